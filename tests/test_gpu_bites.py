"""GPU: one long prompt prefilled in bites chosen by ssd_varlen_align_bite
equals the unsplit forward and the fp64 oracle ("Automatic prefix caching for
GDN hybrid models (mamba_cache_mode=all) with MTP speculative decoding",
Purpose: kernel-chunk-aligned prefill clipping and block-aligned split).

Each bite resumes from the previous bite's final state (num_computed = its
start) and writes the block checkpoints that fall inside it through the same
block table; every block checkpoint, the output of every token and the last
final state must match the oracle of the unsplit prompt.
"""
import numpy as np
import pytest
import torch

import mamba2_ssd_varlen_gb300 as m
import oracle
import workloads

pytestmark = pytest.mark.gpu

ATOL = 5e-3
RTOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mamba2_ssd_varlen_gb300 import build
    build.build()
    oracle.build()
    m.load_library()


def assert_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    ratio = np.abs(got - ref) / (ATOL + RTOL * np.abs(ref))
    k = int(np.argmax(ratio))
    assert ratio.flat[k] <= 1.0, f"{what}: max |err|/tol = {ratio.flat[k]:.3f} at {np.unravel_index(k, ratio.shape)}"


@pytest.mark.parametrize("Q,bs,prefix,budgets", [
    (64, 256, 0, [300, 100, 700, 50, 400, 257]),
    (128, 512, 100, [1500, 90, 2000, 600]),      # a 100-token prefix computed elsewhere
    (32, 64, 37, [40, 64, 65, 7, 200]),
])
def test_prefill_in_aligned_bites(Q, bs, prefix, budgets):
    L = 1700
    spec = workloads.Spec("bites", H=4, P=64, N=128, G=2, chunk_size=Q, dtype="bf16", has_D=True, has_z=True,
                          init="all", pool_slots=L // bs + 8, final_slots=True, block_size=bs)
    prob = workloads.make_problem(spec, seed=31, device="cuda", lengths=[L], canary=-7.0)
    ref = oracle.forward(workloads.to_oracle(prob))
    S = prob["state_pool"].shape[0]
    used = {int(prob["init_slots"][0]), int(prob["final_slots"][0])}
    used.update(int(v) for v in prob["block_table"].flatten().tolist() if v >= 0)
    scratch = [s for s in range(S) if s not in used][:2]
    assert len(scratch) == 2

    pool = prob["state_pool"]
    dev = "cuda"
    pos, cur, k, ys, bites = 0, int(prob["init_slots"][0]), 0, [], []
    while pos < L:
        if pos == 0 and prefix:
            end = prefix
        else:
            end = m.ssd_varlen_align_bite(pos, min(L, pos + budgets[k % len(budgets)]), L, bs)
            k += 1
            if end == pos:  # the budget is below one block: nothing this step
                continue
        nxt = int(prob["final_slots"][0]) if end == L else scratch[k % 2]
        sub = dict(prob)
        for key in ("x", "dt", "B", "C", "z"):
            sub[key] = prob[key][pos:end].clone()  # a fresh, aligned allocation
        sub["cu_seqlens"] = torch.tensor([0, end - pos], dtype=torch.int32, device=dev)
        sub["num_computed"] = torch.tensor([pos], dtype=torch.int32, device=dev)
        sub["init_slots"] = torch.tensor([cur], dtype=torch.int32, device=dev)
        sub["final_slots"] = torch.tensor([nxt], dtype=torch.int32, device=dev)
        call = m.run(sub)
        torch.cuda.synchronize()
        assert call.status() == 0
        ys.append(call.y.float().cpu().numpy())
        bites.append((pos, end))
        pos, cur = end, nxt
    assert bites[0][0] == 0 and bites[-1][1] == L
    last_aligned = L // bs * bs
    assert all(b % bs == 0 or b > last_aligned or a % bs for a, b in bites[1 if prefix else 0:])
    assert_close(np.concatenate(ys), ref["y"], "y over the bites")
    host = pool.cpu().numpy()
    for s in used - {int(prob["init_slots"][0])}:
        assert_close(host[s], ref["state_pool"][s], f"state_pool[{s}]")
