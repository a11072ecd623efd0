"""GPU parity of the decode / speculative-decode step (ssd_varlen_decode) against
the fp64 oracle (oracle.decode), through the C ABI.

Tolerance as for the forward: |gpu - oracle| <= 5e-3 + 5e-3 |oracle| on y and on
every state the step writes.  Slots the step does not write keep their values
bit for bit (canaries), and so do the read anchors.
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
    k = int(np.argmax(ratio)) if ratio.size else 0
    assert ratio.size == 0 or ratio.flat[k] <= 1.0, (
        f"{what}: max |err|/tol = {ratio.flat[k]:.3f} at {np.unravel_index(k, ratio.shape)}")


def run_and_check(prob):
    pool_before = prob["state_pool"].clone()
    ref = oracle.decode(workloads.to_oracle_decode(prob))
    call = m.run_decode(prob)
    torch.cuda.synchronize()
    assert call.status() == 0
    assert_close(call.y.float().cpu().numpy(), ref["y"], "y")
    pool = prob["state_pool"].cpu()
    written = set(ref["writes"])
    for s, v in ref["writes"].items():
        assert_close(pool[s].numpy(), v, f"state_pool[{s}]")
    untouched = [s for s in range(pool.shape[0]) if s not in written]
    assert torch.equal(pool[untouched], pool_before.cpu()[untouched]), "a slot outside the write anchors changed"
    return call, ref


def _spec(**kw):
    base = dict(name="dec", H=8, P=64, N=128, G=2, dtype="bf16", windows=[1, 4, 2, 0, 3, 1, 7, 1],
                has_D=True, has_z=True, read_zero_every=3, write_every=1)
    base.update(kw)
    return workloads.DecodeSpec(**base)


def test_tiny_fp32_config():
    run_and_check(workloads.make_decode_problem("decode_tiny_fp32", device="cuda", canary=-2.0))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
# elements per thread KV and threads per row N / KV: (64, 128) 32 / 4, (128, 128) 64 / 2,
# (32, 64) 8 / 8, (16, 16) 1 / 16, (8, 256) 8 / 32, (33, 64) 16 / 4 with idle threads,
# (256, 64) 64 / 1, (24, 32) 4 / 8, (24, 16) 2 / 8
@pytest.mark.parametrize("P,N", [(64, 128), (128, 128), (32, 64), (16, 16), (8, 256), (33, 64), (256, 64),
                                 (24, 32), (24, 16)])
def test_windows_every_shape(dtype, P, N):
    spec = _spec(P=P, N=N, dtype=dtype)
    run_and_check(workloads.make_decode_problem(spec, seed=11 + P + N, device="cuda", canary=3.5))


def test_sparse_write_anchors_no_gate_no_skip():
    spec = _spec(has_z=False, has_D=False, write_every=3, windows=[5, 1, 6, 2])
    run_and_check(workloads.make_decode_problem(spec, seed=5, device="cuda", canary=-1.0))


def test_plain_decode_one_token_per_request():
    spec = _spec(windows=[1] * 37, G=4)
    run_and_check(workloads.make_decode_problem(spec, seed=9, device="cuda", canary=0.25))


def test_decode_equals_forward_of_the_same_window():
    # The decode step and the prefill forward are two entry points to one
    # recurrence: a window read from slot r that writes on its last token equals
    # a forward of the same tokens from init slot r into that final slot.
    spec = _spec(windows=[3, 2, 4], write_every=99)  # only each window's last token writes
    prob = workloads.make_decode_problem(spec, seed=13, device="cuda", canary=0.0)
    pool_fwd = prob["state_pool"].clone()
    dec = m.run_decode(prob)
    cu = prob["cu_seqlens"].cpu().numpy()
    last = torch.tensor([int(prob["write_slots"][cu[i + 1] - 1]) for i in range(len(cu) - 1)],
                        dtype=torch.int32, device="cuda")
    fwd = {k: prob[k] for k in ("x", "dt", "dt_bias", "A", "B", "C", "D", "z", "cu_seqlens")}
    fwd.update(num_computed=None, chunk_size=16, block_size=0, export_chunks=False, final_dense=False,
               state_pool=pool_fwd, init_slots=prob["read_slots"], final_slots=last, block_table=None)
    call = m.run(fwd)
    torch.cuda.synchronize()
    assert dec.status() == 0 and call.status() == 0
    assert_close(dec.y.float().cpu().numpy(), call.y.float().cpu().numpy(), "y")
    for s in last.tolist():
        assert_close(prob["state_pool"][s].cpu().numpy(), pool_fwd[s].cpu().numpy(), f"slot {s}")


def test_device_error_bits():
    spec = _spec(windows=[2, 1, 3])
    prob = workloads.make_decode_problem(spec, seed=17, device="cuda", canary=1.0)
    S = prob["state_pool"].shape[0]
    prob["read_slots"][1] = S + 3     # out of range: read as zeros
    prob["write_slots"][0] = S        # out of range: write skipped
    pool_before = prob["state_pool"].clone()
    call = m.run_decode(prob)
    torch.cuda.synchronize()
    bits = call.status()
    assert bits & m.DEVERR["INIT_SLOT"] and bits & m.DEVERR["FINAL_SLOT"]
    # request 1 ran from zeros: compare with the oracle given a zero anchor
    o = workloads.to_oracle_decode(prob)
    o["read_slots"] = np.where(o["read_slots"] >= S, -1, o["read_slots"])
    o["write_slots"] = np.where(o["write_slots"] >= S, -1, o["write_slots"])
    ref = oracle.decode(o)
    assert_close(call.y.float().cpu().numpy(), ref["y"], "y")
    for s, v in ref["writes"].items():
        assert_close(prob["state_pool"][s].cpu().numpy(), v, f"state_pool[{s}]")
    written = set(ref["writes"])
    untouched = [s for s in range(S) if s not in written]
    assert torch.equal(prob["state_pool"][untouched].cpu(), pool_before[untouched].cpu())


def test_full_size_spec_decode_sampled():
    # The bench workload (256 requests x 4-token windows, H80 P64 N128, every
    # position keeping its state), in the bench's launch, checked on sampled
    # requests and heads.
    prob = workloads.make_decode_problem("decode_spec_256x4", device="cuda")
    call = m.run_decode(prob)
    torch.cuda.synchronize()
    assert call.status() == 0
    reqs, heads = [0, 77, 128, 255], [0, 13, 79]
    o = workloads.to_oracle_decode(prob, requests=reqs, heads=heads)
    ref = oracle.decode(o)
    hidx = torch.tensor(heads, device="cuda")
    toks = torch.tensor(o["tokens"], device="cuda")
    assert_close(call.y.index_select(0, toks).index_select(1, hidx).float().cpu().numpy(), ref["y"], "y")
    for s, v in ref["writes"].items():
        assert_close(prob["state_pool"][s].index_select(0, hidx).cpu().numpy(), v, f"state_pool[{s}]")


def test_all_windows_empty():
    # T = 0: nothing is read or written; y is empty and the pool keeps its values.
    spec = _spec(windows=[0, 0, 0])
    run_and_check(workloads.make_decode_problem(spec, seed=19, device="cuda", canary=0.5))
