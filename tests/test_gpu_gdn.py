"""GPU parity of the gated-delta-rule prefill (ssd_varlen_gdn_forward) against the
fp64 oracle (oracle.gdn), through the C ABI.

Tolerance as for the SSD path: |gpu - oracle| <= 5e-3 + 5e-3 |oracle| on o and on
every state output; pool slots the call does not write keep their values bit for
bit (canaries).
"""
import numpy as np
import pytest
import torch

import mamba2_ssd_varlen_gb300 as m
import workloads
from oracle.gdn import gdn_forward

pytestmark = pytest.mark.gpu

ATOL = 5e-3
RTOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mamba2_ssd_varlen_gb300 import build
    build.build()
    m.load_library()


def assert_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if got.size == 0:
        return
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    ratio = np.abs(got - ref) / (ATOL + RTOL * np.abs(ref))
    k = int(np.argmax(ratio))
    assert ratio.flat[k] <= 1.0, (f"{what}: max |err|/tol = {ratio.flat[k]:.3f} at "
                                  f"{np.unravel_index(k, ratio.shape)} (got {got.flat[k]:.6g}, ref {ref.flat[k]:.6g})")


def host(t):
    return t.detach().float().cpu().numpy()


def run_full(prob):
    ref = gdn_forward(workloads.to_oracle_gdn(prob))
    call = m.run_gdn(prob)
    torch.cuda.synchronize()
    assert call.status() == 0
    assert_close(host(call.o), ref["o"], "o")
    if call.final_states is not None:
        assert_close(host(call.final_states), ref["final_states"], "final_states")
    if call.chunk_states is not None:
        assert_close(host(call.chunk_states)[: ref["chunk_states"].shape[0]], ref["chunk_states"], "chunk_states")
    if prob["state_pool"] is not None:
        assert_close(host(prob["state_pool"]), ref["state_pool"], "state_pool")
    return call, ref


def _spec(**kw):
    base = dict(name="g", Hk=2, Hv=4, K=128, V=64, lengths=[37, 64, 1, 130, 0, 200], init="all",
                final_slots=True, export_chunks=True, block_size=128)
    base.update(kw)
    return workloads.GdnSpec(**base)


def test_small_config_every_output():
    run_full(workloads.make_gdn_problem("gdn_small", device="cuda", canary=-3.0))


# V = 128 runs the tcgen05 kernel (K = V = 128), other widths the mma.sync kernel.
@pytest.mark.parametrize("V", [64, 128])
def test_every_output_both_kernels(V):
    run_full(workloads.make_gdn_problem(_spec(V=V), seed=30 + V, device="cuda", canary=-3.0))


@pytest.mark.parametrize("V", [64, 128])
def test_resumed_requests_partial_first_chunks(V):
    # num_computed not a multiple of the chunk: partial first chunks, block
    # boundaries at absolute positions, export rows per absolute chunk
    prob = workloads.make_gdn_problem(_spec(V=V), seed=5, device="cuda", num_computed=[3, 64, 0, 100, 5, 70],
                                      canary=2.0)
    run_full(prob)


@pytest.mark.parametrize("V,Hk,Hv", [(32, 1, 1), (128, 2, 4), (256, 1, 4), (96, 3, 3)])
def test_head_shapes(V, Hk, Hv):
    spec = _spec(V=V, Hk=Hk, Hv=Hv, lengths=[70, 5, 129], export_chunks=False, block_size=0)
    run_full(workloads.make_gdn_problem(spec, seed=V + Hk, device="cuda", canary=1.5))


@pytest.mark.parametrize("V", [64, 128])
def test_without_l2norm_and_explicit_scale(V):
    spec = _spec(V=V, l2norm=False, lengths=[90, 64, 17])
    prob = workloads.make_gdn_problem(spec, seed=8, device="cuda", canary=0.5)
    prob["q"] = (prob["q"].float() / 12.0).to(torch.bfloat16)   # keep the un-normalised rule stable
    prob["k"] = (prob["k"].float() / 12.0).to(torch.bfloat16)
    prob["scale"] = 0.7
    run_full(prob)


@pytest.mark.parametrize("V", [64, 128])
def test_long_request_many_chunks(V):
    spec = _spec(V=V, lengths=[1500, 300], block_size=256)
    run_full(workloads.make_gdn_problem(spec, seed=9, device="cuda", canary=-1.0))


@pytest.mark.parametrize("V", [64, 128])
@pytest.mark.parametrize("k", [1, 63, 64, 100])
def test_split_state_resume(k, V):
    L = 333
    spec = _spec(V=V, lengths=[L], export_chunks=False, block_size=0, final_slots=True)
    prob = workloads.make_gdn_problem(spec, seed=12, device="cuda")
    ref = gdn_forward(workloads.to_oracle_gdn(prob))
    first = dict(prob)
    for key in ("q", "k", "v", "g", "beta"):
        first[key] = prob[key][:k].clone()
    first["cu_seqlens"] = torch.tensor([0, k], dtype=torch.int32, device="cuda")
    c1 = m.run_gdn(first)
    torch.cuda.synchronize()
    second = dict(prob)
    for key in ("q", "k", "v", "g", "beta"):
        second[key] = prob[key][k:].clone()
    second["cu_seqlens"] = torch.tensor([0, L - k], dtype=torch.int32, device="cuda")
    second["num_computed"] = torch.tensor([k], dtype=torch.int32, device="cuda")
    second["init_slots"] = prob["final_slots"]            # the first part's final state
    second["final_slots"] = None
    c2 = m.run_gdn(second)
    torch.cuda.synchronize()
    assert c1.status() == 0 and c2.status() == 0
    assert_close(np.concatenate([host(c1.o), host(c2.o)]), ref["o"], "split o")
    assert_close(host(c2.final_states), ref["final_states"], "split final")


@pytest.mark.parametrize("V", [64, 128])
def test_device_error_bits_and_skipped_writes(V):
    spec = _spec(V=V, lengths=[20, 70, 9], export_chunks=False, block_size=64)
    prob = workloads.make_gdn_problem(spec, seed=13, device="cuda", canary=4.0)
    S = prob["state_pool"].shape[0]
    prob["init_slots"][1] = S + 2      # read as zeros
    prob["final_slots"][2] = S         # write skipped
    before = prob["state_pool"].clone()
    call = m.run_gdn(prob)
    torch.cuda.synchronize()
    bits = call.status()
    assert bits & m.DEVERR["INIT_SLOT"] and bits & m.DEVERR["FINAL_SLOT"]
    o = workloads.to_oracle_gdn(prob)
    o["init_slots"] = np.where(o["init_slots"] >= S, -1, o["init_slots"])
    o["final_slots"] = np.where(o["final_slots"] >= S, -1, o["final_slots"])
    ref = gdn_forward(o)
    assert_close(host(call.o), ref["o"], "o")
    assert_close(host(prob["state_pool"]), ref["state_pool"], "state_pool")
    untouched = [s for s in range(S) if np.array_equal(ref["state_pool"][s], host(before[s]))]
    assert torch.equal(prob["state_pool"][untouched].cpu(), before[untouched].cpu())


def test_full_uniform_8x2048_sampled():
    # The bench workload (8 x 2048 tokens, 16 key heads, 32 value heads, 128 x 128
    # states), in the bench's launch, checked on sampled requests and heads.
    prob = workloads.make_gdn_problem("gdn_uniform_8x2048", device="cuda")
    call = m.run_gdn(prob)
    torch.cuda.synchronize()
    assert call.status() == 0
    reqs, heads = [0, 5], [0, 17, 31]
    o = workloads.to_oracle_gdn(prob, requests=reqs, heads=heads)
    ref = gdn_forward(o)
    hidx = torch.tensor(heads, device="cuda")
    toks = torch.tensor(o["tokens"], device="cuda")
    assert_close(host(call.o.index_select(0, toks).index_select(1, hidx)), ref["o"], "o")
    assert_close(host(call.final_states[reqs].index_select(1, hidx)), ref["final_states"], "final_states")


@pytest.mark.parametrize("V", [64, 128])
def test_all_requests_empty(V):
    # T = 0: no chunk runs; every request's final state is its initial state
    # (zeros where the read slot is -1), in the dense output and the final slots.
    spec = _spec(V=V, lengths=[0, 0, 0], export_chunks=False, block_size=0)
    prob = workloads.make_gdn_problem(spec, seed=21, device="cuda", canary=0.75)
    prob["init_slots"][1] = -1
    run_full(prob)
