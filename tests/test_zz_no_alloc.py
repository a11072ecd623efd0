"""The workspace-free forward (ssd_varlen_forward_static) against the regular one.

ssd_varlen_forward_static is for callers that cannot allocate device memory
for a workspace (a plugin inside a host application that owns the device
memory pool, or a loop where cudaMalloc's synchronisation or failure is not
acceptable): it runs the same plan and forward with the library's own fixed
scratch array.  This test calls it through the C ABI on batches in a row --
a small one, a larger one with a request spanning several chained segments,
the small one again (whose call must not be disturbed by what the larger one
left in the shared array), then an fp32 batch on the general path -- and
checks every output against ssd_varlen_plan + ssd_varlen_forward within the
parity tolerance; it also checks that an oversized problem is refused before
anything runs.

The file name sorts last so a run that stops at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mamba2_ssd_varlen_gb300 as m
import workloads

pytestmark = pytest.mark.gpu

ATOL = 5e-3
RTOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mamba2_ssd_varlen_gb300 import build
    build.build()
    m.load_library()


def _close(got, ref, what):
    got = got.detach().float().cpu().numpy().astype(np.float64)
    ref = ref.detach().float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape
    ratio = np.abs(got - ref) / (ATOL + RTOL * np.abs(ref))
    assert np.all(np.isfinite(got)) and ratio.max() <= 1.0, f"{what}: max |err|/tol {ratio.max():.3f}"


def _problem(seed, lengths, ncomp, dtype="bf16"):
    P, N = (64, 128) if dtype == "bf16" else (32, 64)
    spec = workloads.Spec("noalloc", H=4, P=P, N=N, G=2, chunk_size=64, dtype=dtype,
                          has_D=True, has_z=True, init="all", pool_slots=64, final_slots=True,
                          export_chunks=True, block_size=128)
    return workloads.make_problem(spec, seed=seed, device="cuda", lengths=lengths,
                                  num_computed=ncomp, canary=-1.0)


def _static_call(prob):
    """Outputs of ssd_varlen_forward_static for prob (pool updated in place)."""
    call = m.Call(prob)  # builds dims and argument structs; its workspace stays unused
    plan = m.ssd_plan()
    lib = m.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    nc = prob.get("num_computed")
    rc = lib.ssd_varlen_forward_static(ctypes.byref(call.dims), ctypes.c_void_p(prob["cu_seqlens"].data_ptr()),
                                       None if nc is None else ctypes.c_void_p(nc.data_ptr()),
                                       ctypes.byref(call.inputs), ctypes.byref(call.outputs), stream,
                                       ctypes.byref(plan))
    assert rc == 0, m.ssd_varlen_strerror(rc)
    torch.cuda.synchronize()
    assert m.ssd_varlen_status(plan) == 0
    return call


def test_static_scratch_forward_matches_regular_forward_twice():
    small = (41, [300, 0, 1, 700], [37, 5, 0, 128], "bf16")
    cases = [small, (42, [2500, 64], [1000, 0], "bf16"), small, (43, [90, 0, 130], [3, 0, 64], "fp32")]
    for seed, lengths, ncomp, dtype in cases:
        ref_prob = _problem(seed, lengths, ncomp, dtype)
        st_prob = _problem(seed, lengths, ncomp, dtype)
        ref = m.run(ref_prob)
        torch.cuda.synchronize()
        assert ref.status() == 0
        got = _static_call(st_prob)
        _close(got.y, ref.y, f"y (seed {seed})")
        _close(got.final_states, ref.final_states, f"final states (seed {seed})")
        _close(got.chunk_states, ref.chunk_states, f"chunk states (seed {seed})")
        _close(st_prob["state_pool"], ref_prob["state_pool"], f"state pool (seed {seed})")


def test_static_scratch_refuses_oversized_problem():
    lib = m.load_library()
    dims = m.make_dims(T=1 << 24, R=8, H=80, P=64, N=128, G=1, chunk_size=256, dtype=m.DTYPE_BF16)
    assert m.ssd_varlen_workspace_size(dims) > m.STATIC_SCRATCH_BYTES
    rc = lib.ssd_varlen_forward_static(ctypes.byref(dims), ctypes.c_void_p(16), None,
                                       ctypes.byref(m.ssd_inputs()), ctypes.byref(m.ssd_outputs()),
                                       None, None)
    assert rc == -8  # SSD_ERR_WORKSPACE, nothing launched
