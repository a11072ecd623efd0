"""GPU parity of the varlen causal conv1d (ssd_varlen_conv1d) against the fp64
oracle (oracle.conv1d), through the C ABI.

y within |gpu - oracle| <= 5e-3 + 5e-3 |oracle| (the forward's tolerance); the
written conv states are raw inputs and must match bit for bit; slots the call
does not write keep their values.
"""
import numpy as np
import pytest
import torch

import mamba2_ssd_varlen_gb300 as m
import workloads
from oracle.conv1d import conv1d

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
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    ratio = np.abs(got - ref) / (ATOL + RTOL * np.abs(ref))
    k = int(np.argmax(ratio)) if ratio.size else 0
    assert ratio.size == 0 or ratio.flat[k] <= 1.0, (
        f"{what}: max |err|/tol = {ratio.flat[k]:.3f} at {np.unravel_index(k, ratio.shape)}")


def run_and_check(prob):
    pool_before = prob["conv_pool"].clone()
    ref = conv1d(workloads.to_oracle_conv(prob))
    call = m.run_conv1d(prob)
    torch.cuda.synchronize()
    assert call.status() == 0
    assert_close(call.y.float().cpu().numpy(), ref["y"], "y")
    pool = prob["conv_pool"].cpu()
    for s, v in ref["writes"].items():
        np.testing.assert_array_equal(pool[s].double().numpy(), v, err_msg=f"conv_pool[{s}]")
    untouched = [s for s in range(pool.shape[0]) if s not in ref["writes"]]
    assert torch.equal(pool[untouched], pool_before.cpu()[untouched])


def _spec(**kw):
    base = dict(name="conv", D=264, W=4, dtype="bf16", lengths=[1, 63, 64, 65, 0, 2, 130, 3], read_zero_every=3)
    base.update(kw)
    return workloads.ConvSpec(**base)


def test_tiny_fp32_config():
    run_and_check(workloads.make_conv_problem("conv_tiny_fp32", device="cuda", canary=-1.0))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("W", [2, 3, 4])
def test_tiles_across_request_boundaries(dtype, W):
    # lengths put request starts and ends inside and at the edges of 64-token
    # tiles, and requests shorter than the conv state
    run_and_check(workloads.make_conv_problem(_spec(W=W, dtype=dtype), seed=W, device="cuda", canary=2.0))


@pytest.mark.parametrize("lengths", [[331], [100, 0, 231], [7, 300, 24]])
def test_strips_across_channel_groups(lengths):
    # warps take even strips of the (channel group, token) units: with three
    # channel groups (D = 520 bf16: 65 vectors, the last group one lane wide) and
    # 331 tokens, strips start inside requests and one crosses into the next group
    spec = _spec(D=520, lengths=lengths)
    run_and_check(workloads.make_conv_problem(spec, seed=len(lengths), device="cuda", canary=1.25))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_silu_over_a_wide_range_of_arguments(dtype):
    # inputs and conv states scaled by 25: the pre-activation values reach about
    # +-100, through SiLU's saturation on both sides (about zero below, the
    # identity above) and the region in between
    prob = workloads.make_conv_problem(_spec(dtype=dtype, lengths=[130, 64, 1, 200]), seed=21, device="cuda",
                                       canary=3.0)
    prob["x"].mul_(25.0)
    prob["conv_pool"].mul_(25.0)
    run_and_check(prob)


def test_no_activation_no_bias_many_channels():
    spec = _spec(D=2056, silu=False, has_bias=False, lengths=[200, 1, 1, 77])
    run_and_check(workloads.make_conv_problem(spec, seed=8, device="cuda", canary=0.5))


def test_no_slots_means_zero_state_and_no_write():
    prob = workloads.make_conv_problem(_spec(), seed=4, device="cuda")
    prob["read_slots"] = None
    prob["write_slots"] = None
    o = workloads.to_oracle_conv(dict(prob, read_slots=torch.full((8,), -1, dtype=torch.int32),
                                      write_slots=torch.full((8,), -1, dtype=torch.int32)))
    ref = conv1d(o)
    call = m.run_conv1d(prob)
    torch.cuda.synchronize()
    assert call.status() == 0
    assert_close(call.y.float().cpu().numpy(), ref["y"], "y")


def test_split_resume_through_the_conv_state():
    # a request split in two calls, the second reading the state the first wrote,
    # gives the unsplit output
    spec = _spec(lengths=[150], read_zero_every=0)
    full = workloads.make_conv_problem(spec, seed=12, device="cuda")
    whole = m.run_conv1d(full)
    k = 97
    first = dict(full, x=full["x"][:k].clone(), cu_seqlens=torch.tensor([0, k], dtype=torch.int32, device="cuda"),
                 conv_pool=full["conv_pool"].clone())
    a = m.run_conv1d(first)
    second = dict(full, x=full["x"][k:].clone(), cu_seqlens=torch.tensor([0, 150 - k], dtype=torch.int32,
                                                                         device="cuda"),
                  conv_pool=first["conv_pool"].clone(), read_slots=full["write_slots"].clone(),
                  write_slots=full["read_slots"].clone())
    b = m.run_conv1d(second)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([a.y, b.y]), whole.y)
    w, r = int(full["write_slots"][0]), int(full["read_slots"][0])
    assert torch.equal(second["conv_pool"][r], full["conv_pool"][w])


def test_device_error_bits():
    prob = workloads.make_conv_problem(_spec(lengths=[10, 0, 5]), seed=6, device="cuda", canary=1.0)
    S = prob["conv_pool"].shape[0]
    prob["read_slots"][0] = S + 1
    prob["write_slots"][2] = S
    call = m.run_conv1d(prob)
    torch.cuda.synchronize()
    bits = call.status()
    assert bits & m.DEVERR["INIT_SLOT"] and bits & m.DEVERR["FINAL_SLOT"]
    bad_cu = workloads.make_conv_problem(_spec(lengths=[4, 4]), seed=6, device="cuda")
    bad_cu["cu_seqlens"][2] = 9   # does not end at T
    call = m.run_conv1d(bad_cu)
    torch.cuda.synchronize()
    assert call.status() & m.DEVERR["CU_SEQLENS"]


def test_full_size_sampled_channels():
    prob = workloads.make_conv_problem("conv_uniform_8x2048", device="cuda")
    call = m.run_conv1d(prob)
    torch.cuda.synchronize()
    assert call.status() == 0
    ch = [0, 1, 7, 8, 2047, 4096, 5375]
    ref = conv1d(workloads.to_oracle_conv(prob, channels=ch))
    idx = torch.tensor(ch, device="cuda")
    assert_close(call.y.index_select(1, idx).float().cpu().numpy(), ref["y"], "y")
    for s, v in ref["writes"].items():
        np.testing.assert_array_equal(prob["conv_pool"][s].index_select(0, idx).double().cpu().numpy(), v)


def test_all_requests_empty():
    # T = 0: every request passes its conv state (or zeros) to its write slot.
    run_and_check(workloads.make_conv_problem(_spec(lengths=[0, 0, 0]), seed=14, device="cuda", canary=0.25))
