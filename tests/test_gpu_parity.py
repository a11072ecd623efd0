"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerance (the SSD varlen pages settle on atol = rtol = 5e-3 for the varlen
SSD tests, "[Bugfix] Mamba2 SSD varlen bug fix initstates decay", Purpose):
every element of y and of every state output satisfies
    |gpu - oracle| <= 5e-3 + 5e-3 * |oracle|.
Small cases are compared in full; the full-size workloads (in the launch
configuration bench.py times) on sampled requests and heads.
"""
import numpy as np
import pytest
import torch

import mamba2_ssd_varlen_gb300 as m
import oracle
import seg_rule
import workloads
from oracle import checkpoints

pytestmark = pytest.mark.gpu

ATOL = 5e-3
RTOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mamba2_ssd_varlen_gb300 import build
    build.build()
    oracle.build()
    m.load_library()


def assert_close(got, ref, what, scale=1.0):
    """Every element within scale * (ATOL + RTOL |ref|).  scale = 2 compares two GPU
    runs with each other: each is within the tolerance of the exact result (the
    oracle comparisons), so by the triangle inequality the two are within twice
    it -- and two bf16 outputs can differ by one bf16 step (1/8 at 22.4, above
    the 0.117 a single tolerance allows there) while both match the oracle."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if got.size == 0:
        return
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    ratio = err / (scale * (ATOL + RTOL * np.abs(ref)))
    k = int(np.argmax(ratio))
    assert ratio.flat[k] <= 1.0, (f"{what}: max |err|/tol = {ratio.flat[k]:.3f} at "
                                  f"{np.unravel_index(k, ratio.shape)} (got {got.flat[k]:.6g}, "
                                  f"ref {ref.flat[k]:.6g})")


def host(t):
    return t.detach().float().cpu().numpy()


def run_full(prob, check_pool=True):
    """Run the library and compare every output buffer with the oracle."""
    ref = oracle.forward(workloads.to_oracle(prob))
    pool_before = None if prob["state_pool"] is None else prob["state_pool"].clone()
    call = m.run(prob)
    torch.cuda.synchronize()
    hdr = call.workspace[:224].view(torch.int32).cpu().tolist()
    assert call.status() == 0, f"device error; header words 0-55: {hdr}"
    assert_close(host(call.y), ref["y"], "y")
    if call.final_states is not None:
        assert_close(host(call.final_states), ref["final_states"], "final_states")
    if call.chunk_states is not None:
        assert_close(host(call.chunk_states)[: ref["chunk_states"].shape[0]], ref["chunk_states"],
                     "chunk_states")
    if check_pool and prob["state_pool"] is not None:
        assert_close(host(prob["state_pool"]), ref["state_pool"], "state_pool")
    return call, ref, pool_before


SMALL = workloads.Spec("small", H=4, P=64, N=128, G=2, chunk_size=64, dtype="bf16",
                       has_D=True, has_z=True, init="all", pool_slots=96, final_slots=True,
                       export_chunks=True, block_size=128)


def test_tiny_fp32_config():
    prob = workloads.make_problem("tiny_fp32", device="cuda")
    run_full(prob)


@pytest.mark.parametrize("Q", [16, 32, 64, 128, 256])
def test_ragged_batch_every_output(Q):
    lengths = [1, 127, 128, 129, 300, 0, 700, 5]
    ncomp = [0, 5, 128, 0, 37, 3, 1000, 250]
    spec = workloads.Spec(**{**SMALL.__dict__, "chunk_size": Q, "block_size": max(Q, 128)})
    prob = workloads.make_problem(spec, seed=100 + Q, device="cuda", lengths=lengths,
                                  num_computed=ncomp, canary=-3.0)
    run_full(prob)


@pytest.mark.parametrize("P", [64, 128])
def test_long_requests_span_several_segments(P):
    # Requests longer than one work segment (2048 tokens) are split into
    # segments whose entering states are chained on the device; one starts
    # mid-chunk (num_computed 1000) from an initial state.
    spec = workloads.Spec("long", H=2, P=P, N=128, G=1, chunk_size=128, dtype="bf16",
                          has_D=True, has_z=True, init="all", pool_slots=64, final_slots=True,
                          export_chunks=True, block_size=1024)
    prob = workloads.make_problem(spec, seed=31, device="cuda", lengths=[5000, 4096, 3],
                                  num_computed=[1000, 0, 2047], canary=1.5)
    run_full(prob)


HDR_MODE, MODE_PREPASS, MODE_CHAINED = 9, 0, 1  # plan header word: how segment states are carried


def plan_mode(call):
    return int(call.workspace[:64].view(torch.int32)[HDR_MODE].item())


@pytest.mark.parametrize("P", [64, 128])
def test_chained_segment_states(P):
    # Twelve requests of 2000-2600 tokens, most crossing a segment boundary
    # (2048 tokens, 8192 on the one-head path; some from a resume offset), none
    # long next to the batch: the
    # plan chains the segment states through the workspace -- the CTA that ends
    # a segment publishes its state, the one running the next segment picks it
    # up -- with no state pre-pass.  Every output of sampled requests and heads
    # against the oracle.
    spec = workloads.Spec("chain", H=32, P=P, N=128, G=4, chunk_size=128, dtype="bf16", has_D=True,
                          has_z=True, init="all", pool_slots=200, final_slots=True, export_chunks=True,
                          block_size=256)
    lengths = [2600, 2100, 2500, 2300, 2450, 2000, 2550, 2200, 2350, 2400, 2150, 2250]
    ncomp = [0, 100, 1500, 0, 40, 2047, 0, 1000, 7, 0, 300, 1]
    if P == 128:
        # the one-head path cuts at multiples of 8192: resume just below one
        ncomp = [c + 6144 for c in ncomp]
    prob = workloads.make_problem(spec, seed=61 + P, device="cuda", lengths=lengths, num_computed=ncomp,
                                  canary=0.75)
    call = _sampled_check(prob, [0, 2, 5, 7, 11], [0, 13, 31])
    assert plan_mode(call) == MODE_CHAINED


@pytest.mark.parametrize("P", [64, 128])
@pytest.mark.parametrize("H,mode", [(64, 1), (8, 0)])
def test_mid_length_batch_tail_shortened_segments(P, H, mode):
    # Requests averaging between 1024 and 2048 tokens are cut into tail-shortened
    # segments (a 2048-token request: 1280 + 512 + 256); resume offsets put
    # segment, chunk and block boundaries (1024-token checkpoints, 256-token
    # chunks) at different places.  With 64 heads the plan
    # chains the segment states, with 8 (the longest request then outlasts a CTA's
    # share of the work) it takes the pre-pass.  Every output of sampled requests
    # and heads against the oracle.
    spec = workloads.Spec("mid", H=H, P=P, N=128, G=4, chunk_size=256, dtype="bf16", has_D=True,
                          has_z=True, init="all", pool_slots=120, final_slots=True, export_chunks=True,
                          block_size=1024)
    lengths = [2048, 1300, 1700, 900, 2048, 1536, 1100, 1900]
    ncomp = [0, 256, 700, 0, 1024, 5, 0, 2047]
    prob = workloads.make_problem(spec, seed=90 + P + H, device="cuda", lengths=lengths, num_computed=ncomp,
                                  canary=0.5)
    call = _sampled_check(prob, [0, 2, 5, 7], [0, 3, H - 1])
    assert plan_mode(call) == (MODE_CHAINED if mode else MODE_PREPASS)
    assert call.plan.seg_len == 2048 and call.plan.flags & seg_rule.PLAN_TAIL_SEGS


def plan_segments(call, with_order=False):
    """(req_first_seg, segments[, order]) from the plan's workspace: the header (64
    words), then req_first_chunk and req_first_seg (R + 1 words each), the segment
    list (req, first token, length, absolute start; plan.max_segs entries) and the
    order the scan takes the segments in, each region 256-byte aligned."""
    R = call.dims.R
    al = lambda v: (v + 255) // 256 * 256
    off_rfs = al(256 + 4 * (R + 1))
    off_segs = al(off_rfs + 4 * (R + 1))
    off_order = al(off_segs + 16 * call.plan.max_segs)
    ws = call.workspace
    nsegs = int(ws[:64 * 4].view(torch.int32)[2].item())
    rfs = ws[off_rfs:off_rfs + 4 * (R + 1)].view(torch.int32).cpu().tolist()
    segs = ws[off_segs:off_segs + 16 * nsegs].view(torch.int32).view(-1, 4).cpu().tolist()
    if not with_order:
        return rfs, segs
    order = ws[off_order:off_order + 4 * nsegs].view(torch.int32).cpu().tolist()
    return rfs, segs, order


@pytest.mark.parametrize("R", [400, 1300])
def test_many_requests(R):
    # 400 requests (ranked by segment count alone) and 1300 (the plan's CTA has
    # at most 1024 threads, so every per-request pass loops; request order):
    # lengths 1-600 with every 97th request 2500 tokens long (two segments),
    # chained.  The segment list against the rule, the order round by round, and
    # sampled outputs against the oracle.
    rng = np.random.default_rng(5)
    lengths = [2500 if i % 97 == 3 else int(rng.integers(1, 600)) for i in range(R)]
    ncomp = [int(rng.integers(0, 300)) if i % 5 == 0 else 0 for i in range(R)]
    spec = workloads.Spec("many_req", H=8, P=64, N=128, G=2, chunk_size=128, dtype="bf16", has_D=True,
                          has_z=True, init="half_even", pool_slots=2 * R, final_slots=True)
    prob = workloads.make_problem(spec, seed=303, device="cuda", lengths=lengths, num_computed=ncomp)
    rule = seg_rule.rule_of(sum(lengths), R, P=64, H=8, G=2)
    assert rule == (2048, False)
    call = _sampled_check(prob, [0, 3, R // 2, R - 1], [0, 7])
    assert plan_mode(call) == MODE_CHAINED
    rfs, segs, order = plan_segments(call, with_order=True)
    for i in range(R):
        mine = segs[rfs[i]:rfs[i + 1]]
        assert [mine[0][3]] + [sg[3] + sg[2] for sg in mine] == seg_rule.cuts(ncomp[i], lengths[i], *rule), i
    count = [rfs[i + 1] - rfs[i] for i in range(R)]
    if R <= 1024:  # round, more segments first, then request order
        keys = [(sid - rfs[segs[sid][0]], -count[segs[sid][0]], segs[sid][0]) for sid in order]
    else:  # round, then request order
        keys = [(sid - rfs[segs[sid][0]], segs[sid][0]) for sid in order]
    assert keys == sorted(keys) and len(keys) == len(segs)


def test_chained_rounds_take_the_longest_chains_first():
    # Chained mode on a batch whose requests have 1-3 segments (2048-token cuts):
    # the scan takes every request's k-th segment after all (k-1)-th ones, and
    # within a round the requests with more segments first, then the longer ones,
    # ties in request order.
    spec = workloads.Spec("order", H=128, P=64, N=128, G=8, chunk_size=256, dtype="bf16", has_D=True,
                          has_z=True, init="half_even", pool_slots=40, final_slots=True)
    lengths = [4100, 100, 2100, 500, 1, 5000, 700, 1024, 50, 900, 300, 200, 100, 100, 100, 100]
    ncomp = [0, 0, 300, 0, 0, 5, 1000, 0, 0, 200, 0, 0, 0, 0, 0, 0]
    prob = workloads.make_problem(spec, seed=77, device="cuda", lengths=lengths, num_computed=ncomp)
    call = _sampled_check(prob, [0, 5, 15], [0, 127])
    assert plan_mode(call) == MODE_CHAINED
    rfs, segs, order = plan_segments(call, with_order=True)
    count = [rfs[i + 1] - rfs[i] for i in range(len(lengths))]
    assert sorted(order) == list(range(len(segs)))
    keys = []
    for sid in order:
        i = segs[sid][0]
        keys.append((sid - rfs[i], -count[i], -lengths[i], i))  # (round, longer chains, longer, request)
    assert keys == sorted(keys), keys
    assert max(count) == 3 and [k[3] for k in keys[:3]] == [5, 0, 2]  # 3 (5000 tokens), 3, then 2 segments


@pytest.mark.parametrize("lengths,ncomp,P,rule", [
    # mid-length (tail-shortened): a long request whose head is cut in three,
    # resumes, a 1-token and a 300-token request
    ([5000, 1100, 1500, 300, 2048, 600, 1700, 2600, 1, 1000], [0, 256, 700, 5, 1024, 0, 2047, 77, 3, 129],
     64, (2048, True)),
    # short on average: multiples of 2048
    ([900, 300, 2500, 100], [0, 1000, 7, 0], 64, (2048, False)),
    # long on average: multiples of 2048
    ([6000, 10], [100, 0], 64, (2048, False)),
    # tail-shortened with an empty request (one empty segment: final = initial state)
    ([2048, 0, 2048, 1500], [0, 0, 100, 7], 64, (2048, True)),
    # the one-head path, long on average: multiples of 8192
    ([9000, 3000, 17000], [0, 100, 5000], 128, (8192, False)),
])
def test_plan_segments_follow_the_rule(lengths, ncomp, P, rule):
    # The segment list the plan builds on the device, request by request, against
    # the rule restated in seg_rule.py; sampled outputs against the oracle.
    spec = workloads.Spec("segs", H=8, P=P, N=128, G=2, chunk_size=256, dtype="bf16", has_D=True,
                          has_z=True, init="all", pool_slots=40, final_slots=True, export_chunks=True,
                          block_size=1024)
    prob = workloads.make_problem(spec, seed=500 + len(lengths), device="cuda", lengths=lengths, num_computed=ncomp)
    assert seg_rule.rule_of(sum(lengths), len(lengths), P=P, H=8, G=2) == rule
    call = _sampled_check(prob, [0, len(lengths) - 1], [0, 7])
    assert call.plan.seg_len == rule[0] and bool(call.plan.flags & seg_rule.PLAN_TAIL_SEGS) == rule[1]
    rfs, segs = plan_segments(call)
    cu = prob["cu_seqlens"].cpu().tolist()
    for i, (L, s) in enumerate(zip(lengths, ncomp)):
        mine = segs[rfs[i]:rfs[i + 1]]
        assert all(sg[0] == i for sg in mine)
        got = [mine[0][3]] + [sg[3] + sg[2] for sg in mine]
        assert got == seg_rule.cuts(s, L, *rule), (i, got)
        # first tokens are packed positions: request start + (absolute start - s)
        assert [sg[1] for sg in mine] == [cu[i] + (c - s) for c in got[:-1]]


def test_long_request_uses_the_state_pre_pass():
    # One request far longer than the rest of the batch: chaining its segments
    # would make it one serial chain, so the plan computes the segment states
    # in a pre-pass instead.
    spec = workloads.Spec("prepass", H=4, P=64, N=128, G=2, chunk_size=128, dtype="bf16", has_D=True,
                          has_z=False, init="all", pool_slots=16, final_slots=True)
    prob = workloads.make_problem(spec, seed=71, device="cuda", lengths=[6000, 10], num_computed=[100, 0])
    call, _, _ = run_full(prob)
    assert plan_mode(call) == MODE_PREPASS


@pytest.mark.parametrize("P,Q", [(64, 64), (128, 128)])
def test_more_items_than_sms(P, Q):
    # More (segment, head) work items than SMs, so CTAs draw several items
    # each from the work ticket; initial states, a resume offset, chunk exports
    # and block checkpoints on every item.
    spec = workloads.Spec("many", H=64, P=P, N=128, G=4, chunk_size=Q, dtype="bf16",
                          has_D=True, has_z=True, init="all", pool_slots=32, final_slots=True,
                          export_chunks=True, block_size=256)
    prob = workloads.make_problem(spec, seed=41 + P, device="cuda", lengths=[1000, 900, 1100, 1001],
                                  num_computed=[0, 64, 5, 1000], canary=2.5)
    run_full(prob)


def test_initial_state_decay_in_first_chunk_768_tokens_q128():
    # The larger failing shape of the initial-state decay bugfix (768 tokens,
    # chunk_size 128), with an initial state and a resume offset inside a chunk.
    spec = workloads.Spec("p2", H=4, P=64, N=128, G=1, chunk_size=128, dtype="bf16",
                          has_D=True, has_z=False, init="all", pool_slots=8, final_slots=True)
    for ncomp in ([0], [77]):
        prob = workloads.make_problem(spec, seed=21, device="cuda", lengths=[768],
                                      num_computed=ncomp)
        run_full(prob)


def test_chunk_size_does_not_change_results():
    # With the per-chunk export on (and no block table) the tensor-core kernel
    # cuts its pieces at the chunk size, so chunk sizes 16 ... 128 run on
    # different internal tiles (asserted through the path query); y, the final
    # states and the written pool slots must not depend on it.
    outs = {}
    tiles = {}
    for Q in (16, 32, 64, 128, 256):
        spec = workloads.Spec(**{**SMALL.__dict__, "chunk_size": Q, "export_chunks": True,
                                 "block_size": 0})
        prob = workloads.make_problem(spec, seed=7, device="cuda", lengths=[513, 40, 1000],
                                      num_computed=[3, 0, 64])
        call, ref, _ = run_full(prob)
        path, tiles[Q] = call.path()
        assert path == m.PATH_TENSOR_CORE_PAIRED
        outs[Q] = (host(call.y), host(call.final_states), host(prob["state_pool"]))
    assert tiles == {16: 16, 32: 32, 64: 64, 128: 128, 256: 128}
    for Q in (16, 32, 64, 128):
        # y is rounded to bf16 by each run: two runs within twice the tolerance;
        # the fp32 states within the tolerance itself
        assert_close(outs[Q][0], outs[256][0].astype(np.float64), f"y Q={Q} vs 256", scale=2.0)
        assert_close(outs[Q][1], outs[256][1].astype(np.float64), f"final Q={Q} vs 256")
        assert_close(outs[Q][2], outs[256][2].astype(np.float64), f"pool Q={Q} vs 256")


def test_tile_follows_block_size_with_a_block_table():
    # A block table without an export cuts pieces at the largest power of two
    # dividing the block size (at most 128): block size 96 gives 32-token tiles.
    spec = workloads.Spec(**{**SMALL.__dict__, "chunk_size": 32, "export_chunks": False,
                             "block_size": 96})
    prob = workloads.make_problem(spec, seed=17, device="cuda", lengths=[200, 97, 5],
                                  num_computed=[0, 95, 3], canary=-1.0)
    call, _, _ = run_full(prob)
    assert call.path() == (m.PATH_TENSOR_CORE_PAIRED, 32)


def test_every_request_crosses_a_segment_boundary():
    # Each request holds two tokens on either side of a multiple of the work
    # segment length (2048), so every request has one chained segment state:
    # the largest count the workspace is sized for with this many tokens.
    spec = workloads.Spec("cross", H=2, P=64, N=128, G=1, chunk_size=64, dtype="bf16",
                          has_D=True, has_z=True, init="all", pool_slots=16, final_slots=True,
                          export_chunks=True, block_size=64)
    prob = workloads.make_problem(spec, seed=5, device="cuda", lengths=[2, 2, 2],
                                  num_computed=[2047, 4095, 10239], canary=0.25)
    run_full(prob)


def test_packed_equals_separate_runs():
    lengths = [300, 1, 0, 650]
    spec = workloads.Spec(**{**SMALL.__dict__, "export_chunks": False, "block_size": 0,
                             "init": "none", "final_slots": False})
    prob = workloads.make_problem(spec, seed=8, device="cuda", lengths=lengths)
    packed = m.run(prob)
    torch.cuda.synchronize()
    cu = prob["cu_seqlens"].cpu().tolist()
    for i, L in enumerate(lengths):
        sub = dict(prob)
        a, b = cu[i], cu[i + 1]
        for k in ("x", "dt", "B", "C", "z"):
            sub[k] = prob[k][a:b].clone()
        sub["cu_seqlens"] = torch.tensor([0, L], dtype=torch.int32, device="cuda")
        if L == 0:
            continue
        one = m.run(sub)
        torch.cuda.synchronize()
        assert_close(host(one.y), host(packed.y)[a:b].astype(np.float64), f"y req {i}")
        assert_close(host(one.final_states[0]), host(packed.final_states[i]).astype(np.float64),
                     f"final req {i}")


@pytest.mark.parametrize("k", [1, 100, 128, 129, 500])
def test_split_state_resume(k):
    """Run a prefix, feed its final state back as the initial state of the
    suffix (num_computed = k), and compare with the unsplit run."""
    L = 777
    spec = workloads.Spec("split", H=4, P=64, N=128, G=2, chunk_size=128, dtype="bf16",
                          has_D=True, has_z=True, init="none")
    prob = workloads.make_problem(spec, seed=9, device="cuda", lengths=[L])
    whole = m.run(prob)
    pre = dict(prob)
    for key in ("x", "dt", "B", "C", "z"):
        pre[key] = prob[key][:k].clone()
    pre["cu_seqlens"] = torch.tensor([0, k], dtype=torch.int32, device="cuda")
    first = m.run(pre)
    torch.cuda.synchronize()
    post = dict(prob)
    for key in ("x", "dt", "B", "C", "z"):
        post[key] = prob[key][k:].clone()
    post["cu_seqlens"] = torch.tensor([0, L - k], dtype=torch.int32, device="cuda")
    post["num_computed"] = torch.tensor([k], dtype=torch.int32, device="cuda")
    post["state_pool"] = first.final_states.clone()
    post["init_slots"] = torch.tensor([0], dtype=torch.int32, device="cuda")
    second = m.run(post)
    torch.cuda.synchronize()
    ref = oracle.forward(workloads.to_oracle(prob))
    y = np.concatenate([host(first.y), host(second.y)])
    assert_close(y, ref["y"], "split y")
    assert_close(host(second.final_states), ref["final_states"], "split final")
    assert_close(host(whole.y), ref["y"], "whole y")


def test_fp32_path_medium():
    spec = workloads.Spec("f32", H=3, P=32, N=64, G=3, chunk_size=32, dtype="fp32",
                          has_D=True, has_z=True, init="all", pool_slots=40, final_slots=True,
                          export_chunks=True, block_size=64)
    prob = workloads.make_problem(spec, seed=12, device="cuda", lengths=[90, 3, 200],
                                  num_computed=[10, 0, 64], canary=9.0)
    run_full(prob)


def test_device_error_bits_and_skipped_writes():
    spec = workloads.Spec("err", H=2, P=64, N=128, G=1, chunk_size=64, dtype="bf16",
                          has_D=False, init="all", pool_slots=16, final_slots=True)
    prob = workloads.make_problem(spec, seed=13, device="cuda", lengths=[10, 20])
    prob["init_slots"] = torch.tensor([99, -1], dtype=torch.int32, device="cuda")
    prob["final_slots"] = torch.tensor([5, 1000], dtype=torch.int32, device="cuda")
    before = prob["state_pool"].clone()
    call = m.run(prob)
    torch.cuda.synchronize()
    bits = call.status()
    assert bits & m.DEVERR["INIT_SLOT"] and bits & m.DEVERR["FINAL_SLOT"]
    assert call.status() == 0  # status clears the word
    # The bad init slot reads as zeros: request 0 equals a zero-init run.
    ref = oracle.forward(workloads.to_oracle({**prob, "init_slots": None, "final_slots": None,
                                              "state_pool": None}))
    assert_close(host(call.y), ref["y"], "y with zero init")
    after = prob["state_pool"]
    assert torch.equal(torch.cat([after[:5], after[6:]]), torch.cat([before[:5], before[6:]]))

    bad = dict(prob)
    bad["cu_seqlens"] = torch.tensor([0, 20, 10], dtype=torch.int32, device="cuda")
    bad["init_slots"] = None
    bad["final_slots"] = None
    call = m.run(bad)
    torch.cuda.synchronize()
    assert call.status() & m.DEVERR["CU_SEQLENS"]


# ---- full-size workloads, sampled -------------------------------------------

def _sampled_check(prob, requests, heads):
    o = workloads.to_oracle(prob, requests=requests, heads=heads)
    pool_before = None if prob["state_pool"] is None else prob["state_pool"]
    ref = oracle.forward(o)
    call = m.run(prob)
    torch.cuda.synchronize()
    assert call.status() == 0
    cu = prob["cu_seqlens"].cpu().tolist()
    sub_cu = o["cu_seqlens"]
    hidx = torch.tensor(heads, device="cuda")
    for j, i in enumerate(requests):
        a, b = cu[i], cu[i + 1]
        sa, sb = int(sub_cu[j]), int(sub_cu[j + 1])
        assert_close(host(call.y[a:b].index_select(1, hidx)), ref["y"][sa:sb], f"y req {i}")
        if call.final_states is not None:
            assert_close(host(call.final_states[i].index_select(0, hidx)), ref["final_states"][j],
                         f"final req {i}")
    if call.chunk_states is not None:
        lengths = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
        nc = prob["num_computed"]
        _, first = checkpoints.checkpoint_records(lengths, None if nc is None else nc.cpu().tolist(),
                                                  prob["chunk_size"])
        sub_first = ref["first_chunk"]
        for j, i in enumerate(requests):
            got = host(call.chunk_states[first[i]:first[i + 1]].index_select(1, hidx))
            assert_close(got, ref["chunk_states"][sub_first[j]:sub_first[j + 1]], f"chunks req {i}")
    if prob["state_pool"] is not None:
        new_pool = ref["state_pool"]
        for s, v in new_pool.slots.items():
            assert_close(host(prob["state_pool"][s].index_select(0, hidx)), v, f"pool slot {s}")
    return call


def test_full_uniform_8x2048():
    prob = workloads.make_problem("uniform_8x2048", device="cuda")
    _sampled_check(prob, [0, 7], [0, 41, 79])


def test_full_varlen_lognormal_32k():
    prob = workloads.make_problem("varlen_lognormal_32k", device="cuda")
    lens = prob["lengths"]
    order = np.argsort(lens)
    reqs = sorted({int(order[-1]), int(order[0]), 2, 3})
    _sampled_check(prob, reqs, [0, 77, 127])


@pytest.mark.parametrize("Q", [128, 256])
def test_full_long_131072(Q):
    prob = workloads.make_problem("long_131072", device="cuda", chunk_size=Q)
    _sampled_check(prob, [0], [0, 63])


def test_full_long_131072_chunk_sizes_agree():
    # The long request at chunk sizes 64 and 256, both exporting every chunk, so
    # the scan runs on 64- and 128-token tiles (asserted through the path query):
    # y and the final state compared directly between the two runs, on every head
    # and token (on the device), and every fourth Q=64 export row against the
    # Q=256 rows (the same chunk ends).
    runs, tiles = {}, {}
    for Q in (64, 256):
        prob = workloads.make_problem("long_131072", device="cuda", chunk_size=Q)
        call = m.run(prob)
        torch.cuda.synchronize()
        assert call.status() == 0
        tiles[Q] = call.path()[1]
        runs[Q] = call
        del prob
    assert tiles == {64: 64, 256: 128}
    a, b = runs[64], runs[256]

    def ratio(got, ref):
        got, ref = got.float(), ref.float()
        return float(((got - ref).abs() / (ATOL + RTOL * ref.abs())).max())

    # y rounded to bf16 by each run: within twice the tolerance (see assert_close);
    # the fp32 states within the tolerance itself
    assert ratio(a.y, b.y) <= 2.0
    assert ratio(a.final_states, b.final_states) <= 1.0
    assert ratio(a.chunk_states[3::4], b.chunk_states) <= 1.0


def test_full_block_checkpointed_varlen():
    prob = workloads.make_problem("block_ckpt_varlen", device="cuda")
    lens = prob["lengths"]
    order = np.argsort(lens)
    reqs = sorted({int(order[-1]), int(order[0]), 17, 64})
    _sampled_check(prob, reqs, [0, 35, 63])


def test_all_requests_empty():
    # T = 0: no token buffers; every request's final state (dense and in its final
    # slot) is its initial state, zeros where it has no initial slot.
    spec = workloads.Spec("empty", H=4, P=64, N=128, G=2, chunk_size=64, dtype="bf16", has_D=True, has_z=True,
                          init="all", pool_slots=16, final_slots=True)
    prob = workloads.make_problem(spec, seed=23, device="cuda", lengths=[0, 0, 0], canary=-4.0)
    prob["init_slots"][1] = -1
    run_full(prob)


@pytest.mark.parametrize("P,N", [(64, 64), (32, 128), (96, 256), (8, 16)])
def test_bf16_shapes_on_the_general_path(P, N):
    # bf16 shapes the tensor-core kernel does not take (P not 64/128 or N != 128)
    # run on the token-serial path: every output against the oracle.
    spec = workloads.Spec("gen", H=3, P=P, N=N, G=3, chunk_size=32, dtype="bf16", has_D=True, has_z=True,
                          init="all", pool_slots=40, final_slots=True, export_chunks=True, block_size=64)
    prob = workloads.make_problem(spec, seed=P + N, device="cuda", lengths=[90, 0, 200, 1],
                                  num_computed=[3, 0, 64, 10], canary=0.5)
    run_full(prob)
