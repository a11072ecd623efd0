"""The plan and the forward captured into a CUDA graph and replayed.

Both calls only enqueue work on the caller's stream (the forward's kernels as
programmatic dependent launches, waiting in the kernel for the previous one), so
a stream capture turns them into a graph whose replays must give exactly what
the direct calls give.  Which CTA takes which work item varies from run to run,
but each item's arithmetic does not depend on it, so the outputs are compared
bit for bit: y, the final states, the exported chunk states and the state pool
(final slots and block checkpoints).
"""
import pytest
import torch

import mamba2_ssd_varlen_gb300 as m
import workloads

pytestmark = pytest.mark.gpu

HDR_MODE, MODE_PREPASS, MODE_CHAINED = 9, 0, 1  # plan header word: how segment states are carried


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mamba2_ssd_varlen_gb300 import build
    build.build()
    m.load_library()


def _outputs(call, prob):
    outs = {"y": call.y, "final": call.final_states, "chunks": call.chunk_states, "pool": prob["state_pool"]}
    return {k: v.clone() for k, v in outs.items() if v is not None}


def _clear(call):
    for t in (call.y, call.final_states, call.chunk_states):
        if t is not None:
            t.fill_(float("nan"))


def _same(a, b, what):
    assert a.shape == b.shape, what
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"{what}: replay differs from the direct call"


@pytest.mark.parametrize("H,mode", [(64, MODE_CHAINED), (8, MODE_PREPASS)])
def test_graph_replay_matches_direct_calls(H, mode):
    # Requests of 900-2048 tokens with resume offsets (tail-shortened segments, 256-token
    # chunks exported, 1024-token block checkpoints, initial and final pool slots):
    # with 64 heads the scan chains the segment states itself, with 8 the pre-pass
    # and its chain kernel run first.
    spec = workloads.Spec("graph", H=H, P=64, N=128, G=4, chunk_size=256, dtype="bf16", has_D=True,
                          has_z=True, init="all", pool_slots=120, final_slots=True, export_chunks=True,
                          block_size=1024)
    prob = workloads.make_problem(spec, seed=300 + H, device="cuda",
                                  lengths=[2048, 1300, 1700, 900, 2048, 1536, 1100, 1900],
                                  num_computed=[0, 256, 700, 0, 1024, 5, 0, 2047])
    pool0 = prob["state_pool"].clone()

    direct = m.Call(prob)
    direct()
    torch.cuda.synchronize()
    assert direct.status() == 0
    assert int(direct.workspace[:64].view(torch.int32)[HDR_MODE].item()) == mode
    want = _outputs(direct, prob)

    # Warm the captured call up on a side stream (first-use set-up happens outside
    # the capture), then capture plan + forward on it.
    call = m.Call(prob)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        prob["state_pool"].copy_(pool0)
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()

    for replay in range(2):
        prob["state_pool"].copy_(pool0)
        _clear(call)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        got = _outputs(call, prob)
        for k in want:
            _same(got[k], want[k], f"replay {replay}: {k}")
        err = int(call.workspace[:64].view(torch.int32)[0].item())
        assert err == 0, f"device error bits {err:#x} after replay {replay}"
