"""GPU: the slot-aliasing check (ssd_varlen_check_slots) on the workloads' own
slot tables (clean) and on tables with a planted conflict."""
import pytest
import torch

import mamba2_ssd_varlen_gb300 as m
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mamba2_ssd_varlen_gb300 import build
    build.build()
    m.load_library()


def _block_problem():
    spec = workloads.Spec("chk", H=2, P=64, N=128, G=1, chunk_size=64, dtype="bf16", init="all",
                          pool_slots=200, final_slots=True, block_size=128)
    return workloads.make_problem(spec, seed=3, device="cuda", lengths=[300, 0, 5, 700])


def test_clean_tables_pass():
    prob = _block_problem()
    assert m.ssd_varlen_check_slots(4, prob["init_slots"], prob["final_slots"], prob["block_table"]) == 0
    dp = workloads.make_decode_problem("decode_tiny_fp32", device="cuda")
    T = dp["write_slots"].shape[0]
    # the decode step: read anchors per request, write anchors per token
    reads = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    reads[: dp["read_slots"].shape[0]] = dp["read_slots"]
    assert m.ssd_varlen_check_slots(T, reads, dp["write_slots"]) == 0


def test_final_slot_that_is_read_is_flagged():
    prob = _block_problem()
    prob["final_slots"][3] = prob["init_slots"][0]
    assert m.ssd_varlen_check_slots(4, prob["init_slots"], prob["final_slots"], prob["block_table"]) & m.DEVERR["ALIAS"]


def test_slot_written_twice_is_flagged():
    prob = _block_problem()
    bt = prob["block_table"]
    used = bt[bt >= 0]
    assert used.numel() >= 2
    flat = bt.view(-1)
    idx = (flat >= 0).nonzero().flatten()
    flat[idx[1]] = flat[idx[0]]                     # two block boundaries into one slot
    assert m.ssd_varlen_check_slots(4, prob["init_slots"], prob["final_slots"], bt) & m.DEVERR["ALIAS"]
    prob = _block_problem()
    prob["final_slots"][2] = int(prob["block_table"][prob["block_table"] >= 0][0])   # a final slot = a block slot
    assert m.ssd_varlen_check_slots(4, prob["init_slots"], prob["final_slots"], prob["block_table"]) & m.DEVERR["ALIAS"]
