"""Child process of test_gpu_timeout.py: runs the scan from the timeout-test
build of the library (SSD_TIMEOUT_TEST: bounded waits give up after 20 ms; the
header's test word makes block 0's producer publish no work item).

Checks, in order: the forward with the word set returns; the device error word
carries SSD_DEVERR_TIMEOUT and header words 4-6 name a barrier of block 0; the
outputs are complete (the other CTAs took every item); the next plan and
forward on the same workspace are clean and correct.  Prints "timeout ok".
"""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import mamba2_ssd_varlen_gb300 as m  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402

HDR_TIMEOUT_AT, HDR_TEST_HOOK = 4, 11


def close(got, ref):
    got = got.detach().float().cpu().numpy().astype(np.float64)
    return float((np.abs(got - ref) / (5e-3 + 5e-3 * np.abs(ref))).max())


def main(lib_path):
    m.LIB_PATH = lib_path
    m.load_library()
    spec = workloads.Spec("timeout", H=8, P=64, N=128, G=2, chunk_size=64, dtype="bf16", has_D=True,
                          has_z=True, init="all", pool_slots=16, final_slots=True)
    prob = workloads.make_problem(spec, seed=91, device="cuda", lengths=[700, 300, 1000, 5], num_computed=[0, 3, 64, 0])
    ref = oracle.forward(workloads.to_oracle(prob))
    call = m.Call(prob)
    assert call.path()[0] == m.PATH_TENSOR_CORE_PAIRED
    call.make_plan()
    hdr = call.workspace[:256].view(torch.int32)
    hdr[HDR_TEST_HOOK] = 1
    call.forward()
    torch.cuda.synchronize()  # the launch returned: every role gave up and left
    words = hdr.cpu().tolist()
    bits = call.status()
    assert bits & m.DEVERR["TIMEOUT"], f"no timeout bit: {bits:#x}"
    site, block, thread = words[HDR_TIMEOUT_AT:HDR_TIMEOUT_AT + 3]
    assert site > 0 and block == 0 and 0 <= thread < 640, (site, block, thread)
    assert close(call.y, ref["y"]) <= 1.0, "the other CTAs did not take every item"
    assert close(call.final_states, ref["final_states"]) <= 1.0
    # the next normal call on the same workspace: a fresh plan clears the word
    call.make_plan()
    call.forward()
    torch.cuda.synchronize()
    assert call.status() == 0
    assert call.workspace[:256].view(torch.int32)[HDR_TIMEOUT_AT].item() == 0
    assert close(call.y, ref["y"]) <= 1.0 and close(call.final_states, ref["final_states"]) <= 1.0
    print("timeout ok", site, block, thread)


if __name__ == "__main__":
    main(sys.argv[1])
