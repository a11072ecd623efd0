"""A bounded device wait that runs out, on purpose (no fault, no trap, no hang).

The scan's waits are bounded: a wait that gives up records SSD_DEVERR_TIMEOUT
and where it was (header words 4-6), then its CTA drains what it issued and
exits.  A test build of the library (compiled with SSD_TIMEOUT_TEST, never the
default build or the bench) shortens the bound to 20 ms and, when a header word
is set, makes block 0's producer publish no work item: block 0's other roles
then time out on the item ring before issuing any copy or MMA.  The child
process checks the recorded words, that the launch returned with complete
outputs from the other CTAs, and that the next normal call is clean.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_timed_out_wait_is_reported_and_the_next_call_is_clean():
    from mamba2_ssd_varlen_gb300 import build
    pkg = os.path.join(ROOT, "mamba2_ssd_varlen_gb300")
    lib = build.build(extra_flags=["-DSSD_TIMEOUT_TEST"],
                      lib_path=os.path.join(pkg, "_lib", "libssd_varlen_timeout.so"),
                      obj_dir=os.path.join(pkg, "_build", "timeout"))
    import oracle
    oracle.build()
    out = subprocess.run([sys.executable, os.path.join(HERE, "timeout_child.py"), lib], capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-4000:]
    assert "timeout ok" in out.stdout
