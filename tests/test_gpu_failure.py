"""Failure detection on the GPU without a fault: a device-side wait that is made to run out.

The child process (tests/failure_child.py) shortens the device wait limit to 300 ms and runs
the deterministic backward on turn counters that never reach their targets.  Its bounded turn
wait must give up, the library must report ATTN_ERR_TIMEOUT through attn_get_device_status, and
the same CUDA context must afterwards run a normal backward that matches the oracle.  Nothing
here traps, faults or waits without a limit."""
import json
import os
import subprocess
import sys

import pytest

from exact_attention_50_gb300 import _lib

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_turn_wait_times_out_and_context_stays_usable():
    r = subprocess.run([sys.executable, os.path.join(HERE, "failure_child.py")], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["status_before"] == _lib.ATTN_OK
    assert out["launch"] == _lib.ATTN_OK
    assert out["status_after_stuck_call"] == _lib.ATTN_ERR_TIMEOUT, out
    assert out["seconds"] < 30, out  # 300 ms limit per wait, not the 4 s default or a hang
    assert out["status_after_normal_call"] == _lib.ATTN_OK, out
    assert max(out["max_err"]) <= 1e-2, out
