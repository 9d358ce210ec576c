"""Host test of the per-device one-time set-up used by the tcgen05 launchers
for their shared-memory opt-in (a per-device CUDA attribute): compiles a small
C++ harness around csrc/device_once.h with g++ and checks that the set-up runs
once per device id, is retried after a failure, rejects ids outside its table
and runs exactly once under concurrent launches.  No GPU needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HARNESS = os.path.join(ROOT, "tests", "native", "device_once_harness.cpp")
CSRC = os.path.join(ROOT, "long_context_sequence_seq_gb300", "csrc")


def test_per_device_once(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path / "device_once")
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I" + CSRC, HARNESS, "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split("\n")
    got = dict((ln.split(" ", 1)[0], ln.split(" ", 1)[1]) for ln in out if ln)
    assert got["rc"] == "0"
    assert got["dev0"] == "1" and got["dev1"] == "1"      # once per device, not once per process
    assert got["dev2"] == "3"                             # two failures, then one success
    assert got["fail"] == "7 7 good 0 after 0"
    assert got["range"] == "99 99"
    assert got["dev3"] == "1"                             # 8 threads x 2000 launches: one set-up
