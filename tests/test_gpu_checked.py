"""The small-shape GPU parity tests again, against the bounds-checked build
of the library (-DULYSSES_CHECKS, loaded with ULYSSES_CHECKED=1 in a child
process): every kernel checks its global-memory indexes against the buffers
it was given, so an index that strays outside a buffer is reported by
ulysses_check (ULYSSES_ERR_BOUNDS, which fails the test that checks) instead
of touching memory outside it.  Ragged S, documents that cross tiles and
ranks, GQA, kv-head replication, padding, the ring driver, the fused layer,
the projections and the guard-byte checks are all covered; the full-size
workloads are left to the normal build."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FILES = ["tests/test_gpu_checked_variant.py", "tests/test_gpu_attention.py", "tests/test_gpu_relayout.py",
         "tests/test_gpu_rescale.py", "tests/test_gpu_ring.py", "tests/test_gpu_replication.py",
         "tests/test_gpu_fused.py", "tests/test_gpu_proj.py", "tests/test_gpu_guard.py",
         "tests/test_gpu_watchdog.py"]
# the full-size shapes stay with the normal build
DESELECT = "not 65536 and not 8192 and not full_64k and not qwen3_4b_8k and not 1000-2560"


def test_small_suite_under_the_checked_build():
    from long_context_sequence_seq_gb300 import build as B
    B.build(checked=True)
    env = {**os.environ, "ULYSSES_CHECKED": "1"}
    r = subprocess.run([sys.executable, "-m", "pytest", *FILES, "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider",
                        "-k", DESELECT], cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
    assert " passed" in tail and "failed" not in tail, tail
