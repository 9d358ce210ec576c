"""Which build of the library this process runs: the bounds-checked one
exactly when ULYSSES_CHECKED=1 (tests/test_gpu_checked.py runs the small GPU
suite that way)."""
import os

import pytest

from long_context_sequence_seq_gb300 import ulysses as U

pytestmark = pytest.mark.gpu


def test_loaded_variant_matches_the_request():
    want = 1 if os.environ.get("ULYSSES_CHECKED") == "1" else 0
    assert U.lib().ulysses_checked_build() == want
