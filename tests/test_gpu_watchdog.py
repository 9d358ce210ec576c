"""Failure detection without a GPU fault: a bounded wait that runs out.

The self-test kernel waits on an mbarrier that nothing arrives on, with a
50 ms bound.  The wait gives up exactly as any wait of the attention kernels
would, records ULYSSES_ERR_TIMEOUT in the device error word and the kernel
exits; the host reads the status, the word is cleared, and the context stays
usable for the next (checked) attention call.
"""
import numpy as np
import pytest

import oracle
from long_context_sequence_seq_gb300 import ulysses as U
from tests.gpu_util import TOL, f64, max_err, seq_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    U.check()                                   # start from a clean error word
    U.selftest_wait_timeout(50_000_000)
    with pytest.raises(U.UlyssesError) as e:
        U.check()
    assert e.value.code == U.ERR_TIMEOUT
    U.check()                                   # reading cleared the word
    # the device still computes correct results afterwards
    q, k, v, _ = seq_inputs(256, 2, 1, 128, "bf16")
    o, lse = U.layer_fwd(q, k, v, 1, 2)
    U.check()
    ro, _ = oracle.attn_fwd(f64(q)[0].transpose(1, 0, 2), f64(k)[0].transpose(1, 0, 2),
                            f64(v)[0].transpose(1, 0, 2))
    assert max_err(f64(o)[0].transpose(1, 0, 2), ro) <= TOL["bf16"]
