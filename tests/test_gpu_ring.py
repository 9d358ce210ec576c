"""Ring-attention variant on P virtual ranks against the fp64 oracle.

The ring computes the same exact attention as Ulysses, block by block, with
the steps' partial outputs merged by their log-sum-exp weights; so O, the
merged LSE and the summed gradients must match plain attention over the whole
sequence (tolerances as the other bf16 / fp32 tests).
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_sequence_seq_gb300 import ulysses as U
from tests.gpu_util import LSE_TOL, TOL, f64, max_err, seq_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("S,Hq,Hkv,D,P,dtype,causal", [
    (1024, 4, 2, 128, 4, "bf16", True),
    (512, 4, 4, 128, 2, "bf16", True),
    (768, 4, 2, 128, 3, "bf16", False),
    (256, 2, 1, 64, 2, "fp32", True),
])
def test_ring_matches_plain_attention(S, Hq, Hkv, D, P, dtype, causal):
    q, k, v, do = seq_inputs(S, Hq, Hkv, D, dtype)
    o, lse = U.ring_attention_fwd(q, k, v, P, causal=causal)
    dq, dk, dv = U.ring_attention_bwd(q, k, v, o, do, lse, P, causal=causal)
    U.check()
    tr = lambda t: f64(t)[0].transpose(1, 0, 2)
    Q, K, V, DO = tr(q), tr(k), tr(v), tr(do)
    ro, rl = oracle.attn_fwd(Q, K, V, None, causal)
    rq, rk, rv = oracle.attn_bwd(Q, K, V, DO, None, causal)
    L = S // P
    lse_full = f64(lse).transpose(1, 0, 2).reshape(Hq, S)      # [P,H,L] -> [H,S]
    tol = TOL[dtype]
    assert max_err(tr(o), ro) <= tol
    assert max_err(lse_full, rl) <= LSE_TOL[dtype]
    assert max_err(tr(dq), rq) <= tol
    assert max_err(tr(dk), rk) <= tol
    assert max_err(tr(dv), rv) <= tol
