"""The layer with the all-to-alls folded into the attention kernels'
addressing (sequence-layout TMA maps and stores, no head-layout copies).

The kernels run the same arithmetic on the same values as the unfused layer,
so O, LSE, dK and dV must be bit-identical to it; dQ is summed with fp32
reductions in L2 whose order is not fixed, so it is compared to 1e-5 relative.
Both are also checked against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_sequence_seq_gb300 import inputs, ulysses as U
from tests.gpu_util import LSE_TOL, TOL, f64, max_err, seq_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("S,Hq,Hkv,D,P,C,docs,bwd", [
    (640, 8, 2, 128, 2, 4, [300, 340], True),
    (1000, 8, 8, 128, 4, 2, None, True),          # ragged tail of 64-row tiles
    (8192, 32, 8, 128, 4, 8, None, True),         # the 8K Qwen3-4B-shaped layer
    (512, 4, 2, 64, 2, 2, None, False),           # D = 64: forward only
])
def test_fused_layer_equals_unfused(S, Hq, Hkv, D, P, C, docs, bwd):
    q, k, v, do = seq_inputs(S, Hq, Hkv, D, "bf16")
    cu_np = None if docs is None else inputs.cu_seqlens_from_lengths(docs)
    cu = None if cu_np is None else torch.from_numpy(cu_np).cuda()
    o, lse = U.layer_fwd(q, k, v, P, C, cu_seqlens=cu)
    of, lsef = U.layer_fwd_fused(q, k, v, P, C, cu_seqlens=cu)
    U.check()
    assert torch.equal(o, of) and torch.equal(lse, lsef)
    if bwd:
        dq, dk, dv = U.layer_bwd(q, k, v, o, do, lse, P, C, cu_seqlens=cu)
        dqf, dkf, dvf = U.layer_bwd_fused(q, k, v, of, do, lsef, P, C, cu_seqlens=cu)
        U.check()
        assert torch.equal(dk, dkf) and torch.equal(dv, dvf)
        assert float((dq - dqf).abs().max()) <= 1e-5 * max(1.0, float(dq.abs().max()))
    if S <= 1000:
        tr = lambda t: f64(t)[0].transpose(1, 0, 2)
        Q, K, V, DO = tr(q), tr(k), tr(v), tr(do)
        ro, rl = oracle.attn_fwd(Q, K, V, cu_np, True)
        assert max_err(tr(of), ro) <= TOL["bf16"]
        assert max_err(f64(lsef)[0], rl) <= LSE_TOL["bf16"]
        if bwd:
            rq, rk, rv = oracle.attn_bwd(Q, K, V, DO, cu_np, True)
            for got, want in ((dqf, rq), (dkf, rk), (dvf, rv)):
                assert max_err(tr(got), want) <= TOL["bf16"]
