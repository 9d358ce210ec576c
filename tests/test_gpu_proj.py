"""Projections with the re-layout fused into the GEMM (steps 2 and 6 around
the all-to-alls), against the oracle's qkv_proj / out_proj in fp64 on the
same bf16 values.  The oracle projects each rank's token chunk and moves the
heads with its own seq2head / head2seq; the GPU writes (reads) head layout
straight from the GEMM epilogue (operand load).

Bound: the result is rounded to bf16 once (relative 2^-8) after an fp32
accumulation, so |got - ref| <= 2^-8 |ref| + 1e-3 elementwise (the absolute
term covers fp32 accumulation over a few thousand products).
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_sequence_seq_gb300 import inputs, ulysses as U

pytestmark = pytest.mark.gpu


def _bf16(shape, seed, scale=1.0):
    t = inputs.host_tensor(shape, seed, "bf16").float() * scale
    return t.to(torch.bfloat16)


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _within(got, ref):
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3
    assert np.all(err <= bound), float(np.max(err - bound))


@pytest.mark.parametrize("S,hidden,Hq,Hkv,D,P", [(300, 256, 4, 2, 128, 2), (129, 512, 2, 1, 64, 1),
                                                  (1000, 2560, 32, 8, 128, 4)])
def test_qkv_proj_into_head_layout(S, hidden, Hq, Hkv, D, P):
    nf = (Hq + 2 * Hkv) * D
    x = _bf16((S, hidden), 31)
    w = _bf16((nf, hidden), 32, 1.0 / np.sqrt(hidden))
    out = U.qkv_proj(x.cuda(), w.cuda(), Hq, Hkv)
    U.check()
    ref = oracle.qkv_proj(_np(x), _np(w), Hq, Hkv, P)            # [Hq + 2 Hkv, S, D]
    _within(_np(out), ref)


@pytest.mark.parametrize("S,Hq,D,hidden,P", [(300, 4, 128, 256, 2), (77, 2, 64, 512, 1), (1000, 32, 128, 2560, 4)])
def test_out_proj_from_head_layout(S, Hq, D, hidden, P):
    o = _bf16((Hq, S, D), 41)
    w = _bf16((hidden, Hq * D), 42, 1.0 / np.sqrt(Hq * D))
    y = U.out_proj(o.cuda(), w.cuda())
    U.check()
    _within(_np(y), oracle.out_proj(_np(o), _np(w), P))
