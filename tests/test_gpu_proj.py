"""Projections with the re-layout fused into the GEMM, against numpy matmuls
in fp64 on the same bf16 values.

Bound: the result is rounded to bf16 once (relative 2^-8) after an fp32
accumulation, so |got - ref| <= 2^-8 |ref| + 1e-3 elementwise (the absolute
term covers fp32 accumulation over a few thousand products).
"""
import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("S,hidden,Hq,Hkv,D", [(300, 256, 4, 2, 128), (129, 512, 2, 1, 64), (1000, 2560, 32, 8, 128)])
def test_qkv_proj_into_head_layout(S, hidden, Hq, Hkv, D):
    nf = (Hq + 2 * Hkv) * D
    x = _bf16((S, hidden), 31)
    w = _bf16((nf, hidden), 32, 1.0 / np.sqrt(hidden))
    out = U.qkv_proj(x.cuda(), w.cuda(), Hq, Hkv)
    U.check()
    rows = np.arange(S) if S <= 300 else np.unique(np.r_[0:64, S - 64:S, np.linspace(0, S - 1, 64).astype(int)])
    ref = _np(x)[rows] @ _np(w).T                                  # [rows, nf]
    got = _np(out)[:, rows, :].transpose(1, 0, 2).reshape(len(rows), nf)   # head layout -> [rows, nf]
    _within(got, ref)


@pytest.mark.parametrize("S,Hq,D,hidden", [(300, 4, 128, 256), (77, 2, 64, 512), (1000, 32, 128, 2560)])
def test_out_proj_from_head_layout(S, Hq, D, hidden):
    o = _bf16((Hq, S, D), 41)
    w = _bf16((hidden, Hq * D), 42, 1.0 / np.sqrt(Hq * D))
    y = U.out_proj(o.cuda(), w.cuda())
    U.check()
    o_seq = _np(o).transpose(1, 0, 2).reshape(S, Hq * D)         # O_seq[s][h D + d]
    _within(_np(y), o_seq @ _np(w).T)
