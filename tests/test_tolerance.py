"""Host check of the derived bf16 rounding bound used by the online-softmax
stress tests: a CPU emulation of the bf16 operand rounding (P and dS rounded
to bf16 before the second-stage products, O stored as bf16 before D_i is
formed) must stay inside tests.gpu_util.bf16_rounding_bound element by
element, and must exceed the plain 2e-2 somewhere on the wide-score inputs
(otherwise the extra term would not be needed)."""
import math

import numpy as np
import torch

import oracle
from tests.gpu_util import bf16_rounding_bound


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def _emulated(q, k, v, do, causal=True):
    Hq, S, D = q.shape
    G = Hq // k.shape[0]
    sc = 1.0 / math.sqrt(D)
    lo, hi = oracle.key_ranges(S, None, causal)
    j = np.arange(S)
    allowed = (j[None, :] >= lo[:, None]) & (j[None, :] < hi[:, None])
    O, dQ = np.zeros(q.shape), np.zeros(q.shape)
    dK, dV = np.zeros(k.shape), np.zeros(k.shape)
    for h in range(Hq):
        g = h // G
        s = np.where(allowed, sc * (q[h] @ k[g].T), -np.inf)
        e = np.exp(s - s.max(axis=1)[:, None])
        p = e / e.sum(axis=1)[:, None]
        pb = _bf16(p)
        o = _bf16(pb @ v[g])                       # bf16 P into PV, O stored as bf16
        O[h] = o
        dp = do[h] @ v[g].T
        dsb = _bf16(p * (dp - np.sum(do[h] * o, axis=1)[:, None]))   # D_i from the stored O
        dV[g] += pb.T @ do[h]
        dQ[h] = sc * (dsb @ k[g])
        dK[g] += sc * (dsb.T @ q[h])
    return O, dQ, dK, dV


def test_emulated_bf16_operands_stay_inside_the_bound():
    rng = np.random.Generator(np.random.PCG64(5))
    S, D = 256, 64
    q = _bf16(3.0 * rng.standard_normal((2, S, D)))
    k = _bf16(3.0 * rng.standard_normal((1, S, D)))
    v = _bf16(rng.standard_normal((1, S, D)))
    do = _bf16(rng.standard_normal((2, S, D)))
    ro, _ = oracle.attn_fwd(q, k, v)
    rq, rk, rv = oracle.attn_bwd(q, k, v, do)
    got = _emulated(q, k, v, do)
    bounds = bf16_rounding_bound(q, k, v, do)
    worst = 0.0
    for g, r, b in zip(got, (ro, rq, rk, rv), bounds):
        err = np.abs(g - r)
        assert np.all(err <= b + 1e-9), float(np.max(err - b))
        worst = max(worst, float(err.max()))
    assert worst > 2e-2          # the wide scores do need the extra term
