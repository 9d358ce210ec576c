"""Attention parity on inputs that stress the online softmax.

N(0,1) inputs give every row its largest score early, so the forward's
running-max update (which moves the max only once a row's max has grown by
more than 2^8, and otherwise keeps the stale max as the stabiliser) is rarely
taken after the first key tile.  These cases make the row maxima grow along
the sequence (keys aligned with the queries and scaled up with their
position), and spread the scores over a wide range, then compare forward and
backward with the fp64 oracle.

Tolerance: max-abs 2e-2 (the bound of the N(0,1) workloads) plus, element by
element, the worst-case error the bf16 operands of the second-stage MMAs can
add (tests.gpu_util.bf16_rounding_bound: the bf16 unit roundoff 2^-8 on P and
dS, and on the stored O that D_i is formed from).  The "wide" scores give gradients of
magnitude 10-15, where that rounding alone exceeds 2e-2; a wrong lazy
rescale errs by the magnitude of the result, far outside it.  LSE within
1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_sequence_seq_gb300 import inputs, ulysses as U
from tests.gpu_util import bf16_rounding_bound, f64

pytestmark = pytest.mark.gpu


def _head_inputs(S, Hq, Hkv, D, mode, seed=0):
    rng = np.random.Generator(np.random.PCG64(1234 + seed))
    q = rng.standard_normal((1, Hq, S, D))
    k = rng.standard_normal((1, Hkv, S, D))
    v = rng.standard_normal((1, Hkv, S, D))
    do = rng.standard_normal((1, Hq, S, D))
    if mode == "growing":
        # s_ij ~ (|q| |k_j| / sqrt(D)) grows with j: the row max of row i keeps
        # rising tile after tile, by ~6 natural-log units every 1/8 of S
        u = np.ones(D) / np.sqrt(D)
        t = 40.0 * np.arange(S) / S
        q = 0.25 * q + 4.0 * u
        k = 0.25 * k + (t[:, None] * u[None, :])[None, None] * np.sqrt(D) / 4.0
    elif mode == "wide":
        q, k = 3.0 * q, 3.0 * k      # scores with a standard deviation of ~9
    to = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    return to(q), to(k), to(v), to(do)


def _check(name, got, ref, bound):
    err = np.abs(got - ref)
    excess = err - (2e-2 + bound)
    assert np.all(excess <= 0), (name, float(err.max()), float(excess.max()))


@pytest.mark.parametrize("mode,S,docs", [
    ("growing", 1024, None),
    ("growing", 2000, [700, 1300]),
    ("wide", 1024, None),
    ("wide", 640, [1, 300, 339]),
])
def test_online_softmax_stress(mode, S, docs):
    Hq, Hkv, D = 2, 1, 128
    q, k, v, do = _head_inputs(S, Hq, Hkv, D, mode)
    cu_np = None if docs is None else inputs.cu_seqlens_from_lengths(docs)
    cu = None if cu_np is None else torch.from_numpy(cu_np).cuda()
    o, lse = U.attn_fwd(q, k, v, Hq, Hkv, 1, None, None, cu, True)
    dq, dk, dv = U.attn_bwd(q, k, v, o, do, lse, Hq, Hkv, 1, None, None, cu, True)
    U.check()
    Q, K, V, DO = f64(q)[0], f64(k)[0], f64(v)[0], f64(do)[0]
    ro, rl = oracle.attn_fwd(Q, K, V, cu_np, True)
    rq, rk, rv = oracle.attn_bwd(Q, K, V, DO, cu_np, True)
    b_o, b_q, b_k, b_v = bf16_rounding_bound(Q, K, V, DO, cu_np, True)
    _check("O", f64(o)[0], ro, b_o)
    assert float(np.max(np.abs(f64(lse)[0] - rl))) <= 1e-3
    for name, got, ref, bnd in (("dQ", dq, rq, b_q), ("dK", dk, rk, b_k), ("dV", dv, rv, b_v)):
        _check(name, f64(got)[0], ref, bnd)
    if mode == "growing":
        # the construction does what it says: row maxima rise by far more than
        # 8 log2 units over the sequence
        assert float(rl[:, -1].max() - rl[:, S // 8].max()) > 8.0
