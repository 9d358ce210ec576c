"""Full-size parity on the benchmark's own launch configuration.

The layer is run exactly as bench.py times it (per-stage C-ABI calls,
tcgen05 kernels), then checked against the fp64 oracle.  Local attention is
exact softmax attention ("How Ulysses sequence parallelism works", step 4), so
the oracle is the plain definition, run on whole heads where the host can
afford it and on row- or column-local pieces where it cannot:

* 64K layer: the full oracle (every row and every key column) on kv group 0
  (rank 0) and kv group 7 (rank 3): 4 q heads and their kv head each;
* packed 128K layer: the full oracle on the three shortest documents, the
  longest one and the one that crosses the rank 3/4 boundary, all heads of
  kv group 0 (and the shortest ones for the last group too), plus sampled rows
  at every document and rank boundary;
* 1M-token layer: 256 rows of each of two q heads (rank boundaries, tile
  boundaries, the first and last rows and seeded random rows): O, LSE and dQ
  via the oracle's row-local pieces; dK/dV of the last 2048 key columns of one
  kv head (only rows after them see them under the causal mask);
* exact invariants over every kv head and document, at every size:
  sum_j dK_j = 0 (rows of dS sum to D_i - D_i = 0) and
  sum_j dV_j = sum over the group's rows of dO (rows of P sum to 1).
  What the oracle does not reach at 1M is held by these invariants only.
Tolerances: max-abs 2e-2 (bf16 inputs) on O/dQ/dK/dV, 1e-3 on LSE.
"""
import numpy as np
import pytest
import torch

from bench import LayerStep
from long_context_sequence_seq_gb300 import inputs
from tests import oracle_pool
from tests.gpu_util import LSE_TOL, TOL

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy()


def _sample_rows(S, P, n_rows, seed=7):
    """n_rows rows: rank boundaries, tile boundaries, first/last rows, then
    seeded random rows up to the count."""
    Sp = S // P
    cand = {0, 1, 63, 64, 127, 128, 129, S - 2, S - 1}
    for r in range(1, P):
        cand.update({r * Sp - 1, r * Sp, r * Sp + 1})
    rng = np.random.Generator(np.random.PCG64(seed))
    cand = {c for c in cand if 0 <= c < S}
    while len(cand) < min(n_rows, S):
        cand.add(int(rng.integers(0, S)))
    return np.array(sorted(cand), dtype=np.int64)


def _run(w):
    dev = torch.device("cuda")
    cu = inputs.workload_cu_seqlens(w)
    step = LayerStep(w, dev, cu)
    step.run()
    torch.cuda.synchronize()
    step.U.check()
    return step, cu


def _check_groups_full(step, w, groups, a=0, b=None, cu=None):
    """Full oracle on tokens [a, b) (one document, or the whole causal
    sequence) for every q head of the given kv groups, in parallel over heads."""
    G = w.G
    b = w.S if b is None else b
    jobs, where = [], []
    for g in groups:
        K = _np(step.k[0, a:b, g])
        V = _np(step.v[0, a:b, g])
        for h in range(g * G, (g + 1) * G):
            jobs.append((_np(step.q[0, a:b, h]), K, V, _np(step.do[0, a:b, h]), cu, True))
            where.append((g, h))
    res = oracle_pool.run(oracle_pool.head_fwd_bwd, jobs)
    dk_ref = {g: 0.0 for g in groups}
    dv_ref = {g: 0.0 for g in groups}
    for (g, h), (ro, rl, rq, rk, rv) in zip(where, res):
        assert np.max(np.abs(_np(step.o[0, a:b, h]) - ro)) <= TOL["bf16"], (h, a, "O")
        assert np.max(np.abs(_np(step.lse[0, h, a:b]) - rl)) <= LSE_TOL["bf16"], (h, a, "LSE")
        assert np.max(np.abs(_np(step.dq[0, a:b, h]) - rq)) <= TOL["bf16"], (h, a, "dQ")
        dk_ref[g] = dk_ref[g] + rk
        dv_ref[g] = dv_ref[g] + rv
    for g in groups:
        assert np.max(np.abs(_np(step.dk[0, a:b, g]) - dk_ref[g])) <= TOL["bf16"], (g, a, "dK")
        assert np.max(np.abs(_np(step.dv[0, a:b, g]) - dv_ref[g])) <= TOL["bf16"], (g, a, "dV")


def _check_rows(step, w, cu, heads, rows):
    G = w.G
    jobs = []
    for h in heads:
        g = h // G
        jobs.append((_np(step.q[0, rows, h]), _np(step.k[0, :, g]), _np(step.v[0, :, g]),
                     _np(step.do[0, rows, h]), rows, cu, True))
    for h, (ro, rl, rdq) in zip(heads, oracle_pool.run(oracle_pool.head_rows, jobs)):
        assert np.max(np.abs(_np(step.o[0, rows, h]) - ro)) <= TOL["bf16"], (h, "O")
        assert np.max(np.abs(_np(step.lse[0, h, rows]) - rl)) <= LSE_TOL["bf16"], (h, "LSE")
        assert np.max(np.abs(_np(step.dq[0, rows, h]) - rdq)) <= TOL["bf16"], (h, "dQ")


def _check_kv_tail(step, w, cu, kv_heads, tail, row_block=32):
    S, G = w.S, w.G
    j0 = S - tail
    for g in kv_heads:
        K = _np(step.k[0, :, g])
        V = _np(step.v[0, :, g])
        jobs = [(_np(step.q[0, j0:, h]), K, V, _np(step.do[0, j0:, h]), j0, cu, True, row_block)
                for h in range(g * G, (g + 1) * G)]
        parts = oracle_pool.run(oracle_pool.head_kv_tail, jobs, max_workers=4)
        rk = sum(p[0] for p in parts)
        rv = sum(p[1] for p in parts)
        assert np.max(np.abs(_np(step.dk[0, j0:, g]) - rk)) <= TOL["bf16"], (g, "dK tail")
        assert np.max(np.abs(_np(step.dv[0, j0:, g]) - rv)) <= TOL["bf16"], (g, "dV tail")


def _check_invariants(step, w, cu):
    G = w.G
    bounds = [(0, w.S)] if cu is None else list(zip(cu[:-1].tolist(), cu[1:].tolist()))
    for a, b in bounds:
        dk = step.dk[0, a:b].double()           # [L, H_kv, D]
        dv = step.dv[0, a:b].double()
        do = step.do[0, a:b].double().view(b - a, w.H_kv, G, w.D).sum(2)   # sum over the group
        sk = dk.sum(0)
        assert (sk.abs() <= 2e-3 * dk.abs().sum(0) + 1e-3).all(), ("sum dK", a, b)
        sv = dv.sum(0)
        ref = do.sum(0)
        assert ((sv - ref).abs() <= 2e-3 * do.abs().sum(0) + 1e-3).all(), ("sum dV", a, b)


def test_qwen3_4b_64k_layer():
    w = inputs.WORKLOADS["qwen3_4b_64k"]
    step, cu = _run(w)
    _check_groups_full(step, w, groups=(0, w.H_kv - 1))     # kv head 0 (rank 0), kv head 7 (rank 3)
    _check_invariants(step, w, cu)


def test_llama31_8b_packed_layer():
    w = inputs.WORKLOADS["llama31_8b_packed"]
    step, cu = _run(w)
    lengths = np.diff(cu)
    Sp = w.S // w.P
    cross = int(np.searchsorted(cu, 4 * Sp, side="right") - 1)      # the document holding token 4 S/P
    assert cu[cross] < 4 * Sp < cu[cross + 1]                       # it does cross the rank 3/4 boundary
    shortest = [int(d) for d in np.argsort(lengths, kind="stable")[:3]]
    docs = sorted(set(shortest + [int(np.argmax(lengths)), cross]))
    for d in docs:
        a, b = int(cu[d]), int(cu[d + 1])
        groups = (0, w.H_kv - 1) if d in shortest else (0,)
        _check_groups_full(step, w, groups, a, b)
    # sampled rows everywhere (every document and rank boundary) and the key tail
    rows = _sample_rows(w.S, w.P, 64)
    rows = np.unique(np.concatenate([rows, cu[1:-1].astype(np.int64), cu[1:-1].astype(np.int64) - 1]))
    _check_rows(step, w, cu, heads=(0, w.H_q - 1), rows=rows)
    _check_kv_tail(step, w, cu, kv_heads=(0,), tail=256)
    _check_invariants(step, w, cu)


@pytest.mark.slow
def test_million_token_layer():
    w = inputs.WORKLOADS["million_token"]
    step, cu = _run(w)
    rows = _sample_rows(w.S, w.P, 256)
    assert len(rows) == 256
    _check_rows(step, w, cu, heads=(0, w.H_q - 1), rows=rows)
    _check_kv_tail(step, w, cu, kv_heads=(w.H_kv - 1,), tail=2048)
    _check_invariants(step, w, cu)
