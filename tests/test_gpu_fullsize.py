"""Full-size parity on the benchmark's own launch configuration.

The layer is run exactly as bench.py times it (per-stage C-ABI calls,
tcgen05 kernels), then checked against the fp64 oracle on outputs it can
compute one by one, and against properties that hold at any size:

* sampled rows (rank boundaries, tile boundaries, first/last rows and seeded
  random rows) of two q heads from different ranks: O, LSE and dQ via the
  oracle's row-local pieces (each row needs only its own keys);
* dK/dV of the last key columns of two kv heads (only rows after them see
  them under the causal mask);
* for packed documents: the full oracle on the three shortest documents;
* exact invariants over every kv head and document:
  sum_j dK_j = 0 (rows of dS sum to D_i - D_i = 0) and
  sum_j dV_j = sum over the group's rows of dO (rows of P sum to 1).
Tolerances: max-abs 2e-2 (bf16 inputs) on O/dQ/dK/dV, 1e-3 on LSE.
"""
import numpy as np
import pytest
import torch

import oracle
from bench import LayerStep
from long_context_sequence_seq_gb300 import inputs
from tests.gpu_util import LSE_TOL, TOL

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy()


def _sample_rows(S, P, n_random=40, seed=7):
    Sp = S // P
    cand = {0, 1, 63, 64, 127, 128, 129, S - 2, S - 1}
    for r in range(1, P):
        cand.update({r * Sp - 1, r * Sp, r * Sp + 1})
    rng = np.random.Generator(np.random.PCG64(seed))
    cand.update(int(x) for x in rng.integers(0, S, n_random))
    return np.array(sorted(c for c in cand if 0 <= c < S), dtype=np.int64)


def _run(w):
    dev = torch.device("cuda")
    cu = inputs.workload_cu_seqlens(w)
    step = LayerStep(w, dev, cu)
    step.run()
    torch.cuda.synchronize()
    step.U.check()
    return step, cu


def _check_rows(step, w, cu, heads, rows):
    G = w.G
    for h in heads:
        g = h // G
        K = _np(step.k[0, :, g])
        V = _np(step.v[0, :, g])
        q_rows = _np(step.q[0, rows, h])
        do_rows = _np(step.do[0, rows, h])
        ro, rl, rdq = oracle.attn_rows(q_rows, K, V, do_rows, rows, cu, True)
        got_o = _np(step.o[0, rows, h]).astype(np.float64)
        got_l = _np(step.lse[0, h, rows]).astype(np.float64)
        got_dq = _np(step.dq[0, rows, h]).astype(np.float64)
        assert np.max(np.abs(got_o - ro)) <= TOL["bf16"], (h, "O")
        assert np.max(np.abs(got_l - rl)) <= LSE_TOL["bf16"], (h, "LSE")
        assert np.max(np.abs(got_dq - rdq)) <= TOL["bf16"], (h, "dQ")


def _check_kv_tail(step, w, cu, kv_heads, tail):
    S, G, D = w.S, w.G, w.D
    j0 = S - tail
    for g in kv_heads:
        qh = np.zeros((G, S, D), dtype=np.float32)   # only rows >= j0 are read (calloc pages)
        dh = np.zeros((G, S, D), dtype=np.float32)
        qh[:, j0:] = _np(step.q[0, j0:, g * G:(g + 1) * G]).transpose(1, 0, 2)
        dh[:, j0:] = _np(step.do[0, j0:, g * G:(g + 1) * G]).transpose(1, 0, 2)
        K = _np(step.k[0, :, g])
        V = _np(step.v[0, :, g])
        rk, rv = oracle.attn_kv_tail(qh, K, V, dh, j0, cu, True, row_block=32)
        got_k = _np(step.dk[0, j0:, g]).astype(np.float64)
        got_v = _np(step.dv[0, j0:, g]).astype(np.float64)
        assert np.max(np.abs(got_k - rk)) <= TOL["bf16"], (g, "dK tail")
        assert np.max(np.abs(got_v - rv)) <= TOL["bf16"], (g, "dV tail")


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
    rows = _sample_rows(w.S, w.P)
    _check_rows(step, w, cu, heads=(0, w.H_q - 1), rows=rows)
    _check_kv_tail(step, w, cu, kv_heads=(0, w.H_kv - 1), tail=256)
    _check_invariants(step, w, cu)


def test_llama31_8b_packed_layer():
    w = inputs.WORKLOADS["llama31_8b_packed"]
    step, cu = _run(w)
    lengths = np.diff(cu)
    # full oracle on the three shortest documents, every head of kv group 0 and of the last group
    for d in np.argsort(lengths, kind="stable")[:3]:
        a, b = int(cu[d]), int(cu[d + 1])
        for g in (0, w.H_kv - 1):
            hs = slice(g * w.G, (g + 1) * w.G)
            Q = _np(step.q[0, a:b, hs]).transpose(1, 0, 2)
            DO = _np(step.do[0, a:b, hs]).transpose(1, 0, 2)
            K = _np(step.k[0, a:b, g:g + 1]).transpose(1, 0, 2)
            V = _np(step.v[0, a:b, g:g + 1]).transpose(1, 0, 2)
            ro, rl = oracle.attn_fwd(Q, K, V)
            rq, rk, rv = oracle.attn_bwd(Q, K, V, DO)
            assert np.max(np.abs(_np(step.o[0, a:b, hs]).transpose(1, 0, 2) - ro)) <= TOL["bf16"]
            assert np.max(np.abs(_np(step.lse[0, hs, a:b]) - rl)) <= LSE_TOL["bf16"]
            assert np.max(np.abs(_np(step.dq[0, a:b, hs]).transpose(1, 0, 2) - rq)) <= TOL["bf16"]
            assert np.max(np.abs(_np(step.dk[0, a:b, g:g + 1]).transpose(1, 0, 2) - rk)) <= TOL["bf16"]
            assert np.max(np.abs(_np(step.dv[0, a:b, g:g + 1]).transpose(1, 0, 2) - rv)) <= TOL["bf16"]
    # sampled rows everywhere (documents crossing rank boundaries included) and the key tail
    rows = _sample_rows(w.S, w.P)
    rows = np.unique(np.concatenate([rows, cu[1:-1].astype(np.int64), cu[1:-1].astype(np.int64) - 1]))
    _check_rows(step, w, cu, heads=(0, w.H_q - 1), rows=rows)
    _check_kv_tail(step, w, cu, kv_heads=(0,), tail=256)
    _check_invariants(step, w, cu)


@pytest.mark.slow
def test_million_token_layer():
    w = inputs.WORKLOADS["million_token"]
    step, cu = _run(w)
    rows = _sample_rows(w.S, w.P, n_random=24)
    _check_rows(step, w, cu, heads=(0, w.H_q - 1), rows=rows)
    _check_kv_tail(step, w, cu, kv_heads=(w.H_kv - 1,), tail=128)
    _check_invariants(step, w, cu)
