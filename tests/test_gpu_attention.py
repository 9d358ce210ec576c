"""Attention forward/backward on the GPU against the fp64 oracle.

Tolerances (max-abs over every element): 2e-2 for bf16 inputs, 1e-4 for fp32
inputs on O, dQ, dK and dV; LSE within 1e-3 (bf16) / 1e-4 (fp32).
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_sequence_seq_gb300 import inputs, ulysses as U
from tests import oracle_pool
from tests.gpu_util import LSE_TOL, TOL, f64, max_err, seq_inputs

pytestmark = pytest.mark.gpu


def _run_stages(q, k, v, do, P, C, cu, causal):
    """Per-stage C-ABI calls: seq2head -> attn -> head2seq (fwd and bwd)."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty(v.shape, dtype=torch.float32, device=q.device)
    for st in range(P * (Hq // P // C)):
        qh = U.seq2head(q, P, C, st)
        kh = U.seq2head(k, P, C // G, st)
        vh = U.seq2head(v, P, C // G, st)
        oh, lh = U.attn_fwd(qh, kh, vh, Hq, Hkv, P, C, st, cu, causal)
        U.head2seq(oh, o, P, C, st)
        r, c = divmod(st, Hq // P // C)
        h0 = r * (Hq // P) + c * C
        lse[:, h0:h0 + C] = lh
        doh = U.seq2head(do, P, C, st)
        dqh, dkh, dvh = U.attn_bwd(qh, kh, vh, oh, doh, lh, Hq, Hkv, P, C, st, cu, causal)
        U.head2seq(dqh, dq, P, C, st)
        U.head2seq(dkh, dk, P, C // G, st)
        U.head2seq(dvh, dv, P, C // G, st)
    U.check()
    return o, lse, dq, dk, dv


SMALL = [
    # S, Hq, Hkv, D, P, C, dtype, doc lengths (None = one causal doc), causal
    (1, 2, 1, 128, 1, 2, "bf16", None, True),
    (17, 4, 2, 128, 1, 4, "bf16", None, True),
    (200, 4, 2, 128, 2, 2, "bf16", None, True),
    (256, 8, 2, 128, 2, 4, "bf16", None, True),
    (640, 4, 1, 128, 1, 4, "bf16", [300, 340], True),
    (384, 8, 2, 128, 2, 4, "bf16", [100, 200, 84], True),
    (417, 4, 4, 128, 1, 2, "bf16", [1, 129, 130, 157], True),     # ragged tail, 1-token doc
    (300, 4, 2, 128, 2, 2, "bf16", [150, 150], False),
    (260, 4, 2, 64, 2, 2, "bf16", None, True),
    (256, 8, 8, 64, 2, 4, "fp32", None, True),
    (130, 4, 2, 128, 2, 2, "fp32", [60, 70], True),
    # many key blocks of unequal work: the backward's decreasing-work block order
    (3000, 4, 2, 128, 1, 4, "bf16", [700, 5, 123, 1000, 128, 256, 300, 488], True),
    (2100, 4, 2, 128, 1, 4, "bf16", [128, 512, 640, 64, 756], False),
    # G = 8 (the forward's pairs take two of the eight q heads of a kv head)
    (2048, 8, 1, 128, 1, 8, "bf16", None, True),
    # D = 64 at a length where the tensor-core forward runs over many key tiles
    (1536, 4, 2, 64, 1, 4, "bf16", [700, 836], True),
    # bidirectional documents over many tiles, two ranks
    (4096, 4, 2, 128, 2, 2, "bf16", [1000, 3096], False),
]


@pytest.mark.parametrize("S,Hq,Hkv,D,P,C,dtype,docs,causal", SMALL)
def test_attention_small(S, Hq, Hkv, D, P, C, dtype, docs, causal):
    q, k, v, do = seq_inputs(S, Hq, Hkv, D, dtype)
    cu_np = None if docs is None else inputs.cu_seqlens_from_lengths(docs)
    cu = None if cu_np is None else torch.from_numpy(cu_np).cuda()
    o, lse, dq, dk, dv = _run_stages(q, k, v, do, P, C, cu, causal)
    Q, K, V, DO = f64(q), f64(k), f64(v), f64(do)
    ro, rl = oracle.ulysses_attention(Q, K, V, P, C, cu_np, causal)
    rq, rk, rv = oracle.ulysses_attention_bwd(Q, K, V, DO, P, C, cu_np, causal)
    tol = TOL[dtype]
    assert max_err(f64(o), ro) <= tol
    assert max_err(f64(lse), rl) <= LSE_TOL[dtype]
    assert max_err(f64(dq), rq) <= tol
    assert max_err(f64(dk), rk) <= tol
    assert max_err(f64(dv), rv) <= tol
    # the native layer driver gives bit-identical O, LSE, dK and dV.  The
    # bf16 backward sums dQ with fp32 reduce-adds from every key block in the
    # order they reach L2, so two runs may differ in the last bits of dQ.
    lo, ll = U.layer_fwd(q, k, v, P, C, cu_seqlens=cu, causal=causal)
    lq, lk, lv = U.layer_bwd(q, k, v, lo, do, ll, P, C, cu_seqlens=cu, causal=causal)
    U.check()
    for a, b in ((lo, o), (ll, lse), (lk, dk), (lv, dv)):
        assert torch.equal(a, b)
    if dtype == "fp32":
        assert torch.equal(lq, dq)
    else:
        assert float((lq - dq).abs().max()) <= 1e-5 * max(1.0, float(dq.abs().max()))


@pytest.mark.parametrize("S,Hq,Hkv,P,C,causal", [
    (300, 8, 2, 2, 4, True),     # G = 4: pair clusters in the forward, both batch entries
    (257, 8, 1, 1, 8, True),     # G = 8, ragged S
    (200, 4, 4, 2, 2, False),    # G = 1 (no cluster), bidirectional
])
def test_layer_batch_of_two(S, Hq, Hkv, P, C, causal):
    """B = 2 through the layer drivers: the stages' buffers hold both batch
    entries' heads, so kv-head mapping, LSE strides and clusters must not mix
    them."""
    D = 128
    q, k, v, do = seq_inputs(S, Hq, Hkv, D, "bf16", B=2)
    o, lse = U.layer_fwd(q, k, v, P, C, causal=causal)
    dq, dk, dv = U.layer_bwd(q, k, v, o, do, lse, P, C, causal=causal)
    U.check()
    Q, K, V, DO = f64(q), f64(k), f64(v), f64(do)
    ro, rl = oracle.ulysses_attention(Q, K, V, P, C, None, causal)
    rq, rk, rv = oracle.ulysses_attention_bwd(Q, K, V, DO, P, C, None, causal)
    assert max_err(f64(o), ro) <= TOL["bf16"]
    assert max_err(f64(lse), rl) <= LSE_TOL["bf16"]
    assert max_err(f64(dq), rq) <= TOL["bf16"]
    assert max_err(f64(dk), rk) <= TOL["bf16"]
    assert max_err(f64(dv), rv) <= TOL["bf16"]
    # the two batch entries are independent problems
    o1, l1 = U.layer_fwd(q[1:].contiguous(), k[1:].contiguous(), v[1:].contiguous(), P, C, causal=causal)
    U.check()
    assert torch.equal(o1, o[1:]) and torch.equal(l1, lse[1:])


def test_tiny_mha_fp32_workload_all_chunks():
    """S=256, 8 heads, D=64, P=2, fp32: full oracle, head_chunk in {1, 2, 4}."""
    w = inputs.WORKLOADS["tiny_mha_fp32"]
    q, k, v, do = seq_inputs(w.S, w.H_q, w.H_kv, w.D, w.dtype)
    Q, K, V, DO = f64(q), f64(k), f64(v), f64(do)
    ro, rl = oracle.ulysses_attention(Q, K, V, w.P, w.head_chunk)
    rq, rk, rv = oracle.ulysses_attention_bwd(Q, K, V, DO, w.P, w.head_chunk)
    ref = None
    for C in (1, 2, 4):
        o, lse = U.layer_fwd(q, k, v, w.P, C)
        dq, dk, dv = U.layer_bwd(q, k, v, o, do, lse, w.P, C)
        U.check()
        for got, want in ((o, ro), (dq, rq), (dk, rk), (dv, rv)):
            assert max_err(f64(got), want) <= 1e-4
        assert max_err(f64(lse), rl) <= 1e-4
        cur = [x.clone() for x in (o, lse, dq, dk, dv)]
        if ref is not None:                      # independent of the UPipe chunk
            for a, b in zip(ref, cur):
                assert torch.equal(a, b)
        ref = cur


def test_qwen3_4b_8k_all_kv_groups():
    """S=8192, H_q=32, H_kv=8, D=128, P=4, head_chunk=8 (bf16): the full
    oracle on every kv group (all 32 q heads, all 8 kv heads), all elements."""
    w = inputs.WORKLOADS["qwen3_4b_8k"]
    q, k, v, do = seq_inputs(w.S, w.H_q, w.H_kv, w.D, w.dtype)
    o, lse = U.layer_fwd(q, k, v, w.P, w.head_chunk)
    dq, dk, dv = U.layer_bwd(q, k, v, o, do, lse, w.P, w.head_chunk)
    U.check()
    G = w.G
    f32 = lambda t: t.detach().float().cpu().numpy()  # noqa: E731
    qn, kn, vn, don = f32(q[0]), f32(k[0]), f32(v[0]), f32(do[0])
    jobs = [(qn[:, h], kn[:, h // G], vn[:, h // G], don[:, h], None, True) for h in range(w.H_q)]
    res = oracle_pool.run(oracle_pool.head_fwd_bwd, jobs)
    on, ln, dqn, dkn, dvn = f64(o[0]), f64(lse[0]), f64(dq[0]), f64(dk[0]), f64(dv[0])
    for h, (ro, rl, rq, _, _) in enumerate(res):
        assert max_err(on[:, h], ro) <= TOL["bf16"], (h, "O")
        assert max_err(ln[h], rl) <= LSE_TOL["bf16"], (h, "LSE")
        assert max_err(dqn[:, h], rq) <= TOL["bf16"], (h, "dQ")
    for g in range(w.H_kv):
        rk = sum(res[h][3] for h in range(g * G, (g + 1) * G))
        rv = sum(res[h][4] for h in range(g * G, (g + 1) * G))
        assert max_err(dkn[:, g], rk) <= TOL["bf16"], (g, "dK")
        assert max_err(dvn[:, g], rv) <= TOL["bf16"], (g, "dV")


def test_bad_cu_seqlens_flagged_not_faulted():
    S, Hq, Hkv, D = 256, 4, 2, 128
    q, k, v, do = seq_inputs(S, Hq, Hkv, D, "bf16")
    for bad in ([0, 300, 256], [0, 200, 100, 256], [5, 256], [0, 128, 255]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        U.layer_fwd(q, k, v, 2, 2, cu_seqlens=cu)
        with pytest.raises(U.UlyssesError) as e:
            U.check()
        assert e.value.code == U.ERR_BAD_SEQLENS
    U.check()   # the error word was cleared
