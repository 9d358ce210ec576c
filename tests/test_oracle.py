"""Pins for the fp64 oracle against facts fixed by the pages and by mathematics.

Nothing here compares the oracle with itself: each test checks it against a
hand-derived worked example, a closed form, a library routine (torch SDPA and
autograd in fp64), finite differences, brute force on tiny inputs, or an exact
invariant.  ``test_mutants_are_caught`` plants plausible mistakes in copies of
the oracle and checks that these pins catch them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _val(expr):
    ns = {"ln2": math.log(2.0), "ln3": math.log(3.0), "ln6": math.log(6.0)}
    return float(eval(str(expr), {"__builtins__": {}}, ns))


def _rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


# ---------------------------------------------------------------- golden cases

def test_golden_worked_example():
    g = json.load(open(os.path.join(GOLD, "worked_3tok.json")))
    q = np.array(g["q"]).reshape(1, 3, 1)
    k = np.array([_val(x) for x in g["k"]]).reshape(1, 3, 1)
    v = np.array(g["v"]).reshape(1, 3, 1)
    do = np.array(g["do"]).reshape(1, 3, 1)
    for case in g["cases"]:
        cu = case["cu_seqlens"]
        o, lse = O.attn_fwd(q, k, v, cu, case["causal"], g["scale"])
        dq, dk, dv = O.attn_bwd(q, k, v, do, cu, case["causal"], g["scale"])
        for name, got in (("O", o), ("LSE", lse), ("dQ", dq), ("dK", dk), ("dV", dv)):
            want = np.array([_val(x) for x in case[name]])
            np.testing.assert_allclose(got.reshape(-1), want, rtol=0, atol=1e-13,
                                       err_msg=f"{case['name']} {name}")


def test_golden_relayout():
    g = json.load(open(os.path.join(GOLD, "relayout_4tok.json")))
    S, H, D, P = g["S"], g["H"], g["D"], g["P"]
    x = np.array([[[10 * t + h] for h in range(H)] for t in range(S)], dtype=np.int64)[None]
    np.testing.assert_array_equal(O.seq2head(x, P)[0, :, :, 0], np.array(g["x_head_all"]))
    for st, want in g["stages_head_chunk_1"].items():
        np.testing.assert_array_equal(O.seq2head(x, P, 1, int(st))[0, :, :, 0], np.array(want))
    # each rank's heads are the contiguous subset listed by the example
    for r, heads in enumerate(g["rank_heads"]):
        np.testing.assert_array_equal(O.stage_heads(H, P, None, (r, 0)), heads)


# ---------------------------------------------------------------- re-layout

@pytest.mark.parametrize("S,H,D,P,C", [(8, 4, 3, 2, 1), (12, 6, 2, 3, 2), (16, 8, 4, 4, 2),
                                       (6, 4, 5, 1, 4), (10, 10, 1, 5, 1)])
def test_relayout_bruteforce_bit_equal(S, H, D, P, C):
    x = np.arange(2 * S * H * D, dtype=np.int64).reshape(2, S, H, D) * 7919 % 1000003
    hq = H // P
    for st in [None] + list(range(P * (hq // C))):
        a = O.seq2head(x, P, C, st)
        b = O.seq2head_bruteforce(x, P, C, st)
        np.testing.assert_array_equal(a, b)
        y1 = np.full_like(x, -1)
        y2 = np.full_like(x, -1)
        O.head2seq(a, y1, P, C, st)
        O.head2seq_bruteforce(a, y2, P, C, st)
        np.testing.assert_array_equal(y1, y2)


def test_relayout_round_trips():
    x = _rand((1, 24, 8, 4), 5)
    for P in (1, 2, 4, 8):
        hq = 8 // P
        for C in [c for c in range(1, hq + 1) if hq % c == 0]:
            y = np.zeros_like(x)
            for st in range(P * (hq // C)):
                O.head2seq(O.seq2head(x, P, C, st), y, P, C, st)
            np.testing.assert_array_equal(y, x)          # head2seq o seq2head = id
        h = O.seq2head(x, P)
        y = np.zeros_like(x)
        O.head2seq(h, y, P)
        np.testing.assert_array_equal(O.seq2head(y, P), h)  # seq2head o head2seq = id


def test_relayout_P1_is_a_transpose_only():
    x = _rand((1, 5, 3, 2), 6)
    np.testing.assert_array_equal(O.seq2head(x, 1), np.transpose(x, (0, 2, 1, 3)))


def test_relayout_volume_per_rank():
    """Each rank sends its S/P tokens x H x D once per all-to-all: O(n d / P)."""
    S, H, D, P = 32, 8, 4, 4
    x = _rand((1, S, H, D), 7)
    for r in range(P):
        hq = H // P
        got = sum(O.seq2head(x, P, 1, (r, c)).size for c in range(hq))
        # what rank r receives equals what every rank sends (square all-to-all)
        assert got * 2 == O.relayout_bytes_per_rank(S, H, D, P, 2)
    with pytest.raises(ValueError):
        O.seq2head(_rand((1, 30, 8, 4), 1), 4)       # S % P != 0
    with pytest.raises(ValueError):
        O.seq2head(_rand((1, 32, 6, 4), 1), 4)       # H % P != 0


# ---------------------------------------------------------------- forward

SMALL_CASES = [
    dict(Hq=2, Hkv=2, S=9, D=3, cu=None, causal=True),
    dict(Hq=4, Hkv=2, S=13, D=4, cu=None, causal=True),
    dict(Hq=4, Hkv=1, S=17, D=2, cu=[0, 5, 6, 17], causal=True),
    dict(Hq=2, Hkv=1, S=11, D=5, cu=[0, 3, 11], causal=False),
    dict(Hq=3, Hkv=3, S=7, D=3, cu=[0, 1, 2, 7], causal=True),
]


@pytest.mark.parametrize("c", SMALL_CASES)
def test_fwd_bwd_match_bruteforce(c):
    q = _rand((c["Hq"], c["S"], c["D"]), 1)
    k = _rand((c["Hkv"], c["S"], c["D"]), 2)
    v = _rand((c["Hkv"], c["S"], c["D"]), 3)
    do = _rand((c["Hq"], c["S"], c["D"]), 4)
    o, lse = O.attn_fwd(q, k, v, c["cu"], c["causal"], row_block=4)
    o2, lse2 = O.attn_fwd_bruteforce(q, k, v, c["cu"], c["causal"])
    np.testing.assert_allclose(o, o2, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, atol=1e-12)
    g1 = O.attn_bwd(q, k, v, do, c["cu"], c["causal"], row_block=4)
    g2 = O.attn_bwd_bruteforce(q, k, v, do, c["cu"], c["causal"])
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, atol=1e-12)


def _sdpa_ref(q, k, v, causal, scale=None):
    """torch's fp64 scaled_dot_product_attention (a library routine) with
    K/V repeated G times for GQA."""
    G = q.shape[0] // k.shape[0]
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    kk = tk.repeat_interleave(G, dim=0)
    vv = tv.repeat_interleave(G, dim=0)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None], kk[None], vv[None], is_causal=causal, scale=scale)[0]
    return tq, tk, tv, out


@pytest.mark.parametrize("causal", [True, False])
def test_matches_torch_sdpa_fp64(causal):
    Hq, Hkv, S, D = 8, 2, 70, 16
    q, k, v, do = (_rand((Hq, S, D), 11), _rand((Hkv, S, D), 12), _rand((Hkv, S, D), 13),
                   _rand((Hq, S, D), 14))
    tq, tk, tv, out = _sdpa_ref(q, k, v, causal)
    o, _ = O.attn_fwd(q, k, v, None, causal, row_block=16)
    np.testing.assert_allclose(o, out.detach().numpy(), atol=1e-12)
    out.backward(torch.tensor(do))
    dq, dk, dv = O.attn_bwd(q, k, v, do, None, causal, row_block=16)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


def test_lse_matches_library_logsumexp():
    from scipy.special import logsumexp
    Hq, S, D = 2, 40, 8
    q, k, v = _rand((Hq, S, D), 1), _rand((1, S, D), 2), _rand((1, S, D), 3)
    _, lse = O.attn_fwd(q, k, v)
    for h in range(Hq):
        for i in range(S):
            s = (q[h, i] @ k[0, :i + 1].T) / math.sqrt(D)
            assert abs(lse[h, i] - logsumexp(s)) < 1e-12


def test_softmax_rows_sum_to_one():
    # V rows = unit vectors e_j, so O_i is exactly the softmax row i
    Hq, S = 2, 24
    q, k = _rand((Hq, S, 8), 1), _rand((1, S, 8), 2)
    v = np.eye(S)[None]
    for cu, causal in ((None, True), ([0, 10, 24], True), ([0, 7, 24], False)):
        o, _ = O.attn_fwd(q, k, v, cu, causal, scale=0.35)
        np.testing.assert_allclose(o.sum(axis=2), 1.0, atol=1e-12)
        assert np.all(o >= 0)


def test_constant_v_rows():
    Hq, Hkv, S, D = 4, 2, 30, 6
    q, k, do = _rand((Hq, S, D), 1), _rand((Hkv, S, D), 2), _rand((Hq, S, D), 3)
    c = _rand((Hkv, 1, D), 4)
    v = np.repeat(c, S, axis=1)
    o, _ = O.attn_fwd(q, k, v, [0, 11, 30])
    np.testing.assert_allclose(o, np.repeat(c, 2, axis=0).repeat(S, axis=1), atol=1e-12)
    dq, dk, _ = O.attn_bwd(q, k, v, do, [0, 11, 30])
    assert np.max(np.abs(dq)) < 1e-12 and np.max(np.abs(dk)) < 1e-12


def test_first_row_of_each_doc_and_singletons():
    Hq, S, D = 2, 20, 4
    q, k, v = _rand((Hq, S, D), 1), _rand((1, S, D), 2), _rand((1, S, D), 3)
    cu = [0, 1, 2, 9, 10, 20]   # docs of length 1 at tokens 0, 1 and 9
    o, lse = O.attn_fwd(q, k, v, cu)
    for start in cu[:-1]:
        np.testing.assert_allclose(o[:, start], np.repeat(v[:, start], Hq, axis=0), atol=1e-14)
        np.testing.assert_allclose(lse[:, start], q[:, start] @ k[0, start] / math.sqrt(D),
                                   atol=1e-14)


def test_zero_queries_closed_form():
    """q = 0 makes every score 0: O_i is the mean of the allowed v_j and LSE_i
    = log(number of allowed keys)."""
    Hq, S, D = 2, 33, 3
    v = _rand((1, S, D), 5)
    k = _rand((1, S, D), 6)
    q = np.zeros((Hq, S, D))
    cu = [0, 12, 33]
    o, lse = O.attn_fwd(q, k, v, cu)
    for i in range(S):
        a = 0 if i < 12 else 12
        np.testing.assert_allclose(o[:, i], np.mean(v[0, a:i + 1], axis=0)[None].repeat(Hq, 0),
                                   atol=1e-13)
        np.testing.assert_allclose(lse[:, i], math.log(i + 1 - a), atol=1e-13)


def test_causality_bit_identical():
    Hq, S, D = 2, 40, 4
    q, k, v = _rand((Hq, S, D), 1), _rand((1, S, D), 2), _rand((1, S, D), 3)
    o, lse = O.attn_fwd(q, k, v, row_block=8)
    for t in (0, 7, 23, 38):
        q2, k2, v2 = q.copy(), k.copy(), v.copy()
        q2[:, t + 1:] += 3.0
        k2[:, t + 1:] -= 2.0
        v2[:, t + 1:] *= -5.0
        o2, lse2 = O.attn_fwd(q2, k2, v2, row_block=8)
        assert np.array_equal(o[:, :t + 1], o2[:, :t + 1])
        assert np.array_equal(lse[:, :t + 1], lse2[:, :t + 1])


def test_document_isolation_bit_identical():
    Hq, S, D = 2, 30, 4
    cu = [0, 9, 17, 30]
    q, k, v = _rand((Hq, S, D), 1), _rand((1, S, D), 2), _rand((1, S, D), 3)
    for causal in (True, False):
        o, lse = O.attn_fwd(q, k, v, cu, causal, row_block=8)
        q2, k2, v2 = q.copy(), k.copy(), v.copy()
        q2[:, 9:17] = 9.0
        k2[:, 9:17] = -1.0
        v2[:, 9:17] = 4.0
        o2, lse2 = O.attn_fwd(q2, k2, v2, cu, causal, row_block=8)
        keep = np.r_[0:9, 17:30]
        assert np.array_equal(o[:, keep], o2[:, keep])
        assert np.array_equal(lse[:, keep], lse2[:, keep])


def test_gqa_equals_repeated_mha():
    Hq, Hkv, S, D = 8, 2, 19, 4
    q, k, v, do = _rand((Hq, S, D), 1), _rand((Hkv, S, D), 2), _rand((Hkv, S, D), 3), \
        _rand((Hq, S, D), 4)
    G = Hq // Hkv
    kr, vr = np.repeat(k, G, axis=0), np.repeat(v, G, axis=0)
    o, lse = O.attn_fwd(q, k, v, [0, 6, 19])
    o2, lse2 = O.attn_fwd(q, kr, vr, [0, 6, 19])
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    dq, dk, dv = O.attn_bwd(q, k, v, do, [0, 6, 19])
    dq2, dk2, dv2 = O.attn_bwd(q, kr, vr, do, [0, 6, 19])
    np.testing.assert_allclose(dq, dq2, atol=1e-14)
    np.testing.assert_allclose(dk, dk2.reshape(Hkv, G, S, D).sum(1), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(Hkv, G, S, D).sum(1), atol=1e-13)


def test_single_doc_equals_plain_causal():
    q, k, v = _rand((2, 21, 4), 1), _rand((1, 21, 4), 2), _rand((1, 21, 4), 3)
    a = O.attn_fwd(q, k, v, None)
    b = O.attn_fwd(q, k, v, [0, 21])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bad_cu_seqlens_rejected():
    q = _rand((1, 8, 2), 1)
    for cu in ([1, 8], [0, 7], [0, 5, 3, 8]):
        with pytest.raises(ValueError):
            O.attn_fwd(q, q, q, cu)


# ---------------------------------------------------------------- backward

def _loss(q, k, v, do, cu, causal):
    o, _ = O.attn_fwd(q, k, v, cu, causal, row_block=8)
    return float(np.sum(o * do))


@pytest.mark.parametrize("cu,causal", [(None, True), ([0, 7, 16], True), ([0, 9, 16], False)])
def test_bwd_finite_differences(cu, causal):
    Hq, Hkv, S, D = 4, 2, 16, 8
    q, k, v, do = (_rand((Hq, S, D), 21), _rand((Hkv, S, D), 22), _rand((Hkv, S, D), 23),
                   _rand((Hq, S, D), 24))
    grads = O.attn_bwd(q, k, v, do, cu, causal, row_block=8)
    rng = np.random.Generator(np.random.PCG64(9))
    h = 1e-6
    for t, (x, gx) in enumerate(zip((q, k, v), grads)):
        for _ in range(12):
            idx = tuple(rng.integers(0, n) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[t], args_m[t] = xp, xm
            fd = (_loss(*args_p, do, cu, causal) - _loss(*args_m, do, cu, causal)) / (2 * h)
            assert abs(fd - gx[idx]) <= 1e-7 * max(1.0, abs(fd)) + 1e-8, (t, idx, fd, gx[idx])


def test_bwd_sum_invariants():
    """sum_j dK_j = 0 (dS rows sum to D_i - D_i = 0) and sum_j dV_j = sum of dO
    over the kv group's rows (P rows sum to 1), per kv head and document."""
    Hq, Hkv, S, D = 6, 2, 40, 5
    cu = [0, 13, 14, 40]
    q, k, v, do = _rand((Hq, S, D), 31), _rand((Hkv, S, D), 32), _rand((Hkv, S, D), 33), \
        _rand((Hq, S, D), 34)
    dq, dk, dv = O.attn_bwd(q, k, v, do, cu)
    G = Hq // Hkv
    for g in range(Hkv):
        for a, b in zip(cu[:-1], cu[1:]):
            assert np.max(np.abs(dk[g, a:b].sum(0))) < 1e-12
            want = do[g * G:(g + 1) * G, a:b].sum((0, 1))
            np.testing.assert_allclose(dv[g, a:b].sum(0), want, atol=1e-12)


# ---------------------------------------------------------------- the layer

def test_ulysses_layer_independent_of_P_and_chunk():
    B, S, Hq, Hkv, D = 1, 24, 8, 4, 4
    qs, ks, vs, dos = (_rand((B, S, Hq, D), 1), _rand((B, S, Hkv, D), 2),
                       _rand((B, S, Hkv, D), 3), _rand((B, S, Hq, D), 4))
    cu = [0, 5, 24]
    ref_o, ref_l = O.attn_fwd(qs[0].transpose(1, 0, 2), ks[0].transpose(1, 0, 2),
                              vs[0].transpose(1, 0, 2), cu)
    ref_g = O.attn_bwd(qs[0].transpose(1, 0, 2), ks[0].transpose(1, 0, 2),
                       vs[0].transpose(1, 0, 2), dos[0].transpose(1, 0, 2), cu)
    G = Hq // Hkv
    for P in (1, 2, 4):
        hq = Hq // P
        for C in [c for c in range(G, hq + 1, G) if hq % c == 0]:
            o, l = O.ulysses_attention(qs, ks, vs, P, C, cu)
            assert np.array_equal(o[0].transpose(1, 0, 2), ref_o)
            assert np.array_equal(l[0], ref_l)
            g = O.ulysses_attention_bwd(qs, ks, vs, dos, P, C, cu)
            for a, b in zip(g, ref_g):
                assert np.array_equal(a[0].transpose(1, 0, 2), b)


def test_row_and_tail_pieces_agree_with_full():
    Hq, Hkv, S, D = 4, 1, 50, 6
    q, k, v, do = _rand((Hq, S, D), 1), _rand((Hkv, S, D), 2), _rand((Hkv, S, D), 3), \
        _rand((Hq, S, D), 4)
    cu = [0, 20, 21, 50]
    o, lse = O.attn_fwd(q, k, v, cu)
    dq, dk, dv = O.attn_bwd(q, k, v, do, cu)
    rows = [0, 19, 20, 21, 33, 49]
    for h in range(Hq):
        for group in (1, 4, 16):
            ro, rl, rdq = O.attn_rows(q[h], k[0], v[0], do[h], rows, cu, row_group=group)
            np.testing.assert_allclose(ro, o[h, rows], atol=1e-13)
            np.testing.assert_allclose(rl, lse[h, rows], atol=1e-13)
            np.testing.assert_allclose(rdq, dq[h, rows], atol=1e-13)
        # compact form: only the selected rows of q/dO are passed
        ro, rl, rdq = O.attn_rows(q[h][rows], k[0], v[0], do[h][rows], rows, cu)
        np.testing.assert_allclose(rdq, dq[h, rows], atol=1e-13)
    tk, tv = O.attn_kv_tail(q, k[0], v[0], do, 30, cu, row_block=7)
    np.testing.assert_allclose(tk, dk[0, 30:], atol=1e-12)
    np.testing.assert_allclose(tv, dv[0, 30:], atol=1e-12)


def test_num_pairs():
    assert O.num_pairs(8192) == 8192 * 8193 // 2
    assert O.num_pairs(10, [0, 3, 10]) == 6 + 28
    assert O.num_pairs(10, [0, 3, 10], causal=False) == 9 + 49


# ---------------------------------------------------------------- mutants

def _dense_mutant_bwd(variant):
    """A dense re-statement of the backward with one planted mistake."""
    def bwd(q, k, v, do, cu=None, causal=True, scale=None, row_block=512):
        q, k, v, do = (np.asarray(x, float) for x in (q, k, v, do))
        Hq, S, D = q.shape
        G = Hq // k.shape[0]
        sc = 1 / math.sqrt(D) if scale is None else scale
        lo, hi = O.key_ranges(S, cu, causal)
        j = np.arange(S)
        allowed = (j[None] >= lo[:, None]) & (j[None] < hi[:, None])
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for h in range(Hq):
            g = h // G
            s = np.where(allowed, sc * q[h] @ k[g].T, -np.inf)
            p = np.exp(s - s.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            dp = do[h] @ v[g].T
            Di = (p * dp).sum(1, keepdims=True)
            ds = p * dp if variant == "no_delta" else p * (dp - Di)
            if variant == "dk_transposed":
                dk[g] += sc * ds @ q[h]
            else:
                dk[g] += sc * ds.T @ q[h]
            dq[h] = sc * ds @ k[g]
            dv[g] += p.T @ do[h]
        return dq, dk, dv
    return bwd


def test_mutants_are_caught(monkeypatch):
    """Plant plausible mistakes in the oracle (on the CPU) and check a pin fails."""
    real_bwd, real_fwd, real_s2h = O.attn_bwd, O.attn_fwd, O.seq2head

    # the dense restatement without a mistake passes the pins
    monkeypatch.setattr(O, "attn_bwd", _dense_mutant_bwd("none"))
    test_golden_worked_example()
    test_bwd_finite_differences(None, True)

    for variant, pin in (("no_delta", test_golden_worked_example),
                         ("no_delta", lambda: test_bwd_finite_differences(None, True)),
                         ("dk_transposed", test_bwd_sum_invariants)):
        monkeypatch.setattr(O, "attn_bwd", _dense_mutant_bwd(variant))
        with pytest.raises(AssertionError):
            pin()
    monkeypatch.setattr(O, "attn_bwd", real_bwd)

    def fwd_wrong_group(q, k, v, cu=None, causal=True, scale=None, row_block=512):
        # GQA mapping h % Hkv instead of h // G
        Hq, Hkv = q.shape[0], k.shape[0]
        G = Hq // Hkv
        kk = np.asarray(k)[[h % Hkv for h in range(Hq)]]
        vv = np.asarray(v)[[h % Hkv for h in range(Hq)]]
        return real_fwd(q, kk, vv, cu, causal, scale, row_block)

    monkeypatch.setattr(O, "attn_fwd", fwd_wrong_group)
    with pytest.raises(AssertionError):
        test_matches_torch_sdpa_fp64(True)

    def fwd_wrong_scale(q, k, v, cu=None, causal=True, scale=None, row_block=512):
        return real_fwd(q, k, v, cu, causal, 1.0 / q.shape[2] if scale is None else scale,
                        row_block)

    monkeypatch.setattr(O, "attn_fwd", fwd_wrong_scale)
    with pytest.raises(AssertionError):
        test_lse_matches_library_logsumexp()

    def fwd_strict_causal(q, k, v, cu=None, causal=True, scale=None, row_block=512):
        # the diagonal dropped (keys j < i only; row 0 keeps itself to stay finite)
        o, lse = real_fwd(q, k, v, cu, causal, scale, row_block)
        q2 = np.asarray(q, float).copy()
        o2, lse2 = real_fwd(q2[:, 1:], np.asarray(k)[:, :-1], np.asarray(v)[:, :-1], None,
                            causal, scale, row_block)
        o[:, 1:], lse[:, 1:] = o2, lse2
        return o, lse

    monkeypatch.setattr(O, "attn_fwd", fwd_strict_causal)
    with pytest.raises(AssertionError):
        test_golden_worked_example()
    monkeypatch.setattr(O, "attn_fwd", real_fwd)

    def s2h_strided(x, P, head_chunk=None, stage=None):
        # heads dealt round-robin to ranks instead of in contiguous blocks
        H = x.shape[2]
        perm = np.arange(H).reshape(H // P, P).T.reshape(-1)
        return real_s2h(x[:, :, perm], P, head_chunk, stage)

    monkeypatch.setattr(O, "seq2head", s2h_strided)
    with pytest.raises(AssertionError):
        test_golden_relayout()
    monkeypatch.setattr(O, "seq2head", real_s2h)


# ---------------------------------------------------------------- projections (steps 2 and 6)

def test_golden_projections():
    g = json.load(open(os.path.join(GOLD, "proj_2tok.json")))
    for case in g["cases"]:
        x = np.array(case["x"], dtype=np.float64)
        w = np.array(case["w_qkv"], dtype=np.float64)
        got = O.qkv_proj(x, w, case["H_q"], case["H_kv"], case["P"])
        np.testing.assert_array_equal(got, np.array(case["qkv_head"], dtype=np.float64), err_msg=case["name"])
        y = O.out_proj(np.array(case["o_head"], dtype=np.float64), np.array(case["w_o"], dtype=np.float64),
                       case["P"])
        np.testing.assert_array_equal(y, np.array(case["y"], dtype=np.float64), err_msg=case["name"])


def _qkv_bruteforce(x, w, n_heads, D):
    S, hidden = x.shape
    out = np.zeros((n_heads, S, D))
    for h in range(n_heads):
        for s in range(S):
            for d in range(D):
                acc = 0.0
                for c in range(hidden):
                    acc += x[s, c] * w[h * D + d, c]
                out[h, s, d] = acc
    return out


def _out_bruteforce(o, w):
    Hq, S, D = o.shape
    hidden = w.shape[0]
    y = np.zeros((S, hidden))
    for s in range(S):
        for c in range(hidden):
            acc = 0.0
            for h in range(Hq):
                for d in range(D):
                    acc += o[h, s, d] * w[c, h * D + d]
            y[s, c] = acc
    return y


@pytest.mark.parametrize("S,hidden,Hq,Hkv,D,P", [(8, 6, 4, 2, 3, 2), (12, 5, 3, 3, 2, 3), (4, 4, 4, 4, 4, 4)])
def test_projections_bruteforce_and_rank_split(S, hidden, Hq, Hkv, D, P):
    x = _rand((S, hidden), 70)
    w = _rand(((Hq + 2 * Hkv) * D, hidden), 71)
    got = O.qkv_proj(x, w, Hq, Hkv, P)
    np.testing.assert_allclose(got, _qkv_bruteforce(x, w, Hq + 2 * Hkv, D), rtol=0, atol=1e-12)
    # the rank split of the tokens does not change the result
    np.testing.assert_allclose(O.qkv_proj(x, w, Hq, Hkv, 1), got, rtol=0, atol=1e-12)
    o = _rand((Hq, S, D), 72)
    wo = _rand((hidden, Hq * D), 73)
    y = O.out_proj(o, wo, P)
    np.testing.assert_allclose(y, _out_bruteforce(o, wo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(O.out_proj(o, wo, 1), y, rtol=0, atol=1e-12)


def test_projection_identity_round_trip():
    """With hidden = H_q D and identity weights, step 2's Q heads are the
    all-to-all of x itself, and step 6 with identity weights gives x back:
    the two layout maps are inverse to each other."""
    S, Hq, Hkv, D, P = 8, 4, 2, 3, 2
    hidden = Hq * D
    x = _rand((S, hidden), 74)
    w = np.zeros(((Hq + 2 * Hkv) * D, hidden))
    w[:hidden] = np.eye(hidden)
    qkv = O.qkv_proj(x, w, Hq, Hkv, P)
    np.testing.assert_array_equal(qkv[:Hq], O.seq2head(x.reshape(1, S, Hq, D), P)[0])
    assert not np.any(qkv[Hq:])
    np.testing.assert_array_equal(O.out_proj(qkv[:Hq], np.eye(hidden), P), x)


def test_projection_mutants_are_caught():
    """A transposed head/feature order or swapped K/V blocks in a copy of the
    projection fail the brute-force pin."""
    S, hidden, Hq, Hkv, D = 6, 5, 2, 1, 3
    x = _rand((S, hidden), 75)
    w = _rand(((Hq + 2 * Hkv) * D, hidden), 76)
    ref = _qkv_bruteforce(x, w, Hq + 2 * Hkv, D)
    y = x @ w.T
    feature_major = y.reshape(S, D, Hq + 2 * Hkv).transpose(2, 0, 1)     # d-major instead of head-major
    kv_swapped = np.concatenate([ref[:Hq], ref[Hq + Hkv:], ref[Hq:Hq + Hkv]])
    for bad in (feature_major, kv_swapped):
        assert np.max(np.abs(bad - ref)) > 1e-3


def test_oracle_pool_runs_the_oracle_unchanged():
    """The spawn pool used by the full-size GPU checks returns exactly what a
    direct call of the oracle returns (same functions, same inputs)."""
    from tests import oracle_pool
    S, D = 96, 8
    q, k, v, do = (_rand((S, D), 80 + i).astype(np.float32) for i in range(4))
    cu = np.array([0, 40, 96])
    (o, lse, dq, dk, dv), = oracle_pool.run(oracle_pool.head_fwd_bwd, [(q, k, v, do, cu, True)])
    ro, rl = O.attn_fwd(q[None], k[None], v[None], cu, True)
    rq, rk, rv = O.attn_bwd(q[None], k[None], v[None], do[None], cu, True)
    for a, b in ((o, ro[0]), (lse, rl[0]), (dq, rq[0]), (dk, rk[0]), (dv, rv[0])):
        np.testing.assert_array_equal(a, b)
    rows = np.array([0, 39, 40, 95])
    got = oracle_pool.run(oracle_pool.head_rows, [(q[rows], k, v, do[rows], rows, cu, True)])[0]
    want = O.attn_rows(q[rows], k, v, do[rows], rows, cu, True)
    for a, b in zip(got, want):
        np.testing.assert_array_equal(a, b)
    j0 = 64
    tk, tv = oracle_pool.run(oracle_pool.head_kv_tail, [(q[j0:], k, v, do[j0:], j0, cu, True, 16)])[0]
    np.testing.assert_allclose(tk, rk[0, j0:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(tv, rv[0, j0:], rtol=0, atol=1e-12)
