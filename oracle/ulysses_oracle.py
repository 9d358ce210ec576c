"""fp64 CPU oracle for the Ulysses sequence-parallel attention hot path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` call it.  It shares no code with the
CUDA path (the two meet only in the seeded input generators, which hold none of
the method's arithmetic).

What it computes, and where that is defined:

* Sequence sharding and the two all-to-alls.  Page "Ulysses Sequence
  Parallelism for million-token context training" (Hugging Face summary),
  section "How Ulysses sequence parallelism works", steps 1, 3 and 5: every rank
  holds a contiguous token chunk with all heads; the first all-to-all leaves
  each rank with every position for a subset of heads; the second one restores
  the sequence-sharded form.  With P ranks simulated as P partitions of one
  buffer, both all-to-alls are permutations of D-vectors.  Index map used here
  (the plain contiguous split; the pages give no strides):

      X_head[r][h'][t][d] = X_seq[t div (S/P)][t mod (S/P)][r*hq + h'][d]

  UPipe head chunking (page "Ulysses Sequence Parallelism" commentary, section
  on going beyond a million tokens: process only some heads at a time) selects
  the stage (r, c) = q heads [r*hq + c*C, r*hq + (c+1)*C) of rank r.

* Local attention, step 4: dense softmax attention over the full sequence for
  the rank's heads.  FlashAttention computes this exact result (same page,
  "Challenges of long-sequence training": it lowers memory to O(n), the FLOPs
  stay O(n^2)), so the oracle is the plain definition

      s_ij = scale * q_i . k_j,  masked to j <= i (causal) and doc(i) == doc(j)
      O_i  = sum_j softmax_j(s_i) v_j,     LSE_i = log sum_j exp(s_ij)

  The document mask comes from packing (TRL SFTTrainer section) together with
  AutoSP's index recomputation (page "AutoSP", section 2.A step 4): masks are in
  global token indices.  GQA: q head h reads kv head h div G.

* Backward: the analytic gradient of the same definition,

      P_ij = exp(s_ij - LSE_i), dV_j = sum_i P_ij dO_i, dP_ij = dO_i . v_j,
      D_i = sum_j P_ij dP_ij (= dO_i . O_i), dS_ij = P_ij (dP_ij - D_i),
      dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,

  with dK/dV summed over the G q heads that share a kv head.

* Projections, steps 2 and 6 of the same section: every rank projects its own
  token chunk to Q, K and V (a plain matmul with the weights, rows
  independent), the first all-to-all then moves the projected heads; after
  the second all-to-all every rank applies the output projection to its own
  chunk.  Weight rows are ordered Q heads, K heads, V heads, D per head (the
  usual fused QKV weight; the pages give no order).

Readings where the pages are silent: scale 1/sqrt(D) unless given; causal
means j <= i (diagonal included); LSE is the natural log.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "stage_heads", "seq2head", "head2seq", "seq2head_bruteforce", "head2seq_bruteforce",
    "relayout_bytes_per_rank", "key_ranges", "attn_fwd", "attn_bwd",
    "attn_fwd_bruteforce", "attn_bwd_bruteforce", "ulysses_attention",
    "ulysses_attention_bwd", "attn_rows", "attn_kv_tail", "num_pairs", "qkv_proj", "out_proj",
]


# ----------------------------------------------------------------------------
# Re-layout (all-to-all #1 / #2 as permutations)
# ----------------------------------------------------------------------------

def stage_heads(H: int, P: int, head_chunk: int | None, stage):
    """Global head indices a stage owns.

    ``stage`` is None for every head of every rank, else (r, c) or the flat
    index r * (hq // C) + c.  ``H`` is H_q for Q-like tensors and H_kv for
    K/V; for K/V pass the kv chunk C / G.
    """
    if H % P:
        raise ValueError("head count must be divisible by the number of ranks")
    hq = H // P
    if stage is None:
        return np.arange(H)
    C = hq if head_chunk is None else head_chunk
    if C <= 0 or hq % C:
        raise ValueError("head_chunk must divide the per-rank head count")
    if isinstance(stage, (tuple, list)):
        r, c = stage
    else:
        r, c = divmod(int(stage), hq // C)
    if not (0 <= r < P and 0 <= c < hq // C):
        raise ValueError("stage out of range")
    return r * hq + c * C + np.arange(C)


def seq2head(x_seq: np.ndarray, P: int, head_chunk=None, stage=None) -> np.ndarray:
    """All-to-all #1 as a permutation: [B, S, H, D] (P stacked rank chunks) ->
    head layout [B, n_heads, S, D] for the selected stage (all heads if None).

    Ranks' token chunks stacked in rank order are exactly the global sequence,
    so the map is a gather of the stage's heads followed by a (S, H) transpose.
    """
    B, S, H, D = x_seq.shape
    if S % P:
        raise ValueError("S must be divisible by the number of ranks")
    heads = stage_heads(H, P, head_chunk, stage)
    return np.ascontiguousarray(np.transpose(x_seq[:, :, heads, :], (0, 2, 1, 3)))


def head2seq(x_head: np.ndarray, x_seq_out: np.ndarray, P: int, head_chunk=None, stage=None):
    """All-to-all #2: write head layout [B, n_heads, S, D] back into the stage's
    heads of the sequence layout [B, S, H, D] (in place on ``x_seq_out``)."""
    B, S, H, D = x_seq_out.shape
    if S % P:
        raise ValueError("S must be divisible by the number of ranks")
    heads = stage_heads(H, P, head_chunk, stage)
    x_seq_out[:, :, heads, :] = np.transpose(x_head, (0, 2, 1, 3))
    return x_seq_out


def seq2head_bruteforce(x_seq, P, head_chunk=None, stage=None):
    """The same permutation written index by index from the rank view:
    rank r sends its chunk's tokens for head h to the owner of h."""
    B, S, H, D = x_seq.shape
    Sp = S // P
    hq = H // P
    heads = stage_heads(H, P, head_chunk, stage)
    out = np.empty((B, len(heads), S, D), dtype=x_seq.dtype)
    for b in range(B):
        for src in range(P):              # source rank holding tokens [src*Sp, (src+1)*Sp)
            for s_local in range(Sp):
                t = src * Sp + s_local
                for n, h in enumerate(heads):
                    dst, hp = divmod(int(h), hq)   # destination rank and its local head
                    assert dst * hq + hp == h
                    for d in range(D):
                        out[b, n, t, d] = x_seq[b, s_local + src * Sp, h, d]
    return out


def head2seq_bruteforce(x_head, x_seq_out, P, head_chunk=None, stage=None):
    B, S, H, D = x_seq_out.shape
    Sp = S // P
    heads = stage_heads(H, P, head_chunk, stage)
    for b in range(B):
        for n, h in enumerate(heads):
            for t in range(S):
                dst, s_local = divmod(t, Sp)  # rank that owns token t after the return trip
                for d in range(D):
                    x_seq_out[b, dst * Sp + s_local, h, d] = x_head[b, n, t, d]
    return x_seq_out


def relayout_bytes_per_rank(S: int, H: int, D: int, P: int, elt: int) -> int:
    """Bytes one rank sends in one all-to-all: its S/P tokens x H heads x D.

    Matches the O(n d / P) per-GPU communication volume of the "Communication
    complexity" section (n = S, d = H * D)."""
    return (S // P) * H * D * elt


# ----------------------------------------------------------------------------
# Masks
# ----------------------------------------------------------------------------

def key_ranges(S: int, cu_seqlens=None, causal: bool = True):
    """Per query row i the half-open key range [lo_i, hi_i) it may attend to.

    lo_i = start of i's document; hi_i = i + 1 if causal else end of i's
    document.  Without cu_seqlens the whole sequence is one document.
    """
    i = np.arange(S, dtype=np.int64)
    if cu_seqlens is None:
        lo = np.zeros(S, dtype=np.int64)
        end = np.full(S, S, dtype=np.int64)
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        if cu[0] != 0 or cu[-1] != S or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must rise monotonically from 0 to S")
        doc = np.searchsorted(cu, i, side="right") - 1
        lo = cu[doc]
        end = cu[doc + 1]
    hi = i + 1 if causal else end
    return lo, hi


def num_pairs(S: int, cu_seqlens=None, causal: bool = True) -> int:
    """Number of unmasked (i, j) pairs per head."""
    lo, hi = key_ranges(S, cu_seqlens, causal)
    return int(np.sum(hi - lo))


# ----------------------------------------------------------------------------
# Attention (plain definition, fp64)
# ----------------------------------------------------------------------------

def _as64(x):
    return np.asarray(x, dtype=np.float64)


def attn_fwd(q, k, v, cu_seqlens=None, causal=True, scale=None, row_block=512):
    """Masked softmax attention on head-layout inputs.

    q: [Hq, S, D], k/v: [Hkv, S, D] (any float dtype; computed in fp64).
    Returns O [Hq, S, D] and LSE [Hq, S] (natural log), both fp64.
    Rows are processed in blocks; for a block only keys up to its largest
    allowed index are formed.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    Hq, S, D = q.shape
    Hkv = k.shape[0]
    if Hq % Hkv:
        raise ValueError("H_q must be a multiple of H_kv")
    G = Hq // Hkv
    sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
    lo, hi = key_ranges(S, cu_seqlens, causal)
    O = np.zeros((Hq, S, v.shape[2]))
    LSE = np.zeros((Hq, S))
    for h in range(Hq):
        g = h // G
        for i0 in range(0, S, row_block):
            i1 = min(S, i0 + row_block)
            j0, j1 = int(lo[i0:i1].min()), int(hi[i0:i1].max())
            s = sc * (q[h, i0:i1] @ k[g, j0:j1].T)
            j = np.arange(j0, j1)
            allowed = (j[None, :] >= lo[i0:i1, None]) & (j[None, :] < hi[i0:i1, None])
            s = np.where(allowed, s, -np.inf)
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            l = e.sum(axis=1)
            O[h, i0:i1] = (e / l[:, None]) @ v[g, j0:j1]
            LSE[h, i0:i1] = m + np.log(l)
    return O, LSE


def attn_bwd(q, k, v, do, cu_seqlens=None, causal=True, scale=None, row_block=512):
    """Analytic backward of ``attn_fwd`` for upstream gradient dO.

    Returns dQ [Hq,S,D], dK [Hkv,S,D], dV [Hkv,S,D] in fp64.  P is recomputed
    from the definition; nothing from a GPU run is used.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    Hq, S, D = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
    lo, hi = key_ranges(S, cu_seqlens, causal)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for h in range(Hq):
        g = h // G
        for i0 in range(0, S, row_block):
            i1 = min(S, i0 + row_block)
            j0, j1 = int(lo[i0:i1].min()), int(hi[i0:i1].max())
            kk, vv = k[g, j0:j1], v[g, j0:j1]
            s = sc * (q[h, i0:i1] @ kk.T)
            j = np.arange(j0, j1)
            allowed = (j[None, :] >= lo[i0:i1, None]) & (j[None, :] < hi[i0:i1, None])
            s = np.where(allowed, s, -np.inf)
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            Pm = e / e.sum(axis=1)[:, None]
            dOb = do[h, i0:i1]
            dV[g, j0:j1] += Pm.T @ dOb
            dP = dOb @ vv.T
            Di = np.sum(Pm * dP, axis=1)
            dS = Pm * (dP - Di[:, None])
            dQ[h, i0:i1] = sc * (dS @ kk)
            dK[g, j0:j1] += sc * (dS.T @ q[h, i0:i1])
    return dQ, dK, dV


def attn_fwd_bruteforce(q, k, v, cu_seqlens=None, causal=True, scale=None):
    """Scalar triple-loop twin of ``attn_fwd`` (S <= 64 only)."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    Hq, S, D = q.shape
    assert S <= 64, "brute force is for tiny inputs"
    G = Hq // k.shape[0]
    sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
    docs = _doc_of(S, cu_seqlens)
    O = np.zeros((Hq, S, D))
    LSE = np.zeros((Hq, S))
    for h in range(Hq):
        g = h // G
        for i in range(S):
            keys = [j for j in range(S) if docs[j] == docs[i] and (j <= i or not causal)]
            s = {}
            for j in keys:
                acc = 0.0
                for d in range(D):
                    acc += q[h, i, d] * k[g, j, d]
                s[j] = sc * acc
            z = sum(math.exp(s[j]) for j in keys)
            for d in range(D):
                O[h, i, d] = sum(math.exp(s[j]) / z * v[g, j, d] for j in keys)
            LSE[h, i] = math.log(z)
    return O, LSE


def attn_bwd_bruteforce(q, k, v, do, cu_seqlens=None, causal=True, scale=None):
    """Scalar-loop twin of ``attn_bwd`` (S <= 64 only)."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    Hq, S, D = q.shape
    assert S <= 64
    G = Hq // k.shape[0]
    sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
    docs = _doc_of(S, cu_seqlens)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for h in range(Hq):
        g = h // G
        for i in range(S):
            keys = [j for j in range(S) if docs[j] == docs[i] and (j <= i or not causal)]
            s = {j: sc * sum(q[h, i, d] * k[g, j, d] for d in range(D)) for j in keys}
            z = sum(math.exp(s[j]) for j in keys)
            p = {j: math.exp(s[j]) / z for j in keys}
            dp = {j: sum(do[h, i, d] * v[g, j, d] for d in range(D)) for j in keys}
            Di = sum(p[j] * dp[j] for j in keys)
            for j in keys:
                ds = p[j] * (dp[j] - Di)
                for d in range(D):
                    dV[g, j, d] += p[j] * do[h, i, d]
                    dQ[h, i, d] += sc * ds * k[g, j, d]
                    dK[g, j, d] += sc * ds * q[h, i, d]
    return dQ, dK, dV


def _doc_of(S, cu_seqlens):
    if cu_seqlens is None:
        return [0] * S
    cu = [int(x) for x in cu_seqlens]
    out = []
    d = 0
    for i in range(S):
        while i >= cu[d + 1]:
            d += 1
        out.append(d)
    return out


# ----------------------------------------------------------------------------
# The Ulysses layer (steps 3-5) with P virtual ranks and UPipe head chunks
# ----------------------------------------------------------------------------

def ulysses_attention(q_seq, k_seq, v_seq, P, head_chunk=None, cu_seqlens=None,
                      causal=True, scale=None):
    """Steps 3-5 per virtual rank and UPipe stage, in the sequence layout.

    q_seq [B,S,Hq,D], k_seq/v_seq [B,S,Hkv,D].  For every rank r and chunk c:
    all-to-all #1 (seq2head) of the stage's heads, local attention over all S
    positions, all-to-all #2 (head2seq).  Returns O [B,S,Hq,D] and LSE
    [B,Hq,S] (head-major, global head order).
    """
    B, S, Hq, D = q_seq.shape
    Hkv = k_seq.shape[2]
    G = Hq // Hkv
    hq = Hq // P
    C = hq if head_chunk is None else head_chunk
    if C % G:
        raise ValueError("each stage must own whole kv heads (C % G == 0)")
    O = np.zeros((B, S, Hq, D))
    LSE = np.zeros((B, Hq, S))
    for r in range(P):
        for c in range(hq // C):
            qh = seq2head(q_seq, P, C, (r, c))
            kh = seq2head(k_seq, P, C // G, (r, c))
            vh = seq2head(v_seq, P, C // G, (r, c))
            for b in range(B):
                o_h, lse_h = attn_fwd(qh[b], kh[b], vh[b], cu_seqlens, causal, scale)
                heads = stage_heads(Hq, P, C, (r, c))
                LSE[b, heads] = lse_h
                ob = np.zeros((1, S, Hq, D))
                head2seq(o_h[None], ob, P, C, (r, c))
                O[b][:, heads] = ob[0][:, heads]
    return O, LSE


def ulysses_attention_bwd(q_seq, k_seq, v_seq, do_seq, P, head_chunk=None, cu_seqlens=None,
                          causal=True, scale=None):
    """Backward of ``ulysses_attention``: each all-to-all is a permutation, so
    its adjoint is the inverse one (dO goes seq2head, gradients go head2seq)."""
    B, S, Hq, D = q_seq.shape
    Hkv = k_seq.shape[2]
    G = Hq // Hkv
    hq = Hq // P
    C = hq if head_chunk is None else head_chunk
    dQ = np.zeros((B, S, Hq, D))
    dK = np.zeros((B, S, Hkv, D))
    dV = np.zeros((B, S, Hkv, D))
    for r in range(P):
        for c in range(hq // C):
            qh = seq2head(q_seq, P, C, (r, c))
            kh = seq2head(k_seq, P, C // G, (r, c))
            vh = seq2head(v_seq, P, C // G, (r, c))
            doh = seq2head(do_seq, P, C, (r, c))
            for b in range(B):
                dq_h, dk_h, dv_h = attn_bwd(qh[b], kh[b], vh[b], doh[b], cu_seqlens, causal, scale)
                head2seq(dq_h[None], dQ[b:b + 1], P, C, (r, c))
                head2seq(dk_h[None], dK[b:b + 1], P, C // G, (r, c))
                head2seq(dv_h[None], dV[b:b + 1], P, C // G, (r, c))
    return dQ, dK, dV


# ----------------------------------------------------------------------------
# Row- and column-local pieces for sampled checks at full size
# ----------------------------------------------------------------------------

def attn_rows(q_h, k_g, v_g, do_h, rows, cu_seqlens=None, causal=True, scale=None, row_group=16):
    """O_i, LSE_i and dQ_i for selected rows of one q head.

    q_h/do_h: [S, D] of the q head (or just the selected rows, [len(rows), D],
    when their first dimension equals len(rows) < S), k_g/v_g: [S, D] of its
    kv head.  Each row needs only its own keys (cost O(S*D) per row); rows
    are taken ``row_group`` at a time over the union of their key ranges, as
    ``attn_fwd`` does with its row blocks.
    """
    S = k_g.shape[0]
    D = k_g.shape[1]
    sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
    lo, hi = key_ranges(S, cu_seqlens, causal)
    rows = np.asarray(rows, dtype=np.int64)
    compact = q_h.shape[0] == len(rows) and len(rows) < S
    k64 = _as64(k_g)
    v64 = _as64(v_g)
    O = np.zeros((len(rows), v_g.shape[1]))
    LSE = np.zeros(len(rows))
    dQ = np.zeros((len(rows), D))
    for g0 in range(0, len(rows), row_group):
        sel = np.arange(g0, min(len(rows), g0 + row_group))
        r = rows[sel]
        qq = _as64(q_h[sel] if compact else q_h[r])
        dd = _as64(do_h[sel] if compact else do_h[r])
        a, b = int(lo[r].min()), int(hi[r].max())
        j = np.arange(a, b)
        allowed = (j[None, :] >= lo[r, None]) & (j[None, :] < hi[r, None])
        s = np.where(allowed, sc * (qq @ k64[a:b].T), -np.inf)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        l = e.sum(axis=1)
        p = e / l[:, None]
        O[sel] = p @ v64[a:b]
        LSE[sel] = m + np.log(l)
        dp = dd @ v64[a:b].T
        Di = np.sum(p * dp, axis=1)
        dQ[sel] = sc * ((p * (dp - Di[:, None])) @ k64[a:b])
    return O, LSE, dQ


def attn_kv_tail(q_heads, k_g, v_g, do_heads, j0, cu_seqlens=None, causal=True, scale=None,
                 row_block=256):
    """dK_j, dV_j for key columns j in [j0, S) of one kv head (causal only).

    With a causal mask only rows i >= j0 touch these columns, so only those
    rows are formed; each still normalises over all of its keys.
    q_heads/do_heads: [G, S, D] for the q heads sharing this kv head.
    """
    if not causal:
        raise ValueError("column tails are only local under a causal mask")
    G, S, D = q_heads.shape
    sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
    lo, hi = key_ranges(S, cu_seqlens, causal)
    dK = np.zeros((S - j0, D))
    dV = np.zeros((S - j0, D))
    for g in range(G):
        for i0 in range(j0, S, row_block):
            i1 = min(S, i0 + row_block)
            a, b = int(lo[i0:i1].min()), int(hi[i0:i1].max())
            kk, vv = _as64(k_g[a:b]), _as64(v_g[a:b])
            qq, dd = _as64(q_heads[g, i0:i1]), _as64(do_heads[g, i0:i1])
            s = sc * (qq @ kk.T)
            j = np.arange(a, b)
            allowed = (j[None, :] >= lo[i0:i1, None]) & (j[None, :] < hi[i0:i1, None])
            s = np.where(allowed, s, -np.inf)
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            Pm = e / e.sum(axis=1)[:, None]
            dP = dd @ vv.T
            Di = np.sum(Pm * dP, axis=1)
            dS = Pm * (dP - Di[:, None])
            sel = j >= j0
            dV[j[sel] - j0] += Pm[:, sel].T @ dd
            dK[j[sel] - j0] += sc * (dS[:, sel].T @ qq)
    return dK, dV


# ----------------------------------------------------------------------------
# Projections around the all-to-alls (steps 2 and 6)
# ----------------------------------------------------------------------------

def qkv_proj(x, w_qkv, H_q, H_kv, P=1):
    """Step 2 then all-to-all #1: x [S, hidden], w_qkv [(H_q + 2 H_kv) D, hidden].

    Rank r projects its chunk of S/P tokens, y_r = x_r w_qkv^T, viewed as
    [S/P, H_q + 2 H_kv, D]; the chunks stacked in rank order are the sequence
    layout of Q, K and V, and seq2head (all heads) of each gives its head
    layout.  Returns [H_q + 2 H_kv, S, D] fp64: the Q heads, then the K heads,
    then the V heads.
    """
    x, w = _as64(x), _as64(w_qkv)
    S, hidden = x.shape
    n_heads = H_q + 2 * H_kv
    if w.shape[0] % n_heads or w.shape[1] != hidden:
        raise ValueError("w_qkv must be [(H_q + 2 H_kv) D, hidden]")
    D = w.shape[0] // n_heads
    if S % P:
        raise ValueError("S must be divisible by the number of ranks")
    Sp = S // P
    y_seq = np.zeros((1, S, n_heads, D))
    for r in range(P):
        y_seq[0, r * Sp:(r + 1) * Sp] = (x[r * Sp:(r + 1) * Sp] @ w.T).reshape(Sp, n_heads, D)
    q_seq, k_seq, v_seq = y_seq[:, :, :H_q], y_seq[:, :, H_q:H_q + H_kv], y_seq[:, :, H_q + H_kv:]
    return np.concatenate([seq2head(t, P)[0] for t in (q_seq, k_seq, v_seq)])


def out_proj(o_head, w_o, P=1):
    """All-to-all #2 then step 6: o_head [H_q, S, D] (every head, every
    position), w_o [hidden, H_q D].

    head2seq returns each rank its chunk with all heads, [S/P, H_q, D], which
    is flattened to [S/P, H_q D] and projected, y_r = o_r w_o^T.  Returns
    [S, hidden] fp64.
    """
    o, w = _as64(o_head), _as64(w_o)
    Hq, S, D = o.shape
    if w.shape[1] != Hq * D:
        raise ValueError("w_o must be [hidden, H_q D]")
    if S % P:
        raise ValueError("S must be divisible by the number of ranks")
    o_seq = np.zeros((1, S, Hq, D))
    head2seq(o[None], o_seq, P)
    Sp = S // P
    y = np.zeros((S, w.shape[0]))
    for r in range(P):
        y[r * Sp:(r + 1) * Sp] = o_seq[0, r * Sp:(r + 1) * Sp].reshape(Sp, Hq * D) @ w.T
    return y
