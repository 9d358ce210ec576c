"""KV-head replication (H_kv < P) and padding (S % P != 0) on the GPU.

Replication does not change the mathematics: a rank holding a copy of kv
head g computes ordinary grouped-query attention for its q heads, and the
copies' dK/dV add up to dK/dV of g.  So the layer results are checked against
the oracle's plain attention over all heads (q head h uses kv head h // G),
which is independent of P.  Padding places the pad positions in a document of
their own, so the real positions' results equal attention on the unpadded
sequence.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_sequence_seq_gb300 import inputs, ulysses as U
from tests.gpu_util import LSE_TOL, TOL, f64, max_err, seq_inputs

pytestmark = pytest.mark.gpu


def _bits(t):
    t = t.detach().cpu()
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).numpy()


def test_replicated_kv_relayout():
    S, H_kv, D, P = 64, 2, 128, 4
    k = inputs.host_tensor((1, S, H_kv, D), 7, "bf16").cuda()
    R = P // H_kv
    for r in range(P):
        h = U.seq2head(k, P, None, r)
        assert h.shape == (1, 1, S, D)
        assert np.array_equal(_bits(h), _bits(k[:, :, r // R].unsqueeze(1)))
    # the accumulating scatter sums the replicas of a head
    g = inputs.host_tensor((1, S, H_kv, D), 8, "fp32").cuda()
    acc = torch.zeros_like(g)
    parts = [inputs.host_tensor((1, 1, S, D), 20 + r, "fp32").cuda() for r in range(P)]
    for r in range(P):
        (U.head2seq if r % R == 0 else U.head2seq_add)(parts[r], acc, P, None, r)
    U.check()
    for hk in range(H_kv):
        want = sum(parts[r][0, 0] for r in range(P) if r // R == hk)
        assert torch.equal(acc[0, :, hk], want)


def _oracle_layer(q, k, v, do, cu_np, causal):
    Q, K, V, DO = (f64(t)[0].transpose(1, 0, 2) for t in (q, k, v, do))
    ro, rl = oracle.attn_fwd(Q, K, V, cu_np, causal)
    rq, rk, rv = oracle.attn_bwd(Q, K, V, DO, cu_np, causal)
    tr = lambda a: a.transpose(1, 0, 2)
    return tr(ro), rl, tr(rq), tr(rk), tr(rv)


@pytest.mark.parametrize("S,Hq,Hkv,D,P,C,dtype,docs", [
    (512, 8, 2, 128, 4, 2, "bf16", None),          # H_kv = 2 < P = 4, one stage per rank
    (512, 8, 2, 128, 4, 1, "bf16", None),          # two stages per rank share the kv head
    (640, 8, 1, 128, 8, 1, "bf16", [200, 440]),    # H_kv = 1, P = 8, documents
    (64, 4, 1, 64, 2, 2, "fp32", None),            # fp32 SIMT path
])
def test_layer_with_replicated_kv(S, Hq, Hkv, D, P, C, dtype, docs):
    q, k, v, do = seq_inputs(S, Hq, Hkv, D, dtype)
    cu_np = None if docs is None else inputs.cu_seqlens_from_lengths(docs)
    cu = None if cu_np is None else torch.from_numpy(cu_np).cuda()
    o, lse = U.layer_fwd(q, k, v, P, C, cu_seqlens=cu)
    dq, dk, dv = U.layer_bwd(q, k, v, o, do, lse, P, C, cu_seqlens=cu)
    U.check()
    ro, rl, rq, rk, rv = _oracle_layer(q, k, v, do, cu_np, True)
    tol = TOL[dtype]
    assert max_err(f64(o)[0], ro) <= tol
    assert max_err(f64(lse)[0], rl) <= LSE_TOL[dtype]
    assert max_err(f64(dq)[0], rq) <= tol
    assert max_err(f64(dk)[0], rk) <= tol
    assert max_err(f64(dv)[0], rv) <= tol


@pytest.mark.parametrize("S,P,docs", [(1003, 4, None), (771, 8, [300, 471])])
def test_padding_to_multiple_of_P(S, P, docs):
    Hq, Hkv, D = 8, 8, 128
    q, k, v, do = seq_inputs(S, Hq, Hkv, D, "bf16")
    cu_np = None if docs is None else inputs.cu_seqlens_from_lengths(docs)
    cu = None if cu_np is None else torch.from_numpy(cu_np).cuda()
    (qp, kp, vp, dop), cup, S0 = U.pad_to_multiple([q, k, v, do], P, cu)
    assert qp.shape[1] % P == 0 and S0 == S
    o, lse = U.layer_fwd(qp, kp, vp, P, Hq // P, cu_seqlens=cup)
    dq, dk, dv = U.layer_bwd(qp, kp, vp, o, dop, lse, P, Hq // P, cu_seqlens=cup)
    U.check()
    ro, rl, rq, rk, rv = _oracle_layer(q, k, v, do, cu_np, True)
    assert max_err(f64(o[:, :S])[0], ro) <= TOL["bf16"]
    assert max_err(f64(lse[:, :, :S])[0], rl) <= LSE_TOL["bf16"]
    for got, want in ((dq, rq), (dk, rk), (dv, rv)):
        assert max_err(f64(got[:, :S])[0], want) <= TOL["bf16"]


@pytest.mark.parametrize("S,P,B,H,D,dtype,docs", [(10, 4, 2, 3, 64, "bf16", None), (1000, 8, 1, 2, 128, "fp32", [400, 600]),
                                                   (17, 1, 1, 1, 128, "bf16", None), (64, 4, 1, 2, 64, "bf16", [64])])
def test_pad_kernels_bit_exact(S, P, B, H, D, dtype, docs):
    """ulysses_pad_seq copies every real token bit for bit and zeroes the pad
    tokens; ulysses_pad_cu_seqlens appends the pad document."""
    x = inputs.host_tensor((B, S, H, D), 51, dtype).cuda()
    cu = None if docs is None else torch.from_numpy(inputs.cu_seqlens_from_lengths(docs)).cuda()
    (xp,), cup, S0 = U.pad_to_multiple([x], P, cu)
    U.check()
    S_pad = U.padded_length(S, P)
    assert S0 == S and xp.shape == (B, S_pad, H, D)
    bits = lambda t: t.cpu().view(torch.int16 if t.element_size() == 2 else torch.int32)  # noqa: E731
    assert torch.equal(bits(xp[:, :S]), bits(x))
    assert torch.count_nonzero(bits(xp[:, S:])) == 0
    real = [0, S] if docs is None else [0] + list(np.cumsum(docs))
    if S_pad == S:
        assert xp is x and (cup is cu)
    else:
        assert cup.cpu().tolist() == real + [S_pad]
