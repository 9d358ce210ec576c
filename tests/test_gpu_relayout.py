"""K1 re-layout on the GPU: bit-exact against the oracle's permutation."""
import numpy as np
import pytest
import torch

import oracle
from long_context_sequence_seq_gb300 import inputs, ulysses as U

pytestmark = pytest.mark.gpu


def _bits(t):
    t = t.detach().cpu()
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).numpy()


CASES = [
    # S, B, H, D, P, C, dtype
    (8, 1, 4, 64, 2, 1, "bf16"),
    (24, 2, 6, 128, 3, 2, "bf16"),
    (256, 1, 8, 64, 2, 4, "fp32"),
    (1000, 1, 8, 128, 8, 1, "bf16"),      # ragged: S not a tile multiple
    (4, 1, 32, 128, 4, 8, "fp32"),
    (8192, 1, 32, 128, 4, 8, "bf16"),     # Qwen3-4B-shaped layer, 8K tokens
    (8192, 1, 8, 128, 4, 2, "bf16"),      # its K/V (H_kv = 8, kv chunk = 2)
    (0, 1, 8, 128, 4, 2, "bf16"),         # empty
]


@pytest.mark.parametrize("S,B,H,D,P,C,dtype", CASES)
def test_relayout_bit_exact(S, B, H, D, P, C, dtype):
    x = inputs.host_tensor((B, S, H, D), 17, dtype).cuda()
    xb = _bits(x)
    hq = H // P
    stages = [None] + list(range(P * (hq // C)))
    y = torch.full_like(x, float("nan"))
    for st in stages:
        h = U.seq2head(x, P, C, st)
        want = oracle.seq2head(xb, P, C, st)
        assert np.array_equal(_bits(h), want)
        if st is not None:
            U.head2seq(h, y, P, C, st)
    U.check()
    assert np.array_equal(_bits(y), xb)          # head2seq o seq2head = id over all stages
    hall = U.seq2head(x, P)
    z = torch.empty_like(x)
    U.head2seq(hall, z, P)
    assert np.array_equal(_bits(U.seq2head(z, P)), _bits(hall))


@pytest.mark.parametrize("H,C", [(32, 8), (8, 2)])
def test_relayout_full_64k_layer(H, C):
    """The 64K-token Qwen3-4B-shaped layer (P=4): every stage bit-exact."""
    S, D, P = 65536, 128, 4
    x = inputs.device_tensor((1, S, H, D), 23, "bf16")
    xb = _bits(x)
    hq = H // P
    for st in range(P * (hq // C)):
        h = U.seq2head(x, P, C, st)
        assert np.array_equal(_bits(h), oracle.seq2head(xb, P, C, st)), st
    U.check()


@pytest.mark.parametrize("S,B,D,P,dtype", [(256, 1, 128, 4, "bf16"), (1000, 2, 64, 2, "bf16"),
                                           (96, 1, 128, 2, "fp32"), (65536, 1, 128, 4, "bf16")])
def test_batched_relayout_bit_exact(S, B, D, P, dtype):
    """One launch for a stage's Q, K, V, O and dO (and its gradients back):
    every tensor bit-exact against the oracle's permutation, the scatter
    restores the sequence layout, and the accumulating form adds (fp32)."""
    Hq, Hkv = 4 * P, 2 * P if P > 1 else 2
    C, Ckv = Hq // P // 2, max(1, Hkv // P // 2)
    seeds = (31, 32, 33, 34, 35)
    hs = (Hq, Hkv, Hkv, Hq, Hq)
    cs = (C, Ckv, Ckv, C, C)
    xs = [inputs.device_tensor((B, S, h, D), sd, dtype) for h, sd in zip(hs, seeds)]
    bits = [_bits(x) for x in xs]
    n_st = P * (Hq // P // C)
    for st in (0, n_st - 1):
        kst = st * (Hkv // P // Ckv) // (Hq // P // C)
        stg = (st, kst, kst, st, st)
        outs = [torch.empty((B, c, S, D), dtype=x.dtype, device="cuda") for x, c in zip(xs, cs)]
        U.seq2head_n([(x, o, c, s) for x, o, c, s in zip(xs, outs, cs, stg)], P)
        for o, xb, c, s in zip(outs, bits, cs, stg):
            assert np.array_equal(_bits(o), oracle.seq2head(xb, P, c, s)), st
        ys = [torch.zeros_like(x) for x in xs]
        U.head2seq_n([(o, y, c, s) for o, y, c, s in zip(outs, ys, cs, stg)], P)
        for o, y, c, s in zip(outs, ys, cs, stg):
            want = np.zeros_like(_bits(y))
            oracle.head2seq(_bits(o), want, P, c, s)
            assert np.array_equal(_bits(y), want), st
        if dtype == "fp32":
            base = [torch.randn_like(y) for y in ys[:3]]
            acc = [b.clone() for b in base]
            U.head2seq_n([(o, a, c, s, 1) for o, a, c, s in zip(outs[:3], acc, cs[:3], stg[:3])], P)
            for o, a, b, c, s in zip(outs[:3], acc, base, cs[:3], stg[:3]):
                want = b.cpu().numpy().copy()
                heads = oracle.stage_heads(a.shape[2], P, c, s)
                want[:, :, heads] += np.transpose(o.cpu().numpy(), (0, 2, 1, 3))
                assert np.array_equal(a.cpu().numpy(), want), st
    U.check()
