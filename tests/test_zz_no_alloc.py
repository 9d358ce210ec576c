"""GPU test of ulysses_attn_bwd_noalloc, the backward entry point for callers
that cannot allocate device memory (it uses the library's built-in scratch
instead of a caller workspace).

It must agree with ulysses_attn_bwd on the same inputs, call after call: two
calls in a row check that the shared scratch left by one call does not leak
into the next.  The file name makes pytest collect it last.
"""
import pytest
import torch

from long_context_sequence_seq_gb300 import ulysses as U
from tests.gpu_util import TOL, seq_inputs

pytestmark = pytest.mark.gpu


def _stage_buffers(S, Hq, Hkv, D, P, C, seed):
    q, k, v, do = seq_inputs(S, Hq, Hkv, D, "bf16", seed_offset=seed)
    G = Hq // Hkv
    st = 0
    qh, kh, vh = U.seq2head(q, P, C, st), U.seq2head(k, P, C // G, st), U.seq2head(v, P, C // G, st)
    doh = U.seq2head(do, P, C, st)
    oh, lse = U.attn_fwd(qh, kh, vh, Hq, Hkv, P, C, st)
    return qh, kh, vh, oh, doh, lse


@pytest.mark.parametrize("S,Hq,Hkv,D,P,C", [(384, 8, 2, 128, 2, 4), (1000, 8, 2, 64, 2, 4)])
def test_noalloc_matches_workspace_entry_point(S, Hq, Hkv, D, P, C):
    for call, seed in enumerate((10, 20)):            # two calls in a row, different inputs
        qh, kh, vh, oh, doh, lse = _stage_buffers(S, Hq, Hkv, D, P, C, seed)
        ref = U.attn_bwd(qh, kh, vh, oh, doh, lse, Hq, Hkv, P, C, 0)
        got = U.attn_bwd_noalloc(qh, kh, vh, oh, doh, lse, Hq, Hkv, P, C, 0)
        U.check()
        for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
            err = (a - b).abs().max().item()
            assert err <= TOL["bf16"], (call, name, err)


def test_noalloc_rejects_oversized_stage():
    # 2 heads x 4,194,304 tokens is twice the built-in scratch: rejected before
    # any device work (the pointers are never dereferenced)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    S = 1 << 22
    with pytest.raises(U.UlyssesError) as e:
        U.lib()
        import ctypes
        p = ctypes.c_void_p(dummy.data_ptr())
        rc = U.lib().ulysses_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, S, 1, 2, 1, 128, 1, 2, 0,
                                              None, 0, 1, 0.0, U.BF16, None)
        U._ck(rc)
    assert e.value.code == U.ERR_UNSUPPORTED
