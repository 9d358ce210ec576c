"""GPU test of ulysses_attn_bwd_noalloc, the backward entry point for callers
that cannot allocate device memory (it uses the library's built-in scratch
instead of a caller workspace).

It runs the same kernels as ulysses_attn_bwd, so on the same inputs it must
agree with it call after call: dK and dV bit for bit, dQ to 1e-5 of its
largest magnitude (the tcgen05 backward sums dQ with fp32 reduce-adds in the
order they reach L2, so two runs may differ in the last bits).  Two calls in a
row, with different inputs, check that the scratch left by one call does not
leak into the next.  Once the library's device code is loaded, a call must not
change the device's free memory.  The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

from long_context_sequence_seq_gb300 import ulysses as U
from tests.gpu_util import seq_inputs

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
        dq_ref, dk_ref, dv_ref = ref
        dq, dk, dv = got
        assert torch.equal(dk, dk_ref), (call, "dK")
        assert torch.equal(dv, dv_ref), (call, "dV")
        err = float((dq - dq_ref).abs().max())
        assert err <= 1e-5 * max(1.0, float(dq_ref.abs().max())), (call, "dQ", err)


def test_noalloc_call_allocates_nothing():
    S, Hq, Hkv, D, P, C = 512, 8, 2, 128, 2, 4
    qh, kh, vh, oh, doh, lse = _stage_buffers(S, Hq, Hkv, D, P, C, 30)
    dq = torch.empty(qh.shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(kh.shape, dtype=torch.float32, device="cuda")
    dv = torch.empty(vh.shape, dtype=torch.float32, device="cuda")
    # the first call may load the library's device code; after it, no call
    # may take device memory (outputs are passed in, nothing else is needed)
    U.attn_bwd_noalloc(qh, kh, vh, oh, doh, lse, Hq, Hkv, P, C, 0, dq=dq, dk=dk, dv=dv)
    U.check()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        U.attn_bwd_noalloc(qh, kh, vh, oh, doh, lse, Hq, Hkv, P, C, 0, dq=dq, dk=dk, dv=dv)
    U.check()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)


def test_noalloc_rejects_oversized_stage():
    # 2 heads x 4,194,304 tokens is twice the built-in scratch: rejected before
    # any device work (the pointers are never dereferenced)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    S = 1 << 22
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = U.lib().ulysses_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, S, 1, 2, 1, 128, 1, 2, 0,
                                          None, 0, 1, 0.0, U.BF16, None)
    assert rc == U.ERR_UNSUPPORTED
    assert b"built-in scratch" in U.lib().ulysses_last_error()
