"""Out-of-bounds writes, caught without compute-sanitizer.

Every output and workspace buffer handed to the library is a window into a
larger allocation. The window has a 4 KB guard region on each side, and the
padding up to the next 256 bytes counts as guard too; all of it is filled with
a byte pattern. After each call the guards must still hold the pattern. The
shapes have ragged tails (S not a multiple of any tile size) and document
boundaries inside tiles, and every stage of the UPipe loop is run. The windows
start 4 KB into their allocation, so they keep the 16-byte alignment that TMA
needs.
"""
import pytest
import torch

from long_context_sequence_seq_gb300 import inputs, ulysses as U
from tests.gpu_util import seq_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096
PAT = 0xA5


class Guarded:
    def __init__(self):
        self.bufs = []

    def empty(self, shape, dtype):
        n = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        padded = (n + 255) // 256 * 256
        raw = torch.full((GUARD + padded + GUARD,), PAT, dtype=torch.uint8, device="cuda")
        self.bufs.append((raw, n))
        return raw[GUARD:GUARD + n].view(dtype).view(shape)

    def bytes(self, n):
        return self.empty((max(n, 256),), torch.uint8)

    def check(self):
        torch.cuda.synchronize()
        for i, (raw, n) in enumerate(self.bufs):
            assert bool((raw[:GUARD] == PAT).all()), f"buffer {i}: write before its start"
            assert bool((raw[GUARD + n:] == PAT).all()), f"buffer {i}: write past its end"


CASES = [
    # S, Hq, Hkv, D, P, C, doc lengths (None = one causal document)
    (300, 8, 2, 128, 2, 4, [150, 150]),
    (640, 4, 1, 128, 1, 4, [1, 300, 339]),
    (1000, 8, 2, 128, 2, 4, None),
    (260, 4, 2, 64, 2, 2, None),
]


@pytest.mark.parametrize("S,Hq,Hkv,D,P,C,docs", CASES)
def test_stage_calls_stay_in_bounds(S, Hq, Hkv, D, P, C, docs):
    q, k, v, do = seq_inputs(S, Hq, Hkv, D, "bf16")
    cu = None if docs is None else torch.from_numpy(inputs.cu_seqlens_from_lengths(docs)).cuda()
    G = Hq // Hkv
    g = Guarded()
    o = g.empty(q.shape, torch.bfloat16)
    dq = g.empty(q.shape, torch.float32)
    dk = g.empty(k.shape, torch.float32)
    dv = g.empty(v.shape, torch.float32)
    for st in range(P * (Hq // P // C)):
        qh = U.seq2head(q, P, C, st, out=g.empty((1, C, S, D), torch.bfloat16))
        kh = U.seq2head(k, P, C // G, st, out=g.empty((1, C // G, S, D), torch.bfloat16))
        vh = U.seq2head(v, P, C // G, st, out=g.empty((1, C // G, S, D), torch.bfloat16))
        oh, lh = U.attn_fwd(qh, kh, vh, Hq, Hkv, P, C, st, cu, True,
                            out=g.empty((1, C, S, D), torch.bfloat16), lse=g.empty((1, C, S), torch.float32))
        U.head2seq(oh, o, P, C, st)
        doh = U.seq2head(do, P, C, st, out=g.empty((1, C, S, D), torch.bfloat16))
        ws = g.bytes(U.attn_bwd_workspace_bytes(S, 1, Hq, Hkv, D, P, C, st))
        dqh, dkh, dvh = U.attn_bwd(qh, kh, vh, oh, doh, lh, Hq, Hkv, P, C, st, cu, True, workspace=ws,
                                   dq=g.empty((1, C, S, D), torch.float32),
                                   dk=g.empty((1, C // G, S, D), torch.float32),
                                   dv=g.empty((1, C // G, S, D), torch.float32))
        U.head2seq(dqh, dq, P, C, st)
        U.head2seq(dkh, dk, P, C // G, st)
        U.head2seq(dvh, dv, P, C // G, st)
    U.check()
    g.check()


@pytest.mark.parametrize("S,Hq,Hkv,D,P,C,docs", CASES)
def test_layer_calls_stay_in_bounds(S, Hq, Hkv, D, P, C, docs):
    q, k, v, do = seq_inputs(S, Hq, Hkv, D, "bf16")
    cu = None if docs is None else torch.from_numpy(inputs.cu_seqlens_from_lengths(docs)).cuda()
    g = Guarded()
    ws = g.bytes(U.layer_workspace_bytes(S, 1, Hq, Hkv, D, P, C))
    o, lse = U.layer_fwd(q, k, v, P, C, cu_seqlens=cu, workspace=ws, out=g.empty(q.shape, torch.bfloat16),
                         lse=g.empty((1, Hq, S), torch.float32))
    U.layer_bwd(q, k, v, o, do, lse, P, C, cu_seqlens=cu, workspace=ws,
                dq=g.empty(q.shape, torch.float32), dk=g.empty(k.shape, torch.float32),
                dv=g.empty(v.shape, torch.float32))
    U.check()
    g.check()
    if D == 128:
        # the same layer with the all-to-alls folded into the kernels' addressing
        fo, flse = U.layer_fwd_fused(q, k, v, P, C, cu_seqlens=cu, out=g.empty(q.shape, torch.bfloat16),
                                     lse=g.empty((1, Hq, S), torch.float32))
        fws = g.bytes(U.lib().ulysses_layer_fused_workspace(S, 1, Hq, Hkv, D, P, C, U.BF16))
        U.layer_bwd_fused(q, k, v, fo, do, flse, P, C, cu_seqlens=cu, workspace=fws,
                          dq=g.empty(q.shape, torch.float32), dk=g.empty(k.shape, torch.float32),
                          dv=g.empty(v.shape, torch.float32))
        U.check()
        g.check()
