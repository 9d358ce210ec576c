"""Thin ctypes binding over libulysses.so (argument marshalling only).

Every step of the path runs in the library's CUDA kernels; this module only
checks tensor properties, allocates outputs through PyTorch and passes raw
device pointers and the current CUDA stream.  Importing it does not load the
library; the first call does, and fails loudly if the library is missing.

Layouts: sequence layout [B, S, H, D] (P stacked rank chunks of S/P tokens),
head layout [B, n, S, D] (the n heads of one UPipe stage, or all heads).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# ULYSSES_CHECKED=1 loads the bounds-checked build of the same library
LIB_PATH = os.path.join(_PKG, "libulysses_checked.so" if os.environ.get("ULYSSES_CHECKED") == "1"
                        else "libulysses.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_BAD_SEQLENS, ERR_BOUNDS = range(7)
BF16, FP32 = 0, 1
KERNEL_AUTO, KERNEL_SIMT = 0, 1

_lib = None


class RelayoutItem(ctypes.Structure):
    """ulysses_relayout_item: one tensor of a batched re-layout launch."""
    _fields_ = [("src", ctypes.c_void_p), ("dst", ctypes.c_void_p), ("H", ctypes.c_int),
                ("head_chunk", ctypes.c_int), ("stage", ctypes.c_int), ("add", ctypes.c_int)]


class UlyssesError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"ulysses error {code}: {msg}")
        self.code = code


def lib():
    """Load libulysses.so (built by ``build.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "long_context_sequence_seq_gb300.build.build() (checked=True for the "
                           "bounds-checked variant)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.ulysses_seq2head.argtypes = [vp, vp, i64, i32, i32, i32, i32, i32, i32, i32, vp]
    L.ulysses_head2seq.argtypes = [vp, vp, i64, i32, i32, i32, i32, i32, i32, i32, vp]
    L.ulysses_head2seq_add.argtypes = [vp, vp, i64, i32, i32, i32, i32, i32, i32, i32, vp]
    L.ulysses_seq2head_n.argtypes = [ctypes.POINTER(RelayoutItem), i32, i64, i32, i32, i32, i32, vp]
    L.ulysses_head2seq_n.argtypes = [ctypes.POINTER(RelayoutItem), i32, i64, i32, i32, i32, i32, vp]
    L.ulysses_selftest_wait_timeout.argtypes = [i64, vp]
    L.ulysses_ring_workspace.argtypes = [i64, i32, i32, i32, i32, i32]
    L.ulysses_ring_workspace.restype = sz
    L.ulysses_ring_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
    L.ulysses_ring_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, f32, i32,
                                   vp, sz, vp]
    L.ulysses_pad_seq.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, vp]
    L.ulysses_pad_cu_seqlens.argtypes = [vp, i32, vp, i64, i64, vp]
    L.ulysses_lse_merge.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, vp]
    L.ulysses_cast_f32.argtypes = [vp, vp, i64, i32, vp]
    L.ulysses_add_f32.argtypes = [vp, vp, i64, vp]
    L.ulysses_qkv_proj.argtypes = [vp, vp, vp, i64, i32, i32, i32, i32, vp]
    L.ulysses_out_proj.argtypes = [vp, vp, vp, i64, i32, i32, i32, vp]
    L.ulysses_layer_fused_workspace.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32]
    L.ulysses_layer_fused_workspace.restype = ctypes.c_size_t
    L.ulysses_layer_fwd_fused.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, i32, vp, i32,
                                          i32, ctypes.c_float, i32, vp]
    L.ulysses_layer_bwd_fused.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32,
                                          i32, vp, i32, i32, ctypes.c_float, i32, vp, ctypes.c_size_t, vp]
    L.ulysses_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, i32, i32,
                                   vp, i32, i32, f32, i32, vp]
    L.ulysses_attn_bwd_workspace.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32, i32]
    L.ulysses_attn_bwd_workspace.restype = sz
    L.ulysses_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i64, i32, i32,
                                   i32, i32, i32, i32, i32, vp, i32, i32, f32, i32, vp]
    L.ulysses_attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32,
                                           i32, i32, i32, i32, vp, i32, i32, f32, i32, vp]
    L.ulysses_layer_workspace.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32]
    L.ulysses_layer_workspace.restype = sz
    L.ulysses_layer_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, i32, vp,
                                    i32, i32, f32, i32, vp, sz, vp]
    L.ulysses_layer_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32,
                                    i32, i32, vp, i32, i32, f32, i32, vp, sz, vp]
    L.ulysses_check.argtypes = [vp]
    L.ulysses_last_error.restype = ctypes.c_char_p
    L.ulysses_set_kernel.argtypes = [i32]
    L.ulysses_launch_count.restype = ctypes.c_longlong
    L.ulysses_checked_build.restype = ctypes.c_int
    _lib = L
    return L


def _ck(rc):
    if rc != OK:
        raise UlyssesError(rc, lib().ulysses_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cu(cu_seqlens):
    if cu_seqlens is None:
        return None, 0
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    return _p(cu_seqlens), cu_seqlens.numel() - 1


def _stage(stage):
    return -1 if stage is None else int(stage)


# --------------------------------------------------------------- re-layout

def seq2head(x_seq, P, head_chunk=None, stage=None, out=None, stream=None):
    """All-to-all #1: [B,S,H,D] -> [B,n,S,D] for the stage (all heads if None).
    With H < P (kv-head replication) `stage` names a rank and n = 1."""
    B, S, H, D = x_seq.shape
    n = H if stage is None else (1 if H < P else head_chunk)
    if out is None:
        out = torch.empty((B, n, S, D), dtype=x_seq.dtype, device=x_seq.device)
    _ck(lib().ulysses_seq2head(_p(x_seq), _p(out), S, B, H, D, P, head_chunk or 0,
                               _stage(stage), _dtype_code(x_seq), _stream(stream)))
    return out


def head2seq(x_head, x_seq, P, head_chunk=None, stage=None, stream=None):
    """All-to-all #2: write [B,n,S,D] into the stage's heads of [B,S,H,D]."""
    B, S, H, D = x_seq.shape
    if x_head.dtype != x_seq.dtype:
        raise TypeError("dtype mismatch")
    _ck(lib().ulysses_head2seq(_p(x_head), _p(x_seq), S, B, H, D, P, head_chunk or 0,
                               _stage(stage), _dtype_code(x_seq), _stream(stream)))
    return x_seq


def head2seq_add(x_head, x_seq, P, head_chunk=None, stage=None, stream=None):
    """As head2seq, adding into the fp32 sequence tensor (partial gradients of a
    replicated kv head)."""
    B, S, H, D = x_seq.shape
    if x_head.dtype != x_seq.dtype:
        raise TypeError("dtype mismatch")
    _ck(lib().ulysses_head2seq_add(_p(x_head), _p(x_seq), S, B, H, D, P, head_chunk or 0,
                                   _stage(stage), _dtype_code(x_seq), _stream(stream)))
    return x_seq


def _relayout_n(fn, pairs, P, stream, head_seq_index):
    """pairs: (src, dst, head_chunk, stage[, add]) per tensor; the sequence-
    layout tensor of each pair gives S, B, H, D (head_seq_index picks it)."""
    if not pairs:
        return
    items = (RelayoutItem * len(pairs))()
    seq0 = pairs[0][head_seq_index]
    B, S, _, D = seq0.shape
    dt = _dtype_code(seq0)
    for i, pr in enumerate(pairs):
        src, dst, C, stage = pr[:4]
        add = pr[4] if len(pr) > 4 else 0
        seq = pr[head_seq_index]
        if _dtype_code(src) != dt or _dtype_code(dst) != dt:
            raise TypeError("every tensor of a batched re-layout has the same dtype")
        items[i] = RelayoutItem(_p(src).value, _p(dst).value, seq.shape[2], C or 0, _stage(stage), int(add))
    _ck(fn(items, len(pairs), S, B, D, P, dt, _stream(stream)))


def seq2head_n(pairs, P, stream=None):
    """Batched all-to-all #1, one launch: pairs of (x_seq [B,S,H,D], x_head
    [B,n,S,D] out, head_chunk, stage) sharing S, B, D and dtype."""
    _relayout_n(lib().ulysses_seq2head_n, pairs, P, stream, 0)


def head2seq_n(pairs, P, stream=None):
    """Batched all-to-all #2, one launch: (x_head, x_seq, head_chunk, stage[,
    add]) per tensor; add (fp32 only) accumulates into x_seq."""
    _relayout_n(lib().ulysses_head2seq_n, pairs, P, stream, 1)


def padded_length(S, P):
    """S rounded up to a multiple of P."""
    return (S + P - 1) // P * P


def pad_to_multiple(tensors, P, cu_seqlens=None, stream=None):
    """Pad [B,S,H,D] device tensors along S to a multiple of P (as
    pad_to_multiple_of does for sequence parallelism) with the library's pad
    kernels.  Returns (padded tensors, cu_seqlens, S): the padding positions
    form a document of their own, so no real position attends to them or is
    attended by them (S stays the caller's length for slicing the results
    back).  cu_seqlens (int32, device) describes the real documents, or None
    for one document; it is needed with B == 1 only."""
    S = tensors[0].shape[1]
    S_pad = padded_length(S, P)
    if S_pad == S:
        return list(tensors), cu_seqlens, S
    out = []
    for t in tensors:
        B, _, H, D = t.shape
        p = torch.empty((B, S_pad, H, D), dtype=t.dtype, device=t.device)
        _ck(lib().ulysses_pad_seq(_p(t), _p(p), S, S_pad, B, H, D, _dtype_code(t), _stream(stream)))
        out.append(p)
    nd = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    cu = torch.empty(nd + 2, dtype=torch.int32, device=tensors[0].device)
    cp, _ = _cu(cu_seqlens)
    _ck(lib().ulysses_pad_cu_seqlens(cp, nd, _p(cu), S, S_pad, _stream(stream)))
    return out, cu, S


# --------------------------------------------------------------- attention

def attn_fwd(q_h, k_h, v_h, H_q, H_kv, P, head_chunk=None, stage=None, cu_seqlens=None,
             causal=True, scale=None, out=None, lse=None, stream=None):
    """Local attention on head-layout buffers: returns (O [B,n,S,D], LSE [B,n,S])."""
    B, n, S, D = q_h.shape
    if out is None:
        out = torch.empty_like(q_h)
    if lse is None:
        lse = torch.empty((B, n, S), dtype=torch.float32, device=q_h.device)
    cp, nd = _cu(cu_seqlens)
    _ck(lib().ulysses_attn_fwd(_p(q_h), _p(k_h), _p(v_h), _p(out), _p(lse), S, B, H_q, H_kv, D, P,
                               head_chunk or 0, _stage(stage), cp, nd, int(bool(causal)),
                               float(scale or 0.0), _dtype_code(q_h), _stream(stream)))
    return out, lse


def attn_bwd_workspace_bytes(S, B, H_q, H_kv, D, P, head_chunk=None, stage=None, dtype=BF16):
    return lib().ulysses_attn_bwd_workspace(S, B, H_q, H_kv, D, P, head_chunk or 0,
                                            _stage(stage), dtype)


def attn_bwd(q_h, k_h, v_h, o_h, do_h, lse, H_q, H_kv, P, head_chunk=None, stage=None,
             cu_seqlens=None, causal=True, scale=None, workspace=None, dq=None, dk=None, dv=None,
             stream=None):
    """Backward on head-layout buffers: returns fp32 (dQ, dK, dV)."""
    B, n, S, D = q_h.shape
    dev = q_h.device
    dq = torch.empty(q_h.shape, dtype=torch.float32, device=dev) if dq is None else dq
    dk = torch.empty(k_h.shape, dtype=torch.float32, device=dev) if dk is None else dk
    dv = torch.empty(v_h.shape, dtype=torch.float32, device=dev) if dv is None else dv
    ws_b = attn_bwd_workspace_bytes(S, B, H_q, H_kv, D, P, head_chunk, stage, _dtype_code(q_h))
    if workspace is None:
        workspace = torch.empty(max(ws_b, 256), dtype=torch.uint8, device=dev)
    cp, nd = _cu(cu_seqlens)
    _ck(lib().ulysses_attn_bwd(_p(q_h), _p(k_h), _p(v_h), _p(o_h), _p(do_h), _p(lse), _p(dq),
                               _p(dk), _p(dv), _p(workspace), workspace.numel(), S, B, H_q, H_kv,
                               D, P, head_chunk or 0, _stage(stage), cp, nd, int(bool(causal)),
                               float(scale or 0.0), _dtype_code(q_h), _stream(stream)))
    return dq, dk, dv


def attn_bwd_noalloc(q_h, k_h, v_h, o_h, do_h, lse, H_q, H_kv, P, head_chunk=None, stage=None,
                     cu_seqlens=None, causal=True, scale=None, dq=None, dk=None, dv=None,
                     stream=None):
    """attn_bwd through the entry point that needs no workspace (the library's
    built-in scratch holds D_i; see include/ulysses.h for its limit and the
    rule that calls sharing it must not overlap on the GPU)."""
    B, n, S, D = q_h.shape
    dev = q_h.device
    dq = torch.empty(q_h.shape, dtype=torch.float32, device=dev) if dq is None else dq
    dk = torch.empty(k_h.shape, dtype=torch.float32, device=dev) if dk is None else dk
    dv = torch.empty(v_h.shape, dtype=torch.float32, device=dev) if dv is None else dv
    cp, nd = _cu(cu_seqlens)
    _ck(lib().ulysses_attn_bwd_noalloc(_p(q_h), _p(k_h), _p(v_h), _p(o_h), _p(do_h), _p(lse),
                                       _p(dq), _p(dk), _p(dv), S, B, H_q, H_kv, D, P,
                                       head_chunk or 0, _stage(stage), cp, nd, int(bool(causal)),
                                       float(scale or 0.0), _dtype_code(q_h), _stream(stream)))
    return dq, dk, dv


# --------------------------------------------------------------- whole layer

def layer_workspace_bytes(S, B, H_q, H_kv, D, P, head_chunk, dtype=BF16):
    return lib().ulysses_layer_workspace(S, B, H_q, H_kv, D, P, head_chunk, dtype)


def layer_workspace(S, B, H_q, H_kv, D, P, head_chunk, dtype=BF16, device="cuda"):
    n = layer_workspace_bytes(S, B, H_q, H_kv, D, P, head_chunk, dtype)
    if n == 0:
        raise UlyssesError(ERR_INVALID, "invalid layer shape")
    return torch.empty(n, dtype=torch.uint8, device=device)


def layer_fwd(q_seq, k_seq, v_seq, P, head_chunk, cu_seqlens=None, causal=True, scale=None,
              workspace=None, out=None, lse=None, stream=None):
    """Steps 3-5 with the UPipe stage loop: returns (O [B,S,H_q,D], LSE [B,H_q,S])."""
    B, S, H_q, D = q_seq.shape
    H_kv = k_seq.shape[2]
    dt = _dtype_code(q_seq)
    if workspace is None:
        workspace = layer_workspace(S, B, H_q, H_kv, D, P, head_chunk, dt, q_seq.device)
    out = torch.empty_like(q_seq) if out is None else out
    lse = torch.empty((B, H_q, S), dtype=torch.float32, device=q_seq.device) if lse is None else lse
    cp, nd = _cu(cu_seqlens)
    _ck(lib().ulysses_layer_fwd(_p(q_seq), _p(k_seq), _p(v_seq), _p(out), _p(lse), S, B, H_q, H_kv,
                                D, P, head_chunk, cp, nd, int(bool(causal)), float(scale or 0.0),
                                dt, _p(workspace), workspace.numel(), _stream(stream)))
    return out, lse


def layer_bwd(q_seq, k_seq, v_seq, o_seq, do_seq, lse, P, head_chunk, cu_seqlens=None,
              causal=True, scale=None, workspace=None, dq=None, dk=None, dv=None, stream=None):
    """Backward of the layer: returns fp32 (dQ, dK, dV) in sequence layout."""
    B, S, H_q, D = q_seq.shape
    H_kv = k_seq.shape[2]
    dt = _dtype_code(q_seq)
    dev = q_seq.device
    if workspace is None:
        workspace = layer_workspace(S, B, H_q, H_kv, D, P, head_chunk, dt, dev)
    dq = torch.empty(q_seq.shape, dtype=torch.float32, device=dev) if dq is None else dq
    dk = torch.empty(k_seq.shape, dtype=torch.float32, device=dev) if dk is None else dk
    dv = torch.empty(v_seq.shape, dtype=torch.float32, device=dev) if dv is None else dv
    cp, nd = _cu(cu_seqlens)
    _ck(lib().ulysses_layer_bwd(_p(q_seq), _p(k_seq), _p(v_seq), _p(o_seq), _p(do_seq), _p(lse),
                                _p(dq), _p(dk), _p(dv), S, B, H_q, H_kv, D, P, head_chunk, cp, nd,
                                int(bool(causal)), float(scale or 0.0), dt, _p(workspace),
                                workspace.numel(), _stream(stream)))
    return dq, dk, dv


# --------------------------------------------------------------- diagnostics

def check(stream=None):
    """Synchronise and raise if a kernel flagged a timeout or bad cu_seqlens."""
    _ck(lib().ulysses_check(_stream(stream)))


def set_kernel(which: int):
    _ck(lib().ulysses_set_kernel(which))


def launch_count() -> int:
    return int(lib().ulysses_launch_count())


def selftest_wait_timeout(limit_ns=50_000_000, stream=None):
    """Launch the bounded-wait self-test (a wait nothing completes); the next
    check() raises UlyssesError with code ERR_TIMEOUT."""
    _ck(lib().ulysses_selftest_wait_timeout(int(limit_ns), _stream(stream)))


# --------------------------------------------------------------- ring variant

def ring_workspace(S, H_q, H_kv, D, P, dtype=BF16, device="cuda"):
    n = lib().ulysses_ring_workspace(S, H_q, H_kv, D, P, dtype)
    if n == 0:
        raise UlyssesError(ERR_INVALID, "invalid ring shape")
    return torch.empty(n, dtype=torch.uint8, device=device)


def ring_attention_fwd(q_seq, k_seq, v_seq, P, causal=True, scale=None, workspace=None, stream=None):
    """Ring-attention variant of the same layer (the scheme the pages compare
    Ulysses with), on P virtual ranks, run by the library's ring driver: rank
    r keeps query chunk r and meets KV chunk (r - t) mod P at ring step t;
    steps wholly in the future are skipped under the causal mask, the
    diagonal step is causal and the others are full; the steps' (O, LSE) are
    merged with their log-sum-exp weights.  Returns (O [1,S,H_q,D], LSE
    chunks [P,H_q,L])."""
    B, S, Hq, D = q_seq.shape
    Hkv = k_seq.shape[2]
    if B != 1 or S % P:
        raise ValueError("ring variant: B == 1 and S divisible by P")
    dt = _dtype_code(q_seq)
    if workspace is None:
        workspace = ring_workspace(S, Hq, Hkv, D, P, dt, q_seq.device)
    out = torch.empty_like(q_seq)
    lse = torch.empty((P, Hq, S // P), dtype=torch.float32, device=q_seq.device)
    _ck(lib().ulysses_ring_fwd(_p(q_seq), _p(k_seq), _p(v_seq), _p(out), _p(lse), S, Hq, Hkv, D, P,
                               int(bool(causal)), float(scale or 0.0), dt, _p(workspace), workspace.numel(),
                               _stream(stream)))
    return out, lse


def ring_attention_bwd(q_seq, k_seq, v_seq, o_seq, do_seq, lse, P, causal=True, scale=None, workspace=None,
                       stream=None):
    """Backward of ring_attention_fwd (library ring driver): every (query
    chunk, KV chunk) step runs the attention backward with the merged LSE and
    O, and the steps' partial dQ, dK, dV are summed.  Returns fp32 (dQ, dK,
    dV) in sequence layout."""
    B, S, Hq, D = q_seq.shape
    Hkv = k_seq.shape[2]
    if B != 1 or S % P:
        raise ValueError("ring variant: B == 1 and S divisible by P")
    dt = _dtype_code(q_seq)
    dev = q_seq.device
    if workspace is None:
        workspace = ring_workspace(S, Hq, Hkv, D, P, dt, dev)
    dq = torch.empty(q_seq.shape, dtype=torch.float32, device=dev)
    dk = torch.empty(k_seq.shape, dtype=torch.float32, device=dev)
    dv = torch.empty(v_seq.shape, dtype=torch.float32, device=dev)
    _ck(lib().ulysses_ring_bwd(_p(q_seq), _p(k_seq), _p(v_seq), _p(o_seq), _p(do_seq), _p(lse), _p(dq), _p(dk),
                               _p(dv), S, Hq, Hkv, D, P, int(bool(causal)), float(scale or 0.0), dt,
                               _p(workspace), workspace.numel(), _stream(stream)))
    return dq, dk, dv


# --------------------------------------------------------------- projections

def qkv_proj(x, w_qkv, H_q, H_kv, out=None, stream=None):
    """[Q|K|V] = X W_qkv^T written straight into head layout: x [S,hidden]
    bf16, w_qkv [(H_q+2H_kv) D, hidden] bf16 -> [H_q+2H_kv, S, D] bf16."""
    S, hidden = x.shape
    nf = w_qkv.shape[0]
    D = nf // (H_q + 2 * H_kv)
    if out is None:
        out = torch.empty((H_q + 2 * H_kv, S, D), dtype=torch.bfloat16, device=x.device)
    _ck(lib().ulysses_qkv_proj(_p(x), _p(w_qkv), _p(out), S, hidden, H_q, H_kv, D, _stream(stream)))
    return out


def out_proj(o_head, w_o, out=None, stream=None):
    """Y = O W_o^T with O read from head layout: o_head [H_q, S, D] bf16,
    w_o [hidden, H_q D] bf16 -> [S, hidden] bf16."""
    H_q, S, D = o_head.shape
    hidden = w_o.shape[0]
    if out is None:
        out = torch.empty((S, hidden), dtype=torch.bfloat16, device=o_head.device)
    _ck(lib().ulysses_out_proj(_p(o_head), _p(w_o), _p(out), S, H_q, D, hidden, _stream(stream)))
    return out


# --------------------------------------------------------------- fused layer

def layer_fwd_fused(q_seq, k_seq, v_seq, P, head_chunk, cu_seqlens=None, causal=True, scale=None,
                    out=None, lse=None, stream=None):
    """layer_fwd with the all-to-alls folded into the kernels' addressing (no
    head-layout copies): returns (O [1,S,H_q,D], LSE [1,H_q,S])."""
    B, S, H_q, D = q_seq.shape
    H_kv = k_seq.shape[2]
    out = torch.empty_like(q_seq) if out is None else out
    lse = torch.empty((B, H_q, S), dtype=torch.float32, device=q_seq.device) if lse is None else lse
    cp, nd = _cu(cu_seqlens)
    _ck(lib().ulysses_layer_fwd_fused(_p(q_seq), _p(k_seq), _p(v_seq), _p(out), _p(lse), S, B, H_q, H_kv, D, P,
                                      head_chunk, cp, nd, int(bool(causal)), float(scale or 0.0),
                                      _dtype_code(q_seq), _stream(stream)))
    return out, lse


def layer_bwd_fused(q_seq, k_seq, v_seq, o_seq, do_seq, lse, P, head_chunk, cu_seqlens=None, causal=True,
                    scale=None, workspace=None, dq=None, dk=None, dv=None, stream=None):
    """layer_bwd with the all-to-alls folded into the kernels' addressing:
    returns fp32 (dQ, dK, dV) in sequence layout."""
    B, S, H_q, D = q_seq.shape
    H_kv = k_seq.shape[2]
    dt = _dtype_code(q_seq)
    dev = q_seq.device
    if workspace is None:
        nb = lib().ulysses_layer_fused_workspace(S, B, H_q, H_kv, D, P, head_chunk, dt)
        workspace = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
    dq = torch.empty(q_seq.shape, dtype=torch.float32, device=dev) if dq is None else dq
    dk = torch.empty(k_seq.shape, dtype=torch.float32, device=dev) if dk is None else dk
    dv = torch.empty(v_seq.shape, dtype=torch.float32, device=dev) if dv is None else dv
    cp, nd = _cu(cu_seqlens)
    _ck(lib().ulysses_layer_bwd_fused(_p(q_seq), _p(k_seq), _p(v_seq), _p(o_seq), _p(do_seq), _p(lse), _p(dq),
                                      _p(dk), _p(dv), S, B, H_q, H_kv, D, P, head_chunk, cp, nd,
                                      int(bool(causal)), float(scale or 0.0), dt, _p(workspace),
                                      workspace.numel(), _stream(stream)))
    return dq, dk, dv
