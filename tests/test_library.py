"""Host-side checks of the C ABI library (no GPU needed): it builds, loads,
exports every symbol include/ulysses.h declares, and rejects invalid shapes
before touching the device."""
import ctypes
import os
import re

import pytest

from long_context_sequence_seq_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libpath():
    return B.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "ulysses.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ulysses_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_binding_loads(libpath):
    from long_context_sequence_seq_gb300 import ulysses
    L = ulysses.lib()
    assert L.ulysses_launch_count() >= 0


def test_host_validation_without_device(libpath):
    from long_context_sequence_seq_gb300 import ulysses as U
    L = U.lib()
    dummy = ctypes.c_void_p(256)
    # S % P != 0
    assert L.ulysses_seq2head(dummy, ctypes.c_void_p(1 << 20), 30, 1, 8, 128, 4, 2, 0, U.BF16, None) == U.ERR_INVALID
    # heads not divisible by P (num_heads >= sp_size and divisible)
    assert L.ulysses_seq2head(dummy, ctypes.c_void_p(1 << 20), 32, 1, 6, 128, 4, 1, 0, U.BF16, None) == U.ERR_INVALID
    # head_chunk not dividing H/P
    assert L.ulysses_seq2head(dummy, ctypes.c_void_p(1 << 20), 32, 1, 8, 128, 2, 3, 0, U.BF16, None) == U.ERR_INVALID
    # stage out of range
    assert L.ulysses_seq2head(dummy, ctypes.c_void_p(1 << 20), 32, 1, 8, 128, 2, 2, 4, U.BF16, None) == U.ERR_INVALID
    # in place
    assert L.ulysses_seq2head(dummy, dummy, 32, 1, 8, 128, 2, 2, 0, U.BF16, None) == U.ERR_INVALID
    # unaligned
    assert L.ulysses_seq2head(ctypes.c_void_p(264), ctypes.c_void_p(1 << 20), 32, 1, 8, 128, 2, 2, 0, U.BF16, None) == U.ERR_INVALID
    args = [dummy] * 5
    # attention: C % G != 0 (a stage must own whole kv heads)
    rc = L.ulysses_attn_fwd(*args, 64, 1, 32, 8, 128, 4, 2, 0, None, 0, 1, 0.0, U.BF16, None)
    assert rc == U.ERR_INVALID
    # D unsupported
    rc = L.ulysses_attn_fwd(*args, 64, 1, 32, 8, 96, 4, 8, 0, None, 0, 1, 0.0, U.BF16, None)
    assert rc == U.ERR_UNSUPPORTED
    # cu_seqlens with B > 1
    rc = L.ulysses_attn_fwd(*args, 64, 2, 32, 8, 128, 4, 8, 0, dummy, 1, 1, 0.0, U.BF16, None)
    assert rc == U.ERR_UNSUPPORTED
    # H_q not multiple of H_kv
    rc = L.ulysses_attn_fwd(*args, 64, 1, 12, 8, 128, 4, 3, 0, None, 0, 1, 0.0, U.BF16, None)
    assert rc == U.ERR_INVALID
    assert b"kv" in L.ulysses_last_error() or len(L.ulysses_last_error()) > 0
    # empty input is a no-op, never a launch
    before = L.ulysses_launch_count()
    assert L.ulysses_seq2head(dummy, ctypes.c_void_p(1 << 20), 0, 1, 8, 128, 2, 2, 0, U.BF16, None) == U.OK
    assert L.ulysses_attn_fwd(*args, 0, 1, 32, 8, 128, 4, 8, 0, None, 0, 1, 0.0, U.BF16, None) == U.OK
    assert L.ulysses_launch_count() == before


def test_workspace_sizes(libpath):
    from long_context_sequence_seq_gb300 import ulysses as U
    S = 65536
    ws = U.attn_bwd_workspace_bytes(S, 1, 32, 8, 128, 4, 8, 0)
    assert ws == 8 * S * 4
    lw = U.layer_workspace_bytes(S, 1, 32, 8, 128, 4, 8)
    # per stage: q,o,dO (bf16) + k,v (bf16) + dq (fp32) + dk,dv (fp32) + delta
    want = 3 * 8 * S * 128 * 2 + 2 * 2 * S * 128 * 2 + 8 * S * 128 * 4 + 2 * 2 * S * 128 * 4 + 8 * S * 4
    assert lw == want
    assert U.layer_workspace_bytes(S, 1, 32, 8, 128, 4, 3) == 0


def test_kv_replication_validation(libpath):
    """H_kv < P is accepted when H_kv divides P (rank r holds kv head
    r / (P / H_kv)); other head counts are rejected before any launch."""
    from long_context_sequence_seq_gb300 import ulysses as U
    L = U.lib()
    S = 4096
    assert U.layer_workspace_bytes(S, 1, 8, 2, 128, 4, 2) > 0      # H_kv = 2 < P = 4
    assert U.layer_workspace_bytes(S, 1, 8, 1, 128, 8, 1) > 0      # H_kv = 1, P = 8
    assert U.layer_workspace_bytes(S, 1, 12, 3, 128, 4, 3) == 0    # P % H_kv != 0
    dummy = ctypes.c_void_p(256)
    # the rank must be named: stage -1 and stage >= P are rejected
    assert L.ulysses_seq2head(dummy, ctypes.c_void_p(1 << 20), 32, 1, 2, 128, 4, 0, -1, U.BF16, None) == U.ERR_INVALID
    assert L.ulysses_seq2head(dummy, ctypes.c_void_p(1 << 20), 32, 1, 2, 128, 4, 0, 4, U.BF16, None) == U.ERR_INVALID
    # accumulating scatter: fp32 only
    assert L.ulysses_head2seq_add(dummy, ctypes.c_void_p(1 << 20), 32, 1, 2, 128, 4, 0, 1, U.BF16, None) == U.ERR_UNSUPPORTED


def test_pad_to_multiple_host():
    """Padding to a multiple of P puts the pad positions in a document of
    their own (host logic, CPU tensors)."""
    import torch
    from long_context_sequence_seq_gb300 import ulysses as U
    x = torch.arange(2 * 10 * 3 * 2, dtype=torch.float32).reshape(2, 10, 3, 2)
    (p,), cu, S = U.pad_to_multiple([x], 4)
    assert S == 10 and p.shape == (2, 12, 3, 2)
    assert torch.equal(p[:, :10], x) and torch.count_nonzero(p[:, 10:]) == 0
    assert cu.tolist() == [0, 10, 12]
    (q,), cu2, _ = U.pad_to_multiple([x[:1]], 4, torch.tensor([0, 4, 10], dtype=torch.int32))
    assert cu2.tolist() == [0, 4, 10, 12]
    (r,), cu3, _ = U.pad_to_multiple([x[:, :8]], 4)
    assert r.shape[1] == 8 and cu3 is None


def test_selftest_wait_rejects_bad_limits(libpath):
    from long_context_sequence_seq_gb300 import ulysses as U
    L = U.lib()
    assert L.ulysses_selftest_wait_timeout(0, None) == U.ERR_INVALID
    assert L.ulysses_selftest_wait_timeout(3_000_000_000, None) == U.ERR_INVALID


def test_projection_validation(libpath):
    from long_context_sequence_seq_gb300 import ulysses as U
    L = U.lib()
    d = ctypes.c_void_p(256)
    # hidden not a multiple of 64 / features not a multiple of 256 / D unsupported
    assert L.ulysses_qkv_proj(d, d, d, 128, 100, 4, 2, 128, None) == U.ERR_UNSUPPORTED
    assert L.ulysses_qkv_proj(d, d, d, 128, 256, 3, 1, 64, None) == U.ERR_UNSUPPORTED
    assert L.ulysses_qkv_proj(d, d, d, 128, 256, 4, 2, 96, None) == U.ERR_UNSUPPORTED
    assert L.ulysses_out_proj(d, d, d, 128, 4, 128, 300, None) == U.ERR_UNSUPPORTED
    # empty input: a no-op
    assert L.ulysses_out_proj(d, d, d, 0, 4, 128, 256, None) == U.OK


def test_fused_layer_validation(libpath):
    from long_context_sequence_seq_gb300 import ulysses as U
    L = U.lib()
    d = ctypes.c_void_p(256)
    args = [d] * 5
    # B > 1, fp32 and kv-head replication are outside the fused layer
    assert L.ulysses_layer_fwd_fused(*args, 256, 2, 8, 8, 128, 2, 4, None, 0, 1, 0.0, U.BF16, None) == U.ERR_UNSUPPORTED
    assert L.ulysses_layer_fwd_fused(*args, 256, 1, 8, 8, 128, 2, 4, None, 0, 1, 0.0, U.FP32, None) == U.ERR_UNSUPPORTED
    assert L.ulysses_layer_fwd_fused(*args, 256, 1, 8, 2, 128, 4, 2, None, 0, 1, 0.0, U.BF16, None) == U.ERR_UNSUPPORTED
    assert U.lib().ulysses_layer_fused_workspace(4096, 1, 32, 8, 128, 4, 8, U.BF16) == 8 * 4096 * 4
