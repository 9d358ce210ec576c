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


def test_pad_and_ring_validation(libpath):
    """Padding and the ring driver reject bad shapes on the host."""
    from long_context_sequence_seq_gb300 import ulysses as U
    L = U.lib()
    d = ctypes.c_void_p(1 << 20)
    e = ctypes.c_void_p(1 << 24)
    assert U.padded_length(10, 4) == 12 and U.padded_length(12, 4) == 12 and U.padded_length(0, 4) == 0
    # S_pad < S, rows not a multiple of 16 bytes, in place
    assert L.ulysses_pad_seq(d, e, 10, 8, 1, 4, 128, U.BF16, None) == U.ERR_INVALID
    assert L.ulysses_pad_seq(d, e, 10, 12, 1, 1, 4, U.BF16, None) == U.ERR_UNSUPPORTED
    assert L.ulysses_pad_seq(d, ctypes.c_void_p((1 << 20) + 256), 10, 12, 1, 4, 128, U.BF16, None) == U.ERR_INVALID
    assert L.ulysses_pad_seq(d, e, 0, 0, 1, 4, 128, U.BF16, None) == U.OK
    assert L.ulysses_pad_cu_seqlens(d, 0, e, 10, 12, None) == U.ERR_INVALID
    assert L.ulysses_pad_cu_seqlens(None, 0, e, 10, 8, None) == U.ERR_INVALID
    # ring: S % P, workspace size, empty input
    assert L.ulysses_ring_workspace(1000, 4, 2, 128, 3, U.BF16) == 0
    n = L.ulysses_ring_workspace(1024, 4, 2, 128, 4, U.BF16)
    assert n > 0
    args = [d] * 5
    assert L.ulysses_ring_fwd(*args, 1000, 4, 2, 128, 3, 1, 0.0, U.BF16, d, n, None) == U.ERR_INVALID
    assert L.ulysses_ring_fwd(*args, 1024, 4, 2, 128, 4, 1, 0.0, U.BF16, d, n - 256, None) == U.ERR_INVALID
    assert L.ulysses_ring_fwd(*args, 0, 4, 2, 128, 4, 1, 0.0, U.BF16, d, n, None) == U.OK


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


def test_batched_relayout_validation(libpath):
    """ulysses_seq2head_n / head2seq_n reject bad batches on the host."""
    from long_context_sequence_seq_gb300 import ulysses as U
    L = U.lib()
    It = U.RelayoutItem
    a, b, c, d = (1 << 24), (2 << 24), (3 << 24), (4 << 24)   # 16 MiB apart, aligned
    # S=32, B=1, D=128, P=2: Q-like (H=8, chunk 2) and K-like (H=4, chunk 1) items
    ok = (It * 2)(It(a, b, 8, 2, 0, 0), It(c, d, 4, 1, 0, 0))
    arr = lambda *xs: (It * len(xs))(*xs)  # noqa: E731
    # too many items
    many = (It * 7)(*([It(a, b, 8, 2, 0, 0)] * 7))
    assert L.ulysses_seq2head_n(many, 7, 32, 1, 128, 2, U.BF16, None) == U.ERR_INVALID
    # an item's destination overlapping another item's source
    bad = arr(It(a, b, 8, 2, 0, 0), It(b + 256, d, 4, 1, 0, 0))
    assert L.ulysses_seq2head_n(bad, 2, 32, 1, 128, 2, U.BF16, None) == U.ERR_INVALID
    assert b"overlaps source" in L.ulysses_last_error()
    # accumulation is a scatter-only, fp32-only option
    add = arr(It(a, b, 8, 2, 0, 1))
    assert L.ulysses_seq2head_n(add, 1, 32, 1, 128, 2, U.FP32, None) == U.ERR_UNSUPPORTED
    assert L.ulysses_head2seq_n(add, 1, 32, 1, 128, 2, U.BF16, None) == U.ERR_UNSUPPORTED
    # per-item shape rules still apply (chunk 3 does not divide 8/2 heads)
    assert L.ulysses_seq2head_n(arr(It(a, b, 8, 3, 0, 0)), 1, 32, 1, 128, 2, U.BF16, None) == U.ERR_INVALID
    # empty input and an empty batch are no-ops
    assert L.ulysses_seq2head_n(ok, 2, 0, 1, 128, 2, U.BF16, None) == U.OK
    assert L.ulysses_head2seq_n(ok, 0, 32, 1, 128, 2, U.BF16, None) == U.OK


def test_checked_variant_builds_and_loads():
    """The bounds-checked library exports the same symbols and says so."""
    import subprocess
    import sys
    path = B.build(checked=True)
    lib = ctypes.CDLL(path)
    for n in _declared():
        assert hasattr(lib, n), n
    assert lib.ulysses_checked_build() == 1
    assert ctypes.CDLL(B.build()).ulysses_checked_build() == 0
    # ULYSSES_CHECKED=1 makes the binding load it (in a fresh process)
    code = ("from long_context_sequence_seq_gb300 import ulysses as U; "
            "print(U.lib().ulysses_checked_build(), U.LIB_PATH.endswith('libulysses_checked.so'))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env={**os.environ, "ULYSSES_CHECKED": "1"},
                         capture_output=True, text=True, check=True).stdout.split()
    assert out == ["1", "True"]
