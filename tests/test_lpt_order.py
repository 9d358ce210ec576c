"""Host check of the decreasing-work key-block selection the attention
backward runs on the device for packed documents.

Every CTA of the backward grid picks its key block by rank: it evaluates the
work of all key blocks (the 64-query tiles that see the block's keys), bisects
on the work value for the least t with fewer than rank + 1 blocks above it,
then takes the block of its rank among those of work t, counting blocks in
chunks of one per thread (512 threads, 8 chunks).  This restates that
procedure in Python and checks that, over all ranks, it is a permutation in
decreasing work with ties in block order (the longest-processing-time order).
The device kernel itself is checked by the GPU parity tests with documents
(every key block's dK/dV compared with the oracle)."""
import numpy as np
import pytest

from long_context_sequence_seq_gb300 import inputs

BN, BMQ, THREADS, PER = 128, 64, 512, 8


def block_work(kb, cu, S, causal):
    k0 = kb * BN
    last = min(k0 + BN, S) - 1

    def qrange(j):
        d = np.searchsorted(cu, j, side="right") - 1
        ds, de = int(cu[d]), int(cu[d + 1])
        lo = j if causal else max(0, min(S, ds))
        hi = max(0, min(S, de))
        return lo, max(hi, lo)

    q_lo, _ = qrange(k0)
    _, q_hi = qrange(last)
    q_lo = (q_lo // BMQ) * BMQ
    return (q_hi - q_lo + BMQ - 1) // BMQ if q_hi > q_lo else 0


def select(rank, work):
    n = len(work)
    hi, lo = max(work), 0

    def above(t):
        return sum(1 for w in work if w > t)

    while lo < hi:
        mid = (lo + hi) >> 1
        if above(mid) <= rank:
            hi = mid
        else:
            lo = mid + 1
    idx = rank - above(lo)
    for i in range(PER):
        chunk = [kb for kb in range(i * THREADS, min((i + 1) * THREADS, n)) if work[kb] == lo]
        if idx < len(chunk):
            return chunk[idx]
        idx -= len(chunk)
    return 0


def cases():
    rng = np.random.default_rng(7)
    out = [(inputs.workload_cu_seqlens(inputs.WORKLOADS["llama31_8b_packed"]).astype(np.int64), True)]
    for _ in range(5):
        S = int(rng.integers(300, 20000))
        nd = int(rng.integers(1, 12))
        cuts = np.sort(rng.choice(np.arange(1, S), size=nd - 1, replace=False)) if nd > 1 else []
        out.append((np.concatenate([[0], cuts, [S]]).astype(np.int64), bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("case", range(6))
def test_selection_is_decreasing_work_permutation(case):
    cu, causal = cases()[case]
    S = int(cu[-1])
    nkb = (S + BN - 1) // BN
    work = [block_work(kb, cu, S, causal) for kb in range(nkb)]
    perm = [select(r, work) for r in range(nkb)]
    assert sorted(perm) == list(range(nkb))
    assert perm == sorted(range(nkb), key=lambda kb: (-work[kb], kb))
