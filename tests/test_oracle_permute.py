"""Pins for the oracle's dispatch permutation and counts (Stage 4 AllGather
row: sort tokens by expert and return expert token counts; Stage 6: counts
accumulated into moe_load).

Counts are pinned by numpy's bincount; the permutation by its invariants:
bijection, stability, segment membership and permute-then-unpermute
identity.
"""
import numpy as np
import pytest

import oracle


def _check(ids, P):
    T, k = ids.shape
    N = T * k
    counts, offsets, r2t, f2r = oracle.permute(ids, P)
    flat = ids.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat, minlength=P).astype(np.int32))
    assert offsets[0] == 0 and offsets[P] == N and np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(f2r), np.arange(N))                 # bijection
    assert np.array_equal(r2t[f2r], np.arange(N) // k)
    for p in range(P):
        seg = np.nonzero(flat == p)[0]                                   # ascending f
        rows = f2r[seg]
        assert np.array_equal(rows, np.arange(offsets[p], offsets[p + 1]))  # stable
    # permute then unpermute is the identity on row payloads
    x = np.arange(T * 3, dtype=np.int64).reshape(T, 3) * 7 + 1
    x_perm = x[r2t]
    back = x_perm[f2r].reshape(T, k, 3)
    assert np.array_equal(back, np.broadcast_to(x[:, None, :], (T, k, 3)))
    return counts, offsets, r2t, f2r


@pytest.mark.parametrize("T,k,P", [(64, 2, 8), (100, 8, 32), (1, 8, 40), (333, 4, 7)])
def test_permutation_invariants(T, k, P, rng):
    ids = np.stack([rng.permutation(P)[:k] for _ in range(T)]).astype(np.int32)
    _check(ids, P)


def test_degenerate_placements(rng):
    T, k, P = 50, 4, 16
    # every token on the same four experts; twelve experts empty
    ids = np.tile(np.array([3, 0, 9, 15], np.int32), (T, 1))
    counts, offsets, _, _ = _check(ids, P)
    assert counts[3] == T and counts[1] == 0
    # empty input
    counts, offsets, r2t, f2r = oracle.permute(np.zeros((0, k), np.int32), P)
    assert counts.sum() == 0 and offsets[P] == 0 and r2t.size == 0 and f2r.size == 0


def test_counts_accumulate_like_moe_load(rng):
    P = 12
    a = rng.integers(0, P, (30, 3)).astype(np.int32)
    b = rng.integers(0, P, (17, 3)).astype(np.int32)
    load = oracle.expert_counts(a, P)
    load = oracle.expert_counts(b, P, counts=load)
    assert np.array_equal(load, np.bincount(np.concatenate([a.ravel(), b.ravel()]),
                                            minlength=P).astype(np.int32))
