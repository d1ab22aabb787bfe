"""Pins of the oracle's candidate-pool top-k (CPU only).

vllm PR 60834 "Purpose": the MXFP4 indexer has a dense path (the scorer called with no
candidate blocks) and a candidate-pool path for V4.1's two-level indexer. Reading R17 at
orc_topk_cand: a candidate block is one page of P keys; a query ranks only the visible keys
of its candidate blocks. The pins fix the oracle to that reading with brute force written
here in numpy, to the dense top-k when every block is a candidate, and to the special cases.
"""
import numpy as np
import pytest

import oracle as O


def _brute(logits, vis, cand, n_cand, P, k):
    out = np.full((logits.shape[0], k), -1, np.int32)
    for r in range(logits.shape[0]):
        blocks = set(int(b) for b in cand[r, :n_cand[r]])
        keys = [s for s in range(int(vis[r])) if s // P in blocks]
        keys.sort(key=lambda s: (-logits[r, s], s))
        out[r, :min(k, len(keys))] = keys[:k]
    return out


def _case(seed, B=3, P=8, max_len=100, nq=4, causal=1):
    rng = np.random.default_rng(seed)
    lens = rng.integers(nq, max_len + 1, size=B).astype(np.int32)
    cu = (np.arange(B + 1) * nq).astype(np.int32)
    T = B * nq
    ld = int(lens.max())
    logits = rng.standard_normal((T, ld))
    vis = np.array([O.visible(t, lens, cu, causal) for t in range(T)])
    return rng, lens, cu, T, ld, logits, vis


@pytest.mark.parametrize("causal", [0, 1])
def test_cand_against_brute_force(causal):
    for seed in range(6):
        rng, lens, cu, T, ld, logits, vis = _case(100 + seed, causal=causal)
        P, k = 8, 11
        nb = (lens.max() + P - 1) // P
        cand = np.full((T, 9), -7, np.int32)
        n_cand = rng.integers(0, 10, size=T).astype(np.int32)
        for t in range(T):
            cand[t, :n_cand[t]] = rng.integers(-2, nb + 3, size=n_cand[t])  # repeats, out of range
        got = O.topk_cand(logits, lens, cu, causal, cand, n_cand, P, k)
        np.testing.assert_array_equal(got, _brute(logits, vis, cand, n_cand, P, k))


def test_every_block_a_candidate_is_the_dense_topk():
    rng, lens, cu, T, ld, logits, vis = _case(120, causal=1)
    P, k = 8, 13
    nb = (int(lens.max()) + P - 1) // P
    cand = np.tile(rng.permutation(nb).astype(np.int32), (T, 1))
    n_cand = np.full(T, nb, np.int32)
    got = O.topk_cand(logits, lens, cu, 1, cand, n_cand, P, k)
    np.testing.assert_array_equal(got, O.topk(logits, lens, cu, 1, k))


def test_cand_special_cases():
    P, k = 4, 6
    lens = np.array([10], np.int32)          # blocks 0, 1 full; block 2 holds keys 8, 9
    cu = np.array([0, 3], np.int32)
    logits = np.tile(np.arange(10, dtype=np.float64)[::-1], (3, 1))  # key s scores 9 - s
    cand = np.array([[2, 2, 2], [1, 0, 99], [0, 0, 0]], np.int32)
    n_cand = np.array([3, 3, 0], np.int32)
    got = O.topk_cand(logits, lens, cu, 0, cand, n_cand, P, k)
    # a repeated partial block: its 2 keys then padding; blocks 1 and 0 (99 names no block):
    # the 6 best of keys 0..7 in score order; no candidates: all padding
    np.testing.assert_array_equal(got, [[8, 9, -1, -1, -1, -1], [0, 1, 2, 3, 4, 5],
                                        [-1] * 6])
    # causal: the 3 queries see 8, 9, 10 keys; block 2 is invisible to the first
    got = O.topk_cand(logits, lens, cu, 1, np.array([[2, 1, 0]] * 3, np.int32),
                      np.array([2, 2, 2], np.int32), P, k)
    np.testing.assert_array_equal(got, [[4, 5, 6, 7, -1, -1], [4, 5, 6, 7, 8, -1],
                                        [4, 5, 6, 7, 8, 9]])


def test_cand_rows_subset_matches_all_rows():
    rng, lens, cu, T, ld, logits, vis = _case(130, causal=1)
    P, k = 8, 5
    cand = rng.integers(0, 13, size=(T, 4)).astype(np.int32)
    n_cand = rng.integers(0, 5, size=T).astype(np.int32)
    n_cand[[T - 1, 0, 5]] = [4, 1, 3]
    full = O.topk_cand(logits, lens, cu, 1, cand, n_cand, P, k)
    rows = np.array([T - 1, 0, 5], np.int64)
    part = O.topk_cand(logits[rows], lens, cu, 1, cand, n_cand, P, k, rows=rows)
    np.testing.assert_array_equal(part, full[rows])


def test_cand_ties_take_the_lower_key():
    """Equal logits: the lower key positions win (the order is value descending, index
    ascending), across blocks listed in any order."""
    lens = np.array([24], np.int32)
    cu = np.array([0, 1], np.int32)
    logits = np.zeros((1, 24))
    logits[0, 20] = 1.0
    got = O.topk_cand(logits, lens, cu, 0, np.array([[5, 2, 3]], np.int32), np.array([3], np.int32), 4, 5)
    np.testing.assert_array_equal(got, [[20, 8, 9, 10, 11]])
