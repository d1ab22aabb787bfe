"""GPU parity of the candidate-pool path (idx_mqa_topk_cand_paged) through the C ABI.

vllm PR 60834 "Purpose": the candidate-pool path of V4.1's two-level indexer ranks only the
keys of each query's candidate blocks (reading R17 at the oracle's orc_topk_cand). The GPU
set is checked against the oracle's exact scores over the same candidate keys (same size, no
repeats, only candidate keys, -1 padding, and every difference from the exact set within the
logits tolerance of the exact k-th value). Listing every block in order must reproduce the
dense scorer + top-k exactly.
"""
import numpy as np
import pytest

import oracle as O
from sparse_attention_indexer_mqa_gb300 import workloads as W

from helpers import LOGIT_RTOL, Dev, oracle_logits, oracle_q, oracle_store

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as T
    from sparse_attention_indexer_mqa_gb300 import binding
    binding.load()
    return T


def _run_cand(d, cand, n_cand, max_cand, status_ok=True):
    import torch
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    wl = d.wl
    nq = np.diff(wl.cu_seqlens_q)
    max_q, max_k = int(nq.max()), int(wl.seq_lens_k.max())
    n = Bn.idx_mqa_topk_cand_workspace_bytes(wl.T, max_cand, wl.page_size, max_k)
    ws = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")  # no starting value needed
    out = torch.full((wl.T, wl.topk), -7, dtype=torch.int32, device="cuda")
    c = torch.from_numpy(cand).cuda()
    nc = torch.from_numpy(n_cand).cuda()
    Bn.idx_mqa_topk_cand_paged(d.q_codes, d.q_scales, d.w, wl.dtype, d.pool, wl.pool_pages, wl.page_size,
                               wl.page_stride, d.page_table, d.seq_lens_k, d.cu, wl.causal, max_q, max_k,
                               c, nc, max_cand, wl.topk, out, ws, dev_status=d.status)
    torch.cuda.synchronize()
    if status_ok:
        assert int(d.status.item()) == 0
    return out.cpu().numpy()


def _cand_keys(vis, cand_row, n, P):
    blocks = set(int(b) for b in cand_row[:n])
    return np.array([s for s in range(int(vis)) if s // P in blocks], np.int64)


def _assert_cand_valid(got, exact, rows, wl, cand, n_cand, label):
    vis = wl.visible()
    k, P = wl.topk, wl.page_size
    ref = O.topk_cand(exact, wl.seq_lens_k, wl.cu_seqlens_q, wl.causal, cand, n_cand, P, k, rows=rows)
    for i, t in enumerate(rows):
        keys = _cand_keys(vis[t], cand[t], n_cand[t], P)
        g = got[t]
        n = min(k, keys.size)
        assert (g[n:] == -1).all(), f"{label} row {t}: bad padding"
        sel = g[:n]
        assert len(np.unique(sel)) == n, f"{label} row {t}: repeats"
        assert np.isin(sel, keys).all(), f"{label} row {t}: a key outside the candidate blocks"
        if keys.size <= k:
            assert set(sel.tolist()) == set(keys.tolist())
            continue
        e = exact[i]
        ex = ref[i][:n]
        kth = e[ex[-1]]
        tol = LOGIT_RTOL * np.abs(e[:int(vis[t])]).max()
        for s in set(ex.tolist()).symmetric_difference(sel.tolist()):
            assert abs(e[s] - kth) <= tol, f"{label} row {t}: key {s} off by {e[s] - kth:.3e}"


def _check(wl, rows, n_blocks=16, messy=False, label=""):
    d = Dev(wl)
    d.store()
    d.quant()
    cand, n_cand, max_cand = W.candidate_blocks(wl, seed=3, n_blocks=n_blocks, messy=messy)
    got = _run_cand(d, cand, n_cand, max_cand)
    pool_ref = oracle_store(wl)
    qc, qs, w = oracle_q(wl)
    rows = np.asarray(rows, np.int64)
    exact = oracle_logits(wl, pool_ref, qc, qs, w, rows=rows)
    _assert_cand_valid(got, exact, rows, wl, cand, n_cand, label)
    return d, got


def test_cand_tiny_decode_messy_lists(torch):
    wl = W.make("tiny_decode")
    wl.topk = 8
    _check(wl, np.arange(wl.T), n_blocks=2, messy=True, label="tiny")


def test_cand_decode_b64(torch):
    wl = W.make("decode_b64")
    _check(wl, np.arange(wl.T), n_blocks=16, label="decode B64")


def test_cand_decode_compressed_64_key_pages(torch):
    """64-key pages: a 128-key tile of the virtual sequence spans two candidate blocks."""
    wl = W.make("decode_compressed")
    _check(wl, np.arange(0, wl.T, 5), n_blocks=20, messy=True, label="decode compressed")


def test_cand_causal_prefill_partial_blocks(torch):
    """Causal queries: the block at each query's visibility edge is partial."""
    wl = W.make("prefill_8k", T=1000)
    rows = np.concatenate([np.arange(0, 1000, 37), [999, 998, 129, 127, 128]])
    _check(wl, rows, n_blocks=4, messy=True, label="prefill 1000")


def test_cand_fp8(torch):
    wl = W.make("prefill_fp8", B=3, cached=2000, new=5)
    _check(wl, np.arange(wl.T), n_blocks=9, label="fp8")


def test_cand_every_block_is_the_dense_path(torch):
    """All blocks, in order, as candidates: the same logits, so the same indices in the same
    order as the dense scorer followed by idx_topk."""
    wl = W.make("decode_b64", B=16)
    d = Dev(wl)
    d.store()
    d.quant()
    d.score()
    d.select()
    ref = d.host("topk").copy()
    nb = (int(wl.seq_lens_k.max()) + wl.page_size - 1) // wl.page_size
    cand = np.tile(np.arange(nb, dtype=np.int32), (wl.T, 1))
    got = _run_cand(d, cand, np.full(wl.T, nb, np.int32), nb)
    np.testing.assert_array_equal(got, ref)


def test_cand_bad_counts(torch):
    """n_cand above max_cand or negative: the row is all -1 and IDX_STATUS_BAD_LEN is set;
    the other rows are unaffected."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    wl = W.make("decode_b64", B=8)
    d = Dev(wl)
    d.store()
    d.quant()
    cand, n_cand, max_cand = W.candidate_blocks(wl, seed=3, n_blocks=12)
    good = _run_cand(d, cand, n_cand, max_cand)
    n_bad = n_cand.copy()
    n_bad[0] = max_cand + 1
    n_bad[1] = -1
    got = _run_cand(d, cand, n_bad, max_cand, status_ok=False)
    assert int(d.status.item()) & Bn.IDX_STATUS_BAD_LEN
    assert (got[:2] == -1).all()
    np.testing.assert_array_equal(got[2:], good[2:])
