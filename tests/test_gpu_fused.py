"""GPU parity of the fused scorer -> top-k (idx_mqa_topk_paged) through the C ABI.

Its logits come from the same epilogue arithmetic as idx_mqa_logits_paged, so its indices
must equal idx_topk's over the scorer's logits, row for row and in the same order; on the
rows the oracle scores they are also checked against the exact scores (the tolerance rule
of the other top-k tests). A second call on the same workspace checks that the decode
arrival counters are left at zero.
"""
import numpy as np
import pytest

from sparse_attention_indexer_mqa_gb300 import workloads as W

from helpers import Dev, assert_topk_valid, oracle_logits, oracle_q, oracle_store
from test_gpu_parity import _chunked_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as T
    from sparse_attention_indexer_mqa_gb300 import binding
    binding.load()
    return T


def _fused_vs_unfused(wl, oracle_rows=None, label=""):
    import torch
    d = Dev(wl)
    d.store()
    d.quant()
    d.score()
    d.select()
    ref = d.host("topk").copy()
    got_t, ws = d.select_fused()
    got = got_t.cpu().numpy()
    assert int(d.host("status")[0]) == 0, label
    bad = np.nonzero((got != ref).any(axis=1))[0]
    assert bad.size == 0, f"{label}: {bad.size} rows differ from the unfused path, first {bad[:5]}"
    # the same workspace again: the counters were reset
    got2, _ = d.select_fused(workspace=ws)
    np.testing.assert_array_equal(got2.cpu().numpy(), ref, err_msg=f"{label}: second call")
    if oracle_rows is not None:
        pool_ref = oracle_store(wl)
        qc, qs, w = oracle_q(wl)
        rows = np.asarray(oracle_rows)
        exact = oracle_logits(wl, pool_ref, qc, qs, w, rows=rows)
        r = torch.from_numpy(rows.astype(np.int64)).cuda()
        assert_topk_valid(got[rows], exact, d.logits[r].cpu().numpy(), wl.visible()[rows], wl.topk,
                          label=label)
    return d


def test_fused_tiny_decode(torch):
    wl = W.make("tiny_decode")
    _fused_vs_unfused(wl, oracle_rows=np.arange(wl.T), label="tiny")


def test_fused_decode_b64_full(torch):
    _fused_vs_unfused(W.make("decode_b64"), oracle_rows=np.arange(0, 64, 9), label="decode B64")


def test_fused_decode_compressed_full(torch):
    _fused_vs_unfused(W.make("decode_compressed"), oracle_rows=np.arange(0, 256, 37),
                      label="decode compressed")


def test_fused_fp8_decode(torch):
    _fused_vs_unfused(W.make("prefill_fp8", B=5, cached=3001, new=1), oracle_rows=np.arange(5),
                      label="fp8 decode")


def test_fused_decode_many_short_sequences(torch):
    """Many short sequences (a CTA's slice holds many whole sequences; zero-length ones)."""
    rng = np.random.default_rng(44)
    lens = rng.integers(0, 400, 5000)
    lens[rng.random(5000) < 0.05] = 0
    wl = _chunked_prefill(W.MXFP4, 32, 64, 0, lens.tolist(), [1] * 5000, seed=45)
    _fused_vs_unfused(wl, oracle_rows=np.sort(rng.choice(5000, 50, replace=False)), label="many short")


def test_fused_prefill_small(torch):
    wl = W.make("prefill_8k", T=700)
    _fused_vs_unfused(wl, oracle_rows=np.arange(0, 700, 23), label="prefill 700")


def test_fused_prefill_8k_full(torch):
    wl = W.make("prefill_8k")
    rows = np.unique(np.concatenate([np.arange(1020, 1030), np.linspace(0, 8191, 24).astype(int)]))
    _fused_vs_unfused(wl, oracle_rows=rows, label="prefill 8192")


@pytest.mark.parametrize("dtype,H,P,causal", [
    (W.MXFP4, 4, 64, 1), (W.MXFP4, 24, 128, 0), (W.MXFP4, 64, 64, 1), (W.FP8, 64, 64, 1),
    (W.FP8, 8, 128, 0), (W.FP8, 32, 128, 1)])
def test_fused_chunked_prefill(torch, dtype, H, P, causal):
    wl = _chunked_prefill(dtype, H, P, causal, [3000, 517, 129, 1, 2], [237, 200, 129, 1, 3],
                          seed=H * 11 + P)
    wl.topk = 256
    _fused_vs_unfused(wl, oracle_rows=np.arange(0, wl.T, 17), label=f"chunked {dtype} H{H} P{P} c{causal}")


def test_fused_fp8_full(torch):
    wl = W.make("prefill_fp8")
    rows = np.concatenate([b * 4096 + np.array([0, 2047, 4095]) for b in range(8)])
    _fused_vs_unfused(wl, oracle_rows=rows, label="fp8 32K")


def test_fused_bad_lengths(torch):
    """A sequence over max_seq_len_k (decode) or over max_q_len (prefill): its rows are -1
    and IDX_STATUS_BAD_LEN is set; the other rows match the unfused path."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    import torch as T
    for wl, max_q in [(W.make("tiny_decode"), 1),
                      (_chunked_prefill(W.MXFP4, 32, 128, 1, [400, 300], [150, 40], seed=4), 100)]:
        d = Dev(wl)
        d.store(); d.quant()
        d.score(); d.select()
        ref = d.host("topk").copy()
        sl = d.seq_lens_k.clone()
        max_k = int(wl.seq_lens_k.max())
        if max_q == 1:
            sl[1] = max_k + 1
        n = Bn.idx_mqa_topk_workspace_bytes(wl.T, wl.H, wl.B, max_q, max_k)
        ws = T.zeros(max(n, 256), dtype=T.uint8, device="cuda")
        out = T.full((wl.T, wl.topk), -7, dtype=T.int32, device="cuda")
        d.status.zero_()
        Bn.idx_mqa_topk_paged(d.q_codes, d.q_scales, d.w, wl.dtype, d.pool, wl.pool_pages, wl.page_size,
                              wl.page_stride, d.page_table, sl, d.cu, wl.causal, max_q, max_k, wl.topk,
                              out, ws, dev_status=d.status)
        o = out.cpu().numpy()
        assert int(d.host("status")[0]) & Bn.IDX_STATUS_BAD_LEN
        if max_q == 1:
            assert (o[1] == -1).all()
            np.testing.assert_array_equal(o[0], ref[0])
        else:
            assert (o[:150] == -1).all()
            np.testing.assert_array_equal(o[150:], ref[150:])
