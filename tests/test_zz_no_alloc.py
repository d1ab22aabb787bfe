"""The workspace-free decode scorer -> top-k (idx_mqa_topk_paged_noalloc), for callers that
cannot allocate device memory, against the workspace form (idx_mqa_topk_paged) through the C
ABI: the same indices, row for row, on two calls in a row (the library's fixed scratch
array keeps the previous call's contents, so the second call checks that nothing stale is
used). Both run the same decode kernel on the same logits, so the rows must be identical.

This file is named to be collected last: if it fails, a run that stops at the first failure
has already run every other test.
"""
import numpy as np
import pytest

from sparse_attention_indexer_mqa_gb300 import workloads as W

from helpers import Dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as T
    from sparse_attention_indexer_mqa_gb300 import binding
    binding.load()
    return T


def _noalloc(d, out):
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    wl = d.wl
    Bn.idx_mqa_topk_paged_noalloc(d.q_codes, d.q_scales, d.w, wl.dtype, d.pool, wl.pool_pages,
                                  wl.page_size, wl.page_stride, d.page_table, d.seq_lens_k, d.cu,
                                  wl.causal, 1, int(wl.seq_lens_k.max()), wl.topk, out,
                                  dev_status=d.status)


@pytest.mark.parametrize("name,over", [("tiny_decode", {}), ("decode_b64", {}),
                                       ("decode_compressed", {}),
                                       ("prefill_fp8", {"B": 5, "cached": 3001, "new": 1})])
def test_noalloc_matches_workspace_form(torch, name, over):
    wl = W.make(name, **over)
    d = Dev(wl)
    d.store()
    d.quant()
    ref, _ = d.select_fused()
    ref = ref.cpu().numpy()
    for call in range(2):
        out = torch.full((wl.T, wl.topk), -7, dtype=torch.int32, device="cuda")
        _noalloc(d, out)
        got = out.cpu().numpy()
        assert int(d.host("status")[0]) == 0
        np.testing.assert_array_equal(got, ref, err_msg=f"{name}, call {call + 1}")


def test_noalloc_rejects_what_does_not_fit(torch):
    """Prefill shapes, more sequences than counters, and more scratch than the array holds
    are refused before anything runs."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    import ctypes as C
    lib = Bn.load()
    # (T, B, max_q_len, max_seq_len_k): prefill; 16385 sequences; 300 x 8192 floats > 8 MiB
    for T, B, mq, mk in [(64, 2, 32, 1024), (16385, 16385, 1, 64), (300, 300, 1, 8192)]:
        st = lib.idx_mqa_topk_paged_noalloc(16, 16, 16, T, 32, 0, 16, 1, 128, 8704, 16, 64, 16, 16, B,
                                            0, mq, mk, 64, 16, None, None)
        assert st == -2, (T, B, mq, mk, st)
