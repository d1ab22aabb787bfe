"""GPU tests of the decode scorer's dynamic schedule (idx_mqa_logits_paged with a workspace).

The (sequence, tile) units are handed out as jobs claimed from a counter in the workspace
instead of as static slices; every key's logit comes from the same arithmetic, so the logits
must equal the static schedule's bit for bit (and the oracle's within the tolerance), the
workspace must be zero again after each call, and the status bits must be the same.
"""
import numpy as np
import pytest

from sparse_attention_indexer_mqa_gb300 import workloads as W

from helpers import Dev, assert_logits_close, oracle_logits, oracle_q, oracle_store
from test_gpu_parity import _chunked_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as T
    from sparse_attention_indexer_mqa_gb300 import binding
    binding.load()
    return T


def _ws(torch):
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    return torch.zeros(Bn.idx_mqa_logits_workspace_bytes(), dtype=torch.uint8, device="cuda")


def _static_vs_dynamic(torch, wl, label, status=0, oracle_rows=None):
    d = Dev(wl)
    d.store()
    d.quant()
    d.score()
    ref = d.host("logits").copy()
    st_ref = int(d.host("status")[0])
    assert st_ref == status, label
    ws = _ws(torch)
    for rep in range(2):  # the second call reuses the workspace the first one left zeroed
        d.logits.fill_(float("nan"))
        d.status.zero_()
        d.score(workspace=ws)
        got = d.host("logits")
        assert int(d.host("status")[0]) == status, f"{label} call {rep}"
        np.testing.assert_array_equal(got, ref, err_msg=f"{label} call {rep}")
        assert int(ws.count_nonzero().item()) == 0, f"{label}: workspace not zero after call {rep}"
    if oracle_rows is not None:
        pool_ref = oracle_store(wl)
        qc, qs, w = oracle_q(wl)
        rows = np.asarray(oracle_rows)
        exact = oracle_logits(wl, pool_ref, qc, qs, w, rows=rows)
        assert_logits_close(ref[rows], exact, wl.visible()[rows], label=label)
    return d


def test_sched_tiny(torch):
    wl = W.make("tiny_decode")
    _static_vs_dynamic(torch, wl, "tiny", oracle_rows=np.arange(wl.T))


def test_sched_decode_b64(torch):
    _static_vs_dynamic(torch, W.make("decode_b64"), "decode B64", oracle_rows=[0, 31, 63])


def test_sched_decode_compressed_256_sequences(torch):
    """256 sequences (the table's capacity), 64 heads, 64-key pages, ragged lengths."""
    _static_vs_dynamic(torch, W.make("decode_compressed"), "decode compressed", oracle_rows=[0, 100, 255])


def test_sched_fp8(torch):
    _static_vs_dynamic(torch, W.make("prefill_fp8", B=5, cached=3001, new=1), "fp8 decode",
                       oracle_rows=np.arange(5))


def test_sched_ragged_with_empty_sequences(torch):
    """Zero-length sequences, one-tile sequences, odd lengths and one long sequence."""
    rng = np.random.default_rng(91)
    lens = rng.integers(0, 700, 200)
    lens[rng.random(200) < 0.1] = 0
    lens[7] = 20000
    lens[8] = 1
    wl = _chunked_prefill(W.MXFP4, 32, 64, 0, lens.tolist(), [1] * 200, seed=92)
    _static_vs_dynamic(torch, wl, "ragged", oracle_rows=[7, 8, 9, 150])


def test_sched_more_sequences_than_the_table(torch):
    """257 sequences: the static schedule runs (same logits; the workspace stays zero)."""
    rng = np.random.default_rng(93)
    lens = rng.integers(1, 500, 257)
    wl = _chunked_prefill(W.MXFP4, 16, 128, 0, lens.tolist(), [1] * 257, seed=94)
    _static_vs_dynamic(torch, wl, "257 sequences")


def test_sched_length_and_page_faults(torch):
    """A sequence longer than max_seq_len_k is skipped with IDX_STATUS_BAD_LEN and a page-table
    entry past the pool skips its tile with IDX_STATUS_BAD_PAGE, under both schedules alike."""
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    wl = W.make("decode_b64", B=16)
    d = Dev(wl)
    d.store()
    d.quant()
    lens = d.seq_lens_k.clone()
    lens[3] = int(wl.seq_lens_k.max()) + 1
    pt = d.page_table.clone()
    pt[5, 2] = wl.pool_pages + 3
    d.seq_lens_k.copy_(lens)
    out = {}
    for name, ws in (("static", None), ("dynamic", _ws(torch))):
        d.logits.fill_(float("nan"))
        d.status.zero_()
        d.score(page_table=pt, workspace=ws)
        out[name] = (d.host("logits").copy(), int(d.host("status")[0]))
        if ws is not None:
            assert int(ws.count_nonzero().item()) == 0
    st = out["static"][1]
    assert st & Bn.IDX_STATUS_BAD_LEN and st & Bn.IDX_STATUS_BAD_PAGE
    assert out["dynamic"][1] == st
    np.testing.assert_array_equal(out["dynamic"][0], out["static"][0])
    assert np.isnan(out["static"][0][3]).all()


def test_bounded_wait_gives_up_and_reports(torch):
    """A wait on an mbarrier that nothing completes (the wait helper all kernels use) gives
    up after its limit, sets IDX_STATUS_TIMEOUT and returns; the context stays usable (a
    scorer call right after runs normally)."""
    import time
    from sparse_attention_indexer_mqa_gb300 import binding as Bn
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    Bn.idx_debug_wait_timeout(20000, status)  # 20 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) == Bn.IDX_STATUS_TIMEOUT
    assert 0.015 < dt < 5.0
    _static_vs_dynamic(torch, W.make("tiny_decode"), "after a timeout")
