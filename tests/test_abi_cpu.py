"""CPU-side checks of the C ABI: the library builds, loads and exports every entry point of
include/idx.h; the layout query; host-side argument validation (these calls return before
any launch, so no GPU is needed)."""
import ctypes as C

import pytest

from sparse_attention_indexer_mqa_gb300 import binding as Bn


@pytest.fixture(scope="module")
def lib():
    return Bn.load()


def test_exports_every_declared_symbol(lib):
    names = Bn.exported_names()
    assert {"idx_cache_layout", "idx_k_store", "idx_q_quant", "idx_qk_prep",
            "idx_mqa_logits_paged", "idx_topk"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


@pytest.mark.parametrize("dtype,P,per", [(0, 64, 68), (0, 128, 68), (1, 64, 132), (1, 128, 132)])
def test_layout(dtype, P, per):
    lay = Bn.idx_cache_layout(dtype, P)
    assert lay.bytes_per_token == per and lay.page_bytes == per * P
    assert lay.code_offset == 0 and lay.scale_offset == lay.code_bytes
    assert lay.scale_bytes == 4 * P and lay.page_size == P
    assert lay.page_bytes % 16 == 0


def test_layout_rejects_bad_sizes(lib):
    out = Bn.IdxLayout()
    assert lib.idx_cache_layout(0, 32, C.byref(out)) == -2
    assert lib.idx_cache_layout(2, 64, C.byref(out)) == -1
    assert lib.idx_cache_layout(0, 64, None) == -1


def test_host_validation(lib):
    # page size unsupported
    assert lib.idx_k_store(16, 1, 128, 16, None, None, 0, 0, 0, None, None, 1e-6, 0, 16, 1, 32,
                           4352, None, None) == -2
    # misaligned pool
    assert lib.idx_k_store(16, 1, 128, 16, None, None, 0, 0, 0, None, None, 1e-6, 0, 17, 1, 64,
                           4352, None, None) == -1
    # page stride below the page size
    assert lib.idx_k_store(16, 1, 128, 16, None, None, 0, 0, 0, None, None, 1e-6, 0, 16, 1, 64,
                           4000, None, None) == -1
    # RoPE without positions
    assert lib.idx_k_store(16, 1, 128, 16, None, None, 0, 1, 0, None, None, 1e-6, 0, 16, 1, 64,
                           4352, None, None) == -1
    # unaligned k row stride
    assert lib.idx_k_store(16, 1, 130, 16, None, None, 0, 0, 0, None, None, 1e-6, 0, 16, 1, 64,
                           4352, None, None) == -1
    # zero rows is a no-op
    assert lib.idx_k_store(None, 0, 128, None, None, None, 0, 0, 0, None, None, 1e-6, 0, 16, 1,
                           64, 4352, None, None) == 0
    # Q quant: H out of range, MXFP4 without scales
    assert lib.idx_q_quant(16, 1, 65, None, None, 0, 0, 16, 1.0, 1.0, 0, 16, 16, 16, None,
                           None) == -2
    assert lib.idx_q_quant(16, 1, 4, None, None, 0, 0, 16, 1.0, 1.0, 0, 16, None, 16, None,
                           None) == -1
    # top-k: k too large / zero
    assert lib.idx_topk(16, 8, 16, 16, 1, 1, 0, 8, 5000, 16, None, None) == -2
    assert lib.idx_topk(16, 8, 16, 16, 1, 1, 0, 8, 0, 16, None, None) == -2
    # top-k: the scorer's bound may not exceed the row stride
    assert lib.idx_topk(16, 8, 16, 16, 1, 1, 0, 9, 32, 16, None, None) == -1
    # scorer: ld below max_seq_len_k, page table stride too small
    assert lib.idx_mqa_logits_paged(16, 16, 16, 1, 4, 0, 16, 1, 64, 4352, 16, 1, 16, 16, 1, 0, 1,
                                    100, 16, 64, None, 0, None, None) == -1
    assert lib.idx_mqa_logits_paged(16, 16, 16, 1, 4, 0, 16, 1, 64, 4352, 16, 1, 16, 16, 1, 0, 1,
                                    100, 16, 128, None, 0, None, None) == -1
    # scorer: a workspace that is misaligned or too small
    assert lib.idx_mqa_logits_paged(16, 16, 16, 1, 4, 0, 16, 1, 64, 4352, 16, 1, 16, 16, 1, 0, 1,
                                    64, 16, 64, 8, 256, None, None) == -1
    assert lib.idx_mqa_logits_paged(16, 16, 16, 1, 4, 0, 16, 1, 64, 4352, 16, 1, 16, 16, 1, 0, 1,
                                    64, 16, 64, 16, 8, None, None) == -1
    # fused K store + Q quant: bad dtype, H out of range, unsupported page size
    qk = lambda dtype, H, P: lib.idx_qk_prep(16, 1, 128, 16, None, 0, 0, None, None, 1e-6, 16, 1, P,
                                             4352, 16, 1, H, None, 0, 16, 1.0, 1.0, 16, 16, 16,
                                             None, 0, dtype, None, None)
    assert qk(2, 4, 64) == -1
    assert qk(0, 65, 64) == -2
    assert qk(0, 4, 96) == -2
    assert lib.idx_debug_encode(3, 16, 1, 16, None) == -1
    assert Bn.load().idx_status_string(-3) == b"CUDA launch error"
