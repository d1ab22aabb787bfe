"""Thin ctypes binding of libidx_gb300.so (include/idx.h).

The functions carry the C names and only marshal arguments: torch tensors become raw
pointers, the stream defaults to torch's current stream, and a non-zero status raises
IdxError. All computation runs in the library's CUDA kernels; there is no fallback: if the
library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import re
import threading

from . import build as _build

IDX_MXFP4, IDX_FP8 = 0, 1
IDX_ROPE_NONE, IDX_ROPE_NEOX, IDX_ROPE_INTERLEAVED = 0, 1, 2
IDX_STATUS_BAD_SLOT, IDX_STATUS_BAD_POS, IDX_STATUS_BAD_PAGE = 0x1, 0x2, 0x4
IDX_STATUS_TIMEOUT, IDX_STATUS_BAD_LEN = 0x8, 0x10

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "idx.h")

_lock = threading.Lock()
_lib = None


class IdxError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed with status {status} ({_status_str(status)})")
        self.status = status


class IdxLayout(C.Structure):
    _fields_ = [("page_bytes", C.c_int64), ("code_offset", C.c_int64),
                ("code_bytes", C.c_int64), ("scale_offset", C.c_int64),
                ("scale_bytes", C.c_int64), ("bytes_per_token", C.c_int32),
                ("page_size", C.c_int32)]


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load (building first if needed) the CUDA library; raises if that is impossible."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing; run build() first")
            lib = C.CDLL(path)
            _declare(lib)
            _lib = lib
    return _lib


def exported_names():
    """Entry points declared in include/idx.h."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(idx_\w+)\(", txt, re.M)))


def _declare(L):
    vp, i64, i32, f32 = C.c_void_p, C.c_int64, C.c_int32, C.c_float
    L.idx_status_string.argtypes = [C.c_int]; L.idx_status_string.restype = C.c_char_p
    L.idx_cache_layout.argtypes = [i32, i32, C.POINTER(IdxLayout)]
    L.idx_k_store.argtypes = [vp, i64, i64, vp, vp, vp, i32, i32, i32, vp, vp, f32, i32, vp, i64,
                              i32, i64, vp, vp]
    L.idx_q_quant.argtypes = [vp, i64, i32, vp, vp, i32, i32, vp, f32, f32, i32, vp, vp, vp, vp,
                              vp]
    L.idx_qk_prep.argtypes = [vp, i64, i64, vp, vp, i32, i32, vp, vp, f32, vp, i64, i32, i64,
                              vp, i64, i32, vp, i32, vp, f32, f32, vp, vp, vp, vp, i32, i32, vp, vp]
    L.idx_mqa_logits_paged.argtypes = [vp, vp, vp, i64, i32, i32, vp, i64, i32, i64, vp, i32, vp,
                                       vp, i32, i32, i32, i32, vp, i64, vp, C.c_size_t, vp, vp]
    L.idx_mqa_logits_workspace_bytes.argtypes = [C.POINTER(C.c_size_t)]
    L.idx_topk.argtypes = [vp, i64, vp, vp, i32, i64, i32, i32, i32, vp, vp, vp]
    L.idx_debug_encode.argtypes = [i32, vp, i64, vp, vp]
    L.idx_mqa_topk_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, C.POINTER(C.c_size_t)]
    L.idx_mqa_topk_paged.argtypes = [vp, vp, vp, i64, i32, i32, vp, i64, i32, i64, vp, i32, vp, vp,
                                     i32, i32, i32, i32, i32, vp, vp, C.c_size_t, vp, vp]
    L.idx_debug_mma_rate.argtypes = [i32, i32, vp, C.POINTER(C.c_double), vp]
    L.idx_mqa_topk_paged_noalloc.argtypes = [vp, vp, vp, i64, i32, i32, vp, i64, i32, i64, vp, i32,
                                             vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
    L.idx_mqa_topk_cand_workspace_bytes.argtypes = [i64, i32, i32, i32, C.POINTER(C.c_size_t)]
    L.idx_mqa_topk_cand_paged.argtypes = [vp, vp, vp, i64, i32, i32, vp, i64, i32, i64, vp, i32, vp,
                                          vp, i32, i32, i32, i32, vp, i32, vp, i32, i32, vp, vp,
                                          C.c_size_t, vp, vp]
    L.idx_debug_wait_timeout.argtypes = [i32, vp, vp]
    L.idx_compress_k_store.argtypes = [vp, vp, i64, i64, vp, vp, i64, i32, vp, vp, vp, i32, i32, i32,
                                       vp, vp, f32, i32, vp, i64, i32, i64, vp, vp]
    for n in ("idx_cache_layout", "idx_k_store", "idx_q_quant", "idx_qk_prep", "idx_mqa_logits_paged",
              "idx_topk", "idx_debug_encode", "idx_mqa_topk_workspace_bytes", "idx_mqa_topk_paged",
              "idx_debug_mma_rate", "idx_mqa_topk_paged_noalloc", "idx_compress_k_store",
              "idx_mqa_topk_cand_workspace_bytes", "idx_mqa_topk_cand_paged",
              "idx_mqa_logits_workspace_bytes", "idx_debug_wait_timeout"):
        getattr(L, n).restype = C.c_int


def _status_str(s):
    try:
        return load(False).idx_status_string(s).decode()
    except Exception:
        return "?"


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, st):
    if st != 0:
        raise IdxError(fn, st)


def idx_cache_layout(dtype: int, page_size: int) -> IdxLayout:
    out = IdxLayout()
    _check("idx_cache_layout", load().idx_cache_layout(dtype, page_size, C.byref(out)))
    return out


def idx_k_store(k, slot_mapping, positions, cos_sin, rope, apply_norm, dtype, pool, num_pages,
                page_size, page_stride, gamma=None, beta=None, eps=1e-6, dev_status=None,
                stream=None, n_rows=None, k_row_stride=None):
    n = k.shape[0] if n_rows is None else n_rows
    stride = k.stride(0) if k_row_stride is None else k_row_stride
    max_pos = cos_sin.shape[0] if cos_sin is not None else 0
    _check("idx_k_store", load().idx_k_store(
        _ptr(k), n, stride, _ptr(slot_mapping), _ptr(positions), _ptr(cos_sin), max_pos, rope,
        int(apply_norm), _ptr(gamma), _ptr(beta), eps, dtype, _ptr(pool), num_pages, page_size,
        page_stride, _ptr(dev_status), _stream(stream)))


def idx_compress_k_store(k_raw, gate, boundary, first, ratio, slot_mapping, positions, cos_sin, rope,
                         norm, dtype, pool, num_pages, page_size, page_stride, gamma=None, beta=None,
                         eps=1e-6, dev_status=None, stream=None, n_entries=None):
    """k_raw / gate: bf16 (int16/uint16 storage) [n_raw, >=128] sharing one row stride."""
    assert k_raw.stride(0) == gate.stride(0) and k_raw.shape[0] == gate.shape[0]
    n = boundary.shape[0] if n_entries is None else n_entries
    max_pos = cos_sin.shape[0] if cos_sin is not None else 0
    _check("idx_compress_k_store", load().idx_compress_k_store(
        _ptr(k_raw), _ptr(gate), k_raw.shape[0], k_raw.stride(0), _ptr(boundary), _ptr(first), n,
        int(ratio), _ptr(slot_mapping), _ptr(positions), _ptr(cos_sin), max_pos, rope, int(norm),
        _ptr(gamma), _ptr(beta), eps, dtype, _ptr(pool), num_pages, page_size, page_stride,
        _ptr(dev_status), _stream(stream)))


def idx_q_quant(q, positions, cos_sin, rope, w_in, softmax_scale, head_scale, dtype, q_codes,
                q_scales, w_out, dev_status=None, stream=None):
    T, H = q.shape[0], q.shape[1]
    max_pos = cos_sin.shape[0] if cos_sin is not None else 0
    _check("idx_q_quant", load().idx_q_quant(
        _ptr(q), T, H, _ptr(positions), _ptr(cos_sin), max_pos, rope, _ptr(w_in), softmax_scale,
        head_scale, dtype, _ptr(q_codes), _ptr(q_scales), _ptr(w_out), _ptr(dev_status),
        _stream(stream)))


def idx_qk_prep(k, slot_mapping, k_positions, k_rope, apply_norm, pool, num_pages, page_size,
                page_stride, q, q_positions, q_rope, w_in, softmax_scale, head_scale, q_codes,
                q_scales, w_out, cos_sin, dtype, gamma=None, beta=None, eps=1e-6, dev_status=None,
                stream=None):
    n = k.shape[0] if k is not None else 0
    stride = k.stride(0) if k is not None else 128
    T, H = q.shape[0], q.shape[1]
    max_pos = cos_sin.shape[0] if cos_sin is not None else 0
    _check("idx_qk_prep", load().idx_qk_prep(
        _ptr(k), n, stride, _ptr(slot_mapping), _ptr(k_positions), k_rope, int(apply_norm),
        _ptr(gamma), _ptr(beta), eps, _ptr(pool), num_pages, page_size, page_stride, _ptr(q), T, H,
        _ptr(q_positions), q_rope, _ptr(w_in), softmax_scale, head_scale, _ptr(q_codes),
        _ptr(q_scales), _ptr(w_out), _ptr(cos_sin), max_pos, dtype, _ptr(dev_status),
        _stream(stream)))


def idx_mqa_logits_paged(q_codes, q_scales, w, dtype, pool, num_pages, page_size, page_stride,
                         page_table, seq_lens_k, cu_seqlens_q, causal, max_q_len, max_seq_len_k,
                         logits, dev_status=None, stream=None, workspace=None):
    T, H = w.shape
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("idx_mqa_logits_paged", load().idx_mqa_logits_paged(
        _ptr(q_codes), _ptr(q_scales), _ptr(w), T, H, dtype, _ptr(pool), num_pages, page_size,
        page_stride, _ptr(page_table), page_table.shape[1], _ptr(seq_lens_k), _ptr(cu_seqlens_q),
        seq_lens_k.shape[0], int(causal), max_q_len, max_seq_len_k, _ptr(logits),
        logits.stride(0), _ptr(workspace), wsb, _ptr(dev_status), _stream(stream)))


def idx_mqa_logits_workspace_bytes() -> int:
    n = C.c_size_t(0)
    _check("idx_mqa_logits_workspace_bytes", load().idx_mqa_logits_workspace_bytes(C.byref(n)))
    return int(n.value)


def idx_topk(logits, seq_lens_k, cu_seqlens_q, causal, max_seq_len_k, k, out_idx,
             dev_status=None, stream=None, T=None):
    T = logits.shape[0] if T is None else T
    _check("idx_topk", load().idx_topk(
        _ptr(logits), logits.stride(0), _ptr(seq_lens_k), _ptr(cu_seqlens_q),
        seq_lens_k.shape[0], T, int(causal), int(max_seq_len_k), k, _ptr(out_idx),
        _ptr(dev_status), _stream(stream)))


def idx_mqa_topk_workspace_bytes(T, H, B, max_q_len, max_seq_len_k) -> int:
    n = C.c_size_t(0)
    _check("idx_mqa_topk_workspace_bytes",
           load().idx_mqa_topk_workspace_bytes(T, H, B, max_q_len, max_seq_len_k, C.byref(n)))
    return int(n.value)


def idx_mqa_topk_paged(q_codes, q_scales, w, dtype, pool, num_pages, page_size, page_stride,
                       page_table, seq_lens_k, cu_seqlens_q, causal, max_q_len, max_seq_len_k, k,
                       out_idx, workspace, dev_status=None, stream=None):
    T, H = w.shape
    _check("idx_mqa_topk_paged", load().idx_mqa_topk_paged(
        _ptr(q_codes), _ptr(q_scales), _ptr(w), T, H, dtype, _ptr(pool), num_pages, page_size,
        page_stride, _ptr(page_table), page_table.shape[1], _ptr(seq_lens_k), _ptr(cu_seqlens_q),
        seq_lens_k.shape[0], int(causal), max_q_len, max_seq_len_k, k, _ptr(out_idx),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status),
        _stream(stream)))


def idx_mqa_topk_cand_workspace_bytes(T, max_cand, page_size, max_seq_len_k) -> int:
    n = C.c_size_t(0)
    _check("idx_mqa_topk_cand_workspace_bytes",
           load().idx_mqa_topk_cand_workspace_bytes(T, max_cand, page_size, max_seq_len_k, C.byref(n)))
    return int(n.value)


def idx_mqa_topk_cand_paged(q_codes, q_scales, w, dtype, pool, num_pages, page_size, page_stride,
                            page_table, seq_lens_k, cu_seqlens_q, causal, max_q_len, max_seq_len_k,
                            cand_blocks, n_cand, max_cand, k, out_idx, workspace, dev_status=None,
                            stream=None):
    T, H = w.shape
    _check("idx_mqa_topk_cand_paged", load().idx_mqa_topk_cand_paged(
        _ptr(q_codes), _ptr(q_scales), _ptr(w), T, H, dtype, _ptr(pool), num_pages, page_size,
        page_stride, _ptr(page_table), page_table.shape[1], _ptr(seq_lens_k), _ptr(cu_seqlens_q),
        seq_lens_k.shape[0], int(causal), max_q_len, max_seq_len_k, _ptr(cand_blocks),
        cand_blocks.shape[1], _ptr(n_cand), max_cand, k, _ptr(out_idx), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)))


def idx_debug_encode(kind, x, out, stream=None):
    _check("idx_debug_encode", load().idx_debug_encode(kind, _ptr(x), x.numel(), _ptr(out),
                                                       _stream(stream)))


def idx_debug_wait_timeout(limit_us, dev_status, stream=None):
    _check("idx_debug_wait_timeout", load().idx_debug_wait_timeout(int(limit_us), _ptr(dev_status),
                                                                   _stream(stream)))


def idx_debug_mma_rate(dtype, iters, dev_status=None, stream=None) -> float:
    """Launch the tensor-core rate probe; returns the flops one CTA (SM) performs."""
    f = C.c_double(0.0)
    _check("idx_debug_mma_rate", load().idx_debug_mma_rate(dtype, iters, _ptr(dev_status), C.byref(f),
                                                           _stream(stream)))
    return float(f.value)


def idx_mqa_topk_paged_noalloc(q_codes, q_scales, w, dtype, pool, num_pages, page_size, page_stride,
                               page_table, seq_lens_k, cu_seqlens_q, causal, max_q_len, max_seq_len_k,
                               k, out_idx, dev_status=None, stream=None):
    T, H = w.shape
    _check("idx_mqa_topk_paged_noalloc", load().idx_mqa_topk_paged_noalloc(
        _ptr(q_codes), _ptr(q_scales), _ptr(w), T, H, dtype, _ptr(pool), num_pages, page_size,
        page_stride, _ptr(page_table), page_table.shape[1], _ptr(seq_lens_k), _ptr(cu_seqlens_q),
        seq_lens_k.shape[0], int(causal), max_q_len, max_seq_len_k, k, _ptr(out_idx),
        _ptr(dev_status), _stream(stream)))
