"""Python access to the CPU oracle (oracle.c) through ctypes.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of bench.py may import this package. It shares nothing with the
CUDA library and never imports it.

All arrays are numpy arrays in host memory; bf16 tensors are uint16 bit patterns. The
functions mirror oracle.h; see oracle.c for the rule each one follows and the page section
that defines it.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

MXFP4, FP8 = 0, 1
ROPE_NONE, ROPE_NEOX, ROPE_INTERLEAVED = 0, 1, 2

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-pthread"]


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so with gcc (no FMA contraction)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(src),
                                               os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            _declare(_lib)
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _declare(L):
    vp, i64, i32, f32, u8 = C.c_void_p, C.c_int64, C.c_int32, C.c_float, C.c_uint8
    L.orc_e2m1_encode.argtypes = [f32]; L.orc_e2m1_encode.restype = u8
    L.orc_e2m1_decode.argtypes = [u8]; L.orc_e2m1_decode.restype = C.c_double
    L.orc_e4m3_encode.argtypes = [f32]; L.orc_e4m3_encode.restype = u8
    L.orc_e4m3_decode.argtypes = [u8]; L.orc_e4m3_decode.restype = C.c_double
    L.orc_e2m1_encode_n.argtypes = [vp, i64, vp]; L.orc_e2m1_encode_n.restype = None
    L.orc_e4m3_encode_n.argtypes = [vp, i64, vp]; L.orc_e4m3_encode_n.restype = None
    L.orc_mx_shared_exponent.argtypes = [f32]; L.orc_mx_shared_exponent.restype = C.c_int
    L.orc_layernorm128.argtypes = [vp, vp, vp, f32, vp]; L.orc_layernorm128.restype = None
    L.orc_rope128.argtypes = [vp, vp, C.c_int]; L.orc_rope128.restype = None
    L.orc_mxfp4_quant128.argtypes = [vp, vp, vp]; L.orc_mxfp4_quant128.restype = None
    L.orc_fp8_quant128.argtypes = [vp, vp, vp]; L.orc_fp8_quant128.restype = None
    L.orc_page_bytes.argtypes = [C.c_int, C.c_int]; L.orc_page_bytes.restype = i64
    L.orc_code_offset.argtypes = [C.c_int] * 4; L.orc_code_offset.restype = i64
    L.orc_scale_offset.argtypes = [C.c_int] * 4; L.orc_scale_offset.restype = i64
    L.orc_k_store.argtypes = [vp, i64, i64, vp, vp, vp, i32, C.c_int, C.c_int, vp, vp, f32,
                              C.c_int, vp, i64, i32, i64]
    L.orc_k_store.restype = C.c_int
    L.orc_q_quant.argtypes = [vp, i64, i32, vp, vp, i32, C.c_int, vp, f32, f32, C.c_int, vp,
                              vp, vp]
    L.orc_q_quant.restype = C.c_int
    L.orc_visible.argtypes = [i64, vp, vp, i32, C.c_int]; L.orc_visible.restype = i64
    L.orc_exp_neg.argtypes = [f32]; L.orc_exp_neg.restype = f32
    L.orc_rmsnorm128.argtypes = [vp, vp, f32, vp]; L.orc_rmsnorm128.restype = None
    L.orc_compress_pool128.argtypes = [vp, vp, i64, i64, i64, vp]
    L.orc_compress_pool128.restype = None
    L.orc_compress_k_store.argtypes = [vp, vp, i64, i64, vp, vp, i64, i32, vp, vp, vp, i32, C.c_int,
                                       C.c_int, vp, vp, f32, C.c_int, vp, i64, i32, i64]
    L.orc_compress_k_store.restype = C.c_int
    L.orc_topk_cand.argtypes = [vp, i64, vp, vp, i32, C.c_int, vp, i64, vp, i32, vp, i32, i32, vp,
                                C.c_int]
    L.orc_topk_cand.restype = C.c_int
    L.orc_mqa_logits.argtypes = [vp, vp, vp, i64, i32, C.c_int, vp, i64, i32, i64, vp, i32,
                                 vp, vp, i32, C.c_int, vp, i64, vp, i64, C.c_int]
    L.orc_mqa_logits.restype = C.c_int
    L.orc_topk.argtypes = [vp, i64, vp, vp, i32, C.c_int, vp, i64, i32, vp, C.c_int]
    L.orc_topk.restype = C.c_int


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


# --- element encoders ------------------------------------------------------------------

def e2m1_encode(v: float) -> int:
    return int(lib().orc_e2m1_encode(float(v)))


def e2m1_decode(code: int) -> float:
    return float(lib().orc_e2m1_decode(int(code)))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_decode(int(code)))


def e2m1_encode_n(v):
    v = _c(v, np.float32).ravel()
    out = np.empty(v.shape[0], np.uint8)
    lib().orc_e2m1_encode_n(_p(v), v.shape[0], _p(out))
    return out


def e4m3_encode_n(v):
    v = _c(v, np.float32).ravel()
    out = np.empty(v.shape[0], np.uint8)
    lib().orc_e4m3_encode_n(_p(v), v.shape[0], _p(out))
    return out


def mx_shared_exponent(amax: float) -> int:
    return int(lib().orc_mx_shared_exponent(float(amax)))


# --- row steps -------------------------------------------------------------------------

def layernorm128(x, gamma=None, beta=None, eps=1e-6):
    x = _c(x, np.float32)
    g = _c(np.ones(128) if gamma is None else gamma, np.float32)
    b = _c(np.zeros(128) if beta is None else beta, np.float32)
    y = np.empty(128, np.float32)
    lib().orc_layernorm128(_p(x), _p(g), _p(b), C.c_float(eps), _p(y))
    return y


def rope128(x, cos_sin_row, mode):
    x = _c(x, np.float32).copy()
    cs = _c(cos_sin_row, np.float32)
    lib().orc_rope128(_p(x), _p(cs), int(mode))
    return x


def mxfp4_quant128(x):
    x = _c(x, np.float32)
    codes = np.empty(64, np.uint8)
    sc = np.empty(4, np.uint8)
    lib().orc_mxfp4_quant128(_p(x), _p(codes), _p(sc))
    return codes, sc


def fp8_quant128(x):
    x = _c(x, np.float32)
    codes = np.empty(128, np.uint8)
    sc = np.empty(1, np.float32)
    lib().orc_fp8_quant128(_p(x), _p(codes), _p(sc))
    return codes, float(sc[0])


# --- layout ----------------------------------------------------------------------------

def page_bytes(dtype, page_size):
    return int(lib().orc_page_bytes(dtype, page_size))


def code_offset(dtype, page_size, s, j):
    return int(lib().orc_code_offset(dtype, page_size, s, j))


def scale_offset(dtype, page_size, s, b=0):
    return int(lib().orc_scale_offset(dtype, page_size, s, b))


# --- whole steps -----------------------------------------------------------------------

def k_store(pool, k, slot_mapping, positions, cos_sin, rope, apply_norm, dtype, num_pages,
            page_size, page_stride, gamma=None, beta=None, eps=1e-6):
    """Writes into ``pool`` (uint8, modified in place); returns the rejected-row count."""
    assert pool.dtype == np.uint8 and pool.flags.c_contiguous
    k = _c(k, np.uint16)
    n_rows = k.shape[0]
    slot = _c(slot_mapping, np.int64)
    pos = _c(positions if positions is not None else np.zeros(n_rows), np.int32)
    cs = _c(cos_sin if cos_sin is not None else np.zeros((1, 64)), np.float32)
    g = _c(np.ones(128) if gamma is None else gamma, np.float32)
    b = _c(np.zeros(128) if beta is None else beta, np.float32)
    return lib().orc_k_store(_p(k), n_rows, k.shape[1], _p(slot), _p(pos), _p(cs), cs.shape[0],
                             int(rope), int(apply_norm), _p(g), _p(b), C.c_float(eps),
                             int(dtype), _p(pool), int(num_pages), int(page_size),
                             int(page_stride))


def q_quant(q, positions, cos_sin, rope, w_in, softmax_scale, head_scale, dtype):
    """q: uint16 [T, H, 128]. Returns (codes, scales, w_out); FP8 scales are fp32 [T, H]."""
    q = _c(q, np.uint16)
    T, H = q.shape[0], q.shape[1]
    pos = _c(positions if positions is not None else np.zeros(T), np.int32)
    cs = _c(cos_sin if cos_sin is not None else np.zeros((1, 64)), np.float32)
    w_in = _c(w_in, np.float32)
    if dtype == MXFP4:
        codes = np.zeros((T, H, 64), np.uint8)
        scales = np.zeros((T, H, 4), np.uint8)
    else:
        codes = np.zeros((T, H, 128), np.uint8)
        scales = np.zeros((T, H), np.float32)
    w_out = np.zeros((T, H), np.float32)
    bad = lib().orc_q_quant(_p(q), T, H, _p(pos), _p(cs), cs.shape[0], int(rope), _p(w_in),
                            C.c_float(softmax_scale), C.c_float(head_scale), int(dtype),
                            _p(codes), _p(scales), _p(w_out))
    assert bad == 0, f"{bad} Q rows had an out-of-range position"
    return codes, scales, w_out


def visible(t, seq_lens_k, cu_seqlens_q, causal):
    sl = _c(seq_lens_k, np.int32)
    cu = _c(cu_seqlens_q, np.int32)
    return int(lib().orc_visible(int(t), _p(sl), _p(cu), sl.shape[0], int(causal)))


def mqa_logits(q_codes, q_scales, w, dtype, pool, num_pages, page_size, page_stride,
               page_table, seq_lens_k, cu_seqlens_q, causal, ld, rows=None, n_threads=None):
    """Returns fp64 logits [len(rows) or T, ld]; entries past visible(t) are NaN."""
    T, H = w.shape
    qc = _c(q_codes, np.uint8)
    qs = _c(q_scales, np.uint8 if dtype == MXFP4 else np.float32)
    w = _c(w, np.float32)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens_k, np.int32)
    cu = _c(cu_seqlens_q, np.int32)
    rr = None if rows is None else _c(rows, np.int64)
    n = T if rr is None else rr.shape[0]
    out = np.full((n, ld), np.nan, np.float64)
    nt = n_threads or os.cpu_count() or 1
    lib().orc_mqa_logits(_p(qc), _p(qs), _p(w), T, H, int(dtype), _p(pool), int(num_pages),
                         int(page_size), int(page_stride), _p(pt), pt.shape[1], _p(sl), _p(cu),
                         sl.shape[0], int(causal), _p(rr), n, _p(out), int(ld), int(nt))
    return out


def topk(logits, seq_lens_k, cu_seqlens_q, causal, k, rows=None, n_threads=None):
    lg = _c(logits, np.float64)
    sl = _c(seq_lens_k, np.int32)
    cu = _c(cu_seqlens_q, np.int32)
    rr = None if rows is None else _c(rows, np.int64)
    n = lg.shape[0]
    out = np.empty((n, k), np.int32)
    nt = n_threads or os.cpu_count() or 1
    lib().orc_topk(_p(lg), lg.shape[1], _p(sl), _p(cu), sl.shape[0], int(causal), _p(rr), n,
                   int(k), _p(out), int(nt))
    return out


# --- compressor front end --------------------------------------------------------------

def exp_neg(a: float) -> float:
    return float(lib().orc_exp_neg(float(a)))


def rmsnorm128(x, gamma=None, eps=1e-6):
    x = _c(x, np.float32)
    g = _c(np.ones(128) if gamma is None else gamma, np.float32)
    y = np.empty(128, np.float32)
    lib().orc_rmsnorm128(_p(x), _p(g), C.c_float(eps), _p(y))
    return y


def compress_pool128(k_raw, gate, lo, hi):
    """Pooled fp32 row of raw rows lo..hi (inclusive) of k_raw / gate (uint16 [N, 128])."""
    k_raw = _c(k_raw, np.uint16)
    gate = _c(gate, np.uint16)
    out = np.empty(128, np.float32)
    lib().orc_compress_pool128(_p(k_raw), _p(gate), k_raw.shape[1], int(lo), int(hi), _p(out))
    return out


def compress_k_store(pool, k_raw, gate, boundary, first, ratio, slot_mapping, positions, cos_sin,
                     rope, norm, dtype, num_pages, page_size, page_stride, gamma=None, beta=None,
                     eps=1e-6):
    """Writes the compressed entries into ``pool`` (uint8, in place); returns the rejected count."""
    assert pool.dtype == np.uint8 and pool.flags.c_contiguous
    k_raw = _c(k_raw, np.uint16)
    gate = _c(gate, np.uint16)
    bnd = _c(boundary, np.int64)
    fst = _c(first, np.int64)
    n = bnd.shape[0]
    slot = _c(slot_mapping, np.int64)
    pos = _c(positions if positions is not None else np.zeros(n), np.int32)
    cs = _c(cos_sin if cos_sin is not None else np.zeros((1, 64)), np.float32)
    g = _c(np.ones(128) if gamma is None else gamma, np.float32)
    b = _c(np.zeros(128) if beta is None else beta, np.float32)
    return lib().orc_compress_k_store(_p(k_raw), _p(gate), k_raw.shape[0], k_raw.shape[1], _p(bnd), _p(fst), n,
                                      int(ratio), _p(slot), _p(pos), _p(cs), cs.shape[0], int(rope),
                                      int(norm), _p(g), _p(b), C.c_float(eps), int(dtype), _p(pool),
                                      int(num_pages), int(page_size), int(page_stride))


def topk_cand(logits, seq_lens_k, cu_seqlens_q, causal, cand, n_cand, page_size, k, rows=None,
              n_threads=None):
    """Top-k over each query's candidate blocks (reading R17); logits as mqa_logits returns
    them for `rows` (all queries when None); cand int32 [T, cand_stride], n_cand int32 [T]."""
    lg = _c(logits, np.float64)
    sl = _c(seq_lens_k, np.int32)
    cu = _c(cu_seqlens_q, np.int32)
    cd = _c(cand, np.int32)
    nc = _c(n_cand, np.int32)
    rr = None if rows is None else _c(rows, np.int64)
    n = lg.shape[0]
    out = np.empty((n, k), np.int32)
    nt = n_threads or os.cpu_count() or 1
    lib().orc_topk_cand(_p(lg), lg.shape[1], _p(sl), _p(cu), sl.shape[0], int(causal), _p(rr), n,
                        _p(cd), cd.shape[1], _p(nc), int(page_size), int(k), _p(out), int(nt))
    return out
