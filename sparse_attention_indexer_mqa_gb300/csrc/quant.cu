// quant.cu -- the fused K store (LayerNorm -> RoPE -> MXFP4/FP8 -> paged store) and the
// Q quant (RoPE -> MXFP4/FP8, weight fold) kernels, alone or together in one launch.
//
// vllm PR 53094 "Purpose" lists the pre-processing of one indexer layer as five launches
// (LayerNorm on k; RoPE on q and k; per-token-group FP8 quantisation of q; fold of the
// q scale into the weights; FP8 quantisation of k plus the paged cache write) and replaces
// them with one fused kernel; vllm PR 60834 "Changes / K write" and "Q quant" do the same
// for MXFP4 (norm -> RoPE -> MXFP4 -> preshuffled pages; RoPE -> MXFP4 with the softmax
// and head scales folded into fp32 weights). Each of the two steps is one kernel, and
// qk_prep_kernel runs both in a single launch (one block range each). compress_kernel is the
// DeepSeek-V4 form of the K store (vllm PR 60834 "Changes / K write": the indexer's own
// compressor pools raw rows, then RMSNorm -> RoPE -> MXFP4 -> store in one kernel, nothing
// before the norm reaching memory): one entry per compress-ratio boundary token.
//
// Mapping: 16 threads per 128-element row, 8 consecutive elements (one 16-byte load of
// bf16) per thread; a 256-thread CTA handles 16 K rows, or 32 Q rows of one token (two per
// 16 threads, sharing the position and the RoPE table row). Reductions use a fixed tree (group
// of 8 in registers, then xor-butterfly over the 16 lanes), so the result does not depend
// on the launch shape. Every float operation is an explicitly rounded intrinsic (no FMA
// contraction), which makes the bytes reproducible on any IEEE implementation.
#include "common.cuh"
#include "kernels.h"

namespace idx {

namespace {

constexpr int kRowsPerCta = 16;
constexpr int kThreads = 16 * kRowsPerCta;
constexpr int kQHeadsPerCta = 2 * kRowsPerCta;  // Q: two rows per 16 lanes

__device__ __forceinline__ float sum8(const float* e) {
    float a = __fadd_rn(e[0], e[1]);
    float b = __fadd_rn(e[2], e[3]);
    float c = __fadd_rn(e[4], e[5]);
    float d = __fadd_rn(e[6], e[7]);
    return __fadd_rn(__fadd_rn(a, b), __fadd_rn(c, d));
}

// Sum over the 128 values of a row held 8 per lane by 16 lanes (identical in every lane).
__device__ __forceinline__ float row_sum(const float* e) {
    float g = sum8(e);
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) g = __fadd_rn(g, __shfl_xor_sync(kFull, g, off));
    return g;
}

// LayerNorm with biased variance and rstd = 1 / sqrt(var + eps), each op rounded.
__device__ __forceinline__ void layernorm(float* x, int l16, const float* gamma, const float* beta,
                                          float eps) {
    const float inv_d = 0.0078125f;
    float mean = __fmul_rn(row_sum(x), inv_d);
    float d[8], sq[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        d[i] = __fsub_rn(x[i], mean);
        sq[i] = __fmul_rn(d[i], d[i]);
    }
    float var = __fmul_rn(row_sum(sq), inv_d);
    float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float g = gamma ? __ldg(gamma + 8 * l16 + i) : 1.0f;
        float b = beta ? __ldg(beta + 8 * l16 + i) : 0.0f;
        x[i] = __fadd_rn(__fmul_rn(__fmul_rn(d[i], rstd), g), b);
    }
}

// RMSNorm: x * (1 / sqrt(mean(x^2) + eps)) * gamma, each op rounded, the same fixed tree.
__device__ __forceinline__ void rmsnorm(float* x, int l16, const float* gamma, float eps) {
    const float inv_d = 0.0078125f;
    float sq[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sq[i] = __fmul_rn(x[i], x[i]);
    const float ms = __fmul_rn(row_sum(sq), inv_d);
    const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float g = gamma ? __ldg(gamma + 8 * l16 + i) : 1.0f;
        x[i] = __fmul_rn(__fmul_rn(x[i], rstd), g);
    }
}

// exp(a) for a <= 0 by Cody and Waite's argument reduction and a degree-7 Taylor polynomial
// (one fused multiply-add per step): n = rint(a log2 e), f = (a - n ln2_hi) - n ln2_lo with
// ln2_hi holding 16 significant bits so that n ln2_hi is exact, e^f by Horner's rule, the
// result e^f * 2^n. At most 0.86 ulp from exp over [-87, 0]; 0 below -87 (and for NaN).
// Branch-free: the argument is clamped to -87 and the result selected. rint is the add and
// subtract of 1.5 * 2^23 (round to nearest even, exact for |t| < 2^22), and the bits of that
// sum hold n, so 2^n = bits * 2^23 + bits(1.0) in one integer multiply-add.
__device__ __forceinline__ float exp_neg(float a) {
    const float ac = fmaxf(a, -87.0f);
    const float big = __fadd_rn(__fmul_rn(ac, 1.44269504f), 12582912.0f);
    const float n = __fsub_rn(big, 12582912.0f);
    float f = __fmaf_rn(-n, 0.693145752f, ac);
    f = __fmaf_rn(-n, 1.42860677e-06f, f);
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, f, 1.0f / 720.0f);
    p = __fmaf_rn(p, f, 1.0f / 120.0f);
    p = __fmaf_rn(p, f, 1.0f / 24.0f);
    p = __fmaf_rn(p, f, 1.0f / 6.0f);
    p = __fmaf_rn(p, f, 0.5f);
    p = __fmaf_rn(p, f, 1.0f);
    p = __fmaf_rn(p, f, 1.0f);
    const float two_n = __uint_as_float(__float_as_uint(big) * (1u << 23) + 0x3f800000u);
    const float r = __fmul_rn(p, two_n);
    return a > -87.0f ? r : 0.0f;
}

// elementwise max of two pairs of bf16 (exact; a NaN operand yields the other)
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// RoPE on dims 0..63 (lanes 0..7 of the row). NeoX pairs dims (i, i+32): lane l < 4 holds
// the first element of its pairs, lane l+4 the second. Interleaved pairs (2i, 2i+1) lie
// inside one lane. cs = the table row [cos f0..f0+31, sin f0..f0+31] (16-byte aligned). The
// table loads and the rotation are apart, so that rows of one position share the loads.
struct RopeCS {
    float c[8], sn[8];
};

__device__ __forceinline__ void rope_load(int l16, const float* cs, int mode, RopeCS& r) {
    if (mode == IDX_ROPE_NEOX) {
        if (l16 < 8) {
            const int f0 = (8 * l16) & 31;
            const float4 c0 = __ldg(reinterpret_cast<const float4*>(cs + f0));
            const float4 c1 = __ldg(reinterpret_cast<const float4*>(cs + f0 + 4));
            const float4 s0 = __ldg(reinterpret_cast<const float4*>(cs + 32 + f0));
            const float4 s1 = __ldg(reinterpret_cast<const float4*>(cs + 32 + f0 + 4));
            r.c[0] = c0.x; r.c[1] = c0.y; r.c[2] = c0.z; r.c[3] = c0.w;
            r.c[4] = c1.x; r.c[5] = c1.y; r.c[6] = c1.z; r.c[7] = c1.w;
            r.sn[0] = s0.x; r.sn[1] = s0.y; r.sn[2] = s0.z; r.sn[3] = s0.w;
            r.sn[4] = s1.x; r.sn[5] = s1.y; r.sn[6] = s1.z; r.sn[7] = s1.w;
        }
    } else if (mode == IDX_ROPE_INTERLEAVED) {
        if (l16 < 8) {
            const float4 c4 = __ldg(reinterpret_cast<const float4*>(cs + 4 * l16));
            const float4 s4 = __ldg(reinterpret_cast<const float4*>(cs + 32 + 4 * l16));
            r.c[0] = c4.x; r.c[1] = c4.y; r.c[2] = c4.z; r.c[3] = c4.w;
            r.sn[0] = s4.x; r.sn[1] = s4.y; r.sn[2] = s4.z; r.sn[3] = s4.w;
        }
    }
}

__device__ __forceinline__ void rope_apply(float* x, int l16, int mode, const RopeCS& r) {
    if (mode == IDX_ROPE_NEOX) {
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) p[i] = __shfl_xor_sync(kFull, x[i], 4);
        if (l16 < 8) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (l16 < 4) x[i] = __fsub_rn(__fmul_rn(x[i], r.c[i]), __fmul_rn(p[i], r.sn[i]));  // a' = ac - bs
                else         x[i] = __fadd_rn(__fmul_rn(x[i], r.c[i]), __fmul_rn(p[i], r.sn[i]));  // b' = bc + as
            }
        }
    } else if (mode == IDX_ROPE_INTERLEAVED) {
        if (l16 < 8) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float a = x[2 * q], b = x[2 * q + 1];
                x[2 * q] = __fsub_rn(__fmul_rn(a, r.c[q]), __fmul_rn(b, r.sn[q]));
                x[2 * q + 1] = __fadd_rn(__fmul_rn(b, r.c[q]), __fmul_rn(a, r.sn[q]));
            }
        }
    }
}

// One row: the partner elements are exchanged before the table loads (fewer live registers).
__device__ __forceinline__ void rope(float* x, int l16, const float* cs, int mode) {
    if (mode == IDX_ROPE_NEOX) {
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) p[i] = __shfl_xor_sync(kFull, x[i], 4);
        if (l16 < 8) {
            RopeCS r;
            rope_load(l16, cs, mode, r);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (l16 < 4) x[i] = __fsub_rn(__fmul_rn(x[i], r.c[i]), __fmul_rn(p[i], r.sn[i]));  // a' = ac - bs
                else         x[i] = __fadd_rn(__fmul_rn(x[i], r.c[i]), __fmul_rn(p[i], r.sn[i]));  // b' = bc + as
            }
        }
    } else if (mode == IDX_ROPE_INTERLEAVED) {
        RopeCS r;
        rope_load(l16, cs, mode, r);
        rope_apply(x, l16, mode, r);
    }
}

// MXFP4: this lane's 8 elements -> one 32-bit word of nibbles (element 2m low, 2m+1 high
// of byte m) and the E8M0 byte of its 32-element block (lanes 4b..4b+3 = block b).
__device__ __forceinline__ void mx_quant(const float* x, uint32_t& word, uint32_t& sbyte) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    const int e = mx_exponent(amax);
    const float inv = pow2_neg(e);
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(x[i], inv);
    word = e2m1x8(v);
    sbyte = (uint32_t)(e + 127);
}

// FP8: scale = max(amax, 1e-10) / 448 over the 128 values; codes e4m3(x / scale).
__device__ __forceinline__ void f8_quant(const float* x, uint32_t& lo, uint32_t& hi, float& scale) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int off = 1; off <= 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
    scale = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
    lo = hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) lo |= e4m3_code(__fdiv_rn(x[i], scale)) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) hi |= e4m3_code(__fdiv_rn(x[4 + i], scale)) << (8 * i);
}

// eight bf16 (one 16-byte load) -> fp32
__device__ __forceinline__ void unpack8(const uint4 v, float* x) {
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
    x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
    x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
    x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

// Quantise a row held 8 values per lane by 16 lanes and, if ok, write its codes and scale(s)
// into slot s of the page at base. Every lane of the row takes part (shuffles).
template <int kDtype>
__device__ __forceinline__ void quant_store(const float* x, int l16, bool ok, uint8_t* base, int page_size,
                                            int s) {
    if (kDtype == IDX_MXFP4) {
        uint32_t word, sbyte;
        mx_quant(x, word, sbyte);
        pdl_wait();  // the cache may still be read by the previous kernel
        // gather the 4 words of a 16-byte chunk (= one scale block) into its first lane
        uint32_t w1 = __shfl_down_sync(kFull, word, 1);
        uint32_t w2 = __shfl_down_sync(kFull, word, 2);
        uint32_t w3 = __shfl_down_sync(kFull, word, 3);
        uint32_t s1 = __shfl_down_sync(kFull, sbyte, 4);
        uint32_t s2 = __shfl_down_sync(kFull, sbyte, 8);
        uint32_t s3 = __shfl_down_sync(kFull, sbyte, 12);
        if (ok && (l16 & 3) == 0) {
            *reinterpret_cast<uint4*>(base + mx_chunk_off(page_size, s, l16 >> 2)) =
                make_uint4(word, w1, w2, w3);
        }
        if (ok && l16 == 0) {
            *reinterpret_cast<uint32_t*>(base + mx_scale_off(page_size, s)) =
                sbyte | (s1 << 8) | (s2 << 16) | (s3 << 24);
        }
    } else {
        uint32_t lo, hi;
        float scale;
        f8_quant(x, lo, hi, scale);
        pdl_wait();
        uint32_t plo = __shfl_down_sync(kFull, lo, 1);
        uint32_t phi = __shfl_down_sync(kFull, hi, 1);
        if (ok && (l16 & 1) == 0) {
            *reinterpret_cast<uint4*>(base + f8_chunk_off(s, l16 >> 1)) = make_uint4(lo, hi, plo, phi);
        }
        if (ok && l16 == 0) *reinterpret_cast<float*>(base + f8_scale_off(page_size, s)) = scale;
    }
}

// K store of the 16 rows of block `blk` (one row per 16 lanes).
template <int kDtype>
__device__ __forceinline__ void k_store_rows(const KStoreArgs& a, int64_t blk) {
    const int l16 = threadIdx.x & 15;
    const int64_t row = blk * kRowsPerCta + (threadIdx.x >> 4);
    const bool in = row < a.n_rows;
    // the slot, the position and the K row are independent loads: issue them together
    const int64_t slot = in ? __ldg(a.slot_mapping + row) : -1;
    int32_t pos = (in && a.rope != IDX_ROPE_NONE) ? __ldg(a.positions + row) : 0;
    const uint4 raw = in ? __ldg(reinterpret_cast<const uint4*>(a.k + row * a.k_row_stride + 8 * l16))
                         : make_uint4(0, 0, 0, 0);
    bool ok = in && slot >= 0;
    const int lp = a.page_size == 128 ? 7 : 6;  // page sizes are 64 or 128
    const int64_t page = ok ? slot >> lp : 0;
    const int s = ok ? (int)(slot & (a.page_size - 1)) : 0;
    if (ok && page >= a.num_pages) {
        if (l16 == 0) report(a.dev_status, IDX_STATUS_BAD_SLOT);
        ok = false;
    }
    if (a.rope != IDX_ROPE_NONE && ok && (pos < 0 || pos >= a.max_pos)) {
        if (l16 == 0) report(a.dev_status, IDX_STATUS_BAD_POS);
        ok = false;
    }
    if (!ok) pos = 0;
    // every lane keeps going (zeros for skipped rows) so that the shuffles stay converged
    float x[8];
    unpack8(ok ? raw : make_uint4(0, 0, 0, 0), x);
    if (a.apply_norm) layernorm(x, l16, a.gamma, a.beta, a.eps);
    if (a.rope != IDX_ROPE_NONE) rope(x, l16, a.cos_sin + (int64_t)pos * 64, a.rope);

    quant_store<kDtype>(x, l16, ok, a.pool + page * a.page_stride, a.page_size, s);  // 64-bit page rebasing
}

// Compressed K store of the 16 entries of block `blk` (one entry per 16 lanes, 8 dims per
// lane). Entry e pools the raw rows lo..hi, hi = boundary[e], lo = max(first[e], hi - 2r + 1):
// per dimension m = max of the window's gates, e_i = exp(g_i - m), S = sum e_i and
// P = sum e_i x_i in row order (P by fused multiply-adds), pooled = P / S; then the norm
// (none, LayerNorm or RMSNorm), RoPE at positions[e], quantisation and the paged write.
template <int kDtype>
__device__ __forceinline__ void compress_rows(const CompressArgs& a, int64_t blk) {
    const int l16 = threadIdx.x & 15;
    const int64_t e = blk * kRowsPerCta + (threadIdx.x >> 4);
    const bool in = e < a.n_entries;
    const int64_t slot = in ? __ldg(a.slot_mapping + e) : -1;
    int64_t hi = in ? __ldg(a.boundary + e) : 0;
    const int64_t fst = in ? __ldg(a.first + e) : 0;
    int32_t pos = (in && a.rope != IDX_ROPE_NONE) ? __ldg(a.positions + e) : 0;
    bool ok = in && slot >= 0;
    const int lp = a.page_size == 128 ? 7 : 6;  // page sizes are 64 or 128
    const int64_t page = ok ? slot >> lp : 0;
    const int s = ok ? (int)(slot & (a.page_size - 1)) : 0;
    if (ok && page >= a.num_pages) {
        if (l16 == 0) report(a.dev_status, IDX_STATUS_BAD_SLOT);
        ok = false;
    }
    if (ok && (fst < 0 || fst > hi || hi >= a.n_raw)) {
        if (l16 == 0) report(a.dev_status, IDX_STATUS_BAD_LEN);
        ok = false;
    }
    if (a.rope != IDX_ROPE_NONE && ok && (pos < 0 || pos >= a.max_pos)) {
        if (l16 == 0) report(a.dev_status, IDX_STATUS_BAD_POS);
        ok = false;
    }
    if (!ok) pos = 0;
    int64_t lo = hi - 2 * (int64_t)a.ratio + 1;
    if (lo < fst) lo = fst;
    if (!ok) lo = 0, hi = -1;  // no rows: the lanes still reach the shuffles below

    float x[8];
    if (ok) {
        const uint4* gr = reinterpret_cast<const uint4*>(a.gate + lo * a.row_stride) + l16;
        const uint4* kr = reinterpret_cast<const uint4*>(a.k_raw + lo * a.row_stride) + l16;
        const int64_t step = a.row_stride / 8;  // uint4 per row
        const int rows = (int)(hi - lo + 1);    // 1 .. 2 * ratio
        // pass 1: the window's gate maximum per dimension, on packed bf16 pairs
        uint4 mx = __ldg(gr);
        for (int i = 1; i < rows; ++i) {
            const uint4 g = __ldg(gr + i * step);
            mx.x = bf16x2_max(mx.x, g.x); mx.y = bf16x2_max(mx.y, g.y);
            mx.z = bf16x2_max(mx.z, g.z); mx.w = bf16x2_max(mx.w, g.w);
        }
        float m[8];
        unpack8(mx, m);
        // pass 2: weights, their sum and the weighted sum, rows in order; the next row's
        // loads are issued before this row's arithmetic
        float S[8], P[8];
#pragma unroll
        for (int d = 0; d < 8; ++d) S[d] = P[d] = 0.0f;
        uint4 gn = __ldg(gr), vn = __ldg(kr);
        for (int i = 0; i < rows; ++i) {
            const uint4 gc = gn, vc = vn;
            if (i + 1 < rows) {
                gn = __ldg(gr + (i + 1) * step);
                vn = __ldg(kr + (i + 1) * step);
            }
            float g[8], v[8];
            unpack8(gc, g);
            unpack8(vc, v);
#pragma unroll
            for (int d = 0; d < 8; ++d) {
                const float w = exp_neg(__fsub_rn(g[d], m[d]));
                S[d] = __fadd_rn(S[d], w);
                P[d] = __fmaf_rn(w, v[d], P[d]);
            }
        }
#pragma unroll
        for (int d = 0; d < 8; ++d) x[d] = __fdiv_rn(P[d], S[d]);
    } else {
#pragma unroll
        for (int d = 0; d < 8; ++d) x[d] = 0.0f;
    }
    if (a.norm == 1) layernorm(x, l16, a.gamma, a.beta, a.eps);
    else if (a.norm == 2) rmsnorm(x, l16, a.gamma, a.eps);
    if (a.rope != IDX_ROPE_NONE) rope(x, l16, a.cos_sin + (int64_t)pos * 64, a.rope);
    quant_store<kDtype>(x, l16, ok, a.pool + page * a.page_stride, a.page_size, s);
}

// Quantise and store Q row (t, h) held 8 values per lane by 16 lanes (x after RoPE); w_in is
// the row's head weight (lane 0). Heads past H write the zero/neutral padding of the
// tensor-core image (see idx.h for the layout); a real row whose position was rejected (ok
// false) writes nothing.
template <int kDtype>
__device__ __forceinline__ void q_store_row(const QQuantArgs& a, int64_t t, int h, int Hq, bool real, bool ok,
                                            const float* x, float w_in) {
    const int l16 = threadIdx.x & 15;
    const int64_t row = t * a.H + h;  // index of (t, h) in q, w_in, w_out
    if (kDtype == IDX_MXFP4) {
        uint32_t word, sbyte;
        mx_quant(x, word, sbyte);
        pdl_wait();  // the Q image and weights may still be read by the previous kernel
        const uint32_t s1 = __shfl_down_sync(kFull, sbyte, 4);
        const uint32_t s2 = __shfl_down_sync(kFull, sbyte, 8);
        const uint32_t s3 = __shfl_down_sync(kFull, sbyte, 12);
        // gather each 16-byte chunk (4 lanes' words) into its first lane
        const uint32_t w1 = __shfl_down_sync(kFull, word, 1);
        const uint32_t w2 = __shfl_down_sync(kFull, word, 2);
        const uint32_t w3 = __shfl_down_sync(kFull, word, 3);
        if (ok || !real) {
            // canonical image: 8-head groups of [4 chunks][8 heads][16 B]
            uint8_t* img = a.q_codes + t * Hq * 64 + ((h >> 3) * 4 + (l16 >> 2)) * 128 + (h & 7) * 16;
            if ((l16 & 3) == 0)
                *reinterpret_cast<uint4*>(img) = real ? make_uint4(word, w1, w2, w3) : make_uint4(0, 0, 0, 0);
            if (l16 == 0) {
                uint8_t* atom = reinterpret_cast<uint8_t*>(a.q_scales) + t * 512 + (h & 31) * 16 + (h >> 5) * 4;
                *reinterpret_cast<uint32_t*>(atom) = real ? (sbyte | (s1 << 8) | (s2 << 16) | (s3 << 24)) : 0x7f7f7f7fu;
                if (real) a.w_out[row] = __fmul_rn(w_in, a.fold);
            }
        }
    } else {
        uint32_t lo, hi;
        float scale;
        f8_quant(x, lo, hi, scale);
        pdl_wait();
        const uint32_t plo = __shfl_down_sync(kFull, lo, 1);
        const uint32_t phi = __shfl_down_sync(kFull, hi, 1);
        if (ok || !real) {
            uint8_t* img = a.q_codes + t * Hq * 128 + ((h >> 3) * 8 + (l16 >> 1)) * 128 + (h & 7) * 16;
            if ((l16 & 1) == 0)
                *reinterpret_cast<uint4*>(img) = real ? make_uint4(lo, hi, plo, phi) : make_uint4(0, 0, 0, 0);
            if (l16 == 0 && real) {
                if (a.q_scales) reinterpret_cast<float*>(a.q_scales)[row] = scale;
                a.w_out[row] = __fmul_rn(__fmul_rn(w_in, a.fold), scale);
            }
        }
    }
}

// Q rows: CTA (t, y) takes token t's heads hpc*y .. hpc*y + hpc-1 of the Hq = H rounded up to
// 8 heads, hpc = 16 (one row per 16 lanes) or 32 (two: heads h and h + 16, whose loads -- the
// two rows, their weights, the position and the RoPE table row they share -- all go out
// before either row is worked on; more rows in flight per SM, a longer chain per CTA). Hq is
// a multiple of 8, so the rows of a warp are live together.
template <int kDtype>
__device__ __forceinline__ void q_quant_rows(const QQuantArgs& a, int64_t t, int y, int hpc) {
    const int l16 = threadIdx.x & 15;
    const int Hq = (a.H + 7) & ~7;
    const int h0 = y * hpc + (threadIdx.x >> 4), h1 = h0 + 16;
    if (h0 >= Hq) return;
    const bool two = hpc == kQHeadsPerCta && h1 < Hq;
    const bool real0 = h0 < a.H, real1 = two && h1 < a.H;  // real1 implies real0
    const int64_t row0 = t * a.H + h0, row1 = t * a.H + h1;
    const uint4 raw0 = real0 ? __ldg(reinterpret_cast<const uint4*>(a.q + row0 * 128 + 8 * l16))
                             : make_uint4(0, 0, 0, 0);
    const uint4 raw1 = real1 ? __ldg(reinterpret_cast<const uint4*>(a.q + row1 * 128 + 8 * l16))
                             : make_uint4(0, 0, 0, 0);
    const float w0 = (real0 && l16 == 0) ? __ldg(a.w_in + row0) : 0.0f;
    const float w1 = (real1 && l16 == 0) ? __ldg(a.w_in + row1) : 0.0f;
    int32_t pos = (real0 && a.rope != IDX_ROPE_NONE) ? __ldg(a.positions + t) : 0;
    bool pos_ok = true;
    if (a.rope != IDX_ROPE_NONE && real0 && (pos < 0 || pos >= a.max_pos)) {
        if (l16 == 0) report(a.dev_status, IDX_STATUS_BAD_POS);
        pos_ok = false;
    }
    const bool ok0 = real0 && pos_ok, ok1 = real1 && pos_ok;
    if (!ok0) pos = 0;  // a rejected or padding row is zeros, rotated by the table's row 0
    RopeCS cs;
    if (a.rope != IDX_ROPE_NONE) rope_load(l16, a.cos_sin + (int64_t)pos * 64, a.rope, cs);
    float x[8];
    unpack8(ok0 ? raw0 : make_uint4(0, 0, 0, 0), x);
    if (a.rope != IDX_ROPE_NONE) rope_apply(x, l16, a.rope, cs);
    q_store_row<kDtype>(a, t, h0, Hq, real0, ok0, x, w0);
    if (two) {
        unpack8(ok1 ? raw1 : make_uint4(0, 0, 0, 0), x);
        if (a.rope != IDX_ROPE_NONE) rope_apply(x, l16, a.rope, cs);
        q_store_row<kDtype>(a, t, h1, Hq, real1, ok1, x, w1);
    }
}

// The pre-processing kernels let their dependents launch at entry (see common.cuh): all their
// own work follows their wait, and the next kernel's prologue then overlaps the one before.
template <int kDtype>
__global__ void __launch_bounds__(kThreads) k_store_kernel(KStoreArgs a) {
    pdl_launch_dependents();
    k_store_rows<kDtype>(a, blockIdx.x);
}

template <int kDtype>
__global__ void __launch_bounds__(kThreads) q_quant_kernel(QQuantArgs a, int hpc) {
    pdl_launch_dependents();
    q_quant_rows<kDtype>(a, blockIdx.x, blockIdx.y, hpc);
}

// K store and Q quant in one launch: blocks [0, nk) store K rows, the rest quantise Q (block
// nk + t*ny + y takes token t's head block y). The two halves touch disjoint buffers.
template <int kDtype>
__global__ void __launch_bounds__(kThreads) qk_prep_kernel(KStoreArgs ka, QQuantArgs qa, int64_t nk, int ny,
                                                           int hpc) {
    pdl_launch_dependents();
    const int64_t b = blockIdx.x;
    if (b < nk) {
        k_store_rows<kDtype>(ka, b);
    } else {
        // ny = 1..4 and the grid is below 2^31: a 32-bit divide by a constant
        const uint32_t i = (uint32_t)(b - nk);
        const uint32_t t = ny == 1 ? i : (ny == 2 ? i >> 1 : (ny == 4 ? i >> 2 : i / 3u));
        q_quant_rows<kDtype>(qa, t, (int)(i - t * (uint32_t)ny), hpc);
    }
}

template <int kDtype>
__global__ void __launch_bounds__(kThreads) compress_kernel(CompressArgs a) {
    pdl_launch_dependents();
    compress_rows<kDtype>(a, blockIdx.x);
}

__global__ void debug_encode_kernel(int kind, const float* in, int64_t n, uint8_t* out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        float v = in[i];
        float v8[8] = {v, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        out[i] = (uint8_t)(kind == 0 ? (e2m1x8(v8) & 15u) : e4m3_code(v));
    }
}

}  // namespace

cudaError_t launch_k_store(const KStoreArgs& a, cudaStream_t st) {
    if (a.n_rows == 0) return cudaSuccess;
    const int64_t grid = (a.n_rows + kRowsPerCta - 1) / kRowsPerCta;
    return a.dtype == IDX_MXFP4 ? launch_pdl(k_store_kernel<IDX_MXFP4>, dim3((unsigned)grid), dim3(kThreads), 0, st, a)
                                : launch_pdl(k_store_kernel<IDX_FP8>, dim3((unsigned)grid), dim3(kThreads), 0, st, a);
}

namespace {

// Heads per Q CTA: 16 while the Q CTAs fit on the GPU at once (one row per 16 lanes, the
// shortest chain: decode steps), else 32 (two rows per 16 lanes, more rows in flight: prefill).
// Measured: 8192 tokens x 32 heads 40.5 -> 33.5 us with 32; 64 tokens 1.3 -> 1.6 us.
int q_heads_per_cta(int64_t T, int Hq) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 1;
    const int64_t ctas16 = T * ((Hq + kRowsPerCta - 1) / kRowsPerCta);
    return ctas16 <= (int64_t)4 * sms ? kRowsPerCta : kQHeadsPerCta;
}

}  // namespace

cudaError_t launch_q_quant(const QQuantArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    const int Hq = (a.H + 7) & ~7;
    const int hpc = q_heads_per_cta(a.T, Hq);
    const dim3 grid((unsigned)a.T, (unsigned)((Hq + hpc - 1) / hpc));
    return a.dtype == IDX_MXFP4 ? launch_pdl(q_quant_kernel<IDX_MXFP4>, grid, dim3(kThreads), 0, st, a, hpc)
                                : launch_pdl(q_quant_kernel<IDX_FP8>, grid, dim3(kThreads), 0, st, a, hpc);
}

cudaError_t launch_qk_prep(const KStoreArgs& ka, const QQuantArgs& qa, cudaStream_t st) {
    const int64_t nk = (ka.n_rows + kRowsPerCta - 1) / kRowsPerCta;
    const int Hq = (qa.H + 7) & ~7;
    const int hpc = q_heads_per_cta(qa.T, Hq);
    const int ny = (Hq + hpc - 1) / hpc;
    const int64_t grid = nk + qa.T * ny;
    if (grid == 0) return cudaSuccess;
    if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
    return ka.dtype == IDX_MXFP4
               ? launch_pdl(qk_prep_kernel<IDX_MXFP4>, dim3((unsigned)grid), dim3(kThreads), 0, st, ka, qa, nk, ny, hpc)
               : launch_pdl(qk_prep_kernel<IDX_FP8>, dim3((unsigned)grid), dim3(kThreads), 0, st, ka, qa, nk, ny, hpc);
}

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t st) {
    if (a.n_entries == 0) return cudaSuccess;
    const int64_t grid = (a.n_entries + kRowsPerCta - 1) / kRowsPerCta;
    if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
    return a.dtype == IDX_MXFP4 ? launch_pdl(compress_kernel<IDX_MXFP4>, dim3((unsigned)grid), dim3(kThreads), 0, st, a)
                                : launch_pdl(compress_kernel<IDX_FP8>, dim3((unsigned)grid), dim3(kThreads), 0, st, a);
}

cudaError_t launch_debug_encode(int kind, const float* in, int64_t n, uint8_t* out, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 64) blocks = 152 * 64;
    debug_encode_kernel<<<(unsigned)blocks, 256, 0, st>>>(kind, in, n, out);
    return cudaGetLastError();
}

}  // namespace idx
