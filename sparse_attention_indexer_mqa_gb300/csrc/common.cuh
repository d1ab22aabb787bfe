// common.cuh -- device helpers shared by the indexer kernels: bf16 unpacking, the e2m1 /
// e4m3 element encoders, the MX shared exponent, the paged-cache layout, status bits.
//
// Sources: vllm PR 60834 "Purpose" (MXFP4 cache: 4 blocks of 32 e2m1 + one E8M0 scale,
// 68 B/token; FP8: 132 B/token); vllm PR 53094 "Purpose" (the pre-processing steps).
#pragma once

#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/idx.h"

namespace idx {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void report(int32_t* status, int32_t bit) {
    if (status) atomicOr(status, bit);
}

// ---- programmatic dependent launch --------------------------------------------------------
// Every kernel of the library is launched so that it may start while the previous kernel in
// the stream finishes. Before pdl_wait() a kernel only reads caller inputs that no kernel of
// the path writes (lengths, page table, positions, RoPE table, bf16 q / k, head weights) and
// sets up shared and tensor memory; it writes nothing. pdl_wait() returns once the previous
// grid has completed and its memory is visible (at once when there is no such grid).
// pdl_launch_dependents() lets the next kernel start early. The scorers and the top-k issue it
// after their pdl_wait(); the pre-processing kernels (K store, Q quant, both, compressor),
// whose own work all follows their wait, issue it at entry, so that the scorer's prologue also
// overlaps the kernel before them. Either way every CTA of a kernel is resident before its
// dependent launches (no dependent can hold the resources a CTA of it still needs), and a
// kernel's pdl_wait() returning means its predecessor, and everything that one waited for,
// has completed.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialization (the kernel calls pdl_wait()) when pdl is
// true, else as an ordinary stream-ordered launch (the previous kernel has finished, and its
// writes are visible, before this one starts).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
    return launch_k(true, kernel, grid, block, smem, st, std::forward<Args>(args)...);
}

// bf16 pair in a 32-bit word -> two fp32 (exact)
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// e2m1 codes of eight block-scaled values (|v| < 8), packed two per byte (element 2i in the
// low nibble): the hardware conversion cvt.rn.satfinite.e2m1x2.f32, i.e. round to nearest,
// ties to even, saturating at 6, keeping the sign (a negative that rounds to zero is -0).
// vllm PR 60834 "Purpose" names this instruction for DeepSeek-V4's MXFP4 packing.
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
    uint32_t w;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        " mov.b32 %0, {b0, b1, b2, b3};\n}"
        : "=r"(w)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return w;
}

// e4m3 (fn) code of v: the hardware conversion, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_code(float v) {
    return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// OCP MX shared exponent: floor(log2 amax) - 2 read from the exponent field (leading
// mantissa bit for subnormals), clamped to [-127, 127]; amax == 0 gives -127.
__device__ __forceinline__ int mx_exponent(float amax) {
    uint32_t u = __float_as_uint(amax) & 0x7fffffffu;
    if (u == 0) return -127;
    int ef = (int)(u >> 23);
    int fl = ef > 0 ? ef - 127 : (31 - __clz((int)u)) - 149;
    int e = fl - 2;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-E as fp32 for E in [-127, 125] (always a normal number).
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// ---- paged cache layout (see idx.h) ------------------------------------------------------
// MXFP4: byte offset in a page of 16-byte chunk c (scale block c) of in-page token s.
__device__ __forceinline__ int mx_chunk_off(int P, int s, int c) {
    return P == 128 ? ((s >> 3) * 4 + c) * 128 + (s & 7) * 16
                    : (s >> 4) * 1024 + ((s >> 3) & 1) * 512 + c * 128 + (s & 7) * 16;
}
// MXFP4: byte offset of the 4 scale bytes (blocks 0..3, contiguous) of in-page token s.
__device__ __forceinline__ int mx_scale_off(int P, int s) {
    return P == 128 ? 8192 + (s & 31) * 16 + (s >> 5) * 4 : 4096 + (s & 15) * 16 + (s >> 4) * 4;
}
// FP8: byte offset of 16-byte chunk c (elements 16c..16c+15) of token s; scale offset.
__device__ __forceinline__ int f8_chunk_off(int s, int c) { return (s >> 3) * 1024 + c * 128 + (s & 7) * 16; }
__device__ __forceinline__ int f8_scale_off(int P, int s) { return 128 * P + 4 * s; }

// Keys visible to the i-th of nq queries of a sequence with seq_len keys.
__device__ __forceinline__ int64_t visible_keys(int64_t seq_len, int64_t nq, int64_t i, int causal) {
    int64_t v = causal ? seq_len - nq + i + 1 : seq_len;
    return v < 0 ? 0 : (v > seq_len ? seq_len : v);
}

// Sequence b owning global query row t (binary search over cu_seqlens_q[0..B]); -1 if none.
__device__ __forceinline__ int seq_of_query(const int32_t* cu, int B, int64_t t) {
    int lo = 0, hi = B;  // find b with cu[b] <= t < cu[b+1]
    if (t < cu[0] || t >= cu[B]) return -1;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

}  // namespace idx
