// scorer_simt.cu -- paged MQA-logits scorer on the CUDA cores (one thread per key).
//
// logits[t, s] = sum_h w[t,h] * ReLU(q[t,h] . k[s]) over the dequantised operands, K read
// in place through the page table (vllm PR 57517 "Purpose" and "Performance and accuracy";
// vllm PR 60834 "Purpose": the scorer reads the paged cache in place, no gather).
//
// A CTA scores 128 keys of one query: Q is dequantised to fp32 in shared memory, each
// thread dequantises its key row into shared memory, then forms the H dot products with
// fp32 fused multiply-adds. Products of the dequantised values are exact in fp32; the sums
// are rounded fp32.
#include "common.cuh"
#include "kernels.h"

namespace idx {

namespace {

constexpr int kKeys = 128;
constexpr int kRowPad = 129;  // conflict-free column reads of the per-thread key rows

__device__ __forceinline__ float e2m1_value(uint32_t c) {
    const float m[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    float v = m[c & 7];
    return (c & 8) ? -v : v;
}

__device__ __forceinline__ float e4m3_value(uint32_t c) {
    __nv_fp8_e4m3 f;
    f.__x = (__nv_fp8_storage_t)c;
    return (float)f;
}

__device__ __forceinline__ float e8m0_value(uint32_t b) {
    // 2^(b-127); b = 0 is 2^-127 (subnormal)
    return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

template <int kDtype>
__global__ void __launch_bounds__(kKeys) scorer_simt_kernel(ScoreArgs a) {
    extern __shared__ float smem[];
    float* qf = smem;                      // [H][128]
    float* kf = smem + a.H * 128;          // [128][kRowPad]
    const int64_t t = blockIdx.x;
    const int b = seq_of_query(a.cu_seqlens_q, a.B, t);
    if (b < 0) return;
    const int64_t q0 = a.cu_seqlens_q[b];
    int64_t seq_len = a.seq_lens_k[b];
    if (seq_len > a.max_seq_len_k || seq_len < 0) {  // caller's bound broken: clamp, report
        if (threadIdx.x == 0 && blockIdx.y == 0) report(a.dev_status, IDX_STATUS_BAD_LEN);
        seq_len = seq_len < 0 ? 0 : a.max_seq_len_k;
    }
    const int64_t vis = visible_keys(seq_len, a.cu_seqlens_q[b + 1] - q0, t - q0, a.causal);
    const int64_t s0 = (int64_t)blockIdx.y * kKeys;
    if (s0 >= vis) return;
    const int H = a.H;

    const int Hq = (H + 7) & ~7;
    for (int i = threadIdx.x; i < H * 128; i += kKeys) {
        const int h = i >> 7, d = i & 127;
        float v;
        if (kDtype == IDX_MXFP4) {
            // canonical Q image (see idx.h): chunk d/32 of head h, byte (d%32)/2
            const uint32_t byte = a.q_codes[t * Hq * 64 + ((h >> 3) * 4 + (d >> 5)) * 128 + (h & 7) * 16 + ((d & 31) >> 1)];
            const uint32_t sb = a.q_scales[t * 512 + (h & 31) * 16 + (h >> 5) * 4 + (d >> 5)];
            v = e2m1_value((d & 1) ? byte >> 4 : byte & 15) * e8m0_value(sb);
        } else {
            v = e4m3_value(a.q_codes[t * Hq * 128 + ((h >> 3) * 8 + (d >> 4)) * 128 + (h & 7) * 16 + (d & 15)]);
        }
        qf[i] = v;
    }

    const int64_t s = s0 + threadIdx.x;
    bool ok = s < vis;
    float kscale = 1.0f;
    if (ok) {
        const int P = a.page_size;
        const int32_t page = a.page_table[(int64_t)b * a.pt_stride + s / P];
        if (page < 0 || page >= a.num_pages) {
            report(a.dev_status, IDX_STATUS_BAD_PAGE);
            ok = false;
        } else {
            const uint8_t* base = a.pool + (int64_t)page * a.page_stride;
            const int r = (int)(s % P);
            float* kr = kf + threadIdx.x * kRowPad;
            if (kDtype == IDX_MXFP4) {
                const uint32_t sc = *reinterpret_cast<const uint32_t*>(base + mx_scale_off(P, r));
                for (int c = 0; c < 4; ++c) {
                    const uint4 ch = *reinterpret_cast<const uint4*>(base + mx_chunk_off(P, r, c));
                    const uint32_t wds[4] = {ch.x, ch.y, ch.z, ch.w};
                    const float scale = e8m0_value((sc >> (8 * c)) & 255u);
                    for (int wi = 0; wi < 4; ++wi)
                        for (int n = 0; n < 8; ++n)
                            kr[32 * c + 8 * wi + n] = e2m1_value((wds[wi] >> (4 * n)) & 15u) * scale;
                }
            } else {
                for (int c = 0; c < 8; ++c) {
                    const uint4 ch = *reinterpret_cast<const uint4*>(base + f8_chunk_off(r, c));
                    const uint32_t wds[4] = {ch.x, ch.y, ch.z, ch.w};
                    for (int wi = 0; wi < 4; ++wi)
                        for (int n = 0; n < 4; ++n)
                            kr[16 * c + 4 * wi + n] = e4m3_value((wds[wi] >> (8 * n)) & 255u);
                }
                kscale = *reinterpret_cast<const float*>(base + f8_scale_off(P, r));
            }
        }
    }
    __syncthreads();
    if (!ok) return;
    const float* kr = kf + threadIdx.x * kRowPad;
    float logit = 0.0f;
    for (int h = 0; h < H; ++h) {
        const float* qh = qf + h * 128;
        float dot = 0.0f;
#pragma unroll 8
        for (int d = 0; d < 128; ++d) dot = fmaf(qh[d], kr[d], dot);
        logit = fmaf(a.w[t * H + h], fmaxf(dot, 0.0f), logit);
    }
    a.logits[t * a.ld + s] = logit * kscale;
}

}  // namespace

cudaError_t launch_scorer_simt(const ScoreArgs& a, cudaStream_t st) {
    if (a.T == 0 || a.max_seq_len_k == 0) return cudaSuccess;
    const size_t smem = (size_t)(a.H * 128 + kKeys * kRowPad) * sizeof(float);
    dim3 grid((unsigned)a.T, (unsigned)((a.max_seq_len_k + kKeys - 1) / kKeys));
    cudaError_t e;
    if (a.dtype == IDX_MXFP4) {
        e = cudaFuncSetAttribute(scorer_simt_kernel<IDX_MXFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        scorer_simt_kernel<IDX_MXFP4><<<grid, kKeys, smem, st>>>(a);
    } else {
        e = cudaFuncSetAttribute(scorer_simt_kernel<IDX_FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        scorer_simt_kernel<IDX_FP8><<<grid, kKeys, smem, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace idx
