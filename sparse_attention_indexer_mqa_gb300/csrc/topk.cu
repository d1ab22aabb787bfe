// topk.cu -- per-query top-k over the indexer logits by radix select.
//
// vllm PR 60834 "Test Result / GPQA Diamond": the indexer keeps the top-k (1024) keys per
// query once the context exceeds top-k x compress ratio; vllm PR 53094 "Purpose" names the
// per-token topk_indices_buffer it fills. The set of the k largest logits is unique up to
// ties at the k-th value; this kernel returns the indices above the k-th value, then the
// indices equal to it, each group in increasing index order, so the result is
// deterministic.
//
// One CTA per query row. Logits are mapped to order-preserving uint32 keys; three
// histogram passes (11, 11, 10 bits, shared-memory atomics) fix the k-th key exactly; a
// final ordered compaction (block scans over tiles of 512) writes the indices. The row is
// read four times, the later passes mostly from L2.
#include "common.cuh"
#include "kernels.h"

namespace idx {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive sum scan over the CTA; `total` receives the CTA-wide sum.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* warp_sums, uint32_t& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        uint32_t s = lane < kWarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(kFull, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kWarps) warp_sums[lane] = s;
    }
    __syncthreads();
    const uint32_t add = w > 0 ? warp_sums[w - 1] : 0;
    total = warp_sums[kWarps - 1];
    __syncthreads();
    return x + add;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a) {
    __shared__ uint32_t hist[2048];
    __shared__ uint32_t warp_sums[kWarps];
    __shared__ uint32_t sel_bin, sel_above;

    const int64_t t = blockIdx.x;
    const int b = seq_of_query(a.cu_seqlens_q, a.B, t);
    int64_t vis = 0;
    if (b >= 0) {
        const int64_t q0 = a.cu_seqlens_q[b], nq = a.cu_seqlens_q[b + 1] - q0;
        vis = visible_keys(a.seq_lens_k[b], nq, t - q0, a.causal);
    }
    int32_t* out = a.out + t * a.k;
    const float* row = a.logits + t * a.ld;
    if (vis <= a.k) {
        for (int i = threadIdx.x; i < a.k; i += kThreads) out[i] = i < vis ? i : -1;
        return;
    }

    uint32_t prefix = 0, pmask = 0, remaining = (uint32_t)a.k;
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const uint32_t nb = pass == 2 ? 1024u : 2048u;
        for (uint32_t i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (int64_t i = threadIdx.x; i < vis; i += kThreads) {
            const uint32_t key = order_key(row[i]);
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
        }
        __syncthreads();
        // thread r owns the bins [nb - per*(r+1), nb - per*r), highest bins first
        const int per = (int)nb / kThreads;
        const int top = (int)nb - per * (int)threadIdx.x;
        uint32_t local = 0;
        for (int j = 1; j <= per; ++j) local += hist[top - j];
        uint32_t total;
        const uint32_t incl = block_scan(local, warp_sums, total);
        const uint32_t before = incl - local;
        if (before < remaining && remaining <= incl) {
            uint32_t run = before;
            for (int j = 1; j <= per; ++j) {
                const int bin = top - j;
                if (run + hist[bin] >= remaining) {
                    sel_bin = (uint32_t)bin;
                    sel_above = run;
                    break;
                }
                run += hist[bin];
            }
        }
        __syncthreads();
        prefix |= sel_bin << shift;
        pmask |= (nb - 1) << shift;
        remaining -= sel_above;
        __syncthreads();
    }

    // prefix is now the k-th largest key; `remaining` keys equal to it are still needed
    const uint32_t n_gt = (uint32_t)a.k - remaining;
    uint32_t base_gt = 0, base_eq = 0;
    for (int64_t i0 = 0; i0 < vis; i0 += kThreads) {
        const int64_t i = i0 + threadIdx.x;
        const uint32_t key = i < vis ? order_key(row[i]) : 0u;
        const bool gt = i < vis && key > prefix, eq = i < vis && key == prefix;
        const uint32_t packed = (gt ? 1u : 0u) | (eq ? 0x10000u : 0u);
        uint32_t tot;
        const uint32_t ex = block_scan(packed, warp_sums, tot) - packed;
        if (gt) out[base_gt + (ex & 0xffffu)] = (int32_t)i;
        if (eq) {
            const uint32_t r = base_eq + (ex >> 16);
            if (r < remaining) out[n_gt + r] = (int32_t)i;
        }
        base_gt += tot & 0xffffu;
        base_eq += tot >> 16;
    }
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    topk_kernel<<<(unsigned)a.T, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace idx
