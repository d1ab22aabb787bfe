// topk.cu -- per-query top-k over the indexer logits by radix select.
//
// vllm PR 60834 "Test Result / GPQA Diamond": the indexer keeps the top-k (1024) keys per
// query once the context exceeds top-k x compress ratio; vllm PR 53094 "Purpose" names the
// per-token topk_indices_buffer it fills. The set of the k largest logits is unique up to
// ties at the k-th value; this kernel returns the indices above the k-th value, then the
// indices equal to it, each group in increasing index order, so the result is
// deterministic.
//
// One CTA per query row: 1024 threads, or 256 when there are more rows than SMs and the
// rows are short (several rows then share an SM). The row's logits are read from global memory once, mapped to order-preserving uint32 keys and kept in shared memory (rows longer than the
// shared-memory capacity are re-read from global memory instead). Three histogram passes
// (11, 11, 10 bits, shared-memory atomics) fix the k-th key exactly; the final pass gives
// each warp a contiguous chunk of the row, so one scan over the warps orders the output.
#include "common.cuh"
#include "kernels.h"

namespace idx {

namespace {

constexpr int64_t kSmemKeysMax = 48 * 1024;    // 192 KB of keys
constexpr int64_t kNarrowKeysMax = 12 * 1024;  // 48 KB of keys: four 256-thread CTAs per SM

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive sum scan over the CTA; `total` receives the CTA-wide sum.
template <int kThreads, typename T>
__device__ __forceinline__ T block_scan(T v, T* warp_sums, T& total) {
    constexpr int kWarps = kThreads / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        T s = lane < kWarps ? warp_sums[lane] : T(0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            T y = __shfl_up_sync(kFull, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kWarps) warp_sums[lane] = s;
    }
    __syncthreads();
    const T add = w > 0 ? warp_sums[w - 1] : T(0);
    total = warp_sums[kWarps - 1];
    __syncthreads();
    return x + add;
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a, int64_t smem_keys) {
    constexpr int kWarps = kThreads / 32;
    extern __shared__ uint32_t skeys[];
    __shared__ uint32_t hist[2048];
    __shared__ uint64_t warp_sums[kWarps];
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
    const bool cached = vis <= smem_keys;
    auto key_at = [&](int64_t i) -> uint32_t { return cached ? skeys[i] : order_key(row[i]); };

    uint32_t prefix = 0, pmask = 0, remaining = (uint32_t)a.k;
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const uint32_t nb = pass == 2 ? 1024u : 2048u;
        for (uint32_t i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
        __syncthreads();
        if (pass == 0) {
            // rows start 16-byte aligned (ld is a multiple of 4): float4 loads, two in flight
            const int64_t n4 = vis >> 2;
            const float4* row4 = reinterpret_cast<const float4*>(row);
            int64_t j = threadIdx.x;
            for (; j + kThreads < n4; j += 2 * kThreads) {
                const float4 v0 = row4[j], v1 = row4[j + kThreads];
                const uint4 k0 = make_uint4(order_key(v0.x), order_key(v0.y), order_key(v0.z), order_key(v0.w));
                const uint4 k1 = make_uint4(order_key(v1.x), order_key(v1.y), order_key(v1.z), order_key(v1.w));
                if (cached) {
                    reinterpret_cast<uint4*>(skeys)[j] = k0;
                    reinterpret_cast<uint4*>(skeys)[j + kThreads] = k1;
                }
                atomicAdd(&hist[k0.x >> shift], 1u);
                atomicAdd(&hist[k0.y >> shift], 1u);
                atomicAdd(&hist[k0.z >> shift], 1u);
                atomicAdd(&hist[k0.w >> shift], 1u);
                atomicAdd(&hist[k1.x >> shift], 1u);
                atomicAdd(&hist[k1.y >> shift], 1u);
                atomicAdd(&hist[k1.z >> shift], 1u);
                atomicAdd(&hist[k1.w >> shift], 1u);
            }
            for (; j < n4; j += kThreads) {
                const float4 v0 = row4[j];
                const uint4 k0 = make_uint4(order_key(v0.x), order_key(v0.y), order_key(v0.z), order_key(v0.w));
                if (cached) reinterpret_cast<uint4*>(skeys)[j] = k0;
                atomicAdd(&hist[k0.x >> shift], 1u);
                atomicAdd(&hist[k0.y >> shift], 1u);
                atomicAdd(&hist[k0.z >> shift], 1u);
                atomicAdd(&hist[k0.w >> shift], 1u);
            }
            for (int64_t i = 4 * n4 + threadIdx.x; i < vis; i += kThreads) {
                const uint32_t key = order_key(row[i]);
                if (cached) skeys[i] = key;
                atomicAdd(&hist[key >> shift], 1u);
            }
        } else {
            for (int64_t i = threadIdx.x; i < vis; i += kThreads) {
                const uint32_t key = key_at(i);
                if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
            }
        }
        __syncthreads();
        // thread r owns the bins [nb - per*(r+1), nb - per*r), highest bins first
        const int per = (int)nb / kThreads;
        const int top = (int)nb - per * (int)threadIdx.x;
        uint32_t local = 0;
        for (int j = 1; j <= per; ++j) local += hist[top - j];
        uint64_t total;
        const uint32_t incl = (uint32_t)block_scan<kThreads, uint64_t>(local, warp_sums, total);
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

    // prefix is the k-th largest key; `remaining` keys equal to it are still needed. Each
    // warp takes a contiguous chunk of the row (lanes read consecutive keys, so shared-memory
    // reads are conflict-free), counts, and one scan over the warps' counts places each
    // warp's output; inside a warp, ballots keep the index order.
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t n_gt = (uint32_t)a.k - remaining;
    const int64_t chunk = ((vis + kWarps - 1) / kWarps + 31) & ~int64_t(31);
    const int64_t lo = min(vis, chunk * warp), hi = min(vis, lo + chunk);
    uint32_t c_gt = 0, c_eq = 0;
    for (int64_t i = lo + lane; i < hi; i += 32) {
        const uint32_t key = key_at(i);
        c_gt += key > prefix;
        c_eq += key == prefix;
    }
    c_gt = __reduce_add_sync(kFull, c_gt);
    c_eq = __reduce_add_sync(kFull, c_eq);
    __shared__ uint64_t warp_base[kWarps];
    if (lane == 0) warp_base[warp] = (uint64_t)c_gt | ((uint64_t)c_eq << 32);
    __syncthreads();
    if (warp == 0) {  // exclusive scan of the warps' packed (gt, eq) counts
        const uint64_t v = lane < kWarps ? warp_base[lane] : 0;
        uint64_t inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane < kWarps) warp_base[lane] = inc - v;
    }
    __syncthreads();
    const uint64_t ex = warp_base[warp];
    uint32_t og = (uint32_t)ex, oe = (uint32_t)(ex >> 32);
    const uint32_t below = (1u << lane) - 1u;
    for (int64_t base = lo; base < hi && (c_gt > 0 || (c_eq > 0 && oe < remaining)); base += 32) {
        const int64_t i = base + lane;
        const uint32_t key = i < hi ? key_at(i) : 0u;
        const bool gt = i < hi && key > prefix, eq = i < hi && key == prefix;
        const uint32_t mg = __ballot_sync(kFull, gt), me = __ballot_sync(kFull, eq);
        if (gt) out[og + __popc(mg & below)] = (int32_t)i;
        if (eq) {
            const uint32_t r = oe + __popc(me & below);
            if (r < remaining) out[n_gt + r] = (int32_t)i;
        }
        og += __popc(mg);
        oe += __popc(me);
        c_gt -= __popc(mg);
        c_eq -= __popc(me);
    }
}

template <int kThreads>
cudaError_t launch_threads(const TopkArgs& a, cudaStream_t st) {
    const int64_t keys = a.ld < kSmemKeysMax ? a.ld : kSmemKeysMax;
    const size_t smem = (size_t)keys * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel<kThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_kernel<kThreads><<<(unsigned)a.T, kThreads, smem, st>>>(a, keys);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    // more rows than SMs and short rows: narrower CTAs, several resident per SM; otherwise
    // the widest CTA, so that each row finishes soonest
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    return (a.T > sms && a.ld <= kNarrowKeysMax) ? launch_threads<256>(a, st) : launch_threads<1024>(a, st);
}

}  // namespace idx
