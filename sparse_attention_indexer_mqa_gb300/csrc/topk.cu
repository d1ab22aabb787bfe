// topk.cu -- per-query top-k over the indexer logits by radix select.
//
// vllm PR 60834 "Test Result / GPQA Diamond": the indexer keeps the top-k (1024) keys per
// query once the context exceeds top-k x compress ratio; vllm PR 53094 "Purpose" names the
// per-token topk_indices_buffer it fills. The set of the k largest logits is unique up to
// ties at the k-th value; this kernel returns the indices above the k-th value, then the
// indices equal to it, each group in increasing index order, so the result is
// deterministic.
//
// One CTA per query row, in one of three forms chosen per launch:
//   * register-resident (topk_reg_kernel): at most one row per SM, aligned rows of at most
//     16K keys; each thread holds its keys in registers;
//   * linear bins (topk_lin_kernel): aligned rows, more rows than SMs or longer rows; the
//     keys are staged once in shared memory when they fit, and with many rows longer than
//     12K keys each pass re-reads the row instead (four rows per SM);
//   * generic (topk_kernel): any alignment and length; rows longer than shared memory are
//     re-read from global memory.
// 1024 threads per CTA, or 512 (rows up to 12K keys) or 256 (up to 8K) when there are more
// rows than SMs (several rows then share an SM). Warp w owns a contiguous slice of the row and its lanes
// read consecutive keys, so global loads are coalesced and the output keeps index order.
//
// The generic form:
//   1. The row's logits are read once, mapped to order-preserving uint32 keys, kept in
//      shared memory (rows longer than that capacity are re-read from global memory), and
//      histogrammed on their top 11 bits: the bin b0 holding the k-th key is found.
//   2. One pass over the keys counts, per warp, the keys above bin b0 and gathers the keys
//      inside b0 (the candidates: index and key) into a shared list.
//   3. Two more histogram passes (11 and 10 bits) over the listed candidates fix the k-th
//      key exactly (over every key of bin b0 when the list overflowed); when every key of
//      the 22-bit bin found by the first of them is taken (the common case: one key), the
//      k-th key is their minimum and the second pass is skipped.
//   4. Per-warp counts of candidates above / equal to the k-th key complete the warps'
//      counts; one scan over the warps places each warp's output, and a last pass writes
//      the indices with ballots.
// The other two forms bin linearly between the row's smallest and largest value instead
// (few keys share the k-th key's bin) and rank that bin's keys directly.
#include "common.cuh"
#include "kernels.h"

namespace idx {

namespace {

constexpr int kSmemKeysMax = 48 * 1024;    // 192 KB of keys
constexpr int kNarrowKeysMax = 12 * 1024;  // 48 KB of keys: several 512-thread CTAs per SM
// 32 KB of keys: five 256-thread CTAs per SM (measured on 8192 causal rows of up to 8192 keys:
// 122 us against 134 us with 512 threads and 153 us with 128)
constexpr int kNarrowestKeysMax = 8 * 1024;

// Order-preserving map of fp32 to uint32 (-0.0 and +0.0 share a key: they compare equal).
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Find the bin of the `remaining`-th largest key in hist[0..nb): every thread returns the bin
// and the number of keys in higher bins. Thread r owns the bins [nb - per*(r+1), nb - per*r),
// highest bins first; one scan over the CTA orders the owners.
template <int kThreads>
__device__ __forceinline__ void select_bin(const uint32_t* hist, int nb, uint32_t remaining,
                                           uint32_t* warp_sums, uint32_t* sel, uint32_t& bin,
                                           uint32_t& above) {
    constexpr int kWarps = kThreads / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int per = nb / kThreads;
    const int top = nb - per * (int)threadIdx.x;
    uint32_t local = 0;
    for (int j = 1; j <= per; ++j) local += hist[top - j];
    uint32_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    // every warp scans the warps' totals itself (no second barrier); lane w - 1 of the scan
    // holds the bins owned by the warps before this one
    uint32_t s = lane < kWarps ? warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, s, o);
        if (lane >= o) s += y;
    }
    const uint32_t wbefore = __shfl_sync(kFull, s, (w + 31) & 31);
    const uint32_t incl = x + (w > 0 ? wbefore : 0u);
    const uint32_t before = incl - local;
    if (before < remaining && remaining <= incl) {
        uint32_t run = before;
        for (int j = 1; j <= per; ++j) {
            const uint32_t c = hist[top - j];
            if (run + c >= remaining) {
                sel[0] = (uint32_t)(top - j);
                sel[1] = run;
                break;
            }
            run += c;
        }
    }
    __syncthreads();
    bin = sel[0];
    above = sel[1];
}

// The sequence of query row t (-1 when t lies in none). With more than two sequences the
// whole CTA looks: thread i tests the sequences i, i + kT, ... (cu[j] <= t < cu[j + 1]), one
// round of coalesced loads instead of a binary search's chain of dependent ones; with one or
// two the binary search takes at most two rounds and no barrier.
template <int kT>
__device__ __forceinline__ int seq_of_row(const int32_t* cu, int B, int64_t t, int* s_b) {
    if (B <= 2) return seq_of_query(cu, B, t);  // uniform over the CTA
    if (threadIdx.x == 0) *s_b = -1;
    __syncthreads();
    for (int i = threadIdx.x; i < B; i += kT)
        if (cu[i] <= t && t < cu[i + 1]) *s_b = i;
    __syncthreads();
    return *s_b;
}

// The generic form: any alignment, rows longer than shared memory re-read from global
// memory; bins are the top 11 key bits.
template <int kThreads, int kCand>
__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a, int smem_keys) {
    constexpr int kWarps = kThreads / 32;
    extern __shared__ uint32_t skeys[];
    __shared__ uint32_t hist[2048];
    __shared__ int32_t cand[kCand];
    __shared__ uint32_t ckey[kCand];  // the candidates' keys, in list order
    __shared__ uint32_t warp_sums[kWarps], warp_gt[kWarps], warp_eq[kWarps];
    __shared__ uint32_t sel[2], n_cand, bin_min, bin_eq;
    __shared__ int s_b;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = blockIdx.x;
    const int b = seq_of_row<kThreads>(a.cu_seqlens_q, a.B, t, &s_b);
    // the row's length (a caller input, read before the wait so that the row's loads follow it
    // at once)
    int vis = 0;
    bool bad = false;  // the scorer skipped this sequence: no logits to rank
    if (b >= 0) {
        const int64_t q0 = a.cu_seqlens_q[b], nq = a.cu_seqlens_q[b + 1] - q0;
        const int32_t len = a.seq_lens_k[b];
        if (len < 0 || len > a.max_len) bad = true;
        else vis = (int)visible_keys(len, nq, t - q0, a.causal);  // <= len <= max_len <= ld
    }
    pdl_wait();  // the logits come from the previous kernel
    pdl_launch_dependents();
    if (bad && threadIdx.x == 0) report(a.dev_status, IDX_STATUS_BAD_LEN);
    int32_t* out = a.out + t * a.k;
    const float* row = a.logits + t * a.ld;
    if (vis <= a.k) {
        for (int i = threadIdx.x; i < a.k; i += kThreads) out[i] = i < vis ? i : -1;
        return;
    }
    const bool cached = vis <= smem_keys;
    auto key_at = [&](int i) -> uint32_t { return cached ? skeys[i] : order_key(row[i]); };

    for (int i = threadIdx.x; i < 2048; i += kThreads) hist[i] = 0;
    if (threadIdx.x == 0) {
        n_cand = 0;
        bin_min = 0xffffffffu;
        bin_eq = 0;
    }
    __syncthreads();

    // 1. read, stage, histogram the top 11 bits (thread-strided, float4 where aligned)
    const int head = min(vis, (int)(((16u - ((uint32_t)(uintptr_t)row & 15u)) & 15u) >> 2));
    const int n4 = (vis - head) >> 2;
    const float4* row4 = reinterpret_cast<const float4*>(row + head);
    auto put = [&](int i, uint32_t key) {
        if (cached) skeys[i] = key;
        atomicAdd(&hist[key >> 21], 1u);
    };
    if ((int)threadIdx.x < head) put(threadIdx.x, order_key(row[threadIdx.x]));
    int j = threadIdx.x;
    for (; j + kThreads < n4; j += 2 * kThreads) {
        const float4 v0 = row4[j], v1 = row4[j + kThreads];
        const int i0 = head + 4 * j, i1 = head + 4 * (j + kThreads);
        put(i0, order_key(v0.x)); put(i0 + 1, order_key(v0.y));
        put(i0 + 2, order_key(v0.z)); put(i0 + 3, order_key(v0.w));
        put(i1, order_key(v1.x)); put(i1 + 1, order_key(v1.y));
        put(i1 + 2, order_key(v1.z)); put(i1 + 3, order_key(v1.w));
    }
    for (; j < n4; j += kThreads) {
        const float4 v0 = row4[j];
        const int i0 = head + 4 * j;
        put(i0, order_key(v0.x)); put(i0 + 1, order_key(v0.y));
        put(i0 + 2, order_key(v0.z)); put(i0 + 3, order_key(v0.w));
    }
    for (int i = head + 4 * n4 + threadIdx.x; i < vis; i += kThreads) put(i, order_key(row[i]));
    __syncthreads();
    uint32_t b0, above;
    select_bin<kThreads>(hist, 2048, (uint32_t)a.k, warp_sums, sel, b0, above);
    uint32_t remaining = (uint32_t)a.k - above;

    // 2. per-warp count of keys above bin b0; gather bin b0's indices
    constexpr int kStep = 32;  // keys per warp iteration
    const int chunk = ((vis + kWarps - 1) / kWarps + kStep - 1) & ~(kStep - 1);
    const int lo = min(vis, chunk * warp), hi = min(vis, lo + chunk);
    uint32_t c_hi = 0;
    for (int i = lo + lane; i < hi; i += 32) {
        const uint32_t key = key_at(i);
        const uint32_t bin = key >> 21;
        c_hi += bin > b0;
        if (bin == b0) {
            const uint32_t p = atomicAdd(&n_cand, 1u);
            if (p < (uint32_t)kCand) {
                cand[p] = i;
                ckey[p] = key;
            }
        }
    }
    c_hi = __reduce_add_sync(kFull, c_hi);
    if (lane == 0) {
        warp_gt[warp] = c_hi;
        warp_eq[warp] = 0;
    }
    __syncthreads();
    const uint32_t nc = n_cand;
    const bool listed = nc <= (uint32_t)kCand;
    // visit every candidate (key in bin b0): from the list, or by rescanning the row
    auto for_each_cand = [&](auto&& f) {
        if (listed) {
            for (uint32_t j = threadIdx.x; j < nc; j += kThreads) f(cand[j], ckey[j]);
        } else {
            for (int i = threadIdx.x; i < vis; i += kThreads) {
                const uint32_t key = key_at(i);
                if ((key >> 21) == b0) f(i, key);
            }
        }
    };

    // 3. fix the low 21 bits of the k-th key over the candidates (listed, or every key of
    //    bin b0 when the list overflowed)
    uint32_t prefix = b0 << 21;
    bool counted = false;  // per-warp counts of step 4 already complete
    for (int pass = 1; pass < 3; ++pass) {
        const int shift = pass == 1 ? 10 : 0;
        const int nb = pass == 1 ? 2048 : 1024;
        const uint32_t pmask = pass == 1 ? 0xffe00000u : 0xfffffc00u;
        for (int i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
        __syncthreads();
        for_each_cand([&](int, uint32_t key) {
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & (uint32_t)(nb - 1)], 1u);
        });
        __syncthreads();
        uint32_t bin, ab;
        select_bin<kThreads>(hist, nb, remaining, warp_sums, sel, bin, ab);
        const uint32_t cnt = hist[bin];  // read before the next pass clears it
        prefix |= bin << shift;
        remaining -= ab;
        if (pass == 1 && cnt == remaining) {
            // every key with this 22-bit prefix is taken (usually there is one): the k-th key
            // is their minimum, and all copies of it are taken
            for_each_cand([&](int, uint32_t key) {
                if ((key & 0xfffffc00u) == prefix) atomicMin(&bin_min, key);
            });
            __syncthreads();
            const uint32_t mn = bin_min;
            // this pass also completes the per-warp counts of step 4
            for_each_cand([&](int i, uint32_t key) {
                if (key > mn) {
                    atomicAdd(&warp_gt[i / chunk], 1u);
                } else if (key == mn) {
                    atomicAdd(&bin_eq, 1u);
                    atomicAdd(&warp_eq[i / chunk], 1u);
                }
            });
            __syncthreads();
            prefix = mn;
            remaining = bin_eq;
            counted = true;
            break;
        }
    }

    // 4. prefix is the k-th largest key; `remaining` keys equal to it are taken, lowest
    //    indices first. Candidates above / equal to it complete the per-warp counts.
    const uint32_t kth = prefix;
    if (!counted) {
        for_each_cand([&](int i, uint32_t key) {
            if (key > kth) atomicAdd(&warp_gt[i / chunk], 1u);
            else if (key == kth) atomicAdd(&warp_eq[i / chunk], 1u);
        });
        __syncthreads();
    }
    // every warp scans the warps' counts itself: og / oe = the outputs of the warps before
    // this one, c_gt / c_eq = this warp's own counts
    uint32_t og, oe, c_gt, c_eq;
    {
        const uint32_t g = lane < kWarps ? warp_gt[lane] : 0u, e = lane < kWarps ? warp_eq[lane] : 0u;
        uint32_t ig = g, ie = e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t yg = __shfl_up_sync(kFull, ig, o), ye = __shfl_up_sync(kFull, ie, o);
            if (lane >= o) {
                ig += yg;
                ie += ye;
            }
        }
        og = __shfl_sync(kFull, ig - g, warp);
        oe = __shfl_sync(kFull, ie - e, warp);
        c_gt = __shfl_sync(kFull, g, warp);
        c_eq = __shfl_sync(kFull, e, warp);
    }
    const uint32_t n_gt = (uint32_t)a.k - remaining;
    const uint32_t below = (1u << lane) - 1u;
    for (int base = lo; base < hi && (c_gt > 0 || (c_eq > 0 && oe < remaining)); base += 32) {
        const int i = base + lane;
        const uint32_t key = i < hi ? key_at(i) : 0u;
        const bool gt = i < hi && key > kth, eq = i < hi && key == kth;
        const uint32_t mg = __ballot_sync(kFull, gt), me = __ballot_sync(kFull, eq);
        if (gt) out[og + __popc(mg & below)] = i;
        if (eq) {
            const uint32_t r = oe + __popc(me & below);
            if (r < remaining) out[n_gt + r] = i;
        }
        og += __popc(mg);
        oe += __popc(me);
        c_gt -= __popc(mg);
        c_eq -= __popc(me);
    }
}


// Register-resident form for aligned rows of at most kT * kPer keys: thread (w, l) holds the
// kPer consecutive keys from (32 w + l) * kPer on, read with kPer / 4 independent 16-byte
// loads, so warp order, lane order and element order are index order and nothing is staged.
//   1. smallest and largest key of the row;
//   2. a 2048-bin histogram by a monotonic bin function: linear between the row's smallest
//      and largest value (the few bins around the k-th value hold few keys each), or the top
//      11 key bits when that range is not finite; the bin b0 of the k-th key;
//   3. per-warp counts of the keys in higher bins, and the list of bin b0's keys;
//   4. the k-th key among them: by direct ranking when the list is at most kT long, else by
//      11/11/10-bit histograms of the listed keys (or of bin b0's keys re-read from the
//      registers when the list overflowed);
//   5. per-warp counts of listed keys above / equal to it, one scan over the warps, and the
//      output written lane by lane in index order.
template <int kT, int kPer>
__global__ void __launch_bounds__(kT) topk_reg_kernel(TopkArgs a) {
    constexpr int kW = kT / 32;
    constexpr int kCandR = 2048;
    static_assert(kPer % 4 == 0 && kW <= 32 && 2048 % kT == 0, "shape");
    __shared__ uint32_t hist[2048];
    __shared__ int32_t cand[kCandR];
    __shared__ uint32_t ckey[kCandR];
    __shared__ uint32_t warp_sums[kW], warp_gt[kW], warp_eq[kW];
    __shared__ uint32_t sel[2], scal[6];  // scal: listed, min, max, k-th key, copies, taken-min
    __shared__ int s_b;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = blockIdx.x;
    const int b = seq_of_row<kT>(a.cu_seqlens_q, a.B, t, &s_b);
    for (int i = threadIdx.x; i < 2048; i += kT) hist[i] = 0;
    if (threadIdx.x == 0) {
        scal[0] = 0;
        scal[1] = 0xffffffffu;
        scal[2] = 0;
        scal[4] = 0;
        scal[5] = 0xffffffffu;
    }
    __syncthreads();  // the counters are set before any warp's atomics on them
    // the row's length (a caller input, read before the wait so that the row's loads follow it
    // at once)
    int vis = 0;
    bool bad = false;  // the scorer skipped this sequence: no logits to rank
    if (b >= 0) {
        const int64_t q0 = a.cu_seqlens_q[b], nq = a.cu_seqlens_q[b + 1] - q0;
        const int32_t len = a.seq_lens_k[b];
        if (len < 0 || len > a.max_len) bad = true;
        else vis = (int)visible_keys(len, nq, t - q0, a.causal);  // <= max_len <= kT * kPer
    }
    pdl_wait();  // the logits come from the previous kernel
    pdl_launch_dependents();
    if (bad && threadIdx.x == 0) report(a.dev_status, IDX_STATUS_BAD_LEN);
    int32_t* out = a.out + t * a.k;
    if (vis <= a.k) {
        for (int i = threadIdx.x; i < a.k; i += kT) out[i] = i < vis ? i : -1;
        return;
    }
    // 1. the thread's keys (indices i0 .. i0 + kPer - 1; those >= vis are not keys of the row)
    const int i0 = (int)threadIdx.x * kPer;
    const float4* row4 = reinterpret_cast<const float4*>(a.logits + t * a.ld) + threadIdx.x * (kPer / 4);
    uint32_t key[kPer];
    {
        float4 v[kPer / 4];
#pragma unroll
        for (int q = 0; q < kPer / 4; ++q)
            v[q] = i0 + 4 * q < vis ? row4[q] : make_float4(0.f, 0.f, 0.f, 0.f);  // in the row (ld % 4 == 0)
#pragma unroll
        for (int q = 0; q < kPer / 4; ++q) {
            key[4 * q] = order_key(v[q].x);
            key[4 * q + 1] = order_key(v[q].y);
            key[4 * q + 2] = order_key(v[q].z);
            key[4 * q + 3] = order_key(v[q].w);
        }
    }
    const int nv = max(0, min(kPer, vis - i0));  // this thread's keys
    uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        if (e < nv) {
            kmin = min(kmin, key[e]);
            kmax = max(kmax, key[e]);
        }
    }
    kmin = __reduce_min_sync(kFull, kmin);
    kmax = __reduce_max_sync(kFull, kmax);
    if (lane == 0) {
        atomicMin(&scal[1], kmin);
        atomicMax(&scal[2], kmax);
    }
    __syncthreads();

    // 2. histogram by a monotonic bin function; the bin of the k-th key
    auto value_of = [](uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); };
    const float lo = value_of(scal[1]), hi = value_of(scal[2]);
    const float span = hi - lo, scale = 2048.0f / span;
    // x - lo >= 0 and the product are rounded monotonically: equal values share a bin and a
    // larger value never falls into a lower bin
    const bool linear = span > 0.0f && isfinite(span) && isfinite(scale) && isfinite(lo);
    // floor of x in [0, 2^23): the bits of x + 2^23 rounded down (no float-to-int conversion)
    auto bin_of = [&](uint32_t k) -> uint32_t {
        if (!linear) return k >> 21;
        const float x = fminf((value_of(k) - lo) * scale, 2047.0f);
        return __float_as_uint(__fadd_rd(x, 8388608.0f)) - 0x4b000000u;
    };
    // the bins are kept in registers when the thread's keys are few
    constexpr bool kKeepBins = kPer <= 8;
    uint32_t bins[kKeepBins ? kPer : 1];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        const uint32_t bn = bin_of(key[e]);
        if constexpr (kKeepBins) bins[e] = bn;
        if (e < nv) atomicAdd(&hist[bn], 1u);
    }
    auto bin_at = [&](int e) -> uint32_t {
        if constexpr (kKeepBins) return bins[e];
        else return bin_of(key[e]);
    };
    __syncthreads();
    uint32_t b0, above;
    select_bin<kT>(hist, 2048, (uint32_t)a.k, warp_sums, sel, b0, above);
    uint32_t remaining = (uint32_t)a.k - above;

    // 3. keys of higher bins counted per warp; bin b0's keys listed
    uint32_t c_hi = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        if (e < nv) {
            const uint32_t bn = bin_at(e);
            c_hi += bn > b0;
            if (bn == b0) {
                const uint32_t p = atomicAdd(&scal[0], 1u);
                if (p < (uint32_t)kCandR) {
                    cand[p] = i0 + e;
                    ckey[p] = key[e];
                }
            }
        }
    }
    c_hi = __reduce_add_sync(kFull, c_hi);
    if (lane == 0) {
        warp_gt[warp] = c_hi;
        warp_eq[warp] = 0;
    }
    __syncthreads();
    const uint32_t nc = scal[0];
    const bool listed = nc <= (uint32_t)kCandR;
    constexpr int kChunk = 32 * kPer;  // keys per warp
    auto for_each_cand = [&](auto&& f) {
        if (listed) {
            for (uint32_t j = threadIdx.x; j < nc; j += kT) f(cand[j], ckey[j]);
        } else {
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                if (e < nv && bin_at(e) == b0) f(i0 + e, key[e]);
        }
    };

    // 4. the k-th key: the remaining-th largest among bin b0's keys
    uint32_t kth;
    if (listed && nc <= (uint32_t)kT) {
        if (threadIdx.x < nc) {
            const uint32_t mine = ckey[threadIdx.x];
            uint32_t gt = 0, ge = 0;
            for (uint32_t j = 0; j < nc; ++j) {
                const uint32_t o = ckey[j];
                gt += o > mine;
                ge += o >= mine;
            }
            if (gt < remaining && remaining <= ge) {
                scal[3] = mine;
                scal[4] = remaining - gt;  // copies of the k-th key taken
            }
        }
        __syncthreads();
        kth = scal[3];
        remaining = scal[4];
    } else {
        // histograms of the key bits [31:21], [20:10], [9:0] (the top 11 are bin b0's when
        // the bins are the top key bits); when every key of a prefix is taken the k-th key is
        // their minimum
        uint32_t prefix = linear ? 0u : (b0 << 21);
        uint32_t fixed = linear ? 0u : 0xffe00000u;
        bool done = false;
        for (int level = linear ? 0 : 1; level < 3 && !done; ++level) {
            const int shift = level == 0 ? 21 : level == 1 ? 10 : 0;
            const int nb = level == 2 ? 1024 : 2048;
            for (int i = threadIdx.x; i < nb; i += kT) hist[i] = 0;
            __syncthreads();
            for_each_cand([&](int, uint32_t k) {
                if ((k & fixed) == prefix) atomicAdd(&hist[(k >> shift) & (uint32_t)(nb - 1)], 1u);
            });
            __syncthreads();
            uint32_t bin, ab;
            select_bin<kT>(hist, nb, remaining, warp_sums, sel, bin, ab);
            const uint32_t cnt = hist[bin];
            prefix |= bin << shift;
            fixed |= (uint32_t)(nb - 1) << shift;
            remaining -= ab;
            if (level < 2 && cnt == remaining) {
                for_each_cand([&](int, uint32_t k) {
                    if ((k & fixed) == prefix) atomicMin(&scal[5], k);
                });
                __syncthreads();
                const uint32_t mn = scal[5];
                for_each_cand([&](int, uint32_t k) {
                    if (k == mn) atomicAdd(&scal[4], 1u);
                });
                __syncthreads();
                prefix = mn;
                remaining = scal[4];
                done = true;
            }
        }
        kth = prefix;
    }

    // 5. listed keys above / equal to the k-th complete the per-warp counts
    for_each_cand([&](int i, uint32_t k) {
        if (k > kth) atomicAdd(&warp_gt[i / kChunk], 1u);
        else if (k == kth) atomicAdd(&warp_eq[i / kChunk], 1u);
    });
    __syncthreads();
    // every warp scans the warps' counts itself: og / oe = the outputs of the warps before
    // this one, c_gt / c_eq = this warp's own counts
    uint32_t og, oe, c_gt, c_eq;
    {
        const uint32_t g = lane < kW ? warp_gt[lane] : 0u, q = lane < kW ? warp_eq[lane] : 0u;
        uint32_t ig = g, iq = q;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t yg = __shfl_up_sync(kFull, ig, o), yq = __shfl_up_sync(kFull, iq, o);
            if (lane >= o) {
                ig += yg;
                iq += yq;
            }
        }
        og = __shfl_sync(kFull, ig - g, warp);
        oe = __shfl_sync(kFull, iq - q, warp);
        c_gt = __shfl_sync(kFull, g, warp);
        c_eq = __shfl_sync(kFull, q, warp);
    }
    uint32_t fg = 0, fe = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        fg |= (uint32_t)(e < nv && key[e] > kth) << e;
        fe |= (uint32_t)(e < nv && key[e] == kth) << e;
    }
    const uint32_t cnt = (uint32_t)__popc(fg) | ((uint32_t)__popc(fe) << 16);
    uint32_t inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += y;
    }
    const uint32_t ex = inc - cnt;
    const uint32_t n_gt = (uint32_t)a.k - remaining;
    uint32_t pg = og + (ex & 0xffffu), pe = oe + (ex >> 16);
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        if ((fg >> e) & 1u) out[pg++] = i0 + e;
        if ((fe >> e) & 1u) {
            if (pe < remaining) out[n_gt + pe] = i0 + e;
            ++pe;
        }
    }
}

// Shared-memory form with linear bins, for aligned rows that fit in shared memory: the keys
// are staged once, then binned linearly between the row's smallest and largest value (as in
// the register-resident form), so that the k-th key's bin holds few keys and no bin gathers
// a large share of the row's atomic adds; the k-th key is found by direct ranking of that
// bin's keys (or by 11/11/10-bit histograms of them when they are many). Warp w owns the
// slice [w*chunk, (w+1)*chunk) of the row, chunk a multiple of 128, lane L the quads
// 4L..4L+3 of each 128 keys: the output is written in index order with one warp scan per
// 128 keys. kStaged false (many rows too long to stage several per SM): nothing is staged and
// each pass re-reads the row (from L2 after the first), so that several rows share an SM.
template <int kThreads, int kCand, bool kStaged>
__global__ void __launch_bounds__(kThreads, 2048 / kThreads) topk_lin_kernel(TopkArgs a) {
    constexpr int kWarps = kThreads / 32;
    extern __shared__ uint32_t skeys[];
    __shared__ uint32_t hist[2048];
    __shared__ int32_t cand[kCand];
    __shared__ uint32_t ckey[kCand];
    __shared__ uint32_t warp_sums[kWarps], warp_gt[kWarps], warp_eq[kWarps];
    __shared__ uint32_t sel[2], scal[6];  // listed, min, max, k-th key, copies, taken-min
    __shared__ int s_b;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = blockIdx.x;
    const int b = seq_of_row<kThreads>(a.cu_seqlens_q, a.B, t, &s_b);
    for (int i = threadIdx.x; i < 2048; i += kThreads) hist[i] = 0;
    if (threadIdx.x == 0) {
        scal[0] = 0;
        scal[1] = 0xffffffffu;
        scal[2] = 0;
        scal[4] = 0;
        scal[5] = 0xffffffffu;
    }
    __syncthreads();  // the counters are set before any warp's atomics on them
    // the row's length (a caller input, read before the wait so that the row's loads follow it
    // at once)
    int vis = 0;
    bool bad = false;  // the scorer skipped this sequence: no logits to rank
    if (b >= 0) {
        const int64_t q0 = a.cu_seqlens_q[b], nq = a.cu_seqlens_q[b + 1] - q0;
        const int32_t len = a.seq_lens_k[b];
        if (len < 0 || len > a.max_len) bad = true;
        else vis = (int)visible_keys(len, nq, t - q0, a.causal);  // <= len <= max_len <= ld
    }
    pdl_wait();  // the logits come from the previous kernel
    pdl_launch_dependents();
    if (bad && threadIdx.x == 0) report(a.dev_status, IDX_STATUS_BAD_LEN);
    int32_t* out = a.out + t * a.k;
    const float* row = a.logits + t * a.ld;
    if (vis <= a.k) {
        for (int i = threadIdx.x; i < a.k; i += kThreads) out[i] = i < vis ? i : -1;
        return;
    }

    // 1. read and stage the keys; the row's smallest and largest key
    const int n4 = vis >> 2;
    const float4* row4 = reinterpret_cast<const float4*>(row);
    uint4* sk4 = reinterpret_cast<uint4*>(skeys);
    // the keys of quad j / key i: staged, or read again
    auto key4 = [&](int j) -> uint4 {
        if constexpr (kStaged) {
            return sk4[j];
        } else {
            const float4 v = row4[j];
            return make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
        }
    };
    auto key_at = [&](int i) -> uint32_t {
        if constexpr (kStaged) return skeys[i];
        else return order_key(row[i]);
    };
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    auto put4 = [&](int j, const float4 v) {
        const uint4 k = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
        if constexpr (kStaged) sk4[j] = k;
        kmin = min(kmin, min(min(k.x, k.y), min(k.z, k.w)));
        kmax = max(kmax, max(max(k.x, k.y), max(k.z, k.w)));
    };
    {
        int j = threadIdx.x;
        for (; j + kThreads < n4; j += 2 * kThreads) {
            const float4 v0 = row4[j], v1 = row4[j + kThreads];
            put4(j, v0);
            put4(j + kThreads, v1);
        }
        if (j < n4) put4(j, row4[j]);
        if ((int)threadIdx.x < (vis & 3)) {
            const int i = 4 * n4 + threadIdx.x;
            const uint32_t key = order_key(row[i]);
            if constexpr (kStaged) skeys[i] = key;
            kmin = min(kmin, key);
            kmax = max(kmax, key);
        }
    }
    kmin = __reduce_min_sync(kFull, kmin);
    kmax = __reduce_max_sync(kFull, kmax);
    if (lane == 0) {
        atomicMin(&scal[1], kmin);
        atomicMax(&scal[2], kmax);
    }
    __syncthreads();

    // 2. histogram by the monotonic bin function; the bin b0 of the k-th key
    auto value_of = [](uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); };
    const float vlo = value_of(scal[1]), vhi = value_of(scal[2]);
    const float span = vhi - vlo, scale = 2048.0f / span;
    // x - vlo >= 0 and the product are rounded monotonically: equal values share a bin and a
    // larger value never falls into a lower bin (a NaN or an infinity at either end, or a
    // range that overflows, leaves the top 11 key bits as the bins)
    const bool linear = span > 0.0f && isfinite(span) && isfinite(scale) && isfinite(vlo);
    auto bin_of = [&](uint32_t k) -> uint32_t {
        if (!linear) return k >> 21;
        const float x = fminf((value_of(k) - vlo) * scale, 2047.0f);
        return __float_as_uint(__fadd_rd(x, 8388608.0f)) - 0x4b000000u;
    };
    // the histogram and candidate passes run in one of two instances, linear bins or top key
    // bits, so that the per-key bin function has no branch
    auto bin_lin = [&](uint32_t k) -> uint32_t {
        const float x = fminf((value_of(k) - vlo) * scale, 2047.0f);
        return __float_as_uint(__fadd_rd(x, 8388608.0f)) - 0x4b000000u;
    };
    auto bin_top = [](uint32_t k) -> uint32_t { return k >> 21; };
    auto hist_pass = [&](auto binf) {
        for (int j = threadIdx.x; j < n4; j += kThreads) {
            const uint4 k = key4(j);
            atomicAdd(&hist[binf(k.x)], 1u);
            atomicAdd(&hist[binf(k.y)], 1u);
            atomicAdd(&hist[binf(k.z)], 1u);
            atomicAdd(&hist[binf(k.w)], 1u);
        }
        if ((int)threadIdx.x < (vis & 3)) atomicAdd(&hist[binf(key_at(4 * n4 + threadIdx.x))], 1u);
    };
    if (linear) hist_pass(bin_lin);
    else hist_pass(bin_top);
    __syncthreads();
    uint32_t b0, above;
    select_bin<kThreads>(hist, 2048, (uint32_t)a.k, warp_sums, sel, b0, above);
    uint32_t remaining = (uint32_t)a.k - above;

    // 3. per-warp count of keys in higher bins; bin b0's keys listed
    const int chunk = ((vis + kWarps - 1) / kWarps + 127) & ~127;
    const int wlo = min(vis, chunk * warp), whi = min(vis, wlo + chunk);
    uint32_t c_hi = 0;
    auto cand_pass = [&](auto binf) {
        for (int base = wlo; base < whi; base += 128) {
            const int i0 = base + 4 * lane;
            if (i0 >= whi) continue;
            const uint4 k4 = key4(i0 >> 2);
            const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
            const int nv = min(4, whi - i0);  // valid keys of this quad (4 but at the row's end)
            uint32_t bn[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) bn[e] = e < nv ? binf(kk[e]) : 0u;  // bin 0 <= b0: not counted
#pragma unroll
            for (int e = 0; e < 4; ++e) c_hi += bn[e] > b0;
            if (((bn[0] == b0) | (bn[1] == b0) | (bn[2] == b0) | (bn[3] == b0)) != 0) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (e < nv && bn[e] == b0) {
                        const uint32_t p = atomicAdd(&scal[0], 1u);
                        if (p < (uint32_t)kCand) {
                            cand[p] = i0 + e;
                            ckey[p] = kk[e];
                        }
                    }
                }
            }
        }
    };
    if (linear) cand_pass(bin_lin);
    else cand_pass(bin_top);
    c_hi = __reduce_add_sync(kFull, c_hi);
    if (lane == 0) {
        warp_gt[warp] = c_hi;
        warp_eq[warp] = 0;
    }
    __syncthreads();
    const uint32_t nc = scal[0];
    const bool listed = nc <= (uint32_t)kCand;
    // visit bin b0's keys: from the list, or by rescanning the staged row
    auto for_each_cand = [&](auto&& f) {
        if (listed) {
            for (uint32_t j = threadIdx.x; j < nc; j += kThreads) f((int)cand[j], ckey[j]);
        } else {
            for (int i = threadIdx.x; i < vis; i += kThreads) {
                const uint32_t key = key_at(i);
                if (bin_of(key) == b0) f(i, key);
            }
        }
    };

    // 4. the k-th key: the remaining-th largest of bin b0's keys
    uint32_t kth;
    const bool ranked = listed && nc <= (uint32_t)kThreads;  // the k-th key by direct ranking
    if (ranked) {
        if (threadIdx.x < nc) {
            const uint32_t mine = ckey[threadIdx.x];
            uint32_t gt = 0, ge = 0;
            for (uint32_t j = 0; j < nc; ++j) {
                const uint32_t o = ckey[j];
                gt += o > mine;
                ge += o >= mine;
            }
            if (gt < remaining && remaining <= ge) {
                scal[3] = mine;
                scal[4] = remaining - gt;  // copies of the k-th key taken
            }
        }
        __syncthreads();
        kth = scal[3];
        remaining = scal[4];
    } else {
        // histograms of the key bits [31:21], [20:10], [9:0] (the top 11 are bin b0's when
        // the bins are the top key bits); when every key of a prefix is taken the k-th key is
        // their minimum
        uint32_t prefix = linear ? 0u : (b0 << 21);
        uint32_t fixed = linear ? 0u : 0xffe00000u;
        bool done = false;
        for (int level = linear ? 0 : 1; level < 3 && !done; ++level) {
            const int shift = level == 0 ? 21 : level == 1 ? 10 : 0;
            const int nb = level == 2 ? 1024 : 2048;
            for (int i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
            __syncthreads();
            for_each_cand([&](int, uint32_t k) {
                if ((k & fixed) == prefix) atomicAdd(&hist[(k >> shift) & (uint32_t)(nb - 1)], 1u);
            });
            __syncthreads();
            uint32_t bin, ab;
            select_bin<kThreads>(hist, nb, remaining, warp_sums, sel, bin, ab);
            const uint32_t cnt = hist[bin];
            prefix |= bin << shift;
            fixed |= (uint32_t)(nb - 1) << shift;
            remaining -= ab;
            if (level < 2 && cnt == remaining) {
                for_each_cand([&](int, uint32_t k) {
                    if ((k & fixed) == prefix) atomicMin(&scal[5], k);
                });
                __syncthreads();
                const uint32_t mn = scal[5];
                for_each_cand([&](int, uint32_t k) {
                    if (k == mn) atomicAdd(&scal[4], 1u);
                });
                __syncthreads();
                prefix = mn;
                remaining = scal[4];
                done = true;
            }
        }
        kth = prefix;
    }

    if (ranked) {
        // 5'. the keys equal to the k-th are all listed: the first `remaining` of them by index
        //     go to the end of the output, each placed by its rank among them; the pass over
        //     the row then writes only the keys above the k-th
        const uint32_t n_gt = (uint32_t)a.k - remaining;
        if (threadIdx.x < nc && ckey[threadIdx.x] == kth) {
            const int mine = cand[threadIdx.x];
            uint32_t r = 0;
            for (uint32_t j = 0; j < nc; ++j) r += ckey[j] == kth && cand[j] < mine;
            if (r < remaining) out[n_gt + r] = mine;
        }
        for_each_cand([&](int i, uint32_t k) {
            if (k > kth) atomicAdd(&warp_gt[i / chunk], 1u);
        });
        __syncthreads();
        uint32_t og, c_gt;
        {
            const uint32_t g = lane < kWarps ? warp_gt[lane] : 0u;
            uint32_t ig = g;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, ig, o);
                if (lane >= o) ig += y;
            }
            og = __shfl_sync(kFull, ig - g, warp);
            c_gt = __shfl_sync(kFull, g, warp);
        }
        for (int base = wlo; base < whi && c_gt > 0; base += 128) {
            const int i0 = base + 4 * lane;
            const int nv = i0 < whi ? min(4, whi - i0) : 0;
            uint32_t fg = 0;
            if (nv > 0) {
                const uint4 k4 = key4(i0 >> 2);
                fg = ((uint32_t)(k4.x > kth) | ((uint32_t)(k4.y > kth) << 1) | ((uint32_t)(k4.z > kth) << 2) |
                      ((uint32_t)(k4.w > kth) << 3)) & ((1u << nv) - 1u);
            }
            const uint32_t cnt = (uint32_t)__popc(fg);
            uint32_t inc = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, inc, o);
                if (lane >= o) inc += y;
            }
            const uint32_t tot = __shfl_sync(kFull, inc, 31);
            int32_t* dst = out + og + (inc - cnt);
            if (fg & 1u) *dst++ = i0;
            if (fg & 2u) *dst++ = i0 + 1;
            if (fg & 4u) *dst++ = i0 + 2;
            if (fg & 8u) *dst = i0 + 3;
            og += tot;
            c_gt -= tot;
        }
        return;
    }
    // 5. bin b0's keys above / equal to the k-th complete the per-warp counts; one scan over
    //    the warps places each warp's output, written in index order
    for_each_cand([&](int i, uint32_t k) {
        if (k > kth) atomicAdd(&warp_gt[i / chunk], 1u);
        else if (k == kth) atomicAdd(&warp_eq[i / chunk], 1u);
    });
    __syncthreads();
    // every warp scans the warps' counts itself: og / oe = the outputs of the warps before
    // this one, c_gt / c_eq = this warp's own counts
    uint32_t og, oe, c_gt, c_eq;
    {
        const uint32_t g = lane < kWarps ? warp_gt[lane] : 0u, e = lane < kWarps ? warp_eq[lane] : 0u;
        uint32_t ig = g, ie = e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t yg = __shfl_up_sync(kFull, ig, o), ye = __shfl_up_sync(kFull, ie, o);
            if (lane >= o) {
                ig += yg;
                ie += ye;
            }
        }
        og = __shfl_sync(kFull, ig - g, warp);
        oe = __shfl_sync(kFull, ie - e, warp);
        c_gt = __shfl_sync(kFull, g, warp);
        c_eq = __shfl_sync(kFull, e, warp);
    }
    const uint32_t n_gt = (uint32_t)a.k - remaining;
    for (int base = wlo; base < whi && (c_gt > 0 || (c_eq > 0 && oe < remaining)); base += 128) {
        const int i0 = base + 4 * lane;
        uint32_t fg = 0, fe = 0;
        if (i0 < whi) {
            const uint4 k4 = key4(i0 >> 2);
            const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
            const int nv = min(4, whi - i0);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                fg |= (uint32_t)(e < nv && kk[e] > kth) << e;
                fe |= (uint32_t)(e < nv && kk[e] == kth) << e;
            }
        }
        const uint32_t cnt = (uint32_t)__popc(fg) | ((uint32_t)__popc(fe) << 16);
        uint32_t inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += y;
        }
        const uint32_t tot = __shfl_sync(kFull, inc, 31);
        const uint32_t ex = inc - cnt;
        uint32_t pg = og + (ex & 0xffffu), pe = oe + (ex >> 16);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if ((fg >> e) & 1u) out[pg++] = i0 + e;
        if (fe) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if ((fe >> e) & 1u) {
                    if (pe < remaining) out[n_gt + pe] = i0 + e;
                    ++pe;
                }
            }
        }
        og += tot & 0xffffu;
        oe += tot >> 16;
        c_gt -= tot & 0xffffu;
        c_eq -= tot >> 16;
    }
}

template <int kThreads, int kCand>
cudaError_t launch_form(const TopkArgs& a, cudaStream_t st) {
    const int keys = (int)(a.ld < kSmemKeysMax ? a.ld : kSmemKeysMax);
    const size_t smem = (size_t)keys * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel<kThreads, kCand>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_kernel<kThreads, kCand>, dim3((unsigned)a.T), dim3(kThreads), smem, st, a,
                      keys);
}

template <int kThreads, int kCand, bool kStaged>
cudaError_t launch_lin(const TopkArgs& a, cudaStream_t st) {
    const size_t smem = kStaged ? (size_t)a.ld * sizeof(uint32_t) : 0;
    cudaError_t e = cudaFuncSetAttribute(topk_lin_kernel<kThreads, kCand, kStaged>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_lin_kernel<kThreads, kCand, kStaged>, dim3((unsigned)a.T), dim3(kThreads), smem, st, a);
}

template <int kThreads, int kCand>
cudaError_t launch_threads(const TopkArgs& a, cudaStream_t st) {
    const bool vec = a.ld % 4 == 0 && a.ld <= kSmemKeysMax && ((uintptr_t)a.logits & 15) == 0;
    return vec ? launch_lin<kThreads, kCand, true>(a, st) : launch_form<kThreads, kCand>(a, st);
}

}  // namespace

template <int kT, int kPer>
cudaError_t launch_reg(const TopkArgs& a, cudaStream_t st) {
    return launch_pdl(topk_reg_kernel<kT, kPer>, dim3((unsigned)a.T), dim3(kT), 0, st, a);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    // more rows than SMs and short rows: narrower CTAs, several resident per SM; otherwise
    // the widest CTA, so that each row finishes soonest
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // at most one row per SM, aligned rows of at most 16K keys: the register-resident form,
    // whose shorter phase chain finishes a row sooner (16-byte loads need ld % 4 == 0 and a
    // 16-byte aligned base; a row's keys past max_len are never read). With more rows the
    // shared-memory form keeps more rows resident per SM.
    if (a.T <= sms && a.ld % 4 == 0 && ((uintptr_t)a.logits & 15) == 0 && a.max_len <= 16384)
        return a.max_len <= 8192 ? launch_reg<1024, 8>(a, st) : launch_reg<1024, 16>(a, st);
    if (a.T > sms && a.ld <= kNarrowestKeysMax) return launch_threads<256, 512>(a, st);
    // many rows too long to stage several per SM: four 512-thread rows per SM re-read their
    // rows from L2 (measured on 32768 rows of up to 36K keys: 3.21 ms against 3.64 ms staged,
    // one row per SM; 3.24 / 3.63 ms with 256 / 1024 threads)
    if (a.T > sms && a.ld > kNarrowKeysMax && a.ld % 4 == 0 && ((uintptr_t)a.logits & 15) == 0)
        return launch_lin<512, 1024, false>(a, st);
    return (a.T > sms && a.ld <= kNarrowKeysMax) ? launch_threads<512, 1024>(a, st)
                                                 : launch_threads<1024, 2048>(a, st);
}

}  // namespace idx
