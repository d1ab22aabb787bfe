// select.cuh -- exact top-k of one logits row, run by a group of kT threads: the body of
// idx_topk (one CTA per row) and of the fused scorer -> top-k kernels (a warpgroup per row).
//
// vllm PR 60834 "Test Result / GPQA Diamond": the indexer keeps the top-k keys of every query
// once its context passes top-k x compress ratio; vllm PR 53094 "Purpose": the per-token
// topk_indices_buffer. The result is the indices of the values above the k-th value in
// increasing index order, then the indices equal to it in increasing index order, then -1
// padding: a deterministic function of the fp32 row.
//
// The group's threads have ids tid = 0 .. kT-1 and synchronise with sync() (a named barrier
// of kT threads, or __syncthreads when the group is the whole CTA). Warp w of the group owns
// the contiguous slice [w*chunk, (w+1)*chunk) of the row, so its ballots keep index order.
// Values are compared through order-preserving uint32 keys (-0.0 and +0.0 are one key).
//   A. the row is read once (kept in `keys` when it fits, else re-read from L2) and its
//      smallest and largest keys found;
//   B. the keys are histogrammed into 2048 bins by a monotonic function of the value:
//      linear between the row's minimum and maximum, so that the few bins around the k-th
//      value hold few keys each (for an extreme range, the top 11 bits of the key); the bin
//      holding the k-th key is found from the histogram;
//   C. one pass counts, per warp, the keys of higher bins and lists the keys of that bin
//      (the candidates; every key of the bin is revisited when the list overflows);
//   D. the k-th key among the candidates: by direct ranking when they are few, else by
//      histograms of its 11, 11 and 10 key bits (when every key of a prefix is taken, the
//      k-th key is their minimum);
//   E. per-warp counts, one scan over the warps and a ballot pass write the output.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace idx {

// Shared memory a selecting group works in (the caller carves it from its own buffers).
struct SelectSmem {
    uint32_t* hist;       // [2048]
    int32_t* cand;        // [kCand] candidate indices
    uint32_t* ckey;       // [kCand] candidate keys
    uint32_t* warp_sums;  // [kT / 32]
    uint32_t* warp_gt;    // [kT / 32]
    uint32_t* warp_eq;    // [kT / 32]
    uint32_t* scal;       // [8]
    uint32_t* keys;       // staged keys of the row, or nullptr
    int key_cap;          // capacity of `keys`
};

// Order-preserving map of fp32 to uint32 (-0.0 and +0.0 share a key: they compare equal).
__device__ __forceinline__ uint32_t select_order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// Its inverse (the key of -0.0 maps back to +0.0).
__device__ __forceinline__ float select_key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// The bin of the `remaining`-th largest key in hist[0..nb) and the number of keys in higher
// bins, identical in every thread of the group. Thread r owns bins [nb - per*(r+1), nb - per*r).
template <int kT, typename Sync>
__device__ __forceinline__ void select_bin_g(const uint32_t* hist, int nb, uint32_t remaining,
                                             const SelectSmem& sm, int tid, Sync& sync,
                                             uint32_t& bin, uint32_t& above) {
    constexpr int kW = kT / 32;
    const int lane = tid & 31, w = tid >> 5;
    const int per = nb / kT;
    const int top = nb - per * tid;
    uint32_t local = 0;
    for (int j = 1; j <= per; ++j) local += hist[top - j];
    uint32_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.warp_sums[w] = x;
    sync();
    if (w == 0) {
        uint32_t s = lane < kW ? sm.warp_sums[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kW) sm.warp_sums[lane] = s;
    }
    sync();
    const uint32_t incl = x + (w > 0 ? sm.warp_sums[w - 1] : 0u);
    const uint32_t before = incl - local;
    if (before < remaining && remaining <= incl) {
        uint32_t run = before;
        for (int j = 1; j <= per; ++j) {
            const uint32_t c = hist[top - j];
            if (run + c >= remaining) {
                sm.scal[0] = (uint32_t)(top - j);
                sm.scal[1] = run;
                break;
            }
            run += c;
        }
    }
    sync();
    bin = sm.scal[0];
    above = sm.scal[1];
}

// Top-k of row[0 .. vis) into out[0 .. k). An unstaged row is read through L2
// (ld.global.cg): it may have been written by other threads or CTAs of the calling kernel,
// which made their writes visible at GPU scope before a barrier or an acquiring atomic that
// orders them before the call.
template <int kT, int kCand, typename Sync>
__device__ void select_topk_row(const float* row, int vis, int k, int32_t* out, const SelectSmem& sm,
                                int tid, Sync&& sync) {
    constexpr int kW = kT / 32;
    constexpr int kRank = kT < 256 ? kT : 256;  // candidates resolved by direct ranking
    static_assert(kT % 32 == 0 && kW <= 32 && 2048 % kT == 0 && kCand >= kRank, "group shape");
    const int lane = tid & 31, warp = tid >> 5;
    if (vis <= k) {
        for (int i = tid; i < k; i += kT) out[i] = i < vis ? i : -1;
        return;
    }
    const bool cached = sm.keys != nullptr && vis <= sm.key_cap;
    auto key_at = [&](int i) -> uint32_t { return cached ? sm.keys[i] : select_order_key(__ldcg(row + i)); };
    uint32_t* hist = sm.hist;
    for (int i = tid; i < 2048; i += kT) hist[i] = 0;
    if (tid == 0) {
        sm.scal[2] = 0;            // candidates listed
        sm.scal[3] = 0xffffffffu;  // minimum of a fully taken prefix
        sm.scal[4] = 0;            // copies of that minimum
        sm.scal[5] = 0xffffffffu;  // smallest key of the row
        sm.scal[6] = 0;            // largest key of the row
    }
    sync();

    // A. read (16-byte loads after an unaligned head, several in flight), stage, min / max
    {
        uint32_t kmin = 0xffffffffu, kmax = 0u;
        auto put = [&](int i, uint32_t key) {
            if (cached) sm.keys[i] = key;
            kmin = min(kmin, key);
            kmax = max(kmax, key);
        };
        const int head = min(vis, (int)(((16u - ((uint32_t)(uintptr_t)row & 15u)) & 15u) >> 2));
        const int n4 = (vis - head) >> 2;
        const float4* row4 = reinterpret_cast<const float4*>(row + head);
        if (tid < head) put(tid, select_order_key(__ldcg(row + tid)));
        constexpr int U = 4;
        for (int j0 = tid; j0 < n4; j0 += U * kT) {
            float4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (j0 + u * kT < n4) v[u] = __ldcg(row4 + j0 + u * kT);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (j0 + u * kT >= n4) break;
                const int i0 = head + 4 * (j0 + u * kT);
                put(i0, select_order_key(v[u].x));
                put(i0 + 1, select_order_key(v[u].y));
                put(i0 + 2, select_order_key(v[u].z));
                put(i0 + 3, select_order_key(v[u].w));
            }
        }
        for (int i = head + 4 * n4 + tid; i < vis; i += kT) put(i, select_order_key(__ldcg(row + i)));
        kmin = __reduce_min_sync(kFull, kmin);
        kmax = __reduce_max_sync(kFull, kmax);
        if (lane == 0) {
            atomicMin(&sm.scal[5], kmin);
            atomicMax(&sm.scal[6], kmax);
        }
    }
    sync();

    // B. histogram by a monotonic bin function; the bin of the k-th key
    const float lo = select_key_value(sm.scal[5]), hi = select_key_value(sm.scal[6]);
    const float span = hi - lo;
    const float scale = 2048.0f / span;
    // linear bins need a finite, positive range and scale; x - lo >= 0 and the product are
    // rounded monotonically, so equal values share a bin and larger values never fall lower
    const bool linear = span > 0.0f && isfinite(span) && isfinite(scale) && isfinite(lo);
    auto bin_of = [&](uint32_t key) -> uint32_t {
        if (!linear) return key >> 21;
        const float t = (select_key_value(key) - lo) * scale;
        return t >= 2047.0f ? 2047u : (uint32_t)t;
    };
    constexpr int UB = 8;  // keys read per lane before use (independent loads when not staged)
    for (int base = tid; base < vis; base += kT * UB) {
        uint32_t kk[UB];
#pragma unroll
        for (int u = 0; u < UB; ++u) kk[u] = base + kT * u < vis ? key_at(base + kT * u) : 0u;
#pragma unroll
        for (int u = 0; u < UB; ++u)
            if (base + kT * u < vis) atomicAdd(&hist[bin_of(kk[u])], 1u);
    }
    sync();
    uint32_t b0, above;
    select_bin_g<kT>(hist, 2048, (uint32_t)k, sm, tid, sync, b0, above);
    uint32_t remaining = (uint32_t)k - above;

    // C. per-warp count of keys in higher bins; list the bin's keys
    const int chunk = ((vis + kW - 1) / kW + 31) & ~31;
    const int lo_i = min(vis, chunk * warp), hi_i = min(vis, lo_i + chunk);
    uint32_t c_hi = 0;
    for (int base = lo_i + lane; base < hi_i; base += 32 * UB) {
        uint32_t kk[UB];
#pragma unroll
        for (int u = 0; u < UB; ++u) kk[u] = base + 32 * u < hi_i ? key_at(base + 32 * u) : 0u;
#pragma unroll
        for (int u = 0; u < UB; ++u) {
            const int i = base + 32 * u;
            if (i >= hi_i) break;
            const uint32_t bin = bin_of(kk[u]);
            c_hi += bin > b0;
            if (bin == b0) {
                const uint32_t p = atomicAdd(&sm.scal[2], 1u);
                if (p < (uint32_t)kCand) {
                    sm.cand[p] = i;
                    sm.ckey[p] = kk[u];
                }
            }
        }
    }
    c_hi = __reduce_add_sync(kFull, c_hi);
    if (lane == 0) {
        sm.warp_gt[warp] = c_hi;
        sm.warp_eq[warp] = 0;
    }
    sync();
    const uint32_t nc = sm.scal[2];
    const bool listed = nc <= (uint32_t)kCand;
    auto for_each_cand = [&](auto&& f) {
        if (listed) {
            for (uint32_t j = tid; j < nc; j += kT) f(sm.cand[j], sm.ckey[j]);
        } else {
            for (int base = tid; base < vis; base += kT * UB) {
                uint32_t kk[UB];
#pragma unroll
                for (int u = 0; u < UB; ++u) kk[u] = base + kT * u < vis ? key_at(base + kT * u) : 0u;
#pragma unroll
                for (int u = 0; u < UB; ++u)
                    if (base + kT * u < vis && bin_of(kk[u]) == b0) f(base + kT * u, kk[u]);
            }
        }
    };

    // D. the k-th key: the remaining-th largest key among the candidates
    uint32_t kth;
    if (listed && nc <= (uint32_t)kRank) {
        // direct ranking: candidate j is the k-th key when fewer than `remaining` candidates
        // are larger and at least `remaining` are larger or equal
        if ((uint32_t)tid < nc) {
            const uint32_t mine = sm.ckey[tid];
            uint32_t gt = 0, ge = 0;
            for (uint32_t j = 0; j < nc; ++j) {
                const uint32_t o = sm.ckey[j];
                gt += o > mine;
                ge += o >= mine;
            }
            if (gt < remaining && remaining <= ge) {
                sm.scal[3] = mine;
                sm.scal[4] = remaining - gt;  // copies of the k-th key taken
            }
        }
        sync();
        kth = sm.scal[3];
        remaining = sm.scal[4];
        for_each_cand([&](int i, uint32_t key) {
            if (key > kth) atomicAdd(&sm.warp_gt[i / chunk], 1u);
            else if (key == kth) atomicAdd(&sm.warp_eq[i / chunk], 1u);
        });
        sync();
    } else {
        // histograms of the key's bits [31:21], [20:10], [9:0] over the candidates (those of
        // a top-11-bit bin only need the last two)
        uint32_t prefix = linear ? 0u : (b0 << 21);
        uint32_t fixed = linear ? 0u : 0xffe00000u;
        bool counted = false;
        for (int level = linear ? 0 : 1; level < 3; ++level) {
            const int shift = level == 0 ? 21 : level == 1 ? 10 : 0;
            const int nb = level == 2 ? 1024 : 2048;
            for (int i = tid; i < nb; i += kT) hist[i] = 0;
            sync();
            for_each_cand([&](int, uint32_t key) {
                if ((key & fixed) == prefix) atomicAdd(&hist[(key >> shift) & (uint32_t)(nb - 1)], 1u);
            });
            sync();
            uint32_t bin, ab;
            select_bin_g<kT>(hist, nb, remaining, sm, tid, sync, bin, ab);
            const uint32_t cnt = hist[bin];
            prefix |= bin << shift;
            fixed |= (uint32_t)(nb - 1) << shift;
            remaining -= ab;
            if (level < 2 && cnt == remaining) {
                // every key with this prefix is taken (often just one): the k-th key is their
                // minimum, and all copies of it are taken
                for_each_cand([&](int, uint32_t key) {
                    if ((key & fixed) == prefix) atomicMin(&sm.scal[3], key);
                });
                sync();
                const uint32_t mn = sm.scal[3];
                for_each_cand([&](int i, uint32_t key) {
                    if (key > mn) {
                        atomicAdd(&sm.warp_gt[i / chunk], 1u);
                    } else if (key == mn) {
                        atomicAdd(&sm.scal[4], 1u);
                        atomicAdd(&sm.warp_eq[i / chunk], 1u);
                    }
                });
                sync();
                prefix = mn;
                remaining = sm.scal[4];
                counted = true;
                break;
            }
        }
        kth = prefix;
        if (!counted) {
            for_each_cand([&](int i, uint32_t key) {
                if (key > kth) atomicAdd(&sm.warp_gt[i / chunk], 1u);
                else if (key == kth) atomicAdd(&sm.warp_eq[i / chunk], 1u);
            });
            sync();
        }
    }

    // E. kth is the k-th largest key; `remaining` copies of it are taken, lowest indices first
    uint32_t c_gt = sm.warp_gt[warp], c_eq = sm.warp_eq[warp];
    sync();
    if (warp == 0) {  // exclusive scans of the warps' counts
        const uint32_t g = lane < kW ? sm.warp_gt[lane] : 0u, e = lane < kW ? sm.warp_eq[lane] : 0u;
        uint32_t ig = g, ie = e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t yg = __shfl_up_sync(kFull, ig, o), ye = __shfl_up_sync(kFull, ie, o);
            if (lane >= o) {
                ig += yg;
                ie += ye;
            }
        }
        if (lane < kW) {
            sm.warp_gt[lane] = ig - g;
            sm.warp_eq[lane] = ie - e;
        }
    }
    sync();
    const uint32_t n_gt = (uint32_t)k - remaining;
    uint32_t og = sm.warp_gt[warp], oe = sm.warp_eq[warp];
    const uint32_t below = (1u << lane) - 1u;
    for (int base = lo_i; base < hi_i && (c_gt > 0 || (c_eq > 0 && oe < remaining)); base += 32 * UB) {
        uint32_t kk[UB];
#pragma unroll
        for (int u = 0; u < UB; ++u) {
            const int i = base + 32 * u + lane;
            kk[u] = i < hi_i ? key_at(i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < UB; ++u) {
            const int i = base + 32 * u + lane;
            const bool gt = i < hi_i && kk[u] > kth, eq = i < hi_i && kk[u] == kth;
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
    sync();  // the group's shared memory may be reused for the next row
}

// Rows that no unit of a fused scorer -> top-k kernel may write get -1 padding: rows of no
// sequence, rows of a sequence whose lengths break the scorer's bounds (the scorer skips and
// reports it) and rows with no visible key (they have no tile). Strided over `ethreads`
// threads per CTA of the grid (etid in [0, ethreads)); a row's sequence by binary search.
__device__ __forceinline__ void pad_orphan_rows(const ScoreArgs& a, int etid, int ethreads) {
    const int64_t T = a.T;
    for (int64_t t = (int64_t)blockIdx.x * ethreads + etid; t < T; t += (int64_t)gridDim.x * ethreads) {
        const int b = seq_of_query(a.cu_seqlens_q, a.B, t);
        bool bad = b < 0;
        if (!bad) {
            const int64_t q0 = a.cu_seqlens_q[b], nq = (int64_t)a.cu_seqlens_q[b + 1] - q0;
            const int32_t len = a.seq_lens_k[b];
            bad = nq > a.max_q_len || len < 0 || len > a.max_seq_len_k ||
                  visible_keys(len, nq, t - q0, a.causal) == 0;
        }
        if (bad)
            for (int i = 0; i < a.topk_k; ++i) a.out_idx[t * a.topk_k + i] = -1;
    }
}

// Named barrier over `count` threads (a multiple of 32) of the CTA.
struct NamedBarrier {
    uint32_t id, count;
    __device__ __forceinline__ void operator()() const {
        asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
    }
};

}  // namespace idx
