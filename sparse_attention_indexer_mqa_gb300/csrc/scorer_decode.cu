// scorer_decode.cu -- paged MQA-logits scorer for decode (one query per sequence) on the
// 5th-generation tensor cores.
//
//   logits[t, s] = sum_h w[t,h] * ReLU(q[t,h] . k[s])               (MXFP4)
//   logits[t, s] = kscale[s] * sum_h w[t,h] * ReLU(q[t,h] . k[s])   (FP8, w carries q's scale)
//
// vllm PR 57517 "Purpose" / "Performance and accuracy" (decode B64/H32/D128/8K scorer) and
// vllm PR 60834 "Purpose" (the MXFP4 cache is scored in place through the page table,
// without gathering K first).
//
// Operands: the key tile is the A operand (M = 128 keys = one 128-token page or two 64-token
// pages), the query's heads are B (N = H rounded up to 16), K = 128. So each tensor-memory
// lane holds one key and one thread reduces its key's H head scores with no shuffles. Cache
// pages and the quantised Q are stored in the tensor core's canonical K-major order (see
// idx.h): every operand reaches shared memory through cp.async.bulk unchanged, and the
// MXFP4 E8M0 scale atoms go to tensor memory with one tcgen05.cp each. MXFP4 runs
// kind::mxf4 block-scaled MMAs (two of K = 64); FP8 runs kind::f8f6f4 (four of K = 32) and
// applies the per-key scale in the epilogue.
//
// Persistent, warp-specialised: four CTAs per SM (two for 64 heads) each take a contiguous,
// balanced slice of all (sequence, 128-key tile) units, so that one CTA's issue, MMA and
// epilogue latencies overlap the others'. The stage ring is sized from the SM's shared memory
// (about five 8.7 KB tiles per CTA for H <= 32); the code allows G tiles per stage group and
// mbarrier phase, and G = 1 is what every configuration uses.
//   warp 0   producer: bulk copies of the query images (a ring of Q slots; a batch never
//            touches more sequences than there are slots) and of the tiles; each lane of the
//            warp issues one tile, so a batch of tiles goes out at once;
//   warp 1   tensor-memory owner and MMA issuer: scale atoms -> TMEM, a tile's MMAs into one
//            of two accumulators, one commit to free the stage, one to publish the
//            accumulator;
//   warps 2-5 epilogue (one 32-lane TMEM quadrant each): tcgen05.ld, ReLU-weighted head
//            sum in fp32, coalesced logits stores.
// The cache stream is read with an evict-first L2 policy and the lengths and page table with
// evict-last, so that the metadata every launch reads stays in L2 under the stream.
// The prologue scans the sequences once (eight per lane, loads issued together) and keeps the
// 32 sequences from the slice's start in a shared table; it overlaps the previous kernel
// (programmatic dependent launch), and the producer's first page lookups precede its wait.
// Every bounded wait that gives up sets IDX_STATUS_TIMEOUT; the producer then waits (bounded)
// for the copies it armed and the MMA thread for its last tensor-core operations before the
// CTA frees tensor memory.
// Every role walks the same unit sequence, so no metadata is passed between roles.
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"
#include "tc.cuh"

namespace idx {

namespace {

constexpr int kWarps = 6;
constexpr int kThreads = 32 * kWarps;
constexpr int kEpiThreads = 128;
constexpr int kAccG = 2;  // accumulator groups in tensor memory
constexpr int kSeqWin = 32;  // sequences described by the shared-memory table
constexpr int kSelCand = 256;  // select mode: candidate list of the epilogue warps

template <int kDtype, int NP>
struct Cfg {
    // CTAs per SM: independent pipelines that share an SM so that one CTA's issue, MMA and
    // epilogue latencies overlap the others' (tensor memory <= 128 columns each for H <= 32,
    // four CTAs; <= 256 for 64 heads, two CTAs). One tile per stage group and mbarrier phase.
    static constexpr int kCps = NP <= 32 ? 4 : 2;
    static constexpr int G = 1;
    static constexpr int kTileCode = kDtype == IDX_MXFP4 ? 128 * 64 : 128 * 128;
    static constexpr int kTileSf = kDtype == IDX_MXFP4 ? 512 : 0;          // scale atom (MXFP4)
    static constexpr int kTile = kTileCode + kTileSf;
    static constexpr int kGroup = G * kTile;
    static constexpr int kQRow = kDtype == IDX_MXFP4 ? 64 : 128;
    static constexpr int kQImg = NP * kQRow;                               // per Q slot
    static constexpr int kQSf = kDtype == IDX_MXFP4 ? 512 : 0;
    // Q slots (a ring): a producer batch touches at most kQS sequences, so a slot it waits
    // for is always released by tiles of earlier batches
    static constexpr int kQS = NP <= 32 ? 4 : 2;
    // shared memory of one CTA: an SM has 228 KB, of which 1 KB per resident CTA is reserved
    static constexpr int kBudget = (228 * 1024) / kCps - 1024;
    static constexpr int kFixed = kQS * (kQImg + kQSf) + 64 + kSeqWin * 16 + 8 * (2 * kQS + 1 + 2 * kAccG);
    static constexpr int kSG = (kBudget - kFixed) / (kGroup + 16);        // stage groups
    static constexpr uint32_t kSbo = kDtype == IDX_MXFP4 ? 512 : 1024;
    static constexpr int kColsUsed = kAccG * G * (NP + 4) + 4 * kQS;       // acc + SFA + SFB
    static constexpr uint32_t kCols = kColsUsed <= 64 ? 64 : kColsUsed <= 128 ? 128 : kColsUsed <= 256 ? 256 : 512;
    static constexpr int kBatch = G * kSG < 32 ? G * kSG : (32 / G) * G;   // tiles per producer batch
    // shared memory map
    static constexpr int oStages = 0;
    static constexpr int oQ = kSG * kGroup;
    static constexpr int oQSf = oQ + kQS * kQImg;
    static constexpr int oBars = oQSf + kQS * kQSf;
    static constexpr int kBars = 2 * kSG + 2 * kQS + 1 + 2 * kAccG;
    static constexpr int oMisc = oBars + 8 * kBars;
    static constexpr int oSeq = oMisc + 64;
    static constexpr int kSmem = oSeq + kSeqWin * 16;
    static_assert(kBatch % G == 0 && kBatch <= G * kSG, "a batch covers whole, distinct stage groups");
    static_assert(kCols * kCps <= 512, "tensor memory of the CTAs sharing an SM");
    static_assert(kSmem <= kBudget, "shared memory of the CTAs sharing an SM");
};

// Tile count, visible keys and query row of sequence b (0 tiles if it has no query). The
// three loads are issued together. A sequence whose lengths break their bounds (key count
// negative or above max_seq_len_k, query count negative or above max_q_len <= 1) gets 0
// tiles and sets *bad.
struct SeqInfo {  // 32-bit: T <= INT32_MAX and lengths are int32 (checked by the API)
    int32_t t, vis, tiles;
};

// The same from the three values already loaded (cu_seqlens_q[b], cu_seqlens_q[b+1], seq_lens_k[b]).
__device__ __forceinline__ SeqInfo seq_info_of(const ScoreArgs& a, int32_t q0, int32_t q1, int32_t len, bool* bad) {
    SeqInfo r{0, 0, 0};
    const int32_t nq = q1 - q0;
    if (nq == 0) return r;
    if (nq < 0 || nq > a.max_q_len || len < 0 || len > a.max_seq_len_k) {
        *bad = true;
        return r;
    }
    r.t = q0;
    r.vis = (int32_t)visible_keys(len, nq, nq - 1, a.causal);
    r.tiles = (r.vis + 127) / 128;
    return r;
}

__device__ __forceinline__ SeqInfo seq_info(const ScoreArgs& a, int b, uint64_t keep, bool* bad = nullptr) {
    const int32_t q0 = tc::ld_hint(a.cu_seqlens_q + b, keep), q1 = tc::ld_hint(a.cu_seqlens_q + b + 1, keep);
    const int32_t len = tc::ld_hint(a.seq_lens_k + b, keep);
    SeqInfo r{0, 0, 0};
    const int32_t nq = q1 - q0;
    if (nq == 0) return r;
    if (nq < 0 || nq > a.max_q_len || len < 0 || len > a.max_seq_len_k) {
        if (bad) *bad = true;
        return r;
    }
    r.t = q0;
    r.vis = (int32_t)visible_keys(len, nq, nq - 1, a.causal);
    r.tiles = (r.vis + 127) / 128;
    return r;
}

// The kSeqWin sequences from the slice's first one on are described by a table in shared
// memory, written once by the prologue, so that walking from one sequence to the next costs
// no global load (a slice that reaches past the window reads global memory).
struct SeqEnt {
    int32_t t, vis, tiles, pad;
};

struct Seqs {
    const ScoreArgs* a;
    const SeqEnt* tab;
    int b_tab;      // sequence of tab[0]
    uint64_t keep;  // L2 policy of the metadata loads
    __device__ __forceinline__ SeqInfo get(int b) const {
        const unsigned r = (unsigned)(b - b_tab);
        if (r < (unsigned)kSeqWin) {
            const SeqEnt e = tab[r];
            return SeqInfo{e.t, e.vis, e.tiles};
        }
        return seq_info(*a, b, keep);
    }
};

// Walks (sequence, tile) units in order from a starting unit.
struct Walker {
    int b;
    int32_t j;
    SeqInfo si;
    __device__ __forceinline__ void init(const Seqs& S, int b0, int32_t j0) {
        b = b0;
        j = j0;
        si = b0 < S.a->B ? S.get(b0) : SeqInfo{0, 0, 1};
    }
    __device__ __forceinline__ void next(const Seqs& S) {
        if (++j < si.tiles) return;
        j = 0;
        do {
            ++b;
            si = b < S.a->B ? S.get(b) : SeqInfo{0, 0, 1};
        } while (si.tiles == 0);
    }
};

template <int NP>
__device__ __forceinline__ void load_acc(uint32_t taddr, float* v) {
    if constexpr (NP == 16) {
        uint32_t r[16];
        tc::tmem_ld16(taddr, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
    } else {
#pragma unroll
        for (int c = 0; c < NP; c += 32) {
            uint32_t r[32];
            tc::tmem_ld32(taddr + c, r);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[c + i] = __uint_as_float(r[i]);
        }
    }
}

// bar.red.or over the CTA's four epilogue warps (named barrier 1): the OR of the predicates
__device__ __forceinline__ bool epi_barrier_or(bool pred) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r)
                 : "r"((uint32_t)pred), "r"(kEpiThreads)
                 : "memory");
    return r != 0;
}

// kSel: select mode (idx_mqa_topk_paged). The logits go to the workspace's scratch rows; a
// sequence's top-k is selected by the CTA that completes its last tiles: a CTA owns the
// sequences wholly inside its slice, and for the (at most two) sequences it shares with
// other CTAs it adds its tile count to the sequence's arrival counter, the CTA that brings
// the counter to the sequence's tile count selecting (and resetting the counter). The four
// epilogue warps select with the freed stage ring as their work area.
template <int kDtype, int NP, bool kSel>
__global__ void __launch_bounds__(kThreads, Cfg<kDtype, NP>::kCps) decode_kernel(ScoreArgs a) {
    using C = Cfg<kDtype, NP>;
    constexpr int G = C::G;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::oBars);
    uint64_t* k_full = bars;              // per stage group: G arrivals (+ bytes)
    uint64_t* k_empty = k_full + C::kSG;  // per stage group: one commit
    uint64_t* q_full = k_empty + C::kSG;
    uint64_t* q_empty = q_full + C::kQS;
    uint64_t* acc_full = q_empty + C::kQS;
    uint64_t* acc_empty = acc_full + kAccG;
    uint64_t* drain = acc_empty + kAccG;  // the MMA issuer's last commit when it gives up
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::oMisc);
    // misc[0] tmem base, misc[1] start sequence, misc[2..3] start tile, misc[4..5] unit count,
    // misc[6] abort flag
    volatile uint32_t* abort_flag = misc + 6;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, P = a.page_size;
    const int lp = P == 128 ? 7 : 6;  // log2 of the page size (64 or 128)
    const int Hq = (H + 7) & ~7;

    SeqEnt* seq_tab = reinterpret_cast<SeqEnt*>(smem + C::oSeq);
    const uint64_t keep = tc::policy_evict_last();  // lengths and page table: read every launch

    // ---- this CTA's slice of the units: two warp-wide scans over the sequences ----------
    // The first reads every sequence (eight per lane, loads issued together; the first 256
    // sequences' tile counts stay in registers); the second finds the slice's first unit.
    if (warp == 0) {
        int64_t total = 0;
        bool bad = false;  // a sequence broke its length bounds (reported by CTA 0)
        SeqInfo s0[8];  // the first 256 sequences: sequence 32k + lane in s0[k]
        for (int base = 0; base < a.B; base += 256) {
            SeqInfo si[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int b = base + 32 * k + lane;
                si[k] = b < a.B ? seq_info(a, b, keep, &bad) : SeqInfo{0, 0, 0};
            }
            int64_t n = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (base == 0) s0[k] = si[k];
                n += si[k].tiles;
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) n += __shfl_xor_sync(kFull, n, o);
            total += n;
        }
        if (__any_sync(kFull, bad) && blockIdx.x == 0 && lane == 0) report(a.dev_status, IDX_STATUS_BAD_LEN);
        const int64_t u0 = total * blockIdx.x / gridDim.x, u1 = total * (blockIdx.x + 1) / gridDim.x;
        int64_t acc = 0;
        int b0 = a.B;
        int64_t j0 = 0;
        auto scan32 = [&](int base, int64_t n) {  // one chunk of 32 sequences in order
            int64_t inc = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(kFull, inc, o);
                if (lane >= o) inc += y;
            }
            const bool hit = n > 0 && acc + inc - n <= u0 && u0 < acc + inc;
            const unsigned m = __ballot_sync(kFull, hit);
            if (m) {
                const int src = __ffs(m) - 1;
                b0 = base + src;
                j0 = u0 - (acc + __shfl_sync(kFull, inc - n, src));
            }
            acc += __shfl_sync(kFull, inc, 31);
        };
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (32 * k < a.B && b0 == a.B) scan32(32 * k, 32 * k + lane < a.B ? s0[k].tiles : 0);
        for (int base = 256; base < a.B && b0 == a.B; base += 32) {
            const int b = base + lane;
            scan32(base, b < a.B ? seq_info(a, b, keep).tiles : 0);
        }
        {  // the table of the window of sequences from b0 on (from registers when b0 + 31 < 256)
            const int b = b0 + lane;
            SeqInfo si{0, 0, 0};
            if (b0 + 31 < 256) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int32_t t = __shfl_sync(kFull, s0[k].t, b & 31);
                    const int32_t v = __shfl_sync(kFull, s0[k].vis, b & 31);
                    const int32_t n = __shfl_sync(kFull, s0[k].tiles, b & 31);
                    if ((b >> 5) == k && b < a.B) si = SeqInfo{t, v, n};
                }
            } else if (b < a.B) {
                si = seq_info(a, b, keep);
            }
            seq_tab[lane] = SeqEnt{si.t, si.vis, si.tiles, 0};
        }
        if (lane == 0) {
            const int64_t n = b0 < a.B ? u1 - u0 : 0;
            misc[1] = (uint32_t)b0;
            misc[2] = (uint32_t)j0;
            misc[3] = (uint32_t)(j0 >> 32);
            misc[4] = (uint32_t)n;
            misc[5] = (uint32_t)(n >> 32);
            misc[6] = 0;
        }
        // the barriers, spread over the warp's lanes
        for (int i = lane; i < C::kSG; i += 32) {
            tc::mbar_init(&k_full[i], G);
            tc::mbar_init(&k_empty[i], 1);
        }
        if (lane < C::kQS) {
            tc::mbar_init(&q_full[lane], 1);
            tc::mbar_init(&q_empty[lane], 1);
        }
        if (lane == 0) tc::mbar_init(drain, 1);
        if (lane < kAccG) {
            tc::mbar_init(&acc_full[lane], 1);
            tc::mbar_init(&acc_empty[lane], kEpiThreads);
        }
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&misc[0], C::kCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    // the prologue read only the caller's lengths; Q, weights and the cache come from the
    // previous kernels (the producer issues its first page lookups before it waits)
    if (warp != 0) {
        pdl_wait();
        pdl_launch_dependents();
    }
    const uint32_t tbase = misc[0];
    const int b_start = (int)misc[1];
    const Seqs S{&a, seq_tab, b_start, keep};
    const int32_t j_start = (int32_t)misc[2];
    const int64_t n_units = (int64_t)misc[4] | ((int64_t)misc[5] << 32);
    const int64_t n_groups = (n_units + G - 1) / G;
    const int64_t n_slots = n_groups * G;  // tile slots incl. the last group's empty ones
    if constexpr (kSel) {
        if (warp >= 2) pad_orphan_rows(a, tid - 64, kEpiThreads);
    }

    if (warp == 0 && n_units > 0) {
        // ---------------------------------------------------------------- producer warp
        // Tiles go out in batches of up to kBatch: lane L owns tile slot i0+L and issues its
        // page lookups, its stage-group wait and its bulk copies, so the warp issues the
        // batch at once. A batch touches at most kQS sequences: then every wait of a lane
        // (a stage group or a Q slot being released) depends only on tiles of earlier
        // batches, never on a lane of the same batch. Empty slots of the last group arrive
        // without bytes.
        const uint64_t stream = tc::policy_evict_first();  // the cache is read once
        Walker w;  // position of the batch's first unit (same in every lane)
        w.init(S, b_start, j_start);
        int prev_b = -1;     // sequence of the unit before the batch
        int64_t q_base = 0;  // sequences started before the batch
        int64_t armed_g = -1, armed_q = -1;  // last stage group / Q fill armed (warp-wide)
        bool dep_done = false;               // the first batch's page lookups precede pdl_wait
        for (int64_t i0 = 0; i0 < n_slots && !__any_sync(kFull, *abort_flag != 0);) {
            int nb = (int)min((int64_t)C::kBatch, n_units - i0);  // real tiles (may be <= 0)
            Walker my = w;
            for (int k = 0; k < lane && k + 1 < nb; ++k) my.next(S);
            const int b_before = __shfl_up_sync(kFull, my.b, 1);
            unsigned starts = __ballot_sync(kFull, lane < nb && my.b != (lane == 0 ? prev_b : b_before));
            const int allowed = C::kQS - (nb > 0 && w.b == prev_b ? 1 : 0);
            if (__popc(starts) > allowed) {
                unsigned m = starts;  // cut the batch at the (allowed+1)-th sequence start
                for (int r = 0; r < allowed; ++r) m &= m - 1;
                nb = __ffs(m) - 1;
                starts &= (1u << nb) - 1u;
            }
            const bool real = lane < nb;
            const bool newseq = real && ((starts >> lane) & 1u);
            const int ns = i0 + nb >= n_units ? (int)min((int64_t)C::kBatch, n_slots - i0) : nb;  // slots
            if (lane < ns) {
                const int64_t i = i0 + lane;
                const int64_t gi = i / G;
                const int grp = (int)(gi % C::kSG);
                int32_t pg[2] = {-1, -1};
                int halves = 0;
                if (real) {
                    const int64_t key0 = my.j * 128;
                    halves = P == 128 ? 1 : (key0 + 64 < my.si.vis ? 2 : 1);
                    const int32_t* pt = a.page_table + (int64_t)my.b * a.pt_stride;
                    pg[0] = tc::ld_hint(pt + (key0 >> lp), keep);
                    if (halves == 2) pg[1] = tc::ld_hint(pt + ((key0 + 64) >> lp), keep);
                }
                if (!dep_done) {  // Q and the cache come from the previous kernels
                    pdl_wait();
                    pdl_launch_dependents();
                    dep_done = true;
                }
                if (real) {
                    if (newseq) {
                        const int64_t qk = q_base + __popc(starts & ((2u << lane) - 1)) - 1;
                        const int slot = (int)(qk % C::kQS);
                        if (!tc::mbar_wait(&q_empty[slot], (uint32_t)(((qk / C::kQS) & 1) ^ 1))) {
                            *abort_flag = 1;
                        } else {
                            const uint32_t qbytes = (uint32_t)(Hq * C::kQRow);
                            tc::mbar_arrive_expect_tx(&q_full[slot], qbytes + C::kQSf);
                            tc::bulk_g2s(smem + C::oQ + slot * C::kQImg, a.q_codes + (int64_t)my.si.t * Hq * C::kQRow,
                                         qbytes, &q_full[slot]);
                            if (kDtype == IDX_MXFP4)
                                tc::bulk_g2s(smem + C::oQSf + slot * C::kQSf, a.q_scales + (int64_t)my.si.t * 512, 512,
                                             &q_full[slot]);
                        }
                    }
                }
                if (*abort_flag || !tc::mbar_wait(&k_empty[grp], (uint32_t)(((gi / C::kSG) & 1) ^ 1))) {
                    *abort_flag = 1;
                } else {
                    uint32_t bytes = 0;
                    for (int h = 0; h < halves; ++h) {
                        if (pg[h] >= 0 && pg[h] < a.num_pages) {
                            bytes += (uint32_t)(P * (C::kTileCode / 128 + C::kTileSf / 128));
                        } else {
                            report(a.dev_status, IDX_STATUS_BAD_PAGE);
                            pg[h] = -1;
                        }
                    }
                    tc::mbar_arrive_expect_tx(&k_full[grp], bytes);
                    uint8_t* dK = smem + C::oStages + grp * C::kGroup + (int)(i % G) * C::kTile;
                    uint8_t* dS = dK + C::kTileCode;
                    for (int h = 0; h < halves; ++h) {
                        if (pg[h] < 0) continue;
                        const uint8_t* src = a.pool + (int64_t)pg[h] * a.page_stride;
                        if (P == 128) {
                            // codes and scale atom are contiguous in the page and in the stage
                            tc::bulk_g2s_hint(dK, src, C::kTile, &k_full[grp], stream);
                        } else if (kDtype == IDX_MXFP4) {
                            // four 1 KB chunks of 16 keys interleave with the other page's chunks
                            for (int q = 0; q < 4; ++q)
                                tc::bulk_g2s_hint(dK + q * 2048 + h * 1024, src + q * 1024, 1024, &k_full[grp], stream);
                            tc::bulk_g2s_hint(dS + h * 256, src + 4096, 256, &k_full[grp], stream);
                        } else {
                            tc::bulk_g2s_hint(dK + h * 8192, src, 8192, &k_full[grp], stream);
                        }
                    }
                }
            }
            __syncwarp();
            armed_g = (i0 + ns - 1) / G;
            armed_q = q_base + __popc(starts) - 1;
            if (nb <= 0) break;
            // next batch: one unit after this batch's last real unit
            Walker last = my;
            last.b = __shfl_sync(kFull, my.b, nb - 1);
            last.j = __shfl_sync(kFull, my.j, nb - 1);
            last.si.t = __shfl_sync(kFull, my.si.t, nb - 1);
            last.si.vis = __shfl_sync(kFull, my.si.vis, nb - 1);
            last.si.tiles = __shfl_sync(kFull, my.si.tiles, nb - 1);
            prev_b = last.b;
            q_base += __popc(starts);
            w = last;
            if (i0 + nb < n_units) w.next(S);
            i0 += ns;
        }
        if (*abort_flag) {
            // do not leave while copies are in flight: wait (bounded) for the last fill armed
            // in each stage group and each Q slot
            const uint64_t deadline = tc::global_ns() + tc::kWaitLimitNs;
            if (lane < C::kSG && armed_g >= lane) {
                const int64_t g = armed_g - ((armed_g - lane) % C::kSG);
                tc::mbar_wait_until(&k_full[lane], (uint32_t)((g / C::kSG) & 1), deadline);
            }
            if (lane < C::kQS && armed_q >= lane) {
                const int64_t q = armed_q - ((armed_q - lane) % C::kQS);
                tc::mbar_wait_until(&q_full[lane], (uint32_t)((q / C::kQS) & 1), deadline);
            }
        }
        if (lane == 0 && *abort_flag) report(a.dev_status, IDX_STATUS_TIMEOUT);
    } else if (warp == 1 && lane == 0 && n_units > 0) {
        // ---------------------------------------------------------------- MMA issuer
        // tensor memory: accumulators [kAccG][G][NP], then A scale slots [kAccG][G][4] (a slot
        // is rewritten only after the epilogue released its accumulator group, i.e. after the
        // MMAs that read it ended), then the B scale slot of each Q slot [kQS][4]
        const uint32_t t_sfa = tbase + kAccG * G * NP;
        const uint32_t t_sfb = t_sfa + kAccG * G * 4;
        // descriptors of stage 0 / Q slot 0; other tiles, slots and K steps add (bytes >> 4)
        // to the start-address field (shared-memory addresses stay below 256 KB)
        const uint64_t dA0 = tc::smem_desc(tc::smem_u32(smem + C::oStages), 128, C::kSbo);
        const uint64_t dB0 = tc::smem_desc(tc::smem_u32(smem + C::oQ), 128, C::kSbo);
        const uint64_t dSA0 = tc::smem_desc(tc::smem_u32(smem + C::oStages + C::kTileCode), 128, 128);
        const uint64_t dSB0 = tc::smem_desc(tc::smem_u32(smem + C::oQSf), 128, 128);
        const uint32_t id0 = kDtype == IDX_MXFP4 ? tc::idesc_mxf4(128, NP, 0, 0) : tc::idesc_f8(128, NP);
        const uint32_t id1 = kDtype == IDX_MXFP4 ? tc::idesc_mxf4(128, NP, 2, 2) : id0;
        Walker w;
        w.init(S, b_start, j_start);
        int prev_b = -1;
        int64_t qk = -1;
        int slot = 0;
        int grp = 0, ag = 0;
        uint32_t kph = 0, aph = 1;  // parity to wait for: k_full[grp], acc_empty[ag]
        for (int64_t gi = 0; gi < n_groups; ++gi) {
            if (*abort_flag) break;
            if (!tc::mbar_wait(&k_full[grp], kph) || !tc::mbar_wait(&acc_empty[ag], aph)) {
                *abort_flag = 1;
                break;
            }
            tc::tc_fence_after();
            for (int t = 0; t < G; ++t) {
                const int64_t i = gi * G + t;
                if (i >= n_units) break;
                if (w.b != prev_b) {
                    ++qk;
                    slot = (int)(qk % C::kQS);
                    if (!tc::mbar_wait(&q_full[slot], (uint32_t)((qk / C::kQS) & 1))) {
                        *abort_flag = 1;
                        break;
                    }
                    tc::tc_fence_after();
                    if (kDtype == IDX_MXFP4)
                        tc::cp_32x128b_warpx4(t_sfb + 4 * slot, dSB0 + (uint64_t)((slot * C::kQSf) >> 4));
                    prev_b = w.b;
                }
                const int cell = ag * G + t;
                const uint32_t d = tbase + cell * NP;
                const int off = grp * C::kGroup + t * C::kTile;
                const uint64_t da = dA0 + (uint64_t)(off >> 4);
                const uint64_t db = dB0 + (uint64_t)((slot * C::kQImg) >> 4);
                if (kDtype == IDX_MXFP4) {
                    const uint32_t sfa = t_sfa + 4 * cell;
                    tc::cp_32x128b_warpx4(sfa, dSA0 + (uint64_t)(off >> 4));
                    tc::mma_mxf4(d, da, db, id0, sfa, t_sfb + 4 * slot, 0);
                    tc::mma_mxf4(d, da + 16, db + 16, id1, sfa, t_sfb + 4 * slot, 1);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) tc::mma_f8(d, da + 16 * k, db + 16 * k, id0, k);
                }
                const int cur_b = w.b;
                w.next(S);
                if (i + 1 == n_units || w.b != cur_b) tc::mma_commit(&q_empty[slot]);
            }
            if (*abort_flag) break;
            tc::mma_commit(&k_empty[grp]);
            tc::mma_commit(&acc_full[ag]);
            if (++grp == C::kSG) { grp = 0; kph ^= 1; }
            if (++ag == kAccG) { ag = 0; aph ^= 1; }
        }
        if (*abort_flag) {
            // do not free tensor memory under MMAs still running: one more commit tracks
            // every tcgen05 operation issued so far; wait (bounded) for it
            report(a.dev_status, IDX_STATUS_TIMEOUT);
            tc::mma_commit(drain);
            tc::mbar_wait(drain, 0);
        }
    } else if (warp >= 2 && n_units > 0) {
        // ---------------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int m = quad * 32 + lane;
        const uint32_t lane_addr = tbase + ((uint32_t)(quad * 32) << 16);
        // key offset of TMEM row m inside its tile: for two 64-key MXFP4 pages, rows with
        // m % 32 < 16 hold the first page's keys (m % 16) + 16 * (m / 32)
        const bool split = P == 64 && kDtype == IDX_MXFP4;
        const int half = split ? ((m >> 4) & 1) : (m >> 6);
        const int koff = split ? (64 * half + (m & 15) + 16 * (m >> 5)) : m;
        Walker w;
        w.init(S, b_start, j_start);
        int prev_b = -1;
        float wr[NP];
        int ag = 0;
        uint32_t aph = 0;
        for (int64_t gi = 0; gi < n_groups; ++gi) {
            // the group's page lookups are issued before the accumulator wait (their latency
            // hides behind it); their values are used after it
            int32_t pg[G];
            Walker wk = w;
#pragma unroll
            for (int t = 0; t < G; ++t) {
                const int64_t i = gi * G + t;
                const int64_t key = wk.j * 128 + koff;
                pg[t] = (i < n_units && key < wk.si.vis)
                            ? tc::ld_hint(a.page_table + (int64_t)wk.b * a.pt_stride + (key >> lp), keep)
                            : -1;
                if (i + 1 < n_units) wk.next(S);
            }
            // so are the head weights when the group's first tile starts a sequence
            if (w.b != prev_b) {
#pragma unroll
                for (int h = 0; h < NP; ++h) wr[h] = h < H ? __ldg(a.w + (int64_t)w.si.t * H + h) : 0.0f;
                prev_b = w.b;
            }
            const bool got = __all_sync(kFull, tc::mbar_wait(&acc_full[ag], aph));
            if (!got) {
                *abort_flag = 1;
                report(a.dev_status, IDX_STATUS_TIMEOUT);
                break;
            }
            tc::tc_fence_after();
#pragma unroll
            for (int t = 0; t < G; ++t) {
                const int64_t i = gi * G + t;
                if (i >= n_units) break;
                if (w.b != prev_b) {
#pragma unroll
                    for (int h = 0; h < NP; ++h) wr[h] = h < H ? __ldg(a.w + (int64_t)w.si.t * H + h) : 0.0f;
                    prev_b = w.b;
                }
                const int64_t key = w.j * 128 + koff;
                const bool key_ok = key < w.si.vis && pg[t] >= 0 && pg[t] < a.num_pages;
                float kscale = 1.0f;
                if (kDtype == IDX_FP8 && key_ok)
                    kscale = __ldg(reinterpret_cast<const float*>(a.pool + (int64_t)pg[t] * a.page_stride + 128 * P +
                                                                  4 * ((key & (P - 1)))));
                // four independent accumulation chains over the heads, drained 32 columns at a
                // time (head h always in chain h % 4)
                constexpr int CH = NP < 32 ? NP : 32;
                float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int c = 0; c < NP; c += CH) {
                    float v[CH];
                    load_acc<CH>(lane_addr + (ag * G + t) * NP + c, v);
#pragma unroll
                    for (int h = 0; h < CH; ++h)
                        if (c + h < H) part[h & 3] = fmaf(wr[c + h], fmaxf(v[h], 0.0f), part[h & 3]);
                }
                const float logit = (part[0] + part[1]) + (part[2] + part[3]);
                if (key_ok) a.logits[(int64_t)w.si.t * a.ld + key] = logit * kscale;
                w.next(S);
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&acc_empty[ag]);
            if (++ag == kAccG) { ag = 0; aph ^= 1; }
        }
        if constexpr (kSel) {
            // the four epilogue warps' logits stores are done (or given up on); each sequence
            // of the slice, in order: thread 0 settles whether this CTA selects it, and the
            // group selects the sequences it owns. Every warp runs the same barriers.
            __threadfence();
            const bool stop = epi_barrier_or(*abort_flag != 0);
            const int etid = tid - 64;
            volatile int32_t* own = reinterpret_cast<volatile int32_t*>(misc + 8);  // [0] t, [1] vis, [2] more
            SelectSmem sm;
            sm.hist = reinterpret_cast<uint32_t*>(smem + C::oStages);
            sm.cand = reinterpret_cast<int32_t*>(smem + C::oStages + 8192);
            sm.ckey = reinterpret_cast<uint32_t*>(smem + C::oStages + 8192 + 4 * kSelCand);
            sm.warp_sums = reinterpret_cast<uint32_t*>(smem + C::oStages + 8192 + 8 * kSelCand);
            sm.warp_gt = sm.warp_sums + 4;
            sm.warp_eq = sm.warp_gt + 4;
            sm.scal = sm.warp_eq + 4;
            // the rest of the stage ring stages the row's keys (8K keys for MXFP4, 32 heads)
            sm.keys = reinterpret_cast<uint32_t*>(smem + C::oStages + 8192 + 8 * kSelCand + 128);
            sm.key_cap = (int)((C::kSG * C::kGroup - (8192 + 8 * kSelCand + 128)) / 4);
            Walker ws;  // thread 0's walk over the slice's sequences
            ws.init(S, b_start, j_start);
            int64_t left = stop ? 0 : n_units;  // tiles of the slice not yet attributed
            for (;;) {
                if (etid == 0) {
                    int32_t t_sel = -1, vis_sel = 0;
                    while (left > 0 && t_sel < 0) {
                        const int64_t n_b = min((int64_t)(ws.si.tiles - ws.j), left);
                        bool mine = ws.j == 0 && n_b == ws.si.tiles;  // the whole sequence
                        if (!mine) {
                            int32_t old;
                            asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;"
                                         : "=r"(old)
                                         : "l"(a.counters + ws.b), "r"((int32_t)n_b)
                                         : "memory");
                            mine = old + n_b == ws.si.tiles;
                            if (mine) a.counters[ws.b] = 0;  // for the next call
                        }
                        if (mine) {
                            t_sel = ws.si.t;
                            vis_sel = ws.si.vis;
                        }
                        left -= n_b;
                        ws.j = ws.si.tiles - 1;  // step to the next sequence with tiles
                        if (left > 0) ws.next(S);
                    }
                    own[0] = t_sel;
                    own[1] = vis_sel;
                }
                NamedBarrier{1, kEpiThreads}();
                const int32_t t_sel = own[0], vis_sel = own[1];
                NamedBarrier{1, kEpiThreads}();
                if (t_sel < 0) break;
                select_topk_row<kEpiThreads, kSelCand>(a.logits + (int64_t)t_sel * a.ld, vis_sel, a.topk_k,
                                                        a.out_idx + (int64_t)t_sel * a.topk_k, sm, etid,
                                                        NamedBarrier{1, kEpiThreads});
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, C::kCols);
    }
}


// ---- dynamic schedule ---------------------------------------------------------------------
// With a caller workspace and at most kDynB sequences, the units are handed out as jobs of up
// to kJob tiles of one sequence (about half the stage ring; never more than the ring, since a
// job's tiles go out at once, one per lane, and no lane may wait for a stage that a tile of the
// same job has to free): CTA i starts with job i and claims further jobs from a
// counter in the workspace, so CTAs that start late (their SM still busy with the previous
// kernel) or run slow take fewer tiles and the launch ends when the work does, not when the
// last static slice does. The producer publishes each job (sequence, first tile, tile count)
// in a ring of kJR records that the MMA thread and the epilogue warps read in order; every
// job loads its query into its own Q slot. The CTA that finishes last (a second counter)
// zeroes both counters for the next call.
constexpr int kDynB = 256;  // sequences the job tables hold
constexpr int kJR = 8;      // job records in flight

template <int kDtype, int NP>
struct DynCfg {
    using C = Cfg<kDtype, NP>;
    // Q slots: every job loads its query into the next slot, so the slot ring bounds the jobs
    // in flight; four for every head count (the static kernel keeps two for 64 heads)
    static constexpr int kQS = 4;
    static_assert(kAccG * (NP + 4) + 4 * kQS <= (int)C::kCols, "B scale slots fit the tensor memory");
    // records (16-byte aligned int4), then (t, vis) and the job prefix
    static constexpr int kTab = kJR * 16 + kDynB * 8 + (kDynB + 1) * 4;
    static constexpr int kFixed = kQS * (C::kQImg + C::kQSf) + 64 + 16 + kTab +
                                  8 * (2 * kQS + 1 + 2 * kAccG + 2 * kJR);
    static constexpr int kSG = (C::kBudget - kFixed) / (C::kGroup + 16);
    // tiles per job: about half the stage ring, so that the next job's copies overlap this
    // one's (measured: 4 with ten stages, 2 with four; 1 was slower everywhere)
    static constexpr int kJob = kSG >= 8 ? 4 : (kSG >= 2 ? 2 : 1);
    static constexpr int oStages = 0;
    static constexpr int oQ = kSG * C::kGroup;
    static constexpr int oQSf = oQ + kQS * C::kQImg;
    static constexpr int oBars = oQSf + kQS * C::kQSf;
    static constexpr int kBars = 2 * kSG + 2 * kQS + 1 + 2 * kAccG + 2 * kJR;
    static constexpr int oMisc = oBars + 8 * kBars;
    static constexpr int oTab = (oMisc + 64 + 15) & ~15;  // the int4 records need 16-byte alignment
    static constexpr int kSmem = oTab + kTab;
    static_assert(kSG >= kJob, "a job's tiles fit the stage ring at once");
    static_assert(oTab % 16 == 0 && oBars % 8 == 0, "alignment of the records and barriers");
    static_assert(kSmem <= C::kBudget, "shared memory of the CTAs sharing an SM");
};

template <int kDtype, int NP>
__global__ void __launch_bounds__(kThreads, Cfg<kDtype, NP>::kCps) decode_dyn_kernel(ScoreArgs a) {
    using C = Cfg<kDtype, NP>;
    using D = DynCfg<kDtype, NP>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + D::oBars);
    uint64_t* k_full = bars;
    uint64_t* k_empty = k_full + D::kSG;
    uint64_t* q_full = k_empty + D::kSG;
    uint64_t* q_empty = q_full + D::kQS;
    uint64_t* acc_full = q_empty + D::kQS;
    uint64_t* acc_empty = acc_full + kAccG;
    uint64_t* drain = acc_empty + kAccG;
    uint64_t* j_full = drain + 1;     // a record was written (the producer's arrival)
    uint64_t* j_empty = j_full + kJR;  // a record was read (MMA thread + one lane per epilogue warp)
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + D::oMisc);  // [0] tmem, [1] jobs, [2] abort
    volatile uint32_t* abort_flag = misc + 2;
    int4* jrec = reinterpret_cast<int4*>(smem + D::oTab);                    // [kJR] (b, first tile, tiles, -)
    int32_t* seq_t = reinterpret_cast<int32_t*>(smem + D::oTab + kJR * 16);  // [kDynB] query row
    int32_t* seq_vis = seq_t + kDynB;                                         // [kDynB] visible keys
    int32_t* jpre = seq_vis + kDynB;                                          // [kDynB + 1] jobs before b
    int32_t* counters = a.counters;  // [0] next job - gridDim.x, [1] CTAs finished

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, P = a.page_size;
    const int lp = P == 128 ? 7 : 6;
    const int Hq = (H + 7) & ~7;
    const uint64_t keep = tc::policy_evict_last();

    // ---- prologue: every sequence's query row, visible keys and jobs (eight per lane) -------
    int32_t pre_pg[2] = {-1, -1};  // warp 0: the first job's pages (lane L: tile L)
    if (warp == 0) {
        bool bad = false;
        int32_t carry = 0;
        // every sequence's three values are loaded before any is used: one round trip
        int32_t q0[8], q1[8], len[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int b = 32 * k + lane;
            q0[k] = q1[k] = len[k] = 0;
            if (b < a.B) {
                q0[k] = tc::ld_hint(a.cu_seqlens_q + b, keep);
                q1[k] = tc::ld_hint(a.cu_seqlens_q + b + 1, keep);
                len[k] = tc::ld_hint(a.seq_lens_k + b, keep);
            }
        }
        SeqInfo si[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) si[k] = seq_info_of(a, q0[k], q1[k], len[k], &bad);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (32 * k >= a.B) break;
            const int b = 32 * k + lane;
            const int32_t n = (si[k].tiles + D::kJob - 1) / D::kJob;
            int32_t inc = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(kFull, inc, o);
                if (lane >= o) inc += y;
            }
            if (b < a.B) {
                seq_t[b] = si[k].t;
                seq_vis[b] = si[k].vis;
                jpre[b] = carry + inc - n;
            }
            carry += __shfl_sync(kFull, inc, 31);
        }
        if (lane == 0) {
            jpre[a.B] = carry;
            misc[1] = (uint32_t)carry;
            misc[2] = 0;
        }
        __syncwarp();
        if (__any_sync(kFull, bad) && blockIdx.x == 0 && lane == 0) report(a.dev_status, IDX_STATUS_BAD_LEN);
        // the first job's page lookups (job blockIdx.x) go out now: their round trip overlaps
        // the barrier set-up and the CTA barrier below
        if ((int32_t)blockIdx.x < carry) {
            const int32_t c0 = (int32_t)blockIdx.x;
            int lo = 0, hi = a.B;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (jpre[mid] <= c0) lo = mid; else hi = mid;
            }
            const int32_t j00 = D::kJob * (c0 - jpre[lo]);
            const int32_t n0 = min(D::kJob, (seq_vis[lo] + 127) / 128 - j00);
            if (lane < n0) {
                const int64_t key0 = (int64_t)(j00 + lane) * 128;
                const int32_t* pt = a.page_table + (int64_t)lo * a.pt_stride;
                pre_pg[0] = tc::ld_hint(pt + (key0 >> lp), keep);
                if (P == 64 && key0 + 64 < seq_vis[lo]) pre_pg[1] = tc::ld_hint(pt + ((key0 + 64) >> lp), keep);
            }
        }
        for (int i = lane; i < D::kSG; i += 32) {
            tc::mbar_init(&k_full[i], 1);
            tc::mbar_init(&k_empty[i], 1);
        }
        if (lane < D::kQS) {
            tc::mbar_init(&q_full[lane], 1);
            tc::mbar_init(&q_empty[lane], 1);
        }
        if (lane == 0) tc::mbar_init(drain, 1);
        if (lane < kAccG) {
            tc::mbar_init(&acc_full[lane], 1);
            tc::mbar_init(&acc_empty[lane], kEpiThreads);
        }
        if (lane < kJR) {
            tc::mbar_init(&j_full[lane], 1);
            tc::mbar_init(&j_empty[lane], 5);
        }
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&misc[0], C::kCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp != 0) {
        pdl_wait();
        pdl_launch_dependents();
    }
    const uint32_t tbase = misc[0];
    const int32_t n_jobs = (int32_t)misc[1];

    if (warp == 0) {
        // ---------------------------------------------------------------- producer warp
        // Job c of sequence b (jpre[b] <= c < jpre[b + 1]) holds tiles kJob * (c - jpre[b]) on;
        // lane L issues tile L of the job (its page lookups, stage wait and copies).
        const uint64_t stream = tc::policy_evict_first();
        int32_t c = (int32_t)blockIdx.x;  // the first job needs no claim
        int32_t next = -1;
        int64_t i = 0;  // tiles issued so far
        int64_t q = 0;  // jobs published so far
        int64_t armed_g = -1, armed_q = -1;
        bool dep_done = false;
        for (;;) {
            if (__any_sync(kFull, *abort_flag != 0)) break;
            const int slot = (int)(q % kJR);
            const bool end = c >= n_jobs;
            int b = 0, j0 = 0, n = 0;
            if (!end) {
                int lo = 0, hi = a.B;  // the sequence of job c: jpre[lo] <= c < jpre[hi]
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (jpre[mid] <= c) lo = mid; else hi = mid;
                }
                b = lo;
                j0 = D::kJob * (c - jpre[b]);
                n = min(D::kJob, (seq_vis[b] + 127) / 128 - j0);
            }
            // the record: wait until its slot's previous record was read by every consumer
            if (lane == 0) {
                if (!tc::mbar_wait(&j_empty[slot], (uint32_t)(((q / kJR) & 1) ^ 1))) {
                    *abort_flag = 1;
                } else {
                    jrec[slot] = make_int4(end ? -1 : b, j0, n, 0);
                    tc::mbar_arrive(&j_full[slot]);
                }
            }
            __syncwarp();
            if (end || *abort_flag) break;
            int32_t pg[2] = {-1, -1};
            int halves = 0;
            const int vis = seq_vis[b];
            if (lane < n) {
                const int64_t key0 = (int64_t)(j0 + lane) * 128;
                halves = P == 128 ? 1 : (key0 + 64 < vis ? 2 : 1);
                if (q == 0) {  // looked up in the prologue
                    pg[0] = pre_pg[0];
                    pg[1] = pre_pg[1];
                } else {
                    const int32_t* pt = a.page_table + (int64_t)b * a.pt_stride;
                    pg[0] = tc::ld_hint(pt + (key0 >> lp), keep);
                    if (halves == 2) pg[1] = tc::ld_hint(pt + ((key0 + 64) >> lp), keep);
                }
            }
            if (!dep_done) {  // Q, the cache and the counters come from the previous kernels
                pdl_wait();
                pdl_launch_dependents();
                dep_done = true;
            }
            // claim the job after this one (its latency hides behind this job's copies)
            if (lane == 0) next = atomicAdd(counters, 1) + (int32_t)gridDim.x;
            if (lane == 0) {
                const int qs = (int)(q % D::kQS);
                if (!tc::mbar_wait(&q_empty[qs], (uint32_t)(((q / D::kQS) & 1) ^ 1))) {
                    *abort_flag = 1;
                } else {
                    const uint32_t qbytes = (uint32_t)(Hq * C::kQRow);
                    const int32_t t = seq_t[b];
                    tc::mbar_arrive_expect_tx(&q_full[qs], qbytes + C::kQSf);
                    tc::bulk_g2s(smem + D::oQ + qs * C::kQImg, a.q_codes + (int64_t)t * Hq * C::kQRow, qbytes,
                                 &q_full[qs]);
                    if (kDtype == IDX_MXFP4)
                        tc::bulk_g2s(smem + D::oQSf + qs * C::kQSf, a.q_scales + (int64_t)t * 512, 512, &q_full[qs]);
                }
            }
            if (lane < n) {
                const int64_t it = i + lane;
                const int grp = (int)(it % D::kSG);
                if (*abort_flag || !tc::mbar_wait(&k_empty[grp], (uint32_t)(((it / D::kSG) & 1) ^ 1))) {
                    *abort_flag = 1;
                } else {
                    uint32_t bytes = 0;
                    for (int h = 0; h < halves; ++h) {
                        if (pg[h] >= 0 && pg[h] < a.num_pages) {
                            bytes += (uint32_t)(P * (C::kTileCode / 128 + C::kTileSf / 128));
                        } else {
                            report(a.dev_status, IDX_STATUS_BAD_PAGE);
                            pg[h] = -1;
                        }
                    }
                    tc::mbar_arrive_expect_tx(&k_full[grp], bytes);
                    uint8_t* dK = smem + D::oStages + grp * C::kGroup;
                    uint8_t* dS = dK + C::kTileCode;
                    for (int h = 0; h < halves; ++h) {
                        if (pg[h] < 0) continue;
                        const uint8_t* src = a.pool + (int64_t)pg[h] * a.page_stride;
                        if (P == 128) {
                            tc::bulk_g2s_hint(dK, src, C::kTile, &k_full[grp], stream);
                        } else if (kDtype == IDX_MXFP4) {
                            for (int qq = 0; qq < 4; ++qq)
                                tc::bulk_g2s_hint(dK + qq * 2048 + h * 1024, src + qq * 1024, 1024, &k_full[grp], stream);
                            tc::bulk_g2s_hint(dS + h * 256, src + 4096, 256, &k_full[grp], stream);
                        } else {
                            tc::bulk_g2s_hint(dK + h * 8192, src, 8192, &k_full[grp], stream);
                        }
                    }
                }
            }
            __syncwarp();
            armed_g = i + n - 1;
            armed_q = q;
            i += n;
            ++q;
            c = __shfl_sync(kFull, next, 0);
        }
        if (*abort_flag) {
            const uint64_t deadline = tc::global_ns() + tc::kWaitLimitNs;
            if (lane < D::kSG && armed_g >= lane) {
                const int64_t g = armed_g - ((armed_g - lane) % D::kSG);
                tc::mbar_wait_until(&k_full[lane], (uint32_t)((g / D::kSG) & 1), deadline);
            }
            if (lane < D::kQS && armed_q >= lane) {
                const int64_t g = armed_q - ((armed_q - lane) % D::kQS);
                tc::mbar_wait_until(&q_full[lane], (uint32_t)((g / D::kQS) & 1), deadline);
            }
            if (lane == 0) {
                // the consumers stop at the abort flag or at a record that never comes
                report(a.dev_status, IDX_STATUS_TIMEOUT);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        const uint32_t t_sfa = tbase + kAccG * NP;
        const uint32_t t_sfb = t_sfa + kAccG * 4;
        const uint64_t dA0 = tc::smem_desc(tc::smem_u32(smem + D::oStages), 128, C::kSbo);
        const uint64_t dB0 = tc::smem_desc(tc::smem_u32(smem + D::oQ), 128, C::kSbo);
        const uint64_t dSA0 = tc::smem_desc(tc::smem_u32(smem + D::oStages + C::kTileCode), 128, 128);
        const uint64_t dSB0 = tc::smem_desc(tc::smem_u32(smem + D::oQSf), 128, 128);
        const uint32_t id0 = kDtype == IDX_MXFP4 ? tc::idesc_mxf4(128, NP, 0, 0) : tc::idesc_f8(128, NP);
        const uint32_t id1 = kDtype == IDX_MXFP4 ? tc::idesc_mxf4(128, NP, 2, 2) : id0;
        int grp = 0, ag = 0;
        uint32_t kph = 0, aph = 1;
        for (int64_t q = 0;; ++q) {
            const int slot = (int)(q % kJR);
            if (*abort_flag || !tc::mbar_wait(&j_full[slot], (uint32_t)((q / kJR) & 1))) {
                *abort_flag = 1;
                break;
            }
            const int4 r = jrec[slot];
            tc::mbar_arrive(&j_empty[slot]);
            if (r.x < 0) break;
            const int qs = (int)(q % D::kQS);
            if (!tc::mbar_wait(&q_full[qs], (uint32_t)((q / D::kQS) & 1))) {
                *abort_flag = 1;
                break;
            }
            tc::tc_fence_after();
            if (kDtype == IDX_MXFP4) tc::cp_32x128b_warpx4(t_sfb + 4 * qs, dSB0 + (uint64_t)((qs * C::kQSf) >> 4));
            for (int t = 0; t < r.z; ++t) {
                if (!tc::mbar_wait(&k_full[grp], kph) || !tc::mbar_wait(&acc_empty[ag], aph)) {
                    *abort_flag = 1;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t d = tbase + ag * NP;
                const int off = grp * C::kGroup;
                const uint64_t da = dA0 + (uint64_t)(off >> 4);
                const uint64_t db = dB0 + (uint64_t)((qs * C::kQImg) >> 4);
                if (kDtype == IDX_MXFP4) {
                    const uint32_t sfa = t_sfa + 4 * ag;
                    tc::cp_32x128b_warpx4(sfa, dSA0 + (uint64_t)(off >> 4));
                    tc::mma_mxf4(d, da, db, id0, sfa, t_sfb + 4 * qs, 0);
                    tc::mma_mxf4(d, da + 16, db + 16, id1, sfa, t_sfb + 4 * qs, 1);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) tc::mma_f8(d, da + 16 * k, db + 16 * k, id0, k);
                }
                if (t + 1 == r.z) tc::mma_commit(&q_empty[qs]);
                tc::mma_commit(&k_empty[grp]);
                tc::mma_commit(&acc_full[ag]);
                if (++grp == D::kSG) { grp = 0; kph ^= 1; }
                if (++ag == kAccG) { ag = 0; aph ^= 1; }
            }
            if (*abort_flag) break;
        }
        if (*abort_flag) {
            report(a.dev_status, IDX_STATUS_TIMEOUT);
            tc::mma_commit(drain);
            tc::mbar_wait(drain, 0);
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int m = quad * 32 + lane;
        const uint32_t lane_addr = tbase + ((uint32_t)(quad * 32) << 16);
        const bool split = P == 64 && kDtype == IDX_MXFP4;
        const int half = split ? ((m >> 4) & 1) : (m >> 6);
        const int koff = split ? (64 * half + (m & 15) + 16 * (m >> 5)) : m;
        float wr[NP];
        int ag = 0;
        uint32_t aph = 0;
        for (int64_t q = 0;; ++q) {
            const int slot = (int)(q % kJR);
            const bool got = __all_sync(kFull, *abort_flag == 0 && tc::mbar_wait(&j_full[slot], (uint32_t)((q / kJR) & 1)));
            if (!got) {
                *abort_flag = 1;
                report(a.dev_status, IDX_STATUS_TIMEOUT);
                break;
            }
            const int4 r = jrec[slot];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&j_empty[slot]);
            if (r.x < 0) break;
            const int32_t t_q = seq_t[r.x], vis = seq_vis[r.x];
#pragma unroll
            for (int h = 0; h < NP; ++h) wr[h] = h < H ? __ldg(a.w + (int64_t)t_q * H + h) : 0.0f;
            bool stop = false;
            for (int t = 0; t < r.z; ++t) {
                const int64_t key = (int64_t)(r.y + t) * 128 + koff;
                const int32_t pg = key < vis ? tc::ld_hint(a.page_table + (int64_t)r.x * a.pt_stride + (key >> lp), keep)
                                             : -1;
                const bool ok = __all_sync(kFull, tc::mbar_wait(&acc_full[ag], aph));
                if (!ok) {
                    *abort_flag = 1;
                    report(a.dev_status, IDX_STATUS_TIMEOUT);
                    stop = true;
                    break;
                }
                tc::tc_fence_after();
                const bool key_ok = key < vis && pg >= 0 && pg < a.num_pages;
                float kscale = 1.0f;
                if (kDtype == IDX_FP8 && key_ok)
                    kscale = __ldg(reinterpret_cast<const float*>(a.pool + (int64_t)pg * a.page_stride + 128 * P +
                                                                  4 * ((key & (P - 1)))));
                constexpr int CH = NP < 32 ? NP : 32;
                float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int cc = 0; cc < NP; cc += CH) {
                    float v[CH];
                    load_acc<CH>(lane_addr + ag * NP + cc, v);
#pragma unroll
                    for (int h = 0; h < CH; ++h)
                        if (cc + h < H) part[h & 3] = fmaf(wr[cc + h], fmaxf(v[h], 0.0f), part[h & 3]);
                }
                const float logit = (part[0] + part[1]) + (part[2] + part[3]);
                if (key_ok) a.logits[(int64_t)t_q * a.ld + key] = logit * kscale;
                tc::tc_fence_before();
                tc::mbar_arrive(&acc_empty[ag]);
                if (++ag == kAccG) { ag = 0; aph ^= 1; }
            }
            if (stop) break;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, C::kCols);
    }
    if (tid == 0) {
        // every claim of this CTA has returned; the last CTA to get here zeroes the counters
        // (not before the previous kernels are done: they may still be resetting them)
        pdl_wait();
        __threadfence();
        if (atomicAdd(counters + 1, 1) == (int32_t)gridDim.x - 1) {
            counters[0] = 0;
            counters[1] = 0;
        }
    }
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

template <int kDtype, int NP, bool kSel>
cudaError_t launch_np(const ScoreArgs& a, cudaStream_t st) {
    using C = Cfg<kDtype, NP>;
    static_assert(C::kSG * C::kGroup >= 8192 + 8 * kSelCand + 128, "select mode's work area fits the stage ring");
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<kDtype, NP, kSel>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    // an upper bound of the unit count sizes the grid (a CTA with no units exits)
    const int64_t units_max = (int64_t)a.B * ((a.max_seq_len_k + 127) / 128);
    const int ctas = C::kCps * sm_count();
    const int grid = (int)(units_max < ctas ? (units_max > 0 ? units_max : 1) : ctas);
    return launch_k(!a.no_pdl, decode_kernel<kDtype, NP, kSel>, dim3(grid), dim3(kThreads), C::kSmem, st, a);
}

template <int kDtype, int NP>
cudaError_t launch_dyn_np(const ScoreArgs& a, cudaStream_t st) {
    using D = DynCfg<kDtype, NP>;
    cudaError_t e = cudaFuncSetAttribute(decode_dyn_kernel<kDtype, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         D::kSmem);
    if (e != cudaSuccess) return e;
    // no more CTAs than jobs could exist (a CTA whose first job does not exist exits at once)
    const int64_t jobs_max = (int64_t)a.B * (((a.max_seq_len_k + 127) / 128 + D::kJob - 1) / D::kJob);
    const int ctas = Cfg<kDtype, NP>::kCps * sm_count();
    const int grid = (int)(jobs_max < ctas ? (jobs_max > 0 ? jobs_max : 1) : ctas);
    return launch_k(!a.no_pdl, decode_dyn_kernel<kDtype, NP>, dim3(grid), dim3(kThreads), D::kSmem, st, a);
}

template <int kDtype>
cudaError_t launch_dyn_dt(const ScoreArgs& a, cudaStream_t st) {
    if (a.H <= 16) return launch_dyn_np<kDtype, 16>(a, st);
    if (a.H <= 32) return launch_dyn_np<kDtype, 32>(a, st);
    return launch_dyn_np<kDtype, 64>(a, st);
}

template <int kDtype, bool kSel>
cudaError_t launch_dt(const ScoreArgs& a, cudaStream_t st) {
    if (a.H <= 16) return launch_np<kDtype, 16, kSel>(a, st);
    if (a.H <= 32) return launch_np<kDtype, 32, kSel>(a, st);
    return launch_np<kDtype, 64, kSel>(a, st);
}

}  // namespace

cudaError_t launch_scorer_decode(const ScoreArgs& a, cudaStream_t st) {
    if (a.T == 0 || a.max_seq_len_k == 0 || a.B == 0) return cudaSuccess;
    // the dynamic schedule: a workspace for its counters and at most kDynB sequences
    if (a.counters && a.B <= kDynB)
        return a.dtype == IDX_MXFP4 ? launch_dyn_dt<IDX_MXFP4>(a, st) : launch_dyn_dt<IDX_FP8>(a, st);
    return a.dtype == IDX_MXFP4 ? launch_dt<IDX_MXFP4, false>(a, st) : launch_dt<IDX_FP8, false>(a, st);
}

// Select mode: launched whenever there are rows (rows with no key still get their padding).
cudaError_t launch_scorer_decode_select(const ScoreArgs& a, cudaStream_t st) {
    if (a.T == 0 || a.B == 0) return cudaSuccess;
    return a.dtype == IDX_MXFP4 ? launch_dt<IDX_MXFP4, true>(a, st) : launch_dt<IDX_FP8, true>(a, st);
}

}  // namespace idx
