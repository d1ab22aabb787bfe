// scorer_prefill.cu -- paged MQA-logits scorer for prefill / chunked prefill (many queries
// per sequence, optionally causal) on the 5th-generation tensor cores.
//
//   logits[t, s] = sum_h w[t,h] * ReLU(q[t,h] . k[s])               (MXFP4)
//   logits[t, s] = kscale[s] * sum_h w[t,h] * ReLU(q[t,h] . k[s])   (FP8)
//
// vllm PR 57517 "Performance and accuracy" (prefill scorer, 8192 queries / H32 / 8K) and
// vllm PR 60834 "Purpose" (the paged cache is scored in place, so prefill no longer gathers
// K first).
//
// Operands: A = a 128-key tile of the sequence's paged cache (as in the decode scorer), B =
// a block of QB queries: each query's Hq = roundup(H, 8) quantised head rows are placed HP
// rows apart (HP = power of two >= Hq), N = QB * HP <= 224 rows. One block-scaled MMA pair
// (kind::mxf4, K = 64 each) or four kind::f8f6f4 MMAs (K = 32) give D[key][query, head] in
// tensor memory; the ReLU-weighted head sum is the epilogue: each thread owns one key.
//
// Per (query, key) pair the epilogue issues about 1.5H instructions (H maxes for the ReLU,
// H/2 packed fp32x2 fused multiply-adds) while the tensor core does 2*H*128 flops, so the
// epilogue, not the tensor core, is the bound (the maxes run on the half-rate ALU pipe). Two
// accumulator buffers (2 x 224 columns), each fed by its own MMA-issuing warp (even / odd
// tiles) and drained by two epilogue warpgroups (half of the queries each), keep the MMAs of
// the next tiles and the head sums of the current ones in flight together; four epilogue
// warps per scheduler hide the tensor-memory load latency, and each warp loads 64 columns per
// tcgen05.wait::ld (a wait covers every load in flight, so a warp cannot overlap its own loads
// with its sums; fewer, larger loads pay the latency less often). The epilogue is written to
// issue little beyond its sums: compile-time trip counts, head offsets and query indices
// (one instance per warpgroup half), 32-bit key arithmetic, no per-query test on the tiles
// whose keys every query of the half sees (all but the diagonal and the ragged ends),
// per-block row pointers, and the block's head weights in shared memory read 16 bytes at a
// time.
//
// Work: query blocks, heaviest first (causal), in snake order over persistent CTAs (CTA c
// takes ranks c, 2G-1-c, 2G+c, ...). Roles: warp 0 = producer (Q image of the block by bulk
// copy; the block's scale atoms and weights by the warp's lanes; K tiles by bulk copy, one
// tile per lane); warps 1 and 2 = MMA issuers for even and odd tiles (warp 1 also owns the
// tensor memory); warps 3-18 = four epilogue warpgroups: two per accumulator, each taking
// half of the block's queries (one warp per 32-lane TMEM quadrant each).
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"
#include "tc.cuh"

namespace idx {

namespace {

constexpr int kEpiGroups = 4;
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 32 * (3 + kEpiWarps);
constexpr int kNmax = 224;          // B rows per block, at most

template <int kDtype>
struct PCfg {
    static constexpr int kTileCode = kDtype == IDX_MXFP4 ? 128 * 64 : 128 * 128;
    static constexpr int kTileSf = kDtype == IDX_MXFP4 ? 512 : 0;
    static constexpr int kStage = kTileCode + kTileSf;
    static constexpr int kStages = kDtype == IDX_MXFP4 ? 12 : 5;
    static constexpr int kQRow = kDtype == IDX_MXFP4 ? 64 : 128;
    static constexpr int kQImg = 256 * kQRow;                    // Q slot (rows up to 256)
    static constexpr int kQSf = kDtype == IDX_MXFP4 ? 1024 : 0;  // two scale atoms
    static constexpr int kW = kNmax * 4;                         // head weights of a block
    static constexpr uint32_t kSbo = kDtype == IDX_MXFP4 ? 512 : 1024;
    static constexpr uint32_t kCols = 512;  // 2 accumulators of N, A and B scale factors
    static constexpr int oStages = 0;
    static constexpr int oQ = kStages * kStage;   // two Q slots (double-buffered blocks)
    static constexpr int oQSf = oQ + 2 * kQImg;
    static constexpr int oW = oQSf + 2 * kQSf;
    static constexpr int oBars = oW + 2 * kW;
    static constexpr int kBars = 2 * kStages + 10;
    static constexpr int oMisc = oBars + 8 * kBars;
    // select mode: one top-k work area per epilogue warpgroup (histogram, candidate list,
    // per-warp counters)
    static constexpr int kCandS = 512;
    static constexpr int kSelArea = 2048 * 4 + 2 * kCandS * 4 + 3 * 4 * 4 + 8 * 4;
    static constexpr int oSel = oMisc + 64;
    static constexpr int kSmem = oSel;
    static constexpr int kSmemSel = oSel + kEpiGroups * kSelArea;
};

struct Unit {
    int b;
    int64_t q0, nq_blk;   // first query (sequence-local) and queries in this block
    int64_t t0;           // global row of the sequence's first query
    int64_t nq, len;      // queries and keys of the sequence
    int64_t tiles;        // 128-key tiles to score
};

// Unit of virtual rank v: blocks are ranked heaviest first: v -> (jr = v / B, b = v % B),
// block j = MB - 1 - jr of sequence b (empty if the sequence has fewer blocks). A sequence
// whose lengths break their bounds (key count negative or above max_seq_len_k, query count
// negative or above max_q_len) has no units; `report` (one thread of the CTA) sets
// IDX_STATUS_BAD_LEN for it.
__device__ __forceinline__ bool unit_of(const ScoreArgs& a, int QB, int64_t MB, int64_t v, Unit& u,
                                        bool report_bad) {
    const int64_t jr = v / a.B;
    u.b = (int)(v - jr * a.B);
    const int64_t j = MB - 1 - jr;
    u.t0 = a.cu_seqlens_q[u.b];
    u.nq = a.cu_seqlens_q[u.b + 1] - u.t0;
    u.q0 = j * QB;
    const int64_t len = a.seq_lens_k[u.b];
    if (u.nq < 0 || u.nq > a.max_q_len || len < 0 || len > a.max_seq_len_k) {
        if (report_bad) report(a.dev_status, IDX_STATUS_BAD_LEN);
        return false;
    }
    if (u.nq == 0 || u.q0 >= u.nq) return false;
    u.nq_blk = min((int64_t)QB, u.nq - u.q0);
    u.len = len;
    const int64_t vis_last = visible_keys(u.len, u.nq, u.q0 + u.nq_blk - 1, a.causal);
    u.tiles = (vis_last + 127) / 128;
    return u.tiles > 0;
}

// Iterates this CTA's units: ranks c, 2G-1-c, 2G+c, 4G-1-c, ... (snake order).
struct Sched {
    int64_t k, V, MB;
    int c, G, QB;
    __device__ __forceinline__ void init(const ScoreArgs& a, int qb) {
        QB = qb;
        MB = ((int64_t)a.max_q_len + QB - 1) / QB;
        V = MB * a.B;
        k = 0;
        c = blockIdx.x;
        G = gridDim.x;
    }
    __device__ __forceinline__ bool next(const ScoreArgs& a, Unit& u) {
        for (;;) {
            if (k * G >= V) return false;
            const int64_t v = k * G + ((k & 1) ? (G - 1 - c) : c);
            ++k;
            if (v < V && unit_of(a, QB, MB, v, u, threadIdx.x == 0)) return true;
        }
    }
};

// tcgen05.ld of NC consecutive accumulator columns of this warp's lane quadrant
template <int NC>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float* v) {
    if constexpr (NC == 8) {
        uint32_t r[4];
        tc::tmem_ld4(taddr, r);
        uint32_t r2[4];
        tc::tmem_ld4(taddr + 4, r2);
#pragma unroll
        for (int i = 0; i < 4; ++i) { v[i] = __uint_as_float(r[i]); v[4 + i] = __uint_as_float(r2[i]); }
    } else if constexpr (NC == 16) {
        uint32_t r[16];
        tc::tmem_ld16(taddr, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
    } else {
#pragma unroll
        for (int c = 0; c < NC; c += 32) {
            uint32_t r[32];
            tc::tmem_ld32(taddr + c, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[c + i] = __uint_as_float(r[i]);
        }
    }
}

// The work area of selecting warpgroup g (select mode).
template <typename C>
__device__ __forceinline__ SelectSmem sel_smem(uint8_t* smem, int g) {
    uint8_t* p = smem + C::oSel + g * C::kSelArea;
    SelectSmem m;
    m.hist = reinterpret_cast<uint32_t*>(p);
    m.cand = reinterpret_cast<int32_t*>(p + 2048 * 4);
    m.ckey = reinterpret_cast<uint32_t*>(p + 2048 * 4 + C::kCandS * 4);
    m.warp_sums = reinterpret_cast<uint32_t*>(p + 2048 * 4 + 2 * C::kCandS * 4);
    m.warp_gt = m.warp_sums + 4;
    m.warp_eq = m.warp_gt + 4;
    m.scal = m.warp_eq + 4;
    m.keys = nullptr;
    m.key_cap = 0;
    return m;
}

// bar.red.or over the epilogue warpgroups: every participant gets the OR of the predicates
__device__ __forceinline__ bool epi_barrier_or(bool pred) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r)
                 : "r"((uint32_t)pred), "r"(kEpiThreads)
                 : "memory");
    return r != 0;
}

// kAllHeads: H == HP, every accumulator column is a head (no per-head guard in the epilogue).
// kSel: select mode (idx_mqa_topk_paged): a block's logits go to this CTA's rows of the
// scratch, and at the end of the block the four epilogue warpgroups select the top-k of its
// rows (one row per warpgroup at a time) and write the indices.
template <int kDtype, int HP, bool kAllHeads, bool kSel>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(ScoreArgs a) {
    using C = PCfg<kDtype>;
    constexpr int QB = kNmax / HP;  // queries per block
    constexpr int N = QB * HP;      // B rows (224 or 192)
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::oBars);
    uint64_t* k_full = bars;
    uint64_t* k_empty = k_full + C::kStages;
    uint64_t* q_full = k_empty + C::kStages;   // 2
    uint64_t* q_empty = q_full + 2;            // 2
    uint64_t* acc_full = q_empty + 2;          // 2
    uint64_t* acc_empty = acc_full + 2;        // 2
    uint64_t* drain = acc_empty + 2;           // 2: an MMA issuer's last commit when it gives up
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::oMisc);
    volatile uint32_t* abort_flag = misc + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, P = a.page_size;
    const int lp = P == 128 ? 7 : 6;  // log2 of the page size (64 or 128)
    const int Hq = (H + 7) & ~7;

    if (tid == 0) {
        misc[1] = 0;
        for (int i = 0; i < C::kStages; ++i) {
            tc::mbar_init(&k_full[i], 1);
            tc::mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&q_full[i], 1);
            // released by both MMA issuers' commits and by every epilogue thread (they read
            // the slot's head weights after the MMAs are done)
            tc::mbar_init(&q_empty[i], 2 + kEpiThreads);
            tc::mbar_init(&acc_full[i], 1);
            tc::mbar_init(&acc_empty[i], kEpiThreads / 2);  // two warpgroups per buffer
            tc::mbar_init(&drain[i], 1);
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
    // previous kernels
    pdl_wait();
    pdl_launch_dependents();
    const uint32_t tbase = misc[0];
    // tensor memory: accumulators [2][N]; A scale slot per buffer [2][4]; B scale atoms per
    // buffer (MMA issuer) and Q slot [2][2][8]
    const uint32_t t_sfa = tbase + 2 * N;
    const uint32_t t_sfb = t_sfa + 8;

    Sched sch;
    sch.init(a, QB);
    Unit u;

    if (warp == 0) {
        // -------------------------------------------------------------- producer warp
        int64_t n_units = 0, kt = 0;  // units and tiles issued so far
        int64_t q_armed = -1;         // last unit whose Q fill was armed
        while (sch.next(a, u)) {
            if (__any_sync(kFull, *abort_flag != 0)) break;  // warp-uniform exit
            // Q block into slot n % 2, once the MMAs and epilogues of block n-2 are done with it
            const int slot = (int)(n_units & 1);
            if (!__all_sync(kFull, tc::mbar_wait(&q_empty[slot], (uint32_t)(((n_units >> 1) & 1) ^ 1)))) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            // head weights of the block (zero past its queries) and, for MXFP4, B's scale
            // atoms: row n = q*HP + h -> byte (n%32)*16 + ((n/32)%4)*4 of atom n/128, from
            // query q's own atom (head h at (h%32)*16 + (h/32)*4)
            float* wsm = reinterpret_cast<float*>(smem + C::oW + slot * C::kW);
            for (int i = lane; i < QB * H; i += 32) {
                const int q = i / H;
                wsm[i] = q < u.nq_blk ? __ldg(a.w + (u.t0 + u.q0) * H + i) : 0.0f;
            }
            if (kDtype == IDX_MXFP4) {
                uint8_t* sf = smem + C::oQSf + slot * C::kQSf;
                for (int n = lane; n < 256; n += 32) {
                    const int q = n / HP, h = n % HP;
                    uint32_t v = 0x7f7f7f7fu;
                    if (q < u.nq_blk && h < Hq)
                        v = __ldg(reinterpret_cast<const uint32_t*>(a.q_scales + (u.t0 + u.q0 + q) * 512 +
                                                                    (h & 31) * 16 + (h >> 5) * 4));
                    *reinterpret_cast<uint32_t*>(sf + (n >> 7) * 512 + (n & 31) * 16 + ((n >> 5) & 3) * 4) = v;
                }
                tc::fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t qrow_bytes = (uint32_t)(Hq * C::kQRow);  // one query's image
                const uint32_t qbytes = (uint32_t)u.nq_blk * qrow_bytes;
                tc::mbar_arrive_expect_tx(&q_full[slot], qbytes);  // after the lanes' stores (warp-synchronised)
                q_armed = n_units;
                const uint8_t* qsrc = a.q_codes + (u.t0 + u.q0) * Hq * C::kQRow;
                uint8_t* qdst = smem + C::oQ + slot * C::kQImg;
                if (Hq == HP) {
                    tc::bulk_g2s(qdst, qsrc, qbytes, &q_full[slot]);
                } else {  // padded spacing: one copy per query (padding rows are never summed)
                    for (int q = 0; q < u.nq_blk; ++q)
                        tc::bulk_g2s(qdst + q * HP * C::kQRow, qsrc + q * qrow_bytes, qrow_bytes, &q_full[slot]);
                }
            }
            // K tiles in batches: lane L owns tile j0+L (page lookup, stage wait, copies), so
            // the warp issues a batch at once; a batch never reuses a stage, and each lane's
            // wait depends only on tiles of earlier batches
            constexpr int kBatch = C::kStages < 16 ? C::kStages : 16;
            const int32_t* pt = a.page_table + (int64_t)u.b * a.pt_stride;
            for (int64_t j0 = 0; j0 < u.tiles && !__any_sync(kFull, *abort_flag != 0); j0 += kBatch) {
                const int nb = (int)min((int64_t)kBatch, u.tiles - j0);
                if (lane < nb) {
                    const int64_t j = j0 + lane, k = kt + lane;
                    const int64_t key0 = j * 128;
                    const int halves = P == 128 ? 1 : (key0 + 64 < u.len ? 2 : 1);
                    int32_t pg[2] = {__ldg(pt + (key0 >> lp)), halves == 2 ? __ldg(pt + ((key0 + 64) >> lp)) : -1};
                    const int s = (int)(k % C::kStages);
                    if (!tc::mbar_wait(&k_empty[s], (uint32_t)(((k / C::kStages) & 1) ^ 1))) {
                        *abort_flag = 1;
                    } else {
                        uint32_t bytes = 0;
                        for (int hh = 0; hh < halves; ++hh) {
                            if (pg[hh] >= 0 && pg[hh] < a.num_pages) {
                                bytes += (uint32_t)(P * (C::kTileCode / 128 + C::kTileSf / 128));
                            } else {
                                report(a.dev_status, IDX_STATUS_BAD_PAGE);
                                pg[hh] = -1;
                            }
                        }
                        tc::mbar_arrive_expect_tx(&k_full[s], bytes);
                        uint8_t* dK = smem + C::oStages + s * C::kStage;
                        uint8_t* dS = dK + C::kTileCode;
                        for (int hh = 0; hh < halves; ++hh) {
                            if (pg[hh] < 0) continue;
                            const uint8_t* src = a.pool + (int64_t)pg[hh] * a.page_stride;
                            if (P == 128) {
                                // codes and scale atom are contiguous in the page and in the stage
                                tc::bulk_g2s(dK, src, C::kStage, &k_full[s]);
                            } else if (kDtype == IDX_MXFP4) {
                                for (int q = 0; q < 4; ++q)
                                    tc::bulk_g2s(dK + q * 2048 + hh * 1024, src + q * 1024, 1024, &k_full[s]);
                                tc::bulk_g2s(dS + hh * 256, src + 4096, 256, &k_full[s]);
                            } else {
                                tc::bulk_g2s(dK + hh * 8192, src, 8192, &k_full[s]);
                            }
                        }
                    }
                }
                kt += nb;
                __syncwarp();
            }
            ++n_units;
            __syncwarp();
        }
        if (*abort_flag) {
            if (lane == 0) report(a.dev_status, IDX_STATUS_TIMEOUT);
            // do not leave while copies are in flight: wait (bounded) for the last fill armed
            // in each stage and Q slot
            const uint64_t deadline = tc::global_ns() + tc::kWaitLimitNs;
            if (lane < C::kStages && kt - 1 >= lane) {
                const int64_t k = (kt - 1) - ((kt - 1 - lane) % C::kStages);
                tc::mbar_wait_until(&k_full[lane], (uint32_t)((k / C::kStages) & 1), deadline);
            }
            q_armed = __shfl_sync(kFull, q_armed, 0);
            if (lane < 2 && q_armed >= lane) {
                const int64_t n = q_armed - ((q_armed - lane) & 1);
                tc::mbar_wait_until(&q_full[lane], (uint32_t)((n >> 1) & 1), deadline);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // -------------------------------------------------------------- MMA issuers
        // warp 1 issues the even tiles into accumulator 0, warp 2 the odd ones into
        // accumulator 1; each keeps its own A and B scale-factor slots
        const int buf = warp - 1;
        if (lane == 0) {
            // descriptors of stage 0 / Q slot 0; stages, slots and K steps add (bytes >> 4)
            // to the start-address field (shared-memory addresses stay below 256 KB)
            const uint64_t dA0 = tc::smem_desc(tc::smem_u32(smem + C::oStages), 128, C::kSbo);
            const uint64_t dB0 = tc::smem_desc(tc::smem_u32(smem + C::oQ), 128, C::kSbo);
            const uint64_t dSA0 = tc::smem_desc(tc::smem_u32(smem + C::oStages + C::kTileCode), 128, 128);
            const uint64_t dSB0 = tc::smem_desc(tc::smem_u32(smem + C::oQSf), 128, 128);
            const uint32_t id0 = kDtype == IDX_MXFP4 ? tc::idesc_mxf4(128, N, 0, 0) : tc::idesc_f8(128, N);
            const uint32_t id1 = kDtype == IDX_MXFP4 ? tc::idesc_mxf4(128, N, 2, 2) : id0;
            const uint32_t d = tbase + buf * N;
            const uint32_t sfa = t_sfa + 4 * buf;
            int64_t n_units = 0, kt = 0;
            uint32_t aph = 1;
            while (sch.next(a, u)) {
                if (*abort_flag) break;
                const int slot = (int)(n_units & 1);
                if (!tc::mbar_wait(&q_full[slot], (uint32_t)((n_units >> 1) & 1))) {
                    *abort_flag = 1;
                    break;
                }
                tc::tc_fence_after();
                const uint64_t db = dB0 + (uint64_t)((slot * C::kQImg) >> 4);
                const uint32_t sfb = t_sfb + 16 * buf + 8 * slot;
                if (kDtype == IDX_MXFP4) {
                    // B's two scale atoms: rows 0-127 and 128-255
                    const uint64_t dsb = dSB0 + (uint64_t)((slot * C::kQSf) >> 4);
                    tc::cp_32x128b_warpx4(sfb, dsb);
                    tc::cp_32x128b_warpx4(sfb + 4, dsb + 32);
                }
                bool ok = true;
                for (int64_t j = 0; j < u.tiles; ++j, ++kt) {
                    if ((kt & 1) != buf) continue;
                    const int s = (int)(kt % C::kStages);
                    if (!tc::mbar_wait(&k_full[s], (uint32_t)((kt / C::kStages) & 1))) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    // the tile's A scale atom goes to tensor memory before the accumulator
                    // wait: it overwrites only this issuer's scale slot, which the previous
                    // (earlier-issued, in-order) MMA of this issuer has read
                    if (kDtype == IDX_MXFP4) tc::cp_32x128b_warpx4(sfa, dSA0 + (uint64_t)((s * C::kStage) >> 4));
                    if (!tc::mbar_wait(&acc_empty[buf], aph)) {
                        ok = false;
                        break;
                    }
                    aph ^= 1;
                    tc::tc_fence_after();
                    const uint64_t da = dA0 + (uint64_t)((s * C::kStage) >> 4);
                    if (kDtype == IDX_MXFP4) {
                        tc::mma_mxf4(d, da, db, id0, sfa, sfb, 0);
                        tc::mma_mxf4(d, da + 16, db + 16, id1, sfa, sfb, 1);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k) tc::mma_f8(d, da + 16 * k, db + 16 * k, id0, k);
                    }
                    tc::mma_commit(&k_empty[s]);
                    tc::mma_commit(&acc_full[buf]);
                }
                if (!ok) {
                    *abort_flag = 1;
                    break;
                }
                tc::mma_commit(&q_empty[slot]);  // arrives when this warp's MMAs of the block end
                ++n_units;
            }
            if (*abort_flag) {
                // do not free tensor memory under MMAs still running: one more commit tracks
                // every tcgen05 operation of this thread; wait (bounded) for it
                report(a.dev_status, IDX_STATUS_TIMEOUT);
                tc::mma_commit(&drain[buf]);
                tc::mbar_wait(&drain[buf], 0);
            }
        }
    } else {
        // -------------------------------------------------------------- epilogue warpgroups
        // warpgroup g drains accumulator g % 2, i.e. the tiles with (tile count % 2) == g % 2,
        // for half g / 2 of the block's queries; every thread owns one key
        const int g = (warp - 3) >> 2;
        const int gb = g & 1, gh = g >> 1;
        const int quad = warp & 3;        // TMEM lane quadrant this warp may access
        const int m = quad * 32 + lane;
        const bool split = P == 64 && kDtype == IDX_MXFP4;
        const int khalf = split ? ((m >> 4) & 1) : (m >> 6);
        const int koff = split ? (64 * khalf + (m & 15) + 16 * (m >> 5)) : m;
        const bool vec_w = (H & 3) == 0;
        int64_t kt = 0, n_units = 0;
        uint32_t aph = 0;
        constexpr int QC = HP <= 32 ? 32 / HP : 1;  // queries per 32-column load (HP = 64: 2 loads)
        constexpr int CW = QC * HP;                 // columns per chunk
        constexpr int QH0 = (QB + 1) / 2;           // queries of the first half
        constexpr int NCH = (QH0 + QC - 1) / QC;    // chunks per tile, at most
        const int qlo = gh ? QH0 : 0, qhi = gh ? QB : QH0;
        const int nch = (qhi - qlo + QC - 1) / QC;
        if constexpr (kSel) pad_orphan_rows(a, (int)threadIdx.x - 96, kEpiThreads);
        const uint32_t lane_addr = tbase + ((uint32_t)(quad * 32) << 16) + gb * N + qlo * HP;
        while (sch.next(a, u)) {
            const int slot = (int)(n_units & 1);
            // the block's weights: wait for the slot's fill (the same phase the MMA issuers used)
            bool have_q = true;
            if (!__all_sync(kFull, tc::mbar_wait(&q_full[slot], (uint32_t)((n_units >> 1) & 1)))) {
                *abort_flag = 1;
                report(a.dev_status, IDX_STATUS_TIMEOUT);
                if constexpr (!kSel) break;
                have_q = false;  // select mode: no tiles, but the block-end barriers still run
            }
            const float* wsm = reinterpret_cast<const float*>(smem + C::oW + slot * C::kW);
            const int32_t* pt = a.page_table + (int64_t)u.b * a.pt_stride;
            const int nqb = (int)u.nq_blk;
            // query q of the block sees keys < vis0 + q (causal; unclamped, so it also holds when
            // the block has more queries than keys) or keys < len; key < len is checked apart
            // (32-bit key arithmetic: lengths are int32 and the host checks QB * ld < 2^31)
            const int32_t vis0 = (int32_t)(a.causal ? u.len - u.nq + u.q0 + 1 : u.len);
            const int qstep = a.causal ? 1 : 0;
            // the block's first logits row (select mode: this CTA's scratch rows)
            float* lrow = kSel ? a.logits + (int64_t)blockIdx.x * QB * a.ld : a.logits + (u.t0 + u.q0) * a.ld;
            const int32_t ld = (int32_t)a.ld;
            const int tiles = (int)u.tiles;
            // this warpgroup's tiles of the block: every other one, from the parity of the
            // tiles scored before the block
            for (int j = (int)((gb - kt) & 1); j < (have_q ? tiles : 0); j += 2) {
                // page lookups are issued before the accumulator wait (their latency hides
                // behind it) and used after it
                const int32_t key = j * 128 + koff;
                const bool in_seq = key < u.len;
                const int32_t pg = in_seq ? __ldg(pt + (key >> lp)) : -1;
                const bool got = __all_sync(kFull, tc::mbar_wait(&acc_full[gb], aph));
                if (!got) {
                    *abort_flag = 1;
                    report(a.dev_status, IDX_STATUS_TIMEOUT);
                    break;
                }
                aph ^= 1;
                tc::tc_fence_after();
                const bool key_ok = in_seq && pg >= 0 && pg < a.num_pages;
                float kscale = 1.0f;
                if (kDtype == IDX_FP8 && key_ok)
                    kscale = __ldg(reinterpret_cast<const float*>(a.pool + (int64_t)pg * a.page_stride + 128 * P + 4 * ((key & (P - 1)))));
                // this key is visible to queries q >= qmin (all of them off the diagonal)
                const int32_t d = key - vis0 + 1;  // causal: query q sees the key iff q >= d
                const int qmin = !key_ok ? QB : (qstep == 0 ? (key < vis0 ? 0 : QB) : (d <= 0 ? 0 : (d >= QB ? QB : (int)d)));
                if constexpr (kAllHeads) {
                    // drain in 64-column chunks, one tcgen05.wait::ld each (a wait covers every
                    // load in flight, so fewer, larger loads pay the tensor-memory latency less
                    // often); the accumulator is released as soon as this half's last chunk
                    // is in registers. Sub-chunk s of chunk c holds head columns h0 .. h0+15
                    // of query qlo + (64c + 16s) / HP (two queries when HP = 8). The half and,
                    // on tiles whose key every query of the half sees, the queries summed are
                    // compile-time, so such a tile's drain tests nothing per query.
                    auto drain = [&](auto all_c, auto half_c) {
                        constexpr bool kAll = decltype(all_c)::value;
                        constexpr int GH = decltype(half_c)::value;
                        constexpr int CH = 64;
                        constexpr int QPS = HP >= 16 ? 1 : 16 / HP;  // queries per 16 columns
                        constexpr int kColsQ = HP >= 16 ? 16 : HP;   // a query's columns per 16
                        constexpr int QLO = GH ? QH0 : 0, QHI = GH ? QB : QH0;
                        constexpr int NCHK = ((QHI - QLO) * HP + CH - 1) / CH;  // chunks of the half
                        const int qend = kAll ? QHI : min(QHI, nqb);
                        const int nchk = kAll ? NCHK : (qend > QLO ? ((qend - QLO) * HP + CH - 1) / CH : 0);
                        if (nchk == 0) {
                            tc::tc_fence_before();
                            tc::mbar_arrive(&acc_empty[gb]);
                        }
                        float2 acc[QPS][2];
#pragma unroll
                        for (int c = 0; c < NCHK; ++c) {
                            if (!kAll && c >= nchk) break;
                            uint32_t r[CH];
                            tc::tmem_ld32(lane_addr + c * CH, *reinterpret_cast<uint32_t(*)[32]>(r));
                            tc::tmem_ld32(lane_addr + c * CH + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
                            tc::tmem_ld_wait();
                            if (c + 1 == nchk) {  // the last chunk is in registers
                                tc::tc_fence_before();
                                tc::mbar_arrive(&acc_empty[gb]);
                            }
#pragma unroll
                            for (int sc = 0; sc < CH / 16; ++sc) {
#pragma unroll
                                for (int qq = 0; qq < QPS; ++qq) {
                                    const int col = c * CH + 16 * sc;  // compile-time
                                    const int q = QLO + col / HP + qq;  // compile-time
                                    const int h0 = col % HP;
                                    if (q >= QHI) continue;
                                    if (h0 == 0) acc[qq][0] = acc[qq][1] = make_float2(0.0f, 0.0f);
                                    if (!kAll && !(q >= qmin && q < qend)) continue;
                                    const float4* w4p = reinterpret_cast<const float4*>(wsm + q * HP + h0);
#pragma unroll
                                    for (int i = 0; i < kColsQ / 4; ++i) {
                                        const float4 w4 = w4p[i];
                                        const uint32_t* x = r + 16 * sc + qq * kColsQ + 4 * i;
                                        // chain 0: ReLU by max (ALU pipe); chain 1: by x + |x| = 2 ReLU(x)
                                        // (FMA pipe), so chain 1 holds twice its sum, halved below:
                                        // both scalings by 2 are exact, the sum is the same
                                        const float x2 = __uint_as_float(x[2]), x3 = __uint_as_float(x[3]);
                                        const float2 r0 = make_float2(fmaxf(__uint_as_float(x[0]), 0.0f),
                                                                      fmaxf(__uint_as_float(x[1]), 0.0f));
                                        const float2 r1 = make_float2(x2 + fabsf(x2), x3 + fabsf(x3));
                                        acc[qq][0] = __ffma2_rn(make_float2(w4.x, w4.y), r0, acc[qq][0]);
                                        acc[qq][1] = __ffma2_rn(make_float2(w4.z, w4.w), r1, acc[qq][1]);
                                    }
                                    if (h0 + kColsQ == HP) {
                                        const float2 s2 = __ffma2_rn(acc[qq][1], make_float2(0.5f, 0.5f), acc[qq][0]);
                                        lrow[q * ld + key] = (s2.x + s2.y) * kscale;
                                    }
                                }
                            }
                        }
                    };
                    using T0 = std::integral_constant<bool, false>;
                    using T1 = std::integral_constant<bool, true>;
                    using G0 = std::integral_constant<int, 0>;
                    using G1 = std::integral_constant<int, 1>;
                    const bool all = __all_sync(kFull, qmin == 0) && nqb >= (gh ? QB : QH0);
                    if (gh) {
                        if (all) drain(T1{}, G1{});
                        else drain(T0{}, G1{});
                    } else {
                        if (all) drain(T1{}, G0{});
                        else drain(T0{}, G0{});
                    }
                } else {
                    // software-pipelined drain: chunk c+1 is loaded while chunk c is summed; the
                    // accumulator is released as soon as this half's last chunk is in registers
                    float v[2][CW];
                    ld_cols<CW>(lane_addr, v[0]);
                    tc::tmem_ld_wait();
                    if (nch == 1) {
                        tc::tc_fence_before();
                        tc::mbar_arrive(&acc_empty[gb]);
                    }
    #pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        if (c >= nch) break;
                        float* va = v[c & 1];
                        if (c + 1 < nch) ld_cols<CW>(lane_addr + (c + 1) * CW, v[(c + 1) & 1]);
    #pragma unroll
                        for (int qq = 0; qq < QC; ++qq) {
                            const int q = qlo + c * QC + qq;
                            if (q < qhi && q < nqb && q >= qmin) {
                                const float* wq = wsm + q * H;
                                float logit;
                                if constexpr (kAllHeads) {
                                    // eight independent chains as four packed pairs (fma.rn.f32x2:
                                    // each lane an ordinary fp32 fused multiply-add)
                                    float2 acc[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
                                    const float4* w4p = reinterpret_cast<const float4*>(wq);
    #pragma unroll
                                    for (int i = 0; i < HP / 4; ++i) {
                                        const float4 w4 = w4p[i];
                                        const float* x = va + qq * HP + 4 * i;
                                        acc[(2 * i) & 3] = __ffma2_rn(make_float2(w4.x, w4.y),
                                                                      make_float2(fmaxf(x[0], 0.0f), fmaxf(x[1], 0.0f)),
                                                                      acc[(2 * i) & 3]);
                                        acc[(2 * i + 1) & 3] = __ffma2_rn(make_float2(w4.z, w4.w),
                                                                          make_float2(fmaxf(x[2], 0.0f), fmaxf(x[3], 0.0f)),
                                                                          acc[(2 * i + 1) & 3]);
                                    }
                                    const float2 s01 = __fadd2_rn(acc[0], acc[1]), s23 = __fadd2_rn(acc[2], acc[3]);
                                    const float2 s = __fadd2_rn(s01, s23);
                                    logit = s.x + s.y;
                                } else {
                                    float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                                    if (vec_w) {
    #pragma unroll
                                        for (int h = 0; h < HP; h += 4) {
                                            if (h < H) {
                                                const float4 w4 = *reinterpret_cast<const float4*>(wq + h);
                                                part[0] = fmaf(w4.x, fmaxf(va[qq * HP + h], 0.0f), part[0]);
                                                part[1] = fmaf(w4.y, fmaxf(va[qq * HP + h + 1], 0.0f), part[1]);
                                                part[2] = fmaf(w4.z, fmaxf(va[qq * HP + h + 2], 0.0f), part[2]);
                                                part[3] = fmaf(w4.w, fmaxf(va[qq * HP + h + 3], 0.0f), part[3]);
                                            }
                                        }
                                    } else {
    #pragma unroll
                                        for (int h = 0; h < HP; ++h)
                                            if (h < H) part[h & 3] = fmaf(wq[h], fmaxf(va[qq * HP + h], 0.0f), part[h & 3]);
                                    }
                                    logit = (part[0] + part[1]) + (part[2] + part[3]);
                                }
                                lrow[q * ld + key] = logit * kscale;
                            }
                        }
                        if (c + 1 < nch) {
                            tc::tmem_ld_wait();
                            if (c + 2 == nch) {  // the last chunk is in registers
                                tc::tc_fence_before();
                                tc::mbar_arrive(&acc_empty[gb]);
                            }
                        }
                    }
                }
            }
            kt += tiles;
            // done with the slot's weights
            tc::mbar_arrive(&q_empty[slot]);
            ++n_units;
            if constexpr (kSel) {
                // every epilogue warpgroup has written (or given up on) its part of the block's
                // logits: select each row's top-k, warpgroup g taking rows g, g + 4, ...; every
                // warpgroup reaches both barriers once per block, also on the give-up path
                __threadfence();
                NamedBarrier{1, kEpiThreads}();
                const int sg = g;
                const int stid = (int)threadIdx.x - (3 + 4 * sg) * 32;
                const SelectSmem sm = sel_smem<C>(smem, sg);
                for (int q = sg; q < nqb; q += kEpiGroups) {
                    const int vis = (int)visible_keys(u.len, u.nq, u.q0 + q, a.causal);
                    select_topk_row<128, C::kCandS>(lrow + (int64_t)q * a.ld, vis, a.topk_k,
                                                    a.out_idx + (u.t0 + u.q0 + q) * a.topk_k, sm, stid,
                                                    NamedBarrier{(uint32_t)(2 + sg), 128});
                }
                if (epi_barrier_or(*abort_flag != 0)) break;  // uniform over the warpgroups
            } else {
                if (__any_sync(kFull, *abort_flag != 0)) break;  // warp-uniform exit
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

template <int kDtype, int HP, bool kAllHeads, bool kSel>
cudaError_t launch_hp(const ScoreArgs& a, cudaStream_t st) {
    using C = PCfg<kDtype>;
    constexpr int smem = kSel ? C::kSmemSel : C::kSmem;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<kDtype, HP, kAllHeads, kSel>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    constexpr int QB = kNmax / HP;
    const int64_t units = (int64_t)a.B * ((a.max_q_len + QB - 1) / QB);
    // select mode: every CTA runs (the orphan-row pass is strided over the whole grid)
    const int grid = kSel ? sm_count() : (int)(units < sm_count() ? (units > 0 ? units : 1) : sm_count());
    return launch_pdl(prefill_kernel<kDtype, HP, kAllHeads, kSel>, dim3(grid), dim3(kThreads), smem, st, a);
}

template <int kDtype, bool kSel>
cudaError_t launch(const ScoreArgs& a, cudaStream_t st) {
    switch (a.H) {
        case 8: return launch_hp<kDtype, 8, true, kSel>(a, st);
        case 16: return launch_hp<kDtype, 16, true, kSel>(a, st);
        case 32: return launch_hp<kDtype, 32, true, kSel>(a, st);
        case 64: return launch_hp<kDtype, 64, true, kSel>(a, st);
        default: break;
    }
    if (a.H < 8) return launch_hp<kDtype, 8, false, kSel>(a, st);
    if (a.H < 16) return launch_hp<kDtype, 16, false, kSel>(a, st);
    if (a.H < 32) return launch_hp<kDtype, 32, false, kSel>(a, st);
    return launch_hp<kDtype, 64, false, kSel>(a, st);
}

}  // namespace

cudaError_t launch_scorer_prefill(const ScoreArgs& a, cudaStream_t st) {
    if (a.T == 0 || a.max_seq_len_k == 0 || a.B == 0) return cudaSuccess;
    return a.dtype == IDX_MXFP4 ? launch<IDX_MXFP4, false>(a, st) : launch<IDX_FP8, false>(a, st);
}

cudaError_t launch_scorer_prefill_select(const ScoreArgs& a, cudaStream_t st) {
    if (a.T == 0 || a.B == 0) return cudaSuccess;
    return a.dtype == IDX_MXFP4 ? launch<IDX_MXFP4, true>(a, st) : launch<IDX_FP8, true>(a, st);
}

// Queries per prefill block for H heads (HP = H rounded up to a power of two >= 8).
int prefill_queries_per_block(int32_t H) {
    const int hp = H <= 8 ? 8 : H <= 16 ? 16 : H <= 32 ? 32 : 64;
    return kNmax / hp;
}

int device_sm_count() { return sm_count(); }

}  // namespace idx
