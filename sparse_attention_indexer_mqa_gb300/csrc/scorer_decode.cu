// scorer_decode.cu -- paged MQA-logits scorer for decode (one query per sequence) on the
// 5th-generation tensor cores.
//
//   logits[t, s] = sum_h w[t,h] * ReLU(q[t,h] . k[s])          (MXFP4)
//   logits[t, s] = kscale[s] * sum_h w[t,h] * ReLU(q[t,h] . k[s])   (FP8, w carries q's scale)
//
// vllm PR 57517 "Purpose" / "Performance and accuracy" (decode B64/H32/D128/8K scorer) and
// vllm PR 60834 "Purpose" (the MXFP4 cache is scored in place through the page table,
// without gathering K first).
//
// Operand roles: the key tile is the A operand (M = 128 keys = one 128-token page or two
// 64-token pages), the query's heads are B (N = H rounded up to 16), K = 128. So each
// tensor-memory lane holds one key and one thread reduces its key's H head scores with
// no shuffles. The cache pages are laid out in the tensor core's canonical K-major order
// (see idx.h), so each page is bulk-copied (cp.async.bulk) into shared memory unchanged;
// its MXFP4 scale bytes are already in the tensor-memory scale-factor order and go to
// tensor memory with one tcgen05.cp. MXFP4 runs kind::mxf4 block-scaled MMAs (two of
// K = 64, scale factors by 32-block); FP8 runs kind::f8f6f4 (four of K = 32) and applies the
// per-token scale in the epilogue.
//
// A CTA owns up to kTiles consecutive 128-key tiles of one sequence. One thread of warp 4
// issues every tile's bulk copies at once (all bytes in flight immediately: the step is
// HBM bound), then the MMAs tile by tile into two tensor-memory accumulators; warps 0-3
// drain the accumulators (tcgen05.ld), form the ReLU-weighted head sums and write logits.
// Several CTAs share an SM, so one CTA's epilogue overlaps other CTAs' copies.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace idx {

namespace {

constexpr int kEpi = 128;           // warps 0-3: epilogue (one TMEM lane quadrant each)
constexpr int kThreads = kEpi + 32;  // warp 4: copies, tensor-memory allocation, MMAs
constexpr int kIssuer = kEpi;        // the thread that issues copies and MMAs

template <int kDtype>
struct DecodeCfg {
    static constexpr int kTiles = kDtype == IDX_MXFP4 ? 4 : 2;                // tiles per CTA
    static constexpr int kTileCode = kDtype == IDX_MXFP4 ? 128 * 64 : 128 * 128;  // bytes
    static constexpr int kTileAux = 512;     // MXFP4 scale atom / FP8 128 fp32 scales
    static constexpr int kQRow = kDtype == IDX_MXFP4 ? 64 : 128;  // code bytes per head
    static constexpr int kKSteps = kDtype == IDX_MXFP4 ? 2 : 4;   // MMAs per tile
    static constexpr int kStepBytes = 256;   // K advance per MMA in the canonical layout
    static constexpr uint32_t kSbo = kDtype == IDX_MXFP4 ? 512 : 1024;
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

template <int kDtype, int NP>
__global__ void __launch_bounds__(kThreads) decode_kernel(ScoreArgs a) {
    using Cfg = DecodeCfg<kDtype>;
    constexpr int TPC = Cfg::kTiles;
    constexpr uint32_t kCols = (2 * NP + 4 * TPC + 4) <= 64 ? 64 : ((2 * NP + 4 * TPC + 4) <= 128 ? 128 : 256);

    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sK = smem;                                         // TPC x tile codes
    uint8_t* sAux = sK + TPC * Cfg::kTileCode;                  // TPC x 512
    uint8_t* sQ = sAux + TPC * Cfg::kTileAux;                   // NP x kQRow (canonical)
    uint8_t* sSFB = sQ + NP * Cfg::kQRow;                       // 512
    float* sW = reinterpret_cast<float*>(sSFB + 512);           // 64
    uint64_t* bar_load = reinterpret_cast<uint64_t*>(sW + 64);  // TPC
    uint64_t* bar_full = bar_load + TPC;                        // 2
    uint64_t* bar_empty = bar_full + 2;                         // 2
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_empty + 2);
    int32_t* half_ok = reinterpret_cast<int32_t*>(tmem_slot + 1);  // TPC x 2

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y;
    const int64_t t = a.cu_seqlens_q[b];
    if (a.cu_seqlens_q[b + 1] <= t) return;  // sequence without a query
    int64_t seq_len = a.seq_lens_k[b];
    if (seq_len > a.max_seq_len_k || seq_len < 0) {
        if (tid == 0 && blockIdx.x == 0) report(a.dev_status, IDX_STATUS_BAD_LEN);
        seq_len = seq_len < 0 ? 0 : a.max_seq_len_k;
    }
    const int64_t nq = a.cu_seqlens_q[b + 1] - t;
    const int64_t vis = visible_keys(seq_len, nq, nq - 1, a.causal);  // the last query
    const int64_t tile0 = (int64_t)blockIdx.x * TPC;
    const int64_t tiles_total = (vis + 127) / 128;
    if (tile0 >= tiles_total) return;
    const int n_tiles = (int)min((int64_t)TPC, tiles_total - tile0);
    const int H = a.H;
    const int P = a.page_size;

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < TPC; ++i) tc::mbar_init(&bar_load[i], 1);
        tc::mbar_init(&bar_full[0], 1);
        tc::mbar_init(&bar_full[1], 1);
        tc::mbar_init(&bar_empty[0], kEpi);
        tc::mbar_init(&bar_empty[1], kEpi);
        tc::fence_mbar_init();
    }
    __syncthreads();

    // ---- issuer: every page copy of this CTA, issued at once -------------------------------
    if (tid == kIssuer) {
        const int32_t* pt = a.page_table + (int64_t)b * a.pt_stride;
        for (int i = 0; i < n_tiles; ++i) {
            const int64_t key0 = (tile0 + i) * 128;
            const int halves = P == 128 ? 1 : (key0 + 64 < vis ? 2 : 1);
            int32_t pages[2];
            uint32_t bytes = 0;
            for (int h = 0; h < halves; ++h) {
                const int32_t pg = pt[(key0 + 64 * h) / P];
                const bool ok = pg >= 0 && pg < a.num_pages;
                if (!ok) report(a.dev_status, IDX_STATUS_BAD_PAGE);
                pages[h] = ok ? pg : -1;
                half_ok[2 * i + h] = ok;
                if (ok) bytes += (uint32_t)(P * (Cfg::kTileCode / 128 + 4));
            }
            if (halves == 1) half_ok[2 * i + 1] = (P == 128) ? half_ok[2 * i] : 0;
            tc::mbar_arrive_expect_tx(&bar_load[i], bytes);
            uint8_t* dK = sK + i * Cfg::kTileCode;
            uint8_t* dA = sAux + i * Cfg::kTileAux;
            for (int h = 0; h < halves; ++h) {
                if (pages[h] < 0) continue;
                const uint8_t* src = a.pool + (int64_t)pages[h] * a.page_stride;
                if (P == 128) {
                    tc::bulk_g2s(dK, src, Cfg::kTileCode, &bar_load[i]);
                    tc::bulk_g2s(dA, src + Cfg::kTileCode, 512, &bar_load[i]);
                } else if (kDtype == IDX_MXFP4) {
                    // four 1 KB chunks of 16 keys interleave with the other page's chunks
                    for (int q = 0; q < 4; ++q)
                        tc::bulk_g2s(dK + q * 2048 + h * 1024, src + q * 1024, 1024, &bar_load[i]);
                    tc::bulk_g2s(dA + h * 256, src + 4096, 256, &bar_load[i]);
                } else {
                    tc::bulk_g2s(dK + h * 8192, src, 8192, &bar_load[i]);
                    tc::bulk_g2s(dA + h * 256, src + 8192, 256, &bar_load[i]);
                }
            }
        }
    }

    // ---- all threads: Q (canonical image, zero rows past H), its scale atom, weights ------
    {
        const uint8_t* qg = a.q_codes + t * H * Cfg::kQRow;
        constexpr int kChunks = Cfg::kQRow / 16;
        for (int i = tid; i < NP * kChunks; i += kThreads) {
            const int h = i / kChunks, c = i % kChunks;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < H) v = *reinterpret_cast<const uint4*>(qg + h * Cfg::kQRow + 16 * c);
            *reinterpret_cast<uint4*>(sQ + ((h >> 3) * kChunks + c) * 128 + (h & 7) * 16) = v;
        }
        if (kDtype == IDX_MXFP4) {
            for (int h = tid; h < 128; h += kThreads) {
                uint32_t s = 0x7f7f7f7fu;
                if (h < H) s = *reinterpret_cast<const uint32_t*>(a.q_scales + (t * H + h) * 4);
                *reinterpret_cast<uint32_t*>(sSFB + (h & 31) * 16 + (h >> 5) * 4) = s;
            }
        }
        if (tid < 64) sW[tid] = tid < H ? a.w[t * H + tid] : 0.0f;
    }
    tc::fence_proxy_async();
    __syncwarp();
    if (warp == 4) {
        tc::tmem_alloc(tmem_slot, kCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t t_sfa = tbase + 2 * NP;           // 4 columns per tile
    const uint32_t t_sfb = t_sfa + 4 * TPC;          // 4 columns
    bool ok = true;

    // ---- issuer: MMAs, tile by tile, into accumulator buffer i % 2 --------------------------
    if (tid == kIssuer) {
        if (kDtype == IDX_MXFP4) tc::cp_32x128b_warpx4(t_sfb, tc::smem_desc(tc::smem_u32(sSFB), 128, 128));
        for (int i = 0; i < n_tiles && ok; ++i) {
            const int buf = i & 1;
            if (i >= 2) ok = tc::mbar_wait(&bar_empty[buf], ((i - 2) >> 1) & 1);
            ok = ok && tc::mbar_wait(&bar_load[i], 0);
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t d = tbase + buf * NP;
            const uint32_t a0 = tc::smem_u32(sK + i * Cfg::kTileCode), b0 = tc::smem_u32(sQ);
            if (kDtype == IDX_MXFP4) {
                tc::cp_32x128b_warpx4(t_sfa + 4 * i, tc::smem_desc(tc::smem_u32(sAux + i * 512), 128, 128));
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    tc::mma_mxf4(d, tc::smem_desc(a0 + j * 256, 128, Cfg::kSbo),
                                 tc::smem_desc(b0 + j * 256, 128, Cfg::kSbo),
                                 tc::idesc_mxf4(128, NP, 2 * j, 2 * j), t_sfa + 4 * i, t_sfb, j);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tc::mma_f8(d, tc::smem_desc(a0 + j * 256, 128, Cfg::kSbo),
                               tc::smem_desc(b0 + j * 256, 128, Cfg::kSbo), tc::idesc_f8(128, NP), j);
            }
            tc::mma_commit(&bar_full[buf]);
        }
        if (!ok) report(a.dev_status, IDX_STATUS_TIMEOUT);
    }

    // ---- epilogue: lane m of the tile = one key ---------------------------------------------
    const int m = warp * 32 + lane;
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    // key offset of row m inside the tile; for two 64-key pages, rows with m%32 < 16 come from
    // the first page (its keys s%16 + 16*(m/32)... see the page layout in idx.h)
    const int half = (P == 64 && kDtype == IDX_MXFP4) ? ((m >> 4) & 1) : (m >> 6);
    const int koff = (P == 64 && kDtype == IDX_MXFP4) ? (64 * half + (m & 15) + 16 * (m >> 5)) : m;
    float* out = a.logits + t * a.ld;
    for (int i = 0; i < n_tiles && tid < kEpi; ++i) {
        const int buf = i & 1;
        // warp-uniform, since tcgen05.ld is a warp-collective instruction
        const bool got = __all_sync(0xffffffffu, tc::mbar_wait(&bar_full[buf], (i >> 1) & 1));
        tc::tc_fence_after();
        float v[NP];
        if (got) load_acc<NP>(lane_addr + buf * NP, v);
        tc::tc_fence_before();
        tc::mbar_arrive(&bar_empty[buf]);
        if (!got) {
            report(a.dev_status, IDX_STATUS_TIMEOUT);
            break;
        }
        const int64_t key = (tile0 + i) * 128 + koff;
        const bool row_ok = key < vis && half_ok[2 * i + (P == 128 ? 0 : half)];
        float logit = 0.0f;
#pragma unroll
        for (int h = 0; h < NP; ++h)
            if (h < H) logit = fmaf(sW[h], fmaxf(v[h], 0.0f), logit);
        if (kDtype == IDX_FP8) logit *= reinterpret_cast<const float*>(sAux + i * Cfg::kTileAux)[m];
        if (row_ok) out[key] = logit;
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, kCols);
    }
}

template <int kDtype, int NP>
cudaError_t launch_decode_np(const ScoreArgs& a, cudaStream_t st) {
    using Cfg = DecodeCfg<kDtype>;
    const size_t smem = Cfg::kTiles * (Cfg::kTileCode + Cfg::kTileAux) + NP * Cfg::kQRow + 512 +
                        256 + 8 * (Cfg::kTiles + 4) + 4 + 8 * Cfg::kTiles + 64;
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<kDtype, NP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (a.max_seq_len_k + 127) / 128;
    dim3 grid((unsigned)((tiles + Cfg::kTiles - 1) / Cfg::kTiles), (unsigned)a.B);
    decode_kernel<kDtype, NP><<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int kDtype>
cudaError_t launch_decode_dt(const ScoreArgs& a, cudaStream_t st) {
    if (a.H <= 16) return launch_decode_np<kDtype, 16>(a, st);
    if (a.H <= 32) return launch_decode_np<kDtype, 32>(a, st);
    return launch_decode_np<kDtype, 64>(a, st);
}

}  // namespace

cudaError_t launch_scorer_decode(const ScoreArgs& a, cudaStream_t st) {
    if (a.T == 0 || a.max_seq_len_k == 0 || a.B == 0) return cudaSuccess;
    return a.dtype == IDX_MXFP4 ? launch_decode_dt<IDX_MXFP4>(a, st) : launch_decode_dt<IDX_FP8>(a, st);
}

}  // namespace idx
