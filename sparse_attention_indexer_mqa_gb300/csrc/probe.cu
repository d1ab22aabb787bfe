// probe.cu -- dense tensor-core rate of the two MMA kinds the scorers use, for the roofline
// of the prefill scorer: one CTA per SM issues back-to-back block-scaled MXFP4
// (tcgen05.mma kind::mxf4, M = 128, N = 256, K = 64) or FP8 e4m3 (kind::f8f6f4, K = 32) MMAs
// from shared-memory operands, accumulating into one tensor-memory accumulator (as a GEMM's
// K loop does). The operands are zero (the rate does not depend on the values); the results
// are discarded. Each CTA reserves enough shared memory that no two share an SM.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace idx {

namespace {

constexpr int kPerIter = 8;  // MMAs per loop iteration (the issuing thread's loop overhead
                             // is then small next to the tensor work)

template <int kDtype>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int iters, int32_t* status) {
    // A: 128 rows, B: 256 rows, K-major canonical layout; MXFP4 rows are 32 B per K = 64,
    // FP8 rows 32 B per K = 32; plus two 512 B scale atoms for B and one for A
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int kA = 128 * 32, kB = 256 * 32;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kA + kB + 3 * 512);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
    for (int i = threadIdx.x; i < (kA + kB + 3 * 512) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(smem)[i] = kDtype == IDX_MXFP4 && i >= (kA + kB) / 4 ? 0x7f7f7f7fu : 0u;
    if (threadIdx.x == 0) {
        tc::mbar_init(bar, 1);
        tc::fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        tc::tmem_alloc(slot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_proxy_async();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = *slot;
    if (threadIdx.x == 0) {
        const uint32_t sbo = 256;  // 8 rows x 32 B between 8-row groups (K extent 32 B)
        const uint64_t da = tc::smem_desc(tc::smem_u32(smem), 128, sbo);
        const uint64_t db = tc::smem_desc(tc::smem_u32(smem + kA), 128, sbo);
        const uint64_t ds = tc::smem_desc(tc::smem_u32(smem + kA + kB), 128, 128);
        const uint32_t sfa = tbase + 256, sfb = sfa + 4;  // scale columns after the accumulator
        if (kDtype == IDX_MXFP4) {
            tc::cp_32x128b_warpx4(sfa, ds);
            tc::cp_32x128b_warpx4(sfb, ds + 32);
            tc::cp_32x128b_warpx4(sfb + 4, ds + 64);
        }
        const uint32_t id = kDtype == IDX_MXFP4 ? tc::idesc_mxf4(128, 256, 0, 0) : tc::idesc_f8(128, 256);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int m = 0; m < kPerIter; ++m) {
                if (kDtype == IDX_MXFP4) tc::mma_mxf4(tbase, da, db, id, sfa, sfb, it | m);
                else tc::mma_f8(tbase, da, db, id, it | m);
            }
        }
        tc::mma_commit(bar);
        if (!tc::mbar_wait(bar, 0)) report(status, IDX_STATUS_TIMEOUT);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, 512);
    }
}

// One thread waits for phase 0 of an mbarrier whose arrival count is never reached (nothing
// arrives on it), gives up at the deadline and reports the timeout.
__global__ void wait_timeout_kernel(int64_t limit_ns, int32_t* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    const uint64_t deadline = tc::global_ns() + (uint64_t)limit_ns;
    if (!tc::mbar_wait_until(&bar, 0, deadline)) report(status, IDX_STATUS_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout(int32_t limit_us, int32_t* status, cudaStream_t st) {
    wait_timeout_kernel<<<1, 32, 0, st>>>((int64_t)limit_us * 1000, status);
    return cudaGetLastError();
}

cudaError_t launch_mma_rate(int32_t dtype, int32_t iters, int32_t* status, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const size_t smem = 120 * 1024;  // one CTA per SM (it uses the first 14 KB)
    if (dtype == IDX_MXFP4) {
        e = cudaFuncSetAttribute(mma_rate_kernel<IDX_MXFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        mma_rate_kernel<IDX_MXFP4><<<sms, 128, smem, st>>>(iters, status);
    } else {
        e = cudaFuncSetAttribute(mma_rate_kernel<IDX_FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        mma_rate_kernel<IDX_FP8><<<sms, 128, smem, st>>>(iters, status);
    }
    return cudaGetLastError();
}

int mma_rate_flops_per_iter(int32_t dtype) {
    // 2 * M * N * K per MMA
    return (dtype == IDX_MXFP4 ? 2 * 128 * 256 * 64 : 2 * 128 * 256 * 32) * kPerIter;
}

}  // namespace idx
