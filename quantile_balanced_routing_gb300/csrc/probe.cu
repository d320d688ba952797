// Tensor-core rate probe: back-to-back tcgen05.mma on fixed shared-memory
// tiles, one CTA per SM, no TMA and no epilogue.  It measures the rate of one
// MMA kind on this GPU at its current clocks, so that a contraction can be
// compared with the peak of the MMA kind it actually issues.
//
// Kinds: QBMOE_PROBE_BF16 = kind::f16 with bf16 A and B (M = 128, N = 256,
// K = 16 per instruction); QBMOE_PROBE_MXF4F8 = kind::mxf8f6f4 block-scaled
// with E2M1 A and E4M3 B, one E8M0 scale per 32 K (M = 128, N = 256, K = 32),
// the instruction the MXFP4 expert GEMMs issue.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kProbeThreads = 128;
constexpr int kRowBytes = 128;                   // one 128-byte swizzled row per operand row
constexpr int kABytes = 128 * kRowBytes;         // 16 KB
constexpr int kBBytes = 256 * kRowBytes;         // 32 KB
constexpr int kProbeSmem = 1024 + kABytes + kBBytes + 64;
// requested per CTA so that at most one CTA runs on an SM (it holds all 512
// TMEM columns)
constexpr int kProbeSmemLaunch = 120 * 1024;
constexpr uint32_t kAccCol = 0, kSfbCol = 256, kSfaCol = 264;

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352dU;
    x ^= x >> 15;
    x *= 0x846ca68bU;
    x ^= x >> 16;
    return x;
}

template <int KIND>
__global__ void __launch_bounds__(kProbeThreads, 1) k_mma_probe(int iters, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* A = smem;
    uint8_t* B = smem + kABytes;
    uint64_t* done = reinterpret_cast<uint64_t*>(B + kBBytes);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // operands: finite, nonzero bit patterns (bf16 with a small exponent
    // range; E2M1 any code; E4M3 without the NaN codes)
    for (int i = threadIdx.x; i < (kABytes + kBBytes) / 4; i += blockDim.x) {
        uint32_t h = mix32(i * 2654435761u + blockIdx.x);
        if (KIND == QBMOE_PROBE_BF16) h = (h & 0x807F807Fu) | 0x3C003C00u;
        else if (i >= kABytes / 4) h &= 0x77777777u;
        reinterpret_cast<uint32_t*>(smem)[i] = h;
    }
    if (threadIdx.x == 0) {
        tc::mbar_init(done, 1);
        tc::fence_mbar_init();
    }
    tc::fence_proxy_async_smem();
    if (warp == 0) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = *tslot;
    if (KIND == QBMOE_PROBE_MXF4F8) {
        // all scales 2^0: each warp writes its TMEM lane quarter
        const uint32_t lanes = static_cast<uint32_t>(32 * warp) << 16;
        constexpr uint32_t one = 0x7F7F7F7Fu;
        tc::tmem_st4(tbase + lanes + kSfbCol, one, one, one, one);
        tc::tmem_st4(tbase + lanes + kSfbCol + 4, one, one, one, one);
        tc::tmem_st4(tbase + lanes + kSfaCol, one, one, one, one);
        tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (threadIdx.x == 0) {
        const uint64_t ad = tc::desc_sw128(tc::smem_u32(A));
        const uint64_t bd = tc::desc_sw128(tc::smem_u32(B));
        uint32_t id[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            id[kk] = KIND == QBMOE_PROBE_BF16 ? tc::idesc_bf16_m128(256) : tc::idesc_mx_e2m1_e4m3_m128(256, kk, 0);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                if (KIND == QBMOE_PROBE_BF16)
                    tc::tc_mma_bf16(tbase + kAccCol, ad + 2 * kk, bd + 2 * kk, id[kk], (it | kk) != 0);
                else
                    tc::tc_mma_mxf8f6f4(tbase + kAccCol, ad + 2 * kk, bd + 2 * kk, id[kk], tbase + kSfaCol,
                                        tbase + kSfbCol, (it | kk) != 0);
            }
        }
        tc::tc_commit(done);
        if (!tc::mbar_wait(done, 0, 1LL << 17)) qb::set_status(status, QBMOE_ETIMEOUT);
    }
    __syncwarp();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tbase, 512);
}

}  // namespace

extern "C" int qbmoe_mma_probe(int kind, int iters, float* ms_out, double* flops_out) {
    if (!ms_out || !flops_out || iters < 1 || iters > (1 << 22)) return QBMOE_EINVAL;
    if (kind != QBMOE_PROBE_BF16 && kind != QBMOE_PROBE_MXF4F8) return QBMOE_EINVAL;
    int rc = qbh::device_init();
    if (rc) return rc;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return QBMOE_ECUDA;
    auto kern = kind == QBMOE_PROBE_BF16 ? k_mma_probe<QBMOE_PROBE_BF16> : k_mma_probe<QBMOE_PROBE_MXF4F8>;
    int* status = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    static_assert(kProbeSmem <= kProbeSmemLaunch, "probe shared memory");
    bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmemLaunch) ==
                  cudaSuccess &&
              cudaMalloc(&status, sizeof(int)) == cudaSuccess && cudaMemset(status, 0, sizeof(int)) == cudaSuccess &&
              cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess;
    float ms = 0.0f;
    int st = 0;
    if (ok) {
        kern<<<sms, kProbeThreads, kProbeSmemLaunch>>>(1, status);   // warm-up
        cudaEventRecord(e0);
        kern<<<sms, kProbeThreads, kProbeSmemLaunch>>>(iters, status);
        cudaEventRecord(e1);
        ok = cudaGetLastError() == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
             cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess &&
             cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess;
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (status) cudaFree(status);
    if (!ok) {
        cudaGetLastError();
        return QBMOE_ECUDA;
    }
    if (st) return st;
    const double k_per = kind == QBMOE_PROBE_BF16 ? 16.0 : 32.0;
    *ms_out = ms;
    *flops_out = (double)sms * iters * 4.0 * 2.0 * 128.0 * 256.0 * k_per;
    return QBMOE_OK;
}
