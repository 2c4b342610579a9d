// Measurement diagnostic: the issue rate of the block-scaled MMA form of the
// pair GEMM kernel (nvfp4_mma_issue_rate in nvfp4.h).  One cluster of two
// CTAs; the even CTA issues the kernel's fused K-stage block (12 scale
// copies and 4 MMAs of M=256, N=256, K=64) back to back on operands already
// in shared memory, then one commit; the cycles between the first issue and
// that commit's arrival give the sustained rate.  The operand bytes are
// arbitrary (the rate does not depend on them); the accumulator is never
// read.  Every wait is bounded.
#include "common.cuh"
#include "internal.h"
#include "nvfp4.h"

namespace nvfp4 {

namespace {

constexpr int kProbeStages = 4096;
constexpr int kProbeSmem = 65536 + 24576 + 1024;   // codes, scales, alignment
__device__ long long g_probe_cycles;
__device__ int g_probe_status;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1) mma_rate_kernel()
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t done, sink;
    __shared__ uint32_t tbase;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    for (int i = threadIdx.x; i < (65536 + 24576) / 16; i += 128)
        reinterpret_cast<uint4*>(sm)[i] = make_uint4(0x22222222u, 0x22222222u, 0x38383838u, 0x38383838u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&done), 1);
        mbar_init(smem_u32(&sink), 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc2(smem_u32(&tbase), 512);
        tmem_relinquish2();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the fills above, for the tensor core
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tm = tbase;
    if (warp == 0) {
        const uint64_t dsw = make_smem_desc(base, 16, 1024, 2);
        const uint64_t dsf = make_smem_desc(base + 65536, 128, 128, 0);
        const uint32_t a_lo = (uint32_t)dsw, sw_hi = (uint32_t)(dsw >> 32);
        const uint32_t f_lo = (uint32_t)dsf, sf_hi = (uint32_t)(dsf >> 32);
        // kind::mxf4nvf4: E2M1 A and B, UE4M3 scales, K-major, N = 256, M = 256
        const uint32_t idesc = (1u << 7) | (1u << 10) | ((256u >> 3) << 17) | ((256u >> 4) << 24);
        __syncwarp();
        const long long t0 = clock64();
        if (rank == 0) {
            for (int i = 0; i < kProbeStages; i++) {
                // five rotating scale slots and two operand stages, as in the kernel
                const uint32_t sfc = tm + 256 + (uint32_t)(i % 5) * 48;
                const uint32_t a = a_lo + (uint32_t)(i & 1) * (32768u >> 4);
                stage_issue_2sm(tm, sfc, f_lo, sf_hi, a, a + (16384u >> 4), sw_hi, idesc, i != 0, smem_u32(&sink),
                                0x1);
            }
            mma_commit2_mc_warp(smem_u32(&done), 0x3);
        }
        bool ok = true;
        if (lane == 0) {
            const long long w0 = clock64();
            while (!mbar_try_wait(smem_u32(&done), 0))
                if (clock64() - w0 > (long long)kWaitLimitCycles) {
                    ok = false;
                    break;
                }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        const long long t1 = clock64();
        if (rank == 0 && lane == 0) {
            g_probe_cycles = ok ? t1 - t0 : -1;
            if (!ok) g_probe_status = NVFP4_ERR_TIMEOUT;
        }
        if (!ok && lane == 0) mbar_wait_teardown(smem_u32(&done), 0);   // the MMAs in flight (bounded)
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 0) tmem_dealloc2(tm, 512);
}

}  // namespace

}  // namespace nvfp4

using namespace nvfp4;

extern "C" int nvfp4_mma_issue_rate(double* mac_per_clk)
{
    if (!mac_per_clk) return NVFP4_ERR_INVALID_ARG;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (!(major == 10 && minor == 3)) return NVFP4_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    const long long zero = 0;
    const int izero = 0;
    if (cudaMemcpyToSymbol(g_probe_cycles, &zero, sizeof zero) != cudaSuccess ||
        cudaMemcpyToSymbol(g_probe_status, &izero, sizeof izero) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    mma_rate_kernel<<<2, 128, kProbeSmem>>>();
    if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return NVFP4_ERR_CUDA;
    long long cycles = 0;
    int st = 0;
    if (cudaMemcpyFromSymbol(&cycles, g_probe_cycles, sizeof cycles) != cudaSuccess ||
        cudaMemcpyFromSymbol(&st, g_probe_status, sizeof st) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (st != 0 || cycles <= 0) return NVFP4_ERR_TIMEOUT;
    // per SM: 128 of the 256 rows x 256 columns x 256 (four K-steps of 64) per stage
    *mac_per_clk = (double)kProbeStages * 128.0 * 256.0 * 256.0 / (double)cycles;
    return NVFP4_OK;
}
