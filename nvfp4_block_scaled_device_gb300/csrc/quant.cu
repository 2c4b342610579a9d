// Row kernels of the NVFP4 path: the device global scale (amax reduction,
// optionally of the RMSNorm of the rows) and the bf16 -> NVFP4 quantizer
// (optionally fused with that RMSNorm).  Both are single HBM passes with
// 16-byte vector loads; reductions use warp shuffles.
//
// Sources: "PERFORMANCE -- verified hot-path audit and prioritized fixes"
// P0 (scale = max(amax, 1e-8) / (6 * 448), computed on the device, handed on
// as a (1,) device tensor) and P8 item 2 (RMSNorm fused into the next
// linear's input quantization); "CUDA: NVFP4 prefill on Blackwell leaves
// ~1.45x performance on the table", item 2 (batched-row rms_norm).
#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

namespace {

__device__ __forceinline__ void unpack8(const uint4& p, float* f)
{
    f[0] = bf16_lo(p.x); f[1] = bf16_hi(p.x);
    f[2] = bf16_lo(p.y); f[3] = bf16_hi(p.y);
    f[4] = bf16_lo(p.z); f[5] = bf16_hi(p.z);
    f[6] = bf16_lo(p.w); f[7] = bf16_hi(p.w);
}

// 1 / sqrt(mean(x^2) + eps) of one row, computed by the whole block
// (kRowThreads threads) in a fixed order; every thread gets the result.
// The square of a bf16 value is exact in binary32; each thread sums its
// squares as an unevaluated pair hi + lo (TwoSum keeps every addition's
// rounding error), the pairs are combined in binary64, and the mean is
// rounded once to binary32 -- the binary64 mean-square of the definition,
// to well below half a binary32 ulp.
__device__ float row_inv_rms(const uint4* xr, int64_t nvec, int64_t cols, float eps, double* red)
{
    float hi = 0.0f, lo = 0.0f;
    for (int64_t v = threadIdx.x; v < nvec; v += kRowThreads) {
        float f[8];
        unpack8(xr[v], f);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float p = __fmul_rn(f[i], f[i]);
            const float s = __fadd_rn(hi, p);
            const float bp = __fsub_rn(s, hi);
            const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
            hi = s;
            lo = __fadd_rn(lo, e);
        }
    }
    double t = (double)hi + (double)lo;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    const int warp = threadIdx.x >> 5;
    __syncthreads();  // red[] may still be read from the previous row
    if ((threadIdx.x & 31) == 0) red[warp] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
        double sum = 0.0;
        for (int w = 0; w < kRowThreads / 32; w++) sum += red[w];
        const float ms = (float)(sum / (double)cols);
        red[kRowThreads / 32] = (double)__fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    }
    __syncthreads();
    return (float)red[kRowThreads / 32];
}

// y = bf16( (x * r) * w ), one rounding per step.
__device__ __forceinline__ void norm8(float* f, float r, const uint4& wp)
{
    float w[8];
    unpack8(wp, w);
#pragma unroll
    for (int i = 0; i < 8; i++) f[i] = bf16_round(__fmul_rn(__fmul_rn(f[i], r), w[i]));
}

template <bool NORM>
__global__ void __launch_bounds__(kRowThreads) amax_scale_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                                                 int64_t cols, int64_t ldx,
                                                                 const __nv_bfloat16* __restrict__ norm_w,
                                                                 float eps, float* __restrict__ g_out,
                                                                 uint32_t* __restrict__ ws)
{
    __shared__ double red[kRowThreads / 32 + 1];
    const int64_t nvec = cols / 8;
    float amax = 0.0f;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const uint4* xr = reinterpret_cast<const uint4*>(x + row * ldx);
        float r = 1.0f;
        if (NORM) r = row_inv_rms(xr, nvec, cols, eps, red);
        for (int64_t v = threadIdx.x; v < nvec; v += kRowThreads) {
            float f[8];
            unpack8(xr[v], f);
            if (NORM) norm8(f, r, reinterpret_cast<const uint4*>(norm_w)[v]);
#pragma unroll
            for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(f[i]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float wmax[kRowThreads / 32];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kRowThreads / 32; w++) amax = fmaxf(amax, wmax[w]);
        // non-negative binary32 values order like their bit patterns
        atomicMax(&ws[0], __float_as_uint(amax));
        __threadfence();
        const uint32_t ticket = atomicAdd(&ws[1], 1u);
        if (ticket == gridDim.x - 1) {
            __threadfence();
            const float a = __uint_as_float(atomicExch(&ws[0], 0u));
            g_out[0] = __fdiv_rn(fmaxf(a, 1e-8f), 2688.0f);
            atomicExch(&ws[1], 0u);
        }
    }
}

template <bool NORM>
__global__ void __launch_bounds__(kRowThreads) quantize_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                                               int64_t cols, int64_t ldx,
                                                               const __nv_bfloat16* __restrict__ norm_w, float eps,
                                                               const float* __restrict__ g_ptr,
                                                               uint8_t* __restrict__ codes, int64_t ld_codes,
                                                               uint8_t* __restrict__ sf,
                                                               __nv_bfloat16* __restrict__ y_out)
{
    __shared__ double red[kRowThreads / 32 + 1];
    const float g = *g_ptr;
    const int64_t nvec = cols / 8;          // a multiple of 8: cols % 64 == 0
    const int64_t kb_pad = cols / 16;       // already a multiple of 4
    const int64_t pad_rows = (rows + 127) / 128 * 128;
    for (int64_t row = blockIdx.x; row < pad_rows; row += gridDim.x) {
        if (row >= rows) {
            // padding rows of the scale layout are zero
            for (int64_t c4 = threadIdx.x; c4 < kb_pad / 4; c4 += kRowThreads)
                *reinterpret_cast<uint32_t*>(sf + sf_offset(row, c4 * 4, kb_pad)) = 0u;
            continue;
        }
        const uint4* xr = reinterpret_cast<const uint4*>(x + row * ldx);
        float r = 1.0f;
        if (NORM) r = row_inv_rms(xr, nvec, cols, eps, red);
        for (int64_t v0 = 0; v0 < nvec; v0 += kRowThreads) {
            const int64_t v = v0 + threadIdx.x;
            const bool valid = v < nvec;   // uniform over each group of 8 lanes
            float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (valid) {
                unpack8(xr[v], f);
                if (NORM) {
                    norm8(f, r, reinterpret_cast<const uint4*>(norm_w)[v]);
                    if (y_out) {
                        uint4 o;
                        o.x = pack_bf16x2(f[0], f[1]);
                        o.y = pack_bf16x2(f[2], f[3]);
                        o.z = pack_bf16x2(f[4], f[5]);
                        o.w = pack_bf16x2(f[6], f[7]);
                        reinterpret_cast<uint4*>(y_out + row * cols)[v] = o;
                    }
                }
            }
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; i++) a = fmaxf(a, fabsf(f[i]));
            const float a16 = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            uint32_t sc;
            const uint32_t cw = quant_half_block(f, g, a16, &sc);
            const uint32_t s1 = __shfl_down_sync(0xffffffffu, sc, 2);
            const uint32_t s2 = __shfl_down_sync(0xffffffffu, sc, 4);
            const uint32_t s3 = __shfl_down_sync(0xffffffffu, sc, 6);
            if (valid) {
                *reinterpret_cast<uint32_t*>(codes + row * ld_codes + v * 4) = cw;
                if ((v & 7) == 0)
                    *reinterpret_cast<uint32_t*>(sf + sf_offset(row, v / 2, kb_pad)) =
                        sc | (s1 << 8) | (s2 << 16) | (s3 << 24);
            }
        }
    }
}

__global__ void finalize_scale_kernel(uint32_t* ws, float* g_out)
{
    const float a = __uint_as_float(atomicExch(&ws[0], 0u));
    g_out[0] = __fdiv_rn(fmaxf(a, 1e-8f), 2688.0f);
}

}  // namespace

cudaError_t launch_amax_scale(const __nv_bfloat16* x, int64_t rows, int64_t cols, int64_t ldx,
                              const __nv_bfloat16* norm_w, float eps, float* g_out, uint32_t* ws, int num_sms,
                              cudaStream_t stream)
{
    const int64_t cap = (int64_t)num_sms * 8;
    const unsigned grid = (unsigned)(rows < cap ? rows : cap);
    if (norm_w)
        amax_scale_kernel<true><<<grid, kRowThreads, 0, stream>>>(x, rows, cols, ldx, norm_w, eps, g_out, ws);
    else
        amax_scale_kernel<false><<<grid, kRowThreads, 0, stream>>>(x, rows, cols, ldx, norm_w, eps, g_out, ws);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const __nv_bfloat16* x, int64_t rows, int64_t cols, int64_t ldx,
                            const __nv_bfloat16* norm_w, float eps, const float* g, uint8_t* codes,
                            int64_t ld_codes, uint8_t* sf, __nv_bfloat16* y_out, cudaStream_t stream)
{
    const int64_t pad_rows = (rows + 127) / 128 * 128;
    const unsigned grid = (unsigned)(pad_rows < 2147483647 ? pad_rows : 2147483647);
    if (norm_w)
        quantize_kernel<true><<<grid, kRowThreads, 0, stream>>>(x, rows, cols, ldx, norm_w, eps, g, codes, ld_codes,
                                                                sf, y_out);
    else
        quantize_kernel<false><<<grid, kRowThreads, 0, stream>>>(x, rows, cols, ldx, norm_w, eps, g, codes, ld_codes,
                                                                 sf, y_out);
    return cudaGetLastError();
}

cudaError_t launch_finalize_scale(uint32_t* ws, float* g_out, cudaStream_t stream)
{
    finalize_scale_kernel<<<1, 1, 0, stream>>>(ws, g_out);
    return cudaGetLastError();
}

}  // namespace nvfp4
