// Row kernels of the NVFP4 path: the device global scale (amax reduction,
// optionally of the RMSNorm of the rows) and the bf16 -> NVFP4 quantizer
// (optionally fused with that RMSNorm).  One warp per row (8 rows per
// block, no block-wide barriers), 16-byte vector loads with 4 in flight per
// lane, shuffle reductions; both kernels share one row routine so the
// RMSNorm they compute is bit-identical.
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

constexpr int kRowsPerBlock = kRowThreads / 32;   // one warp per row
constexpr int kUnroll = 4;                          // 16-byte loads in flight per lane

__device__ __forceinline__ void unpack8(const uint4& p, float* f)
{
    f[0] = bf16_lo(p.x); f[1] = bf16_hi(p.x);
    f[2] = bf16_lo(p.y); f[3] = bf16_hi(p.y);
    f[4] = bf16_lo(p.z); f[5] = bf16_hi(p.z);
    f[6] = bf16_lo(p.w); f[7] = bf16_hi(p.w);
}

// Unevaluated sum hi + lo of binary32 values (error-free additions).
struct FF {
    float hi, lo;
};

__device__ __forceinline__ FF ff_add_f(FF a, float p)
{
    const float s = __fadd_rn(a.hi, p);
    const float bp = __fsub_rn(s, a.hi);
    const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
    return {s, __fadd_rn(a.lo, e)};
}

__device__ __forceinline__ FF ff_add(FF a, FF b)
{
    FF s = ff_add_f(a, b.hi);
    s.lo = __fadd_rn(s.lo, b.lo);
    // renormalise so |lo| stays below half an ulp of hi
    const float h = __fadd_rn(s.hi, s.lo);
    return {h, __fsub_rn(s.lo, __fsub_rn(h, s.hi))};
}

__device__ __forceinline__ FF ff_sumsq8(FF acc, const uint4& p)
{
    float f[8];
    unpack8(p, f);
#pragma unroll
    for (int i = 0; i < 8; i++) acc = ff_add_f(acc, __fmul_rn(f[i], f[i]));   // bf16^2 is exact
    return acc;
}

// y = bf16( (x * r) * w ), one rounding per step.
__device__ __forceinline__ void norm8(float* f, float r, const uint4& wp)
{
    float w[8];
    unpack8(wp, w);
#pragma unroll
    for (int i = 0; i < 8; i++) f[i] = bf16_round(__fmul_rn(__fmul_rn(f[i], r), w[i]));
}

// 1 / sqrt(mean(x^2) + eps) of one row, computed by one warp in a fixed
// order.  The squares of bf16 values are exact in binary32; each lane sums
// its squares as a float-float pair, the pairs are reduced by shuffles, and
// lane 0 forms the mean in binary64 and rounds it once to binary32 -- the
// binary64 mean-square of the definition, to far below half a binary32 ulp.
// Every lane gets lane 0's result.
__device__ __forceinline__ float warp_inv_rms(const uint4* __restrict__ xr, int64_t nvec, int64_t cols, float eps)
{
    const int lane = threadIdx.x & 31;
    FF part{0.0f, 0.0f};
    for (int64_t v0 = 0; v0 < nvec; v0 += 32 * kUnroll) {
        uint4 b[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; k++) {
            const int64_t v = v0 + 32 * k + lane;
            b[k] = v < nvec ? xr[v] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; k++) part = ff_sumsq8(part, b[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        FF other{__shfl_xor_sync(0xffffffffu, part.hi, o), __shfl_xor_sync(0xffffffffu, part.lo, o)};
        part = ff_add(part, other);
    }
    float r = 0.0f;
    if (lane == 0) {
        const double sum = (double)part.hi + (double)part.lo;
        const float ms = (float)(sum / (double)cols);
        r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    }
    return __shfl_sync(0xffffffffu, r, 0);
}

// One row, one warp.  QUANT: quantize and store the row; otherwise
// accumulate the amax of the (normalised) row into *amax.  The amax and the
// quantize kernels both go through here, so their RMSNorm is bit-identical.
template <bool NORM, bool QUANT>
__device__ __forceinline__ void row_warp(const uint4* __restrict__ xr, int64_t row, int64_t nvec, int64_t cols,
                                         const uint4* __restrict__ w, float eps, float g,
                                         uint8_t* __restrict__ codes, int64_t ld_codes, uint8_t* __restrict__ sf,
                                         int64_t kb_pad, __nv_bfloat16* __restrict__ y_out, float* amax)
{
    const int lane = threadIdx.x & 31;
    const float r = NORM ? warp_inv_rms(xr, nvec, cols, eps) : 1.0f;
    for (int64_t v0 = 0; v0 < nvec; v0 += 32 * kUnroll) {
        uint4 b[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; k++) {
            const int64_t v = v0 + 32 * k + lane;
            b[k] = v < nvec ? xr[v] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; k++) {
            const int64_t v = v0 + 32 * k + lane;
            const bool valid = v < nvec;            // uniform over each group of 8 lanes
            float f[8];
            unpack8(b[k], f);
            if (NORM && valid) norm8(f, r, w[v]);
            if (QUANT) {
                if (NORM && y_out && valid) {
                    uint4 o;
                    o.x = pack_bf16x2(f[0], f[1]);
                    o.y = pack_bf16x2(f[2], f[3]);
                    o.z = pack_bf16x2(f[4], f[5]);
                    o.w = pack_bf16x2(f[6], f[7]);
                    reinterpret_cast<uint4*>(y_out + row * cols)[v] = o;
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
            } else if (valid) {
#pragma unroll
                for (int i = 0; i < 8; i++) *amax = fmaxf(*amax, fabsf(f[i]));
            }
        }
    }
}

template <bool NORM>
__global__ void __launch_bounds__(kRowThreads) amax_scale_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                                                 int64_t cols, int64_t ldx,
                                                                 const __nv_bfloat16* __restrict__ norm_w,
                                                                 float eps, float* __restrict__ g_out,
                                                                 uint32_t* __restrict__ ws)
{
    const int64_t nvec = cols / 8;
    float amax = 0.0f;
    for (int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); row < rows;
         row += (int64_t)gridDim.x * kRowsPerBlock)
        row_warp<NORM, false>(reinterpret_cast<const uint4*>(x + row * ldx), row, nvec, cols,
                              reinterpret_cast<const uint4*>(norm_w), eps, 0.0f, nullptr, 0, nullptr, 0, nullptr,
                              &amax);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float wmax[kRowsPerBlock];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kRowsPerBlock; w++) amax = fmaxf(amax, wmax[w]);
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
    const float g = *g_ptr;
    const int64_t nvec = cols / 8;          // a multiple of 8: cols % 64 == 0
    const int64_t kb_pad = cols / 16;       // already a multiple of 4
    const int64_t pad_rows = (rows + 127) / 128 * 128;
    const int lane = threadIdx.x & 31;
    for (int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); row < pad_rows;
         row += (int64_t)gridDim.x * kRowsPerBlock) {
        if (row >= rows) {
            // padding rows of the scale layout are zero
            for (int64_t c4 = lane; c4 < kb_pad / 4; c4 += 32)
                *reinterpret_cast<uint32_t*>(sf + sf_offset(row, c4 * 4, kb_pad)) = 0u;
            continue;
        }
        row_warp<NORM, true>(reinterpret_cast<const uint4*>(x + row * ldx), row, nvec, cols,
                             reinterpret_cast<const uint4*>(norm_w), eps, g, codes, ld_codes, sf, kb_pad, y_out,
                             nullptr);
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
    const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    const int64_t cap = (int64_t)num_sms * 8;
    const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
    if (norm_w)
        amax_scale_kernel<true><<<grid, kRowThreads, 0, stream>>>(x, rows, cols, ldx, norm_w, eps, g_out, ws);
    else
        amax_scale_kernel<false><<<grid, kRowThreads, 0, stream>>>(x, rows, cols, ldx, norm_w, eps, g_out, ws);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const __nv_bfloat16* x, int64_t rows, int64_t cols, int64_t ldx,
                            const __nv_bfloat16* norm_w, float eps, const float* g, uint8_t* codes,
                            int64_t ld_codes, uint8_t* sf, __nv_bfloat16* y_out, int num_sms, cudaStream_t stream)
{
    const int64_t pad_rows = (rows + 127) / 128 * 128;
    const int64_t blocks = (pad_rows + kRowsPerBlock - 1) / kRowsPerBlock;
    const int64_t cap = (int64_t)num_sms * 8;
    const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
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
