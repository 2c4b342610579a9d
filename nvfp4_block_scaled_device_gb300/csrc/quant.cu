// Row kernels of the NVFP4 path: the device global scale (amax reduction,
// optionally of the RMSNorm of the rows) and the bf16 -> NVFP4 quantizer
// (optionally fused with that RMSNorm), as two kernels and as one
// cooperative launch with a grid barrier between them (the path's form), in
// three variants by size: resident (every row held in registers across the
// barrier), streaming (rows staged in shared memory by bulk copies) and
// looping (rows read from global memory in both phases).
// Four warps per row, 16-byte vector loads, a row share of up to 1536
// columns per warp held in registers, shuffle reductions; all kernels compute
// the RMSNorm with the same routines, so it is bit-identical among them.
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

// Pairs of binary32 values in one 64-bit register, for the packed f32x2
// arithmetic of sm_100-class GPUs (each lane rounded to nearest, as the
// scalar operation): element 0 in the low half.
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_dup(float a)
{
    return ((uint64_t)__float_as_uint(a) << 32) | __float_as_uint(a);
}
// two bf16 (element 0 in the low half of w) -> their binary32 values (exact)
__device__ __forceinline__ uint64_t bf16x2_f2(uint32_t w)
{
    return ((uint64_t)(w & 0xFFFF0000u) << 32) | (uint64_t)(w << 16);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// Two float-float sums side by side (the element pairs' even and odd
// members): the error-free additions of ff_add_f on f32x2 registers.
struct FF2 {
    uint64_t hi, lo;
};

__device__ __forceinline__ FF2 ff2_add_f2(FF2 a, uint64_t p)
{
    const uint64_t s = f2_add(a.hi, p);
    const uint64_t bp = f2_sub(s, a.hi);
    const uint64_t e = f2_add(f2_sub(a.hi, f2_sub(s, bp)), f2_sub(p, bp));
    return {s, f2_add(a.lo, e)};
}

__device__ __forceinline__ FF2 ff2_sumsq8(FF2 acc, const uint4& p)
{
    const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint64_t v = bf16x2_f2(w[i]);
        acc = ff2_add_f2(acc, f2_mul(v, v));            // bf16^2 is exact
    }
    return acc;
}

// the two chains of an FF2, even member first
__device__ __forceinline__ FF ff2_sum(FF2 a)
{
    return ff_add(FF{f2_lo(a.hi), f2_lo(a.lo)}, FF{f2_hi(a.hi), f2_hi(a.lo)});
}

// y = bf16( (x * r) * w ) of 8 bf16 values, one rounding per step (packed).
__device__ __forceinline__ uint4 norm8p(const uint4& xp, uint64_t r2, const uint4& wp)
{
    const uint32_t x[4] = {xp.x, xp.y, xp.z, xp.w};
    const uint32_t w[4] = {wp.x, wp.y, wp.z, wp.w};
    uint32_t y[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint64_t t = f2_mul(f2_mul(bf16x2_f2(x[i]), r2), bf16x2_f2(w[i]));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(y[i]) : "f"(f2_hi(t)), "f"(f2_lo(t)));
    }
    return make_uint4(y[0], y[1], y[2], y[3]);
}

// Running max of |bf16| over packed pairs (exact; no NaN among the inputs).
__device__ __forceinline__ uint32_t amax_bf16x8(uint32_t m, const uint4& p)
{
    uint32_t r = m;
    const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint32_t a;
        asm("abs.bf16x2 %0, %1;" : "=r"(a) : "r"(w[i]));
        asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(r), "r"(a));
    }
    return r;
}
__device__ __forceinline__ float amax_bf16x2_value(uint32_t m) { return fmaxf(bf16_lo(m), bf16_hi(m)); }

// A row is shared by kWarpsPerRow warps: warp q of the row takes the
// 256-column groups q, q + kWarpsPerRow, ... (group j = vectors 32j..32j+31,
// lane l holding vector 32j + l), so a 16-element block sits in a lane pair
// and a 64-element scale word in 8 lanes of one warp.  Up to kRegGroups
// groups of a warp's share are held in registers (rows of up to
// kWarpsPerRow * kRegGroups * 256 = 6144 columns are read once); longer rows
// are read twice (sum of squares, then the row).
constexpr int kWarpsPerRow = 4;
constexpr int kRowsPerBlock = kRowThreads / 32 / kWarpsPerRow;   // 2
constexpr int kRegGroups = 6;

// Per-row scratch of a block: each warp's float-float sum of squares.
struct RowShared {
    float hi[kRowsPerBlock][kWarpsPerRow];
    float lo[kRowsPerBlock][kWarpsPerRow];
};

// Float-float sum of squares of this lane's vectors in its warp's share of
// the row (four independent chains: the even and the odd vectors, each as
// the even and the odd elements of its pairs, then combined in that order),
// shuffle-reduced over the warp (fixed order).
__device__ __forceinline__ FF warp_sumsq(const uint4* __restrict__ b, int ng)
{
    FF2 p0{0, 0}, p1{0, 0};
    for (int k = 0; k < ng; k += 2) {
        p0 = ff2_sumsq8(p0, b[k]);
        if (k + 1 < ng) p1 = ff2_sumsq8(p1, b[k + 1]);
    }
    FF part = ff_add(ff2_sum(p0), ff2_sum(p1));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        FF other{__shfl_xor_sync(0xffffffffu, part.hi, o), __shfl_xor_sync(0xffffffffu, part.lo, o)};
        part = ff_add(part, other);
    }
    return part;
}

// 1 / sqrt(mean(x^2) + eps) of the row from its warps' sums, combined in
// warp order (lane 0 of every warp of the row computes the same value).  The
// squares of bf16 values are exact in binary32 and the float-float sum S =
// hi + lo carries far more precision than binary32.  The mean S / cols is
// rounded once to binary32 without binary64 (slow here): q = hi / n, the
// exact remainder hi - q n by a fused multiply-add, and the correction
// (remainder + lo) / n added to q.  The result is the correctly rounded
// quotient except within about 2^-24 of an ulp of a tie -- the same margin at
// which the float-float sum itself may differ from the exact sum.  Both
// divisions by n are correctly rounded quotients formed from rcp_n = RN(1/n)
// (div_by_recip; a full division where the quotient would be subnormal), and
// 1/sqrt is the correctly rounded reciprocal of the correctly rounded root.
__device__ __forceinline__ float div_by_n(float a, float n, float rcp_n)
{
    const float q = div_by_recip(a, n, rcp_n);
    return fabsf(q) < 1.17549435e-38f ? __fdiv_rn(a, n) : q;
}

__device__ __forceinline__ float row_inv_rms(const RowShared& sh, int rb, int64_t cols, float rcp_n, float eps)
{
    FF t{sh.hi[rb][0], sh.lo[rb][0]};
#pragma unroll
    for (int q = 1; q < kWarpsPerRow; q++) t = ff_add(t, FF{sh.hi[rb][q], sh.lo[rb][q]});
    const float n = (float)cols;                        // exact: cols < 2^24
    const float q0 = div_by_n(t.hi, n, rcp_n);
    const float rem = __fmaf_rn(-q0, n, t.hi);          // exact
    const float ms = __fadd_rn(q0, div_by_n(__fadd_rn(rem, t.lo), n, rcp_n));
    return __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
}

// The quantizer's constants for one global scale g, as quant_half_block
// forms them: d = RN(6 g), rd = RN(1 / d), and for every E4M3 scale code c
// (c = 127, never produced, included) den = RN(dec(c) g) with RN(1 / den),
// in shared memory (built by quant_table once g is known), or tab = NULL:
// each block's den and RN(1 / den) computed where it is quantized (saves the
// table's block barrier where few blocks follow it).
struct QuantK {
    float d, rd;
    const float2* tab;
    float g;
};

__device__ __forceinline__ QuantK quant_direct(float g)
{
    QuantK k;
    k.d = __fmul_rn(6.0f, g);
    k.rd = __frcp_rn(k.d);
    k.tab = nullptr;
    k.g = g;
    return k;
}

// Every thread of the block calls it (one block barrier inside); nt >= 128.
template <int NT>
__device__ __forceinline__ QuantK quant_table(float2* tab, float g)
{
    static_assert(NT >= 128, "one table entry per thread");
    if (threadIdx.x < 128) {
        const float den = __fmul_rn(e4m3_to_f32(threadIdx.x), g);
        tab[threadIdx.x] = make_float2(den, __frcp_rn(den));
    }
    __syncthreads();
    QuantK k = quant_direct(g);
    k.tab = tab;
    return k;
}

// One 8-element vector v of a row, packed bf16 in p (normalised when NORM):
// QUANT: its half of a 16-element block quantized (quant_half_block's
// arithmetic, the per-block divisor from the table) and stored (lanes 2j
// and 2j+1 hold the two halves of a block); otherwise its amax folded in.
template <bool NORM, bool QUANT>
__device__ __forceinline__ void vec_step(const uint4& p, int64_t v, bool valid, int64_t row, int64_t cols,
                                         const QuantK& qk, uint8_t* __restrict__ codes, int64_t ld_codes,
                                         uint8_t* __restrict__ sf, int64_t kb_pad, __nv_bfloat16* __restrict__ y_out,
                                         float* amax)
{
    const float a = amax_bf16x2_value(amax_bf16x8(0u, p));   // exact: bf16 values, no NaN
    if (QUANT) {
        if (NORM && y_out && valid) reinterpret_cast<uint4*>(y_out + row * cols)[v] = p;
        const float a16 = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        const uint32_t sc = cvt_e4m3(div_by_recip(a16, qk.d, qk.rd));
        uint32_t cw = 0u;
        if (sc != 0) {
            float2 t;
            if (qk.tab) {
                t = qk.tab[sc];
            } else {
                t.x = __fmul_rn(e4m3_to_f32(sc), qk.g);
                t.y = __frcp_rn(t.x);
            }
            float f[8];
            unpack8(p, f);
#pragma unroll
            for (int i = 0; i < 8; i++) f[i] = div_by_recip(f[i], t.x, t.y);
            cw = cvt_e2m1x8(f);
        }
        if (valid) {
            const int vi = (int)v;                      // vectors of a row: < 2^31
            *reinterpret_cast<uint32_t*>(codes + row * ld_codes + vi * 4) = cw;
            // the block's scale byte, from the lane holding its first half
            // (sf_offset with the row's part apart: the four bytes of a
            // scale word come from four lanes of one store)
            if ((vi & 1) == 0)
                sf[sf_offset(row, 0, kb_pad) + (vi >> 3) * 512 + ((vi >> 1) & 3)] = (uint8_t)sc;
        }
    } else if (valid) {
        *amax = fmaxf(*amax, a);
    }
}

// This warp's share of one row (row < rows; rb = the row's slot in the
// block, q = the warp's index within the row).  QUANT: quantize and store
// the share; otherwise accumulate its amax (of the normalised row) into
// *amax.  The amax and the quantize kernels both go through here, so the
// RMSNorm they compute is bit-identical.  The block's barrier is executed
// by every warp (NORM only), whatever its row.
// HAVE_R: the row's 1 / rms is given (r_in; no sum of squares, no block
// barrier); otherwise computed and, if r_out is set, stored there by one
// lane of the row.
template <bool NORM, bool QUANT, bool HAVE_R = false>
__device__ __forceinline__ void row_share(const uint4* __restrict__ xr, int64_t row, bool row_valid, int rb, int q,
                                          int64_t nvec, int64_t cols, const uint4* __restrict__ w, float eps,
                                          const QuantK& qk, uint8_t* __restrict__ codes, int64_t ld_codes,
                                          uint8_t* __restrict__ sf, int64_t kb_pad, __nv_bfloat16* __restrict__ y_out,
                                          float* amax, RowShared& sh, float r_in = 1.0f, float* r_out = nullptr)
{
    const int lane = threadIdx.x & 31;
    const int64_t ngroups = (nvec + 31) / 32;
    const int ng = row_valid ? (int)((ngroups - q + kWarpsPerRow - 1) / kWarpsPerRow) : 0;   // this warp's groups
    if (ng <= kRegGroups) {
        uint4 b[kRegGroups];
#pragma unroll
        for (int k = 0; k < kRegGroups; k++) {
            const int64_t v = (int64_t)(q + k * kWarpsPerRow) * 32 + lane;
            b[k] = (k < ng && v < nvec) ? xr[v] : make_uint4(0, 0, 0, 0);
        }
        float r = 1.0f;
        if (NORM && HAVE_R) r = r_in;
        if (NORM && !HAVE_R) {
            const FF part = warp_sumsq(b, kRegGroups);   // zero padding adds exact zeros
            if (lane == 0) {
                sh.hi[rb][q] = part.hi;
                sh.lo[rb][q] = part.lo;
            }
            __syncthreads();
            // one lane per warp (binary64 is slow on this GPU), then broadcast
            if (row_valid && lane == 0) r = row_inv_rms(sh, rb, cols, __frcp_rn((float)cols), eps);
            r = __shfl_sync(0xffffffffu, r, 0);
            if (r_out && q == 0 && lane == 0) *r_out = r;
            __syncthreads();                            // sh is reused by the block's next rows
        }
#pragma unroll
        for (int k = 0; k < kRegGroups; k++) {
            if (k >= ng) break;                         // uniform over the warp
            const int64_t v = (int64_t)(q + k * kWarpsPerRow) * 32 + lane;
            const bool valid = v < nvec;                // uniform over each group of 8 lanes
            const uint4 pv = (NORM && valid) ? norm8p(b[k], f2_dup(r), w[v]) : b[k];
            vec_step<NORM, QUANT>(pv, v, valid, row, cols, qk, codes, ld_codes, sf, kb_pad, y_out, amax);
        }
        return;
    }
    // long rows: sum of squares over the share, then the share again
    float r = 1.0f;
    if (NORM && HAVE_R) r = r_in;
    if (NORM && !HAVE_R) {
        FF2 acc{0, 0};
        for (int k = 0; k < ng; k++) {
            const int64_t v = (int64_t)(q + k * kWarpsPerRow) * 32 + lane;
            acc = ff2_sumsq8(acc, v < nvec ? xr[v] : make_uint4(0, 0, 0, 0));
        }
        FF part = ff2_sum(acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            FF other{__shfl_xor_sync(0xffffffffu, part.hi, o), __shfl_xor_sync(0xffffffffu, part.lo, o)};
            part = ff_add(part, other);
        }
        if (lane == 0) {
            sh.hi[rb][q] = part.hi;
            sh.lo[rb][q] = part.lo;
        }
        __syncthreads();
        if (lane == 0) r = row_inv_rms(sh, rb, cols, __frcp_rn((float)cols), eps);
        r = __shfl_sync(0xffffffffu, r, 0);
        if (r_out && q == 0 && lane == 0) *r_out = r;
        __syncthreads();
    }
    for (int k = 0; k < ng; k++) {
        const int64_t v = (int64_t)(q + k * kWarpsPerRow) * 32 + lane;
        const bool valid = v < nvec;
        const uint4 xv = v < nvec ? xr[v] : make_uint4(0, 0, 0, 0);
        const uint4 pv = (NORM && valid) ? norm8p(xv, f2_dup(r), w[v]) : xv;
        vec_step<NORM, QUANT>(pv, v, valid, row, cols, qk, codes, ld_codes, sf, kb_pad, y_out, amax);
    }
}

template <bool NORM>
__global__ void __launch_bounds__(kRowThreads, 3) amax_scale_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                                                 int64_t cols, int64_t ldx,
                                                                 const __nv_bfloat16* __restrict__ norm_w,
                                                                 float eps, float* __restrict__ g_out,
                                                                 uint32_t* __restrict__ ws)
{
    griddep_launch_dependents();   // a following GEMM may be scheduled early
    __shared__ RowShared sh;
    const int64_t nvec = cols / 8;
    const int wib = threadIdx.x >> 5, rb = wib / kWarpsPerRow, q = wib % kWarpsPerRow;
    float amax = 0.0f;
    // every warp of the block runs the same number of iterations (barriers)
    for (int64_t r0 = (int64_t)blockIdx.x * kRowsPerBlock; r0 < rows; r0 += (int64_t)gridDim.x * kRowsPerBlock) {
        const int64_t row = r0 + rb;
        const bool ok = row < rows;
        row_share<NORM, false>(reinterpret_cast<const uint4*>(x + (ok ? row : 0) * ldx), row, ok, rb, q, nvec, cols,
                               reinterpret_cast<const uint4*>(norm_w), eps, QuantK{}, nullptr, 0, nullptr, 0, nullptr,
                               &amax, sh);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float wmax[kRowThreads / 32];
    if ((threadIdx.x & 31) == 0) wmax[wib] = amax;
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
__global__ void __launch_bounds__(kRowThreads, 3) quantize_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                                               int64_t cols, int64_t ldx,
                                                               const __nv_bfloat16* __restrict__ norm_w, float eps,
                                                               const float* __restrict__ g_ptr,
                                                               uint8_t* __restrict__ codes, int64_t ld_codes,
                                                               uint8_t* __restrict__ sf,
                                                               __nv_bfloat16* __restrict__ y_out)
{
    griddep_launch_dependents();   // a following GEMM may be scheduled early
    __shared__ RowShared sh;
    __shared__ float2 tab[128];
    const QuantK qk = quant_table<kRowThreads>(tab, *g_ptr);
    const int64_t nvec = cols / 8;          // a multiple of 8: cols % 64 == 0
    const int64_t kb_pad = cols / 16;       // already a multiple of 4
    const int64_t pad_rows = (rows + 127) / 128 * 128;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5, rb = wib / kWarpsPerRow, q = wib % kWarpsPerRow;
    // every warp of the block runs the same number of iterations (barriers)
    for (int64_t r0 = (int64_t)blockIdx.x * kRowsPerBlock; r0 < pad_rows; r0 += (int64_t)gridDim.x * kRowsPerBlock) {
        const int64_t row = r0 + rb;
        if (row >= rows && row < pad_rows) {
            // padding rows of the scale layout are zero
            for (int64_t c4 = (int64_t)q * 32 + lane; c4 < kb_pad / 4; c4 += 32 * kWarpsPerRow)
                *reinterpret_cast<uint32_t*>(sf + sf_offset(row, c4 * 4, kb_pad)) = 0u;
        }
        const bool ok = row < rows;
        row_share<NORM, true>(reinterpret_cast<const uint4*>(x + (ok ? row : 0) * ldx), row, ok, rb, q, nvec, cols,
                              reinterpret_cast<const uint4*>(norm_w), eps, qk, codes, ld_codes, sf, kb_pad, y_out,
                              nullptr, sh);
    }
}

__global__ void finalize_scale_kernel(uint32_t* ws, float* g_out)
{
    const float a = __uint_as_float(atomicExch(&ws[0], 0u));
    g_out[0] = __fdiv_rn(fmaxf(a, 1e-8f), 2688.0f);
}

// ---------------------------------------------- scale + quantize, one launch
// The global scale needs the amax of the whole matrix before any block can
// quantize, so the fused kernels run as cooperative launches (every block
// resident) with one grid-wide barrier between the two phases.  Workspace
// words: [0] amax bits (atomicMax), [kArriveWord] arrivals,
// [kDepartWord] departures, in separate L2 sectors (the arrival word is
// polled by every block while the others are updated); the last block to
// depart returns all three to zero.
constexpr int kArriveWord = 32;    // byte 128
constexpr int kDepartWord = 48;    // byte 192

// Block-wide amax of the per-thread values, merged into ws[0]; then the grid
// barrier; returns the global scale to every thread of the block, or -1 if
// the barrier wait gave up (status recorded).  Block 0 writes *g_out.  One
// thread per block touches the words: an atomicMax of the amax, then an
// arrival whose release orders it before the count; the blocks poll the
// count with acquire loads, spaced out so that the polls do not crowd the
// arrivals at the word's L2 slice.  NT: threads of the block.
template <int NT>
__device__ float grid_global_scale(float amax, uint32_t* ws, float* g_out, int* status, int site)
{
    __shared__ float wmax[NT / 32];
    __shared__ float s_g;
    const int wib = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) wmax[wib] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < NT / 32; w++) amax = fmaxf(amax, wmax[w]);
        // non-negative binary32 values order like their bit patterns
        atomicMax(&ws[0], __float_as_uint(amax));
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ws + kArriveWord) : "memory");
        const uint64_t t0 = clock64();
        float g = -1.0f;
        for (;;) {
            uint32_t arrived;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(arrived) : "l"(ws + kArriveWord) : "memory");
            if (arrived >= gridDim.x) {
                uint32_t bits;
                asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(bits) : "l"(ws) : "memory");
                g = __fdiv_rn(fmaxf(__uint_as_float(bits), 1e-8f), 2688.0f);
                break;
            }
            if ((uint64_t)(clock64() - t0) > kWaitLimitCycles) {
                if (status) atomicCAS(status, 0, kErrTimeout * 100 + site);
                break;
            }
            __nanosleep(128);
        }
        s_g = g;
    }
    __syncthreads();
    const float g = s_g;
    if (threadIdx.x == 0 && g >= 0.0f) {
        // off the block's path to its second phase: block 0 publishes the
        // scale; every block has read the amax before it departs, and the
        // last one to depart clears the words for the next call
        if (blockIdx.x == 0) g_out[0] = g;
        uint32_t before;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(before) : "l"(ws + kDepartWord) : "memory");
        if (before == gridDim.x - 1) {
            atomicExch(&ws[0], 0u);
            atomicExch(&ws[kArriveWord], 0u);
            atomicExch(&ws[kDepartWord], 0u);
        }
    }
    return g;
}

// Scale rows [rows, pad128(rows)) of the swizzled layout must be zero.  The
// last 128-row tile of the layout is one contiguous run of bytes: before the
// grid barrier the whole grid clears it with 16-byte stores, and the
// quantization after the barrier writes the tile's real rows over it.
template <int NT>
__device__ __forceinline__ void zero_last_scale_tile(uint8_t* __restrict__ sf, int64_t rows, int64_t kb_pad)
{
    if (rows % 128 == 0) return;
    uint4* t = reinterpret_cast<uint4*>(sf + (rows / 128) * (kb_pad / 4) * 512);
    const int64_t n = kb_pad * 8;                        // (kb_pad / 4) tiles of 32 vectors
    for (int64_t i = (int64_t)blockIdx.x * NT + threadIdx.x; i < n; i += (int64_t)gridDim.x * NT)
        t[i] = make_uint4(0, 0, 0, 0);
}

// Resident variant: every row is held by one block at once (up to kResRows
// rows per block of kResThreads threads, row rb of block b being row
// b + rb * gridDim.x, so the rows spread evenly over the SMs) and each warp's
// share of its row (at most kResGroups 256-column groups) stays in registers
// across the barrier: the row is read once, its RMSNorm computed once and
// held as bf16 for the quantizer.  Few large blocks keep the grid barrier's
// arrivals few.
constexpr int kResGroups = 5;
constexpr int kResMaxCols = kWarpsPerRow * kResGroups * 256;   // 5120
constexpr int kResThreads = 896;
constexpr int kResRows = kResThreads / 32 / kWarpsPerRow;     // 7

struct ResShared {
    float hi[kResRows][kWarpsPerRow];
    float lo[kResRows][kWarpsPerRow];
};

// row_inv_rms over a ResShared (the same combination order as RowShared).
__device__ __forceinline__ float res_inv_rms(const ResShared& sh, int rb, int64_t cols, float rcp_n, float eps)
{
    FF t{sh.hi[rb][0], sh.lo[rb][0]};
#pragma unroll
    for (int q = 1; q < kWarpsPerRow; q++) t = ff_add(t, FF{sh.hi[rb][q], sh.lo[rb][q]});
    const float n = (float)cols;                        // exact: cols < 2^24
    const float q0 = div_by_n(t.hi, n, rcp_n);
    const float rem = __fmaf_rn(-q0, n, t.hi);          // exact
    const float ms = __fadd_rn(q0, div_by_n(__fadd_rn(rem, t.lo), n, rcp_n));
    return __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
}

template <bool NORM>
__global__ void __launch_bounds__(kResThreads, 1)
    scale_quantize_resident_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                                   const __nv_bfloat16* __restrict__ norm_w, float eps, float* __restrict__ g_out,
                                   uint8_t* __restrict__ codes, int64_t ld_codes, uint8_t* __restrict__ sf,
                                   uint32_t* __restrict__ ws, int* status)
{
    griddep_launch_dependents();   // a following GEMM may be scheduled early
    __shared__ ResShared sh;
    __shared__ uint4 w_sh[NORM ? kResMaxCols / 8 : 1];   // the RMSNorm weight, for all rows of the block
    const int64_t nvec = cols / 8;
    const int64_t kb_pad = cols / 16;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5, rb = wib / kWarpsPerRow, q = wib % kWarpsPerRow;
    const int64_t row = (int64_t)blockIdx.x + (int64_t)gridDim.x * rb;
    const bool ok = row < rows;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (ok ? row : 0) * ldx);
    const uint4* w = reinterpret_cast<const uint4*>(norm_w);
    const int64_t ngroups = (nvec + 31) / 32;
    const int ng = ok ? (int)((ngroups - q + kWarpsPerRow - 1) / kWarpsPerRow) : 0;

    uint4 b[kResGroups];
#pragma unroll
    for (int k = 0; k < kResGroups; k++) {
        const int64_t v = (int64_t)(q + k * kWarpsPerRow) * 32 + lane;
        b[k] = (k < ng && v < nvec) ? xr[v] : make_uint4(0, 0, 0, 0);
    }
    if (NORM) {
        // the weight goes to shared memory by asynchronous copies, in flight
        // with the row's loads; the block barrier below makes it visible
        for (int64_t i = threadIdx.x; i < nvec; i += kResThreads)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_u32(&w_sh[i])), "l"(w + i) : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    zero_last_scale_tile<kResThreads>(sf, rows, kb_pad);
    float r = 1.0f;
    if (NORM) {
        const float rcp_n = __frcp_rn((float)cols);    // off the row's critical path
        const FF part = warp_sumsq(b, kResGroups);     // zero padding adds exact zeros
        if (lane == 0) {
            sh.hi[rb][q] = part.hi;
            sh.lo[rb][q] = part.lo;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
        if (ok && lane == 0) r = res_inv_rms(sh, rb, cols, rcp_n, eps);
        r = __shfl_sync(0xffffffffu, r, 0);
    }
    // phase 1: the row (normalised when NORM, kept as bf16) and its amax
    uint32_t amax2 = 0;                                  // packed bf16 running max of |y|
    const uint64_t r2 = f2_dup(r);
#pragma unroll
    for (int k = 0; k < kResGroups; k++) {
        if (k >= ng) break;                             // uniform over the warp
        const int64_t v = (int64_t)(q + k * kWarpsPerRow) * 32 + lane;
        if (v >= nvec) break;                           // uniform over each group of 8 lanes
        if (NORM) b[k] = norm8p(b[k], r2, w_sh[v]);
        amax2 = amax_bf16x8(amax2, b[k]);
    }
    const float g = grid_global_scale<kResThreads>(amax_bf16x2_value(amax2), ws, g_out, status, 7);
    if (g < 0.0f) return;
    const QuantK qk = quant_direct(g);
    // phase 2: quantize the held row
#pragma unroll
    for (int k = 0; k < kResGroups; k++) {
        if (k >= ng) break;
        const int64_t v = (int64_t)(q + k * kWarpsPerRow) * 32 + lane;
        const bool valid = v < nvec;
        vec_step<false, true>(b[k], v, valid, row, cols, qk, codes, ld_codes, sf, kb_pad, nullptr, nullptr);
    }
}

// General variant: blocks loop over the rows in both phases (the rows are
// read twice, as by the two separate kernels).  Phase 2 walks each block's
// rows in the reverse order, so the rows read last in phase 1, still in L2,
// come first; with RMSNorm, phase 1 keeps each row's 1 / rms in shared
// memory (up to kStashIters row pairs per block), so phase 2 does not
// recompute it.
constexpr int kStashIters = 32;

template <bool NORM>
__global__ void __launch_bounds__(kRowThreads, 3)
    scale_quantize_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                          const __nv_bfloat16* __restrict__ norm_w, float eps, float* __restrict__ g_out,
                          uint8_t* __restrict__ codes, int64_t ld_codes, uint8_t* __restrict__ sf,
                          uint32_t* __restrict__ ws, int* status)
{
    griddep_launch_dependents();   // a following GEMM may be scheduled early
    __shared__ RowShared sh;
    __shared__ float r_sh[NORM ? kStashIters : 1][kRowsPerBlock];
    const int64_t nvec = cols / 8;
    const int64_t kb_pad = cols / 16;
    const int wib = threadIdx.x >> 5, rb = wib / kWarpsPerRow, q = wib % kWarpsPerRow;
    const int64_t step = (int64_t)gridDim.x * kRowsPerBlock;
    const int64_t first = (int64_t)blockIdx.x * kRowsPerBlock;
    const int64_t iters = first < rows ? (rows - first + step - 1) / step : 0;   // row pairs of this block
    zero_last_scale_tile<kRowThreads>(sf, rows, kb_pad);
    float amax = 0.0f;
    for (int64_t it = 0; it < iters; it++) {
        const int64_t row = first + it * step + rb;
        const bool ok = row < rows;
        row_share<NORM, false>(reinterpret_cast<const uint4*>(x + (ok ? row : 0) * ldx), row, ok, rb, q, nvec, cols,
                               reinterpret_cast<const uint4*>(norm_w), eps, QuantK{}, nullptr, 0, nullptr, 0, nullptr,
                               &amax, sh, 1.0f, (NORM && it < kStashIters) ? &r_sh[NORM ? it : 0][rb] : nullptr);
    }
    const float g = grid_global_scale<kRowThreads>(amax, ws, g_out, status, 8);
    if (g < 0.0f) return;
    __shared__ float2 tab[128];
    const QuantK qk = quant_table<kRowThreads>(tab, g);
    for (int64_t it = iters - 1; it >= 0; it--) {
        const int64_t row = first + it * step + rb;
        const bool ok = row < rows;
        const uint4* xr = reinterpret_cast<const uint4*>(x + (ok ? row : 0) * ldx);
        if (NORM && it < kStashIters)
            row_share<NORM, true, true>(xr, row, ok, rb, q, nvec, cols, reinterpret_cast<const uint4*>(norm_w), eps, qk,
                                        codes, ld_codes, sf, kb_pad, nullptr, nullptr, sh, r_sh[NORM ? it : 0][rb]);
        else
            row_share<NORM, true>(xr, row, ok, rb, q, nvec, cols, reinterpret_cast<const uint4*>(norm_w), eps, qk, codes,
                                  ld_codes, sf, kb_pad, nullptr, nullptr, sh);
    }
}

// Streaming variant, for more rows than the resident one holds: one block per
// SM of kStrGroups groups of four warps; each group owns kStrSlots row slots
// of shared memory, filled by 1-D bulk copies (one per row, issued by one
// lane, counted on the slot's mbarrier), so the bytes in flight per SM do
// not depend on registers.  Group g of block b takes rows
// (j * kStrGroups + g) * G + b, j = 0, 1, ... (G blocks), so that the grid
// sweeps the matrix in row order.  Phase 1 walks a group's rows forward, a
// slot being refilled with row j + kStrSlots once the group has finished
// row j; the group's last kStrSlots rows stay in their slots.  Phase 2 walks
// them backward: first those held rows (no copy), then the others, each slot
// refilled with row j - kStrSlots once row j is done, so the rows read last
// in phase 1 (the likeliest to be still in L2) are read again first.  Each
// row is handled with the looping variant's arithmetic: the same register
// share per warp, the same float-float sum of squares and the same
// quantizer, so the results are bit-identical to the other variants.
constexpr int kStrGroups = 7;
constexpr int kStrThreads = kStrGroups * kWarpsPerRow * 32;   // 896
constexpr int kStrSlots = 3;
constexpr int kStrStash = 64;                                 // rows per group whose 1 / rms is kept
constexpr int kStrRegGroups = 5;                              // 256-column groups per warp
constexpr int kStrMaxCols = kWarpsPerRow * kStrRegGroups * 256;  // 5120
constexpr int kStrSiteWait = 25;
constexpr int kStrSiteGrid = 26;

__host__ __device__ constexpr size_t str_smem_bytes(int64_t cols)
{
    return (size_t)kStrGroups * kStrSlots * (size_t)cols * 2;
}

// The four warps of group grp (named barrier 1 + grp).
__device__ __forceinline__ void group_sync(int grp)
{
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kWarpsPerRow * 32) : "memory");
}

// row_inv_rms over one group's four warp sums (the same order and arithmetic).
__device__ __forceinline__ float grp_inv_rms(const float* hi, const float* lo, int64_t cols, float rcp_n, float eps)
{
    FF t{hi[0], lo[0]};
#pragma unroll
    for (int q = 1; q < kWarpsPerRow; q++) t = ff_add(t, FF{hi[q], lo[q]});
    const float n = (float)cols;                        // exact: cols < 2^24
    const float q0 = div_by_n(t.hi, n, rcp_n);
    const float rem = __fmaf_rn(-q0, n, t.hi);          // exact
    const float ms = __fadd_rn(q0, div_by_n(__fadd_rn(rem, t.lo), n, rcp_n));
    return __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
}

template <bool NORM>
__global__ void __launch_bounds__(kStrThreads, 1)
    scale_quantize_stream_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                                 const __nv_bfloat16* __restrict__ norm_w, float eps, float* __restrict__ g_out,
                                 uint8_t* __restrict__ codes, int64_t ld_codes, uint8_t* __restrict__ sf,
                                 uint32_t* __restrict__ ws, int* status)
{
    griddep_launch_dependents();   // a following GEMM may be scheduled early
    extern __shared__ __align__(128) uint8_t str_slots[];
    __shared__ __align__(8) uint64_t full[kStrGroups][kStrSlots];
    __shared__ float sh_hi[kStrGroups][kWarpsPerRow], sh_lo[kStrGroups][kWarpsPerRow];
    __shared__ float r_sh[NORM ? kStrGroups : 1][NORM ? kStrStash : 1];
    __shared__ float2 tab[128];
    __shared__ int abort_flag;
    const int64_t nvec = cols / 8;
    const int64_t kb_pad = cols / 16;
    const uint32_t row_bytes = (uint32_t)(cols * 2);
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5, grp = wib / kWarpsPerRow, q = wib % kWarpsPerRow;
    const int64_t stride = (int64_t)gridDim.x * kStrGroups;           // rows per step j
    const int64_t base = (int64_t)grp * gridDim.x + blockIdx.x;      // the group's row at j = 0
    const int m = base < rows ? (int)((rows - base + stride - 1) / stride) : 0;
    const int64_t ngroups = (nvec + 31) / 32;
    const int ng = (int)((ngroups - q + kWarpsPerRow - 1) / kWarpsPerRow);   // this warp's 256-column groups
    const uint4* w = reinterpret_cast<const uint4*>(norm_w);
    const bool leader = q == 0;                                      // issues the group's copies
    uint8_t* my_slots = str_slots + (size_t)grp * kStrSlots * row_bytes;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStrGroups * kStrSlots; i++) mbar_init(smem_u32(&full[i / kStrSlots][i % kStrSlots]), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    uint32_t ph = 0;     // per slot: parity of its next fill
    uint32_t pend = 0;   // leader: slots with a fill issued and not yet waited for
    auto issue = [&](int j) {
        const int s = j % kStrSlots;
        const uint32_t bar = smem_u32(&full[grp][s]);
        if (elect_one()) {
            mbar_arrive_expect_tx(bar, row_bytes);
            bulk_load(smem_u32(my_slots + (size_t)s * row_bytes), x + (base + (int64_t)j * stride) * ldx, row_bytes,
                      bar);
        }
        __syncwarp();
        pend |= 1u << s;
    };
    // wait for row j's fill; false (nothing done) once the block has aborted
    auto wait = [&](int j) -> bool {
        const int s = j % kStrSlots;
        if (__shfl_sync(0xffffffffu, *(volatile int*)&abort_flag, 0)) return false;
        if (!mbar_wait_warp(smem_u32(&full[grp][s]), (ph >> s) & 1u, &abort_flag, status, kStrSiteWait))
            return false;
        ph ^= 1u << s;
        pend &= ~(1u << s);
        return true;
    };
    auto load_share = [&](int j, bool ok, uint4* b) {
        const uint4* rs = reinterpret_cast<const uint4*>(my_slots + (size_t)(j % kStrSlots) * row_bytes);
#pragma unroll
        for (int k = 0; k < kStrRegGroups; k++) {
            const int64_t v = (int64_t)(q + k * kWarpsPerRow) * 32 + lane;
            b[k] = (ok && k < ng && v < nvec) ? rs[v] : make_uint4(0, 0, 0, 0);
        }
    };
    // 1 / rms of the row whose share is in b (every warp of the group calls it)
    const float rcp_n = __frcp_rn((float)cols);
    auto inv_rms = [&](const uint4* b) -> float {
        const FF part = warp_sumsq(b, kStrRegGroups);       // zero padding adds exact zeros
        if (lane == 0) {
            sh_hi[grp][q] = part.hi;
            sh_lo[grp][q] = part.lo;
        }
        group_sync(grp);
        float r = 1.0f;
        if (lane == 0) r = grp_inv_rms(sh_hi[grp], sh_lo[grp], cols, rcp_n, eps);
        return __shfl_sync(0xffffffffu, r, 0);
    };

    if (leader)
        for (int j = 0; j < kStrSlots && j < m; j++) issue(j);

    // phase 1: amax of the rows (normalised when NORM)
    uint32_t amax2 = 0;
    for (int j = 0; j < m; j++) {
        const bool ok = wait(j);
        uint4 b[kStrRegGroups];
        load_share(j, ok, b);
        if (NORM) {
            const float r = inv_rms(b);
            if (q == 0 && lane == 0 && j < kStrStash) r_sh[NORM ? grp : 0][NORM ? j : 0] = r;
            const uint64_t r2 = f2_dup(r);
#pragma unroll
            for (int k = 0; k < kStrRegGroups; k++) {
                const int64_t v = (int64_t)(q + k * kWarpsPerRow) * 32 + lane;
                if (ok && k < ng && v < nvec) amax2 = amax_bf16x8(amax2, norm8p(b[k], r2, w[v]));
            }
        } else {
#pragma unroll
            for (int k = 0; k < kStrRegGroups; k++) amax2 = amax_bf16x8(amax2, b[k]);   // zeros elsewhere
        }
        group_sync(grp);   // the group is done with the slot (and with sh_hi / sh_lo)
        const bool ab = __shfl_sync(0xffffffffu, *(volatile int*)&abort_flag, 0);   // uniform per warp
        if (leader && j + kStrSlots < m && !ab) issue(j + kStrSlots);
    }
    zero_last_scale_tile<kStrThreads>(sf, rows, kb_pad);
    const float g = grid_global_scale<kStrThreads>(amax_bf16x2_value(amax2), ws, g_out, status, kStrSiteGrid);
    if (g >= 0.0f) {
        const QuantK qk = quant_table<kStrThreads>(tab, g);
        // phase 2: quantize, last rows first
        for (int j = m - 1; j >= 0; j--) {
            const bool held = j >= m - kStrSlots;   // still in its slot from phase 1
            const bool ok = held ? !__shfl_sync(0xffffffffu, *(volatile int*)&abort_flag, 0) : wait(j);
            uint4 b[kStrRegGroups];
            load_share(j, ok, b);
            float r = 1.0f;
            if (NORM) r = j < kStrStash ? r_sh[NORM ? grp : 0][NORM ? j : 0] : inv_rms(b);
            const uint64_t r2 = f2_dup(r);
            const int64_t row = base + (int64_t)j * stride;
#pragma unroll
            for (int k = 0; k < kStrRegGroups; k++) {
                if (!ok || k >= ng) break;                   // uniform over the warp
                const int64_t v = (int64_t)(q + k * kWarpsPerRow) * 32 + lane;
                const bool valid = v < nvec;                 // uniform over each group of 8 lanes
                const uint4 pv = (NORM && valid) ? norm8p(b[k], r2, w[v]) : b[k];
                vec_step<false, true>(pv, v, valid, row, cols, qk, codes, ld_codes, sf, kb_pad, nullptr, nullptr);
            }
            group_sync(grp);
            const bool ab = __shfl_sync(0xffffffffu, *(volatile int*)&abort_flag, 0);
            if (leader && j - kStrSlots >= 0 && !ab) issue(j - kStrSlots);
        }
    }
    // after an abort: let the copies still in flight land before the block exits
    if (leader && pend)
        for (int s = 0; s < kStrSlots; s++)
            if (pend & (1u << s)) mbar_wait_teardown(smem_u32(&full[grp][s]), (ph >> s) & 1u);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_cooperative(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                               cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Blocks of a kernel that can be resident on one SM at once.
int blocks_per_sm(const void* kernel, int threads, size_t smem = 0)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) return 0;
    return n;
}

// Dynamic shared memory the streaming variant may take (its static shared
// memory is a few KB).
constexpr size_t kStrSmemLimit = 220 * 1024;

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

cudaError_t launch_scale_quantize(const __nv_bfloat16* x, int64_t rows, int64_t cols, int64_t ldx,
                                  const __nv_bfloat16* norm_w, float eps, float* g_out, uint8_t* codes,
                                  int64_t ld_codes, uint8_t* sf, uint32_t* ws, int* status, int num_sms,
                                  cudaStream_t stream)
{
    // resident blocks per SM of the four kernels, per device
    // (the streaming kernels' with their largest shared memory size)
    static int occ[64][6];
    static bool have[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    if (!have[dev]) {
        e = cudaFuncSetAttribute((const void*)scale_quantize_stream_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStrSmemLimit);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute((const void*)scale_quantize_stream_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStrSmemLimit);
        if (e != cudaSuccess) return e;
        occ[dev][0] = blocks_per_sm((const void*)scale_quantize_resident_kernel<false>, kResThreads);
        occ[dev][1] = blocks_per_sm((const void*)scale_quantize_resident_kernel<true>, kResThreads);
        occ[dev][2] = blocks_per_sm((const void*)scale_quantize_kernel<false>, kRowThreads);
        occ[dev][3] = blocks_per_sm((const void*)scale_quantize_kernel<true>, kRowThreads);
        occ[dev][4] = blocks_per_sm((const void*)scale_quantize_stream_kernel<false>, kStrThreads, kStrSmemLimit);
        occ[dev][5] = blocks_per_sm((const void*)scale_quantize_stream_kernel<true>, kStrThreads, kStrSmemLimit);
        for (int i = 0; i < 4; i++)
            if (occ[dev][i] < 1) return cudaErrorInvalidConfiguration;
        have[dev] = true;
    }
    const bool norm = norm_w != nullptr;
    // resident: a grid of min(rows, resident blocks) blocks, each holding
    // rows b, b + grid, ... (at most kResRows of them)
    const int64_t res_blocks = (int64_t)occ[dev][norm ? 1 : 0] * num_sms;
    if (cols <= kResMaxCols && rows <= res_blocks * kResRows) {
        const unsigned grid = (unsigned)(rows < res_blocks ? rows : res_blocks);
        if (norm)
            return launch_cooperative(scale_quantize_resident_kernel<true>, grid, kResThreads, 0, stream, x, rows, cols,
                                      ldx, norm_w, eps, g_out, codes, ld_codes, sf, ws, status);
        return launch_cooperative(scale_quantize_resident_kernel<false>, grid, kResThreads, 0, stream, x, rows, cols, ldx,
                                  norm_w, eps, g_out, codes, ld_codes, sf, ws, status);
    }
    // streaming: rows of up to kStrMaxCols columns whose slots fit in shared
    // memory, one block per SM
    const size_t str_smem = str_smem_bytes(cols);
    if (cols <= kStrMaxCols && str_smem <= kStrSmemLimit && occ[dev][norm ? 5 : 4] >= 1) {
        const unsigned grid = (unsigned)num_sms;
        if (norm)
            return launch_cooperative(scale_quantize_stream_kernel<true>, grid, kStrThreads, str_smem, stream, x, rows,
                                      cols, ldx, norm_w, eps, g_out, codes, ld_codes, sf, ws, status);
        return launch_cooperative(scale_quantize_stream_kernel<false>, grid, kStrThreads, str_smem, stream, x, rows,
                                  cols, ldx, norm_w, eps, g_out, codes, ld_codes, sf, ws, status);
    }
    const int64_t pairs = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    const int64_t cap = (int64_t)occ[dev][norm ? 3 : 2] * num_sms;
    const unsigned grid = (unsigned)(pairs < cap ? pairs : cap);
    if (norm)
        return launch_cooperative(scale_quantize_kernel<true>, grid, kRowThreads, 0, stream, x, rows, cols, ldx, norm_w,
                                  eps, g_out, codes, ld_codes, sf, ws, status);
    return launch_cooperative(scale_quantize_kernel<false>, grid, kRowThreads, 0, stream, x, rows, cols, ldx, norm_w, eps,
                              g_out, codes, ld_codes, sf, ws, status);
}

}  // namespace nvfp4
