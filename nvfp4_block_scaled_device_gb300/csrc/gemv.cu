// Decode-regime NVFP4 GEMM: out[m, n] = alpha * sum_k dA[m, k] * dW[n, k]
// for a handful of activation rows m (T = 1, 2 tokens per step), with the
// same epilogues as the tensor-core kernels (bf16 [+ residual]; SwiGLU
// requantized to FP4, or stored as bf16 with its amax).
//
// At T <= 2 the GEMM is a weight stream: every weight byte is used for one
// or two multiply-adds, so the bound is HBM bandwidth, not the tensor pipe
// (the tensor-core kernels, whose smallest tile has 128 activation rows, run
// such shapes at a fraction of HBM speed, limited by their fixed latencies
// where the weights are small; see kDecodeMaxWeightBytes).
// This kernel reads each weight byte once, with coalesced 16-byte loads, and
// does the arithmetic on the CUDA cores in integers:
//   - an E2M1 code times two is an integer in [-12, 12], so one 16-element
//     block's sum of code products is an exact int32 from eight dp4a
//     (positive and negative weight codes taken apart by a byte permute, one
//     dp4a each);
//   - that sum times the two E4M3 block scales is exact in fp32, and the
//     blocks accumulate in fp32 (the same arithmetic as the tensor pipe's
//     block-scaled MMA, in another summation order).
// Sources: "tp>1 prefill is host-bound: per-token fp4 GEMM + per-layer H2D
// activation staging" (vllm.cpp issue 2144), whose profile compares the fp4
// MLP of a decode step (T=1) with T=5; "PERFORMANCE -- verified hot-path
// audit and prioritized fixes", which targets the single-GPU per-token
// decode step (its CUDA-graph item, roadmap E9).
//
// Work split.  One CTA of 16 warps per SM.  CTA c owns a contiguous range of
// output columns (whole column pairs, which the rotary embedding rotates;
// whole 16-column blocks for the SwiGLU epilogues, whose requantization
// needs them); its weight rows (gate rows, then up rows, for
// SwiGLU) are cut into units of 512 code bytes (1024 elements; 16 bytes per
// lane), and warp w takes the contiguous unit range [w U/16, (w+1) U/16).
// Each lane keeps kDepth units in flight in registers (loaded ahead of the
// arithmetic), so an SM has ~64 KB of weight loads outstanding.  A warp
// reduces its lanes' partial sums at each row boundary into a shared-memory
// slot; after the stream the CTA adds a row's slots in warp order
// (deterministic), and runs the epilogue.  The activation rows are expanded
// once per CTA into shared memory as int8 (2 x E2M1) and fp32 scales.
#include "common.cuh"
#include "decode_epilogue.cuh"
#include "gemv.h"

#ifndef NVFP4_DECODE_MAX_ROWS
#define NVFP4_DECODE_MAX_ROWS kDecodeMaxRows
#endif

namespace nvfp4 {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kDepth = 8;              // units in flight per lane
constexpr int kUnitBytes = 512;        // code bytes of a unit (16 per lane)
constexpr int kUnitElems = 1024;
constexpr int kMaxKernelRows = 4;      // instantiated activation row counts: 1..4
constexpr size_t kMaxSmem = 200 * 1024;

// Magnitude table of 2 x E2M1 (code & 7 -> 0, 1, 2, 3, 4, 6, 8, 12), as the
// eight source bytes of a byte permute.
constexpr uint32_t kMagLo = 0x03020100u;
constexpr uint32_t kMagHi = 0x0C080604u;

struct DecodeParams {
    GemmArgs g;
    DecodeOperands op;
    int segs;    // units per weight row: ceil(K / 1024)
    int slots;   // partial-sum slots per warp
};

// Byte permute: result byte i = source byte (sel nibble i & 7) of {b, a};
// a selector nibble with bit 3 set gives instead the sign of that byte
// replicated (0x00 for the table bytes above, which are all < 0x80).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The four E2M1 codes in the low 16 bits of w -> four bytes 2*|value| of
// the positive codes (negative codes give 0), and of the negative codes.
__device__ __forceinline__ uint32_t mag_pos(uint32_t w) { return prmt(kMagLo, kMagHi, w); }
__device__ __forceinline__ uint32_t mag_neg(uint32_t w) { return prmt(kMagLo, kMagHi, w ^ 0x8888u); }

// Four E2M1 codes (low 16 bits) -> four signed int8 values 2 x E2M1.
__device__ __forceinline__ uint32_t e2m1x4_to_s8(uint32_t w) { return __vsub4(mag_pos(w), mag_neg(w)); }

// Streamed 16-byte weight load (read once: not kept in L1).
__device__ __forceinline__ uint4 ldg_stream(const uint8_t* p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Two weight scale bytes (kept in L1: the CTA's neighbouring rows share
// their 32-byte sectors).
__device__ __forceinline__ uint32_t ldg_sf2(const uint8_t* p)
{
    uint16_t v;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

template <int kM>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const DecodeParams prm)
{
    extern __shared__ __align__(16) uint8_t smem[];
    griddep_launch_dependents();
    const GemmArgs& args = prm.g;
    const bool swiglu = args.epilogue != kEpiBf16;
    const int S = prm.segs;
    const int code_bytes = (int)(args.K / 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this CTA's output columns [n0, n0 + C) and weight rows (R of them)
    int64_t n0;
    int C, R;
    if (swiglu) {
        const int64_t nb = args.N / 16;
        const int64_t b0 = (int64_t)blockIdx.x * nb / gridDim.x, b1 = (int64_t)(blockIdx.x + 1) * nb / gridDim.x;
        n0 = 16 * b0;
        C = (int)(16 * (b1 - b0));
        R = 2 * C;
    } else {
        // whole column pairs (the rotary embedding rotates pairs)
        const int64_t np = args.N / 2;
        const int64_t p0 = (int64_t)blockIdx.x * np / gridDim.x, p1 = (int64_t)(blockIdx.x + 1) * np / gridDim.x;
        n0 = 2 * p0;
        C = (int)(2 * (p1 - p0));
        R = C;
    }
    const int U = R * S;
    const int u_beg = warp * U / kWarps, u_end = (warp + 1) * U / kWarps;

    // shared memory: A as int8 [kM][S][64 chunks of 16], chunk c of a unit
    // at position (c & 1) * 32 + c / 2 (so that lane l's chunks 2l and 2l+1
    // are two conflict-free 512-byte rows); A scales * 2^119 [kM][S][64];
    // partial sums [kWarps][slots][kM]; row sums [R][kM]
    int8_t* a_q = reinterpret_cast<int8_t*>(smem);
    float* a_s = reinterpret_cast<float*>(smem + (size_t)kM * S * kUnitElems);
    float* part = a_s + (size_t)kM * S * 64;
    float* racc = part + (size_t)kWarps * prm.slots * kM;

    // ---- weight stream: load cursor (row lr, unit lj of the row)
    uint4 buf[kDepth];
    uint32_t bsf[kDepth];
    int lu = u_beg, lr = u_beg / S, lj = u_beg % S;
    const uint8_t* lcp = nullptr;   // this lane's 16 bytes of unit 0 of row lr
    const uint8_t* lsp = nullptr;   // this lane's 2 scale bytes of unit 0 of row lr
    auto row_ptrs = [&](int r) {
        const uint8_t* w = prm.op.b0_codes;
        const uint8_t* sf = args.sfb0;
        int64_t ld = prm.op.ldb0;
        int64_t n = n0 + r;
        if (swiglu && r >= C) {
            w = prm.op.b1_codes;
            sf = args.sfb1;
            ld = prm.op.ldb1;
            n -= C;
        }
        lcp = w + n * ld + 16 * lane;
        // scale column 64 j + 2 lane (+1) of row n: tile 16 j + lane / 2
        lsp = sf + (n >> 7) * args.sfb_tile_stride + (n & 31) * 16 + ((n & 127) >> 5) * 4 + (lane >> 1) * 512 +
              2 * (lane & 1);
    };
    auto issue = [&](uint4& wc, uint32_t& ws) {
        if (lu < u_end) {
            const bool ok = kUnitBytes * lj + 16 * lane < code_bytes;   // ragged last unit of a row
            wc = ok ? ldg_stream(lcp + (size_t)kUnitBytes * lj) : make_uint4(0u, 0u, 0u, 0u);
            ws = ok ? ldg_sf2(lsp + (size_t)(16 * 512) * lj) : 0u;
            ++lu;
            if (++lj == S) {
                lj = 0;
                ++lr;
                if (lu < u_end) row_ptrs(lr);
            }
        }
    };
    if (u_beg < u_end) row_ptrs(lr);
    // The weights may be read before the previous kernel of the stream has
    // completed only when the caller vouches they were complete before it.
    if (!args.weights_early) griddep_wait();
#pragma unroll
    for (int i = 0; i < kDepth; i++) issue(buf[i], bsf[i]);
    griddep_wait();

    // ---- activations -> shared memory
    for (int t = threadIdx.x; t < kM * S * 64; t += kThreads) {
        const int m = t / (S * 64), j = (t / 64) % S, c = t % 64;
        const int64_t e0 = (int64_t)j * kUnitElems + 16 * c;
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        if (e0 < args.K) {
            const uint2 w = *reinterpret_cast<const uint2*>(prm.op.a_codes + m * prm.op.lda + e0 / 2);
            q.x = e2m1x4_to_s8(w.x);
            q.y = e2m1x4_to_s8(w.x >> 16);
            q.z = e2m1x4_to_s8(w.y);
            q.w = e2m1x4_to_s8(w.y >> 16);
        }
        const int p = (c & 1) * 32 + (c >> 1);
        *reinterpret_cast<uint4*>(a_q + ((size_t)(m * S + j) * 64 + p) * 16) = q;
        // scale of block (m, 64 j + c), times 2^119 (exact: at most 448 * 2^119 < 2^128)
        const int64_t blk = (int64_t)j * 64 + c;
        float s = 0.0f;
        if (blk < args.K / 16) {
            const int64_t off = (blk >> 2) * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4 + (blk & 3);
            s = __fmul_rn(e4m3_to_f32(args.sfa[off]), 0x1p119f);
        }
        a_s[t] = s;   // t == (m * S + j) * 64 + c
    }
    __syncthreads();

    // ---- the stream: unit u of this warp is (row cr, unit cj of the row)
    float acc[kM];
#pragma unroll
    for (int m = 0; m < kM; m++) acc[m] = 0.0f;
    int cj = u_beg % S, slot = 0;
    const uint32_t aq_lane = smem_u32(a_q) + 16u * lane;
    auto flush = [&]() {
#pragma unroll
        for (int m = 0; m < kM; m++) {
            float v = acc[m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0 && slot < prm.slots) part[(warp * prm.slots + slot) * kM + m] = v;
            acc[m] = 0.0f;
        }
        ++slot;
    };
    for (int base = u_beg; base < u_end; base += kDepth) {
#pragma unroll
        for (int i = 0; i < kDepth; i++) {
            if (base + i < u_end) {
                const uint4 wc = buf[i];
                const uint32_t wsf = bsf[i];
                issue(buf[i], bsf[i]);   // refill the slot with the unit kDepth ahead
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    // block 64 cj + 2 lane + h: 16 codes in two words
                    const uint32_t w0 = h ? wc.z : wc.x, w1 = h ? wc.w : wc.y;
                    const uint32_t p0 = mag_pos(w0), p1 = mag_pos(w0 >> 16), p2 = mag_pos(w1), p3 = mag_pos(w1 >> 16);
                    const uint32_t q0 = mag_neg(w0), q1 = mag_neg(w0 >> 16), q2 = mag_neg(w1), q3 = mag_neg(w1 >> 16);
                    // E4M3 scale * 2^-120 (exact, subnormal range included)
                    const float swr = __uint_as_float(((wsf >> (8 * h)) & 0xFFu) << 20);
#pragma unroll
                    for (int m = 0; m < kM; m++) {
                        const uint32_t ua = (uint32_t)(((m * S + cj) * 64 + h * 32) * 16);
                        const uint4 av = lds128(aq_lane + ua);
                        const float sa = a_s[(m * S + cj) * 64 + 2 * lane + h];
                        int sp = __dp4a((int)av.x, (int)p0, 0);
                        sp = __dp4a((int)av.y, (int)p1, sp);
                        sp = __dp4a((int)av.z, (int)p2, sp);
                        sp = __dp4a((int)av.w, (int)p3, sp);
                        int sn = __dp4a((int)av.x, (int)q0, 0);
                        sn = __dp4a((int)av.y, (int)q1, sn);
                        sn = __dp4a((int)av.z, (int)q2, sn);
                        sn = __dp4a((int)av.w, (int)q3, sn);
                        // (4 x code-product sum) * sA * sW / 2: exact; one rounding in the sum
                        acc[m] = __fmaf_rn((float)(sp - sn), __fmul_rn(sa, swr), acc[m]);
                    }
                }
                if (++cj == S) {
                    cj = 0;
                    flush();
                }
            }
        }
    }
    if (cj != 0) flush();   // the warp's range ended inside a row
    __syncthreads();

    // ---- row sums: a row's slots in warp order; acc holds 2 x the dot product
    for (int t = threadIdx.x; t < R * kM; t += kThreads) {
        const int r = t / kM, m = t % kM;
        float s = 0.0f;
        for (int w = 0; w < kWarps; w++) {
            const int b = w * U / kWarps, e = (w + 1) * U / kWarps;
            if (b == e) continue;
            const int rf = b / S, rl = (e - 1) / S;
            if (r >= rf && r <= rl) s = __fadd_rn(s, part[(w * prm.slots + (r - rf)) * kM + m]);
        }
        racc[t] = __fmul_rn(s, 0.5f);
    }
    __syncthreads();

    // ---- epilogue
    decode_epilogue<kThreads>(args, epi_scalars(args), racc, kM, n0, C, threadIdx.x);
}

// Grid, slots and shared memory of one launch.
struct DecodeShape {
    int grid, segs, slots;
    size_t smem;
};

DecodeShape decode_shape(const GemmArgs& a, int num_sms)
{
    DecodeShape d{};
    const bool swiglu = a.epilogue != kEpiBf16;
    const int64_t units = swiglu ? a.N / 16 : a.N / 2;   // column pairs, or 16-column blocks
    d.grid = (int)(units < num_sms ? units : num_sms);
    d.segs = (int)((a.K + kUnitElems - 1) / kUnitElems);
    const int64_t per = (units + d.grid - 1) / d.grid;
    const int64_t rmax = swiglu ? 32 * per : 2 * per;              // weight rows of a CTA, at most
    const int64_t umax = (rmax * d.segs + kWarps - 1) / kWarps;    // units of a warp, at most
    d.slots = (int)((umax + 2 * d.segs - 2) / d.segs);             // rows a warp's range touches, at most
    d.smem = (size_t)a.M * d.segs * (kUnitElems + 64 * 4) + (size_t)kWarps * d.slots * a.M * 4 +
             (size_t)rmax * a.M * 4;
    if (rmax * d.segs > (int64_t)1 << 26) d.smem = ~(size_t)0;     // keep the unit counts far from overflow
    return d;
}

template <int kM>
cudaError_t launch_rows(const DecodeParams& prm, const DecodeShape& d, cudaStream_t stream)
{
    static int attr_set_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set_for_device[dev]) {
        e = cudaFuncSetAttribute(gemv_kernel<kM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    return launch_programmatic(gemv_kernel<kM>, dim3((unsigned)d.grid), dim3(kThreads), d.smem, stream, prm);
}

}  // namespace

bool gemv_eligible(const GemmArgs& args, int num_sms)
{
    static_assert(NVFP4_DECODE_MAX_ROWS <= kMaxKernelRows, "decode kernel instantiated for at most 4 rows");
    if (args.M < 1 || args.M > NVFP4_DECODE_MAX_ROWS || num_sms < 1) return false;
    const int64_t weight_bytes = (args.epilogue != kEpiBf16 ? 2 : 1) * args.N * (args.K / 2);
    if (weight_bytes > kDecodeMaxWeightBytes) return false;
    return decode_shape(args, num_sms).smem <= kMaxSmem;
}

cudaError_t launch_gemv(const DecodeOperands& ops, const GemmArgs& args, int num_sms, cudaStream_t stream)
{
    if (!gemv_eligible(args, num_sms)) return cudaErrorInvalidValue;
    const DecodeShape d = decode_shape(args, num_sms);
    DecodeParams prm;
    prm.g = args;
    prm.op = ops;
    prm.segs = d.segs;
    prm.slots = d.slots;
    switch (args.M) {
        case 1: return launch_rows<1>(prm, d, stream);
        case 2: return launch_rows<2>(prm, d, stream);
        case 3: return launch_rows<3>(prm, d, stream);
        default: return launch_rows<4>(prm, d, stream);
    }
}

}  // namespace nvfp4
