// Epilogue of the decode-regime kernels (a handful of activation rows):
// from one block of finished dot products in shared memory to the outputs,
// with the same arithmetic as the tensor-core kernels' per-row epilogue.
//   racc[r * M + m]: dot product of activation row m with weight row r of
//   the block, r < R; bf16 epilogue: R = C output columns n0 .. n0 + C - 1;
//   SwiGLU: R = 2C, gate rows first, then the up rows of the same columns.
// Every thread of the kNT taking part calls it (the SwiGLU branch
// exchanges values between neighbouring lanes).
#pragma once

#include "common.cuh"
#include "gemm_epilogue.cuh"
#include "internal.h"

namespace nvfp4 {

// The epilogue's scalars: alpha of the (gate) weights and of the up
// weights, fp32(gA * gW); the intermediate scale (FP4 SwiGLU epilogue).
struct EpiScalars {
    float alpha0, alpha1, g_inter;
};

__device__ __forceinline__ EpiScalars epi_scalars(const GemmArgs& args)
{
    EpiScalars e;
    const float ga = *args.ga;
    e.alpha0 = __fmul_rn(ga, *args.gb0);
    e.alpha1 = args.epilogue != kEpiBf16 ? __fmul_rn(ga, *args.gb1) : e.alpha0;
    e.g_inter = args.epilogue == kEpiSwigluFp4 ? *args.g_inter : 1.0f;
    return e;
}

template <int kNT>
__device__ __forceinline__ void decode_epilogue(const GemmArgs& args, const EpiScalars& es, const float* racc, int M,
                                                int64_t n0, int C, int tid)
{
    const float alpha0 = es.alpha0;
    if (args.epilogue == kEpiBf16) {
        // out = bf16(alpha * acc) [rotated] [then bf16(residual + that)];
        // consecutive threads take consecutive column pairs
        const int pairs = C / 2;
        for (int t = tid; t < M * pairs; t += kNT) {
            const int m = t / pairs, r = 2 * (t % pairs);
            const int64_t n = n0 + r;
            uint32_t o;
            if (args.rope_pos) {
                // rotated in binary32 from the rounded values (no residual)
                float y0 = bf16_round(__fmul_rn(racc[r * M + m], alpha0));
                float y1 = bf16_round(__fmul_rn(racc[(r + 1) * M + m], alpha0));
                RopeCursor rk = rope_begin(args, m, n);
                rope_step(args, rk, y0, y1);
                o = pack_bf16x2(y0, y1);
            } else {
                o = cvt_bf16x2(__fmul_rn(racc[r * M + m], alpha0), __fmul_rn(racc[(r + 1) * M + m], alpha0));
                if (args.residual)
                    o = add_bf16x2(*reinterpret_cast<const uint32_t*>(args.residual + m * args.ldr + n), o);
            }
            *reinterpret_cast<uint32_t*>(args.out + m * args.ldo + n) = o;
        }
        return;
    }
    const float alpha1 = es.alpha1;
    const float g_inter = es.g_inter;
    float wamax = 0.0f;
    // s = bf16(silu(gate) * up), gate and up rounded to bf16 first; a thread
    // takes 8 columns of one row, lanes 2q and 2q+1 one 16-column block
    const int groups = M * (C / 8);
    for (int g0 = 0; g0 < groups; g0 += kNT) {   // the same trip count for every thread
        const int t = g0 + tid;
        const bool act = t < groups;
        const int m = act ? t / (C / 8) : 0, i0 = act ? 8 * (t % (C / 8)) : 0;
        float v[8];
        float a8 = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            v[k] = 0.0f;
            if (act) {
                const float gate = bf16_round(__fmul_rn(racc[(i0 + k) * M + m], alpha0));
                const float up = bf16_round(__fmul_rn(racc[(C + i0 + k) * M + m], alpha1));
                v[k] = bf16_round(silu_mul(gate, up));
                a8 = fmaxf(a8, fabsf(v[k]));
            }
        }
        const float a16 = fmaxf(a8, __shfl_xor_sync(0xffffffffu, a8, 1));
        if (act) {
            const int64_t n = n0 + i0;
            if (args.s_bf16) {
                uint4 o;
                o.x = pack_bf16x2(v[0], v[1]);
                o.y = pack_bf16x2(v[2], v[3]);
                o.z = pack_bf16x2(v[4], v[5]);
                o.w = pack_bf16x2(v[6], v[7]);
                *reinterpret_cast<uint4*>(args.s_bf16 + m * args.ld_s + n) = o;
            }
            if (args.epilogue == kEpiSwigluFp4) {
                uint32_t sc;
                const uint32_t cw = quant_half_block(v, g_inter, a16, &sc);
                *reinterpret_cast<uint32_t*>(args.s_codes + m * args.ld_s_codes + n / 2) = cw;
                if ((i0 & 8) == 0) args.s_sf[sf_offset(m, n / 16, args.s_kb_pad)] = (uint8_t)sc;
            } else {
                wamax = fmaxf(wamax, a8);
            }
        }
    }
    if (args.epilogue == kEpiSwigluFp4) {
        // scale rows M..127 of this block's 16-column blocks are padding: zero
        const int nblk = C / 16;
        for (int t = tid; t < (128 - M) * nblk; t += kNT)
            args.s_sf[sf_offset(M + t / nblk, n0 / 16 + t % nblk, args.s_kb_pad)] = 0;
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wamax = fmaxf(wamax, __shfl_xor_sync(0xffffffffu, wamax, o));
        if ((tid & 31) == 0) atomicMax(args.amax_ws, __float_as_uint(wamax));
    }
}

}  // namespace nvfp4
