// The epilogue of one accumulator row, shared by the 1-SM and 2-SM GEMM
// kernels: scale, round and store (bf16, optional residual), or SwiGLU and
// FP4 requantization / bf16 store with amax (SwiGLU epilogues).
//   v[0..127]: this thread's accumulator values (bf16 epilogue: output
//   columns nt*256 + h*128 + j; SwiGLU: v[0..63] gate and v[64..127] up of
//   intermediate columns nt*128 + h*64 + j), row: output row of this thread.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

__device__ __forceinline__ float silu_mul(float gate, float up)
{
    return __fmul_rn(__fdividef(gate, __fadd_rn(1.0f, __expf(-gate))), up);
}

__device__ __forceinline__ void epilogue_row(const GemmArgs& args, bool swiglu, float (&v)[128], int64_t row,
                                             int64_t nt, int h, float alpha0, float alpha1, float g_inter,
                                             float& wamax)
{
    if (!swiglu) {
        if (row < args.M) {
            const int64_t n_base = nt * 256 + h * 128;
            __nv_bfloat16* orow = args.out + row * args.ldo;
            const __nv_bfloat16* rrow = args.residual ? args.residual + row * args.ldr : nullptr;
            // Eight 16-byte vectors per batch: the batch's residual loads are
            // all issued before its stores.  The output may alias the
            // residual only element for element (same pitch), and each
            // thread reads exactly the residual elements it then overwrites,
            // so the early loads see the values the stores replace.
#pragma unroll
            for (int jb = 0; jb < 128; jb += 64) {
                uint4 rp[8];
#pragma unroll
                for (int t = 0; t < 8; t++) {
                    const int64_t n = n_base + jb + 8 * t;
                    rp[t] = (rrow && n < args.N) ? *reinterpret_cast<const uint4*>(rrow + n) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int t = 0; t < 8; t++) {
                    const int j = jb + 8 * t;
                    const int64_t n = n_base + j;
                    if (n < args.N) {
                        float y[8];
#pragma unroll
                        for (int i = 0; i < 8; i++) y[i] = bf16_round(__fmul_rn(v[j + i], alpha0));
                        if (rrow) {
                            y[0] = __fadd_rn(bf16_lo(rp[t].x), y[0]);
                            y[1] = __fadd_rn(bf16_hi(rp[t].x), y[1]);
                            y[2] = __fadd_rn(bf16_lo(rp[t].y), y[2]);
                            y[3] = __fadd_rn(bf16_hi(rp[t].y), y[3]);
                            y[4] = __fadd_rn(bf16_lo(rp[t].z), y[4]);
                            y[5] = __fadd_rn(bf16_hi(rp[t].z), y[5]);
                            y[6] = __fadd_rn(bf16_lo(rp[t].w), y[6]);
                            y[7] = __fadd_rn(bf16_hi(rp[t].w), y[7]);
                        }
                        uint4 o;
                        o.x = pack_bf16x2(y[0], y[1]);
                        o.y = pack_bf16x2(y[2], y[3]);
                        o.z = pack_bf16x2(y[4], y[5]);
                        o.w = pack_bf16x2(y[6], y[7]);
                        *reinterpret_cast<uint4*>(orow + n) = o;
                    }
                }
            }
        }
    } else {
        const int64_t col0 = nt * 128 + h * 64;   // intermediate column of v[0]
        if (row < args.M) {
            // s = bf16( silu(gate) * up ), gate/up rounded to bf16 first
#pragma unroll
            for (int i = 0; i < 64; i++) {
                const float gate = bf16_round(__fmul_rn(v[i], alpha0));
                const float up = bf16_round(__fmul_rn(v[64 + i], alpha1));
                v[i] = bf16_round(silu_mul(gate, up));
            }
            if (args.s_bf16) {
                __nv_bfloat16* srow = args.s_bf16 + row * args.ld_s + col0;
#pragma unroll
                for (int j = 0; j < 64; j += 8) {
                    uint4 o;
                    o.x = pack_bf16x2(v[j + 0], v[j + 1]);
                    o.y = pack_bf16x2(v[j + 2], v[j + 3]);
                    o.z = pack_bf16x2(v[j + 4], v[j + 5]);
                    o.w = pack_bf16x2(v[j + 6], v[j + 7]);
                    *reinterpret_cast<uint4*>(srow + j) = o;
                }
            }
            if (args.epilogue == kEpiSwigluFp4) {
                uint32_t cw[8];
                uint32_t scw = 0;
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    float a = 0.0f;
#pragma unroll
                    for (int i = 0; i < 16; i++) a = fmaxf(a, fabsf(v[16 * b + i]));
                    uint32_t sc;
                    cw[2 * b] = quant_half_block(v + 16 * b, g_inter, a, &sc);
                    cw[2 * b + 1] = quant_half_block(v + 16 * b + 8, g_inter, a, &sc);
                    scw |= sc << (8 * b);
                }
                uint8_t* crow = args.s_codes + row * args.ld_s_codes + col0 / 2;
                *reinterpret_cast<uint4*>(crow) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                *reinterpret_cast<uint4*>(crow + 16) = make_uint4(cw[4], cw[5], cw[6], cw[7]);
                *reinterpret_cast<uint32_t*>(args.s_sf + sf_offset(row, col0 / 16, args.s_kb_pad)) = scw;
            } else {
#pragma unroll
                for (int i = 0; i < 64; i++) wamax = fmaxf(wamax, fabsf(v[i]));
            }
        } else if (args.epilogue == kEpiSwigluFp4) {
            // rows past M inside the last 128-row tile: zero scale padding
            *reinterpret_cast<uint32_t*>(args.s_sf + sf_offset(row, col0 / 16, args.s_kb_pad)) = 0u;
        }
    }
}

}  // namespace nvfp4
