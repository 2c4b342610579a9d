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

// Rotary embedding of a row's bf16 outputs, pair by pair from an even
// column: a cursor holds the rotated-head index and the column within the
// head, so that no division runs per pair.  Each step rotates the pair
// (e, o) at the cursor if it lies in the last rope_rd columns of a rotated
// head, in binary32 steps on the bf16-rounded outputs:
//   forward: e' = e*c - o*s, o' = e*s + o*c; inverse: e' = e*c + o*s, o' = o*c - e*s
// ("PERFORMANCE -- verified hot-path audit" P5, RoPE fused into the Q/KV
// projection's epilogue), then advances two columns.
struct RopeCursor {
    int32_t head;     // rotated-head index of the cursor column (outside [0, heads): none)
    int32_t within;   // cursor column within its head (even)
    const float* c;   // the cos / sin table row of the row's position
    const float* s;
};

__device__ __forceinline__ RopeCursor rope_begin(const GemmArgs& a, int64_t row, int64_t n)
{
    RopeCursor k;
    const int64_t rel = n - a.rope_col0;
    const int64_t head = rel >= 0 ? rel / a.rope_hd : -((-rel + a.rope_hd - 1) / a.rope_hd);
    k.head = (int32_t)head;
    k.within = (int32_t)(rel - head * a.rope_hd);
    const int64_t p = a.rope_pos[row];
    k.c = a.rope_cos + p * a.rope_ld;
    k.s = a.rope_sin + p * a.rope_ld;
    return k;
}

__device__ __forceinline__ void rope_step(const GemmArgs& a, RopeCursor& k, float& e, float& o)
{
    const int32_t hd = (int32_t)a.rope_hd, nope = (int32_t)(a.rope_hd - a.rope_rd);
    if (k.head >= 0 && k.head < a.rope_heads && k.within >= nope) {
        const int32_t i = (k.within - nope) >> 1;
        const float c = __ldg(k.c + i), s = __ldg(k.s + i);
        const float ec = __fmul_rn(e, c), os = __fmul_rn(o, s), es = __fmul_rn(e, s), oc = __fmul_rn(o, c);
        if (a.rope_inverse) {
            e = __fadd_rn(ec, os);
            o = __fsub_rn(oc, es);
        } else {
            e = __fsub_rn(ec, os);
            o = __fadd_rn(es, oc);
        }
    }
    k.within += 2;
    if (k.within >= hd) {
        k.within -= hd;
        ++k.head;
    }
}

// bf16 output rows can go out through a per-warp shared-memory staging area
// of kStageRows rows (4 or 8, as the kernel's shared memory allows): a thread
// holds one row's 128 columns, so storing them straight from registers makes
// every warp store touch 32 rows; staged, each warp store writes two whole
// 256-byte row segments.
constexpr int kEpiStageRowBytes = 256 + 16;            // padded: the staged rows' 16-byte chunks hit distinct banks
__host__ __device__ constexpr int epi_stage_bytes(int stage_rows) { return stage_rows * kEpiStageRowBytes; }   // per epilogue warp
constexpr int kEpiStageBytes = epi_stage_bytes(4);

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// v: this thread's accumulator values; row: its output row (warp-converged
// call: every lane of the warp, rows >= M included); stage: this warp's
// epi_stage_bytes(kStageRows) of shared memory (shared-space address), or 0
// for the direct bf16 stores (fewer steps: for a tile of few rows).
// kRope: the rotary embedding of the bf16 output (args.rope_*) is compiled
// in; the kernels run that instantiation only for a call that asks for it,
// so the others carry none of its code or registers.
template <bool kRope, int kStageRows = 4>
__device__ __forceinline__ void epilogue_row(const GemmArgs& args, bool swiglu, float (&v)[128], int64_t row,
                                             int64_t nt, int h, float alpha0, float alpha1, float g_inter,
                                             float& wamax, uint32_t stage)
{
    if (!swiglu && stage == 0u) {
        // direct: each thread stores its own row; four 16-byte vectors per
        // batch, the batch's residual loads issued before its stores (an
        // output aliasing the residual element for element is read by the
        // thread that then overwrites it)
        if (row < args.M) {
            const int64_t n_base = nt * 256 + h * 128;
            __nv_bfloat16* orow = args.out + row * args.ldo;
            const __nv_bfloat16* rrow = args.residual ? args.residual + row * args.ldr : nullptr;
            RopeCursor rk{};
            if (kRope) rk = rope_begin(args, row, n_base);
#pragma unroll
            for (int jb = 0; jb < 128; jb += 32) {
                uint4 rp[4];
#pragma unroll
                for (int t = 0; t < 4; t++) {
                    const int64_t n = n_base + jb + 8 * t;
                    rp[t] = (rrow && n < args.N) ? *reinterpret_cast<const uint4*>(rrow + n) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int t = 0; t < 4; t++) {
                    const int j = jb + 8 * t;
                    const int64_t n = n_base + j;
                    uint4 o;
                    if (kRope) {
                        // rotated in binary32 from the rounded values, then
                        // rounded (the rotation has no residual)
                        float y[8];
#pragma unroll
                        for (int i = 0; i < 8; i++) y[i] = bf16_round(__fmul_rn(v[j + i], alpha0));
#pragma unroll
                        for (int q = 0; q < 4; q++) rope_step(args, rk, y[2 * q], y[2 * q + 1]);
                        o.x = pack_bf16x2(y[0], y[1]);
                        o.y = pack_bf16x2(y[2], y[3]);
                        o.z = pack_bf16x2(y[4], y[5]);
                        o.w = pack_bf16x2(y[6], y[7]);
                    } else {
                        o.x = cvt_bf16x2(__fmul_rn(v[j], alpha0), __fmul_rn(v[j + 1], alpha0));
                        o.y = cvt_bf16x2(__fmul_rn(v[j + 2], alpha0), __fmul_rn(v[j + 3], alpha0));
                        o.z = cvt_bf16x2(__fmul_rn(v[j + 4], alpha0), __fmul_rn(v[j + 5], alpha0));
                        o.w = cvt_bf16x2(__fmul_rn(v[j + 6], alpha0), __fmul_rn(v[j + 7], alpha0));
                    }
                    if (n < args.N) {
                        if (rrow) {
                            // out = bf16(residual + bf16(alpha * acc))
                            o.x = add_bf16x2(rp[t].x, o.x);
                            o.y = add_bf16x2(rp[t].y, o.y);
                            o.z = add_bf16x2(rp[t].z, o.z);
                            o.w = add_bf16x2(rp[t].w, o.w);
                        }
                        *reinterpret_cast<uint4*>(orow + n) = o;
                    }
                }
            }
        }
    } else if (!swiglu) {
        // staged: t = bf16(alpha * acc) of this lane's row (rotated), packed
        const int64_t n_base = nt * 256 + h * 128;
        uint32_t pk[64];
        if (kRope && row < args.M) {
            RopeCursor rk = rope_begin(args, row, n_base);
#pragma unroll
            for (int i = 0; i < 64; i++) {
                float e = bf16_round(__fmul_rn(v[2 * i], alpha0)), o = bf16_round(__fmul_rn(v[2 * i + 1], alpha0));
                rope_step(args, rk, e, o);
                pk[i] = pack_bf16x2(e, o);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 64; i++) pk[i] = cvt_bf16x2(__fmul_rn(v[2 * i], alpha0), __fmul_rn(v[2 * i + 1], alpha0));
        }
        const int lane = threadIdx.x & 31;
        const int64_t row0 = row - lane;                 // the warp's first row
        const int c = lane & 15;                         // 16-byte chunk (8 columns) of a staged row
        const int64_t n = n_base + 8 * c;
        static_assert(kStageRows == 4 || kStageRows == 8, "staging rows");
        constexpr int kRounds = 32 / kStageRows;
        constexpr int kPerRound = kStageRows / 2;         // chunks a lane stores per round
        constexpr int kAhead = kStageRows == 4 ? 3 : 1;   // rounds of residual loads in flight
        // this lane's output chunk (round r, part hh): row
        // row0 + kStageRows * r + 2 * hh + lane / 16, columns n .. n + 7.
        // Residual loads run kAhead rounds ahead of the stores (an output
        // aliasing the residual element for element is read by the thread
        // that later overwrites it, before it does).
        auto chunk_row = [&](int r, int hh) { return row0 + kStageRows * r + 2 * hh + (lane >> 4); };
        auto load_res = [&](int r, int hh) {
            const int64_t orow = chunk_row(r, hh);
            return (args.residual && orow < args.M && n < args.N)
                       ? *reinterpret_cast<const uint4*>(args.residual + orow * args.ldr + n)
                       : make_uint4(0, 0, 0, 0);
        };
        uint4 rp[kAhead * kPerRound];
#pragma unroll
        for (int i = 0; i < kAhead * kPerRound; i++) rp[i] = load_res(i / kPerRound, i % kPerRound);
#pragma unroll
        for (int r = 0; r < kRounds; r++) {
            if ((lane / kStageRows) == r) {
                const uint32_t dst = stage + (uint32_t)(lane % kStageRows) * kEpiStageRowBytes;
#pragma unroll
                for (int j = 0; j < 16; j++)
                    st_shared_v4(dst + 16u * j, make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]));
            }
            __syncwarp();
#pragma unroll
            for (int hh = 0; hh < kPerRound; hh++) {
                const int rr = 2 * hh + (lane >> 4);      // staged row of this lane's chunk
                const int64_t orow = chunk_row(r, hh);
                const uint4 t = ld_shared_v4(stage + (uint32_t)rr * kEpiStageRowBytes + 16u * c);
                const int slot = (r % kAhead) * kPerRound + hh;
                if (orow < args.M && n < args.N) {
                    uint4 o = t;
                    if (args.residual) {
                        // out = bf16(residual + t)
                        const uint4 q = rp[slot];
                        o.x = add_bf16x2(q.x, t.x);
                        o.y = add_bf16x2(q.y, t.y);
                        o.z = add_bf16x2(q.z, t.z);
                        o.w = add_bf16x2(q.w, t.w);
                    }
                    *reinterpret_cast<uint4*>(args.out + orow * args.ldo + n) = o;
                }
                if (r + kAhead < kRounds) rp[slot] = load_res(r + kAhead, hh);
            }
            __syncwarp();
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
