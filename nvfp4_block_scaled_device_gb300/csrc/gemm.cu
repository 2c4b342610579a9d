// Block-scaled NVFP4 GEMM for sm_103a: tcgen05.mma kind::mxf4nvf4 with
// UE4M3 scales per 16 elements (scale_vec::4X), fp32 accumulation in tensor
// memory, operands staged by TMA into a 4-stage mbarrier ring.
//
// Sources: "CUDA: NVFP4 prefill on Blackwell leaves ~1.45x performance on
// the table" -- NVFP4 tiles fed by TMA with mbarriers and the FP4 MMA
// accumulated in place (item 3); GLU output quantized straight into the next
// GEMM's activation format and gate/up sharing one quantized input (item 2).
// "tp>1 prefill is host-bound" fix direction 1: one launch covers all T rows
// and the grid grows with T.
//
// Tile: 128 rows of A x 256 rows of B per MMA (M=128, N=256, K=64 per
// instruction, 4 instructions per 256-element K stage).  For the SwiGLU
// epilogues the 256 B rows are 128 rows of W_gate followed by the same 128
// rows of W_up, so one MMA produces gate and up for 128 intermediate columns.
//
// Warp roles (320 threads):
//   warp 0      TMA producer (one lane): codes by 2-D TMA, scales by 1-D bulk
//               copies (the 512-byte scale tiles are contiguous along K).
//   warp 1      tensor-memory allocator; one lane issues tcgen05.cp (scales
//               shared -> tensor memory) and tcgen05.mma, and commits.
//   warps 2-9   epilogue: drain the accumulator to registers, release it to
//               the MMA warp, then scale / SwiGLU / requantize / store while
//               the next tile accumulates.
// Persistent: grid = min(#tiles, #SMs); tile t -> (m = t % Mt, n = t / Mt),
// so CTAs running together share the same weight tiles through L2.
#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

namespace {

constexpr int kStages = 4;
constexpr int kABytes = 128 * 128;             // 128 rows x 256 FP4
constexpr int kBHalfBytes = 128 * 128;         // 128 rows x 256 FP4
constexpr int kBBytes = 2 * kBHalfBytes;
constexpr int kSfTile = 512;                   // 128 rows x 4 scales
constexpr int kSfaBytes = 4 * kSfTile;         // 4 K-steps of 64
constexpr int kSfbBytes = 8 * kSfTile;         // 2 row tiles x 4 K-steps
constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;  // 55296
constexpr int kCtrlBytes = 256;
constexpr int kSmemBytes = kStages * kStageBytes + kCtrlBytes + 1024;   // + alignment slack

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kSfColsPerKK = 12;          // 4 (A) + 4 + 4 (two B row tiles)
constexpr uint32_t kSfColsPerStage = 4 * kSfColsPerKK;
static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");

constexpr int kNumThreads = 320;
constexpr int kEpiWarps = 8;

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1 (format 1), UE4M3
// scales (bit 23 = 0), K-major A and B, N = 256 (bits 17-22 = N/8),
// M = 128 (bits 24-28 = M/16), dense, scale-factor ids 0.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((256u >> 3) << 17) | ((128u >> 4) << 24);

#ifdef NVFP4_TRACE
// Debug timeline of CTA 0 (built only with -DNVFP4_TRACE): SM clock at each
// pipeline handoff.  [0,256) producer empty-wait done, [256,512) producer
// issued, [512,768) MMA full-wait done, [768,1024) MMA issued, [1024,1088)
// MMA acc-empty done, [1088,1152) epilogue acc-full done, [1152,1216) drained.
__device__ unsigned long long g_trace[1216];
#define TRACE(slot, i) \
    do { if (blockIdx.x == 0 && (i) < 64 * ((slot) < 1024 ? 4 : 1)) g_trace[(slot) + (i)] = clock64(); } while (0)
#else
#define TRACE(slot, i) do { } while (0)
#endif

struct Ctrl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t teardown;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

// The 12 scale-tile copies of a full stage (A, B rows 0-127, B rows
// 128-255, for each of 4 K-steps), straight-line.
__device__ __forceinline__ void issue_sf4(uint32_t c, uint32_t f, uint32_t hi)
{
    constexpr uint32_t kB0 = kSfaBytes >> 4, kB1 = (kSfaBytes + 4 * kSfTile) >> 4, kT = kSfTile >> 4;
    tmem_copy_sf_warp(c, desc_from(f, hi));
    tmem_copy_sf_warp(c + 4, desc_from(f + kB0, hi));
    tmem_copy_sf_warp(c + 8, desc_from(f + kB1, hi));
    tmem_copy_sf_warp(c + kSfColsPerKK, desc_from(f + kT, hi));
    tmem_copy_sf_warp(c + kSfColsPerKK + 4, desc_from(f + kT + kB0, hi));
    tmem_copy_sf_warp(c + kSfColsPerKK + 8, desc_from(f + kT + kB1, hi));
    tmem_copy_sf_warp(c + 2 * kSfColsPerKK, desc_from(f + 2 * kT, hi));
    tmem_copy_sf_warp(c + 2 * kSfColsPerKK + 4, desc_from(f + 2 * kT + kB0, hi));
    tmem_copy_sf_warp(c + 2 * kSfColsPerKK + 8, desc_from(f + 2 * kT + kB1, hi));
    tmem_copy_sf_warp(c + 3 * kSfColsPerKK, desc_from(f + 3 * kT, hi));
    tmem_copy_sf_warp(c + 3 * kSfColsPerKK + 4, desc_from(f + 3 * kT + kB0, hi));
    tmem_copy_sf_warp(c + 3 * kSfColsPerKK + 8, desc_from(f + 3 * kT + kB1, hi));
}

__device__ __forceinline__ float silu_mul(float gate, float up)
{
    return __fmul_rn(__fdividef(gate, __fadd_rn(1.0f, __expf(-gate))), up);
}

__global__ void __launch_bounds__(kNumThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                const __grid_constant__ CUtensorMap map_b1, const GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + kStages * kStageBytes);
    volatile int* abort_flag = &ctrl->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool swiglu = args.epilogue != kEpiBf16;

    const int64_t num_m = (args.M + 127) / 128;
    const int64_t num_n = swiglu ? args.N / 128 : (args.N + 255) / 256;
    const int64_t num_tiles = num_m * num_n;
    const int num_kk = (int)(args.K / 64);
    const int num_kstages = (num_kk + 3) / 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(smem_u32(&ctrl->full[s]), 1);
            mbar_init(smem_u32(&ctrl->empty[s]), 1);
        }
        mbar_init(smem_u32(&ctrl->acc_full), 1);
        mbar_init(smem_u32(&ctrl->acc_empty), kEpiWarps);
        mbar_init(smem_u32(&ctrl->teardown), 1);
        ctrl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&map_a);
        prefetch_tmap(&map_b0);
        if (swiglu) prefetch_tmap(&map_b1);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        // The whole warp runs the loop; one elected lane issues each copy.
        const uint64_t pol_a = l2_policy_evict_last();
        const uint64_t pol_b = l2_policy_evict_first();
        const uint32_t full0 = smem_u32(&ctrl->full[0]);
        const uint32_t empty0 = smem_u32(&ctrl->empty[0]);
        int s = 0;
        uint32_t ph = 0, issued = 0, issued_ph = 0;
        int kcount = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const int64_t mt = tile % num_m, nt = tile / num_m;
            const int32_t ya = (int32_t)(mt * 128);
            int32_t yb0, yb1;
            const uint8_t *pb0, *pb1;
            bool has_b1;
            if (swiglu) {
                yb0 = yb1 = (int32_t)(nt * 128);
                pb0 = args.sfb0 + nt * args.sfb_tile_stride;
                pb1 = args.sfb1 + nt * args.sfb_tile_stride;
                has_b1 = true;
            } else {
                yb0 = (int32_t)(nt * 256);
                yb1 = yb0 + 128;
                pb0 = args.sfb0 + (2 * nt) * args.sfb_tile_stride;
                pb1 = args.sfb0 + (2 * nt + 1) * args.sfb_tile_stride;
                has_b1 = yb1 < args.N;   // else the scale tile does not exist
            }
            const uint8_t* pa = args.sfa + mt * args.sfa_tile_stride;
            const CUtensorMap* mb1 = swiglu ? &map_b1 : &map_b0;
            const uint32_t tx_full = kABytes + kBHalfBytes * (has_b1 ? 2u : 1u) + 4u * kSfTile * (has_b1 ? 3u : 2u);
            for (int kb = 0; kb < num_kstages; kb++) {
                if (!mbar_wait_warp(empty0 + 8u * (uint32_t)s, ph ^ 1u, abort_flag, args.status, 1)) {
                    ok = false;
                    break;
                }
                if (lane == 0) TRACE(0, kcount);
                // a B half entirely past N is not loaded: its stale shared
                // memory only feeds accumulator columns >= N, never stored
                const bool tail = kb == num_kstages - 1;
                const uint32_t sf_bytes = tail ? (uint32_t)(num_kk - kb * 4) * kSfTile : 4u * kSfTile;
                const uint32_t tx =
                    tail ? kABytes + kBHalfBytes * (has_b1 ? 2u : 1u) + sf_bytes * (has_b1 ? 3u : 2u) : tx_full;
                const uint32_t full = full0 + 8u * (uint32_t)s;
                const uint32_t st = base + (uint32_t)s * kStageBytes;
                const uint32_t sf_st = st + kABytes + kBBytes;
                const int32_t xk = kb * 128;
                mbar_arrive_expect_tx_warp(full, tx);
                if (has_b1) {   // straight-line common case
                    tma_load_2d_warp(st, &map_a, full, xk, ya, pol_a);
                    tma_load_2d_warp(st + kABytes, &map_b0, full, xk, yb0, pol_b);
                    tma_load_2d_warp(st + kABytes + kBHalfBytes, mb1, full, xk, yb1, pol_b);
                    bulk_load_warp(sf_st, pa, sf_bytes, full);
                    bulk_load_warp(sf_st + kSfaBytes, pb0, sf_bytes, full);
                    bulk_load_warp(sf_st + kSfaBytes + 4 * kSfTile, pb1, sf_bytes, full);
                } else {
                    tma_load_2d_warp(st, &map_a, full, xk, ya, pol_a);
                    tma_load_2d_warp(st + kABytes, &map_b0, full, xk, yb0, pol_b);
                    bulk_load_warp(sf_st, pa, sf_bytes, full);
                    bulk_load_warp(sf_st + kSfaBytes, pb0, sf_bytes, full);
                }
                pa += 4 * kSfTile;
                pb0 += 4 * kSfTile;
                pb1 += 4 * kSfTile;
                if (lane == 0) TRACE(256, kcount);
                kcount++;
                issued |= 1u << s;
                issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            // stopped early: let the copies already issued land before the
            // CTA's shared memory goes away (bounded)
            for (int i = 0; i < kStages; i++)
                if (issued & (1u << i)) mbar_wait_teardown(full0 + 8u * (uint32_t)i, (issued_ph >> i) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA
        // The whole warp runs the loop; one elected lane issues the scale
        // copies, the MMAs and the commits (always the same lane, so each
        // commit tracks all MMAs before it).
        // K-major, 128-byte swizzle, 8-row groups 1024 B apart (codes);
        // no swizzle, 16-byte rows, 8-row groups 128 B apart (scales)
        const uint64_t dsw = make_smem_desc(base, 16, 1024, 2);
        const uint64_t dsf = make_smem_desc(base + kABytes + kBBytes, 128, 128, 0);
        const uint32_t desc_a_lo = (uint32_t)dsw, desc_sw_hi = (uint32_t)(dsw >> 32);
        const uint32_t desc_sf_lo = (uint32_t)dsf, desc_sf_hi = (uint32_t)(dsf >> 32);
        const uint32_t full0 = smem_u32(&ctrl->full[0]);
        const uint32_t empty0 = smem_u32(&ctrl->empty[0]);
        int s = 0;
        uint32_t ph = 0, acc_ph = 0;
        bool ok = true;
        int kcount = 0, tcount = 0;
        for (int64_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            if (!mbar_wait_warp(smem_u32(&ctrl->acc_empty), acc_ph ^ 1u, abort_flag, args.status, 2)) break;
            if (lane == 0) TRACE(1024, tcount);
            tcount++;
            tc_fence_after();
            for (int kb = 0; kb < num_kstages; kb++) {
                if (!mbar_wait_warp(full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 3)) {
                    ok = false;
                    break;
                }
                if (lane == 0) TRACE(512, kcount);
                tc_fence_after();
                // descriptors of this stage: only 32-bit adds in the loop
                const uint32_t soff = (uint32_t)s * (kStageBytes >> 4);
                const uint32_t a_lo = desc_a_lo + soff;
                const uint32_t b_lo = a_lo + (kABytes >> 4);
                const uint32_t f_lo = desc_sf_lo + soff;
                const uint32_t sf_stage = tmem + kAccCols + (uint32_t)s * kSfColsPerStage;
                const int nkk = min(4, num_kk - kb * 4);
                const uint32_t acc0 = kb != 0 ? 1u : 0u;
                if (nkk == 4) {
                    // full stage: straight-line issue (no branches between
                    // tcgen05 instructions keeps the tensor pipe fed)
                    issue_sf4(sf_stage, f_lo, desc_sf_hi);
                    mma_mxf4nvf4_warp(tmem, desc_from(a_lo, desc_sw_hi), desc_from(b_lo, desc_sw_hi), kIdesc,
                                      sf_stage, sf_stage + 4, acc0);
                    mma_mxf4nvf4_warp(tmem, desc_from(a_lo + 2u, desc_sw_hi), desc_from(b_lo + 2u, desc_sw_hi),
                                      kIdesc, sf_stage + kSfColsPerKK, sf_stage + kSfColsPerKK + 4, 1u);
                    mma_mxf4nvf4_warp(tmem, desc_from(a_lo + 4u, desc_sw_hi), desc_from(b_lo + 4u, desc_sw_hi),
                                      kIdesc, sf_stage + 2 * kSfColsPerKK, sf_stage + 2 * kSfColsPerKK + 4, 1u);
                    mma_mxf4nvf4_warp(tmem, desc_from(a_lo + 6u, desc_sw_hi), desc_from(b_lo + 6u, desc_sw_hi),
                                      kIdesc, sf_stage + 3 * kSfColsPerKK, sf_stage + 3 * kSfColsPerKK + 4, 1u);
                } else {
                    // K tail: fewer than 4 K-steps
                    for (int kk = 0; kk < nkk; kk++) {
                        const uint32_t c = sf_stage + (uint32_t)kk * kSfColsPerKK;
                        const uint32_t f = f_lo + (uint32_t)kk * (kSfTile >> 4);
                        tmem_copy_sf_warp(c, desc_from(f, desc_sf_hi));
                        tmem_copy_sf_warp(c + 4, desc_from(f + (kSfaBytes >> 4), desc_sf_hi));
                        tmem_copy_sf_warp(c + 8, desc_from(f + ((kSfaBytes + 4 * kSfTile) >> 4), desc_sf_hi));
                    }
                    for (int kk = 0; kk < nkk; kk++) {
                        const uint32_t c = sf_stage + (uint32_t)kk * kSfColsPerKK;
                        mma_mxf4nvf4_warp(tmem, desc_from(a_lo + 2u * kk, desc_sw_hi),
                                          desc_from(b_lo + 2u * kk, desc_sw_hi), kIdesc, c, c + 4,
                                          (kb | kk) != 0 ? 1u : 0u);
                    }
                }
                mma_commit_warp(empty0 + 8u * (uint32_t)s);
                if (lane == 0) TRACE(768, kcount);
                kcount++;
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            mma_commit_warp(smem_u32(&ctrl->acc_full));
            acc_ph ^= 1u;
        }
        // every MMA issued has completed before teardown
        mma_commit_warp(smem_u32(&ctrl->teardown));
        if (lane == 0) mbar_wait_teardown(smem_u32(&ctrl->teardown), 0);
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;             // tensor-memory lane quarter of this warp
        const int h = (warp - 2) >> 2;      // which half of the tile's columns
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        const float ga = *args.ga;
        const float alpha0 = __fmul_rn(ga, *args.gb0);
        const float alpha1 = swiglu ? __fmul_rn(ga, *args.gb1) : alpha0;
        const float g_inter = args.epilogue == kEpiSwigluFp4 ? *args.g_inter : 1.0f;
        uint32_t acc_ph = 0;
        float wamax = 0.0f;
        int ecount = 0;
        for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int64_t mt = tile % num_m, nt = tile / num_m;
            // one lane waits; the warp then proceeds converged (tcgen05.ld is warp-wide)
            int ok = 1;
            if (lane == 0) ok = mbar_wait<true>(smem_u32(&ctrl->acc_full), acc_ph, abort_flag, args.status, 4) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            if (!ok) break;
            if (warp == 2 && lane == 0) TRACE(1088, ecount);
            tc_fence_after();
            float v[128];
            if (!swiglu) {
                tmem_ld32(lane_addr + h * 128 + 0, v + 0);
                tmem_ld32(lane_addr + h * 128 + 32, v + 32);
                tmem_ld32(lane_addr + h * 128 + 64, v + 64);
                tmem_ld32(lane_addr + h * 128 + 96, v + 96);
            } else {
                tmem_ld32(lane_addr + h * 64 + 0, v + 0);
                tmem_ld32(lane_addr + h * 64 + 32, v + 32);
                tmem_ld32(lane_addr + 128 + h * 64 + 0, v + 64);
                tmem_ld32(lane_addr + 128 + h * 64 + 32, v + 96);
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctrl->acc_empty));
            if (warp == 2 && lane == 0) TRACE(1152, ecount);
            ecount++;
            acc_ph ^= 1u;

            const int64_t row = mt * 128 + q * 32 + lane;
            if (!swiglu) {
                if (row < args.M) {
                    const int64_t n_base = nt * 256 + h * 128;
                    __nv_bfloat16* orow = args.out + row * args.ldo;
                    const __nv_bfloat16* rrow = args.residual ? args.residual + row * args.ldr : nullptr;
#pragma unroll
                    for (int j = 0; j < 128; j += 8) {
                        const int64_t n = n_base + j;
                        if (n < args.N) {
                            float y[8];
#pragma unroll
                            for (int i = 0; i < 8; i++) y[i] = bf16_round(__fmul_rn(v[j + i], alpha0));
                            if (rrow) {
                                const uint4 rp = *reinterpret_cast<const uint4*>(rrow + n);
                                y[0] = __fadd_rn(bf16_lo(rp.x), y[0]);
                                y[1] = __fadd_rn(bf16_hi(rp.x), y[1]);
                                y[2] = __fadd_rn(bf16_lo(rp.y), y[2]);
                                y[3] = __fadd_rn(bf16_hi(rp.y), y[3]);
                                y[4] = __fadd_rn(bf16_lo(rp.z), y[4]);
                                y[5] = __fadd_rn(bf16_hi(rp.z), y[5]);
                                y[6] = __fadd_rn(bf16_lo(rp.w), y[6]);
                                y[7] = __fadd_rn(bf16_hi(rp.w), y[7]);
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
        if (args.epilogue == kEpiSwigluBf16) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wamax = fmaxf(wamax, __shfl_xor_sync(0xffffffffu, wamax, o));
            if (lane == 0) atomicMax(args.amax_ws, __float_as_uint(wamax));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t gemm_smem_bytes() { return kSmemBytes; }

cudaError_t launch_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b0, const CUtensorMap& map_b1,
                        const GemmArgs& args, int num_sms, cudaStream_t stream)
{
    static int attr_set_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set_for_device[dev]) {
        e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    const bool swiglu = args.epilogue != kEpiBf16;
    const int64_t num_m = (args.M + 127) / 128;
    const int64_t num_n = swiglu ? args.N / 128 : (args.N + 255) / 256;
    const int64_t tiles = num_m * num_n;
    const unsigned grid = (unsigned)(tiles < num_sms ? tiles : num_sms);
    gemm_kernel<<<grid, kNumThreads, kSmemBytes, stream>>>(map_a, map_b0, map_b1, args);
    return cudaGetLastError();
}

}  // namespace nvfp4

#ifdef NVFP4_TRACE
extern "C" int nvfp4_debug_trace(unsigned long long* out, int n)
{
    if (n > 1216) n = 1216;
    return cudaMemcpyFromSymbol(out, nvfp4::g_trace, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : 4;
}
#endif
