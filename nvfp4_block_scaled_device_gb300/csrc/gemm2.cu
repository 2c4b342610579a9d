// Block-scaled NVFP4 GEMM on SM pairs (sm_103a): tcgen05.mma.cta_group::2
// kind::mxf4nvf4 with UE4M3 scales per 16 elements, M = 256 rows per
// instruction split over the two SMs of a cluster of 2, N = 256, K = 64.
//
// Sources: as the 1-SM kernel ("CUDA: NVFP4 prefill on Blackwell leaves
// ~1.45x performance on the table", items 2 and 3; "tp>1 prefill is
// host-bound", fix direction 1).
//
// Why pairs: each SM holds its own 128 rows of A but only half of the 256 B
// rows; the pair's tensor cores share the B halves.  Per SM and per K step
// the operand bytes drop from 12 KB (1-SM, 128x256) to 8 KB for the same
// work, and one issued instruction covers twice the work.
//
// Each CTA of the pair loads, into its own shared memory: its 128 rows of A
// and their scales, its 128-row half of B (rows 0-127 in the even CTA, rows
// 128-255 in the odd one; for SwiGLU the W_gate and the W_up rows), and the
// scales of all 256 B rows.  The even CTA ("leader") issues the scale copies
// and MMAs for both CTAs once both halves of a stage have landed: the odd
// CTA's otherwise idle MMA warp relays "stage landed" to the leader by a
// remote mbarrier arrive.  The leader's commits are multicast to both CTAs
// (stage free, accumulator ready); both CTAs' epilogue warps arrive on the
// leader's accumulator-free barrier.  Each CTA's epilogue reads its own
// tensor memory (its 128 rows of the 256-row tile).
#include "common.cuh"
#include "gemm_epilogue.cuh"
#include "internal.h"

namespace nvfp4 {

namespace {

constexpr int kStages = 5;
constexpr int kABytes = 128 * 128;             // own 128 rows x 256 FP4
constexpr int kBBytes = 128 * 128;             // own 128-row half of B
constexpr int kSfTile = 512;                   // 128 rows x 4 scales
constexpr int kSfaBytes = 4 * kSfTile;         // own rows, 4 K-steps of 64
constexpr int kSfbBytes = 8 * kSfTile;         // both 128-row halves of B, 4 K-steps
constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;  // 38912
constexpr int kCtrlBytes = 256;
constexpr int kSmemBytes = kStages * kStageBytes + kCtrlBytes + 1024;
static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment (128-byte swizzle atoms)");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kSfColsPerKK = 12;          // 4 (A) + 8 (B: two 128-row halves)
constexpr uint32_t kSfColsPerStage = 4 * kSfColsPerKK;
static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");

// Warp roles (16 warps, 4 warpgroups): warps 0-3 and 5-7 are copy
// producers (each a separate copy stream), warp 4 the MMA warp (leader) or
// the stage relay (odd CTA), warps 8-15 the epilogue.  Launched at 128
// registers per thread; warpgroups 0-1 drop to 56 and 2-3 rise to 200.
constexpr int kProducers = 7;
constexpr int kMmaWarp = 4;
constexpr int kEpiWarp0 = 8;
constexpr int kEpiWarps = 8;
constexpr int kNumThreads = 512;
constexpr uint32_t kRegsSmall = 56;
constexpr uint32_t kRegsEpi = 200;
static_assert(2 * kRegsSmall + 2 * kRegsEpi == 512, "register split per sub-partition");
constexpr uint16_t kPairMask = 0x3;            // both CTAs of the cluster

// Instruction descriptor, kind::mxf4nvf4: E2M1 A and B (format 1), UE4M3
// scales, K-major, N = 256 (bits 17-22 = N/8), M = 256 (bits 24-28 = M/16).
constexpr uint32_t kIdesc2 = (1u << 7) | (1u << 10) | ((256u >> 3) << 17) | ((256u >> 4) << 24);

#ifdef NVFP4_TRACE
// Debug timeline of the first CTA pair (built only with -DNVFP4_TRACE),
// %globaltimer ns: [0,256) leader stage-free seen, [256,512) leader issued,
// [512,768) odd stage-free seen, [768,1024) odd issued, [1024,1280) leader
// own-full seen, [1280,1536) leader peer-full seen, [1536,1792) leader MMAs
// issued, [1792,2048) odd relay sent.
__device__ unsigned long long g_trace2[2048];
#define TRACE2(slot, i)                                                 \
    do {                                                                \
        if (blockIdx.x < 2 && (i) < 256) g_trace2[(slot) + (i)] = globaltimer(); \
    } while (0)
#else
#define TRACE2(slot, i) do { } while (0)
#endif

struct Ctrl {
    uint64_t full[kStages];       // this CTA's loads of the stage landed
    uint64_t peer_full[kStages];  // (leader) the odd CTA's loads of the stage landed
    uint64_t empty[kStages];      // the pair's MMAs finished reading the stage
    uint64_t acc_full;            // the tile's accumulator is complete
    uint64_t acc_empty;           // (leader) both CTAs' epilogues drained the accumulator
    uint64_t teardown;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kNumThreads, 1)
    gemm2_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
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
    const uint32_t rank = cluster_ctarank();   // 0: leader (issues the pair's MMAs)
    const bool leader = rank == 0;
    const bool swiglu = args.epilogue != kEpiBf16;

    const int64_t num_m = (args.M + 255) / 256;
    const int64_t num_n = swiglu ? args.N / 128 : (args.N + 255) / 256;
    const int64_t num_tiles = num_m * num_n;
    const int64_t pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
    const int num_kk = (int)(args.K / 64);
    const int num_kstages = (num_kk + 3) / 4;
    const int full_kstages = num_kk / 4;       // stages of 4 K-steps
    const int tail_kk = num_kk % 4;            // K-steps of a last, partial stage

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(smem_u32(&ctrl->full[s]), kProducers);
            mbar_init(smem_u32(&ctrl->peer_full[s]), 1);
            mbar_init(smem_u32(&ctrl->empty[s]), 1);
        }
        mbar_init(smem_u32(&ctrl->acc_full), 1);
        mbar_init(smem_u32(&ctrl->acc_empty), 2 * kEpiWarps);
        mbar_init(smem_u32(&ctrl->teardown), 1);
        ctrl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&map_a);
        prefetch_tmap(&map_b0);
        if (swiglu) prefetch_tmap(&map_b1);
    }
    if (warp == kMmaWarp) {
        tmem_alloc2(smem_u32(&ctrl->tmem_base), kTmemCols);
        tmem_relinquish2();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // both CTAs' barriers are initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;

    if (warp < kEpiWarp0) {
        // warpgroups 0-1: one register-budget instruction for all eight warps
        setmaxnreg_dec<kRegsSmall>();
        if (warp != kMmaWarp) {
            // ------------------------------------------------------ producers
            // Seven warps, one lane each, share every stage's copies (copies
            // issued by one thread are served one after the other): producers
            // 0-3 fetch the 64-row code boxes (this CTA's A rows 0-63, 64-127, its
            // B half's rows 0-63, 64-127), producers 4-6 the scale tiles (A, B
            // rows 0-127, B rows 128-255).  Each arrives once per stage on its
            // CTA's full barrier with its own byte count.  Boxes past the
            // operand's rows are not fetched: their stale shared memory only
            // feeds accumulator rows >= M or columns >= N.
            const int p = warp < kMmaWarp ? warp : warp - 1;
            const uint32_t full0 = smem_u32(&ctrl->full[0]);
            const uint32_t empty0 = smem_u32(&ctrl->empty[0]);
            constexpr uint32_t kBox = kCodeBoxRows * 128u;
            const uint64_t pol = p < 2 ? l2_policy_evict_last() : l2_policy_evict_first();
            const uint32_t my_off = (uint32_t)p * kBox;     // A then the B half, contiguous
            int s = 0;
            uint32_t ph = 0, issued = 0, issued_ph = 0;
            bool ok = true;
            int kcount = 0;
            for (int64_t tile = pair; tile < num_tiles && ok; tile += num_pairs) {
                const int64_t mt = tile % num_m, nt = tile / num_m;
                const int64_t row0 = mt * 256 + rank * 128;          // this CTA's first A row
                const bool has_a = row0 < args.M;                    // else its rows (and scale tile) do not exist
                int32_t yb;
                const CUtensorMap* mb;
                const uint8_t *pb0, *pb1;
                bool has_b1;
                if (swiglu) {
                    yb = (int32_t)(nt * 128);
                    mb = rank ? &map_b1 : &map_b0;
                    pb0 = args.sfb0 + nt * args.sfb_tile_stride;
                    pb1 = args.sfb1 + nt * args.sfb_tile_stride;
                    has_b1 = true;
                } else {
                    yb = (int32_t)(nt * 256 + rank * 128);
                    mb = &map_b0;
                    pb0 = args.sfb0 + (2 * nt) * args.sfb_tile_stride;
                    pb1 = args.sfb0 + (2 * nt + 1) * args.sfb_tile_stride;
                    has_b1 = nt * 256 + 128 < args.N;               // the second B scale tile exists
                }
                const CUtensorMap* my_map = p < 2 ? &map_a : mb;
                const int32_t my_y = (p < 2 ? (int32_t)row0 : yb) + (p & 1) * kCodeBoxRows;
                const bool my_box = p < 4 && my_y < (p < 2 ? args.M : args.N);
                const bool my_sf = p == 4 ? has_a : p == 5 ? true : p == 6 ? has_b1 : false;
                const uint8_t* my_sf_src = p == 4 ? args.sfa + (row0 / 128) * args.sfa_tile_stride : p == 5 ? pb0 : pb1;
                const uint32_t my_sf_off = kABytes + kBBytes + (p == 4 ? 0u : p == 5 ? (uint32_t)kSfaBytes
                                                                                      : (uint32_t)(kSfaBytes + 4 * kSfTile));
                for (int kb = 0; kb < num_kstages; kb++) {
                    if (!mbar_wait_cluster_warp(empty0 + 8u * (uint32_t)s, ph ^ 1u, abort_flag, args.status, 11)) {
                        ok = false;
                        break;
                    }
                    if (p == 0 && lane == 0) TRACE2(rank * 512, kcount);
                    const uint32_t sf_bytes = (uint32_t)min(4, num_kk - kb * 4) * kSfTile;
                    const uint32_t tx = my_box ? kBox : my_sf ? sf_bytes : 0u;
                    const uint32_t full = full0 + 8u * (uint32_t)s;
                    const uint32_t st = base + (uint32_t)s * kStageBytes;
                    const int32_t xk = kb * 128;
                    if (lane == 0) {
                        if (tx == 0) {
                            mbar_arrive(full);
                        } else {
                            mbar_arrive_expect_tx(full, tx);
                            if (my_box) tma_load_2d(st + my_off, my_map, full, xk, my_y, pol);
                            else bulk_load(st + my_sf_off, my_sf_src + (size_t)kb * (4 * kSfTile), sf_bytes, full);
                        }
                    }
                    __syncwarp();
                    if (p == 0 && lane == 0) TRACE2(rank * 512 + 256, kcount);
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
                for (int i = 0; i < kStages; i++)
                    if (issued & (1u << i)) mbar_wait_teardown(full0 + 8u * (uint32_t)i, (issued_ph >> i) & 1u);
            }
            __syncwarp();
        } else {
            const uint32_t full0 = smem_u32(&ctrl->full[0]);
            const uint32_t peer_full0 = smem_u32(&ctrl->peer_full[0]);
            const uint32_t empty0 = smem_u32(&ctrl->empty[0]);
            if (leader) {
                // ----------------------------------------------- MMA (pair)
                const uint64_t dsw = make_smem_desc(base, 16, 1024, 2);
                const uint64_t dsf = make_smem_desc(base + kABytes + kBBytes, 128, 128, 0);
                const uint32_t desc_a_lo = (uint32_t)dsw, desc_sw_hi = (uint32_t)(dsw >> 32);
                const uint32_t desc_sf_lo = (uint32_t)dsf, desc_sf_hi = (uint32_t)(dsf >> 32);
                int s = 0;
                uint32_t ph = 0, acc_ph = 0;
                bool ok = true;
                int kcount = 0;
                for (int64_t tile = pair; tile < num_tiles && ok; tile += num_pairs) {
                    if (!mbar_wait_cluster_warp(smem_u32(&ctrl->acc_empty), acc_ph ^ 1u, abort_flag, args.status, 12))
                        break;
                    tc_fence_after();
                    // full stages: nothing but the waits and one fused issue block
                    for (int kb = 0; kb < full_kstages; kb++) {
                        if (!mbar_wait_warp(full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 13) ||
                            !mbar_wait_cluster_warp(peer_full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 14)) {
                            ok = false;
                            break;
                        }
                        TRACE2(1280, kcount);
                        tc_fence_after();
                        const uint32_t soff = (uint32_t)s * (kStageBytes >> 4);
                        const uint32_t a_lo = desc_a_lo + soff;
                        stage_issue_2sm(tmem, tmem + kAccCols + (uint32_t)s * kSfColsPerStage, desc_sf_lo + soff,
                                        desc_sf_hi, a_lo, a_lo + (kABytes >> 4), desc_sw_hi, kIdesc2,
                                        kb != 0 ? 1u : 0u, empty0 + 8u * (uint32_t)s, kPairMask);
                        TRACE2(1536, kcount);
                        kcount++;
                        if (++s == kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (ok && tail_kk != 0) {
                        // K tail: a last stage of fewer than 4 K-steps
                        if (!mbar_wait_warp(full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 13) ||
                            !mbar_wait_cluster_warp(peer_full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 14)) {
                            ok = false;
                        } else {
                            tc_fence_after();
                            const uint32_t soff = (uint32_t)s * (kStageBytes >> 4);
                            const uint32_t a_lo = desc_a_lo + soff;
                            const uint32_t b_lo = a_lo + (kABytes >> 4);
                            const uint32_t f_lo = desc_sf_lo + soff;
                            const uint32_t sf_stage = tmem + kAccCols + (uint32_t)s * kSfColsPerStage;
                            for (int kk = 0; kk < tail_kk; kk++) {
                                const uint32_t c = sf_stage + (uint32_t)kk * kSfColsPerKK;
                                const uint32_t f = f_lo + (uint32_t)kk * (kSfTile >> 4);
                                tmem_copy_sf2_warp(c, desc_from(f, desc_sf_hi));
                                tmem_copy_sf2_warp(c + 4, desc_from(f + (kSfaBytes >> 4), desc_sf_hi));
                                tmem_copy_sf2_warp(c + 8, desc_from(f + ((kSfaBytes + 4 * kSfTile) >> 4), desc_sf_hi));
                            }
                            for (int kk = 0; kk < tail_kk; kk++) {
                                const uint32_t c = sf_stage + (uint32_t)kk * kSfColsPerKK;
                                mma2_mxf4nvf4_warp(tmem, desc_from(a_lo + 2u * kk, desc_sw_hi),
                                                   desc_from(b_lo + 2u * kk, desc_sw_hi), kIdesc2, c, c + 4,
                                                   (full_kstages | kk) != 0 ? 1u : 0u);
                            }
                            // the stage is free in both CTAs once these MMAs complete
                            mma_commit2_mc_warp(empty0 + 8u * (uint32_t)s, kPairMask);
                            kcount++;
                            if (++s == kStages) {
                                s = 0;
                                ph ^= 1u;
                            }
                        }
                    }
                    if (!ok) break;
                    mma_commit2_mc_warp(smem_u32(&ctrl->acc_full), kPairMask);
                    acc_ph ^= 1u;
                }
                // every MMA issued has completed before teardown
                mma_commit2_mc_warp(smem_u32(&ctrl->teardown), 0x1);
                if (lane == 0) mbar_wait_teardown(smem_u32(&ctrl->teardown), 0);
                __syncwarp();
            } else {
                // ------------------------------ relay (odd CTA): stage landed
                const uint32_t leader_peer_full0 = map_to_cta(peer_full0, 0);
                int s = 0;
                uint32_t ph = 0;
                bool ok = true;
                int kcount = 0;
                for (int64_t tile = pair; tile < num_tiles && ok; tile += num_pairs) {
                    for (int kb = 0; kb < num_kstages; kb++) {
                        if (!mbar_wait_warp(full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 15)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) mbar_arrive_remote(leader_peer_full0 + 8u * (uint32_t)s);
                        if (lane == 0 && kcount < 8) TRACE2(1792, kcount);
                        kcount++;
                        __syncwarp();
                        if (++s == kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        setmaxnreg_inc<kRegsEpi>();                        // warpgroups 2-3
        const int q = warp & 3;             // tensor-memory lane quarter of this warp
        const int h = (warp - kEpiWarp0) >> 2;   // which half of the tile's columns
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        const uint32_t acc_empty_leader = map_to_cta(smem_u32(&ctrl->acc_empty), 0);
        const float ga = *args.ga;
        const float alpha0 = __fmul_rn(ga, *args.gb0);
        const float alpha1 = swiglu ? __fmul_rn(ga, *args.gb1) : alpha0;
        const float g_inter = args.epilogue == kEpiSwigluFp4 ? *args.g_inter : 1.0f;
        uint32_t acc_ph = 0;
        float wamax = 0.0f;
        for (int64_t tile = pair; tile < num_tiles; tile += num_pairs) {
            const int64_t mt = tile % num_m, nt = tile / num_m;
            if (!mbar_wait_cluster_warp<true>(smem_u32(&ctrl->acc_full), acc_ph, abort_flag, args.status, 16)) break;
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
            if (lane == 0) mbar_arrive_remote(acc_empty_leader);
            acc_ph ^= 1u;
            const int64_t row = mt * 256 + rank * 128 + q * 32 + lane;
            epilogue_row(args, swiglu, v, row, nt, h, alpha0, alpha1, g_inter, wamax);
        }
        if (args.epilogue == kEpiSwigluBf16) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wamax = fmaxf(wamax, __shfl_xor_sync(0xffffffffu, wamax, o));
            if (lane == 0) atomicMax(args.amax_ws, __float_as_uint(wamax));
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // no CTA leaves while the other may still signal it or read its memory
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc2(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_gemm2(const CUtensorMap& map_a, const CUtensorMap& map_b0, const CUtensorMap& map_b1,
                         const GemmArgs& args, int num_sms, cudaStream_t stream)
{
    static int attr_set_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set_for_device[dev]) {
        e = cudaFuncSetAttribute(gemm2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    const bool swiglu = args.epilogue != kEpiBf16;
    const int64_t num_m = (args.M + 255) / 256;
    const int64_t num_n = swiglu ? args.N / 128 : (args.N + 255) / 256;
    const int64_t tiles = num_m * num_n;
    const int64_t pairs = tiles < num_sms / 2 ? tiles : num_sms / 2;
    gemm2_kernel<<<(unsigned)(2 * pairs), kNumThreads, kSmemBytes, stream>>>(map_a, map_b0, map_b1, args);
    return cudaGetLastError();
}

}  // namespace nvfp4

#ifdef NVFP4_TRACE
extern "C" int nvfp4_debug_trace2(unsigned long long* out, int n)
{
    if (n > 2048) n = 2048;
    return cudaMemcpyFromSymbol(out, nvfp4::g_trace2, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : 4;
}
#endif
