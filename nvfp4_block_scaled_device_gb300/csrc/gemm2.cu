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
// scales of all 256 B rows.  Every copy of both CTAs, scale tiles included
// (through 1-D tensor maps), completes its bytes on the full
// barrier of the pair's even CTA ("leader"), whose producer 0 alone arrives
// on it with the byte count of both CTAs; the leader then issues the scale
// copies and MMAs for both CTAs.  The leader's commits are multicast to both
// CTAs (stage free, accumulator ready); both CTAs' epilogue warps arrive on
// the leader's accumulator-free barrier.  Each CTA's epilogue reads its own
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
// ring, control block, the epilogue warps' bf16 staging areas, alignment slack
constexpr int kEpiRows = 8;                            // bf16 staging rows per epilogue warp
constexpr int kSmemBytes = kStages * kStageBytes + kCtrlBytes + 8 * epi_stage_bytes(kEpiRows) + 1024;   // 8 epilogue warps
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment (128-byte swizzle atoms)");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kSfColsPerKK = 12;          // 4 (A) + 8 (B: two 128-row halves)
constexpr uint32_t kSfColsPerStage = 4 * kSfColsPerKK;
static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");

// Warp roles (16 warps, 4 warpgroups): warps 0-3 and 5-7 are copy
// producers (each a separate copy stream), warp 4 the MMA warp (leader; in
// the odd CTA it only allocates tensor memory), warps 8-15 the epilogue.  Launched at 128
// registers per thread; warpgroups 0-1 drop to 56 and 2-3 rise to 200.
constexpr int kProducers = 7;
constexpr int kMmaWarp = 4;
constexpr int kEpiWarp0 = 8;
constexpr int kEpiWarps = 8;
static_assert(kEpiWarps == 8, "shared memory holds 8 epilogue staging areas");
constexpr int kNumThreads = 512;
constexpr uint32_t kRegsSmall = 56;
constexpr uint32_t kRegsEpi = 200;
static_assert(2 * kRegsSmall + 2 * kRegsEpi == 512, "register split per sub-partition");
static_assert(kProducers == kEpiWarp0 - 1, "producers: warpgroups 0-1 less the MMA warp");
constexpr uint16_t kPairMask = 0x3;            // both CTAs of the cluster
// Shallowest K (stages of 256) for which a partial last wave of tiles is
// split over all pairs.
#ifndef NVFP4_PAIR_SPLIT_MIN_STAGES
#define NVFP4_PAIR_SPLIT_MIN_STAGES 32
#endif
constexpr int kPairSplitMinStages = NVFP4_PAIR_SPLIT_MIN_STAGES;

// Instruction descriptor, kind::mxf4nvf4: E2M1 A and B (format 1), UE4M3
// scales, K-major, N = 256 (bits 17-22 = N/8), M = 256 (bits 24-28 = M/16).
constexpr uint32_t kIdesc2 = (1u << 7) | (1u << 10) | ((256u >> 3) << 17) | ((256u >> 4) << 24);

#ifdef NVFP4_TRACE
// Debug timeline of the first CTA pair (built only with -DNVFP4_TRACE),
// %globaltimer ns: [0,256) leader stage-free seen, [256,512) leader issued,
// [512,768) odd stage-free seen, [768,1024) odd issued, [1280,1536) leader
// stage full seen, [1536,1792) leader MMAs issued.
__device__ unsigned long long g_trace2[2048];
#define TRACE2(slot, i)                                                 \
    do {                                                                \
        if (blockIdx.x < 2 && (i) < 256) g_trace2[(slot) + (i)] = globaltimer(); \
    } while (0)
#else
#define TRACE2(slot, i) do { } while (0)
#endif

struct Ctrl {
    uint64_t full[kStages];       // (leader) both CTAs' copies of the stage landed
    uint64_t empty[kStages];      // the pair's MMAs finished reading the stage
    uint64_t acc_full;            // the tile's accumulator is complete
    uint64_t acc_empty;           // (leader) both CTAs' epilogues drained the accumulator
    uint64_t teardown;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

// Work schedule of one SM pair, walked as segments (tile, first K stage, end
// K stage) by every role of both CTAs alike, P pairs: whole tiles p, p + P,
// ...; or (split, stream-K) the contiguous run [p*U/P, (p+1)*U/P) of the
// U = tiles x stages flattened (tile, K stage) units, a tile split between
// pairs being finished by the pair holding its first K stage.  (32-bit
// counts: the launcher keeps tiles x stages below 2^31.)
struct PairSchedule {
    int next;         // whole tiles: next tile; split: next unit
    int end;          // split: end of this pair's units
    int tiles;
    int stages;       // K stages per tile
    int pairs;
    bool split;
};

__device__ __forceinline__ int pair_first_unit(int64_t pair, int64_t units, int64_t pairs)
{
    return (int)(pair * units / pairs);
}

__device__ __forceinline__ PairSchedule make_pair_schedule(int64_t pair, int64_t pairs, int64_t tiles, int stages,
                                                          bool split)
{
    PairSchedule sc;
    sc.tiles = (int)tiles;
    sc.stages = stages;
    sc.pairs = (int)pairs;
    sc.split = split;
    if (split) {
        sc.next = pair_first_unit(pair, tiles * stages, pairs);
        sc.end = pair_first_unit(pair + 1, tiles * stages, pairs);
    } else {
        sc.next = (int)pair;
        sc.end = 0;
    }
    return sc;
}

__device__ __forceinline__ bool next_pair_segment(PairSchedule& sc, int64_t& tile, int& ks, int& ke)
{
    if (!sc.split) {
        if (sc.next >= sc.tiles) return false;
        tile = sc.next;
        ks = 0;
        ke = sc.stages;
        sc.next += sc.pairs;
        return true;
    }
    if (sc.next >= sc.end) return false;
    const int t = sc.next / sc.stages;
    tile = t;
    ks = sc.next - t * sc.stages;
    const int left = sc.end - sc.next;
    ke = left < sc.stages - ks ? ks + left : sc.stages;
    sc.next += ke - ks;
    return true;
}

// One past the last pair holding a piece of the tile that `pair` finishes
// (its contributors are pairs pair + 1 .. end - 1).
__device__ __forceinline__ int64_t pair_finisher_end(const PairSchedule& sc, int64_t pair, int64_t tile)
{
    const int64_t units = (int64_t)sc.tiles * sc.stages, tile_end = (tile + 1) * sc.stages;
    int64_t e = pair + 1;
    while (e < sc.pairs && pair_first_unit(e, units, sc.pairs) < tile_end) e++;
    return e;
}

__device__ __forceinline__ void flag_set_release2(int* f, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

__device__ __forceinline__ int flag_get_relaxed2(const int* f)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}

// Warp-wide bounded wait (every lane polls its own ready flag, or none when
// f is null; a vote decides); gives up like mbar_wait_warp.  Relaxed polls:
// the caller orders its reads of the flagged data with one acquire fence.
__device__ __forceinline__ bool flag_wait_warp2(const int* f, volatile int* abort_flag, int* status, int site)
{
    const uint64_t t0 = clock64();
    for (uint32_t i = 0;; i++) {
        if (__all_sync(0xffffffffu, f == nullptr || flag_get_relaxed2(f) != 0)) return true;
        if ((i & 255u) == 255u) {
            int stop = *abort_flag ? 1 : ((uint64_t)(clock64() - t0) > kWaitLimitCycles ? 2 : 0);
            stop = __shfl_sync(0xffffffffu, stop, 0);
            if (stop != 0) {
                if (stop == 2 && (threadIdx.x & 31) == 0) {
                    *abort_flag = 1;
                    if (status) atomicCAS(status, 0, kErrTimeout * 100 + site);
                }
                __syncwarp();
                return false;
            }
        }
    }
}

// kSplit: the split schedule (its fix-up code is compiled into this
// instantiation only).
// kRope: the bf16 epilogue's rotary embedding compiled in (whole tiles only).
template <bool kSplit, bool kRope = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kNumThreads, 1)
    gemm2_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                 const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_sfa,
                 const __grid_constant__ CUtensorMap map_sfb0, const __grid_constant__ CUtensorMap map_sfb1,
                 const GemmArgs args)
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
            mbar_init(smem_u32(&ctrl->full[s]), 1);     // leader's producer 0 + both CTAs' bytes
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
        prefetch_tmap(&map_sfa);
        prefetch_tmap(&map_sfb0);
        if (swiglu) {
            prefetch_tmap(&map_b1);
            prefetch_tmap(&map_sfb1);
        }
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
    // the next kernel of the stream may be scheduled from here on (it waits
    // for this one before touching its outputs)
    griddep_launch_dependents();

    if (warp < kEpiWarp0) {
        // warpgroups 0-1: one register-budget instruction for all eight warps
        setmaxnreg_dec<kRegsSmall>();
        if (warp != kMmaWarp) {
            // ------------------------------------------------------ producers
            // Seven warps, one lane each, share every stage's copies (copies
            // issued by one thread are served one after the other): producers
            // 0-3 fetch the 64-row code boxes (this CTA's A rows 0-63, 64-127,
            // its B half's rows 0-63, 64-127), producers 4-6 the 2 KB scale
            // runs (A, B rows 0-127, B rows 128-255) of the stage.  All copies
            // complete on the leader's full barrier; the leader's producer 0
            // arrives on it once per stage with both CTAs' byte count (a slot
            // is refilled only after the MMAs that read it completed, so no
            // copy of a later fill can land in the current phase).  Boxes past
            // the operand's rows are not fetched: their stale shared memory
            // only feeds accumulator rows >= M or columns >= N.  A scale box
            // of a partial last stage also carries the scales of the next K
            // stages or of the next rows (or zero fill past the end), which no
            // MMA reads.
            const int p = warp < kMmaWarp ? warp : warp - 1;
            // A and its scales (producers 0, 1, 4) wait for the previous
            // kernel to complete; the weight boxes and scales (producers 2,
            // 3, 5, 6) start at once when the caller vouches that the weights
            // were complete before that kernel started.
            if (p < 2 || p == 4 || !args.weights_early) griddep_wait();
            const uint32_t full_leader0 = map_to_cta(smem_u32(&ctrl->full[0]), 0);
            const uint32_t empty0 = smem_u32(&ctrl->empty[0]);
            constexpr uint32_t kBox = kCodeBoxRows * 128u;
            constexpr uint32_t kSfBox = 4u * kSfTile;                       // 2048 bytes
            const uint64_t pol = p < 2 ? l2_policy_evict_last() : l2_policy_evict_first();
            const uint32_t my_off = p < 4 ? (uint32_t)p * kBox                // A then the B half, contiguous
                                          : (uint32_t)(kABytes + kBBytes) + (uint32_t)(p - 4) * kSfBox;
            const CUtensorMap* sf_map = p == 4 ? &map_sfa : (p == 6 && swiglu) ? &map_sfb1 : &map_sfb0;
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int kcount = 0;
            PairSchedule sched = make_pair_schedule(pair, num_pairs, num_tiles, num_kstages, kSplit);
            int64_t tile;
            int ks, ke;
            while (ok && next_pair_segment(sched, tile, ks, ke)) {
                const int64_t mt = tile % num_m, nt = tile / num_m;
                const int64_t row0 = mt * 256 + rank * 128;          // this CTA's first A row
                int32_t yb;
                const CUtensorMap* mb;
                int64_t sfb_block0, sfb_block1;                      // 128-row scale blocks of B
                if (swiglu) {
                    yb = (int32_t)(nt * 128);
                    mb = rank ? &map_b1 : &map_b0;
                    sfb_block0 = sfb_block1 = nt;
                } else {
                    yb = (int32_t)(nt * 256 + rank * 128);
                    mb = &map_b0;
                    sfb_block0 = 2 * nt;
                    sfb_block1 = 2 * nt + 1;
                }
                const bool has_b1 = swiglu || nt * 256 + 128 < args.N;   // the second B scale block exists
                // this producer's copy: code box (first row), or scale box
                // (first 8-byte element of its 2 KB run at K stage 0)
                const CUtensorMap* my_map = p < 2 ? &map_a : p < 4 ? mb : sf_map;
                const int32_t my_y = p < 4 ? (p < 2 ? (int32_t)row0 : yb) + (p & 1) * kCodeBoxRows
                                           : (int32_t)(((p == 4 ? (row0 / 128) * args.sfa_tile_stride
                                                                : (p == 5 ? sfb_block0 : sfb_block1) * args.sfb_tile_stride)) /
                                                       8);
                const bool my_copy = p < 4 ? my_y < (p < 2 ? args.M : args.N)
                                           : p == 4 ? row0 < args.M : p == 5 ? true : has_b1;
                // bytes of the stage's copies in both CTAs (the leader's producer 0 expects them)
                uint32_t tx = 0;
                if (leader && p == 0) {
                    for (int r = 0; r < 2; r++) {
                        const int64_t r0 = mt * 256 + r * 128;
                        const int64_t yr = swiglu ? nt * 128 : nt * 256 + r * 128;
                        tx += kBox * ((r0 < args.M) + (r0 + kCodeBoxRows < args.M) + (yr < args.N) +
                                      (yr + kCodeBoxRows < args.N));
                        tx += kSfBox * ((r0 < args.M) + 1 + (has_b1 ? 1 : 0));
                    }
                }
                for (int kb = ks; kb < ke; kb++) {
                    if (!mbar_wait_cluster_warp(empty0 + 8u * (uint32_t)s, ph ^ 1u, abort_flag, args.status, 11)) {
                        ok = false;
                        break;
                    }
                    if (p == 0 && lane == 0) TRACE2(rank * 512, kcount);
                    const uint32_t full = full_leader0 + 8u * (uint32_t)s;
                    const uint32_t st = base + (uint32_t)s * kStageBytes;
                    if (lane == 0) {
                        if (leader && p == 0) mbar_arrive_expect_tx(smem_u32(&ctrl->full[0]) + 8u * (uint32_t)s, tx);
                        if (my_copy) {
                            if (p < 4)
                                tma_load_2d_pair(st + my_off, my_map, full, kb * 128, my_y, pol);
                            else
                                tma_load_1d_pair(st + my_off, my_map, full, my_y + kb * (int32_t)(kSfBox / 8), pol);
                        }
                    }
                    __syncwarp();
                    if (p == 0 && lane == 0) TRACE2(rank * 512 + 256, kcount);
                    kcount++;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // on an early stop, the leader's teardown waits for the copies in
            // flight (its full barriers count both CTAs' bytes); the final
            // cluster barrier keeps this CTA alive until then
            __syncwarp();
        } else {
            const uint32_t full0 = smem_u32(&ctrl->full[0]);
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
                PairSchedule sched = make_pair_schedule(pair, num_pairs, num_tiles, num_kstages, kSplit);
                int64_t tile;
                int ks, ke;
                while (ok && next_pair_segment(sched, tile, ks, ke)) {
                    if (!mbar_wait_cluster_warp(smem_u32(&ctrl->acc_empty), acc_ph ^ 1u, abort_flag, args.status, 12))
                        break;
                    tc_fence_after();
                    // full stages: nothing but the wait and one fused issue block
                    const int kb_full_end = ke < full_kstages ? ke : full_kstages;
                    for (int kb = ks; kb < kb_full_end; kb++) {
                        if (!mbar_wait_cluster_warp(full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 13)) {
                            ok = false;
                            break;
                        }
                        TRACE2(1280, kcount);
                        tc_fence_after();
                        const uint32_t soff = (uint32_t)s * (kStageBytes >> 4);
                        const uint32_t a_lo = desc_a_lo + soff;
                        stage_issue_2sm(tmem, tmem + kAccCols + (uint32_t)s * kSfColsPerStage, desc_sf_lo + soff,
                                        desc_sf_hi, a_lo, a_lo + (kABytes >> 4), desc_sw_hi, kIdesc2,
                                        kb != ks ? 1u : 0u, empty0 + 8u * (uint32_t)s, kPairMask);
                        TRACE2(1536, kcount);
                        kcount++;
                        if (++s == kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (ok && ke > full_kstages) {
                        // K tail: a last stage of fewer than 4 K-steps
                        if (!mbar_wait_cluster_warp(full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 13)) {
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
                                                   (full_kstages != ks || kk != 0) ? 1u : 0u);
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
                if (!ok && lane == 0) {
                    // stopped early: let the copies of the stages not consumed
                    // land in both CTAs before their shared memory goes away
                    // (bounded); the next fill of each slot (phase ph of slot s
                    // onwards) may be in flight
                    for (int i = 0; i < kStages; i++) {
                        const int si = (s + i) % kStages;
                        const uint32_t pi = si >= s ? ph : ph ^ 1u;
                        mbar_wait_teardown(full0 + 8u * (uint32_t)si, pi);
                    }
                }
                __syncwarp();
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        setmaxnreg_inc<kRegsEpi>();                        // warpgroups 2-3
        griddep_wait();                     // scales, residual, outputs: after the previous kernel
        const int q = warp & 3;             // tensor-memory lane quarter of this warp
        const int h = (warp - kEpiWarp0) >> 2;   // which half of the tile's columns
        // this warp's bf16 staging area, after the ring and the control block
        const uint32_t epi_stage = base + (uint32_t)(kStages * kStageBytes + kCtrlBytes) +
                                   (uint32_t)((warp - kEpiWarp0) * epi_stage_bytes(kEpiRows));
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        const uint32_t acc_empty_leader = map_to_cta(smem_u32(&ctrl->acc_empty), 0);
        const float ga = *args.ga;
        const float alpha0 = __fmul_rn(ga, *args.gb0);
        const float alpha1 = swiglu ? __fmul_rn(ga, *args.gb1) : alpha0;
        const float g_inter = args.epilogue == kEpiSwigluFp4 ? *args.g_inter : 1.0f;
        uint32_t acc_ph = 0;
        float wamax = 0.0f;
        const int we = warp - kEpiWarp0;   // epilogue warp index (its slice of a partial slot)
        PairSchedule sched = make_pair_schedule(pair, num_pairs, num_tiles, num_kstages, kSplit);
        int64_t tile;
        int ks, ke;
        while (next_pair_segment(sched, tile, ks, ke)) {
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
            if (kSplit && ks != 0) {
                // later K stages of a tile finished by another pair: this
                // warp's 32 x 128 partial into the CTA's slot (values
                // 4j..4j+3 of lane l as one 16-byte vector at [we][j][l]),
                // then its ready flag (release: after the warp's stores)
                float4* slot = reinterpret_cast<float4*>(args.sk_partials + (int64_t)blockIdx.x * kSplitSlotFloats) +
                               we * 1024 + lane;
                if (row < args.M) {
#pragma unroll
                    for (int j = 0; j < 32; j++)
                        __stcg(slot + j * 32, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
                }
                __syncwarp();
                if (lane == 0) flag_set_release2(args.sk_flags + blockIdx.x * kSplitFlagsPerCta + we, 1);
                continue;
            }
            if (kSplit && ke != num_kstages) {
                // first K stages of a tile whose later stages other pairs
                // hold: wait for the partials of this CTA's rank in those
                // pairs (lane i polls pair + 1 + i (+ 32k)), add them in pair
                // order, return their flags to zero
                const int64_t p_end = pair_finisher_end(sched, pair, tile);
                bool got = true;
                for (int64_t cb = pair + 1; cb < p_end && got; cb += 32) {
                    const int64_t c = cb + lane;
                    got = flag_wait_warp2(c < p_end ? args.sk_flags + (2 * c + rank) * kSplitFlagsPerCta + we : nullptr,
                                          abort_flag, args.status, 17);
                }
                if (!got) break;
                asm volatile("fence.acq_rel.gpu;" ::: "memory");
                if (row < args.M) {
                    for (int64_t c = pair + 1; c < p_end; c++) {
                        const float4* slot = reinterpret_cast<const float4*>(args.sk_partials +
                                                                             (2 * c + rank) * kSplitSlotFloats) +
                                             we * 1024 + lane;
#pragma unroll
                        for (int jb = 0; jb < 32; jb += 16) {   // 16 loads in flight, then their adds
                            float4 t[16];
#pragma unroll
                            for (int j = 0; j < 16; j++) t[j] = __ldcg(slot + (jb + j) * 32);
#pragma unroll
                            for (int j = 0; j < 16; j++) {
                                v[4 * (jb + j)] += t[j].x;
                                v[4 * (jb + j) + 1] += t[j].y;
                                v[4 * (jb + j) + 2] += t[j].z;
                                v[4 * (jb + j) + 3] += t[j].w;
                            }
                        }
                    }
                }
                __syncwarp();
                for (int64_t c = pair + 1 + lane; c < p_end; c += 32)
                    args.sk_flags[(2 * c + rank) * kSplitFlagsPerCta + we] = 0;
            }
            // bf16 stores staged through shared memory: whole 256-byte row
            // segments per warp store
            epilogue_row<kRope, kEpiRows>(args, swiglu, v, row, nt, h, alpha0, alpha1, g_inter, wamax, epi_stage);
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
                         const CUtensorMap& map_sfa, const CUtensorMap& map_sfb0, const CUtensorMap& map_sfb1,
                         const GemmArgs& args, int num_sms, cudaStream_t stream)
{
    static int attr_set_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set_for_device[dev]) {
        e = cudaFuncSetAttribute(gemm2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm2_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm2_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    const bool swiglu = args.epilogue != kEpiBf16;
    const int64_t num_m = (args.M + 255) / 256;
    const int64_t num_n = swiglu ? args.N / 128 : (args.N + 255) / 256;
    const int64_t tiles = num_m * num_n;
    const int64_t stages = (args.K / 64 + 3) / 4;
    const int64_t all_pairs = num_sms / 2;
    // Whole tiles strided over min(tiles, pairs) pairs, unless (given a
    // workspace) their last wave leaves more than a tenth of the pairs idle
    // and the tiles are deep in K (>= 32 stages): then every pair takes an
    // equal run of the (tile, K stage) units, as the 1-SM kernel's split.
    const int64_t waves = (tiles + all_pairs - 1) / all_pairs;
    const bool rope = args.rope_pos != nullptr;
    const bool split = !rope && args.sk_partials != nullptr && args.sk_flags != nullptr && num_sms <= kSplitMaxCtas &&
                       tiles * stages >= all_pairs && tiles * 10 < waves * all_pairs * 9 &&
                       stages >= kPairSplitMinStages &&
                       tiles * stages < (int64_t)1 << 31;
    const int64_t pairs = split ? all_pairs : (tiles < all_pairs ? tiles : all_pairs);
    // programmatic launch: the CTAs may start on SMs the previous kernel has
    // left, and fetch weights before it completes when args.weights_early
    if (split)
        return launch_programmatic(gemm2_kernel<true>, dim3((unsigned)(2 * pairs)), dim3(kNumThreads), kSmemBytes,
                                   stream, map_a, map_b0, map_b1, map_sfa, map_sfb0, map_sfb1, args);
    if (rope)
        return launch_programmatic(gemm2_kernel<false, true>, dim3((unsigned)(2 * pairs)), dim3(kNumThreads),
                                   kSmemBytes, stream, map_a, map_b0, map_b1, map_sfa, map_sfb0, map_sfb1, args);
    return launch_programmatic(gemm2_kernel<false>, dim3((unsigned)(2 * pairs)), dim3(kNumThreads), kSmemBytes, stream,
                               map_a, map_b0, map_b1, map_sfa, map_sfb0, map_sfb1, args);
}

}  // namespace nvfp4

#ifdef NVFP4_TRACE
extern "C" int nvfp4_debug_trace2(unsigned long long* out, int n)
{
    if (n > 2048) n = 2048;
    return cudaMemcpyFromSymbol(out, nvfp4::g_trace2, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : 4;
}
#endif
