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
// Warp roles (512 threads):
//   warps 0-3, 5-7  TMA producers, one copy stream each: codes by 2-D TMA in
//               64-row boxes, scales by 1-D bulk copies (the 512-byte scale
//               tiles are contiguous along K).
//   warp 4      tensor-memory allocator; one lane issues tcgen05.cp (scales
//               shared -> tensor memory) and tcgen05.mma, and commits.
//   warps 8-15  epilogue: drain the accumulator to registers, release it to
//               the MMA warp, then scale / SwiGLU / requantize / store while
//               the next tile accumulates.
// Persistent: grid = min(#tiles, #SMs), tile t -> (m = t % Mt, n = t / Mt),
// so CTAs running together share the same weight tiles through L2; or, for
// deep-K tiles whose last wave would leave more than a tenth of the GPU
// idle, a split schedule over all SMs (stream-K: each CTA an equal run of
// the flattened (tile, K stage) units; a tile's CTAs combine fp32 partials
// through a workspace, the one holding its first K stage finishing it).
#include "common.cuh"
#include "gemm_epilogue.cuh"
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
// ring, control block, the epilogue warps' bf16 staging areas, alignment slack
constexpr int kSmemBytes = kStages * kStageBytes + kCtrlBytes + 8 * kEpiStageBytes + 1024;   // 8 epilogue warps
static_assert(kSmemBytes <= 232448, "shared memory per block");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kSfColsPerKK = 12;          // 4 (A) + 4 + 4 (two B row tiles)
constexpr uint32_t kSfColsPerStage = 4 * kSfColsPerKK;
static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");

// Warp roles (16 warps, 4 warpgroups): warps 0-3 and 5-7 are copy
// producers (each a separate copy stream), warp 4 is the MMA warp, warps
// 8-15 the epilogue.  Launched at 128 registers per thread; warpgroups 0-1
// drop to 64 and warpgroups 2-3 rise to 192 (64 + 64 + 192 + 192 = 512 per
// lane of each sub-partition, its 16384 registers).
constexpr int kProducers = 7;
constexpr int kMmaWarp = 4;
constexpr int kEpiWarp0 = 8;
constexpr int kEpiWarps = 8;
static_assert(kEpiWarps == 8, "shared memory holds 8 epilogue staging areas");
constexpr int kNumThreads = 512;
constexpr uint32_t kRegsSmall = 64;
constexpr uint32_t kRegsEpi = 192;
// Split fix-up: warps with at most this many valid rows fetch the partials
// with their lanes spread over the columns instead of over the rows.
constexpr int kFixRowsByLane = 4;
static_assert(2 * kRegsSmall + 2 * kRegsEpi == 512, "register split per sub-partition");
static_assert(kProducers == kEpiWarp0 - 1, "producers: warpgroups 0-1 less the MMA warp");

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1 (format 1), UE4M3
// scales (bit 23 = 0), K-major A and B, N = 256 (bits 17-22 = N/8),
// M = 128 (bits 24-28 = M/16), dense, scale-factor ids 0.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((256u >> 3) << 17) | ((128u >> 4) << 24);

#ifdef NVFP4_TRACE
// Debug timeline of CTA NVFP4_TRACE_CTA (default 0; built only with
// -DNVFP4_TRACE): SM clock at each
// pipeline handoff.  [0,256) producer empty-wait done, [256,512) producer
// issued, [512,768) MMA full-wait done, [768,1024) MMA issued, [1024,1088)
// MMA acc-empty done, [1088,1152) epilogue acc-full done, [1152,1216) drained,
// [1216,1280) split partials added (or partial stored).
__device__ unsigned long long g_trace[1280];
#ifndef NVFP4_TRACE_CTA
#define NVFP4_TRACE_CTA 0
#endif
#define TRACE(slot, i) \
    do { if (blockIdx.x == NVFP4_TRACE_CTA && (i) < 64 * ((slot) < 1024 ? 4 : 1)) g_trace[(slot) + (i)] = clock64(); } while (0)
// Per-CTA events on the global timer (ns): [c][0] start, [c][1] first
// accumulator ready, [c][2] first segment's partial stored or first tile
// finished, [c][3] last segment finished.
__device__ unsigned long long g_trace_cta[256][4];
__device__ unsigned long long g_trace_fix[16];   // CTA 0, first epilogue warp: [1] all flags seen, [0] partials added
#define TRACE_CTA(k) \
    do { if (blockIdx.x < 256) g_trace_cta[blockIdx.x][k] = globaltimer(); } while (0)
#else
#define TRACE(slot, i) do { } while (0)
#define TRACE_CTA(k) do { } while (0)
#endif

struct Ctrl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t teardown;
    uint32_t tmem_base;
    int abort_flag;
    int fix_arrive;       // split fix-up: arrivals of the epilogue warps (epi_sync)
    uint64_t fix_full;    // split fix-up: the contributors' partial rows landed in the ring
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

// Work schedule of one CTA, walked as segments (tile, first K stage, end K
// stage) by every role alike, on a grid of G CTAs: whole tiles c, c + G, ...;
// or (split, stream-K) a contiguous range of the flattened (tile, K stage)
// units, CTA c taking [c*U/G, (c+1)*U/G) of U = tiles x stages.
// (32-bit counts: the launcher keeps tiles x stages below 2^31.)
struct Schedule {
    int next;         // whole tiles: next tile; split: next unit
    int end;          // split: end of this CTA's units
    int tiles;
    int stages;       // K stages per tile
    bool split;
};

__device__ __forceinline__ int split_first_unit(int64_t cta, int64_t units)
{
    return (int)(cta * units / gridDim.x);
}

__device__ __forceinline__ Schedule make_schedule(int64_t tiles, int stages, bool split)
{
    Schedule sc;
    sc.tiles = (int)tiles;
    sc.stages = stages;
    sc.split = split;
    if (split) {
        sc.next = split_first_unit(blockIdx.x, tiles * stages);
        sc.end = split_first_unit(blockIdx.x + 1, tiles * stages);
    } else {
        sc.next = (int)blockIdx.x;
        sc.end = 0;
    }
    return sc;
}

// One past the last CTA holding a piece of the tile that the calling CTA
// finishes (its contributors are the CTAs blockIdx.x + 1 .. end - 1).
__device__ __forceinline__ int64_t finisher_end(const Schedule& sc, int64_t tile)
{
    const int64_t units = (int64_t)sc.tiles * sc.stages, tile_end = (tile + 1) * sc.stages;
    int64_t c_end = (int64_t)blockIdx.x + 1;
    while (c_end < (int64_t)gridDim.x && split_first_unit(c_end, units) < tile_end) c_end++;
    return c_end;
}

__device__ __forceinline__ bool next_segment(Schedule& sc, int64_t& tile, int& ks, int& ke)
{
    if (!sc.split) {
        if (sc.next >= sc.tiles) return false;
        tile = sc.next;
        ks = 0;
        ke = sc.stages;
        sc.next += (int)gridDim.x;
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

// Ready flag of a partial accumulator: set with release semantics after the
// slot's stores, read with acquire semantics before its loads.
__device__ __forceinline__ void flag_set_release(int* f, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

__device__ __forceinline__ int flag_get_relaxed(const int* f)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}

// Warp-wide bounded wait (converged: every lane polls its own ready flag,
// or none when f is null, and a vote decides); gives up like mbar_wait_warp.
// The polls are relaxed: the caller orders its reads of the flagged data
// after the wait with one acquire fence.
__device__ __forceinline__ bool flag_wait_warp(const int* f, volatile int* abort_flag, int* status, int site)
{
    const uint64_t t0 = clock64();
    for (uint32_t i = 0;; i++) {
        if (__all_sync(0xffffffffu, f == nullptr || flag_get_relaxed(f) != 0)) return true;
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
// instantiation only; the whole-tile instantiation carries none of it).
// kGrouped: the expert-indexed mode (GemmArgs::grp_*; whole tiles, bf16
// epilogue without residual): tile m of the device table takes its A rows
// from the expert-sorted operand and its B rows from that expert's block of
// the stacked weights, and each output row goes where the row map says.
// kRope: the bf16 epilogue's rotary embedding compiled in (whole tiles only).
template <bool kSplit, bool kGrouped = false, bool kRope = false>
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

    int64_t num_m = (args.M + 127) / 128;
    if (kGrouped) {
        // the tile table is written by the previous kernel of the stream
        griddep_wait();
        num_m = *reinterpret_cast<const volatile int*>(args.grp_count);
    }
    const int64_t num_n = swiglu ? args.N / 128 : (args.N + 255) / 256;
    const int64_t num_tiles = num_m * num_n;
    const int num_kk = (int)(args.K / 64);
    const int num_kstages = (num_kk + 3) / 4;
    const int full_kstages = num_kk / 4;       // stages of 4 K-steps
    const int tail_kk = num_kk % 4;            // K-steps of a last, partial stage
    constexpr bool split = kSplit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(smem_u32(&ctrl->full[s]), 1);      // producer 0's arrival + all copies' bytes
            mbar_init(smem_u32(&ctrl->empty[s]), 1);
        }
        mbar_init(smem_u32(&ctrl->acc_full), 1);
        mbar_init(smem_u32(&ctrl->acc_empty), kEpiWarps);
        mbar_init(smem_u32(&ctrl->teardown), 1);
        mbar_init(smem_u32(&ctrl->fix_full), kEpiWarps);
        ctrl->abort_flag = 0;
        ctrl->fix_arrive = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&map_a);
        prefetch_tmap(&map_b0);
        if (swiglu) prefetch_tmap(&map_b1);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    if (threadIdx.x == 0) TRACE_CTA(0);
    // the next kernel of the stream may be scheduled from here on (it waits
    // for this one before touching its outputs)
    griddep_launch_dependents();

    if (warp < kEpiWarp0) {
        // warpgroups 0-1: one register-budget instruction for all eight warps
        setmaxnreg_dec<kRegsSmall>();
        if (warp != kMmaWarp) {
            // ------------------------------------------------------ producers
            // Seven warps, one lane each, share every stage's copies (copies
            // issued by one thread are served one after the other, about 25
            // bytes per clock): producer p < 6 fetches the 64-row code box p of
            // the stage (A rows 0-63, 64-127, B rows 0-63, ..., 192-255), producer
            // 6 the A and B scale tiles.  Producer 0 alone arrives on the stage's
            // full barrier, with the byte count of all seven producers' copies;
            // the others' copies only complete bytes on it, so the stage is full
            // when every byte has landed, whatever order the producers run in
            // (a slot is refilled only after the MMAs that read it completed,
            // so no copy of a later fill can land in the current phase).  A box
            // whose first row is past the operand's rows is not fetched: its
            // stale shared memory only feeds accumulator rows >= M or columns
            // >= N, never stored.
            const int p = warp < kMmaWarp ? warp : warp - 1;
            // A and the scale tiles (producers 0, 1, 6) wait for the previous
            // kernel to complete (programmatic launch); the weight boxes
            // (producers 2-5) start at once when the caller vouches that the
            // weights were complete before that kernel started.
            if (p < 2 || p == 6 || !args.weights_early) griddep_wait();
            const uint32_t full0 = smem_u32(&ctrl->full[0]);
            const uint32_t empty0 = smem_u32(&ctrl->empty[0]);
            constexpr uint32_t kBox = kCodeBoxRows * 128u;
            const uint64_t pol = p < 2 ? l2_policy_evict_last() : l2_policy_evict_first();
            const uint32_t my_off = (uint32_t)p * kBox;     // A, B rows 0-127, B rows 128-255 are contiguous
            int s = 0;
            uint32_t ph = 0, issued = 0, issued_ph = 0;
            int kcount = 0;
            bool ok = true;
            Schedule sched = make_schedule(num_tiles, num_kstages, split);
            int64_t tile;
            int ks, ke;
            while (ok && next_segment(sched, tile, ks, ke)) {
                const int64_t mt = tile % num_m, nt = tile / num_m;
                int32_t ya = (int32_t)(mt * 128);
                int32_t yb0, yb1;
                const uint8_t *pb0, *pb1;
                bool has_b1;
                int64_t b_base = 0;        // grouped: first row of the tile's expert in the stacked weights
                if (kGrouped) {
                    const int4 td = args.grp_tiles[mt];
                    ya = td.y;
                    b_base = (int64_t)td.x * args.N;
                }
                if (kGrouped) {
                    yb0 = (int32_t)(b_base + nt * 256);
                    yb1 = yb0 + 128;
                    pb0 = args.sfb0 + (b_base / 128 + 2 * nt) * args.sfb_tile_stride;
                    pb1 = pb0 + args.sfb_tile_stride;
                    has_b1 = nt * 256 + 128 < args.N;
                } else if (swiglu) {
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
                const CUtensorMap* my_map = p < 2 ? &map_a : p < 4 ? &map_b0 : (swiglu ? &map_b1 : &map_b0);
                const int32_t my_y = (p < 2 ? ya : p < 4 ? yb0 : yb1) + (p & 1) * kCodeBoxRows;
                // bounds: B rows are checked within the (expert's) N rows
                const int64_t yb0r = yb0 - b_base, yb1r = yb1 - b_base;
                const bool my_box = p < 6 && (p < 2 ? my_y < args.M : my_y - b_base < args.N);
                // code boxes of the stage that are fetched (A rows +64, B rows +64, +128, +192)
                const uint32_t code_bytes =
                    kBox * (1u + (ya + kCodeBoxRows < args.M ? 1u : 0u) + 1u + (yb0r + kCodeBoxRows < args.N ? 1u : 0u) +
                            (yb1r < args.N ? 1u : 0u) + (yb1r + kCodeBoxRows < args.N ? 1u : 0u));
                const uint8_t* pa = args.sfa + (int64_t)(ya / 128) * args.sfa_tile_stride + (size_t)ks * 4 * kSfTile;
                pb0 += (size_t)ks * 4 * kSfTile;
                pb1 += (size_t)ks * 4 * kSfTile;
                for (int kb = ks; kb < ke; kb++) {
                    if (!mbar_wait_warp(empty0 + 8u * (uint32_t)s, ph ^ 1u, abort_flag, args.status, 1)) {
                        ok = false;
                        break;
                    }
                    if (p == 0 && lane == 0) TRACE(0, kcount);
                    const uint32_t sf_bytes = (uint32_t)min(4, num_kk - kb * 4) * kSfTile;
                    const uint32_t full = full0 + 8u * (uint32_t)s;
                    const uint32_t st = base + (uint32_t)s * kStageBytes;
                    const uint32_t sf_st = st + kABytes + kBBytes;
                    const int32_t xk = kb * 128;
                    if (lane == 0) {
                        if (p == 0) mbar_arrive_expect_tx(full, code_bytes + sf_bytes * (has_b1 ? 3u : 2u));
                        if (my_box) {
                            tma_load_2d(st + my_off, my_map, full, xk, my_y, pol);
                        } else if (p == 6) {
                            bulk_load(sf_st, pa, sf_bytes, full);
                            bulk_load(sf_st + kSfaBytes, pb0, sf_bytes, full);
                            if (has_b1) bulk_load(sf_st + kSfaBytes + 4 * kSfTile, pb1, sf_bytes, full);
                        }
                    }
                    __syncwarp();
                    pa += 4 * kSfTile;
                    pb0 += 4 * kSfTile;
                    pb1 += 4 * kSfTile;
                    if (p == 0 && lane == 0) TRACE(256, kcount);
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
        } else {
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
            Schedule sched = make_schedule(num_tiles, num_kstages, split);
            int64_t tile;
            int ks, ke;
            while (ok && next_segment(sched, tile, ks, ke)) {
                if (!mbar_wait_warp(smem_u32(&ctrl->acc_empty), acc_ph ^ 1u, abort_flag, args.status, 2)) break;
                TRACE(1024, tcount);
                tcount++;
                tc_fence_after();
                // full stages of the segment: nothing but the wait and one
                // fused issue block
                const int kfull_end = ke < full_kstages ? ke : full_kstages;
                for (int kb = ks; kb < kfull_end; kb++) {
                    if (!mbar_wait_warp(full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 3)) {
                        ok = false;
                        break;
                    }
                    TRACE(512, kcount);
                    tc_fence_after();
                    // descriptors of this stage: only 32-bit adds in the loop
                    const uint32_t soff = (uint32_t)s * (kStageBytes >> 4);
                    const uint32_t a_lo = desc_a_lo + soff;
                    stage_issue_1sm(tmem, tmem + kAccCols + (uint32_t)s * kSfColsPerStage, desc_sf_lo + soff,
                                    desc_sf_hi, a_lo, a_lo + (kABytes >> 4), desc_sw_hi, kIdesc, kb != ks ? 1u : 0u,
                                    empty0 + 8u * (uint32_t)s);
                    TRACE(768, kcount);
                    kcount++;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok && ke > full_kstages) {
                    // K tail: a last stage of fewer than 4 K-steps
                    if (!mbar_wait_warp(full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 3)) {
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
                            tmem_copy_sf_warp(c, desc_from(f, desc_sf_hi));
                            tmem_copy_sf_warp(c + 4, desc_from(f + (kSfaBytes >> 4), desc_sf_hi));
                            tmem_copy_sf_warp(c + 8, desc_from(f + ((kSfaBytes + 4 * kSfTile) >> 4), desc_sf_hi));
                        }
                        for (int kk = 0; kk < tail_kk; kk++) {
                            const uint32_t c = sf_stage + (uint32_t)kk * kSfColsPerKK;
                            mma_mxf4nvf4_warp(tmem, desc_from(a_lo + 2u * kk, desc_sw_hi),
                                              desc_from(b_lo + 2u * kk, desc_sw_hi), kIdesc, c, c + 4,
                                              (full_kstages != ks || kk != 0) ? 1u : 0u);
                        }
                        mma_commit_warp(empty0 + 8u * (uint32_t)s);
                        kcount++;
                        if (++s == kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
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
        }
    } else {
        // ------------------------------------------------------ epilogue
        setmaxnreg_inc<kRegsEpi>();                        // warpgroups 2-3
        griddep_wait();                     // scales, residual, outputs: after the previous kernel
        const int q = warp & 3;             // tensor-memory lane quarter of this warp
        const int h = (warp - kEpiWarp0) >> 2;   // which half of the tile's columns
        // this warp's bf16 staging area, after the ring and the control block
        const uint32_t epi_stage = base + (uint32_t)(kStages * kStageBytes + kCtrlBytes) +
                                   (uint32_t)((warp - kEpiWarp0) * kEpiStageBytes);
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        const float ga = *args.ga;
        const float alpha0 = __fmul_rn(ga, *args.gb0);
        const float alpha1 = swiglu ? __fmul_rn(ga, *args.gb1) : alpha0;
        const float g_inter = args.epilogue == kEpiSwigluFp4 ? *args.g_inter : 1.0f;
        uint32_t acc_ph = 0;
        float wamax = 0.0f;
        int ecount = 0;
        const int we = warp - kEpiWarp0;   // epilogue warp index (its slice of a partial slot)
        Schedule sched = make_schedule(num_tiles, num_kstages, split);
        int64_t tile;
        int ks, ke;
        GemmArgs gargs = args;              // grouped: rows are output rows of the row map
        if (kGrouped) gargs.M = args.grp_out_rows;
        while (next_segment(sched, tile, ks, ke)) {
            const int64_t mt = tile % num_m, nt = tile / num_m;
            if (!mbar_wait_warp<true>(smem_u32(&ctrl->acc_full), acc_ph, abort_flag, args.status, 4)) break;
            if (warp == kEpiWarp0 && lane == 0) TRACE(1088, ecount);
            if (warp == kEpiWarp0 && lane == 0 && ecount == 0) TRACE_CTA(1);
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
            if (warp == kEpiWarp0 && lane == 0) TRACE(1152, ecount);
            ecount++;
            acc_ph ^= 1u;

            const int64_t row = mt * 128 + q * 32 + lane;
            if (split && ks != 0) {
                // later K stages of a tile finished by another CTA: this
                // warp's 32 x 128 partial into the CTA's slot (values 4j..4j+3
                // of lane l as one 16-byte vector at [we][j][l]: each store
                // instruction of the warp writes 512 contiguous bytes), then
                // its ready flag
                float4* slot = reinterpret_cast<float4*>(args.sk_partials + (int64_t)blockIdx.x * kSplitSlotFloats) +
                               we * 1024 + lane;
                if (row < args.M) {
#pragma unroll
                    for (int j = 0; j < 32; j++)
                        __stcg(slot + j * 32, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
                }
                // the warp's stores, ordered by __syncwarp before lane 0's
                // release store of the flag, are visible to whoever acquires it
                __syncwarp();
                if (lane == 0) flag_set_release(args.sk_flags + blockIdx.x * kSplitFlagsPerCta + we, 1);
                if (warp == kEpiWarp0 && lane == 0) TRACE(1216, ecount - 1);
                if (warp == kEpiWarp0 && lane == 0) TRACE_CTA(2);
                continue;
            }
            if (split && ke != num_kstages) {
                // first K stages of a tile whose later stages other CTAs
                // hold (each as the first segment of its range): wait for
                // their partials, add them, then return their flags to zero
                const int64_t c_end = finisher_end(sched, tile);
                // lane i waits for contributor blockIdx.x + 1 + i (+ 32k)
                bool got = true;
                for (int64_t cb = (int64_t)blockIdx.x + 1; cb < c_end && got; cb += 32) {
                    const int64_t c = cb + lane;
                    got = flag_wait_warp(c < c_end ? args.sk_flags + c * kSplitFlagsPerCta + we : nullptr, abort_flag,
                                         args.status, 5);
                }
#ifdef NVFP4_TRACE
                if (blockIdx.x == 0 && warp == kEpiWarp0 && lane == 0) g_trace_fix[1] = globaltimer();
#endif
                if (got) asm volatile("fence.acq_rel.gpu;" ::: "memory");
                const int64_t wrow0 = mt * 128 + q * 32;             // first row of this warp
                const int nrows = (int)(args.M - wrow0 < 32 ? (args.M - wrow0 > 0 ? args.M - wrow0 : 0) : 32);
                // When the contributors' partial slots of the warps with valid
                // rows fit in the ring (idle now: this is the CTA's last
                // segment, its MMAs are done), they come in at once by bulk
                // copies, so that the fix-up costs one memory round trip
                // instead of two per contributor.  A slot holds an epilogue
                // warp's 32 rows as [column unit j][row l] (16 KB); warps
                // h*4 + qq with qq < nq hold valid rows, each half's nq slots
                // contiguous.  Ring layout: [contributor][half][qq][j][l].
                const int vrows = (int)(args.M - mt * 128 < 128 ? args.M - mt * 128 : 128);
                const int nq = (vrows + 31) / 32;
                const int nc = (int)(c_end - blockIdx.x - 1);
                const bool staged = (int64_t)nc * nq * 2 * 16384 <= (int64_t)kStages * kStageBytes;
                bool synced = epi_sync(&ctrl->fix_arrive, kEpiWarps, abort_flag, args.status, 6);   // flags all seen
                if (staged) {
                    // epilogue warp we copies run r = we, we + 8, ... (r = ci * 2
                    // + half: nq slots of 16 KB), lane 0 alone; every warp
                    // arrives with its bytes before issuing them
                    const bool issue = got && synced && !*abort_flag;
                    const uint32_t fix_full = smem_u32(&ctrl->fix_full);
                    const uint32_t run_bytes = 16384u * (uint32_t)nq;
                    uint32_t my_bytes = 0;
                    if (issue)
                        for (int r = we; r < nc * 2; r += kEpiWarps) my_bytes += run_bytes;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(fix_full, my_bytes);
                        if (issue) {
                            asm volatile("fence.proxy.async.global;" ::: "memory");
                            for (int r = we; r < nc * 2; r += kEpiWarps) {
                                const int ci = r >> 1, hh = r & 1;
                                const float* src = args.sk_partials + ((int64_t)blockIdx.x + 1 + ci) * kSplitSlotFloats +
                                                   (int64_t)hh * 4 * 4096;
                                bulk_load(base + run_bytes * (uint32_t)r, src, run_bytes, fix_full);
                            }
                        }
                    }
                    __syncwarp();
                    // every warp's copies have landed (or, on giving up, they
                    // still land before the CTA's shared memory goes away)
                    if (!mbar_wait_warp(fix_full, 0, abort_flag, args.status, 6)) {
                        if (lane == 0) mbar_wait_teardown(fix_full, 0);
                        synced = false;
                    }
                }
                if (!got || !synced) break;
                if (staged) {
                    if (row < args.M) {
                        // this warp's slot in contributor ci: ring run ci * 2 + h, slot q
                        for (int ci = 0; ci < nc; ci++) {
                            const uint32_t src = base + 16384u * (uint32_t)((ci * 2 + h) * nq + q) + 16u * (uint32_t)lane;
#pragma unroll
                            for (int j = 0; j < 32; j++) {
                                const uint4 t = ld_shared_v4(src + 512u * (uint32_t)j);
                                v[4 * j] += __uint_as_float(t.x);
                                v[4 * j + 1] += __uint_as_float(t.y);
                                v[4 * j + 2] += __uint_as_float(t.z);
                                v[4 * j + 3] += __uint_as_float(t.w);
                            }
                        }
                    }
                } else if (nrows > 0 && nrows <= kFixRowsByLane) {
                    // few rows (decode): lane j fetches the 4 columns 4j..4j+3
                    // of each row from up to 4 partials at once, sums them
                    // in CTA order and hands them to the row's lane
                    for (int rr = 0; rr < nrows; rr++) {
                        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        for (int64_t c0 = (int64_t)blockIdx.x + 1; c0 < c_end; c0 += 4) {
                            float4 t[4];
#pragma unroll
                            for (int i = 0; i < 4; i++)
                                t[i] = c0 + i < c_end ? __ldcg(reinterpret_cast<const float4*>(
                                                                   args.sk_partials + (c0 + i) * kSplitSlotFloats) +
                                                               we * 1024 + lane * 32 + rr)
                                                         : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                            for (int i = 0; i < 4; i++) {
                                if (c0 + i < c_end) {
                                    acc.x += t[i].x;
                                    acc.y += t[i].y;
                                    acc.z += t[i].z;
                                    acc.w += t[i].w;
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 32; j++) {
                            const float ax = __shfl_sync(0xffffffffu, acc.x, j);
                            const float ay = __shfl_sync(0xffffffffu, acc.y, j);
                            const float az = __shfl_sync(0xffffffffu, acc.z, j);
                            const float aw = __shfl_sync(0xffffffffu, acc.w, j);
                            if (lane == rr) {
                                v[4 * j] += ax;
                                v[4 * j + 1] += ay;
                                v[4 * j + 2] += az;
                                v[4 * j + 3] += aw;
                            }
                        }
                    }
                } else if (row < args.M) {
                    for (int64_t c = (int64_t)blockIdx.x + 1; c < c_end; c++) {
                        const float4* slot =
                            reinterpret_cast<const float4*>(args.sk_partials + c * kSplitSlotFloats) + we * 1024 + lane;
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
#ifdef NVFP4_TRACE
                if (blockIdx.x == 0 && warp == kEpiWarp0 && lane == 0) g_trace_fix[0] = globaltimer();
#endif
                for (int64_t c = (int64_t)blockIdx.x + 1 + lane; c < c_end; c += 32)
                    args.sk_flags[c * kSplitFlagsPerCta + we] = 0;
                if (warp == kEpiWarp0 && lane == 0) TRACE(1216, ecount - 1);
            }
            // bf16 stores through the shared-memory staging (whole 256-byte
            // row segments per warp store); with few rows (a tile of at most
            // 64) the thread of each row stores it directly, which costs less
            // than the staging's rounds
            const uint32_t stage_arg = args.M > 64 ? epi_stage : 0u;
            if (kGrouped) {
                // the tile's expert scale; the A row's output row (rows past
                // the tile's valid rows are padding: sent past the last
                // output row, not stored); each row stored by its own thread
                const int4 td = args.grp_tiles[mt];
                const int64_t arow = (int64_t)td.y + q * 32 + lane;
                const int orow = q * 32 + lane < td.z ? args.grp_rowmap[arow] : -1;
                const float alpha_e = __fmul_rn(ga, args.gb0[td.x]);
                epilogue_row<false>(gargs, false, v, orow >= 0 ? (int64_t)orow : args.grp_out_rows, nt, h, alpha_e, alpha_e,
                             1.0f, wamax, 0u);
            } else {
                epilogue_row<kRope>(args, swiglu, v, row, nt, h, alpha0, alpha1, g_inter, wamax, stage_arg);
            }
            if (warp == kEpiWarp0 && lane == 0 && ecount == 1) TRACE_CTA(2);
            if (warp == kEpiWarp0 && lane == 0) TRACE_CTA(3);
        }
        if (args.epilogue == kEpiSwigluBf16) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wamax = fmaxf(wamax, __shfl_xor_sync(0xffffffffu, wamax, o));
            if (lane == 0) atomicMax(args.amax_ws, __float_as_uint(wamax));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b0, const CUtensorMap& map_b1,
                        const GemmArgs& args, int num_sms, cudaStream_t stream)
{
    static int attr_set_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set_for_device[dev]) {
        e = cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm_kernel<false, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    const bool swiglu = args.epilogue != kEpiBf16;
    const bool rope = args.rope_pos != nullptr;
    const int64_t num_m = (args.M + 127) / 128;
    const int64_t num_n = swiglu ? args.N / 128 : (args.N + 255) / 256;
    const int64_t tiles = num_m * num_n;
    const int64_t stages = (args.K / 64 + 3) / 4;
    // Whole tiles strided over min(tiles, SMs) CTAs, unless their last wave
    // leaves more than a tenth of the GPU idle and the tiles are deep in K:
    // then (given a workspace) every SM takes an equal share of the (tile,
    // K stage) units.  A tile split over CTAs costs its finishing CTA a few
    // microseconds of partial reads, which only deep tiles (>= 32 stages,
    // K >= 8192) repay; spreading shallow tiles over all SMs also makes
    // every CTA stream its own weight slab, which defeats the L2 sharing of
    // concurrently running whole tiles.
    // (Splitting the partial last wave of shallow-K tiles over the idle SMs
    // was measured slower: each CTA streams its K stages at a rate set by
    // its own load latency, so the idle SMs buy little, and the partials
    // and the split instantiation cost more.)
    const int64_t waves = (tiles + num_sms - 1) / num_sms;
    const bool split = !rope && args.sk_partials != nullptr && args.sk_flags != nullptr && num_sms <= kSplitMaxCtas &&
                       tiles * stages >= num_sms && tiles * 10 < waves * num_sms * 9 && stages >= 32 &&
                       tiles * stages < (int64_t)1 << 31;
    // programmatic launch: the CTAs may start on SMs the previous kernel has
    // left, and fetch weights before it completes when args.weights_early
    // split: at most as many CTAs per tile as let a finisher hold all its
    // contributors' valid partial rows in its ring at once (the fix-up's
    // one round trip); CTA c of G takes units [c*U/G, (c+1)*U/G)
    const int64_t tile_rows = args.M < 128 ? args.M : 128;
    const int64_t per_tile = 1 + (int64_t)kStages * kStageBytes / (2 * 16384 * ((tile_rows + 31) / 32));
    const int64_t split_ctas = tiles * per_tile < num_sms ? tiles * per_tile : num_sms;
    if (split)
        return launch_programmatic(gemm_kernel<true>, dim3((unsigned)split_ctas), dim3(kNumThreads), kSmemBytes, stream,
                                   map_a, map_b0, map_b1, args);
    if (rope)
        return launch_programmatic(gemm_kernel<false, false, true>, dim3((unsigned)(tiles < num_sms ? tiles : num_sms)),
                                   dim3(kNumThreads), kSmemBytes, stream, map_a, map_b0, map_b1, args);
    return launch_programmatic(gemm_kernel<false>, dim3((unsigned)(tiles < num_sms ? tiles : num_sms)),
                               dim3(kNumThreads), kSmemBytes, stream, map_a, map_b0, map_b1, args);
}

cudaError_t launch_gemm_grouped(const CUtensorMap& map_a, const CUtensorMap& map_b, const GemmArgs& args, int num_sms,
                                int64_t max_tiles, cudaStream_t stream)
{
    static int attr_set_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set_for_device[dev]) {
        e = cudaFuncSetAttribute(gemm_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    const int64_t grid = max_tiles < num_sms ? max_tiles : num_sms;
    return launch_programmatic(gemm_kernel<false, true>, dim3((unsigned)(grid > 0 ? grid : 1)), dim3(kNumThreads),
                               kSmemBytes, stream, map_a, map_b, map_b, args);
}

}  // namespace nvfp4

#ifdef NVFP4_TRACE
extern "C" int nvfp4_debug_trace_ctas(unsigned long long* out)
{
    if (cudaMemcpyFromSymbol(out, nvfp4::g_trace_cta, sizeof(nvfp4::g_trace_cta)) != cudaSuccess) return 4;
    return cudaMemcpyFromSymbol(out + 1024, nvfp4::g_trace_fix, sizeof(nvfp4::g_trace_fix)) == cudaSuccess ? 0 : 4;
}

extern "C" int nvfp4_debug_trace(unsigned long long* out, int n)
{
    if (n > 1280) n = 1280;
    return cudaMemcpyFromSymbol(out, nvfp4::g_trace, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : 4;
}
#endif
