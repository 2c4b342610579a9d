// Decode-regime NVFP4 GEMM on the tensor cores: out[m, n] = alpha *
// sum_k dA[m, k] dW[n, k] for a handful of activation rows (M <= 8), with
// the epilogues of the other GEMM kernels (bf16 [+ residual] [+ rotary
// embedding]; SwiGLU requantized to FP4, or bf16 with its amax).
//
// At M <= 8 the GEMM is a weight stream: every weight byte feeds at most
// eight multiply-adds, so the bound is HBM bandwidth.  The CUDA-core decode
// kernel spends about one instruction per weight code on decoding and
// integer dot products, which caps it near half of HBM speed; here the
// tensor pipe does that work and the SMs only move bytes.
// Sources: "PERFORMANCE -- verified hot-path audit and prioritized fixes"
// (the per-token decode step, its CUDA-graph item, roadmap E9); "tp>1
// prefill is host-bound" (the fp4 MLP of a decode step, T=1 vs T=5).
//
// Operand roles are swapped against the prefill kernels: the weights are
// the MMA's M side (128 weight rows per MMA), the activations its N side
// (N = 128, of which the first M columns are real).  One MMA of M=128,
// N=128, K=64 takes 64 tensor-pipe cycles for 4 KB of weight codes, about
// three times the rate at which HBM supplies an SM, so the pipe idles most
// of the time and the copies set the pace.  The activation rows of a
// stage (8 rows x 256 FP4, one 1 KB area per stage, the layout a 128-row
// operand has in its first 8 rows) are the B operand; its other 120 rows
// are whatever shared memory follows the area (later areas, weight codes):
// they only feed accumulator columns >= 8, which are never read.  Every
// 4-bit pattern is a finite E2M1 value and the activations' padding scale
// rows are zero, so those columns stay finite.
//
// Work split (stream-K): the weight rows are cut into parts of 128 rows
// (SwiGLU: gate block b is part 2b, up block b part 2b+1), each part into K
// stages of 256; CTA c of G = min(#SMs, units) takes the contiguous run
// [c U / G, (c+1) U / G) of the U = parts x stages units, so every SM
// streams the same number of weight bytes.  A run cut into segments at part
// boundaries leaves one fp32 partial per segment (M x 128 values) in the
// workspace; a per-block ticket counts the segments that have stored
// theirs, and the CTA taking the last ticket adds the block's partials in
// CTA order (deterministic), runs the epilogue and returns the ticket to
// zero.  No CTA waits for another.
//
// Warp roles (384 threads): warp 0 weight copies (2-D TMA of two 64-row
// boxes, 1-D bulk copy of the four scale tiles), warp 2 activation copies
// (one 8-row TMA box, the activation scale tiles), warp 1 tensor-memory
// allocation and the MMAs, warps 4-11 the epilogue (two teams of four, one
// per accumulator; each warp of a team one tensor-memory lane quarter);
// warp 3 idles.  A segment's ticket and partial reads are global round
// trips, slow while the weight stream loads the memory system: with two
// accumulators and two teams, one segment's epilogue overlaps the next
// segment's MMAs and the other team's epilogue.
#include <string.h>

#include "common.cuh"
#include "decode_epilogue.cuh"
#include "gemv.h"

namespace nvfp4 {
namespace {

constexpr int kStages = 8;
constexpr int kWBytes = 128 * 128;            // weight codes of a stage: 128 rows x 256 FP4
constexpr int kBoxBytes = kCodeBoxRows * 128; // one 64-row weight box
constexpr int kSfTile = 512;                  // 128 rows x 4 scales (one K-step of 64)
constexpr int kSfBytes = 4 * kSfTile;         // the 4 K-steps of a stage
constexpr int kActBytes = kDecodeTcMaxRows * 128;
constexpr int kOffW = kStages * kActBytes;
constexpr int kOffWsf = kOffW + kStages * kWBytes;
constexpr int kOffAsf = kOffWsf + kStages * kSfBytes;
constexpr int kOffCtrl = kOffAsf + kStages * kSfBytes;
constexpr int kCtrlBytes = 256;
constexpr int kOffRacc = kOffCtrl + kCtrlBytes;
constexpr int kRaccBytes = 2 * 256 * kDecodeTcMaxRows * 4;   // one block's dot products per epilogue team
constexpr int kSmemBytes = kOffRacc + kRaccBytes + 1024;     // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(kActBytes % 1024 == 0, "activation areas start on 1024-byte swizzle atoms");
static_assert((kStages - 1) * kActBytes + 128 * 128 <= kOffCtrl, "the B operand's 128 rows stay inside the ring");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;            // two accumulators of 128 columns (segments alternate)
constexpr uint32_t kSfColsPerStage = 32;      // per K-step: weight scales +0..3, activation scales +4..7
static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");

constexpr int kNumThreads = 384;
constexpr int kWarpW = 0, kWarpMma = 1, kWarpA = 2, kEpiWarp0 = 4;
constexpr int kEpiThreads = 128;              // one epilogue team: 4 warps, one per lane quarter
constexpr int kMaxContrib = 8;                // partials fetched together by the finishing CTA

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1, UE4M3 scales,
// K-major A and B, N = 128 (bits 17-22 = N/8), M = 128 (bits 24-28 = M/16).
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

struct Ctrl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t teardown;
    uint32_t tmem_base;
    int abort_flag;
    int last[2];       // epilogue team t: this CTA took the block's last ticket
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

#ifdef NVFP4_TRACE_DECODE
// Debug timeline (built only with -DNVFP4_TRACE_DECODE): global timer (ns)
// per CTA at [0] entry, [1] set-up done, [2] first stage full (MMA warp),
// [3] last segment issued, [4] first accumulator full (epilogue), [5] last
// ticket taken, [6] last block finished (if any), [7] exit.  Totals (ns) at
// [8] weight producer waiting for a free slot, [9] MMA waiting for a full
// stage, [10] MMA waiting for a free accumulator, [11] epilogue from
// accumulator drained to segment done; of that, [12] partial stored, [13]
// ticket, [14] partials combined, [15] block epilogue.
__device__ unsigned long long g_dtrace[256][16];
#define DTRACE(k) \
    do { if (blockIdx.x < 256) g_dtrace[blockIdx.x][k] = globaltimer(); } while (0)
#define DT_T0() const uint64_t dt0_ = globaltimer()
#define DT_ADD(k) \
    do { if (blockIdx.x < 256 && (threadIdx.x & 31) == 0) g_dtrace[blockIdx.x][k] += globaltimer() - dt0_; } while (0)
#define DT_MARK(k, tvar)                                                           \
    do {                                                                          \
        const uint64_t now_ = globaltimer();                                      \
        if (blockIdx.x < 256 && et == 0) g_dtrace[blockIdx.x][k] += now_ - tvar; \
        tvar = now_;                                                              \
    } while (0)
#else
#define DTRACE(k) do { } while (0)
#define DT_T0() do { } while (0)
#define DT_ADD(k) do { } while (0)
#define DT_MARK(k, tvar) do { } while (0)
#endif

struct DecodeTcParams {
    CUtensorMap map_a;    // activation codes, boxes of kDecodeTcMaxRows rows
    CUtensorMap map_b0;   // weights (gate for SwiGLU)
    CUtensorMap map_b1;   // up weights (SwiGLU)
    GemmArgs g;
    int ks;               // K stages per part
    int maxseg;           // partial slots per CTA
    // first unit of CTA c's run (c <= grid), and the part of CTA c's first
    // unit (its partial slot 0): tables, so that no division runs on the
    // device
    int32_t run_b[kSplitMaxCtas + 1];
    int32_t part_first[kSplitMaxCtas];
};

// The CTA whose run holds unit u: the last c < grid with run_b[c] <= u.
__device__ __forceinline__ int owner_of_unit(const DecodeTcParams& P, int grid, int u)
{
    int lo = 0, hi = grid - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.run_b[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int atom_add_acq_rel(int* p, int v)
{
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v)
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = __uint_as_float(r[i]);
}

// Named barrier of an epilogue team (barrier 1 + team); epi_any: the same
// barrier, returning whether any of its threads passed true (a decision the
// team's four warps take alike).
__device__ __forceinline__ void epi_sync(int team)
{
    asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "n"(kEpiThreads) : "memory");
}
__device__ __forceinline__ bool epi_any(int team, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(1 + team), "n"(kEpiThreads)
        : "memory");
    return r != 0;
}

// One full stage (4 K-steps): its 8 scale-tile copies shared -> tensor
// memory (weight tile j to column sfc + 8j, activation tile j to sfc + 8j +
// 4), its 4 MMAs and the commit that frees the stage, from one converged
// warp with a single elect.sync (see stage_issue_1sm).
//   w_lo / a_lo / sw_hi: weight and activation code descriptors of the stage
//   wsf_lo / asf_lo / sf_hi: scale-tile descriptors (tiles 512 B apart)
__device__ __forceinline__ void stage_issue_decode(uint32_t acc, uint32_t sfc, uint32_t wsf_lo, uint32_t asf_lo,
                                                   uint32_t sf_hi, uint32_t w_lo, uint32_t a_lo, uint32_t sw_hi,
                                                   uint32_t acc0, uint32_t bar)
{
    asm volatile(
        "{\n"
        " .reg .pred e, p, pt;\n"
        " .reg .b32 el, t, u, lo;\n"
        " .reg .b64 d, da, db;\n"
        " elect.sync el|e, 0xffffffff;\n"
        " setp.ne.b32 p, %8, 0;\n"
        " setp.eq.b32 pt, 0, 0;\n"
        " add.u32 t, %1, 0; add.u32 lo, %2, 0; mov.b64 d, {lo, %4};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 4; add.u32 lo, %3, 0; mov.b64 d, {lo, %4};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 8; add.u32 lo, %2, 32; mov.b64 d, {lo, %4};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 12; add.u32 lo, %3, 32; mov.b64 d, {lo, %4};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 16; add.u32 lo, %2, 64; mov.b64 d, {lo, %4};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 20; add.u32 lo, %3, 64; mov.b64 d, {lo, %4};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 24; add.u32 lo, %2, 96; mov.b64 d, {lo, %4};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 28; add.u32 lo, %3, 96; mov.b64 d, {lo, %4};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 lo, %5, 0; mov.b64 da, {lo, %7}; add.u32 lo, %6, 0; mov.b64 db, {lo, %7};\n"
        " add.u32 t, %1, 0; add.u32 u, %1, 4;\n"
        " @e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %9, [t], [u], p;\n"
        " add.u32 lo, %5, 2; mov.b64 da, {lo, %7}; add.u32 lo, %6, 2; mov.b64 db, {lo, %7};\n"
        " add.u32 t, %1, 8; add.u32 u, %1, 12;\n"
        " @e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %9, [t], [u], pt;\n"
        " add.u32 lo, %5, 4; mov.b64 da, {lo, %7}; add.u32 lo, %6, 4; mov.b64 db, {lo, %7};\n"
        " add.u32 t, %1, 16; add.u32 u, %1, 20;\n"
        " @e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %9, [t], [u], pt;\n"
        " add.u32 lo, %5, 6; mov.b64 da, {lo, %7}; add.u32 lo, %6, 6; mov.b64 db, {lo, %7};\n"
        " add.u32 t, %1, 24; add.u32 u, %1, 28;\n"
        " @e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %9, [t], [u], pt;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n"
        "}\n" ::"r"(acc),
        "r"(sfc), "r"(wsf_lo), "r"(asf_lo), "r"(sf_hi), "r"(w_lo), "r"(a_lo), "r"(sw_hi), "r"(acc0), "r"(kIdesc),
        "r"(bar)
        : "memory");
}

__global__ void __launch_bounds__(kNumThreads, 1) decode_tc_kernel(const __grid_constant__ DecodeTcParams prm)
{
    extern __shared__ uint8_t smem_raw[];
    if (threadIdx.x == 0) DTRACE(0);
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_addr);
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + kOffCtrl);
    float* racc = reinterpret_cast<float*>(smem + kOffRacc);
    volatile int* abort_flag = &ctrl->abort_flag;

    const GemmArgs& args = prm.g;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int M = (int)args.M;
    const bool swiglu = args.epilogue != kEpiBf16;
    const int ks = prm.ks;
    const int num_kk = (int)(args.K / 64);
    const int grid = (int)gridDim.x;
    const int cta = blockIdx.x;
    const int u_beg = prm.run_b[cta], u_end = prm.run_b[cta + 1];

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(smem_u32(&ctrl->full[s]), 1);   // the weight producer's arrival + all bytes
            mbar_init(smem_u32(&ctrl->empty[s]), 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(smem_u32(&ctrl->acc_full[a]), 1);
            mbar_init(smem_u32(&ctrl->acc_empty[a]), kEpiThreads / 32);
        }
        mbar_init(smem_u32(&ctrl->teardown), 1);
        ctrl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kWarpW && lane == 0) {
        prefetch_tmap(&prm.map_b0);
        if (swiglu) prefetch_tmap(&prm.map_b1);
    }
    if (warp == kWarpA && lane == 0) prefetch_tmap(&prm.map_a);
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    griddep_launch_dependents();
    if (threadIdx.x == 0) DTRACE(1);

    if (warp == kWarpW || warp == kWarpA) {
        // ---------------------------------------------------------- copies
        // Both producers walk the same units and wait on the same empty
        // barriers; the weight producer alone arrives on a stage's full
        // barrier, with the byte count of both producers' copies (the
        // activation copies only complete bytes on it).  The weights may be
        // fetched before the previous kernel completes when the caller
        // vouches they were complete before it; the activations never.
        const bool wside = warp == kWarpW;
        if (!wside || !args.weights_early) griddep_wait();
        const uint64_t pol = wside ? l2_policy_evict_first() : l2_policy_evict_last();
        const uint32_t full0 = smem_u32(&ctrl->full[0]);
        const uint32_t empty0 = smem_u32(&ctrl->empty[0]);
        int s = 0;
        uint32_t ph = 0, issued = 0, issued_ph = 0;
        bool ok = true;
        int p = u_beg / ks, kb = u_beg - p * ks;   // the unit's part and K stage
        for (int u = u_beg; u < u_end; u++) {
            {
                DT_T0();
                const bool w_ok = mbar_wait_warp(empty0 + 8u * (uint32_t)s, ph ^ 1u, abort_flag, args.status, 21);
                if (wside) DT_ADD(8);
                if (!w_ok) {
                    ok = false;
                    break;
                }
            }
            const uint32_t nk = (uint32_t)min(4, num_kk - 4 * kb);   // K-steps of this stage
            const uint32_t full = full0 + 8u * (uint32_t)s;
            if (lane == 0) {
                if (wside) {
                    const int blk = swiglu ? p >> 1 : p;
                    const bool up = swiglu && (p & 1);
                    const int32_t y = blk * 128;
                    const bool box1 = y + kCodeBoxRows < args.N;   // else its rows are past N: not fetched
                    mbar_arrive_expect_tx(full, (uint32_t)kActBytes + 2u * nk * kSfTile + (box1 ? 2u : 1u) * kBoxBytes);
                    const CUtensorMap* map = up ? &prm.map_b1 : &prm.map_b0;
                    const uint32_t dst = base + kOffW + (uint32_t)s * kWBytes;
                    tma_load_2d(dst, map, full, kb * 128, y, pol);
                    if (box1) tma_load_2d(dst + kBoxBytes, map, full, kb * 128, y + kCodeBoxRows, pol);
                    const uint8_t* sf = (up ? args.sfb1 : args.sfb0) + (int64_t)blk * args.sfb_tile_stride +
                                        (size_t)kb * kSfBytes;
                    bulk_load(base + kOffWsf + (uint32_t)s * kSfBytes, sf, nk * kSfTile, full);
                } else {
                    tma_load_2d(base + (uint32_t)s * kActBytes, &prm.map_a, full, kb * 128, 0, pol);
                    bulk_load(base + kOffAsf + (uint32_t)s * kSfBytes, args.sfa + (size_t)kb * kSfBytes, nk * kSfTile,
                              full);
                }
            }
            __syncwarp();
            issued |= 1u << s;
            issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
            if (++s == kStages) {
                s = 0;
                ph ^= 1u;
            }
            if (++kb == ks) {
                kb = 0;
                ++p;
            }
        }
        if (!ok && lane == 0) {
            // stopped early: let the copies already issued land before the
            // CTA's shared memory goes away (bounded)
            for (int i = 0; i < kStages; i++)
                if (issued & (1u << i)) mbar_wait_teardown(full0 + 8u * (uint32_t)i, (issued_ph >> i) & 1u);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------- MMA
        // K-major, 128-byte swizzle, 8-row groups 1024 B apart (codes); no
        // swizzle, 16-byte rows, 8-row groups 128 B apart (scales)
        const uint64_t dsw = make_smem_desc(base, 16, 1024, 2);
        const uint64_t dsf = make_smem_desc(base + kOffWsf, 128, 128, 0);
        const uint32_t sw_lo = (uint32_t)dsw, sw_hi = (uint32_t)(dsw >> 32);
        const uint32_t sf_lo = (uint32_t)dsf, sf_hi = (uint32_t)(dsf >> 32);
        const uint32_t full0 = smem_u32(&ctrl->full[0]);
        const uint32_t empty0 = smem_u32(&ctrl->empty[0]);
        int s = 0;
        uint32_t ph = 0, acc_ph = 0;   // acc_ph: bit a = phase of accumulator a
        int acc = 0;                   // accumulator of the current segment
        bool ok = true;
        bool first = true;
        int u = u_beg;
        while (ok && u < u_end) {
            // segment: the stages [kb0, kb1) of one part
            const int p = u / ks;
            const int kb0 = u - p * ks;
            const int kb1 = u_end - u < ks - kb0 ? kb0 + (u_end - u) : ks;
            u += kb1 - kb0;
            {
                DT_T0();
                const bool a_ok = mbar_wait_warp(smem_u32(&ctrl->acc_empty[acc]), ((acc_ph >> acc) & 1u) ^ 1u,
                                                 abort_flag, args.status, 22);
                DT_ADD(10);
                if (!a_ok) break;
            }
            tc_fence_after();
            const uint32_t dacc = tmem + (uint32_t)acc * 128u;
            for (int kb = kb0; kb < kb1; kb++) {
                {
                    DT_T0();
                    const bool f_ok = mbar_wait_warp(full0 + 8u * (uint32_t)s, ph, abort_flag, args.status, 23);
                    DT_ADD(9);
                    if (!f_ok) {
                        ok = false;
                        break;
                    }
                }
                if (first && lane == 0) DTRACE(2);
                first = false;
                tc_fence_after();
                const int nk = min(4, num_kk - 4 * kb);
                const uint32_t w_lo = sw_lo + ((uint32_t)(kOffW + s * kWBytes) >> 4);
                const uint32_t a_lo = sw_lo + ((uint32_t)(s * kActBytes) >> 4);
                const uint32_t wsf_lo = sf_lo + ((uint32_t)(s * kSfBytes) >> 4);
                const uint32_t asf_lo = wsf_lo + ((uint32_t)(kOffAsf - kOffWsf) >> 4);
                const uint32_t sfc = tmem + kAccCols + (uint32_t)s * kSfColsPerStage;
                const uint32_t bar = empty0 + 8u * (uint32_t)s;
                if (nk == 4) {
                    stage_issue_decode(dacc, sfc, wsf_lo, asf_lo, sf_hi, w_lo, a_lo, sw_hi, kb != kb0 ? 1u : 0u, bar);
                } else {
                    // K tail: a last stage of fewer than 4 K-steps
                    for (int k = 0; k < nk; k++) {
                        tmem_copy_sf_warp(sfc + 8u * k, desc_from(wsf_lo + 32u * k, sf_hi));
                        tmem_copy_sf_warp(sfc + 8u * k + 4u, desc_from(asf_lo + 32u * k, sf_hi));
                    }
                    for (int k = 0; k < nk; k++)
                        mma_mxf4nvf4_warp(dacc, desc_from(w_lo + 2u * k, sw_hi), desc_from(a_lo + 2u * k, sw_hi),
                                          kIdesc, sfc + 8u * k, sfc + 8u * k + 4u, (kb != kb0 || k != 0) ? 1u : 0u);
                    mma_commit_warp(bar);
                }
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            mma_commit_warp(smem_u32(&ctrl->acc_full[acc]));
            acc_ph ^= 1u << acc;
            acc ^= 1;
            if (lane == 0) DTRACE(3);
        }
        // every MMA issued has completed before teardown
        mma_commit_warp(smem_u32(&ctrl->teardown));
        if (lane == 0) mbar_wait_teardown(smem_u32(&ctrl->teardown), 0);
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        // -------------------------------------------------------- epilogue
        // Team t takes the segments of accumulator t (every other segment
        // of the CTA).
        griddep_wait();   // workspace, residual, outputs, scales: after the previous kernel
        const int team = (warp - kEpiWarp0) >> 2;
        const int q = warp & 3;                                                // tensor-memory lane quarter
        const int et = (threadIdx.x - kEpiWarp0 * 32) & (kEpiThreads - 1);   // weight row: q * 32 + lane
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)team * 128u;
        racc += team * 256 * kDecodeTcMaxRows;
        const int64_t slot_floats = (int64_t)128 * M;
        const int nparts = swiglu ? 2 : 1;
        const EpiScalars es = epi_scalars(args);   // read while the stream runs
        uint32_t acc_ph = 0;   // phase of this team's accumulator
        int seg = 0;           // segment index in the CTA (team seg % 2 takes it)
        bool first = true;
        int u = u_beg;
        while (u < u_end) {
            const int p = u / ks;
            const int kb0 = u - p * ks;
            const int kb1 = u_end - u < ks - kb0 ? kb0 + (u_end - u) : ks;
            u += kb1 - kb0;
            if ((seg++ & 1) != team) continue;   // the other team's segment
            const bool got = mbar_wait_warp<true>(smem_u32(&ctrl->acc_full[team]), acc_ph, abort_flag, args.status, 24);
            float v[8];
            if (got) {
                tc_fence_after();
                tmem_ld8(lane_addr, v);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctrl->acc_empty[team]));
            }
            // a wait that gave up in any warp of the team stops all four
            // here, before the team's next named barrier
            if (epi_any(team, !got)) break;
            if (first && et == 0 && team == 0) DTRACE(4);
            first = false;
            acc_ph ^= 1u;
#ifdef NVFP4_TRACE_DECODE
            uint64_t dtm = globaltimer();
            const uint64_t dt_seg0 = dtm;
#endif

            // this segment's partial: [m][row] in the CTA's slot of part p
            float* slot = args.sk_partials + ((int64_t)cta * prm.maxseg + (p - prm.part_first[cta])) * slot_floats;
#pragma unroll
            for (int m = 0; m < kDecodeTcMaxRows; m++)
                if (m < M) __stcg(slot + m * 128 + et, v[m]);
            epi_sync(team);
            DT_MARK(12, dtm);
            // the block's ticket (acquire-release: the partials stored before
            // the barrier are visible to whoever takes the last)
            const int blk = swiglu ? p >> 1 : p;
            const int pfirst = swiglu ? 2 * blk : blk;   // the block's first part
            if (et == 0) {
                int expected = 0;
                for (int i = 0; i < nparts; i++) {
                    const int U0 = (pfirst + i) * ks;
                    expected += owner_of_unit(prm, grid, U0 + ks - 1) - owner_of_unit(prm, grid, U0) + 1;
                }
                int* ticket = args.sk_flags + blk;
                const int last = atom_add_acq_rel(ticket, 1) == expected - 1;
                if (last) *ticket = 0;   // every segment has arrived: ready for the next launch
                ctrl->last[team] = last;
                DTRACE(5);
            }
            epi_sync(team);
            DT_MARK(13, dtm);
            if (ctrl->last[team]) {
                // sum the block's partials in CTA order, up to kMaxContrib
                // loads in flight
                for (int i = 0; i < nparts; i++) {
                    const int pp = pfirst + i;
                    const int c0 = owner_of_unit(prm, grid, pp * ks), c1 = owner_of_unit(prm, grid, pp * ks + ks - 1);
                    float sum[kDecodeTcMaxRows];
#pragma unroll
                    for (int m = 0; m < kDecodeTcMaxRows; m++) sum[m] = 0.0f;
                    for (int cb = c0; cb <= c1; cb += kMaxContrib) {
                        float t[kMaxContrib][kDecodeTcMaxRows];
#pragma unroll
                        for (int k = 0; k < kMaxContrib; k++) {
                            const int c = cb + k;
                            const float* src =
                                c <= c1 ? args.sk_partials +
                                              ((int64_t)c * prm.maxseg + (pp - prm.part_first[c])) * slot_floats + et
                                        : nullptr;
#pragma unroll
                            for (int m = 0; m < kDecodeTcMaxRows; m++)
                                t[k][m] = (src && m < M) ? __ldcg(src + m * 128) : 0.0f;
                        }
#pragma unroll
                        for (int k = 0; k < kMaxContrib; k++)
                            if (cb + k <= c1) {
#pragma unroll
                                for (int m = 0; m < kDecodeTcMaxRows; m++) sum[m] = __fadd_rn(sum[m], t[k][m]);
                            }
                    }
#pragma unroll
                    for (int m = 0; m < kDecodeTcMaxRows; m++)
                        if (m < M) racc[(i * 128 + et) * M + m] = sum[m];
                }
                epi_sync(team);
                DT_MARK(14, dtm);
                const int64_t n0 = (int64_t)blk * 128;
                const int C = (int)(args.N - n0 < 128 ? args.N - n0 : 128);
                decode_epilogue<kEpiThreads>(args, es, racc, M, n0, C, et);
                epi_sync(team);   // the block's outputs stored; racc is rewritten by the next block
                if (et == 0) DTRACE(6);
                DT_MARK(15, dtm);
            }
#ifdef NVFP4_TRACE_DECODE
            if (cta < 256 && et == 0) g_dtrace[cta][11] += globaltimer() - dt_seg0;
#endif
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0) DTRACE(7);
}

// Grid, units and partial slots per CTA of a launch.
struct DecodeTcShape {
    int64_t units, grid, ks, blocks;
    int maxseg;
};

DecodeTcShape decode_tc_shape(const GemmArgs& a, int num_sms)
{
    DecodeTcShape d{};
    d.blocks = (a.N + 127) / 128;
    const int64_t parts = a.epilogue != kEpiBf16 ? 2 * d.blocks : d.blocks;
    d.ks = (a.K / 64 + 3) / 4;
    d.units = parts * d.ks;
    d.grid = d.units < num_sms ? d.units : num_sms;
    if (d.grid < 1) return d;
    // parts a CTA's run touches, at most (walked exactly: at most 256 CTAs)
    for (int64_t c = 0; c < d.grid; c++) {
        const int64_t b = c * d.units / d.grid, e = (c + 1) * d.units / d.grid;
        const int64_t n = (e - 1) / d.ks - b / d.ks + 1;
        if (n > d.maxseg) d.maxseg = (int)n;
    }
    return d;
}

}  // namespace

bool decode_tc_eligible(const GemmArgs& a, int num_sms)
{
    if (a.M < 1 || a.M > kDecodeTcMaxRows || num_sms < 1 || num_sms > kSplitMaxCtas) return false;
    if (!a.sk_partials || !a.sk_flags || a.grp_count) return false;
    if (a.epilogue != kEpiBf16 && a.N % 128 != 0) return false;
    if (a.K < 64 || a.K % 64 != 0 || a.N < 16 || a.N % 16 != 0) return false;
    const DecodeTcShape d = decode_tc_shape(a, num_sms);
    if (d.grid < 1 || d.units >= ((int64_t)1 << 31)) return false;
    if (d.blocks > (int64_t)kSplitMaxCtas * kSplitFlagsPerCta) return false;   // one ticket word per block
    // partial slots: grid x maxseg x (M x 128) floats within the workspace's slots
    return d.grid * d.maxseg * 128 * a.M * 4 <= (int64_t)split_partial_bytes(num_sms);
}

cudaError_t launch_decode_tc(const CUtensorMap& map_a, const CUtensorMap& map_b0, const CUtensorMap& map_b1,
                             const GemmArgs& args, int num_sms, cudaStream_t stream)
{
    if (!decode_tc_eligible(args, num_sms)) return cudaErrorInvalidValue;
    static int attr_set_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set_for_device[dev]) {
        e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    const DecodeTcShape d = decode_tc_shape(args, num_sms);
    DecodeTcParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.map_a = map_a;
    prm.map_b0 = map_b0;
    prm.map_b1 = map_b1;
    prm.g = args;
    prm.ks = (int)d.ks;
    prm.maxseg = d.maxseg;
    for (int64_t c = 0; c <= d.grid; c++) prm.run_b[c] = (int32_t)(c * d.units / d.grid);
    for (int64_t c = 0; c < d.grid; c++) prm.part_first[c] = (int32_t)(prm.run_b[c] / d.ks);
    return launch_programmatic(decode_tc_kernel, dim3((unsigned)d.grid), dim3(kNumThreads), kSmemBytes, stream, prm);
}

}  // namespace nvfp4

#ifdef NVFP4_TRACE_DECODE
extern "C" int nvfp4_debug_decode_trace(unsigned long long* out)
{
    return cudaMemcpyFromSymbol(out, nvfp4::g_dtrace, sizeof(nvfp4::g_dtrace)) == cudaSuccess ? 0 : 4;
}

extern "C" int nvfp4_debug_decode_trace_clear(void)
{
    static unsigned long long zero[256 * 16];
    return cudaMemcpyToSymbol(nvfp4::g_dtrace, zero, sizeof(zero)) == cudaSuccess ? 0 : 4;
}
#endif
