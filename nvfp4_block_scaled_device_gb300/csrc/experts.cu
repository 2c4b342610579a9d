// Expert-indexed NVFP4 GEMM (the routed projection of a mixture-of-experts
// layer, MUL_MAT_ID in llama.cpp's terms): every routed (token, slot) pair
// is one GEMM row of its token's activations with its expert's weights.
// Three launches, no host synchronisation (the routing table stays on the
// device):
//   1. route_kernel: counts the pairs per expert, lays out each expert's
//      rows as a segment padded to 128 rows, numbers the pairs within their
//      expert, and writes the M-tile table and the row maps;
//   2. gather_kernel: copies each pair's token row (codes and its scales, in
//      the 128 x 4 scale layout) into the expert-sorted operand;
//   3. the 1-SM tcgen05 GEMM in its grouped mode over the tile table.
// The order of the pairs within an expert depends on the order of atomic
// increments, but every output row depends only on its own token row and
// expert, so the outputs do not.
//
// Sources: "CUDA: NVFP4 prefill on Blackwell leaves ~1.45x performance on
// the table", the MUL_MAT_ID tests its patch passes; "PERFORMANCE --
// verified hot-path audit and prioritized fixes", the routed experts run
// without a host round trip (its CUDA-graph item lists a host read of the
// routing table, topk_ids.max().item(), as a blocker).
#include "common.cuh"
#include "internal.h"
#include "nvfp4.h"

namespace nvfp4 {

namespace {

constexpr int kRouteThreads = 1024;
constexpr int kMaxExperts = 4096;                          // the API's bound on E
constexpr int kExpertsPerThread = kMaxExperts / kRouteThreads;
constexpr int kIdsAhead = 4;                               // id loads in flight per thread

// One block.  The per-expert counts and cursors live in shared memory
// (atomics there, not on global words that every pair of a popular expert
// would serialise on; aggregating a warp's equal ids with match.any first
// was slower), and the experts' tile offsets come from a block-wide prefix
// sum; an expert's rows start at 128 x its first tile.
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_kernel(const int32_t* __restrict__ ids, int64_t pairs, int64_t topk, int E, int* __restrict__ hdr,
                 int4* __restrict__ tiles, int* __restrict__ rowmap, int* __restrict__ src, int* status)
{
    __shared__ int s_count[kMaxExperts];     // pairs per expert, then the cursor within its segment
    __shared__ int s_tile0[kMaxExperts];     // the expert's first tile
    __shared__ int s_warp[kRouteThreads / 32];
    griddep_wait();                 // the ids may come from the previous kernel
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    for (int e = t; e < E; e += kRouteThreads) s_count[e] = 0;
    __syncthreads();
    bool bad = false;
    for (int64_t i0 = 0; i0 < pairs; i0 += kRouteThreads * kIdsAhead) {
        int ev[kIdsAhead];
#pragma unroll
        for (int u = 0; u < kIdsAhead; u++) {      // the loads first, one round trip for all
            const int64_t i = i0 + u * kRouteThreads + t;
            ev[u] = i < pairs ? __ldg(ids + i) : 0;
            if (i < pairs && (ev[u] < 0 || ev[u] >= E)) bad = true;
            if (i >= pairs || ev[u] >= E) ev[u] = -1;
        }
#pragma unroll
        for (int u = 0; u < kIdsAhead; u++) {
            const int e = ev[u];
            if (e >= 0) atomicAdd(&s_count[e], 1);
        }
    }
    if (bad) {
        hdr[2] = 1;
        if (status) atomicCAS(status, 0, NVFP4_ERR_INVALID_ARG * 100 + 30);
    }
    __syncthreads();
    // exclusive prefix sum of the experts' tile counts: thread t takes the
    // experts kExpertsPerThread * t .. + kExpertsPerThread - 1
    int n_tiles[kExpertsPerThread];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < kExpertsPerThread; j++) {
        const int e = t * kExpertsPerThread + j;
        n_tiles[j] = e < E ? (s_count[e] + 127) / 128 : 0;
        sum += n_tiles[j];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;                       // inclusive over warps
    }
    __syncthreads();
    int run = (warp ? s_warp[warp - 1] : 0) + incl - sum;
#pragma unroll
    for (int j = 0; j < kExpertsPerThread; j++) {
        const int e = t * kExpertsPerThread + j;
        if (e < E) s_tile0[e] = run;
        run += n_tiles[j];
    }
    if (t == 0) {
        hdr[0] = s_warp[kRouteThreads / 32 - 1];
        hdr[1] = 128 * s_warp[kRouteThreads / 32 - 1];
    }
    __syncthreads();
    // the tile table (tile by tile: consecutive threads, consecutive
    // entries); a tile's expert is the last one whose first tile is at or
    // before it.  Padding rows are not marked: the gather and the GEMM's
    // epilogue take a tile's valid rows from its entry.
    const int n_tiles_all = s_warp[kRouteThreads / 32 - 1];
    for (int tl = t; tl < n_tiles_all; tl += kRouteThreads) {
        int lo = 0, hi = E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_tile0[mid] <= tl) lo = mid; else hi = mid - 1;
        }
        tiles[tl] = make_int4(lo, 128 * tl, min(128, s_count[lo] - 128 * (tl - s_tile0[lo])), 0);
    }
    __syncthreads();
    for (int e = t; e < E; e += kRouteThreads) s_count[e] = 0;   // now the cursors
    __syncthreads();
    // each pair's row within its expert's segment
    for (int64_t i0 = 0; i0 < pairs; i0 += kRouteThreads * kIdsAhead) {
        int ev[kIdsAhead];
#pragma unroll
        for (int u = 0; u < kIdsAhead; u++) {
            const int64_t i = i0 + u * kRouteThreads + t;
            ev[u] = i < pairs ? __ldg(ids + i) : -1;
            if (ev[u] >= E) ev[u] = -1;
        }
#pragma unroll
        for (int u = 0; u < kIdsAhead; u++) {
            const int64_t i = i0 + u * kRouteThreads + t;
            const int e = ev[u];
            if (e >= 0) {
                const int r = 128 * s_tile0[e] + atomicAdd(&s_count[e], 1);
                rowmap[r] = (int)i;
                src[r] = (int)i / (int)topk;   // pairs < 2^31
            }
        }
    }
    griddep_launch_dependents();
}

// One 32-lane warp per sorted row: the codes (16-byte vectors) and the
// 32-bit scale words (four consecutive 16-element blocks each) of its
// token row.  Padding rows (past their tile's valid rows) are left as they
// are: each GEMM output row depends on its own A row only, and those rows
// are never stored.
__global__ void __launch_bounds__(256) gather_kernel(const uint8_t* __restrict__ a_codes, int64_t lda,
                                                     const uint8_t* __restrict__ a_sf, int64_t K,
                                                     const int* __restrict__ hdr, const int4* __restrict__ tiles,
                                                     const int* __restrict__ src, uint8_t* __restrict__ p_codes,
                                                     uint8_t* __restrict__ p_sf)
{
    griddep_wait();                 // the tables of route_kernel
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    const int lane = threadIdx.x & 31;
    const int64_t rows = hdr[1];
    const int64_t kb = K / 16;                  // scale columns (a multiple of 4: K % 64 == 0)
    const int64_t nvec = K / 32;                // 16-byte vectors of codes per row
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
        if ((r & 127) >= tiles[r >> 7].z) continue;   // a padding row (uniform over the warp)
        const int s = src[r];
        const uint4* in = reinterpret_cast<const uint4*>(a_codes + (int64_t)s * lda);
        uint4* out = reinterpret_cast<uint4*>(p_codes + r * (K / 2));
        for (int64_t v = lane; v < nvec; v += 32) out[v] = in[v];
        for (int64_t c4 = lane; c4 < kb / 4; c4 += 32)
            *reinterpret_cast<uint32_t*>(p_sf + sf_offset(r, c4 * 4, kb)) =
                *reinterpret_cast<const uint32_t*>(a_sf + sf_offset(s, c4 * 4, kb));
    }
    griddep_launch_dependents();
}

}  // namespace

ExpertsLayout experts_layout(int64_t T, int64_t topk, int64_t K, int64_t E)
{
    ExpertsLayout L;
    const int64_t pairs = T * topk;
    const int64_t pad_experts = E < pairs ? E : pairs;
    L.max_rows = (pairs + 127 * pad_experts + 127) / 128 * 128;
    L.max_tiles = L.max_rows / 128;
    auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
    size_t off = 256;                               // header words
    L.tiles = off;
    off += al((size_t)L.max_tiles * 16);
    L.rowmap = off;
    off += al((size_t)L.max_rows * 4);
    L.src = off;
    off += al((size_t)L.max_rows * 4);
    L.codes = off;
    off += al((size_t)L.max_rows * (size_t)(K / 2));
    L.sf = off;
    off += al((size_t)L.max_rows * (size_t)((K / 16 + 3) / 4 * 4));
    L.total = off;
    return L;
}

cudaError_t launch_experts(const uint8_t* a_codes, int64_t lda, const uint8_t* a_sf, const float* a_g, int64_t T,
                           int64_t K, const uint8_t* w_codes, int64_t ldw, const uint8_t* w_sf, const float* w_g,
                           int64_t N, int64_t E, const int32_t* ids, int64_t topk, __nv_bfloat16* out, int64_t ldo,
                           uint8_t* ws, const CUtensorMap& map_a, const CUtensorMap& map_b, int* status, int num_sms,
                           cudaStream_t stream)
{
    const ExpertsLayout L = experts_layout(T, topk, K, E);
    int* hdr = reinterpret_cast<int*>(ws);
    int4* tiles = reinterpret_cast<int4*>(ws + L.tiles);
    int* rowmap = reinterpret_cast<int*>(ws + L.rowmap);
    int* src = reinterpret_cast<int*>(ws + L.src);
    uint8_t* p_codes = ws + L.codes;
    uint8_t* p_sf = ws + L.sf;
    const int64_t pairs = T * topk;
    cudaError_t e = launch_programmatic(route_kernel, dim3(1), dim3(kRouteThreads), 0, stream, ids, pairs, topk, (int)E,
                                        hdr, tiles, rowmap, src, status);
    if (e != cudaSuccess) return e;
    const int64_t gblocks = (L.max_rows + 7) / 8;
    const unsigned ggrid = (unsigned)(gblocks < (int64_t)num_sms * 8 ? gblocks : (int64_t)num_sms * 8);
    e = launch_programmatic(gather_kernel, dim3(ggrid), dim3(256), 0, stream, a_codes, lda, a_sf, K,
                            static_cast<const int*>(hdr), static_cast<const int4*>(tiles), static_cast<const int*>(src),
                            p_codes, p_sf);
    if (e != cudaSuccess) return e;
    GemmArgs a = {};
    a.epilogue = kEpiBf16;
    a.M = L.max_rows;
    a.N = N;
    a.K = K;
    a.sfa = p_sf;
    a.sfb0 = w_sf;
    a.sfa_tile_stride = (K / 16 + 3) / 4 * 512;
    a.sfb_tile_stride = (K / 16 + 3) / 4 * 512;
    a.ga = a_g;
    a.gb0 = w_g;
    a.gb1 = w_g;
    a.out = out;
    a.ldo = ldo;
    a.status = status;
    a.grp_count = hdr;
    a.grp_tiles = tiles;
    a.grp_rowmap = rowmap;
    a.grp_out_rows = pairs;
    (void)w_codes;
    (void)ldw;
    return launch_gemm_grouped(map_a, map_b, a, num_sms, L.max_tiles * ((N + 255) / 256), stream);
}

}  // namespace nvfp4
