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

__global__ void __launch_bounds__(kRouteThreads, 1)
    route_kernel(const int32_t* __restrict__ ids, int64_t pairs, int64_t topk, int E, int* __restrict__ hdr,
                 int* __restrict__ counts, int* __restrict__ cursor, int* __restrict__ seg,
                 int* __restrict__ tile_start, int4* __restrict__ tiles, int* __restrict__ rowmap,
                 int* __restrict__ src, int* status)
{
    griddep_wait();                 // the ids may come from the previous kernel
    for (int e = threadIdx.x; e < E; e += kRouteThreads) {
        counts[e] = 0;
        cursor[e] = 0;
    }
    __syncthreads();
    bool bad = false;
    for (int64_t i = threadIdx.x; i < pairs; i += kRouteThreads) {
        const int e = ids[i];
        if (e >= 0 && e < E)
            atomicAdd(&counts[e], 1);
        else
            bad = true;
    }
    if (bad) {
        hdr[2] = 1;
        if (status) atomicCAS(status, 0, NVFP4_ERR_INVALID_ARG * 100 + 30);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int rows = 0, t = 0;
        for (int e = 0; e < E; e++) {
            const int n = counts[e];
            seg[e] = rows;
            tile_start[e] = t;
            rows += (n + 127) / 128 * 128;
            t += (n + 127) / 128;
        }
        hdr[0] = t;
        hdr[1] = rows;
    }
    __syncthreads();
    // the tile table, and the padding rows of each segment (no output)
    for (int e = threadIdx.x; e < E; e += kRouteThreads) {
        const int n = counts[e];
        for (int m = 0; m * 128 < n; m++)
            tiles[tile_start[e] + m] = make_int4(e, seg[e] + 128 * m, min(128, n - 128 * m), 0);
        for (int r = n; r < (n + 127) / 128 * 128; r++) {
            rowmap[seg[e] + r] = -1;
            src[seg[e] + r] = -1;
        }
    }
    // each pair's row within its expert's segment
    for (int64_t i = threadIdx.x; i < pairs; i += kRouteThreads) {
        const int e = ids[i];
        if (e < 0 || e >= E) continue;
        const int r = seg[e] + atomicAdd(&cursor[e], 1);
        rowmap[r] = (int)i;
        src[r] = (int)(i / topk);
    }
    griddep_launch_dependents();
}

// One 32-lane warp per sorted row: the codes (16-byte vectors) and the
// 32-bit scale words (four consecutive 16-element blocks each) of its
// token row, or zeros for a padding row.
__global__ void __launch_bounds__(256) gather_kernel(const uint8_t* __restrict__ a_codes, int64_t lda,
                                                     const uint8_t* __restrict__ a_sf, int64_t K,
                                                     const int* __restrict__ hdr, const int* __restrict__ src,
                                                     uint8_t* __restrict__ p_codes, uint8_t* __restrict__ p_sf)
{
    griddep_wait();                 // the tables of route_kernel
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    const int lane = threadIdx.x & 31;
    const int64_t rows = hdr[1];
    const int64_t kb = K / 16;                  // scale columns (a multiple of 4: K % 64 == 0)
    const int64_t nvec = K / 32;                // 16-byte vectors of codes per row
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
        const int s = src[r];
        const uint4* in = reinterpret_cast<const uint4*>(a_codes + (int64_t)(s < 0 ? 0 : s) * lda);
        uint4* out = reinterpret_cast<uint4*>(p_codes + r * (K / 2));
        for (int64_t v = lane; v < nvec; v += 32) out[v] = s < 0 ? make_uint4(0, 0, 0, 0) : in[v];
        for (int64_t c4 = lane; c4 < kb / 4; c4 += 32) {
            const uint32_t w = s < 0 ? 0u : *reinterpret_cast<const uint32_t*>(a_sf + sf_offset(s, c4 * 4, kb));
            *reinterpret_cast<uint32_t*>(p_sf + sf_offset(r, c4 * 4, kb)) = w;
        }
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
    L.counts = off;
    off += al((size_t)E * 4);
    L.cursor = off;
    off += al((size_t)E * 4);
    L.seg = off;
    off += al((size_t)E * 4);
    L.tile_start = off;
    off += al((size_t)E * 4);
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
    int* counts = reinterpret_cast<int*>(ws + L.counts);
    int* cursor = reinterpret_cast<int*>(ws + L.cursor);
    int* seg = reinterpret_cast<int*>(ws + L.seg);
    int* tile_start = reinterpret_cast<int*>(ws + L.tile_start);
    int4* tiles = reinterpret_cast<int4*>(ws + L.tiles);
    int* rowmap = reinterpret_cast<int*>(ws + L.rowmap);
    int* src = reinterpret_cast<int*>(ws + L.src);
    uint8_t* p_codes = ws + L.codes;
    uint8_t* p_sf = ws + L.sf;
    const int64_t pairs = T * topk;
    cudaError_t e = launch_programmatic(route_kernel, dim3(1), dim3(kRouteThreads), 0, stream, ids, pairs, topk, (int)E,
                                        hdr, counts, cursor, seg, tile_start, tiles, rowmap, src, status);
    if (e != cudaSuccess) return e;
    const int64_t gblocks = (L.max_rows + 7) / 8;
    const unsigned ggrid = (unsigned)(gblocks < (int64_t)num_sms * 8 ? gblocks : (int64_t)num_sms * 8);
    e = launch_programmatic(gather_kernel, dim3(ggrid), dim3(256), 0, stream, a_codes, lda, a_sf, K,
                            static_cast<const int*>(hdr), static_cast<const int*>(src), p_codes, p_sf);
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
