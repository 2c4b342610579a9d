// Internal (C++) launcher interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4.h"

namespace nvfp4 {

// Block size of the row kernels (amax / quantize).  Both kernels reduce a
// row's sum of squares with this many threads in the same order, so the
// RMSNorm they compute is bit-identical.
constexpr int kRowThreads = 256;

// Rows per TMA box of the FP4 code tensors (128 bytes wide, 128-byte
// swizzle).  A 128-row operand tile is fetched as two boxes, issued by two
// different threads: the copies one thread issues are served one after the
// other (about 25 bytes per clock each), so a stage's copies are spread over
// several issuing lanes.
constexpr int kCodeBoxRows = 64;

// Workspace words used by the amax reduction: [0] amax bits, [1] ticket;
// the grid barrier of the fused scale + quantize kernels also counts
// arrivals at word 32 and departures at word 48 (bytes 128 and 192).
constexpr size_t kAmaxWorkspaceBytes = 256;

cudaError_t launch_amax_scale(const __nv_bfloat16* x, int64_t rows, int64_t cols, int64_t ldx,
                              const __nv_bfloat16* norm_w, float eps, float* g_out, uint32_t* ws,
                              int num_sms, cudaStream_t stream);

cudaError_t launch_quantize(const __nv_bfloat16* x, int64_t rows, int64_t cols, int64_t ldx,
                            const __nv_bfloat16* norm_w, float eps, const float* g, uint8_t* codes,
                            int64_t ld_codes, uint8_t* sf, __nv_bfloat16* y_out, int num_sms,
                            cudaStream_t stream);

// g_out = max(amax(ws), 1e-8) / 2688, and the amax word is reset to zero.
cudaError_t launch_finalize_scale(uint32_t* ws, float* g_out, cudaStream_t stream);

// Launch `kernel` on `stream` with the programmatic-serialization attribute:
// it may start while the previous kernel of the stream still runs, and must
// call griddep_wait() before touching anything that kernel writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// launch_amax_scale followed by launch_quantize in one cooperative launch
// (bit-identical results); sf padding rows are zero-filled.  A barrier wait
// that gives up records a timeout in *status.
cudaError_t launch_scale_quantize(const __nv_bfloat16* x, int64_t rows, int64_t cols, int64_t ldx,
                                  const __nv_bfloat16* norm_w, float eps, float* g_out, uint8_t* codes,
                                  int64_t ld_codes, uint8_t* sf, uint32_t* ws, int* status, int num_sms,
                                  cudaStream_t stream);

enum EpilogueKind : int {
    kEpiBf16 = 0,        // out = bf16(alpha * acc) [+ residual]
    kEpiSwigluFp4 = 1,   // s = SwiGLU(gate, up) requantized to FP4 with a given scale
    kEpiSwigluBf16 = 2,  // s stored as bf16 + its amax accumulated into a workspace word
};

struct GemmArgs {
    int epilogue;
    int64_t M, N, K;  // N: output columns (kEpiBf16) or intermediate columns (SwiGLU)
    // scale factors (swizzled) and global scales of A and of the B operand(s)
    const uint8_t* sfa;
    const uint8_t* sfb0;
    const uint8_t* sfb1;
    int64_t sfa_tile_stride;  // bytes between consecutive 128-row scale tiles
    int64_t sfb_tile_stride;
    const float* ga;
    const float* gb0;
    const float* gb1;
    // kEpiBf16
    __nv_bfloat16* out;
    int64_t ldo;
    const __nv_bfloat16* residual;
    int64_t ldr;
    // SwiGLU epilogues
    const float* g_inter;
    uint8_t* s_codes;
    int64_t ld_s_codes;
    uint8_t* s_sf;
    int64_t s_kb_pad;
    __nv_bfloat16* s_bf16;
    int64_t ld_s;
    uint32_t* amax_ws;
    int* status;
    // split schedule (1-SM kernel): sk_partials (slots for at least as many
    // CTAs as the device has SMs) and sk_flags set = the launcher may split
    // (it then launches the split instantiation of the kernel).  Each CTA
    // then takes a contiguous range of the flattened (tile, K stage) units;
    // a tile split between CTAs is finished by the CTA holding its first K
    // stage, from the others' partial accumulators (one fp32 slot of
    // kSplitSlotFloats per CTA) and per-warp ready flags.
    float* sk_partials;
    int* sk_flags;
    // nonzero: the weight operands (B0/B1 codes and scales) were complete
    // before the previous kernel of the stream started, so their loads may
    // run ahead of griddep_wait(); zero: every load waits for that kernel
    // (which may be the one that wrote them) to complete
    int weights_early;
    // rotary embedding of the bf16 output (kEpiBf16 without residual;
    // rope_pos NULL: none).  In each of the rope_heads heads of rope_hd
    // columns from column rope_col0, the last rope_rd columns form (even,
    // odd) pairs rotated by the angles of table row rope_pos[row] (rope_cos,
    // rope_sin: rope_ld floats a row); rope_inverse: the inverse rotation
    const int32_t* rope_pos;
    const float* rope_cos;
    const float* rope_sin;
    int64_t rope_ld, rope_col0, rope_heads, rope_hd, rope_rd;
    int rope_inverse;
    // grouped (expert-indexed) mode of the 1-SM kernel, from tables built on
    // the device (launch_gemm_grouped): A is the expert-sorted operand of
    // args.M rows (each expert's rows padded to 128); B the experts' weights
    // stacked [E * N x K] (N per expert), gb0 fp32[E]; *grp_count M tiles,
    // grp_tiles[m] = {expert, first A row, valid rows, 0}; an A row r goes
    // to output row grp_rowmap[r] (< 0: padding); grp_out_rows output rows.
    const int* grp_count;
    const int4* grp_tiles;
    const int* grp_rowmap;
    int64_t grp_out_rows;
};

// Split-schedule workspace: a fixed block of ready flags (one per epilogue
// warp of up to kSplitMaxCtas CTAs; zero before first use, and every
// completed launch leaves them zero), and one 128 x 256 fp32 accumulator
// slot per CTA of the launch.
constexpr int64_t kSplitSlotFloats = 128 * 256;
constexpr int kSplitFlagsPerCta = 8;
constexpr int kSplitMaxCtas = 256;
constexpr size_t kSplitFlagBytes = (size_t)kSplitMaxCtas * kSplitFlagsPerCta * 4;   // 8 KB
inline size_t split_partial_bytes(int ctas) { return (size_t)ctas * (size_t)kSplitSlotFloats * 4; }

// maps: A [M x K/2 bytes], B0 and B1 (B1 only for SwiGLU) with a 128x128-byte
// box and 128-byte swizzle.
cudaError_t launch_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b0, const CUtensorMap& map_b1,
                        const GemmArgs& args, int num_sms, cudaStream_t stream);

// Grouped mode of the 1-SM kernel (args.grp_* set, bf16 epilogue, no
// residual, no split): a persistent grid of min(SMs, max_tiles) CTAs walks
// the device tile table.
cudaError_t launch_gemm_grouped(const CUtensorMap& map_a, const CUtensorMap& map_b, const GemmArgs& args, int num_sms,
                                int64_t max_tiles, cudaStream_t stream);

// Workspace of the expert-indexed GEMM (byte offsets): a 256-byte header of
// int32 words ([0] M tiles, [1] rows of the expert-sorted operand, [2] an id
// outside [0, E) was seen), the M-tile table (int4), the row map and source
// rows of the sorted operand (int32), then that operand's codes and scales.
// max_rows bounds the sorted rows: pairs + 127 per expert that has any,
// rounded up to 128.
struct ExpertsLayout {
    size_t tiles, rowmap, src, codes, sf, total;
    int64_t max_rows, max_tiles;
};
ExpertsLayout experts_layout(int64_t T, int64_t topk, int64_t K, int64_t E);

// The three launches of the expert-indexed GEMM (routing, gather, grouped
// GEMM); map_a covers the sorted operand's codes in the workspace, map_b the
// stacked weights' codes (boxes of kCodeBoxRows rows).
cudaError_t launch_experts(const uint8_t* a_codes, int64_t lda, const uint8_t* a_sf, const float* a_g, int64_t T,
                           int64_t K, const uint8_t* w_codes, int64_t ldw, const uint8_t* w_sf, const float* w_g,
                           int64_t N, int64_t E, const int32_t* ids, int64_t topk, __nv_bfloat16* out, int64_t ldo,
                           uint8_t* ws, const CUtensorMap& map_a, const CUtensorMap& map_b, int* status, int num_sms,
                           cudaStream_t stream);

// SM-pair version (clusters of 2 CTAs, 256-row tiles): same arguments and
// results, plus 1-D tensor maps of the scale factors of A, B0 and B1 (8-byte
// elements, boxes of 256 elements = 2048 bytes).
cudaError_t launch_gemm2(const CUtensorMap& map_a, const CUtensorMap& map_b0, const CUtensorMap& map_b1,
                         const CUtensorMap& map_sfa, const CUtensorMap& map_sfb0, const CUtensorMap& map_sfb1,
                         const GemmArgs& args, int num_sms, cudaStream_t stream);

// Workspace of nvfp4_gemm_swiglu / nvfp4_mlp without the split schedule's
// partial slots (the least a call accepts; it then runs unsplit).  The
// public size helpers add the slots for the current device.
size_t swiglu_base_workspace_bytes(int64_t T, int64_t I, int inter_mode);
size_t mlp_base_workspace_bytes(int64_t T, int64_t H, int64_t I, int inter_mode);

// nvfp4_mlp's argument checks, all but the workspace's: NVFP4_OK or the
// status nvfp4_mlp returns for these arguments.
int check_mlp_args(const void* x, int64_t T, int64_t H, int64_t ldx, const void* norm_w,
                   const nvfp4_tensor_t* W_gate, const nvfp4_tensor_t* W_up, const nvfp4_tensor_t* W_down,
                   int inter_mode, const float* g_inter, const void* out, int64_t ldo, int add_residual);

}  // namespace nvfp4
