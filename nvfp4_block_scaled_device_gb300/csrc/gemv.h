// Decode-regime NVFP4 GEMM (a handful of activation rows): launcher
// interface between the C-ABI layer and gemv.cu.
#pragma once

#include "internal.h"

namespace nvfp4 {

// Most activation rows the decode kernel takes; more rows go to the
// tensor-core kernels.
constexpr int kDecodeMaxRows = 2;

// Most weight code bytes (both weights for SwiGLU) the CUDA-core decode
// kernel takes (used without the split workspace, which the tensor-core
// decode kernel needs).  It streams weights at ~3 TB/s, against ~5 TB/s
// for the prefill kernels once their pipelines run, but starts at once: it
// wins where the latter's fixed latencies (launch, first round trip,
// fix-up, epilogue) dominate, on weights of tens of MB (measured on GB300
// at T=1, launches back to back: 7168x5120 11.1 vs 18.1 us, 5120x5120 9.2
// vs 13.2 us, 5120x17408 17.6 vs 18.8 us, gate/up 2x17408x5120 33.0 vs
// 20.8 us).
constexpr int64_t kDecodeMaxWeightBytes = int64_t(32) << 20;

// The operands' code arrays (the tensor-core kernels take them as tensor
// maps): A [M x K/2 bytes] with row pitch lda, weights B0 (and B1 for the
// SwiGLU epilogues) [N x K/2 bytes] with row pitches ldb0, ldb1 (bytes).
struct DecodeOperands {
    const uint8_t* a_codes;
    int64_t lda;
    const uint8_t* b0_codes;
    int64_t ldb0;
    const uint8_t* b1_codes;
    int64_t ldb1;
};

// True when the decode kernel takes this problem: args.M <= kDecodeMaxRows,
// weights of at most kDecodeMaxWeightBytes, and its shared memory (which
// grows with K) fits.
bool gemv_eligible(const GemmArgs& args, int num_sms);

// Same arguments and results as launch_gemm (the split-schedule fields of
// args are not used).
cudaError_t launch_gemv(const DecodeOperands& ops, const GemmArgs& args, int num_sms, cudaStream_t stream);

// Tensor-core decode kernel (gemm_decode.cu): at most this many activation
// rows; its activation tensor map has boxes of this many rows.
constexpr int kDecodeTcMaxRows = 8;

// True when the tensor-core decode kernel takes this problem: args.M <=
// kDecodeTcMaxRows, the split-schedule workspace present (its flag words
// serve as per-block tickets, its slots hold the per-segment partials),
// SwiGLU N a multiple of 128.
bool decode_tc_eligible(const GemmArgs& args, int num_sms);

// Same arguments and results as launch_gemm; map_a: the activation codes
// with boxes of 128 bytes x kDecodeTcMaxRows rows (128-byte swizzle),
// map_b0 / map_b1 as for launch_gemm.
cudaError_t launch_decode_tc(const CUtensorMap& map_a, const CUtensorMap& map_b0, const CUtensorMap& map_b1,
                             const GemmArgs& args, int num_sms, cudaStream_t stream);

}  // namespace nvfp4
