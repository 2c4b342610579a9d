/*
 * nvfp4.h -- C ABI of libnvfp4.so: the NVFP4 (E2M1 codes + E4M3 scale per 16
 * elements + FP32 per-tensor scale) W4A4 linear and MLP hot path on one
 * Blackwell GPU (sm_103a).
 *
 * Sources, by page title and section:
 *  - "PERFORMANCE -- verified hot-path audit and prioritized fixes"
 *    (nvfp4-megamoe-kernel PERFORMANCE_AUDIT.md): P0 (activation global
 *    scale amax/(6*448) computed on the device and handed to the kernel as a
 *    (1,) device tensor, never read back by the host), P8 items 1-2
 *    (quantization fused into the producer: RMSNorm + quantize), DOCTRINE 1
 *    (no host state on the hot path).
 *  - "CUDA: NVFP4 prefill on Blackwell leaves ~1.45x performance on the
 *    table. Comparison + PoC" (llama.cpp discussion 28514), "What the patch
 *    does": GLU output quantized straight into the next GEMM's activation
 *    format, gate/up sharing one quantized input, batched-row rms_norm,
 *    TMA + mbarrier fed FP4 MMA tiles; and its ncu finding that a 36-byte
 *    interleaved FP4 block is only 4-byte aligned -- codes and scales are
 *    therefore kept in separate, 16-byte aligned arrays here.
 *  - "tp>1 prefill is host-bound: per-token fp4 GEMM + per-layer H2D
 *    activation staging" (vllm.cpp issue 2144), "Fix directions" 1-3: one
 *    launch set per T-token batch with a grid that scales with T,
 *    activations resident on the device, quantization on the device.
 *
 * Conventions (all functions):
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise, owned
 *    by the caller.  No function allocates, frees or synchronises; all work is
 *    enqueued on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *  - The GEMM kernels use programmatic dependent launch: they may start
 *    while the previous kernel of the stream still runs, and read their
 *    operands only after it has completed -- except inside nvfp4_mlp, whose
 *    GEMMs fetch the weights early (the weights were complete before the
 *    call's first, plainly launched kernel started): a tensor quantized by
 *    the launch just before a GEMM call is safe to use as its weight.
 *  - The return value is a status (NVFP4_OK = 0).  Argument errors are
 *    detected on the host before anything is enqueued.  NVFP4_ERR_CUDA
 *    reports a launch error (cudaGetLastError); asynchronous failures show
 *    up in the stream as usual.
 *  - bf16 tensors are row-major with a row pitch given in ELEMENTS; bf16
 *    base pointers and pitches must be 16-byte aligned (pitch % 8 == 0).
 *  - A quantized tensor (nvfp4_tensor_t) of logical shape [rows x cols]:
 *      codes: byte (r, k/2) at codes + r*ld + k/2 holds element k in its low
 *             nibble when k is even, in its high nibble when k is odd; each
 *             nibble is an E2M1 code (bit 3 sign, magnitudes 0, .5, 1, 1.5,
 *             2, 3, 4, 6).  cols % 64 == 0; ld % 16 == 0; codes 16-B aligned.
 *      sf:    one unsigned E4M3 scale per 16 consecutive elements of a row,
 *             in 512-byte tiles of 128 rows x 4 scales: rows padded to a
 *             multiple of 128, scale columns (cols/16) padded to a multiple of
 *             4, tiles row-tile-major, and inside a tile the scale of row r,
 *             column c at (r%32)*16 + (r%128)/32*4 + c%4.  Size:
 *             nvfp4_sf_bytes(rows, cols); 128-B aligned; padding bytes are 0.
 *      g:     fp32[1] per-tensor global scale (> 0).
 *    Element value = E2M1(code) * E4M3(scale) * g.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvfp4_stream_t; /* identical to cudaStream_t */

enum nvfp4_status {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1, /* NULL pointer, bad shape (rows < 1, cols % 64 != 0, ...) */
    NVFP4_ERR_MISALIGNED = 2,  /* pointer or pitch not aligned as documented */
    NVFP4_ERR_UNSUPPORTED = 3, /* device is not compute capability 10.3 (sm_103a) */
    NVFP4_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
    NVFP4_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required */
    NVFP4_ERR_TIMEOUT = 6      /* device-side: a pipeline wait exceeded its time limit */
};

/* Intermediate (SwiGLU output) global-scale modes of the fused gate/up GEMM. */
enum nvfp4_inter_mode {
    /* g_inter is an input: a scale fixed ahead of time (e.g. by one DYNAMIC
     * warm-up call), used by the GEMM epilogue to requantize SwiGLU output
     * straight into FP4 ("keep the warm-up scale as a device tensor"). */
    NVFP4_INTER_STATIC = 0,
    /* g_inter is an output: the epilogue stores bf16 SwiGLU output and its
     * amax, then the scale max(amax,1e-8)/2688 is written to *g_inter on the
     * device and the SwiGLU output is quantized with it (exact per-call
     * scale, two extra HBM passes over T x I bf16). */
    NVFP4_INTER_DYNAMIC = 1
};

/* A quantized matrix; see the conventions above. */
typedef struct {
    const uint8_t* codes;
    const uint8_t* sf;
    const float* g;
    int64_t rows;
    int64_t cols;
    int64_t ld; /* bytes */
} nvfp4_tensor_t;

/* ------------------------------------------------------------ host helpers */

/* Bytes of a codes array with ld = cols/2: rows * cols / 2. */
size_t nvfp4_codes_bytes(int64_t rows, int64_t cols);
/* Bytes of a scale array: pad128(rows) * pad4(cols/16). */
size_t nvfp4_sf_bytes(int64_t rows, int64_t cols);
/* Workspace of nvfp4_amax_scale and nvfp4_scale_quantize (256 bytes, 256-B aligned). */
size_t nvfp4_amax_workspace_bytes(void);
/* Workspace that lets nvfp4_gemm split its work evenly over all SMs of the
 * current device (8 KB of ready flags + 128 KB per SM; 0 when no device is
 * usable). */
size_t nvfp4_gemm_workspace_bytes(void);
/* Workspace of nvfp4_gemm_swiglu for an A of T rows and an intermediate of I
 * columns on the current device: 256 + 8192 bytes, + T*I*2 (DYNAMIC), + the
 * split schedule's 128 KB per SM.  A workspace without the last part is
 * accepted (the call then runs unsplit). */
size_t nvfp4_swiglu_workspace_bytes(int64_t T, int64_t I, int inter_mode);
/* Workspace of nvfp4_mlp (T tokens, hidden H, intermediate I) on the current
 * device; likewise, its last 128 KB per SM (the split schedule's) may be
 * left out. */
size_t nvfp4_mlp_workspace_bytes(int64_t T, int64_t H, int64_t I, int inter_mode);
/* Workspace of nvfp4_gemm_experts for T tokens, topk slots, K columns and E
 * experts: the routing tables plus the expert-sorted operand (at most
 * T*topk + 127*min(E, T*topk) rows, rounded up to 128, of K/2 + K/16 bytes). */
size_t nvfp4_experts_workspace_bytes(int64_t T, int64_t topk, int64_t K, int64_t num_experts);
/* Static description of a status code. */
const char* nvfp4_status_string(int status);
/* Reads (and if clear != 0 resets) the library's device-side status word of
 * the current device, which kernels set when a pipeline wait times out.
 * SYNCHRONOUS (a device-to-host copy); diagnostics and tests only. */
int nvfp4_device_status(int* status_out, int clear);
/* Measures the issue rate of the tensor-core instruction form the GEMM
 * kernels use (tcgen05.mma.cta_group::2 kind::mxf4nvf4 scale_vec::4X,
 * M=256 N=256 K=64, with its scale copies), fed back to back from operands
 * already in shared memory on one SM pair of the current device: writes
 * the multiply-adds per SM per clock cycle to *mac_per_clk.  Returns
 * NVFP4_ERR_TIMEOUT if the measurement's bounded wait ran out.  SYNCHRONOUS;
 * a measurement diagnostic (the dense NVFP4 peak of this instruction is
 * 2 * mac_per_clk * SMs * SM clock), not part of the path.  No counterpart
 * in the pages, which give no peak. */
int nvfp4_mma_issue_rate(double* mac_per_clk);

/* ------------------------------------------------------------- the path */

/*
 * nvfp4_amax_scale -- device per-tensor global scale.
 *   g_out[0] = max(amax, 1e-8) / (6 * 448)  (binary32 division),
 *   amax = max |v| over the bf16 matrix v.
 * Source: "PERFORMANCE -- verified hot-path audit and prioritized fixes", P0
 * (the runtime scale, computed on the device instead of via .item()).
 *   x        bf16 [rows x cols], row pitch ldx elements.
 *   norm_w   NULL, or bf16 [cols]: then v is the RMSNorm of x,
 *            v = bf16(x * r * w), r = 1/sqrt(mean(x^2) + eps) per row
 *            (the batched-row RMSNorm prologue).
 *   g_out    fp32[1], written.
 *   workspace >= nvfp4_amax_workspace_bytes(), 256-B aligned.  It must be
 *            zero-filled ONCE after allocation; every call returns it to zero.
 *            Calls sharing one workspace must be stream-ordered.
 * Requires rows >= 1, cols >= 8, cols % 8 == 0.
 */
int nvfp4_amax_scale(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                     const void* norm_w, float eps, float* g_out,
                     void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_quantize -- bf16 -> NVFP4 with the device global scale g.
 * Per 16-element block (binary32, one rounding per step):
 *   s = E4M3_rne_satfinite( amax16 / (6*g) ),
 *   code_i = s == 0 ? +0 : E2M1_rne_satfinite( v_i / (E4M3(s) * g) ).
 * Sources: "PERFORMANCE -- verified hot-path audit and prioritized fixes",
 * P0 and P8 item 2 (rmsnorm_quantize); "CUDA: NVFP4 prefill on Blackwell
 * leaves ~1.45x performance on the table", item 2 (batched-row rms_norm).
 *   x, ldx, norm_w, eps  as nvfp4_amax_scale (norm_w != NULL: quantize the
 *            RMSNorm of x, computed exactly as nvfp4_amax_scale computes it).
 *   g        fp32[1] device global scale.
 *   codes    [rows][ld_codes] bytes, ld_codes >= cols/2, % 16 == 0.
 *   sf       nvfp4_sf_bytes(rows, cols) bytes, 128-B aligned; padding written 0.
 *   y_out    NULL, or bf16 [rows x cols] (pitch cols): receives v (export for
 *            tests of the norm prologue).
 * Requires rows >= 1, cols % 64 == 0.
 */
int nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                   const void* norm_w, float eps, const float* g,
                   uint8_t* codes, int64_t ld_codes, uint8_t* sf, void* y_out,
                   nvfp4_stream_t stream);

/*
 * nvfp4_scale_quantize -- nvfp4_amax_scale then nvfp4_quantize with the
 * scale just computed, as ONE kernel launch: *g_out, codes and sf are bit for
 * bit those of the two calls.  The kernel is a cooperative launch with one
 * grid-wide barrier between the amax and the quantization (every block is
 * resident; when the grid covers all rows at once each row is read once).
 * Sources: as nvfp4_amax_scale and nvfp4_quantize.
 *   x, ldx, norm_w, eps  as nvfp4_amax_scale.
 *   g_out    fp32[1], written with the global scale.
 *   codes, ld_codes, sf  as nvfp4_quantize.
 *   workspace as nvfp4_amax_scale (>= nvfp4_amax_workspace_bytes(), zero-filled
 *            once; calls leave it zeroed).  After a call that reported a
 *            timeout through nvfp4_device_status it must be zero-filled again.
 * Requires rows >= 1, cols % 64 == 0.
 */
int nvfp4_scale_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                         const void* norm_w, float eps, float* g_out,
                         uint8_t* codes, int64_t ld_codes, uint8_t* sf,
                         void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_gemm -- block-scaled GEMM on the tensor cores (tcgen05
 * kind::mxf4nvf4, fp32 accumulation in tensor memory):
 *   out[m][n] = bf16( alpha * sum_k A[m,k] W[n,k] ),  alpha = fp32(gA * gW),
 *   or, with residual != NULL, bf16( residual[m][n] + that bf16 ).
 * Source: "CUDA: NVFP4 prefill on Blackwell leaves ~1.45x performance on the
 * table" item 3 (TMA + mbarrier fed FP4 MMA accumulated in place);
 * "tp>1 prefill is host-bound" fix direction 1 (one launch for all T rows).
 *   A        activations, rows M = T (any M >= 1), cols K.
 *   W        weights [N x K] (K-major, as nn.Linear stores them).
 *   out      bf16 [M x N], pitch ldo; may alias residual (same pitch).
 *   workspace NULL, or >= 8192 bytes, 256-B aligned, zero-filled once after
 *            allocation (calls leave it zeroed); calls sharing one workspace
 *            must be stream-ordered.  With nvfp4_gemm_workspace_bytes() bytes
 *            the GEMM may split its tiles' K ranges over all SMs when whole
 *            tiles would leave part of the GPU idle (fp32 partials combined
 *            in the workspace); otherwise whole tiles are spread over the SMs.
 * With M <= 8 and such a workspace the GEMM runs instead as a weight stream
 * on the tensor cores (the weights as the MMA's 128-row side, split over
 * all SMs along K, fp32 partials combined in the workspace in a fixed
 * order); without one, with M <= 2 and at most 32 MiB of weight codes, as
 * a weight stream on the CUDA cores (exact int32 sums of E2M1 code
 * products per 16-element block, block scales applied exactly in fp32,
 * fp32 accumulation).  Either gives the same result up to the fp32
 * summation order.  nvfp4_gemm_swiglu and nvfp4_mlp do the same, except
 * that a SwiGLU GEMM whose 128-column blocks fill at least 85% of the SMs
 * runs as whole tiles.
 * Requires K == A->cols == W->cols, K % 64 == 0, N % 16 == 0.
 */
int nvfp4_gemm(const nvfp4_tensor_t* A, const nvfp4_tensor_t* W,
               void* out, int64_t ldo, const void* residual, int64_t ldr,
               void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Rotary embedding applied by nvfp4_gemm_rope (all pointers DEVICE). */
typedef struct {
    const int32_t* pos;   /* int32 [M]: position of each output row, in [0, positions) (not checked on the device) */
    const float* cos_t;   /* fp32 [positions x table_ld]: cos of the angle of (position, pair i) at [p*table_ld + i] */
    const float* sin_t;   /* fp32, the same layout: sin of that angle */
    int64_t table_ld;     /* floats per table row, >= rope_dim / 2 */
    int64_t positions;    /* rows of the tables, >= 1 */
    int64_t col0;         /* first output column of the first rotated head; even */
    int64_t heads;        /* rotated heads (col0 + heads * head_dim <= N) */
    int64_t head_dim;     /* columns per head; even */
    int64_t rope_dim;     /* rotated columns per head: the LAST rope_dim of each head; even, <= head_dim */
    int inverse;          /* nonzero: the inverse rotation */
} nvfp4_rope_t;

/*
 * nvfp4_gemm_rope -- nvfp4_gemm (no residual) with a rotary position
 * embedding applied to its bf16 output in the GEMM's epilogue, e.g. the Q
 * and K heads of a QKV projection.  Source: "PERFORMANCE -- verified
 * hot-path audit and prioritized fixes", P5 (RoPE on the last rope_dim
 * columns of each head, float32 arithmetic from bf16 and back) and the
 * structural target "fuse RoPE into the Q/KV GEMM epilogue".
 * In a rotated head, the pairs (e, o) = (y[2i], y[2i+1]) of the last rope_dim
 * columns of y = nvfp4_gemm's bf16 output are rotated with
 * c = cos_t[pos[m]*table_ld + i], s = sin_t[...]:
 *   forward: e' = e*c - o*s,  o' = e*s + o*c;  inverse: e' = e*c + o*s,  o' = o*c - e*s
 * each product, sum and difference one binary32 operation, then rounded to
 * bf16; every other column is nvfp4_gemm's output.
 *   A, W, out, ldo, workspace  as nvfp4_gemm.
 *   rope     the embedding's tables and geometry (above).
 */
int nvfp4_gemm_rope(const nvfp4_tensor_t* A, const nvfp4_tensor_t* W, void* out, int64_t ldo,
                    const nvfp4_rope_t* rope, void* workspace, size_t workspace_bytes,
                    nvfp4_stream_t stream);

/*
 * nvfp4_gemm_experts -- expert-indexed GEMM, the routed projection of a
 * mixture-of-experts layer (llama.cpp's MUL_MAT_ID).  For token t and routing
 * slot j < topk, with e = ids[t*topk + j]:
 *   out[(t*topk + j) * ldo + n] = bf16( fp32(A->g[0] * W->g[e]) * sum_k A[t,k] W_e[n,k] ),
 * the sum and the rounding as in nvfp4_gemm.  The routing table stays on
 * the device: three launches (routing, gather of the routed rows into an
 * expert-sorted operand, grouped tcgen05 GEMM over a tile table built on the
 * device), no host synchronisation.  Sources: "CUDA: NVFP4 prefill on
 * Blackwell leaves ~1.45x performance on the table" (the MUL_MAT_ID tests
 * its patch passes); "PERFORMANCE -- verified hot-path audit and prioritized
 * fixes" (the routed experts run without a host read of the routing table).
 *   A            [T x K] quantized activations.
 *   W            the E experts' weights stacked: rows E*N (expert e = rows
 *                e*N .. e*N + N - 1), cols K; W->g points to fp32[E], expert
 *                e's global scale.  N = W->rows / E, a multiple of 128.
 *   num_experts  E, 1 .. 4096.
 *   ids          DEVICE int32 [T * topk]: the expert of each (token, slot).
 *                An id outside [0, E) leaves that output row unwritten and
 *                records NVFP4_ERR_INVALID_ARG * 100 + 30 in the device
 *                status word (nvfp4_device_status).
 *   topk         routing slots per token, >= 1 (T * topk < 2^31).
 *   out          bf16 [T*topk x N], row pitch ldo (elements).
 *   workspace    nvfp4_experts_workspace_bytes(T, topk, K, E) bytes,
 *                256-byte aligned; no zero-fill needed; not shared with a
 *                call that may run at the same time.
 */
int nvfp4_gemm_experts(const nvfp4_tensor_t* A, const nvfp4_tensor_t* W, int64_t num_experts, const int32_t* ids,
                       int64_t topk, void* out, int64_t ldo, void* workspace, size_t workspace_bytes,
                       nvfp4_stream_t stream);

/*
 * nvfp4_gemm_swiglu -- fused gate/up GEMM with SwiGLU epilogue and FP4
 * requantization into the down projection's activation format:
 *   gate = bf16(alpha_g * A Wg^T), up = bf16(alpha_u * A Wu^T),
 *   s = bf16( gate * sigmoid(gate) * up ),  S = NVFP4(s) with scale g_inter.
 * Source: "CUDA: NVFP4 prefill on Blackwell leaves ~1.45x performance on the
 * table" item 2 (GLU output quantized directly into the next GEMM's
 * activation format; gate and up share one quantized input).
 *   A            [T x K] quantized input, shared by both GEMMs.
 *   W_gate, W_up [I x K] each, same shape.
 *   inter_mode   NVFP4_INTER_STATIC (g_inter read) or NVFP4_INTER_DYNAMIC
 *                (g_inter written with the per-call scale).
 *   s_codes      [T][ld_s_codes] bytes (I/2 per row); s_sf nvfp4_sf_bytes(T, I).
 *   s_bf16       NULL, or bf16 [T x I] (pitch I): receives s (export).
 *   workspace    nvfp4_swiglu_workspace_bytes(T, I, inter_mode), 256-B aligned,
 *                zero-filled once after allocation (calls leave it zeroed).
 * Requires I % 128 == 0, K % 64 == 0.
 */
int nvfp4_gemm_swiglu(const nvfp4_tensor_t* A, const nvfp4_tensor_t* W_gate,
                      const nvfp4_tensor_t* W_up, int inter_mode, float* g_inter,
                      uint8_t* s_codes, int64_t ld_s_codes, uint8_t* s_sf, void* s_bf16,
                      void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_mlp -- the whole NVFP4 MLP block for a batch of T tokens in one
 * launch set, activations device-resident, no host synchronisation:
 *   h   = NVFP4( RMSNorm(x; norm_w, eps) )   (scale g_h computed on device)
 *   S   = nvfp4_gemm_swiglu(h, W_gate, W_up, inter_mode, g_inter)
 *   out = bf16( [x +] alpha_d * S W_down^T )
 * Sources: all three pages (see top of file).
 *   x        bf16 [T x H], pitch ldx.
 *   W_gate, W_up [I x H]; W_down [H x I].
 *   out      bf16 [T x H], pitch ldo; may alias x (in-place residual, ldo == ldx).
 *   workspace nvfp4_mlp_workspace_bytes(T, H, I, inter_mode), 256-B aligned,
 *            zero-filled once after allocation (calls leave it zeroed).
 * Requires H % 64 == 0, I % 128 == 0, T >= 1.
 */
int nvfp4_mlp(const void* x, int64_t T, int64_t H, int64_t ldx,
              const void* norm_w, float eps,
              const nvfp4_tensor_t* W_gate, const nvfp4_tensor_t* W_up,
              const nvfp4_tensor_t* W_down, int inter_mode, float* g_inter,
              void* out, int64_t ldo, int add_residual,
              void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_mlp_noalloc -- nvfp4_mlp for callers that cannot allocate device
 * memory (no counterpart on the source pages; an addition of this library).
 * Examples: a plugin that only receives borrowed tensor pointers from its host
 * application and has no allocator, or a latency-critical caller for which
 * cudaMalloc -- which may synchronise the whole device -- is not acceptable.
 *
 * Same computation, arguments, requirements and results as nvfp4_mlp, minus
 * the workspace: the intermediates live in a fixed 32 MiB array inside this
 * library (every GPU that loads the library holds it until the process
 * exits).  The array must hold nvfp4_mlp's workspace without the split
 * schedule's partial slots (those slots are used too when they also fit,
 * which at H=5120, I=17408 and 152 SMs is up to T ~1070 with
 * NVFP4_INTER_STATIC): a larger call returns NVFP4_ERR_WORKSPACE.  At
 * H=5120, I=17408 the largest T is 2642 with NVFP4_INTER_STATIC and 704 with
 * NVFP4_INTER_DYNAMIC.
 *   - Argument errors (the statuses nvfp4_mlp returns) and
 *     NVFP4_ERR_WORKSPACE are returned before anything is enqueued.
 *   - Allocates nothing and calls no allocator.  It enqueues one small
 *     cudaMemsetAsync that clears the array's amax words and the split
 *     schedule's flag words (a call that stopped early may have left them
 *     non-zero), then the nvfp4_mlp launches.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it for the life of the process; make
 *     that first call before any stream capture.  The cached address is not
 *     looked up again: do not use the library across cudaDeviceReset or
 *     anything else that destroys the device's primary context.
 *   - Every call shares the one array: calls that can overlap on the GPU
 *     (different streams, or several host threads) race with each other and
 *     must be serialised by the caller.
 */
int nvfp4_mlp_noalloc(const void* x, int64_t T, int64_t H, int64_t ldx,
                      const void* norm_w, float eps,
                      const nvfp4_tensor_t* W_gate, const nvfp4_tensor_t* W_up,
                      const nvfp4_tensor_t* W_down, int inter_mode, float* g_inter,
                      void* out, int64_t ldo, int add_residual, nvfp4_stream_t stream);

/*
 * nvfp4_noalloc_scratch -- diagnostics: the device address (on the current
 * device) and the size of nvfp4_mlp_noalloc's fixed array.  The array
 * belongs to nvfp4_mlp_noalloc; a caller may read it, or clear it between
 * calls, but anything it writes there is overwritten or cleared by the next
 * call.  Same caching as nvfp4_mlp_noalloc.
 */
int nvfp4_noalloc_scratch(void** device_ptr, size_t* bytes);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H */
