// C ABI of libnvfp4.so (declared in include/nvfp4.h): argument validation on
// the host, tensor-map construction, and the launch sets of the NVFP4 path.
// Nothing here allocates device memory or synchronises the stream (except
// nvfp4_device_status, a diagnostic).
#include <cudaTypedefs.h>

#include <mutex>

#include "gemv.h"
#include "internal.h"
#include "nvfp4.h"

using namespace nvfp4;

// Device-side status word: kernels record a timed-out pipeline wait here.
__device__ int g_nvfp4_status_word = 0;

namespace {

struct DeviceInfo {
    bool init;
    int cc_major, cc_minor, num_sms;
    int* status;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_info(DeviceInfo** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        if (d.cc_major == 10 && d.cc_minor == 3) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_nvfp4_status_word) != cudaSuccess) return NVFP4_ERR_CUDA;
            d.status = static_cast<int*>(p);
        }
        d.init = true;
    }
    if (!(d.cc_major == 10 && d.cc_minor == 3)) return NVFP4_ERR_UNSUPPORTED;
    *out = &d;
    return NVFP4_OK;
}

int encoder()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return NVFP4_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return NVFP4_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return NVFP4_OK;
}

// 2-D byte tensor [rows x row_bytes], pitch ld, boxes of 128 bytes x
// box_rows rows, 128-B swizzle.
int make_codes_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes, int64_t ld,
                   int box_rows = nvfp4::kCodeBoxRows)
{
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// Scale factors viewed as a 1-D array of 8-byte elements, boxes of 256
// elements: one box is the 2048 contiguous bytes of four 512-byte scale
// tiles (one K stage of a 128-row block).
int make_sf_map(CUtensorMap* m, const void* base, size_t bytes)
{
    cuuint64_t dims[1] = {(cuuint64_t)(bytes / 8)};
    cuuint64_t strides[1] = {0};
    cuuint32_t box[1] = {256};
    cuuint32_t estr[1] = {1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 1, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline int64_t pad_to(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

int check_bf16_matrix(const void* p, int64_t rows, int64_t cols, int64_t ld)
{
    if (!p || rows < 1 || cols < 1 || ld < cols) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(p, 16) || ld % 8 != 0) return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

int check_tensor(const nvfp4_tensor_t* t)
{
    if (!t || !t->codes || !t->sf || !t->g) return NVFP4_ERR_INVALID_ARG;
    if (t->rows < 1 || t->cols < 64 || t->cols % 64 != 0 || t->ld < t->cols / 2) return NVFP4_ERR_INVALID_ARG;
    if (t->rows > INT32_MAX || t->cols / 2 > INT32_MAX) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(t->codes, 16) || t->ld % 16 != 0 || !aligned(t->sf, 128) || !aligned(t->g, 4))
        return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

int64_t sf_tile_stride(int64_t cols) { return pad_to(cols / 16, 4) / 4 * 512; }

#define NVFP4_TRY(expr)                 \
    do {                                \
        int _st = (expr);               \
        if (_st != NVFP4_OK) return _st; \
    } while (0)

#define NVFP4_CUDA(expr)                                   \
    do {                                                   \
        if ((expr) != cudaSuccess) return NVFP4_ERR_CUDA; \
    } while (0)

// The SM-pair kernel (256 x 256 tiles on two SMs) takes M >= kPairMinRows
// when its tiles fill at least one wave of SM pairs; otherwise the 1-SM
// kernel (128 x 256 tiles, split schedule over all SMs when given a
// workspace) runs.  With the weights streaming from HBM, as in a layer
// block whose weights exceed L2, the pair kernel's smaller per-SM operand
// stages (38 KB vs 54 KB for the same MMA work, five stages in flight
// instead of four) cover more of the load latency: measured faster on
// every GEMM of the prefill block, the O projection's partial last wave
// included.
#ifdef NVFP4_PAIR_MIN_ROWS
constexpr int64_t kPairMinRows = NVFP4_PAIR_MIN_ROWS;   // probe builds only
#else
constexpr int64_t kPairMinRows = 129;
#endif

cudaError_t run_gemm(const CUtensorMap& ma, const CUtensorMap& mb0, const CUtensorMap& mb1, const GemmArgs& a,
                     const DecodeOperands& ops, const DeviceInfo* d, cudaStream_t stream)
{
    // a handful of activation rows: a weight stream, on the tensor cores
    // given the split workspace (tickets and partials), else (one or two
    // rows) on the CUDA cores.  A SwiGLU GEMM whose 128-column blocks
    // nearly fill the GPU (>= 85% of the SMs) runs as whole tiles on the
    // prefill kernel instead: no split-K partials to combine.
    const bool whole_tiles = a.epilogue != kEpiBf16 && (a.N / 128) * 20 >= (int64_t)17 * d->num_sms;
    if (!whole_tiles && decode_tc_eligible(a, d->num_sms)) {
        CUtensorMap ma8;
        if (make_codes_map(&ma8, ops.a_codes, a.M, a.K / 2, ops.lda, kDecodeTcMaxRows) != NVFP4_OK)
            return cudaErrorInvalidValue;
        return launch_decode_tc(ma8, mb0, mb1, a, d->num_sms, stream);
    }
    if (gemv_eligible(a, d->num_sms)) return launch_gemv(ops, a, d->num_sms, stream);
    const bool swiglu = a.epilogue != kEpiBf16;
    const int64_t pair_tiles = (a.M + 255) / 256 * (swiglu ? a.N / 128 : (a.N + 255) / 256);
    if (a.M >= kPairMinRows && pair_tiles * 2 >= d->num_sms) {
        // the pair kernel fetches the scale tiles through tensor maps too
        CUtensorMap msa, msb0, msb1;
        if (make_sf_map(&msa, a.sfa, nvfp4_sf_bytes(a.M, a.K)) != NVFP4_OK ||
            make_sf_map(&msb0, a.sfb0, nvfp4_sf_bytes(a.N, a.K)) != NVFP4_OK ||
            make_sf_map(&msb1, a.sfb1 ? a.sfb1 : a.sfb0, nvfp4_sf_bytes(a.N, a.K)) != NVFP4_OK)
            return cudaErrorInvalidValue;
        return launch_gemm2(ma, mb0, mb1, msa, msb0, msb1, a, d->num_sms, stream);
    }
    return launch_gemm(ma, mb0, mb1, a, d->num_sms, stream);
}

// Shared by nvfp4_gemm_swiglu and nvfp4_mlp.
// Split-schedule scratch of one call: the flag block and, when the
// workspace has room for one slot per SM, the partial slots (else nullptr:
// no split).
struct SplitScratch {
    int* flags = nullptr;
    float* partials = nullptr;
};

SplitScratch split_scratch(const DeviceInfo* d, uint8_t* flags, uint8_t* partials, size_t partial_room)
{
    SplitScratch sp;
    if (d->num_sms <= kSplitMaxCtas && partial_room >= split_partial_bytes(d->num_sms)) {
        sp.flags = reinterpret_cast<int*>(flags);
        sp.partials = reinterpret_cast<float*>(partials);
    }
    return sp;
}

// The gate/up GEMM's arguments common to both SwiGLU modes (the caller
// sets the epilogue and its outputs).
GemmArgs swiglu_gemm_args(const DeviceInfo* d, const nvfp4_tensor_t* A, const nvfp4_tensor_t* Wg,
                          const nvfp4_tensor_t* Wu, uint8_t* s_codes, int64_t ld_s_codes, uint8_t* s_sf,
                          SplitScratch split, bool weights_early)
{
    const int64_t T = A->rows, I = Wg->rows;
    GemmArgs a = {};
    a.M = T;
    a.N = I;
    a.K = A->cols;
    a.sfa = A->sf;
    a.sfb0 = Wg->sf;
    a.sfb1 = Wu->sf;
    a.sfa_tile_stride = sf_tile_stride(A->cols);
    a.sfb_tile_stride = sf_tile_stride(Wg->cols);
    a.ga = A->g;
    a.gb0 = Wg->g;
    a.gb1 = Wu->g;
    a.status = d->status;
    a.weights_early = weights_early ? 1 : 0;
    a.s_codes = s_codes;
    a.ld_s_codes = ld_s_codes;
    a.s_sf = s_sf;
    a.s_kb_pad = pad_to(I / 16, 4);
    a.sk_flags = split.flags;
    a.sk_partials = split.partials;
    return a;
}

int run_swiglu(const DeviceInfo* d, const nvfp4_tensor_t* A, const nvfp4_tensor_t* Wg, const nvfp4_tensor_t* Wu,
               int mode, float* g_inter, uint8_t* s_codes, int64_t ld_s_codes, uint8_t* s_sf,
               __nv_bfloat16* s_bf16_user, uint32_t* amax_ws, __nv_bfloat16* s_bf16_scratch, SplitScratch split,
               bool weights_early, cudaStream_t stream)
{
    const int64_t T = A->rows, I = Wg->rows;
    CUtensorMap ma, mg, mu;
    NVFP4_TRY(make_codes_map(&ma, A->codes, T, A->cols / 2, A->ld));
    NVFP4_TRY(make_codes_map(&mg, Wg->codes, I, Wg->cols / 2, Wg->ld));
    NVFP4_TRY(make_codes_map(&mu, Wu->codes, I, Wu->cols / 2, Wu->ld));
    const DecodeOperands ops = {A->codes, A->ld, Wg->codes, Wg->ld, Wu->codes, Wu->ld};
    GemmArgs a = swiglu_gemm_args(d, A, Wg, Wu, s_codes, ld_s_codes, s_sf, split, weights_early);
    if (mode == NVFP4_INTER_STATIC) {
        a.epilogue = kEpiSwigluFp4;
        a.g_inter = g_inter;
        a.s_bf16 = s_bf16_user;
        a.ld_s = I;
        NVFP4_CUDA(run_gemm(ma, mg, mu, a, ops, d, stream));
    } else {
        __nv_bfloat16* s_bf16 = s_bf16_user ? s_bf16_user : s_bf16_scratch;
        a.epilogue = kEpiSwigluBf16;
        a.s_bf16 = s_bf16;
        a.ld_s = I;
        a.amax_ws = amax_ws;
        NVFP4_CUDA(run_gemm(ma, mg, mu, a, ops, d, stream));
        NVFP4_CUDA(launch_finalize_scale(amax_ws, g_inter, stream));
        NVFP4_CUDA(launch_quantize(s_bf16, T, I, I, nullptr, 0.0f, g_inter, s_codes, ld_s_codes, s_sf, nullptr,
                                   d->num_sms, stream));
    }
    return NVFP4_OK;
}

int check_swiglu_args(const nvfp4_tensor_t* A, const nvfp4_tensor_t* Wg, const nvfp4_tensor_t* Wu, int mode,
                      const float* g_inter)
{
    NVFP4_TRY(check_tensor(A));
    NVFP4_TRY(check_tensor(Wg));
    NVFP4_TRY(check_tensor(Wu));
    if (Wg->rows != Wu->rows || Wg->cols != Wu->cols || A->cols != Wg->cols) return NVFP4_ERR_INVALID_ARG;
    if (Wg->rows % 128 != 0) return NVFP4_ERR_INVALID_ARG;
    if (mode != NVFP4_INTER_STATIC && mode != NVFP4_INTER_DYNAMIC) return NVFP4_ERR_INVALID_ARG;
    if (!g_inter) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(g_inter, 4)) return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

// SMs of the current device (0 without a usable device): the split
// schedule's partial slots in the workspace sizes are one per SM.
int current_device_sms()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sms <= kSplitMaxCtas ? sms : 0;
}

// nvfp4_gemm and nvfp4_gemm_rope (rope NULL: no rotary embedding).
int run_linear(const nvfp4_tensor_t* A, const nvfp4_tensor_t* W, void* out, int64_t ldo, const void* residual,
               int64_t ldr, const nvfp4_rope_t* rope, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

}  // namespace

// Every argument check of nvfp4_mlp but the workspace's (nvfp4_mlp_noalloc
// runs them before it touches its fixed array).
int nvfp4::check_mlp_args(const void* x, int64_t T, int64_t H, int64_t ldx, const void* norm_w,
                          const nvfp4_tensor_t* W_gate, const nvfp4_tensor_t* W_up, const nvfp4_tensor_t* W_down,
                          int inter_mode, const float* g_inter, const void* out, int64_t ldo, int add_residual)
{
    NVFP4_TRY(check_bf16_matrix(x, T, H, ldx));
    if (H % 64 != 0 || !norm_w) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(norm_w, 16)) return NVFP4_ERR_MISALIGNED;
    NVFP4_TRY(check_tensor(W_gate));
    NVFP4_TRY(check_tensor(W_up));
    NVFP4_TRY(check_tensor(W_down));
    const int64_t I = W_gate->rows;
    if (W_gate->cols != H || W_up->cols != H || W_up->rows != I || W_down->rows != H || W_down->cols != I ||
        I % 128 != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (inter_mode != NVFP4_INTER_STATIC && inter_mode != NVFP4_INTER_DYNAMIC) return NVFP4_ERR_INVALID_ARG;
    if (!g_inter) return NVFP4_ERR_INVALID_ARG;
    NVFP4_TRY(check_bf16_matrix(out, T, H, ldo));
    if (add_residual && out == x && ldo != ldx) return NVFP4_ERR_INVALID_ARG;
    return NVFP4_OK;
}

// Workspace layouts (all offsets 256-B aligned).  Without the trailing
// partial slots a call still runs, unsplit.
//   swiglu: [256 amax words][split flags][DYNAMIC: bf16 T x I][partials]
//   mlp:    [256 amax words][split flags][h codes][h scales][s codes]
//           [s scales][DYNAMIC: bf16 T x I][partials]
size_t nvfp4::swiglu_base_workspace_bytes(int64_t T, int64_t I, int inter_mode)
{
    size_t b = 256 + kSplitFlagBytes;
    if (inter_mode == NVFP4_INTER_DYNAMIC) b += align256((size_t)T * (size_t)I * 2);
    return b;
}

size_t nvfp4::mlp_base_workspace_bytes(int64_t T, int64_t H, int64_t I, int inter_mode)
{
    size_t b = 256 + kSplitFlagBytes;                 // amax words, split flags
    b += align256(nvfp4_codes_bytes(T, H));           // h codes
    b += align256(nvfp4_sf_bytes(T, H));              // h scales
    b += align256(nvfp4_codes_bytes(T, I));           // s codes
    b += align256(nvfp4_sf_bytes(T, I));              // s scales
    if (inter_mode == NVFP4_INTER_DYNAMIC) b += align256((size_t)T * (size_t)I * 2);
    return b;
}

extern "C" {

size_t nvfp4_codes_bytes(int64_t rows, int64_t cols)
{
    if (rows < 0 || cols < 0) return 0;
    return (size_t)(rows * (cols / 2));
}

size_t nvfp4_sf_bytes(int64_t rows, int64_t cols)
{
    if (rows < 0 || cols < 0) return 0;
    return (size_t)(pad_to(rows, 128) * pad_to(cols / 16, 4));
}

size_t nvfp4_amax_workspace_bytes(void) { return kAmaxWorkspaceBytes; }

size_t nvfp4_gemm_workspace_bytes(void) { return kSplitFlagBytes + split_partial_bytes(current_device_sms()); }

size_t nvfp4_swiglu_workspace_bytes(int64_t T, int64_t I, int inter_mode)
{
    return nvfp4::swiglu_base_workspace_bytes(T, I, inter_mode) + split_partial_bytes(current_device_sms());
}

size_t nvfp4_mlp_workspace_bytes(int64_t T, int64_t H, int64_t I, int inter_mode)
{
    return nvfp4::mlp_base_workspace_bytes(T, H, I, inter_mode) + split_partial_bytes(current_device_sms());
}

size_t nvfp4_experts_workspace_bytes(int64_t T, int64_t topk, int64_t K, int64_t num_experts)
{
    if (T < 1 || topk < 1 || K < 64 || num_experts < 1) return 0;
    return nvfp4::experts_layout(T, topk, K, num_experts).total;
}

const char* nvfp4_status_string(int status)
{
    switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_MISALIGNED: return "misaligned pointer or pitch";
    case NVFP4_ERR_UNSUPPORTED: return "unsupported device (needs compute capability 10.3, sm_103a)";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_ERR_TIMEOUT: return "device pipeline wait timed out";
    default: return "unknown status";
    }
}

int nvfp4_device_status(int* status_out, int clear)
{
    if (!status_out) return NVFP4_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    NVFP4_TRY(device_info(&d));
    int v = 0;
    NVFP4_CUDA(cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost));
    *status_out = v;
    if (clear) {
        const int zero = 0;
        NVFP4_CUDA(cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice));
    }
    return NVFP4_OK;
}

int nvfp4_amax_scale(const void* x, int64_t rows, int64_t cols, int64_t ldx, const void* norm_w, float eps,
                     float* g_out, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    NVFP4_TRY(check_bf16_matrix(x, rows, cols, ldx));
    if (cols % 8 != 0 || !g_out) return NVFP4_ERR_INVALID_ARG;
    if (norm_w && !aligned(norm_w, 16)) return NVFP4_ERR_MISALIGNED;
    if (!workspace || workspace_bytes < kAmaxWorkspaceBytes) return NVFP4_ERR_WORKSPACE;
    if (!aligned(workspace, 256) || !aligned(g_out, 4)) return NVFP4_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    NVFP4_TRY(device_info(&d));
    NVFP4_CUDA(launch_amax_scale(static_cast<const __nv_bfloat16*>(x), rows, cols, ldx,
                                 static_cast<const __nv_bfloat16*>(norm_w), eps, g_out,
                                 static_cast<uint32_t*>(workspace), d->num_sms, (cudaStream_t)stream));
    return NVFP4_OK;
}

int nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, const void* norm_w, float eps,
                   const float* g, uint8_t* codes, int64_t ld_codes, uint8_t* sf, void* y_out,
                   nvfp4_stream_t stream)
{
    NVFP4_TRY(check_bf16_matrix(x, rows, cols, ldx));
    if (cols % 64 != 0 || !g || !codes || !sf || ld_codes < cols / 2) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(codes, 16) || ld_codes % 16 != 0 || !aligned(sf, 128) || !aligned(g, 4))
        return NVFP4_ERR_MISALIGNED;
    if ((norm_w && !aligned(norm_w, 16)) || (y_out && !aligned(y_out, 16))) return NVFP4_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    NVFP4_TRY(device_info(&d));
    NVFP4_CUDA(launch_quantize(static_cast<const __nv_bfloat16*>(x), rows, cols, ldx,
                               static_cast<const __nv_bfloat16*>(norm_w), eps, g, codes, ld_codes, sf,
                               static_cast<__nv_bfloat16*>(y_out), d->num_sms, (cudaStream_t)stream));
    return NVFP4_OK;
}

int nvfp4_scale_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, const void* norm_w, float eps,
                         float* g_out, uint8_t* codes, int64_t ld_codes, uint8_t* sf, void* workspace,
                         size_t workspace_bytes, nvfp4_stream_t stream)
{
    NVFP4_TRY(check_bf16_matrix(x, rows, cols, ldx));
    if (cols % 64 != 0 || !g_out || !codes || !sf || ld_codes < cols / 2) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(codes, 16) || ld_codes % 16 != 0 || !aligned(sf, 128) || !aligned(g_out, 4))
        return NVFP4_ERR_MISALIGNED;
    if (norm_w && !aligned(norm_w, 16)) return NVFP4_ERR_MISALIGNED;
    if (!workspace || workspace_bytes < kAmaxWorkspaceBytes) return NVFP4_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return NVFP4_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    NVFP4_TRY(device_info(&d));
    NVFP4_CUDA(launch_scale_quantize(static_cast<const __nv_bfloat16*>(x), rows, cols, ldx,
                                     static_cast<const __nv_bfloat16*>(norm_w), eps, g_out, codes, ld_codes, sf,
                                     static_cast<uint32_t*>(workspace), d->status, d->num_sms,
                                     (cudaStream_t)stream));
    return NVFP4_OK;
}

int nvfp4_gemm(const nvfp4_tensor_t* A, const nvfp4_tensor_t* W, void* out, int64_t ldo, const void* residual,
               int64_t ldr, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    return run_linear(A, W, out, ldo, residual, ldr, nullptr, workspace, workspace_bytes, stream);
}

int nvfp4_gemm_rope(const nvfp4_tensor_t* A, const nvfp4_tensor_t* W, void* out, int64_t ldo,
                    const nvfp4_rope_t* rope, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    if (!rope || !rope->pos || !rope->cos_t || !rope->sin_t) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(rope->pos, 4) || !aligned(rope->cos_t, 4) || !aligned(rope->sin_t, 4)) return NVFP4_ERR_MISALIGNED;
    if (rope->head_dim < 2 || rope->head_dim % 2 != 0 || rope->rope_dim < 2 || rope->rope_dim % 2 != 0 ||
        rope->rope_dim > rope->head_dim || rope->col0 < 0 || rope->col0 % 2 != 0 || rope->heads < 0 ||
        rope->table_ld < rope->rope_dim / 2 || rope->positions < 1 || !W ||
        rope->col0 + rope->heads * rope->head_dim > W->rows)
        return NVFP4_ERR_INVALID_ARG;
    return run_linear(A, W, out, ldo, nullptr, 0, rope, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

int run_linear(const nvfp4_tensor_t* A, const nvfp4_tensor_t* W, void* out, int64_t ldo, const void* residual,
               int64_t ldr, const nvfp4_rope_t* rope, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    NVFP4_TRY(check_tensor(A));
    NVFP4_TRY(check_tensor(W));
    if (A->cols != W->cols || W->rows % 16 != 0) return NVFP4_ERR_INVALID_ARG;
    NVFP4_TRY(check_bf16_matrix(out, A->rows, W->rows, ldo));
    if (residual) NVFP4_TRY(check_bf16_matrix(residual, A->rows, W->rows, ldr));
    if (workspace && workspace_bytes < kSplitFlagBytes) return NVFP4_ERR_WORKSPACE;
    if (workspace && !aligned(workspace, 256)) return NVFP4_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    NVFP4_TRY(device_info(&d));
    NVFP4_TRY(encoder());
    CUtensorMap ma, mb;
    NVFP4_TRY(make_codes_map(&ma, A->codes, A->rows, A->cols / 2, A->ld));
    NVFP4_TRY(make_codes_map(&mb, W->codes, W->rows, W->cols / 2, W->ld));
    GemmArgs a = {};
    a.epilogue = kEpiBf16;
    a.M = A->rows;
    a.N = W->rows;
    a.K = A->cols;
    a.sfa = A->sf;
    a.sfb0 = W->sf;
    a.sfa_tile_stride = sf_tile_stride(A->cols);
    a.sfb_tile_stride = sf_tile_stride(W->cols);
    a.ga = A->g;
    a.gb0 = W->g;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.ldo = ldo;
    a.residual = static_cast<const __nv_bfloat16*>(residual);
    a.ldr = ldr;
    a.status = d->status;
    if (rope) {
        a.rope_pos = rope->pos;
        a.rope_cos = rope->cos_t;
        a.rope_sin = rope->sin_t;
        a.rope_ld = rope->table_ld;
        a.rope_col0 = rope->col0;
        a.rope_heads = rope->heads;
        a.rope_hd = rope->head_dim;
        a.rope_rd = rope->rope_dim;
        a.rope_inverse = rope->inverse ? 1 : 0;
    }
    if (workspace) {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        const SplitScratch sp =
            split_scratch(d, ws, ws + kSplitFlagBytes, workspace_bytes - kSplitFlagBytes);
        a.sk_flags = sp.flags;
        a.sk_partials = sp.partials;
    }
    const DecodeOperands ops = {A->codes, A->ld, W->codes, W->ld, W->codes, W->ld};
    NVFP4_CUDA(run_gemm(ma, mb, mb, a, ops, d, (cudaStream_t)stream));
    return NVFP4_OK;
}

}  // namespace

extern "C" {

int nvfp4_gemm_experts(const nvfp4_tensor_t* A, const nvfp4_tensor_t* W, int64_t num_experts, const int32_t* ids,
                       int64_t topk, void* out, int64_t ldo, void* workspace, size_t workspace_bytes,
                       nvfp4_stream_t stream)
{
    NVFP4_TRY(check_tensor(A));
    NVFP4_TRY(check_tensor(W));
    const int64_t E = num_experts;
    if (E < 1 || E > 4096 || topk < 1 || !ids || A->cols != W->cols || W->rows % E != 0)
        return NVFP4_ERR_INVALID_ARG;
    const int64_t N = W->rows / E, T = A->rows, K = A->cols;
    if (N % 128 != 0 || T * topk >= ((int64_t)1 << 31)) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(ids, 4)) return NVFP4_ERR_MISALIGNED;
    NVFP4_TRY(check_bf16_matrix(out, T * topk, N, ldo));
    const ExpertsLayout L = experts_layout(T, topk, K, E);
    if (!workspace || workspace_bytes < L.total) return NVFP4_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return NVFP4_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    NVFP4_TRY(device_info(&d));
    NVFP4_TRY(encoder());
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    CUtensorMap ma, mb;
    NVFP4_TRY(make_codes_map(&ma, ws + L.codes, L.max_rows, K / 2, K / 2));
    NVFP4_TRY(make_codes_map(&mb, W->codes, W->rows, K / 2, W->ld));
    NVFP4_CUDA(launch_experts(A->codes, A->ld, A->sf, A->g, T, K, W->codes, W->ld, W->sf, W->g, N, E, ids, topk,
                              static_cast<__nv_bfloat16*>(out), ldo, ws, ma, mb, d->status, d->num_sms,
                              (cudaStream_t)stream));
    return NVFP4_OK;
}

int nvfp4_gemm_swiglu(const nvfp4_tensor_t* A, const nvfp4_tensor_t* W_gate, const nvfp4_tensor_t* W_up,
                      int inter_mode, float* g_inter, uint8_t* s_codes, int64_t ld_s_codes, uint8_t* s_sf,
                      void* s_bf16, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    NVFP4_TRY(check_swiglu_args(A, W_gate, W_up, inter_mode, g_inter));
    const int64_t T = A->rows, I = W_gate->rows;
    if (!s_codes || !s_sf || ld_s_codes < I / 2) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(s_codes, 16) || ld_s_codes % 16 != 0 || !aligned(s_sf, 128)) return NVFP4_ERR_MISALIGNED;
    if (s_bf16 && !aligned(s_bf16, 16)) return NVFP4_ERR_MISALIGNED;
    const size_t base = swiglu_base_workspace_bytes(T, I, inter_mode);
    if (!workspace || workspace_bytes < base) return NVFP4_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return NVFP4_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    NVFP4_TRY(device_info(&d));
    NVFP4_TRY(encoder());
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    return run_swiglu(d, A, W_gate, W_up, inter_mode, g_inter, s_codes, ld_s_codes, s_sf,
                      static_cast<__nv_bfloat16*>(s_bf16), reinterpret_cast<uint32_t*>(ws),
                      reinterpret_cast<__nv_bfloat16*>(ws + 256 + kSplitFlagBytes),
                      split_scratch(d, ws + 256, ws + base, workspace_bytes - base), false,
                      (cudaStream_t)stream);
}

int nvfp4_mlp(const void* x, int64_t T, int64_t H, int64_t ldx, const void* norm_w, float eps,
              const nvfp4_tensor_t* W_gate, const nvfp4_tensor_t* W_up, const nvfp4_tensor_t* W_down,
              int inter_mode, float* g_inter, void* out, int64_t ldo, int add_residual, void* workspace,
              size_t workspace_bytes, nvfp4_stream_t stream)
{
    NVFP4_TRY(nvfp4::check_mlp_args(x, T, H, ldx, norm_w, W_gate, W_up, W_down, inter_mode, g_inter, out, ldo,
                                    add_residual));
    const int64_t I = W_gate->rows;
    const size_t base = mlp_base_workspace_bytes(T, H, I, inter_mode);
    if (!workspace || workspace_bytes < base) return NVFP4_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return NVFP4_ERR_MISALIGNED;
    DeviceInfo* d = nullptr;
    NVFP4_TRY(device_info(&d));
    NVFP4_TRY(encoder());
    cudaStream_t st = (cudaStream_t)stream;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint32_t* amax_ws = reinterpret_cast<uint32_t*>(ws);          // words 0, 1, 32, 48 (g_h: word 16)
    float* g_h = reinterpret_cast<float*>(ws + 64);
    const SplitScratch split = split_scratch(d, ws + 256, ws + base, workspace_bytes - base);
    size_t off = 256 + kSplitFlagBytes;
    uint8_t* h_codes = ws + off;
    off += align256(nvfp4_codes_bytes(T, H));
    uint8_t* h_sf = ws + off;
    off += align256(nvfp4_sf_bytes(T, H));
    uint8_t* s_codes = ws + off;
    off += align256(nvfp4_codes_bytes(T, I));
    uint8_t* s_sf = ws + off;
    off += align256(nvfp4_sf_bytes(T, I));
    __nv_bfloat16* s_bf16_scratch = reinterpret_cast<__nv_bfloat16*>(ws + off);   // DYNAMIC only

    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    const __nv_bfloat16* nw = static_cast<const __nv_bfloat16*>(norm_w);
    // 1-2: RMSNorm prologue -> device scale -> FP4 input
    NVFP4_CUDA(launch_scale_quantize(xb, T, H, ldx, nw, eps, g_h, h_codes, H / 2, h_sf, amax_ws, d->status,
                                     d->num_sms, st));
    // 3: fused gate/up GEMM + SwiGLU + FP4 requant
    const nvfp4_tensor_t h = {h_codes, h_sf, g_h, T, H, H / 2};
    // the gate/up kernel and the down kernel run one after the other on the
    // stream, so they share the split scratch
    // the weights were complete before the call's first launch (the plain
    // launch of step 1 waits for all earlier work), and no launch of the call
    // writes them: the GEMMs may fetch them early
    NVFP4_TRY(run_swiglu(d, &h, W_gate, W_up, inter_mode, g_inter, s_codes, I / 2, s_sf, nullptr, amax_ws,
                         s_bf16_scratch, split, true, st));
    // 4: down GEMM (+ residual)
    const nvfp4_tensor_t s = {s_codes, s_sf, g_inter, T, I, I / 2};
    GemmArgs a = {};
    a.epilogue = kEpiBf16;
    a.M = T;
    a.N = H;
    a.K = I;
    a.sfa = s.sf;
    a.sfb0 = W_down->sf;
    a.sfa_tile_stride = sf_tile_stride(I);
    a.sfb_tile_stride = sf_tile_stride(I);
    a.ga = g_inter;
    a.gb0 = W_down->g;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.ldo = ldo;
    a.residual = add_residual ? xb : nullptr;
    a.ldr = ldx;
    a.status = d->status;
    a.sk_flags = split.flags;
    a.sk_partials = split.partials;
    a.weights_early = 1;
    CUtensorMap ma, mb;
    NVFP4_TRY(make_codes_map(&ma, s.codes, T, I / 2, I / 2));
    NVFP4_TRY(make_codes_map(&mb, W_down->codes, H, I / 2, W_down->ld));
    const DecodeOperands ops = {s.codes, I / 2, W_down->codes, W_down->ld, W_down->codes, W_down->ld};
    NVFP4_CUDA(run_gemm(ma, mb, mb, a, ops, d, st));
    return NVFP4_OK;
}

#ifdef NVFP4_TRACE
// Debug builds only: copy the GEMM timeline of CTA 0 to the host.
int nvfp4_debug_trace(unsigned long long* out, int n);
#endif

}  // extern "C"
