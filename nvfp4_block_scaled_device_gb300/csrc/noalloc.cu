// nvfp4_mlp_noalloc: the MLP launch set of nvfp4_mlp with its scratch memory
// taken from a fixed array compiled into this library instead of a
// caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory -- for example a
// plugin that only receives borrowed tensor pointers from its host
// application and has no allocator of its own, or code on a latency-critical
// path where cudaMalloc is not acceptable because it may synchronise the
// whole device.  Such callers still pass their inputs and outputs; only the
// intermediates (the quantized normalised input, the quantized SwiGLU
// output, the amax words, and in the per-call-scale mode the bf16 SwiGLU
// output) live in the array below.
#include <mutex>

#include "internal.h"
#include "nvfp4.h"

// The scratch array: every GPU that loads this library holds these bytes
// until the process exits.  Its host-side name is only a stand-in; host code
// must use the device address obtained with cudaGetSymbolAddress.
static constexpr size_t kNoallocScratchBytes = size_t(32) << 20;   // 32 MiB
static __device__ __align__(256) unsigned char g_mlp_scratch[kNoallocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
int scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_mlp_scratch) != cudaSuccess || p == nullptr) return NVFP4_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return NVFP4_OK;
}

}  // namespace

extern "C" int nvfp4_noalloc_scratch(void** device_ptr, size_t* bytes)
{
    if (!device_ptr || !bytes) return NVFP4_ERR_INVALID_ARG;
    const int st = scratch_address(device_ptr);
    if (st != NVFP4_OK) return st;
    *bytes = kNoallocScratchBytes;
    return NVFP4_OK;
}

extern "C" int nvfp4_mlp_noalloc(const void* x, int64_t T, int64_t H, int64_t ldx, const void* norm_w, float eps,
                                 const nvfp4_tensor_t* W_gate, const nvfp4_tensor_t* W_up,
                                 const nvfp4_tensor_t* W_down, int inter_mode, float* g_inter, void* out,
                                 int64_t ldo, int add_residual, nvfp4_stream_t stream)
{
    // every argument error is returned before anything is enqueued
    const int arg = nvfp4::check_mlp_args(x, T, H, ldx, norm_w, W_gate, W_up, W_down, inter_mode, g_inter, out, ldo,
                                          add_residual);
    if (arg != NVFP4_OK) return arg;
    // the intermediates of this call must fit the fixed array (the split
    // schedule's partial slots are used when they fit as well)
    if (nvfp4::mlp_base_workspace_bytes(T, H, W_gate->rows, inter_mode) > kNoallocScratchBytes)
        return NVFP4_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != NVFP4_OK) return st;
    // The array keeps whatever the previous call left.  The amax words and
    // the split schedule's ready flags and tickets at its start must be zero
    // when a call begins (a completed call leaves them zero; a call that
    // stopped early might not), so clear them first.
    if (cudaMemsetAsync(scratch, 0, 256 + nvfp4::kSplitFlagBytes, (cudaStream_t)stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return nvfp4_mlp(x, T, H, ldx, norm_w, eps, W_gate, W_up, W_down, inter_mode, g_inter, out, ldo, add_residual,
                     scratch, kNoallocScratchBytes, stream);
}
