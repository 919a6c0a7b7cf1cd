// vsa_coarse_select_noalloc: the coarse selection without a caller-supplied
// workspace, for callers that cannot allocate device memory themselves.
//
// Who needs it: code that runs inside a host application which owns every
// device allocation (for example an inference-server plugin handed a fixed
// memory plan), or latency-critical loops that must not call cudaMalloc /
// cudaFree because those calls can synchronise the device.  Such callers
// still own and pass the inputs and the output; only the scratch space of
// the coarse stage comes from the library.
//
// The scratch is one file-scope device array of kScratchBytes (64 MiB).
// Every GPU that loads this library reserves it for the life of the process.
// Its device address is looked up with cudaGetSymbolAddress (with the
// device current) on every call made outside a stream capture, so a device
// reset, which reloads the module and may move the array, is picked up by
// the next call; a call made while its stream is capturing uses the address
// found by the last call on that device outside a capture, so make one call
// on each device before capturing.  All calls on a device share the one
// array: calls whose kernels overlap on the GPU (e.g. on two streams at once)
// race on it and must be serialised by the caller.  The array keeps whatever
// the last call left; the kernels here overwrite every byte they read, so no
// clearing is needed.  No cudaMalloc, cudaFree or allocating library routine
// is called.
#include <math.h>

#include <mutex>

#include "vsa_common.cuh"

// Scratch of the allocation-free coarse selection (file scope, one per device).
static __device__ __align__(256) unsigned char g_coarse_scratch[(size_t)64 << 20];

namespace vsa {

namespace {

constexpr size_t kScratchBytes = sizeof(g_coarse_scratch);  // 64 MiB

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device: looked up
// afresh unless `stream` is capturing, then the last address found.
cudaError_t scratch_for_current_device(cudaStream_t stream, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_coarse_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    } else if (!g_scratch_ptr[dev]) {
        return cudaErrorStreamCaptureUnsupported;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace vsa

extern "C" vsa_status vsa_coarse_select_noalloc(const void* qt, const void* kt, const int32_t* vbs, int32_t B,
                                                int32_t ncubes, int32_t heads, int32_t D, int32_t topk,
                                                float sm_scale, int32_t* topk_idx, vsa_stream_t stream) {
    using namespace vsa;
    if (!qt || !kt || !vbs || !topk_idx) return VSA_ERR_INVALID_ARG;
    if (B <= 0 || ncubes <= 0 || heads <= 0 || topk <= 0 || topk > ncubes) return VSA_ERR_INVALID_ARG;
    if (!(sm_scale == sm_scale)) return VSA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return VSA_ERR_UNSUPPORTED;
    if (ncubes > 4096 || !sizes_fit(B, (int64_t)ncubes * 64, heads, D)) return VSA_ERR_UNSUPPORTED;
    // The problem must fit the fixed scratch array: scores through memory when
    // that path is the default and its score matrix fits, else the fused path.
    bool split = coarse_split_default(ncubes, D);
    if (split && coarse_workspace_bytes(B, heads, ncubes, D, true) > kScratchBytes) split = false;
    if (coarse_workspace_bytes(B, heads, ncubes, D, split) > kScratchBytes) return VSA_ERR_UNSUPPORTED;
    if (!aligned16(qt) || !aligned16(kt) || !aligned16(vbs) || (reinterpret_cast<uintptr_t>(topk_idx) & 3u))
        return VSA_ERR_ALIGNMENT;
    DevCtx ctx;
    if (get_dev_ctx(&ctx) != cudaSuccess) return VSA_ERR_CUDA;
    if (coarse_smem_bytes(ncubes, D, split) > (size_t)ctx.max_smem_optin)
        return VSA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (scratch_for_current_device(static_cast<cudaStream_t>(stream), &scratch) != cudaSuccess) return VSA_ERR_CUDA;
    if (sm_scale <= 0.f) sm_scale = 1.0f / sqrtf((float)D);
    return launch_coarse(qt, kt, vbs, B, ncubes, heads, D, topk, sm_scale, scratch, topk_idx, split, false,
                         static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? VSA_OK
               : VSA_ERR_CUDA;
}
