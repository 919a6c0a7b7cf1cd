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
// Its device address is looked up once per device (cudaGetSymbolAddress,
// with that device current) on the first call made on that device; make that
// first call before any stream capture.  All calls on a device share the one
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

// Device address of the scratch array on the current device (set up on the
// first call per device).
cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_coarse_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
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
    if (ncubes > 4096) return VSA_ERR_UNSUPPORTED;
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
    if (scratch_for_current_device(&scratch) != cudaSuccess) return VSA_ERR_CUDA;
    if (sm_scale <= 0.f) sm_scale = 1.0f / sqrtf((float)D);
    return launch_coarse(qt, kt, vbs, B, ncubes, heads, D, topk, sm_scale, scratch, topk_idx, split,
                         static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? VSA_OK
               : VSA_ERR_CUDA;
}
