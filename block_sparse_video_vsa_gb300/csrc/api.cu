// C ABI of the VSA library: argument validation on the host, then dispatch
// to the kernels of tile.cu, coarse.cu, pair.cu, fine.cu, coarse_attn.cu and
// block_select.cu
// (coarse_noalloc.cu holds the allocation-free coarse entry point).  See
// include/vsa.h for the contract of each entry point.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "vsa_common.cuh"

namespace vsa {

// Library-wide device error word (one per device that loads the library).
__device__ unsigned int g_device_error;

namespace {
constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_launches{0};
std::mutex g_ctx_mu;
DevCtx g_ctx[kMaxDevices];
bool g_ctx_ok[kMaxDevices];
}  // namespace

void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

// Element counts that index int32 loops in the kernels must stay below 2^31.
bool sizes_fit(int64_t B, int64_t rows, int64_t heads, int64_t D) {
    const int64_t lim = (int64_t)1 << 31;
    return heads * D < lim / 64 && B * rows < lim && B * heads * rows / 64 < lim;
}

cudaError_t get_dev_ctx(DevCtx* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_ctx_mu);
    if (!g_ctx_ok[dev]) {
        DevCtx c;
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_error);
        if (e != cudaSuccess) return e;
        c.err = static_cast<unsigned int*>(p);
        e = cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&c.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        g_ctx[dev] = c;
        g_ctx_ok[dev] = true;
    }
    *out = g_ctx[dev];
    return cudaSuccess;
}

}  // namespace vsa

using namespace vsa;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

vsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? VSA_OK : VSA_ERR_CUDA; }

bool grid_ok(const vsa_grid* g) {
    return g && g->B > 0 && g->T > 0 && g->H > 0 && g->W > 0 && g->heads > 0 && g->D > 0;
}

int64_t cubes_of(const vsa_grid* g) {
    return (int64_t)((g->T + 3) / 4) * ((g->H + 3) / 4) * ((g->W + 3) / 4);
}

}  // namespace

extern "C" {

const char* vsa_status_string(vsa_status s) {
    switch (s) {
        case VSA_OK: return "VSA_OK";
        case VSA_ERR_INVALID_ARG: return "VSA_ERR_INVALID_ARG";
        case VSA_ERR_UNSUPPORTED: return "VSA_ERR_UNSUPPORTED";
        case VSA_ERR_ALIGNMENT: return "VSA_ERR_ALIGNMENT";
        case VSA_ERR_INDEX_RANGE: return "VSA_ERR_INDEX_RANGE";
        case VSA_ERR_TIMEOUT: return "VSA_ERR_TIMEOUT";
        case VSA_ERR_CUDA: return "VSA_ERR_CUDA";
    }
    return "VSA_ERR_UNKNOWN";
}

int64_t vsa_num_cubes(const vsa_grid* g) {
    if (!grid_ok(g)) return -1;
    return cubes_of(g);
}

vsa_status vsa_tile(const vsa_grid* g, const void* x, void* xt, int32_t* vbs, vsa_stream_t stream) {
    if (!grid_ok(g) || !x || !xt) return VSA_ERR_INVALID_ARG;
    if ((g->heads * (int64_t)g->D) % 8 != 0) return VSA_ERR_UNSUPPORTED;
    const int64_t N = cubes_of(g);
    if (!sizes_fit(g->B, N * 64, g->heads, g->D) || (int64_t)g->T * g->H * g->W >= ((int64_t)1 << 31))
        return VSA_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(xt) || (vbs && (reinterpret_cast<uintptr_t>(vbs) & 3u)))
        return VSA_ERR_ALIGNMENT;
    return from_cuda(launch_tile(*g, (int)N, x, xt, vbs, static_cast<cudaStream_t>(stream)));
}

vsa_status vsa_untile(const vsa_grid* g, const void* yt, void* y, vsa_stream_t stream) {
    if (!grid_ok(g) || !yt || !y) return VSA_ERR_INVALID_ARG;
    if ((g->heads * (int64_t)g->D) % 8 != 0) return VSA_ERR_UNSUPPORTED;
    const int64_t N = cubes_of(g);
    if (!sizes_fit(g->B, N * 64, g->heads, g->D) || (int64_t)g->T * g->H * g->W >= ((int64_t)1 << 31))
        return VSA_ERR_UNSUPPORTED;
    if (!aligned16(yt) || !aligned16(y)) return VSA_ERR_ALIGNMENT;
    return from_cuda(launch_untile(*g, (int)N, yt, y, static_cast<cudaStream_t>(stream)));
}

size_t vsa_coarse_workspace_bytes(int32_t B, int32_t heads, int32_t ncubes, int32_t D) {
    if (B <= 0 || heads <= 0 || ncubes <= 0 || D <= 0) return 0;
    return coarse_workspace_bytes(B, heads, ncubes, D, coarse_split_default(ncubes, D));
}

vsa_status vsa_coarse_select(const void* qt, const void* kt, const int32_t* vbs, int32_t B, int32_t ncubes,
                             int32_t heads, int32_t D, int32_t topk, float sm_scale, void* workspace,
                             int32_t* topk_idx, vsa_stream_t stream) {
    if (!qt || !kt || !vbs || !workspace || !topk_idx) return VSA_ERR_INVALID_ARG;
    if (B <= 0 || ncubes <= 0 || heads <= 0 || topk <= 0 || topk > ncubes) return VSA_ERR_INVALID_ARG;
    if (!(sm_scale == sm_scale)) return VSA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return VSA_ERR_UNSUPPORTED;
    if (ncubes > 4096 || !sizes_fit(B, (int64_t)ncubes * 64, heads, D)) return VSA_ERR_UNSUPPORTED;
    if (!aligned16(qt) || !aligned16(kt) || !aligned16(workspace) || !aligned16(vbs) ||
        (reinterpret_cast<uintptr_t>(topk_idx) & 3u))
        return VSA_ERR_ALIGNMENT;
    DevCtx ctx;
    cudaError_t e = get_dev_ctx(&ctx);
    if (e != cudaSuccess) return VSA_ERR_CUDA;
    const bool split = coarse_split_default(ncubes, D);
    const size_t smem = coarse_smem_bytes(ncubes, D, split);
    if (smem > (size_t)ctx.max_smem_optin) return VSA_ERR_UNSUPPORTED;
    if (sm_scale <= 0.f) sm_scale = 1.0f / sqrtf((float)D);
    return from_cuda(launch_coarse(qt, kt, vbs, B, ncubes, heads, D, topk, sm_scale, workspace, topk_idx, split, false,
                                   static_cast<cudaStream_t>(stream)));
}

vsa_status vsa_tile_pool(const vsa_grid* g, const void* q, const void* k, void* qt, void* kt, int32_t* vbs,
                         void* workspace, vsa_stream_t stream) {
    if (!grid_ok(g) || !q || !k || !workspace) return VSA_ERR_INVALID_ARG;
    if (g->D != 64 && g->D != 128) return VSA_ERR_UNSUPPORTED;
    const int64_t N = cubes_of(g);
    if (N > 4096 || !sizes_fit(g->B, N * 64, g->heads, g->D) || (int64_t)g->T * g->H * g->W >= ((int64_t)1 << 31))
        return VSA_ERR_UNSUPPORTED;
    if ((int64_t)g->B * N > 2147483647 || g->heads > 65535) return VSA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || (qt && !aligned16(qt)) || (kt && !aligned16(kt)) || !aligned16(workspace) ||
        (vbs && (reinterpret_cast<uintptr_t>(vbs) & 3u)))
        return VSA_ERR_ALIGNMENT;
    return from_cuda(launch_tile_pool(*g, (int)N, q, k, qt, kt, vbs, workspace, static_cast<cudaStream_t>(stream)));
}

vsa_status vsa_coarse_select_pooled(const int32_t* vbs, int32_t B, int32_t ncubes, int32_t heads, int32_t D,
                                    int32_t topk, float sm_scale, void* workspace, int32_t* topk_idx,
                                    vsa_stream_t stream) {
    if (!vbs || !workspace || !topk_idx) return VSA_ERR_INVALID_ARG;
    if (B <= 0 || ncubes <= 0 || heads <= 0 || topk <= 0 || topk > ncubes) return VSA_ERR_INVALID_ARG;
    if (!(sm_scale == sm_scale)) return VSA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return VSA_ERR_UNSUPPORTED;
    if (ncubes > 4096 || !sizes_fit(B, (int64_t)ncubes * 64, heads, D)) return VSA_ERR_UNSUPPORTED;
    if (!aligned16(workspace) || !aligned16(vbs) || (reinterpret_cast<uintptr_t>(topk_idx) & 3u))
        return VSA_ERR_ALIGNMENT;
    DevCtx ctx;
    cudaError_t e = get_dev_ctx(&ctx);
    if (e != cudaSuccess) return VSA_ERR_CUDA;
    const bool split = coarse_split_default(ncubes, D);
    if (coarse_smem_bytes(ncubes, D, split) > (size_t)ctx.max_smem_optin) return VSA_ERR_UNSUPPORTED;
    if (sm_scale <= 0.f) sm_scale = 1.0f / sqrtf((float)D);
    return from_cuda(launch_coarse(nullptr, nullptr, vbs, B, ncubes, heads, D, topk, sm_scale, workspace, topk_idx,
                                   split, true, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Every fine-stage entry point: validation, then one launch of the fine kernel.
vsa_status fine_entry(const void* qt, const void* kt, const void* vt, const int32_t* topk_idx, const int32_t* counts,
                      const int32_t* vbs, const uint32_t* pairs, int32_t B, int32_t ncubes, int32_t heads, int32_t D,
                      int32_t topk, float sm_scale, const float* coarse_out, const void* gate_c, const void* gate_f,
                      void* out, float* lse, float* max_prob, vsa_stream_t stream, const vsa_grid* raster = nullptr) {
    if (!qt || !kt || !vt || !topk_idx || !vbs || !out) return VSA_ERR_INVALID_ARG;
    const bool gated = coarse_out || gate_c || gate_f;
    if (gated && (!coarse_out || !gate_c || !gate_f)) return VSA_ERR_INVALID_ARG;
    if (raster) {
        // q and out in raster order of this grid; k, v, topk_idx on its cubes.
        if (!grid_ok(raster) || gated) return VSA_ERR_INVALID_ARG;
        if (raster->B != B || raster->heads != heads || raster->D != D || cubes_of(raster) != ncubes)
            return VSA_ERR_INVALID_ARG;
        if ((int64_t)B * raster->T * raster->H * raster->W >= ((int64_t)1 << 31)) return VSA_ERR_UNSUPPORTED;
    }
    if (B <= 0 || ncubes <= 0 || heads <= 0 || topk <= 0 || topk > ncubes) return VSA_ERR_INVALID_ARG;
    if (!(sm_scale == sm_scale)) return VSA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return VSA_ERR_UNSUPPORTED;
    if (!sizes_fit(B, (int64_t)ncubes * 64, heads, D) || (int64_t)B * ncubes * 64 >= ((int64_t)1 << 31) ||
        (int64_t)B * heads * ncubes >= ((int64_t)1 << 31))
        return VSA_ERR_UNSUPPORTED;
    if (heads > 65535) return VSA_ERR_UNSUPPORTED;  // TMA box coordinate range
    if (topk > fine_max_topk() || ncubes > fine_max_cubes()) return VSA_ERR_UNSUPPORTED;
    if (!aligned16(qt) || !aligned16(kt) || !aligned16(vt) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(topk_idx) & 3u) || (reinterpret_cast<uintptr_t>(vbs) & 3u) ||
        (reinterpret_cast<uintptr_t>(pairs) & 3u) || (reinterpret_cast<uintptr_t>(counts) & 3u) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
        (max_prob && (reinterpret_cast<uintptr_t>(max_prob) & 3u)) ||
        (gated && (!aligned16(coarse_out) || !aligned16(gate_c) || !aligned16(gate_f))))
        return VSA_ERR_ALIGNMENT;
    DevCtx ctx;
    cudaError_t e = get_dev_ctx(&ctx);
    if (e != cudaSuccess) return VSA_ERR_CUDA;
    if (fine_smem_bytes() > ctx.max_smem_optin) return VSA_ERR_UNSUPPORTED;
    if (sm_scale <= 0.f) sm_scale = 1.0f / sqrtf((float)D);
    return from_cuda(launch_fine(qt, kt, vt, topk_idx, counts, vbs, pairs, B, ncubes, heads, D, topk, sm_scale,
                                 coarse_out, gate_c, gate_f, out, lse, max_prob, raster, ctx.err, ctx.num_sms,
                                 static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

vsa_status vsa_sparse_attn_fwd_gated(const void* qt, const void* kt, const void* vt, const int32_t* topk_idx,
                                     const int32_t* counts, const int32_t* vbs, const uint32_t* pairs, int32_t B,
                                     int32_t ncubes, int32_t heads, int32_t D, int32_t topk, float sm_scale,
                                     const float* coarse_out, const void* gate_c, const void* gate_f, void* out,
                                     float* lse, vsa_stream_t stream) {
    return fine_entry(qt, kt, vt, topk_idx, counts, vbs, pairs, B, ncubes, heads, D, topk, sm_scale, coarse_out,
                      gate_c, gate_f, out, lse, nullptr, stream);
}

vsa_status vsa_sparse_attn_fwd_peak(const void* qt, const void* kt, const void* vt, const int32_t* topk_idx,
                                    const int32_t* counts, const int32_t* vbs, const uint32_t* pairs, int32_t B,
                                    int32_t ncubes, int32_t heads, int32_t D, int32_t topk, float sm_scale, void* out,
                                    float* lse, float* max_prob, vsa_stream_t stream) {
    if (!max_prob) return VSA_ERR_INVALID_ARG;
    return fine_entry(qt, kt, vt, topk_idx, counts, vbs, pairs, B, ncubes, heads, D, topk, sm_scale, nullptr, nullptr,
                      nullptr, out, lse, max_prob, stream);
}


vsa_status vsa_sparse_attn_fwd_raster(const vsa_grid* g, const void* q, const void* kt, const void* vt,
                                      const int32_t* topk_idx, const int32_t* counts, const int32_t* vbs,
                                      const uint32_t* pairs, int32_t topk, float sm_scale, void* out, float* lse,
                                      vsa_stream_t stream) {
    if (!grid_ok(g)) return VSA_ERR_INVALID_ARG;
    const int64_t N = cubes_of(g);
    if (N > 2147483647) return VSA_ERR_UNSUPPORTED;
    return fine_entry(q, kt, vt, topk_idx, counts, vbs, pairs, g->B, (int32_t)N, g->heads, g->D, topk, sm_scale,
                      nullptr, nullptr, nullptr, out, lse, nullptr, stream, g);
}

vsa_status vsa_sparse_attn_fwd_ex(const void* qt, const void* kt, const void* vt, const int32_t* topk_idx,
                                  const int32_t* counts, const int32_t* vbs, const uint32_t* pairs, int32_t B,
                                  int32_t ncubes, int32_t heads, int32_t D, int32_t topk, float sm_scale,
                                  void* out, float* lse, vsa_stream_t stream) {
    return vsa_sparse_attn_fwd_gated(qt, kt, vt, topk_idx, counts, vbs, pairs, B, ncubes, heads, D, topk, sm_scale,
                                     nullptr, nullptr, nullptr, out, lse, stream);
}

size_t vsa_coarse_attn_workspace_bytes(int32_t B, int32_t heads, int32_t ncubes, int32_t D) {
    if (B <= 0 || heads <= 0 || ncubes <= 0 || (D != 64 && D != 128)) return 0;
    return coarse_attn_workspace_bytes(B, heads, ncubes, D);
}

vsa_status vsa_coarse_attn(const void* qt, const void* kt, const void* vt, const int32_t* vbs, int32_t B,
                           int32_t ncubes, int32_t heads, int32_t D, float sm_scale, void* workspace,
                           float* coarse_out, vsa_stream_t stream) {
    if (!qt || !kt || !vt || !vbs || !workspace || !coarse_out) return VSA_ERR_INVALID_ARG;
    if (B <= 0 || ncubes <= 0 || heads <= 0) return VSA_ERR_INVALID_ARG;
    if (!(sm_scale == sm_scale)) return VSA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return VSA_ERR_UNSUPPORTED;
    if (!sizes_fit(B, (int64_t)ncubes * 64, heads, D) || B > 65535 || heads > 65535 ||
        (int64_t)B * ncubes >= ((int64_t)1 << 31))
        return VSA_ERR_UNSUPPORTED;
    if (!aligned16(qt) || !aligned16(kt) || !aligned16(vt) || !aligned16(workspace) || !aligned16(coarse_out) ||
        (reinterpret_cast<uintptr_t>(vbs) & 3u))
        return VSA_ERR_ALIGNMENT;
    if (sm_scale <= 0.f) sm_scale = 1.0f / sqrtf((float)D);
    return from_cuda(launch_coarse_attn(qt, kt, vt, vbs, B, ncubes, heads, D, sm_scale, workspace, coarse_out,
                                        static_cast<cudaStream_t>(stream)));
}

vsa_status vsa_sparse_attn_fwd_paired(const void* qt, const void* kt, const void* vt, const int32_t* topk_idx,
                                      const int32_t* vbs, const uint32_t* pairs, int32_t B, int32_t ncubes,
                                      int32_t heads, int32_t D, int32_t topk, float sm_scale, void* out, float* lse,
                                      vsa_stream_t stream) {
    return vsa_sparse_attn_fwd_ex(qt, kt, vt, topk_idx, nullptr, vbs, pairs, B, ncubes, heads, D, topk, sm_scale,
                                  out, lse, stream);
}

vsa_status vsa_sparse_attn_fwd(const void* qt, const void* kt, const void* vt, const int32_t* topk_idx,
                               const int32_t* vbs, int32_t B, int32_t ncubes, int32_t heads, int32_t D,
                               int32_t topk, float sm_scale, void* out, float* lse, vsa_stream_t stream) {
    return vsa_sparse_attn_fwd_ex(qt, kt, vt, topk_idx, nullptr, vbs, nullptr, B, ncubes, heads, D, topk,
                                  sm_scale, out, lse, stream);
}

size_t vsa_block_select_workspace_bytes(int32_t B, int32_t S, int32_t heads, int32_t D) {
    if (B <= 0 || heads <= 0 || S <= 0 || S % 128 || (D != 64 && D != 128)) return 0;
    return block_select_workspace_bytes(B, heads, S / 128, D);
}

vsa_status vsa_block_select(const void* q, const void* k, int32_t B, int32_t S, int32_t heads, int32_t D, float tau,
                            float sm_scale, void* workspace, int32_t* cube_idx, int32_t* cube_counts,
                            vsa_stream_t stream) {
    if (!q || !k || !workspace || !cube_idx || !cube_counts) return VSA_ERR_INVALID_ARG;
    if (B <= 0 || S <= 0 || heads <= 0 || S % 128) return VSA_ERR_INVALID_ARG;
    if (!(tau > 0.f && tau <= 1.f) || !(sm_scale == sm_scale)) return VSA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return VSA_ERR_UNSUPPORTED;
    if (S / 128 > block_select_max_blocks() || B > 65535 || heads > 65535 ||
        !sizes_fit(B, S, heads, D))
        return VSA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(cube_idx) & 3u) ||
        (reinterpret_cast<uintptr_t>(cube_counts) & 3u))
        return VSA_ERR_ALIGNMENT;
    if (sm_scale <= 0.f) sm_scale = 1.0f / sqrtf((float)D);
    return from_cuda(launch_block_select(q, k, B, S, heads, D, tau, sm_scale, workspace, cube_idx, cube_counts,
                                         static_cast<cudaStream_t>(stream)));
}

size_t vsa_pair_workspace_bytes(int32_t B, int32_t heads, int32_t ncubes, int32_t topk) {
    if (B <= 0 || heads <= 0 || ncubes <= 0 || topk <= 0) return 0;
    return pair_workspace_bytes(B, heads, ncubes, topk);
}

vsa_status vsa_pair_cubes(const int32_t* topk_idx, int32_t B, int32_t ncubes, int32_t heads, int32_t topk,
                          void* workspace, uint32_t* pairs, vsa_stream_t stream) {
    if (!topk_idx || !workspace || !pairs) return VSA_ERR_INVALID_ARG;
    if (B <= 0 || ncubes <= 0 || heads <= 0 || topk <= 0 || topk > ncubes) return VSA_ERR_INVALID_ARG;
    if (ncubes > pair_max_cubes() || topk > pair_max_topk() || (int64_t)B * heads > 65535 ||
        (int64_t)B * heads * ncubes >= ((int64_t)1 << 31) ||
        (int64_t)B * heads * ncubes * topk >= ((int64_t)1 << 40))
        return VSA_ERR_UNSUPPORTED;
    if (!aligned16(workspace) || (reinterpret_cast<uintptr_t>(topk_idx) & 3u) ||
        (reinterpret_cast<uintptr_t>(pairs) & 3u))
        return VSA_ERR_ALIGNMENT;
    DevCtx ctx;
    if (get_dev_ctx(&ctx) != cudaSuccess) return VSA_ERR_CUDA;
    return from_cuda(launch_pair(topk_idx, B, ncubes, heads, topk, workspace, pairs, ctx.num_sms,
                                 ctx.max_smem_optin, static_cast<cudaStream_t>(stream)));
}

vsa_status vsa_validate_indices_ex(const int32_t* topk_idx, const int32_t* counts, const int32_t* vbs, int32_t B,
                                   int32_t heads, int32_t ncubes, int32_t topk, int32_t* dev_flag,
                                   vsa_stream_t stream) {
    if (!topk_idx || !vbs || !dev_flag) return VSA_ERR_INVALID_ARG;
    if (B <= 0 || heads <= 0 || ncubes <= 0 || topk <= 0) return VSA_ERR_INVALID_ARG;
    if (ncubes > validate_max_cubes() || (int64_t)B * heads * ncubes >= ((int64_t)1 << 31))
        return VSA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(topk_idx) & 3u) || (reinterpret_cast<uintptr_t>(vbs) & 3u) ||
        (reinterpret_cast<uintptr_t>(counts) & 3u) || (reinterpret_cast<uintptr_t>(dev_flag) & 3u))
        return VSA_ERR_ALIGNMENT;
    return from_cuda(launch_validate(topk_idx, counts, vbs, B * heads * ncubes, ncubes, topk, dev_flag,
                                     static_cast<cudaStream_t>(stream)));
}

vsa_status vsa_validate_indices(const int32_t* topk_idx, const int32_t* vbs, int32_t B, int32_t heads,
                                int32_t ncubes, int32_t topk, int32_t* dev_flag, vsa_stream_t stream) {
    return vsa_validate_indices_ex(topk_idx, nullptr, vbs, B, heads, ncubes, topk, dev_flag, stream);
}

vsa_status vsa_device_error(uint32_t* out, int32_t reset) {
    if (!out) return VSA_ERR_INVALID_ARG;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return VSA_ERR_CUDA;
    *out = v;
    if (reset) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_device_error, &z, sizeof z) != cudaSuccess) return VSA_ERR_CUDA;
    }
    return VSA_OK;
}

vsa_status vsa_debug_wait_timeout(int64_t limit_ns, int32_t* dev_result, vsa_stream_t stream) {
    if (!dev_result || limit_ns < 1000 || limit_ns > 10000000000ll) return VSA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(dev_result) & 3u) return VSA_ERR_ALIGNMENT;
    DevCtx ctx;
    if (get_dev_ctx(&ctx) != cudaSuccess) return VSA_ERR_CUDA;
    return from_cuda(launch_debug_wait((long long)limit_ns, dev_result, ctx.err, static_cast<cudaStream_t>(stream)));
}

uint64_t vsa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

vsa_status vsa_table_from_csr(const int64_t* lut_ptr, const int32_t* kv_idx, int64_t nnz, int64_t rows,
                              int32_t width, int32_t ncubes, int32_t* table, int32_t* counts) {
    if (!lut_ptr || !table || !counts || rows <= 0 || width <= 0 || nnz < 0 || ncubes <= 0)
        return VSA_ERR_INVALID_ARG;
    if (lut_ptr[0] != 0) return VSA_ERR_INVALID_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t n = lut_ptr[r + 1] - lut_ptr[r];
        if (n < 0 || n > width) return VSA_ERR_INVALID_ARG;
    }
    if (lut_ptr[rows] > nnz) return VSA_ERR_INVALID_ARG;  // the offsets run past kv_idx
    if (lut_ptr[rows] > 0 && !kv_idx) return VSA_ERR_INVALID_ARG;
    for (int64_t e = 0; e < lut_ptr[rows]; ++e)
        if (kv_idx[e] < 0 || kv_idx[e] >= ncubes) return VSA_ERR_INDEX_RANGE;
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t b = lut_ptr[r];
        const int32_t n = (int32_t)(lut_ptr[r + 1] - b);
        int32_t* row = table + r * (int64_t)width;
        for (int32_t e = 0; e < n; ++e) row[e] = kv_idx[b + e];
        for (int32_t e = n; e < width; ++e) row[e] = -1;
        counts[r] = n;
    }
    return VSA_OK;
}

}  // extern "C"
