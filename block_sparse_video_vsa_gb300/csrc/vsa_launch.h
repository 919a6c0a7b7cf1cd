// Host-side launchers shared between the kernel files and the C ABI layer
// (internal; not part of the public interface).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/vsa.h"

namespace vsa {

// api.cu: counts kernel launches (n kernels enqueued by the caller).
void note_launches(int n);
// api.cu: element counts that index int32 loops in the kernels stay below 2^31.
bool sizes_fit(int64_t B, int64_t rows, int64_t heads, int64_t D);

// tile.cu
cudaError_t launch_tile(const vsa_grid& g, int ncubes, const void* x, void* xt, int32_t* vbs,
                        cudaStream_t stream);
cudaError_t launch_untile(const vsa_grid& g, int ncubes, const void* yt, void* y, cudaStream_t stream);
cudaError_t launch_tile_pool(const vsa_grid& g, int ncubes, const void* q, const void* k, void* qt, void* kt,
                             int32_t* vbs, void* workspace, cudaStream_t stream);

// coarse.cu
bool coarse_split_default(int ncubes, int D);
size_t coarse_workspace_bytes(int B, int heads, int ncubes, int D, bool split);
size_t coarse_smem_bytes(int N, int D, bool split);
int coarse_rows_per_block(int ncubes, int D);
cudaError_t launch_coarse(const void* qt, const void* kt, const int32_t* vbs, int B, int ncubes, int heads,
                          int D, int topk, float sm_scale, void* workspace, int32_t* topk_idx,
                          bool split, bool pooled, cudaStream_t stream);
cudaError_t launch_validate(const int32_t* idx, const int32_t* counts, const int32_t* vbs, int rows, int ncubes,
                            int topk, int32_t* flag, cudaStream_t stream);
int validate_max_cubes();
cudaError_t launch_debug_wait(long long limit_ns, int32_t* result, unsigned int* err, cudaStream_t stream);

// fine.cu
int fine_smem_bytes();
int fine_max_topk();
int fine_max_cubes();
cudaError_t launch_fine(const void* qt, const void* kt, const void* vt, const int32_t* topk_idx,
                        const int32_t* counts, const int32_t* vbs, const uint32_t* pairs, int B, int ncubes,
                        int heads, int D, int topk, float sm_scale, const float* coarse_out, const void* gate_c,
                        const void* gate_f, void* out, float* lse, float* max_prob, const vsa_grid* raster,
                        unsigned int* err, int num_sms, cudaStream_t stream);

// coarse_attn.cu
size_t coarse_attn_workspace_bytes(int B, int heads, int ncubes, int D);
cudaError_t launch_coarse_attn(const void* qt, const void* kt, const void* vt, const int32_t* vbs, int B,
                               int ncubes, int heads, int D, float sm_scale, void* workspace, float* out,
                               cudaStream_t stream);

// block_select.cu
size_t block_select_workspace_bytes(int B, int heads, int nb, int D);
int block_select_max_blocks();
cudaError_t launch_block_select(const void* q, const void* k, int B, int S, int heads, int D, float tau,
                                float sm_scale, void* workspace, int32_t* cube_idx, int32_t* cube_counts,
                                cudaStream_t stream);

// pair.cu
int pair_words(int ncubes);
size_t pair_workspace_bytes(int B, int heads, int ncubes, int topk);
int pair_max_cubes();
int pair_max_topk();
cudaError_t launch_pair(const int32_t* topk_idx, int B, int ncubes, int heads, int topk, void* workspace,
                        uint32_t* pairs, int num_sms, int max_smem, cudaStream_t stream);

}  // namespace vsa
