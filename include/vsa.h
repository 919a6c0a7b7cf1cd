/*
 * vsa.h -- C ABI of the GB300 (sm_103a) Video Sparse Attention hot path.
 *
 * The library implements the data path of Video Sparse Attention (VSA):
 *   1. vsa_tile            cube tiling of a (T, H, W) latent token grid into
 *                          zero-padded 4x4x4 cubes plus the per-cube real-token
 *                          count vbs;
 *   2. vsa_coarse_select   cube mean-pool of Q and K, cube-to-cube scores and
 *                          the top-k key/value cubes per query cube;
 *      (vsa_tile_pool + vsa_coarse_select_pooled: steps 1 and 2 with one
 *                          read of q and k; vsa_sparse_attn_fwd_raster:
 *                          step 3 on raster q and out; same results)
 *   3. vsa_sparse_attn_fwd non-causal block-sparse attention over the selected
 *                          cubes, padded tokens masked (bf16 out + fp32 LSE);
 *      (vsa_pair_cubes     optional schedule for step 3: which query cubes
 *                          share a tensor-core tile; results are unchanged)
 *   4. vsa_untile          the inverse permutation of step 1.
 * and, beside them, the coarse stage's own attention output
 * (vsa_coarse_attn) and its gated sum with the fine output
 * (vsa_sparse_attn_fwd_gated), and a mean-pool block selector with a
 * cumulative threshold for sequences in 128-token blocks
 * (vsa_block_select).
 *
 * Sources (page title, section):
 *   [VSA-AMD] "VSA: Accelerating Video Diffusion Inference with Sparse
 *             Attention on AMD GPUs": Two-Stage Architecture, Block-Sparse
 *             Encoding, Kernel Architecture, Sparse Traversal, Generating
 *             Sparsity Patterns.
 *   [WAN-VSA] "Wan2.2 Production Values -- VSA Block-Sparse Attention Inputs +
 *             Reference": Shapes, Operator contract.
 *   [STA]     "FastVideo Guide: Sliding Tile Attention": Implementation
 *             (tile partition and inverse permutation).
 *   [INT8-WAN] "Optimizing block-sparse INT8 attention and multi-expert step
 *             caching for Wan 2.2": Decoupling Block Selection from Sparse
 *             CUDA Kernels, Dynamic Sparsity Budgeting via Softmax
 *             Normalizer Registers.
 *
 * Conventions shared by every entry point
 *   - Layout: token tensors are BSHD, i.e. [B, S, heads, D] row-major,
 *     contiguous, bf16 (IEEE bfloat16 bit patterns).  "Tiled" tensors have
 *     S = S_pad = 64 * ncubes; "raster" tensors have S = T * H * W with token
 *     n = (t * H + h) * W + w.
 *   - Cube order is raster over the cube grid: cube c = (ct * nh + ch) * nw + cw
 *     with nt = ceil(T/4), nh = ceil(H/4), nw = ceil(W/4).  Inside a cube the
 *     real tokens of its clipped sub-box occupy slots 0 .. vbs[c]-1 in raster
 *     (t, h, w) order; slots vbs[c] .. 63 are padding.
 *   - vbs is int32 [ncubes], shared by every batch entry and head.
 *   - Ownership: the caller allocates and owns every buffer (device memory
 *     unless stated) and the stream.  The library allocates no memory.
 *     Every call is asynchronous on `stream`; results are ready when the
 *     stream reaches that point.
 *   - Host threads: entry points may be called from several host threads at
 *     once, on any streams; the only state they share is a per-device
 *     context set up once under a lock and the launch counter (atomic).
 *     vsa_coarse_select_noalloc's device scratch is the exception (see there).
 *   - Alignment: device pointers must be 16-byte aligned.
 *   - Errors: argument checks run on the host before any launch and return a
 *     status without touching memory.  Launch failures return VSA_ERR_CUDA.
 *     Faults of a launched kernel surface at the caller's next
 *     synchronisation.  Kernels never trap: a bounded wait that runs out sets
 *     a device error word (see vsa_device_error) and the kernel returns.
 *   - In-place operation is not supported (outputs must not alias inputs).
 *   - Results are bit-reproducible from run to run on the same device.
 */
#ifndef VSA_H_
#define VSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t / CUstream); NULL = legacy default stream. */
typedef void* vsa_stream_t;

typedef enum {
    VSA_OK = 0,
    VSA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, topk out of range */
    VSA_ERR_UNSUPPORTED = 2, /* D not in {64, 128}, or a size beyond a stated limit */
    VSA_ERR_ALIGNMENT = 3,   /* a device pointer is not 16-byte aligned */
    VSA_ERR_INDEX_RANGE = 4, /* vsa_validate_indices found a bad index or count */
    VSA_ERR_TIMEOUT = 5,     /* a device-side bounded wait ran out */
    VSA_ERR_CUDA = 6         /* a CUDA runtime/driver call failed */
} vsa_status;

/* Latent token grid: batch B, T x H x W tokens, `heads` heads of size D. */
typedef struct {
    int32_t B, T, H, W, heads, D;
} vsa_grid;

/* Device error word bits (vsa_device_error). */
#define VSA_DEVERR_TIMEOUT 0x1u /* a bounded mbarrier wait in a kernel ran out */

/* Human-readable name of a status code.  Never NULL. */
const char* vsa_status_string(vsa_status s);

/*
 * Number of 4x4x4 cubes covering the grid: ceil(T/4) * ceil(H/4) * ceil(W/4)
 * ([WAN-VSA] Shapes: 624 = 6 x 8 x 13 for 21 x 30 x 52).  Returns -1 for a
 * NULL or non-positive grid.
 */
int64_t vsa_num_cubes(const vsa_grid* g);

/*
 * Cube tiling ([VSA-AMD] Two-Stage Architecture, Pre-stage and Stage 1 cube
 * partition; [WAN-VSA] Shapes "cube-major tiled/padded").
 *   x   : raster bf16 [B, T*H*W, heads, D]              (read)
 *   xt  : tiled  bf16 [B, 64*ncubes, heads, D]         (written in full;
 *         padding slots are written as zero)
 *   vbs : int32 [ncubes] real tokens per cube, or NULL   (written)
 * Any D >= 8 with heads * D a multiple of 8 is accepted (rows are copied as
 * 16-byte vectors).
 */
vsa_status vsa_tile(const vsa_grid* g, const void* x, void* xt, int32_t* vbs, vsa_stream_t stream);

/*
 * Inverse of vsa_tile on the real slots ([STA] Implementation, inverse
 * permutation); padding slots of yt are ignored.
 *   yt : tiled  bf16 [B, 64*ncubes, heads, D]   (read)
 *   y  : raster bf16 [B, T*H*W, heads, D]      (written in full)
 */
vsa_status vsa_untile(const vsa_grid* g, const void* yt, void* y, vsa_stream_t stream);

/*
 * Bytes of device workspace vsa_coarse_select needs: 16 * B * heads * ncubes
 * * D + 8 * B * heads * ncubes (per cube and head: the fp32 mean of Q and K,
 * an fp32 residual that makes the channel sums exact to ~2^-48, and the norm
 * of each mean), plus 4 * B * heads * ncubes^2 for the fp32 score matrix
 * when ncubes >= 256 (the scores then go through memory: a score GEMM, then
 * a per-row selection).  0 for bad sizes.
 */
size_t vsa_coarse_workspace_bytes(int32_t B, int32_t heads, int32_t ncubes, int32_t D);

/*
 * Coarse selection ([VSA-AMD] Stage 1: Coarse Selection and Generating
 * Sparsity Patterns).  For every (b, head, query cube i):
 *   q_mean_i = (1 / vbs[i]) * sum_{s < vbs[i]} qt[b, 64 i + s, head, :]
 *   k_mean_j likewise from kt,
 *   score_ij = sm_scale * (q_mean_i . k_mean_j),
 *   topk_idx[b, head, i, :] = the topk cubes j with the largest score_ij,
 *   ties broken toward the lower cube index; the row lists them in
 *   ascending cube index.
 * A cube with vbs = 0 pools to the zero vector.  Scores are formed in fp32
 * with a proven error bound; rows whose k-th boundary falls inside that bound
 * are re-ranked with exact cube sums in fp64, so the selected set equals the
 * exact-arithmetic top-k except where exact scores tie to ~1e-13 relative.
 *   qt, kt    : tiled bf16 [B, 64*ncubes, heads, D]
 *   vbs       : int32 [ncubes], each in [0, 64]
 *   topk      : 1 <= topk <= ncubes
 *   sm_scale  : score scale; <= 0 means 1/sqrt(D)
 *   workspace : device buffer of vsa_coarse_workspace_bytes(...) bytes,
 *               16-byte aligned; contents need not be initialised
 *   topk_idx  : int32 [B, heads, ncubes, topk] (written)
 * Limits: D in {64, 128}; ncubes <= 4096.
 */
vsa_status vsa_coarse_select(const void* qt, const void* kt, const int32_t* vbs, int32_t B,
                             int32_t ncubes, int32_t heads, int32_t D, int32_t topk,
                             float sm_scale, void* workspace, int32_t* topk_idx,
                             vsa_stream_t stream);

/*
 * Steps 1 and 2 with one read of q and k: vsa_tile of q and of k in a single
 * launch that also writes, into `workspace`, the pooled cube statistics the
 * coarse selection starts from (the same bits vsa_coarse_select computes from
 * the tiled tensors), then vsa_coarse_select_pooled scores and selects from
 * them without reading qt and kt again.  Same sources as vsa_tile and
 * vsa_coarse_select; no counterpart of its own on the pages: it fuses two of
 * their steps.
 *   q, k      : raster bf16 [B, T*H*W, heads, D]        (read)
 *   qt, kt    : tiled bf16 [B, 64*ncubes, heads, D]    (written as vsa_tile),
 *               or NULL: that tiled copy is skipped (the statistics are
 *               still computed; vsa_sparse_attn_fwd_raster reads raster q)
 *   vbs       : int32 [ncubes] or NULL                  (written as vsa_tile)
 *   workspace : vsa_coarse_workspace_bytes(B, heads, ncubes, D) bytes,
 *               16-byte aligned; its pooled-statistics head is written
 * Limits: D in {64, 128}; ncubes <= 4096 (those of vsa_coarse_select).
 */
vsa_status vsa_tile_pool(const vsa_grid* g, const void* q, const void* k, void* qt, void* kt, int32_t* vbs,
                         void* workspace, vsa_stream_t stream);

/*
 * vsa_coarse_select on statistics vsa_tile_pool left in `workspace` (same
 * B, heads, ncubes, D; nothing else may have written the workspace since):
 * the same topk_idx bits, without reading the tiled q and k.
 *   vbs       : int32 [ncubes] as vsa_tile_pool wrote it
 *   workspace : the buffer vsa_tile_pool wrote (read; its score area written)
 *   other arguments, results and errors as vsa_coarse_select.
 */
vsa_status vsa_coarse_select_pooled(const int32_t* vbs, int32_t B, int32_t ncubes, int32_t heads, int32_t D,
                                    int32_t topk, float sm_scale, void* workspace, int32_t* topk_idx,
                                    vsa_stream_t stream);

/*
 * vsa_coarse_select without a workspace argument, for callers that cannot
 * allocate device memory: code running inside a host application that owns
 * every device allocation (e.g. a plugin given a fixed memory plan), or
 * loops that must avoid cudaMalloc/cudaFree because those can synchronise
 * the device.  The paper has no counterpart; it is a deployment variant.
 * Same arguments, results and errors as vsa_coarse_select, except:
 *   - the scratch is a 64 MiB device array inside the library, reserved on
 *     every GPU that loads the library until the process exits.  The
 *     problem uses the score-matrix form of the selection when that is
 *     vsa_coarse_select's choice and its workspace (the value
 *     vsa_coarse_workspace_bytes returns) fits in 64 MiB; otherwise the
 *     fused form, whose workspace is 16 * B * heads * ncubes * D
 *     + 8 * B * heads * ncubes bytes.  VSA_ERR_UNSUPPORTED when that too
 *     exceeds 64 MiB, or the fused form's shared memory does not fit;
 *   - every call made outside a stream capture looks up the array's device
 *     address (cudaGetSymbolAddress, with the call's device current), so a
 *     device reset is picked up; a call made while its stream is capturing
 *     reuses the address its device's last such lookup found (VSA_ERR_CUDA
 *     if there was none), so make one call per device before capturing;
 *   - all calls on a device share the array, so calls whose kernels overlap
 *     on the GPU race and must be serialised by the caller;
 *   - no cudaMalloc, cudaFree or other allocating routine is called.
 */
vsa_status vsa_coarse_select_noalloc(const void* qt, const void* kt, const int32_t* vbs, int32_t B,
                                     int32_t ncubes, int32_t heads, int32_t D, int32_t topk,
                                     float sm_scale, int32_t* topk_idx, vsa_stream_t stream);

/*
 * Fine stage: non-causal block-sparse attention ([WAN-VSA] Operator contract;
 * [VSA-AMD] Stage 2: Fine Computation, Kernel Architecture, Sparse Traversal).
 * For every (b, head, query cube i) and each of its 64 rows r (padding rows
 * included), with the attended keys
 *   X = { 64 j + s : j in topk_idx[b, head, i, :], s < vbs[j] }:
 *   s_x   = sm_scale * (q_r . k_x)
 *   out_r = sum_x softmax(s)_x v_x          (bf16, round to nearest even)
 *   lse_r = log(sum_x exp(s_x))             (fp32, natural log)
 * The softmax subtracts a running row maximum, so logits of any finite size
 * are safe.  A row with no attended key gets out = 0 and lse = -inf.
 *   qt, kt, vt : tiled bf16 [B, 64*ncubes, heads, D]; padding slots must hold
 *                finite values (vsa_tile writes zeros)
 *   topk_idx   : int32 [B, heads, ncubes, topk], entries in [0, ncubes),
 *                distinct within a row (order is free)
 *   vbs        : int32 [ncubes], each in [0, 64]
 *   out        : bf16 [B, 64*ncubes, heads, D] (written in full)
 *   lse        : fp32 [B, heads, 64*ncubes] (written), or NULL
 * Limits: D in {64, 128}; 1 <= topk <= min(ncubes, 1024); ncubes <= 8192;
 * 64*ncubes*B < 2^31.
 * Index validity is a precondition (check with vsa_validate_indices).
 */
vsa_status vsa_sparse_attn_fwd(const void* qt, const void* kt, const void* vt,
                               const int32_t* topk_idx, const int32_t* vbs, int32_t B,
                               int32_t ncubes, int32_t heads, int32_t D, int32_t topk,
                               float sm_scale, void* out, float* lse, vsa_stream_t stream);

/*
 * Schedule for the fine stage (no counterpart in the pages: a GB300 tiling
 * choice that leaves every result unchanged).  The fine kernel processes
 * query cubes in pairs, one 128-row tensor-core tile per pair, walking the
 * union of the two cubes' selections; a pair costs ceil(|sel(i) u sel(j)| / 2)
 * steps.  vsa_pair_cubes chooses, per (b, head), a pairing with large
 * selection overlaps: mutual-best matching over each cube's own selection,
 * then over a window of the unpaired cubes, the rest in index order
 * (deterministic, integer only).
 *   topk_idx  : int32 [B, heads, ncubes, topk], as for vsa_sparse_attn_fwd
 *   workspace : device buffer of vsa_pair_workspace_bytes(...) bytes,
 *               16-byte aligned, overwritten
 *   pairs     : uint32 [B, heads, (ncubes + 1) / 2] (written): unit u holds
 *               cubes i | (j << 16), i < j, j = 0xFFFF for a single cube;
 *               units in increasing i; every cube appears exactly once
 * Limits: ncubes <= 8192, topk <= 512, B * heads <= 65535.  Entries of
 * topk_idx outside [0, ncubes) are ignored.
 */
size_t vsa_pair_workspace_bytes(int32_t B, int32_t heads, int32_t ncubes, int32_t topk);
vsa_status vsa_pair_cubes(const int32_t* topk_idx, int32_t B, int32_t ncubes, int32_t heads,
                          int32_t topk, void* workspace, uint32_t* pairs, vsa_stream_t stream);

/*
 * vsa_sparse_attn_fwd with the query-cube pairing given: `pairs` as written
 * by vsa_pair_cubes (uint32 [B, heads, (ncubes + 1) / 2]), or NULL for the
 * pairs (2u, 2u + 1).  A pairing must list every cube exactly once (cube
 * indices >= ncubes mean "none"); the results are those of
 * vsa_sparse_attn_fwd up to the order of floating-point accumulation.
 * Same arguments, limits and errors otherwise.
 */
vsa_status vsa_sparse_attn_fwd_paired(const void* qt, const void* kt, const void* vt,
                                      const int32_t* topk_idx, const int32_t* vbs,
                                      const uint32_t* pairs, int32_t B, int32_t ncubes,
                                      int32_t heads, int32_t D, int32_t topk, float sm_scale,
                                      void* out, float* lse, vsa_stream_t stream);

/*
 * The fine stage with a variable number of selected cubes per query cube
 * ([VSA-AMD] Block-Sparse Encoding: a per-row count of valid blocks beside the
 * block-index table).  Row (b, head, i) attends the cubes
 * topk_idx[b, head, i, 0 .. counts[b, head, i] - 1] only; entries past the
 * count are not read (fill them with -1 so that vsa_pair_cubes, which reads
 * whole rows, ignores them).  A count of 0 gives out = 0 and lse = -inf.
 *   counts : int32 [B, heads, ncubes], values clamped to [0, topk], or NULL
 *            for topk everywhere
 *   pairs  : as for vsa_sparse_attn_fwd_paired, or NULL
 * Same arguments, limits and errors as vsa_sparse_attn_fwd otherwise.
 */
vsa_status vsa_sparse_attn_fwd_ex(const void* qt, const void* kt, const void* vt,
                                  const int32_t* topk_idx, const int32_t* counts,
                                  const int32_t* vbs, const uint32_t* pairs, int32_t B,
                                  int32_t ncubes, int32_t heads, int32_t D, int32_t topk,
                                  float sm_scale, void* out, float* lse, vsa_stream_t stream);

/*
 * vsa_sparse_attn_fwd_ex with q read and the output written in raster token
 * order, so the tiling of q and the untiling of the output (steps 1 and 4
 * for those tensors) are not separate passes: same arithmetic, so `out`
 * equals vsa_untile of vsa_sparse_attn_fwd_ex's output bit for bit, and lse
 * is the same.  No counterpart of its own on the pages: it fuses the
 * permutation of [STA] Implementation into step 3.
 *   g        : the grid (B, T, H, W, heads, D); ncubes = vsa_num_cubes(g)
 *   q        : raster bf16 [B, T*H*W, heads, D]
 *   kt, vt   : tiled bf16 [B, 64*ncubes, heads, D] (vsa_tile / vsa_tile_pool)
 *   topk_idx, counts, vbs, pairs, topk, sm_scale, lse: as vsa_sparse_attn_fwd_ex
 *   out      : raster bf16 [B, T*H*W, heads, D] (written in full)
 * Limits and errors as vsa_sparse_attn_fwd_ex, and B * T * H * W < 2^31.
 */
vsa_status vsa_sparse_attn_fwd_raster(const vsa_grid* g, const void* q, const void* kt, const void* vt,
                                      const int32_t* topk_idx, const int32_t* counts, const int32_t* vbs,
                                      const uint32_t* pairs, int32_t topk, float sm_scale, void* out, float* lse,
                                      vsa_stream_t stream);

/*
 * vsa_sparse_attn_fwd_ex that also returns each row's peakedness ([INT8-WAN]
 * Dynamic Sparsity Budgeting via Softmax Normalizer Registers: with m the
 * row's largest logit and l = sum_x exp(s_x - m), 1 / l is the row's largest
 * softmax weight):
 *   max_prob_r = exp(m_r - lse_r),  m_r = the largest attended s_x of row r,
 * formed from the exact row maximum the kernel tracks beside its lazily
 * updated softmax offset.  A row with no attended key gets 0.
 *   max_prob : fp32 [B, heads, 64*ncubes] (written; required)
 * Other arguments, limits and errors as for vsa_sparse_attn_fwd_ex (lse may
 * be NULL).
 */
vsa_status vsa_sparse_attn_fwd_peak(const void* qt, const void* kt, const void* vt,
                                    const int32_t* topk_idx, const int32_t* counts,
                                    const int32_t* vbs, const uint32_t* pairs, int32_t B,
                                    int32_t ncubes, int32_t heads, int32_t D, int32_t topk,
                                    float sm_scale, void* out, float* lse, float* max_prob,
                                    vsa_stream_t stream);

/*
 * Coarse-stage attention output ([VSA-AMD] Two-Stage Architecture, Stage 1:
 * each cube is mean-pooled into cube-level Qc, Kc, Vc and attends cube to
 * cube; the final output gates the coarse and fine outputs together):
 *   coarse_out[b, head, i, :] = sum_j w_ij Vc[b, head, j, :],
 *   w_ij = softmax_j(sm_scale * Qc[i] . Kc[j]) over the key cubes j with
 *          vbs[j] > 0,
 * with Qc, Kc, Vc the means over each cube's vbs real tokens, computed in
 * fp32.  A query cube with vbs = 0 gets zeros.
 *   qt, kt, vt : tiled bf16 [B, 64 * ncubes, heads, D]
 *   vbs        : int32 [ncubes]
 *   sm_scale   : <= 0 selects 1 / sqrt(D)
 *   workspace  : device buffer of vsa_coarse_attn_workspace_bytes(...) bytes
 *                (the fp32 cube means [3][B][heads][ncubes][D]), overwritten
 *   coarse_out : fp32 [B, heads, ncubes, D] (written)
 * Limits: D in {64, 128}; B, heads <= 65535.  Two kernel launches.
 */
size_t vsa_coarse_attn_workspace_bytes(int32_t B, int32_t heads, int32_t ncubes, int32_t D);
vsa_status vsa_coarse_attn(const void* qt, const void* kt, const void* vt, const int32_t* vbs,
                           int32_t B, int32_t ncubes, int32_t heads, int32_t D, float sm_scale,
                           void* workspace, float* coarse_out, vsa_stream_t stream);

/*
 * vsa_sparse_attn_fwd_ex whose output is the gated sum of the two stages
 * ([VSA-AMD] Two-Stage Architecture: the final output combines the coarse
 * and fine outputs through gates): for token slot s of cube i,
 *   out[b, 64 i + s, head, :] = gate_c[...] * coarse_out[b, head, i, :]
 *                             + gate_f[...] * fine[b, 64 i + s, head, :],
 * with [...] = [b, 64 i + s, head, :] and fine the normalised fine-stage
 * output, formed in fp32 inside the fine kernel's epilogue and rounded to
 * bf16 once.  lse stays the fine stage's.
 *   coarse_out     : fp32 [B, heads, ncubes, D] (e.g. from vsa_coarse_attn)
 *   gate_c, gate_f : bf16 in the layout of out, [B, 64 * ncubes, heads, D]
 * All three are required together (any one NULL with another set is
 * VSA_ERR_INVALID_ARG; all NULL is vsa_sparse_attn_fwd_ex) and must be
 * 16-byte aligned.  Other arguments, limits and errors as for
 * vsa_sparse_attn_fwd_ex.
 */
vsa_status vsa_sparse_attn_fwd_gated(const void* qt, const void* kt, const void* vt,
                                     const int32_t* topk_idx, const int32_t* counts,
                                     const int32_t* vbs, const uint32_t* pairs, int32_t B,
                                     int32_t ncubes, int32_t heads, int32_t D, int32_t topk,
                                     float sm_scale, const float* coarse_out, const void* gate_c,
                                     const void* gate_f, void* out, float* lse,
                                     vsa_stream_t stream);

/*
 * Mean-pool block selector with a cumulative threshold ([INT8-WAN]
 * "Optimizing block-sparse INT8 attention and multi-expert step caching for
 * Wan 2.2", Decoupling Block Selection from Sparse CUDA Kernels), for token
 * sequences attended in contiguous 128-token blocks (no cube grid):
 *   qbar_i, kbar_j = means of the 128 token rows of block i of q, j of k
 *                    (all 128 rows, padding included; fp32),
 *   S_ij           = qbar_i . kbar_j,
 *   row i keeps its key blocks in descending S_ij (equal scores: lower index
 *   first) until their share of softmax_j(sm_scale * S_ij) reaches tau: at
 *   least one block, all of them if the share never reaches tau.
 * Scores, weights and the share are formed in fp32, so a block whose
 * cumulative share lies within rounding of tau, or whose score ties another
 * within rounding, may be decided the other way than in exact arithmetic.
 * The result is written as the fine stage's cube-level table: block j is the
 * 64-token slot groups 2j and 2j + 1, and query groups 2i and 2i + 1 (block i)
 * both list the groups of every kept block, ascending, then -1; their count
 * is twice the kept blocks.  Pass it to vsa_sparse_attn_fwd_ex with
 * topk = S / 64, these counts, pairs = NULL (the default pairs (2u, 2u + 1)
 * are then exactly the blocks) and vbs = the real tokens of each 64-token
 * group (64, or fewer in a zero-padded tail).
 *   q, k        : bf16 [B, S, heads, D] in the sequence's token order;
 *                 S a multiple of 128
 *   tau         : in (0, 1]
 *   sm_scale    : <= 0 selects 1 / sqrt(D)
 *   workspace   : vsa_block_select_workspace_bytes(B, S, heads, D) bytes
 *                 (the fp32 block means), 16-byte aligned, overwritten
 *   cube_idx    : int32 [B, heads, S / 64, S / 64] (written in full)
 *   cube_counts : int32 [B, heads, S / 64] (written)
 * Limits: S <= 32768 (256 blocks); D in {64, 128}; B, heads <= 65535.
 * Two kernel launches (pooling, selection).
 */
size_t vsa_block_select_workspace_bytes(int32_t B, int32_t S, int32_t heads, int32_t D);
vsa_status vsa_block_select(const void* q, const void* k, int32_t B, int32_t S, int32_t heads, int32_t D,
                            float tau, float sm_scale, void* workspace, int32_t* cube_idx,
                            int32_t* cube_counts, vsa_stream_t stream);

/*
 * Debug aid for the block-sparse encoding ([VSA-AMD] Block-Sparse Encoding):
 * checks every topk_idx entry is in [0, ncubes), that no row repeats an
 * index, and that every vbs entry is in [0, 64].  ORs into *dev_flag (device
 * int32, caller-initialised): 1 = index out of range, 2 = duplicate index,
 * 4 = vbs out of range.  Read the flag after the stream synchronises;
 * VSA_ERR_INDEX_RANGE is the status a caller should report for a non-zero
 * flag.
 */
vsa_status vsa_validate_indices(const int32_t* topk_idx, const int32_t* vbs, int32_t B,
                                int32_t heads, int32_t ncubes, int32_t topk, int32_t* dev_flag,
                                vsa_stream_t stream);

/*
 * vsa_validate_indices for a table with per-row counts (the variable-length
 * encoding vsa_sparse_attn_fwd_ex takes): row r is checked on its first
 * counts[r] entries only, so padding entries (vsa_table_from_csr writes -1)
 * are not flagged.  A count outside [0, topk] sets flag bit 8 and the row is
 * checked on its entries clamped to that range.  counts: int32
 * [B, heads, ncubes] (device), or NULL for topk everywhere (the same check as
 * vsa_validate_indices).
 */
vsa_status vsa_validate_indices_ex(const int32_t* topk_idx, const int32_t* counts, const int32_t* vbs,
                                   int32_t B, int32_t heads, int32_t ncubes, int32_t topk,
                                   int32_t* dev_flag, vsa_stream_t stream);

/*
 * Reads (and with reset != 0 clears) the library's device error word on the
 * current device; synchronous.  Bits: VSA_DEVERR_*.  A kernel whose bounded
 * wait ran out sets VSA_DEVERR_TIMEOUT, stops, and leaves its outputs
 * unspecified.
 */
vsa_status vsa_device_error(uint32_t* out, int32_t reset);

/*
 * Self-test of the bounded-wait mechanism the kernels use: launches one
 * block that waits on an mbarrier nobody arrives on, with a limit of
 * `limit_ns` nanoseconds (1e3 .. 1e10).  When the wait runs out the kernel
 * sets VSA_DEVERR_TIMEOUT in the device error word and writes 1 to
 * *dev_result (device int32), else 0.  The kernel then returns normally.
 */
vsa_status vsa_debug_wait_timeout(int64_t limit_ns, int32_t* dev_result, vsa_stream_t stream);

/*
 * Number of kernels this library has launched in this process so far, over
 * every entry point, device and stream (a host-side counter, incremented when
 * a launch is enqueued; thread safe; never reset).  The difference of two
 * reads is the number of kernels launched between them.
 */
uint64_t vsa_kernel_launches(void);

/*
 * HOST-side conversion of a block table in compressed-row form ([VSA-AMD]
 * Block-Sparse Encoding: the K/V block indices of all query blocks in one
 * array, with per-row offsets and a per-row number of valid blocks) into the
 * padded table and counts that vsa_sparse_attn_fwd_ex takes.  All pointers
 * are host memory; synchronous; no CUDA call.
 *   lut_ptr : int64 [rows + 1], lut_ptr[0] = 0, non-decreasing: row r owns
 *             kv_idx[lut_ptr[r] .. lut_ptr[r + 1])
 *   kv_idx  : int32 [nnz] (may be NULL when lut_ptr[rows] is 0)
 *   nnz     : the number of entries kv_idx holds; lut_ptr[rows] <= nnz
 *   rows    : B * heads * ncubes, in the row order of topk_idx
 *   width   : the table width (topk); every row must hold <= width entries
 *   ncubes  : cubes per (batch, head); every used entry must be in
 *             [0, ncubes)
 *   table   : int32 [rows, width] (written): each row's entries, then -1
 *   counts  : int32 [rows] (written): lut_ptr[r + 1] - lut_ptr[r]
 * Returns VSA_ERR_INVALID_ARG on a null pointer, non-positive sizes,
 * lut_ptr[0] != 0, a decreasing offset, a row longer than width or offsets
 * that run past nnz, and VSA_ERR_INDEX_RANGE on an entry outside
 * [0, ncubes); in both cases nothing is written.
 */
vsa_status vsa_table_from_csr(const int64_t* lut_ptr, const int32_t* kv_idx, int64_t nnz, int64_t rows,
                              int32_t width, int32_t ncubes, int32_t* table, int32_t* counts);

#ifdef __cplusplus
}
#endif

#endif /* VSA_H_ */
