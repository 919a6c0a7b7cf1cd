// Mean-pool block selector with a cumulative threshold ("Optimizing
// block-sparse INT8 attention and multi-expert step caching for Wan 2.2",
// Decoupling Block Selection from Sparse CUDA Kernels), for token sequences
// attended in contiguous 128-token blocks: each 128-token block of q and k is
// mean-pooled, block pairs are scored by dot products S_ij = qbar_i . kbar_j,
// and each query block keeps its key blocks in descending score (equal
// scores: lower index first) until their share of softmax_j(sm_scale * S_ij)
// reaches tau (at least one block; all of them if the share never does).
//
// The kept blocks are written as the fine stage's cube-level table: a
// 128-token block j is the two 64-token slot groups ("cubes") 2j and 2j + 1,
// so query cubes 2i and 2i + 1 (block i) both list the cubes of every kept
// block, ascending, then -1, with the count beside.  The fine stage's default
// pairing (2u, 2u + 1) then puts exactly one block in each tile.
//
// GB300 design: pooling is a streaming read of q and k (one pass, 16-byte
// loads, fp32 sums in token order); selection is one warp per query block,
// the head's key-block means staged once per CTA in shared memory: scores in
// fp32 against every key block, the softmax weights, and the
// threshold found by a 32-step bitwise search over order-preserving integer
// keys of the scores (the largest key t whose blocks with key >= t hold at
// least tau of the mass), so no sort is needed; blocks tied at that key are
// taken in index order while the kept mass is still short of tau.
#include <math.h>

#include "vsa_common.cuh"

namespace vsa {

namespace {

constexpr int kBlockTokens = 128;
constexpr int kSelWarps = 32;  // query blocks per CTA (one warp each): the staged key means serve 32 rows
constexpr int kMaxBlocks = 256;  // key blocks per row: cube table rows of up to 512 entries
constexpr int kPerLane = kMaxBlocks / 32;

// Order-preserving map of a float to an unsigned key (larger float, larger key).
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// grid (B * nb, 2 [q, k]): fp32 channel means of 128 consecutive token rows,
// summed in token order; written as [2][B][heads][nb][D].
__global__ void __launch_bounds__(256) block_pool_kernel(const uint4* __restrict__ q, const uint4* __restrict__ k,
                                                         float* __restrict__ means, int B, int nb, int heads, int D) {
    const int blk = blockIdx.x % nb;
    const int b = blockIdx.x / nb;
    const uint4* src = blockIdx.y == 0 ? q : k;
    const int row_vecs = heads * D / 8;
    const uint4* base = src + ((size_t)b * nb + blk) * kBlockTokens * row_vecs;
    for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int r = 0; r < kBlockTokens; r += 16) {  // sixteen loads in flight, summed in token order
            uint4 w[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) w[u] = __ldcs(base + (size_t)(r + u) * row_vecs + v);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const uint32_t ww[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[2 * e] += __uint_as_float(ww[e] << 16);
                    acc[2 * e + 1] += __uint_as_float(ww[e] & 0xFFFF0000u);
                }
            }
        }
        const int ch = v * 8;
        const int h = ch / D;
        const int d = ch - h * D;
        float* o = means + ((((size_t)blockIdx.y * B + b) * heads + h) * nb + blk) * D + d;
        const float inv = 1.f / kBlockTokens;
        *reinterpret_cast<float4*>(o) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<float4*>(o + 4) = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// grid (ceil(nb / kSelWarps), heads, B): one warp per query block for the
// selection.  The CTA stages the head's key-block means (rows padded to D + 4
// floats: a float4 read by 32 lanes of 32 rows is 4 conflict-free phases) and
// its 32 query-block means in shared memory, forms the 32 x nb score tile with
// each thread holding 4 query rows x 2 key blocks (float4 reads, every score
// summed channel by channel in order), and parks it in shared memory, from
// where each warp takes its row.
constexpr int kScoreLd = kMaxBlocks + 4;

template <int D>
__host__ __device__ constexpr size_t select_smem_bytes() {
    return ((size_t)kMaxBlocks * (D + 4) + (size_t)kSelWarps * D + (size_t)kSelWarps * kScoreLd) * sizeof(float);
}

template <int D>
__global__ void __launch_bounds__(kSelWarps * 32) block_select_kernel(const float* __restrict__ means, int B, int nb,
                                                                      int heads, float scale_log2, float tau,
                                                                      int32_t* __restrict__ cube_idx,
                                                                      int32_t* __restrict__ cube_counts) {
    static_assert(kSelWarps == 32 && kMaxBlocks == 256, "the score tile covers 32 rows x 256 key blocks");
    constexpr int LD = D + 4;
    constexpr int kV = D / 4;  // float4 vectors per row
    extern __shared__ __align__(16) float sel_smem[];
    float* ks = sel_smem;                             // [kMaxBlocks][LD] key-block means
    float* qs = ks + (size_t)kMaxBlocks * LD;         // [kSelWarps][D] query-block means
    float* ss = qs + (size_t)kSelWarps * D;           // [kSelWarps][kScoreLd] scores
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int i0 = blockIdx.x * kSelWarps;
    const int i = i0 + warp;
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const size_t plane = (size_t)B * heads * nb * D;
    const size_t hoff = ((size_t)b * heads + h) * nb * D;
    // Key means: eight 16-byte loads per thread in flight (at most 8 each).
#pragma unroll
    for (int e0 = 0; e0 < kMaxBlocks * kV; e0 += 8 * kSelWarps * 32) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + u * kSelWarps * 32 + threadIdx.x;
            if (e < nb * kV) v[u] = *reinterpret_cast<const float4*>(means + plane + hoff + (size_t)e * 4);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + u * kSelWarps * 32 + threadIdx.x;
            if (e < nb * kV) {
                const int j = e / kV, c = e - j * kV;
                *reinterpret_cast<float4*>(ks + j * LD + 4 * c) = v[u];
            }
        }
    }
    // Query means of the CTA's rows (zeros past nb).
    for (int e = threadIdx.x; e < kSelWarps * kV; e += kSelWarps * 32) {
        const int r = e / kV, c = e - r * kV;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i0 + r < nb) v = *reinterpret_cast<const float4*>(means + hoff + (size_t)(i0 + r) * D + 4 * c);
        *reinterpret_cast<float4*>(qs + r * D + 4 * c) = v;
    }
    __syncthreads();
    {
        // Tile: rows 4 (warp & 7) .. + 3; key blocks lane + 32 (2 (warp >> 3) + {0, 1}).
        const int r0 = 4 * (warp & 7);
        const int j0 = lane + 64 * (warp >> 3), j1 = j0 + 32;
        const float* k0 = ks + (j0 < nb ? j0 : 0) * LD;
        const float* k1 = ks + (j1 < nb ? j1 : 0) * LD;
        float acc[4][2];
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r][0] = acc[r][1] = 0.f;
#pragma unroll 4
        for (int c = 0; c < kV; ++c) {
            const float4 a0 = *reinterpret_cast<const float4*>(k0 + 4 * c);
            const float4 a1 = *reinterpret_cast<const float4*>(k1 + 4 * c);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float4 q = *reinterpret_cast<const float4*>(qs + (r0 + r) * D + 4 * c);
                acc[r][0] = fmaf(q.x, a0.x, acc[r][0]);
                acc[r][0] = fmaf(q.y, a0.y, acc[r][0]);
                acc[r][0] = fmaf(q.z, a0.z, acc[r][0]);
                acc[r][0] = fmaf(q.w, a0.w, acc[r][0]);
                acc[r][1] = fmaf(q.x, a1.x, acc[r][1]);
                acc[r][1] = fmaf(q.y, a1.y, acc[r][1]);
                acc[r][1] = fmaf(q.z, a1.z, acc[r][1]);
                acc[r][1] = fmaf(q.w, a1.w, acc[r][1]);
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            ss[(r0 + r) * kScoreLd + j0] = acc[r][0];
            ss[(r0 + r) * kScoreLd + j1] = acc[r][1];
        }
    }
    __syncthreads();
    if (i >= nb) return;  // no block-wide barrier below
    // Row i's scores: lane t holds key blocks j = t + 32 s (s < kPerLane).
    float sc[kPerLane];
#pragma unroll
    for (int s2 = 0; s2 < kPerLane; ++s2) {
        const int j = lane + 32 * s2;
        sc[s2] = j < nb ? ss[warp * kScoreLd + j] : -INFINITY;
    }
    // Softmax weights of the row (exp2 with log2(e) folded into the scale).
    float smax = -INFINITY;
#pragma unroll
    for (int s = 0; s < kPerLane; ++s) smax = fmaxf(smax, sc[s]);
    smax = warp_max(smax);
    float w[kPerLane];
    uint32_t key[kPerLane];
    float wsum = 0.f;
#pragma unroll
    for (int s = 0; s < kPerLane; ++s) {
        const bool in = lane + 32 * s < nb;
        w[s] = in ? exp2f((sc[s] - smax) * scale_log2) : 0.f;
        key[s] = in ? order_key(sc[s]) : 0u;
        wsum += w[s];
    }
    wsum = warp_sum(wsum);
    const float target = tau * wsum;  // unnormalised masses are compared
    // The largest key t with mass(key >= t) >= target, bit by bit.
    uint32_t ans = 0u;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = ans | (1u << bit);
        float mass = 0.f;
#pragma unroll
        for (int s = 0; s < kPerLane; ++s) mass += key[s] >= cand ? w[s] : 0.f;
        if (warp_sum(mass) >= target) ans = cand;
    }
    // Kept: every block above ans, then the blocks tied at ans in index
    // order while the mass kept before each is still short of the target.
    float mass_gt = 0.f;
#pragma unroll
    for (int s = 0; s < kPerLane; ++s) mass_gt += key[s] > ans ? w[s] : 0.f;
    float run = warp_sum(mass_gt);
    int pos = 0;                                   // blocks written so far
    const int nc = 2 * nb;                         // cubes per row of the sequence
    const size_t row0 = ((size_t)b * heads + h) * nc + 2 * (size_t)i;
    int32_t* out0 = cube_idx + row0 * (size_t)nc;  // query cube 2i; 2i + 1 follows
    int32_t* out1 = out0 + nc;
#pragma unroll
    for (int s = 0; s < kPerLane; ++s) {
        const int j = lane + 32 * s;
        const bool tie = j < nb && key[s] == ans;
        // Tie blocks in index order: inclusive prefix of their weights across the warp.
        float pre = tie ? w[s] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_up_sync(0xffffffffu, pre, o);
            if (lane >= o) pre += v;
        }
        const float excl = pre - (tie ? w[s] : 0.f);
        const bool keep = j < nb && (key[s] > ans || (tie && run + excl < target));
        run += __shfl_sync(0xffffffffu, pre, 31);
        const uint32_t bal = __ballot_sync(0xffffffffu, keep);
        if (keep) {
            const int at = pos + __popc(bal & ((1u << lane) - 1u));
            out0[2 * at] = 2 * j;
            out0[2 * at + 1] = 2 * j + 1;
            out1[2 * at] = 2 * j;
            out1[2 * at + 1] = 2 * j + 1;
        }
        pos += __popc(bal);
    }
    for (int e = 2 * pos + lane; e < nc; e += 32) {
        out0[e] = -1;
        out1[e] = -1;
    }
    if (lane == 0) {
        cube_counts[row0] = 2 * pos;
        cube_counts[row0 + 1] = 2 * pos;
    }
}

}  // namespace

size_t block_select_workspace_bytes(int B, int heads, int nb, int D) {
    return (size_t)2 * B * heads * nb * D * sizeof(float);
}

int block_select_max_blocks() { return kMaxBlocks; }

cudaError_t launch_block_select(const void* q, const void* k, int B, int S, int heads, int D, float tau,
                                float sm_scale, void* workspace, int32_t* cube_idx, int32_t* cube_counts,
                                cudaStream_t stream) {
    const int nb = S / kBlockTokens;
    float* means = static_cast<float*>(workspace);
    const int row_vecs = heads * D / 8;
    const int pool_threads = row_vecs < 256 ? ((row_vecs + 31) / 32) * 32 : 256;
    block_pool_kernel<<<dim3(B * nb, 2), pool_threads, 0, stream>>>(
        static_cast<const uint4*>(q), static_cast<const uint4*>(k), means, B, nb, heads, D);
    note_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto kernel = D == 128 ? block_select_kernel<128> : block_select_kernel<64>;
    const size_t smem = D == 128 ? select_smem_bytes<128>() : select_smem_bytes<64>();
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<dim3((nb + kSelWarps - 1) / kSelWarps, heads, B), kSelWarps * 32, smem, stream>>>(
        means, B, nb, heads, sm_scale * 1.4426950408889634f, tau, cube_idx, cube_counts);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace vsa
