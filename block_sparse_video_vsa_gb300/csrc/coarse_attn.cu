// Coarse-stage attention output ("VSA: Accelerating Video Diffusion Inference
// with Sparse Attention on AMD GPUs", Two-Stage Architecture: Stage 1 pools
// each cube into cube-level Qc, Kc, Vc and attends cube to cube; the final
// output gates the coarse and the fine outputs together):
//     O_c[b, h, i, :] = softmax_j(sm_scale * Qc[i] . Kc[j]) Vc[j]
// over the key cubes j that hold a real token (vbs > 0); a query cube
// without a real token gets 0.  Means are over the vbs real tokens.
//
// Two kernels:
//  1. pool_means_kernel -- per (batch, cube, q|k|v): fp32 channel means into
//     the workspace [3][B][heads][ncubes][D].  HBM bound: each tiled tensor is
//     read once.
//  2. coarse_attn_kernel -- per (batch, head, 32 query cubes): the head's key
//     and value means stream through shared memory in tiles of 32 cubes; each
//     warp owns 4 query cubes, scores one key per lane, keeps an online
//     softmax in fp32 (exp2, with log2(e) folded into the scale) and D / 32
//     output channels per lane.  The work is 4 N^2 D FLOP per (batch, head),
//     small beside the fine stage, so it runs on the FMA pipes in fp32.
#include <math.h>

#include "vsa_common.cuh"

namespace vsa {

namespace {

constexpr int kAttnRows = 32;   // query cubes per block
constexpr int kAttnKeys = 32;   // key cubes per shared-memory tile (one per lane)
constexpr int kAttnWarps = 8;
constexpr int kRowsPerWarp = kAttnRows / kAttnWarps;  // 4 (the score loop holds them in a float4)
static_assert(kRowsPerWarp == 4, "the score loop reads a warp's query cubes as one float4");

__device__ __forceinline__ void add_bf16x8(const uint4 w, float (&acc)[8]) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        acc[2 * e] += __uint_as_float(ww[e] << 16);
        acc[2 * e + 1] += __uint_as_float(ww[e] & 0xFFFF0000u);
    }
}

// grid: (B * ncubes, 3 [q, k, v]); threads stride over the 8-channel vectors
// of a token row; tokens are summed in slot order.
__global__ void __launch_bounds__(256) pool_means_kernel(const uint4* __restrict__ qt, const uint4* __restrict__ kt,
                                                         const uint4* __restrict__ vt, const int32_t* __restrict__ vbs,
                                                         float* __restrict__ means, int B, int ncubes, int heads,
                                                         int D) {
    const int c = blockIdx.x % ncubes;
    const int b = blockIdx.x / ncubes;
    const int which = blockIdx.y;
    const uint4* src = which == 0 ? qt : which == 1 ? kt : vt;
    const int row_vecs = heads * D / 8;
    const int vb = min(max(vbs[c], 0), kCubeTokens);
    const float fv = (float)vb;
    const size_t s_pad = (size_t)ncubes * kCubeTokens;
    const uint4* base = src + ((size_t)b * s_pad + (size_t)c * kCubeTokens) * row_vecs;
    for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        int r = 0;
        for (; r + 8 <= vb; r += 8) {  // eight loads in flight
            uint4 w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) w[u] = __ldcs(base + (size_t)(r + u) * row_vecs + v);
#pragma unroll
            for (int u = 0; u < 8; ++u) add_bf16x8(w[u], acc);
        }
        for (; r < vb; ++r) add_bf16x8(__ldcs(base + (size_t)r * row_vecs + v), acc);
        float m[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m[e] = vb > 0 ? acc[e] / fv : 0.f;
        const int ch = v * 8;
        const int h = ch / D;
        const int d = ch - h * D;
        float* o = means + ((((size_t)which * B + b) * heads + h) * ncubes + c) * D + d;
        *reinterpret_cast<float4*>(o) = make_float4(m[0], m[1], m[2], m[3]);
        *reinterpret_cast<float4*>(o + 4) = make_float4(m[4], m[5], m[6], m[7]);
    }
}

template <int D>
__global__ void __launch_bounds__(kAttnWarps * 32) coarse_attn_kernel(const float* __restrict__ means,
                                                                     const int32_t* __restrict__ vbs,
                                                                     float* __restrict__ out, int B, int ncubes,
                                                                     int heads, float scale_log2) {
    constexpr int C = D / 32;  // output channels per lane
    extern __shared__ __align__(16) float attn_smem[];
    float* qs = attn_smem;                  // [warp][D][kRowsPerWarp]: a warp's 4 rows side by side per channel
    float* ks = qs + kAttnRows * D;         // [kAttnKeys][D + 1] (padded: one key per lane, no bank conflict)
    float* vs = ks + kAttnKeys * (D + 1);   // [kAttnKeys][D]
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const int i0 = blockIdx.x * kAttnRows;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const size_t plane = (size_t)B * heads * ncubes * D;
    const size_t head_off = ((size_t)b * heads + h) * ncubes * D;
    const float* qm = means + head_off;
    const float* km = means + plane + head_off;
    const float* vm = means + 2 * plane + head_off;
    for (int e = threadIdx.x; e < kAttnRows * D; e += blockDim.x) {
        const int rg = e / D;  // row of the block
        const int d = e - rg * D;
        const int i = i0 + rg;
        qs[((rg / kRowsPerWarp) * D + d) * kRowsPerWarp + rg % kRowsPerWarp] =
            i < ncubes ? qm[(size_t)i0 * D + e] : 0.f;
    }
    float m[kRowsPerWarp], l[kRowsPerWarp], o[kRowsPerWarp][C];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) o[rr][c] = 0.f;
    }
    for (int j0 = 0; j0 < ncubes; j0 += kAttnKeys) {
        __syncthreads();  // the previous tile has been consumed (first pass: qs is staged)
        for (int e = threadIdx.x; e < kAttnKeys * D; e += blockDim.x) {
            const int jj = e / D;
            const int d = e - jj * D;
            const bool in = j0 + jj < ncubes;
            ks[jj * (D + 1) + d] = in ? km[(size_t)j0 * D + e] : 0.f;
            vs[e] = in ? vm[(size_t)j0 * D + e] : 0.f;
        }
        __syncthreads();
        const int j = j0 + lane;
        const bool live = j < ncubes && __ldg(vbs + j) > 0;
        const float* krow = ks + lane * (D + 1);
        const float4* qw = reinterpret_cast<const float4*>(qs + warp * D * kRowsPerWarp);
        // Scores of this lane's key against the warp's 4 query cubes.
        // Two partial sums per query cube (even and odd channels) halve the dependent chains.
        float sa[kRowsPerWarp] = {0.f, 0.f, 0.f, 0.f}, sb[kRowsPerWarp] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int d = 0; d < D; d += 2) {
            const float k0 = krow[d], k1 = krow[d + 1];
            const float4 q0 = qw[d], q1 = qw[d + 1];  // broadcast
            sa[0] = fmaf(q0.x, k0, sa[0]);
            sa[1] = fmaf(q0.y, k0, sa[1]);
            sa[2] = fmaf(q0.z, k0, sa[2]);
            sa[3] = fmaf(q0.w, k0, sa[3]);
            sb[0] = fmaf(q1.x, k1, sb[0]);
            sb[1] = fmaf(q1.y, k1, sb[1]);
            sb[2] = fmaf(q1.z, k1, sb[2]);
            sb[3] = fmaf(q1.w, k1, sb[3]);
        }
        float sc[kRowsPerWarp];
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) sc[rr] = sa[rr] + sb[rr];
        float pj[kRowsPerWarp];
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            const float s = live ? sc[rr] * scale_log2 : -INFINITY;
            float tmax = s;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            const float mn = fmaxf(m[rr], tmax);
            const float alpha = m[rr] == -INFINITY ? 0.f : exp2f(m[rr] - mn);
            pj[rr] = s == -INFINITY ? 0.f : exp2f(s - mn);
            float ps = pj[rr];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            l[rr] = l[rr] * alpha + ps;
            m[rr] = mn;
#pragma unroll
            for (int c = 0; c < C; ++c) o[rr][c] *= alpha;
        }
        // O += P V over the tile's keys: each value row is read once for the 4 query cubes.
#pragma unroll 4
        for (int jj = 0; jj < kAttnKeys; ++jj) {
            const float* vrow = vs + jj * D + lane;
            float vv[C];
#pragma unroll
            for (int c = 0; c < C; ++c) vv[c] = vrow[32 * c];
#pragma unroll
            for (int rr = 0; rr < kRowsPerWarp; ++rr) {
                const float w = __shfl_sync(0xffffffffu, pj[rr], jj);
#pragma unroll
                for (int c = 0; c < C; ++c) o[rr][c] = fmaf(w, vv[c], o[rr][c]);
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int i = i0 + warp * kRowsPerWarp + rr;
        if (i >= ncubes) continue;
        const bool row_live = __ldg(vbs + i) > 0 && l[rr] > 0.f;
        const float inv = row_live ? 1.f / l[rr] : 0.f;
        float* dst = out + head_off + (size_t)i * D + lane;
#pragma unroll
        for (int c = 0; c < C; ++c) dst[32 * c] = o[rr][c] * inv;
    }
}

}  // namespace

size_t coarse_attn_workspace_bytes(int B, int heads, int ncubes, int D) {
    return (size_t)3 * B * heads * ncubes * D * sizeof(float);
}

cudaError_t launch_coarse_attn(const void* qt, const void* kt, const void* vt, const int32_t* vbs, int B,
                               int ncubes, int heads, int D, float sm_scale, void* workspace, float* out,
                               cudaStream_t stream) {
    float* means = static_cast<float*>(workspace);
    const int row_vecs = heads * D / 8;
    pool_means_kernel<<<dim3(B * ncubes, 3), row_vecs < 256 ? ((row_vecs + 31) / 32) * 32 : 256, 0, stream>>>(
        static_cast<const uint4*>(qt), static_cast<const uint4*>(kt), static_cast<const uint4*>(vt), vbs, means, B,
        ncubes, heads, D);
    note_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = (size_t)(kAttnRows * D + kAttnKeys * (D + 1) + kAttnKeys * D) * sizeof(float);
    auto kernel = D == 128 ? coarse_attn_kernel<128> : coarse_attn_kernel<64>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const float scale_log2 = sm_scale * 1.4426950408889634f;
    kernel<<<dim3((ncubes + kAttnRows - 1) / kAttnRows, heads, B), kAttnWarps * 32, smem, stream>>>(
        means, vbs, out, B, ncubes, heads, scale_log2);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace vsa
