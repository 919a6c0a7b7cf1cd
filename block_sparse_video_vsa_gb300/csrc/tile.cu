// Cube tiling and untiling: the token permutation between raster (t, h, w)
// order and cube-major order with zero padding.
//
// Follows "VSA: Accelerating Video Diffusion Inference with Sparse Attention
// on AMD GPUs" (Two-Stage Architecture: Pre-stage reordering so each block is
// a contiguous spatio-temporal region; Stage 1: (4, 4, 4) cubes of 64 tokens)
// and "Wan2.2 Production Values -- VSA Block-Sparse Attention Inputs +
// Reference" (Shapes: cube-major tiled/padded, vbs = real tokens per cube;
// Operator contract: attention reads only the leading vbs[c] slots of a cube).
//
// Work decomposition: one thread block per (batch, cube).  Each token row is
// heads * D * 2 contiguous bytes; rows move as 16-byte vectors with the block's
// threads striding over the row, so every warp-level access is a fully
// coalesced 512-byte transaction.  Pure data movement: HBM bound.
#include "vsa_common.cuh"

namespace vsa {

namespace {

struct CubeGeom {
    int T, H, W, nh, nw;
};

// Source token of slot `s` of cube `c`, or -1 for a padding slot.  The real
// tokens of the cube's clipped sub-box fill slots 0 .. vbs-1 in raster order.
__device__ __forceinline__ int slot_token(const CubeGeom& g, int c, int s, int* vbs_out) {
    const int cw = c % g.nw;
    const int ch = (c / g.nw) % g.nh;
    const int ct = c / (g.nw * g.nh);
    const int et = min(kCube, g.T - kCube * ct);
    const int eh = min(kCube, g.H - kCube * ch);
    const int ew = min(kCube, g.W - kCube * cw);
    const int vb = et * eh * ew;
    if (vbs_out) *vbs_out = vb;
    if (s >= vb) return -1;
    const int lt = s / (eh * ew);
    const int r = s - lt * (eh * ew);
    const int lh = r / ew;
    const int lw = r - lh * ew;
    return ((kCube * ct + lt) * g.H + (kCube * ch + lh)) * g.W + (kCube * cw + lw);
}

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) tile_kernel(const int4* __restrict__ x,
                                                        int4* __restrict__ xt,
                                                        int32_t* __restrict__ vbs, CubeGeom g,
                                                        int ncubes, int row_vecs,
                                                        long long tokens) {
    __shared__ int src_tok[kCubeTokens];
    const int c = blockIdx.x % ncubes;
    const int b = blockIdx.x / ncubes;
    if (threadIdx.x < kCubeTokens) {
        int vb;
        src_tok[threadIdx.x] = slot_token(g, c, threadIdx.x, &vb);
        if (threadIdx.x == 0 && b == 0 && vbs) vbs[c] = vb;
    }
    __syncthreads();
    const size_t s_pad = (size_t)ncubes * kCubeTokens;
    const int total = kCubeTokens * row_vecs;
    const int4* xb = x + (size_t)b * (size_t)tokens * row_vecs;
    int4* xtb = xt + ((size_t)b * s_pad + (size_t)c * kCubeTokens) * row_vecs;
    // Four vectors per thread in flight: all loads are issued before the stores.
    for (int e0 = threadIdx.x; e0 < total; e0 += 4 * kThreads) {
        int4 val[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads;
            val[u] = make_int4(0, 0, 0, 0);
            if (e < total) {
                const int s = e / row_vecs;
                const int n = src_tok[s];
                if (n >= 0) val[u] = __ldcs(xb + (size_t)n * row_vecs + (e - s * row_vecs));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads;
            if (e < total) __stcs(xtb + e, val[u]);
        }
    }
}

__global__ void __launch_bounds__(kThreads) untile_kernel(const int4* __restrict__ yt,
                                                          int4* __restrict__ y, CubeGeom g,
                                                          int ncubes, int row_vecs,
                                                          long long tokens) {
    __shared__ int dst_tok[kCubeTokens];
    __shared__ int vb_s;
    const int c = blockIdx.x % ncubes;
    const int b = blockIdx.x / ncubes;
    if (threadIdx.x < kCubeTokens) {
        int vb;
        dst_tok[threadIdx.x] = slot_token(g, c, threadIdx.x, &vb);
        if (threadIdx.x == 0) vb_s = vb;
    }
    __syncthreads();
    const size_t s_pad = (size_t)ncubes * kCubeTokens;
    const int total = vb_s * row_vecs;
    const int4* ytb = yt + ((size_t)b * s_pad + (size_t)c * kCubeTokens) * row_vecs;
    int4* yb = y + (size_t)b * (size_t)tokens * row_vecs;
    for (int e0 = threadIdx.x; e0 < total; e0 += 4 * kThreads) {
        int4 val[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads;
            if (e < total) val[u] = __ldcs(ytb + e);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads;
            if (e < total) {
                const int s = e / row_vecs;
                __stcs(yb + (size_t)dst_tok[s] * row_vecs + (e - s * row_vecs), val[u]);
            }
        }
    }
}

CubeGeom make_geom(const vsa_grid& g) {
    CubeGeom cg;
    cg.T = g.T;
    cg.H = g.H;
    cg.W = g.W;
    cg.nh = (g.H + kCube - 1) / kCube;
    cg.nw = (g.W + kCube - 1) / kCube;
    return cg;
}

}  // namespace

cudaError_t launch_tile(const vsa_grid& g, int ncubes, const void* x, void* xt, int32_t* vbs,
                        cudaStream_t stream) {
    const int row_vecs = g.heads * g.D / 8;
    const long long tokens = (long long)g.T * g.H * g.W;
    tile_kernel<<<g.B * ncubes, kThreads, 0, stream>>>(static_cast<const int4*>(x),
                                                      static_cast<int4*>(xt), vbs, make_geom(g),
                                                      ncubes, row_vecs, tokens);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_untile(const vsa_grid& g, int ncubes, const void* yt, void* y,
                          cudaStream_t stream) {
    const int row_vecs = g.heads * g.D / 8;
    const long long tokens = (long long)g.T * g.H * g.W;
    untile_kernel<<<g.B * ncubes, kThreads, 0, stream>>>(static_cast<const int4*>(yt),
                                                        static_cast<int4*>(y), make_geom(g),
                                                        ncubes, row_vecs, tokens);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace vsa
