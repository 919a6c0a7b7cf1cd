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
#include "pool_sum.cuh"

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
constexpr int kPoolThreadsMax = 320;

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

// Tiling of q and k fused with the coarse stage's cube mean-pool: one pass
// over the raster q and k writes the tiled tensors and the pooled statistics
// (pool_sum.cuh), so the selection does not read the tiled q and k again.
// A null qt or kt skips that tiled copy (the statistics are still written).
// grid (B * ncubes, 2 [q, k]); every 8-channel column of the cube's token
// rows belongs to one thread, which copies its 64 slots eight at a time and
// sums the first vbs of them in slot order, the order pool_kernel sums the
// tiled rows in (the statistics are the same bits).  The block size is a
// multiple of 32 and of D / 8, so one head's columns sit in consecutive lanes
// for the norm's shuffle reduction.
__global__ void __launch_bounds__(kPoolThreadsMax) tile_pool_kernel(const uint4* __restrict__ q,
                                                                   const uint4* __restrict__ k,
                                                                   uint4* __restrict__ qt, uint4* __restrict__ kt,
                                                                   int32_t* __restrict__ vbs, CubeGeom g,
                                                                   int ncubes, int heads, int D, long long tokens,
                                                                   PoolOut o, int B) {
    __shared__ int src_tok[kCubeTokens];
    __shared__ int vb_s;
    const int c = blockIdx.x % ncubes;
    const int b = blockIdx.x / ncubes;
    const int which = blockIdx.y;
    if (threadIdx.x < kCubeTokens) {
        int vb;
        src_tok[threadIdx.x] = slot_token(g, c, threadIdx.x, &vb);
        if (threadIdx.x == 0) {
            vb_s = vb;
            if (b == 0 && which == 0 && vbs) vbs[c] = vb;
        }
    }
    __syncthreads();
    const int row_vecs = heads * D / 8;
    const int vb = vb_s;
    const size_t s_pad = (size_t)ncubes * kCubeTokens;
    const uint4* xb = (which == 0 ? q : k) + (size_t)b * (size_t)tokens * row_vecs;
    uint4* const dst = which == 0 ? qt : kt;  // null: statistics only, no tiled copy
    uint4* xtb = dst ? dst + ((size_t)b * s_pad + (size_t)c * kCubeTokens) * row_vecs : nullptr;
    for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) {
        float hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) hi[e] = lo[e] = 0.f;
#pragma unroll 1
        for (int s0 = 0; s0 < kCubeTokens; s0 += 8) {  // eight slots in flight
            uint4 w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int n = src_tok[s0 + u];
                w[u] = n >= 0 ? __ldcs(xb + (size_t)n * row_vecs + v) : make_uint4(0u, 0u, 0u, 0u);
            }
            if (xtb) {
#pragma unroll
                for (int u = 0; u < 8; ++u) __stcs(xtb + (size_t)(s0 + u) * row_vecs + v, w[u]);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (s0 + u < vb) accumulate8(w[u], hi, lo);
        }
        pool_finish(hi, lo, vb, v, which, b, c, o, B, ncubes, heads, D);
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

// Block size of tile_pool_kernel: the largest multiple of 32 (and of D / 8)
// up to kPoolThreadsMax that divides the row's column count, so no thread
// idles in the last pass (640 columns at 40 heads x 128 -> 320: two columns
// per thread); 256 when none divides it.  At least 64 threads: the first 64
// fill the cube's slot table.
static int tile_pool_threads(int row_vecs, int D) {
    const int step = D / 8 > 32 ? D / 8 : 32;
    if (row_vecs <= kPoolThreadsMax) {
        const int t = ((row_vecs + step - 1) / step) * step;
        return t < kCubeTokens ? kCubeTokens : t;
    }
    for (int t = kPoolThreadsMax / step * step; t >= 64; t -= step)
        if (row_vecs % t == 0) return t;
    return 256;
}

cudaError_t launch_tile_pool(const vsa_grid& g, int ncubes, const void* q, const void* k, void* qt, void* kt,
                             int32_t* vbs, void* workspace, cudaStream_t stream) {
    const int row_vecs = g.heads * g.D / 8;
    const long long tokens = (long long)g.T * g.H * g.W;
    const PoolOut po = pool_planes(workspace, g.B, g.heads, ncubes, g.D);
    tile_pool_kernel<<<dim3(g.B * ncubes, 2), tile_pool_threads(row_vecs, g.D), 0, stream>>>(
        static_cast<const uint4*>(q), static_cast<const uint4*>(k), static_cast<uint4*>(qt),
        static_cast<uint4*>(kt), vbs, make_geom(g), ncubes, g.heads, g.D, tokens, po, g.B);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace vsa
