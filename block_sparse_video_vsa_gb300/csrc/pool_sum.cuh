// Cube mean-pool statistics of the coarse stage, shared by the two kernels
// that produce them (coarse.cu's pool_kernel over tiled q and k, and tile.cu's
// tile_pool_kernel that tiles q and k and pools them in the same pass), so
// that both give the same bits.
//
// "VSA: Accelerating Video Diffusion Inference with Sparse Attention on AMD
// GPUs" (Two-Stage Architecture, Stage 1: Coarse Selection): each cube is
// mean-pooled into one vector over its vbs real tokens.
//
// Per (cube, head, channel) one thread sums the cube's real tokens in slot
// order, error-free as an fp32 (hi, lo) pair (TwoSum), and stores the fp32
// mean m = fl(fl(hi + lo) / vbs) and the fp32 residual r = (hi + lo) - m * vbs
// (TwoProduct, exact up to one rounding), plus the fp32 norm of each cube's
// mean vector per head.  The residual lets the selection rebuild the exact
// channel sum m * vbs + r in fp64.
#pragma once

#include "vsa_common.cuh"

namespace vsa {

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Adds the eight bf16 channels of one 16-byte vector to the (hi, lo) sums.
__device__ __forceinline__ void accumulate8(const uint4 w, float (&hi)[8], float (&lo)[8]) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float s, err;
        two_sum(hi[2 * e], bf16_lo(ww[e]), s, err);
        hi[2 * e] = s;
        lo[2 * e] += err;
        two_sum(hi[2 * e + 1], bf16_hi(ww[e]), s, err);
        hi[2 * e + 1] = s;
        lo[2 * e + 1] += err;
    }
}

// Workspace planes (floats): mean [2][B][heads][ncubes][D] (q then k),
// residual likewise, then norm [2][B][heads][ncubes].
struct PoolOut {
    float* mean;
    float* resid;
    float* norm;
};

__host__ __device__ inline PoolOut pool_planes(void* workspace, int B, int heads, int ncubes, int D) {
    float* ws = static_cast<float*>(workspace);
    const size_t half = (size_t)B * heads * ncubes * D;  // one [B][heads][N][D] plane
    PoolOut po;
    po.mean = ws;              // q, then k
    po.resid = ws + 2 * half;  // q, then k
    po.norm = ws + 4 * half;   // q [B][heads][N], then k
    return po;
}

// Mean, residual and norm of the 8-channel column v (channels 8v .. 8v + 7 of
// the token row) of cube c, from its (hi, lo) sums over vb tokens.  The D / 8
// lanes of one head's row must be active together (consecutive lanes, the
// first at a multiple of D / 8): the norm is a shuffle reduction over them.
__device__ __forceinline__ void pool_finish(const float (&hi)[8], const float (&lo)[8], int vb, int v, int which,
                                            int b, int c, const PoolOut& o, int B, int ncubes, int heads, int D) {
    const float fv = (float)vb;
    float m[8], rr[8];
    float s2 = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        if (vb > 0) {
            m[e] = (hi[e] + lo[e]) / fv;
            const float p = m[e] * fv;
            const float pe = fmaf(m[e], fv, -p);  // m * vb = p + pe exactly
            rr[e] = (hi[e] - p) + (lo[e] - pe);
        } else {
            m[e] = rr[e] = 0.f;
        }
        s2 = fmaf(m[e], m[e], s2);
    }
    const int gsz = D / 8;
    const int ch = v * 8;
    const int h = ch / D;
    const int d = ch - h * D;
    const size_t row = (((size_t)which * B + b) * heads + h) * ncubes + c;
    const size_t off = row * D + d;
    *reinterpret_cast<float4*>(o.mean + off) = make_float4(m[0], m[1], m[2], m[3]);
    *reinterpret_cast<float4*>(o.mean + off + 4) = make_float4(m[4], m[5], m[6], m[7]);
    *reinterpret_cast<float4*>(o.resid + off) = make_float4(rr[0], rr[1], rr[2], rr[3]);
    *reinterpret_cast<float4*>(o.resid + off + 4) = make_float4(rr[4], rr[5], rr[6], rr[7]);
    const unsigned act = __activemask();
    for (int x = 1; x < gsz; x <<= 1) s2 += __shfl_xor_sync(act, s2, x);
    if ((v & (gsz - 1)) == 0) o.norm[row] = sqrtf(s2);
}

}  // namespace vsa
