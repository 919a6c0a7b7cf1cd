// Coarse stage: cube mean-pool of Q and K, cube-to-cube scores, top-k cubes.
//
// Follows "VSA: Accelerating Video Diffusion Inference with Sparse Attention
// on AMD GPUs" (Two-Stage Architecture, Stage 1: Coarse Selection -- each
// cube mean-pooled into one vector, cube-to-cube scores, Top-K key/value
// cubes per query cube; Generating Sparsity Patterns -- pool, score einsum,
// top-k over the last axis) with the score scaled by sm_scale.
//
// Pipeline (two kernels):
//  1. pool_sums_kernel -- exact per-cube channel sums of q and k as fp32
//     (hi, lo) pairs (error-free TwoSum accumulation over the vbs real
//     tokens).  HBM bound: reads each tiled tensor once.
//  2. score_topk_kernel -- per (batch, head, block of R query cubes): fp32
//     scores against every key cube (FFMA, shared-memory tiled), then per row
//     a bitwise radix select of the k-th largest score.  Scores within a
//     proven fp32 error bound of that boundary are re-ranked with exact cube
//     sums in fp64, so the set matches exact-arithmetic top-k.
#include <float.h>

#include "vsa_common.cuh"

namespace vsa {

namespace {

// ------------------------------------------------------------------ pooling
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// grid: (B * ncubes, 2 [q, k]); threads stride over 8-channel vectors of a
// token row (heads * D / 8 of them).  ws layout: [2][B][heads][ncubes][D] for
// hi, then the same for lo.
__global__ void __launch_bounds__(256) pool_sums_kernel(const uint4* __restrict__ qt,
                                                        const uint4* __restrict__ kt,
                                                        const int32_t* __restrict__ vbs,
                                                        float* __restrict__ ws_hi,
                                                        float* __restrict__ ws_lo, int B,
                                                        int ncubes, int heads, int D) {
    const int c = blockIdx.x % ncubes;
    const int b = blockIdx.x / ncubes;
    const int which = blockIdx.y;
    const uint4* src = which == 0 ? qt : kt;
    const int row_vecs = heads * D / 8;
    const int vb = min(max(vbs[c], 0), kCubeTokens);
    const size_t s_pad = (size_t)ncubes * kCubeTokens;
    const uint4* base = src + ((size_t)b * s_pad + (size_t)c * kCubeTokens) * row_vecs;
    for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) {
        float hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) hi[e] = lo[e] = 0.f;
        for (int r = 0; r < vb; ++r) {
            const uint4 w = __ldcs(base + (size_t)r * row_vecs + v);
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
        const int ch = v * 8;
        const int h = ch / D;
        const int d = ch - h * D;
        const size_t o = ((((size_t)which * B + b) * heads + h) * ncubes + c) * D + d;
#pragma unroll
        for (int e = 0; e < 8; e += 4) {
            *reinterpret_cast<float4*>(ws_hi + o + e) = make_float4(hi[e], hi[e + 1], hi[e + 2], hi[e + 3]);
            *reinterpret_cast<float4*>(ws_lo + o + e) = make_float4(lo[e], lo[e + 1], lo[e + 2], lo[e + 3]);
        }
    }
}

// ------------------------------------------------------------ score + top-k
constexpr int kScoreThreads = 256;
constexpr int kWarps = kScoreThreads / 32;
constexpr int kTileJ = 32;       // key cubes per shared-memory tile
constexpr int kCandCap = 128;    // stored candidates per warp for re-ranking

// Monotone map from float to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f2key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ unsigned long long d2key(double f) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(f);
    return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

struct ScoreArgs {
    const float* qh;  // [B][heads][N][D] exact sums, hi part
    const float* ql;
    const float* kh;
    const float* kl;
    const int32_t* vbs;
    int32_t* topk_idx;
    int B, N, heads, topk, R;
    float sm_scale;
};

// Exact (to ~1e-16) score of cube pair (i, j) from the hi/lo cube sums:
// sm_scale * (Q_i . K_j) / (vbs_i * vbs_j), evaluated in fp64.
template <int D>
__device__ double precise_score(const double* __restrict__ qsum, const ScoreArgs& a, size_t krow,
                                int j, double inv_vq) {
    const float* kh = a.kh + krow + (size_t)j * D;
    const float* kl = a.kl + krow + (size_t)j * D;
    double acc = 0.0;
#pragma unroll 4
    for (int d = 0; d < D; ++d) {
        const double kd = (double)kh[d] + (double)kl[d];
        acc = fma(qsum[d], kd, acc);
    }
    const int vk = a.vbs[j];
    if (vk <= 0) return 0.0;
    return (double)a.sm_scale * acc * inv_vq / (double)vk;
}

template <int D>
__global__ void __launch_bounds__(kScoreThreads) score_topk_kernel(ScoreArgs a) {
    constexpr int LD = D + 4;  // padded row (floats): conflict-free float4 reads
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int R = a.R;
    const int N = a.N;
    float* qs = reinterpret_cast<float*>(smem_raw);                    // [R][LD]
    float* ks = qs + R * LD;                                          // [kTileJ][LD]
    float* sc = ks + kTileJ * LD;                                     // [R][N]
    float* qnorm = sc + (size_t)R * N;                                // [R]
    float* kmax_s = qnorm + R;                                        // [kWarps]
    double* qsum_w = reinterpret_cast<double*>(kmax_s + kWarps + (kWarps & 1 ? 1 : 0));  // [kWarps][D]
    double* cand_s = qsum_w + kWarps * D;                             // [kWarps][kCandCap]
    int* cand_j = reinterpret_cast<int*>(cand_s + kWarps * kCandCap); // [kWarps][kCandCap]

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int i0 = blockIdx.x * R;
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const size_t hrow = ((size_t)b * a.heads + h) * (size_t)N * D;

    // Stage the fp32 query means of this block's rows.
    for (int e = tid; e < R * D; e += kScoreThreads) {
        const int r = e / D, d = e - r * D;
        const int i = i0 + r;
        float v = 0.f;
        if (i < N) {
            const int vq = a.vbs[i];
            const size_t o = hrow + (size_t)i * D + d;
            v = vq > 0 ? (a.qh[o] + a.ql[o]) / (float)vq : 0.f;
        }
        qs[r * LD + d] = v;
    }
    __syncthreads();
    for (int r = warp; r < R; r += kWarps) {
        float s2 = 0.f;
        for (int d = lane; d < D; d += 32) s2 = fmaf(qs[r * LD + d], qs[r * LD + d], s2);
#pragma unroll
        for (int o = 16; o; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        if (lane == 0) qnorm[r] = sqrtf(s2);
    }

    // fp32 scores: thread (row group, column) -> R/8 rows x 1 column per tile.
    const int col = tid & 31;
    const int rg = tid >> 5;  // rows rg, rg + 8, ...
    const int rows_per = R / kWarps;
    float kmax = 0.f;
    for (int j0 = 0; j0 < N; j0 += kTileJ) {
        __syncthreads();
        for (int e = tid; e < kTileJ * D; e += kScoreThreads) {
            const int r = e / D, d = e - r * D;
            const int j = j0 + r;
            float v = 0.f;
            if (j < N) {
                const int vk = a.vbs[j];
                const size_t o = hrow + (size_t)j * D + d;
                v = vk > 0 ? (a.kh[o] + a.kl[o]) / (float)vk : 0.f;
            }
            ks[r * LD + d] = v;
        }
        __syncthreads();
        {   // running max of key-mean norms (warp w handles tile rows w*4 .. w*4+3)
            for (int r = warp * 4; r < warp * 4 + 4; ++r) {
                float s2 = 0.f;
                for (int d = lane; d < D; d += 32) s2 = fmaf(ks[r * LD + d], ks[r * LD + d], s2);
#pragma unroll
                for (int o = 16; o; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
                kmax = fmaxf(kmax, sqrtf(s2));
            }
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const float* kp = ks + col * LD;
#pragma unroll 4
        for (int d = 0; d < D; d += 4) {
            const float4 kv = *reinterpret_cast<const float4*>(kp + d);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (t < rows_per) {
                    const float4 qv = *reinterpret_cast<const float4*>(qs + (rg + kWarps * t) * LD + d);
                    acc[t] = fmaf(qv.x, kv.x, acc[t]);
                    acc[t] = fmaf(qv.y, kv.y, acc[t]);
                    acc[t] = fmaf(qv.z, kv.z, acc[t]);
                    acc[t] = fmaf(qv.w, kv.w, acc[t]);
                }
            }
        }
        const int j = j0 + col;
        if (j < N) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (t < rows_per) sc[(size_t)(rg + kWarps * t) * N + j] = a.sm_scale * acc[t];
        }
    }
    if (lane == 0) kmax_s[warp] = kmax;
    __syncthreads();
    float kmax_all = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) kmax_all = fmaxf(kmax_all, kmax_s[w]);

    // Selection: one warp per row.
    const int k = a.topk;
    for (int r = warp; r < R; r += kWarps) {
        const int i = i0 + r;
        if (i >= N) break;
        float* row = sc + (size_t)r * N;
        // k-th largest key by bitwise search: largest T with count(key >= T) >= k.
        uint32_t T = 0;
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = T | (1u << bit);
            int cnt = 0;
            for (int j = lane; j < N; j += 32) cnt += f2key(row[j]) >= cand;
            cnt = __reduce_add_sync(0xffffffffu, cnt);
            if (cnt >= k) T = cand;
        }
        const float tau = key2f(T);
        // Error bound of an fp32 score against the exact one (dot of rounded
        // means with fp32 accumulation, then the scale): (D + 8) u |q||k|,
        // doubled for margin; the band is twice that around tau.
        const float eps = 2.f * (float)(D + 8) * 5.9604645e-8f * a.sm_scale * qnorm[r] * kmax_all;
        const float band = 2.f * eps + 1e-30f;
        const float lo = tau - band, hi = tau + band;
        int cA = 0, cC = 0;
        for (int j = lane; j < N; j += 32) {
            const float s = row[j];
            cA += s > hi;
            cC += (s >= lo) && (s <= hi);
        }
        cA = __reduce_add_sync(0xffffffffu, cA);
        cC = __reduce_add_sync(0xffffffffu, cC);
        const int need = k - cA;  // 1 <= need <= cC
        const bool take_band = (cC == need);  // the whole band is selected: no re-ranking
        if (!take_band) {
            // Re-rank the boundary band with exact cube sums in fp64.
            double* qsum = qsum_w + warp * D;
            const size_t qrow = hrow + (size_t)i * D;
            for (int d = lane; d < D; d += 32) qsum[d] = (double)a.qh[qrow + d] + (double)a.ql[qrow + d];
            __syncwarp();
            const int vq = a.vbs[i];
            const double inv_vq = vq > 0 ? 1.0 / (double)vq : 0.0;
            if (cC <= kCandCap) {
                double* cs = cand_s + warp * kCandCap;
                int* cj = cand_j + warp * kCandCap;
                int pos = 0;
                for (int j0 = 0; j0 < N; j0 += 32) {
                    const int j = j0 + lane;
                    const bool inC = j < N && row[j] >= lo && row[j] <= hi;
                    const unsigned m = __ballot_sync(0xffffffffu, inC);
                    if (inC) cj[pos + __popc(m & ((1u << lane) - 1u))] = j;
                    pos += __popc(m);
                }
                __syncwarp();
                for (int c = lane; c < cC; c += 32)
                    cs[c] = precise_score<D>(qsum, a, hrow, cj[c], inv_vq);
                __syncwarp();
                // rank among candidates: (score desc, index asc); chosen if rank < need.
                for (int c = lane; c < cC; c += 32) {
                    const double s = cs[c];
                    const int jc = cj[c];
                    int rank = 0;
                    for (int o = 0; o < cC; ++o) {
                        const double so = cs[o];
                        rank += (so > s) || (so == s && cj[o] < jc);
                    }
                    row[jc] = rank < need ? INFINITY : -INFINITY;
                }
                __syncwarp();
            } else {
                // Degenerate band (many near-equal scores): 64-bit bitwise search
                // over the exact scores of the band, recomputed per pass.
                unsigned long long T2 = 0;
                for (int bit = 63; bit >= 0; --bit) {
                    const unsigned long long cand = T2 | (1ull << bit);
                    int cnt = 0;
                    for (int j = lane; j < N; j += 32)
                        if (row[j] >= lo && row[j] <= hi)
                            cnt += d2key(precise_score<D>(qsum, a, hrow, j, inv_vq)) >= cand;
                    cnt = __reduce_add_sync(0xffffffffu, cnt);
                    if (cnt >= need) T2 = cand;
                }
                int greater = 0;
                for (int j = lane; j < N; j += 32)
                    if (row[j] >= lo && row[j] <= hi)
                        greater += d2key(precise_score<D>(qsum, a, hrow, j, inv_vq)) > T2;
                greater = __reduce_add_sync(0xffffffffu, greater);
                int eq_left = need - greater;  // equal-to-T2 members to take, lowest index first
                for (int j0 = 0; j0 < N; j0 += 32) {
                    const int j = j0 + lane;
                    bool inC = j < N && row[j] >= lo && row[j] <= hi;
                    unsigned long long kk = 0;
                    if (inC) kk = d2key(precise_score<D>(qsum, a, hrow, j, inv_vq));
                    const bool eq = inC && kk == T2;
                    const unsigned m = __ballot_sync(0xffffffffu, eq);
                    const int before = __popc(m & ((1u << lane) - 1u));
                    if (inC) row[j] = (kk > T2 || (eq && before < eq_left)) ? INFINITY : -INFINITY;
                    eq_left -= __popc(m);
                }
                __syncwarp();
            }
        }
        // Emit the selected set in ascending cube index.  After re-ranking the
        // band members hold +inf (chosen) or -inf (not chosen).
        int32_t* out = a.topk_idx + (((size_t)b * a.heads + h) * N + i) * (size_t)k;
        int pos = 0;
        for (int j0 = 0; j0 < N; j0 += 32) {
            const int j = j0 + lane;
            const bool sel = j < N && (row[j] > hi || (take_band && row[j] >= lo));
            const unsigned m = __ballot_sync(0xffffffffu, sel);
            if (sel) out[pos + __popc(m & ((1u << lane) - 1u))] = j;
            pos += __popc(m);
        }
    }
}

// --------------------------------------------------------------- validator
constexpr int kValWarps = 4;
constexpr int kValMaxCubes = 65536;

__global__ void __launch_bounds__(kValWarps * 32) validate_kernel(const int32_t* __restrict__ idx,
                                                                  const int32_t* __restrict__ vbs,
                                                                  int rows, int ncubes, int topk,
                                                                  int32_t* flag) {
    extern __shared__ unsigned int bits[];  // [kValWarps][ceil(ncubes/32)]
    const int words = (ncubes + 31) / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned int* my = bits + warp * words;
    int f = 0;
    if (blockIdx.x == 0)
        for (int c = threadIdx.x; c < ncubes; c += blockDim.x)
            if (vbs[c] < 0 || vbs[c] > kCubeTokens) f |= 4;
    for (int row = blockIdx.x * kValWarps + warp; row < rows; row += gridDim.x * kValWarps) {
        for (int w = lane; w < words; w += 32) my[w] = 0u;
        __syncwarp();
        const int32_t* p = idx + (size_t)row * topk;
        for (int t = lane; t < topk; t += 32) {
            const int j = p[t];
            if (j < 0 || j >= ncubes) {
                f |= 1;
            } else {
                const unsigned int old = atomicOr(&my[j >> 5], 1u << (j & 31));
                if (old & (1u << (j & 31))) f |= 2;
            }
        }
        __syncwarp();
    }
    f = __reduce_or_sync(0xffffffffu, f);
    if (lane == 0 && f) atomicOr(flag, f);
}

__global__ void debug_wait_kernel(long long limit_ns, int32_t* result, unsigned int* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
    }
    __syncthreads();
    // Nobody arrives on `bar`: the bounded wait must run out.
    const bool ok = mbar_wait_bounded(b, 0, &abort_flag, err, (uint64_t)limit_ns);
    if (threadIdx.x == 0) *result = ok ? 0 : 1;
}

}  // namespace

size_t coarse_workspace_bytes(int B, int heads, int ncubes, int D) {
    return (size_t)16 * B * heads * ncubes * D;
}

int coarse_rows_per_block(int ncubes) {
    if (ncubes <= 1024) return 32;
    if (ncubes <= 2048) return 16;
    return 8;
}

size_t coarse_smem_bytes(int R, int N, int D) {
    const size_t LD = D + 4;
    size_t f = (size_t)R * LD + (size_t)kTileJ * LD + (size_t)R * N + R + kWarps + 1;
    size_t bytes = f * 4;
    bytes = (bytes + 7) & ~(size_t)7;
    bytes += (size_t)kWarps * D * 8 + (size_t)kWarps * kCandCap * 8 + (size_t)kWarps * kCandCap * 4;
    return bytes;
}

cudaError_t launch_coarse(const void* qt, const void* kt, const int32_t* vbs, int B, int ncubes,
                          int heads, int D, int topk, float sm_scale, void* workspace,
                          int32_t* topk_idx, cudaStream_t stream) {
    float* ws = static_cast<float*>(workspace);
    const size_t plane = (size_t)2 * B * heads * ncubes * D;  // q then k
    float* hi = ws;
    float* lo = ws + plane;
    const int row_vecs = heads * D / 8;
    dim3 pg(B * ncubes, 2);
    pool_sums_kernel<<<pg, row_vecs < 256 ? ((row_vecs + 31) / 32) * 32 : 256, 0, stream>>>(
        static_cast<const uint4*>(qt), static_cast<const uint4*>(kt), vbs, hi, lo, B, ncubes,
        heads, D);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    ScoreArgs a;
    const size_t half = (size_t)B * heads * ncubes * D;
    a.qh = hi;
    a.kh = hi + half;
    a.ql = lo;
    a.kl = lo + half;
    a.vbs = vbs;
    a.topk_idx = topk_idx;
    a.B = B;
    a.N = ncubes;
    a.heads = heads;
    a.topk = topk;
    a.R = coarse_rows_per_block(ncubes);
    a.sm_scale = sm_scale;
    const size_t smem = coarse_smem_bytes(a.R, ncubes, D);
    dim3 grid((ncubes + a.R - 1) / a.R, heads, B);
    if (D == 128) {
        e = cudaFuncSetAttribute(score_topk_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        score_topk_kernel<128><<<grid, kScoreThreads, smem, stream>>>(a);
    } else {
        e = cudaFuncSetAttribute(score_topk_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        score_topk_kernel<64><<<grid, kScoreThreads, smem, stream>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_validate(const int32_t* idx, const int32_t* vbs, int rows, int ncubes, int topk,
                            int32_t* flag, cudaStream_t stream) {
    const int words = (ncubes + 31) / 32;
    const size_t smem = (size_t)kValWarps * words * 4;
    int blocks = (rows + kValWarps - 1) / kValWarps;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    cudaError_t e = cudaFuncSetAttribute(validate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    validate_kernel<<<blocks, kValWarps * 32, smem, stream>>>(idx, vbs, rows, ncubes, topk, flag);
    return cudaGetLastError();
}

int validate_max_cubes() { return kValMaxCubes; }

cudaError_t launch_debug_wait(long long limit_ns, int32_t* result, unsigned int* err,
                              cudaStream_t stream) {
    debug_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, result, err);
    return cudaGetLastError();
}

}  // namespace vsa
