// Coarse stage: cube mean-pool of Q and K, cube-to-cube scores, top-k cubes.
//
// Follows "VSA: Accelerating Video Diffusion Inference with Sparse Attention
// on AMD GPUs" (Two-Stage Architecture, Stage 1: Coarse Selection -- each
// cube mean-pooled into one vector, cube-to-cube scores, Top-K key/value
// cubes per query cube; Generating Sparsity Patterns -- pool, score einsum,
// top-k over the last axis) with the score scaled by sm_scale.
//
// Pipeline:
//  1. pool_kernel -- per (batch, cube, q|k): channel sums over the vbs real
//     tokens, accumulated error-free as fp32 (hi, lo) pairs (TwoSum), stored
//     as the fp32 mean m = fl(fl(hi + lo) / vbs) and the fp32 residual
//     r = (hi + lo) - m * vbs (TwoProduct, exact up to one rounding), plus the
//     fp32 norm of every cube's mean vector per head (pool_sum.cuh).  HBM
//     bound: reads each tiled tensor once.  Skipped when tile_pool_kernel
//     (tile.cu) already wrote the same statistics while tiling q and k.
//  2. score_topk_kernel -- per (batch, head, block of R query cubes): fp32
//     scores against every key cube (FFMA; key means streamed into shared
//     memory by asynchronous copies, double buffered), then per row a bitwise radix
//     select of the k-th largest score.  Scores within a proven fp32 error
//     bound of that boundary are re-ranked in fp64 with the exact cube sums
//     m * vbs + r, so the set matches exact-arithmetic top-k.  From 256 cubes
//     the scores go through memory instead (score_gemm_kernel, then
//     select_kernel, one warp per row, with the same selection).
#include <float.h>

#include <type_traits>

#include "pool_sum.cuh"

namespace vsa {

namespace {

// ------------------------------------------------------------------ pooling
// grid: (B * ncubes, 2 [q, k]); threads stride over the 8-channel vectors of
// a token row (heads * D / 8 of them); D / 8 consecutive threads hold one
// head's row, so the norm is a reduction over that lane group.
__global__ void __launch_bounds__(256) pool_kernel(const uint4* __restrict__ qt, const uint4* __restrict__ kt,
                                                   const int32_t* __restrict__ vbs, PoolOut o, int B,
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
        int r = 0;
        for (; r + 8 <= vb; r += 8) {  // eight loads in flight, summed in token order
            uint4 w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) w[u] = __ldcs(base + (size_t)(r + u) * row_vecs + v);
#pragma unroll
            for (int u = 0; u < 8; ++u) accumulate8(w[u], hi, lo);
        }
        for (; r < vb; ++r) accumulate8(__ldcs(base + (size_t)r * row_vecs + v), hi, lo);
        pool_finish(hi, lo, vb, v, which, b, c, o, B, ncubes, heads, D);
    }
}

// ------------------------------------------------------------ score + top-k
constexpr int kTileJ = 64;       // key cubes per shared-memory tile (two per lane)
constexpr int kCandCap = 128;    // stored candidates per warp for re-ranking
constexpr size_t kSmemCap = 232448;  // 227 KB opt-in shared memory per block

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

// Key of the k-th largest score of a row (warp-wide): the largest T with
// count(key >= T) >= k, found bit by bit from the top.  The row's keys are
// held in registers (KPL per lane, N <= 32 * KPL); slots past N hold 0,
// which no candidate threshold (>= 1) counts.
template <int KPL>
__device__ __forceinline__ uint32_t kth_key(const float* row, int N, int k, int lane) {
    uint32_t key[KPL];
#pragma unroll
    for (int q = 0; q < KPL; ++q) {
        const int j = lane + 32 * q;
        key[q] = j < N ? f2key(row[j]) : 0u;
    }
    uint32_t T = 0;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = T | (1u << bit);
        int cnt[4] = {0, 0, 0, 0};  // four independent chains (latency)
#pragma unroll
        for (int q = 0; q < KPL; ++q) cnt[q & 3] += key[q] >= cand;
        const int c = __reduce_add_sync(0xffffffffu, (cnt[0] + cnt[1]) + (cnt[2] + cnt[3]));
        if (c >= k) T = cand;
    }
    return T;
}
// Same search reading the row from shared memory on every pass (long rows).
__device__ __noinline__ uint32_t kth_key_smem(const float* row, int N, int k, int lane) {
    uint32_t T = 0;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = T | (1u << bit);
        int cnt = 0;
        for (int j = lane; j < N; j += 32) cnt += f2key(row[j]) >= cand;
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        if (cnt >= k) T = cand;
    }
    return T;
}

// Byte offsets of the score kernel's shared-memory regions.
struct ScoreLayout {
    size_t qs, kb, sc, qnorm, red, qsum, cand_s, cand_j, total;
};
__host__ __device__ inline size_t take(size_t& o, size_t bytes, size_t align) {
    o = (o + align - 1) / align * align;
    const size_t r = o;
    o += bytes;
    return r;
}
__host__ __device__ inline ScoreLayout score_layout(int R, int N, int D, int warps) {
    const size_t LD = (size_t)D + 4;  // padded row (floats): conflict-free float4 reads
    ScoreLayout L;
    size_t o = 0;
    L.qs = take(o, (size_t)R * LD * 4, 16);
    L.kb = take(o, 2 * (size_t)kTileJ * LD * 4, 16);
    L.sc = take(o, (size_t)R * N * 4, 16);
    L.qnorm = take(o, (size_t)R * 4, 4);
    L.red = take(o, (size_t)warps * 4, 4);
    L.qsum = take(o, (size_t)warps * D * 8, 8);
    L.cand_s = take(o, (size_t)warps * kCandCap * 8, 8);
    L.cand_j = take(o, (size_t)warps * kCandCap * 4, 4);
    L.total = o;
    return L;
}

struct ScoreArgs {
    const float* qm;  // [B][heads][N][D] means
    const float* qr;  //                  residuals
    const float* km;
    const float* kr;
    const float* qn;  // [B][heads][N] norms of the means
    const float* kn;
    const int32_t* vbs;
    int32_t* topk_idx;
    int B, N, heads, topk, R;
    float sm_scale;
};

__device__ __forceinline__ int clamp_vbs(int v) { return min(max(v, 0), kCubeTokens); }

// Exact (to ~1e-16) score of cube pair (i, j): sm_scale * (S_i . S_j) /
// (vbs_i * vbs_j) in fp64, with the channel sums S = m * vbs + r.
template <int D>
__device__ double precise_score(const double* __restrict__ qsum, const ScoreArgs& a, size_t hrow, int j,
                                double inv_vq) {
    const int vk = clamp_vbs(a.vbs[j]);
    if (vk <= 0) return 0.0;
    const float* km = a.km + hrow + (size_t)j * D;
    const float* kr = a.kr + hrow + (size_t)j * D;
    double acc = 0.0;
#pragma unroll 4
    for (int d = 0; d < D; ++d) acc = fma(qsum[d], fma((double)km[d], (double)vk, (double)kr[d]), acc);
    return (double)a.sm_scale * acc * inv_vq / (double)vk;
}

// Top-k of one score row (one warp): the k-th largest fp32 score by bitwise
// search, then the scores within the fp32 error band of that boundary are
// re-ranked in fp64 from the exact cube sums; the selected cube ids are
// written in ascending order.  `row` (shared or global memory) is scratch:
// band members are overwritten with +inf (chosen) or -inf.  kMaxCase bounds
// the register-held search (N <= 128 * kMaxCase); longer rows are searched in
// place.
template <int D, int kMaxCase>
__device__ void select_row(float* row, const ScoreArgs& a, size_t bh, size_t hrow, int i, float qnorm_i,
                           float kmax_all, double* qsum, double* cs, int* cj, int lane) {
    const int N = a.N;
    const int k = a.topk;
    uint32_t T;
    switch ((N + 127) / 128) {  // register slots per lane: N / 32 rounded up to a multiple of 4
        case 1: T = kth_key<4>(row, N, k, lane); break;
        case 2: T = kth_key<8>(row, N, k, lane); break;
        case 3: T = kth_key<12>(row, N, k, lane); break;
        case 4: T = kth_key<16>(row, N, k, lane); break;
        case 5: T = kth_key<20>(row, N, k, lane); break;
        case 6: T = kth_key<24>(row, N, k, lane); break;
        case 7: T = kth_key<28>(row, N, k, lane); break;
        case 8: T = kth_key<32>(row, N, k, lane); break;
        default:
            if constexpr (kMaxCase >= 16) {
                const int c = (N + 127) / 128;
                if (c <= 10) T = kth_key<40>(row, N, k, lane);
                else if (c <= 12) T = kth_key<48>(row, N, k, lane);
                else if (c <= 14) T = kth_key<56>(row, N, k, lane);
                else if (c <= 16) T = kth_key<64>(row, N, k, lane);
                else T = kth_key_smem(row, N, k, lane);
            } else {
                T = kth_key_smem(row, N, k, lane);
            }
            break;
    }
    const float tau = key2f(T);
    // Error bound of an fp32 score against the exact one (dot of rounded
    // means with fp32 accumulation, then the scale): (D + 8) u |q||k|,
    // doubled for margin; the band is twice that around tau.
    const float eps = 2.f * (float)(D + 8) * 5.9604645e-8f * a.sm_scale * qnorm_i * kmax_all;
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
        const size_t qrow = hrow + (size_t)i * D;
        const int vq = clamp_vbs(a.vbs[i]);
        for (int d = lane; d < D; d += 32)
            qsum[d] = fma((double)a.qm[qrow + d], (double)vq, (double)a.qr[qrow + d]);
        __syncwarp();
        const double inv_vq = vq > 0 ? 1.0 / (double)vq : 0.0;
        if (cC <= kCandCap) {
            int pos = 0;
            for (int j0b = 0; j0b < N; j0b += 32) {
                const int j = j0b + lane;
                const bool inC = j < N && row[j] >= lo && row[j] <= hi;
                const unsigned m = __ballot_sync(0xffffffffu, inC);
                if (inC) cj[pos + __popc(m & ((1u << lane) - 1u))] = j;
                pos += __popc(m);
            }
            __syncwarp();
            for (int c = lane; c < cC; c += 32) cs[c] = precise_score<D>(qsum, a, hrow, cj[c], inv_vq);
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
            for (int j0b = 0; j0b < N; j0b += 32) {
                const int j = j0b + lane;
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
    int32_t* out = a.topk_idx + (bh * N + i) * (size_t)k;
    int pos = 0;
    const unsigned below = (1u << lane) - 1u;
    for (int j0b = 0; j0b < N; j0b += 128) {  // four 32-wide slices per pass: loads batched
        bool sel[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = j0b + 32 * q + lane;
            const float x = j < N ? row[j] : -INFINITY;
            sel[q] = j < N && (x > hi || (take_band && x >= lo));
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const unsigned m = __ballot_sync(0xffffffffu, sel[q]);
            if (sel[q]) out[pos + __popc(m & below)] = j0b + 32 * q + lane;
            pos += __popc(m);
        }
    }
}

// WARPS warps; each thread scores RT query rows (R = WARPS * RT rows per block).
template <int D, int RT, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) score_topk_kernel(ScoreArgs a) {
    constexpr int kWarps = WARPS;
    constexpr int kScoreThreads = WARPS * 32;
    constexpr int LD = D + 4;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int R = a.R;
    const int N = a.N;
    const ScoreLayout L = score_layout(R, N, D, WARPS);
    float* qs = reinterpret_cast<float*>(smem_raw + L.qs);        // [R][LD]
    float* kb = reinterpret_cast<float*>(smem_raw + L.kb);        // [2][kTileJ][LD]
    float* sc = reinterpret_cast<float*>(smem_raw + L.sc);        // [R][N]
    float* qnorm = reinterpret_cast<float*>(smem_raw + L.qnorm);  // [R]
    float* red = reinterpret_cast<float*>(smem_raw + L.red);      // [kWarps]
    double* qsum_w = reinterpret_cast<double*>(smem_raw + L.qsum);  // [kWarps][D]
    double* cand_s = reinterpret_cast<double*>(smem_raw + L.cand_s);
    int* cand_j = reinterpret_cast<int*>(smem_raw + L.cand_j);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int i0 = blockIdx.x * R;
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const size_t bh = (size_t)b * a.heads + h;
    const size_t hrow = bh * (size_t)N * D;  // element offset of this (b, head) in a [B][heads][N][D] plane
    const int ntiles = (N + kTileJ - 1) / kTileJ;

    // Copy key-mean tile t (rows j0 .. j0 + 63, 16-byte pieces into the
    // padded layout) into buffer t & 1 with asynchronous copies.
    auto issue_tile = [&](int t) {
        const int j0 = t * kTileJ;
        const int rows = min(kTileJ, N - j0);
        float* dst = kb + (size_t)(t & 1) * kTileJ * LD;
        const float* src = a.km + hrow + (size_t)j0 * D;
        for (int e = tid; e < rows * (D / 4); e += kScoreThreads) {
            const int r = e / (D / 4), c = e - r * (D / 4);
            cp_async16(smem_u32(dst + r * LD + 4 * c), src + (size_t)r * D + 4 * c);
        }
        cp_async_commit();
    };
    issue_tile(0);

    // Stage the query means of this block's rows and their norms.
    for (int e = tid; e < R * (D / 4); e += kScoreThreads) {
        const int r = e / (D / 4), d4 = e - r * (D / 4);
        const int i = i0 + r;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < N) v = *reinterpret_cast<const float4*>(a.qm + hrow + (size_t)i * D + d4 * 4);
        *reinterpret_cast<float4*>(qs + r * LD + d4 * 4) = v;
    }
    for (int r = tid; r < R; r += kScoreThreads) qnorm[r] = (i0 + r < N) ? a.qn[bh * N + i0 + r] : 0.f;
    float kmax = 0.f;  // largest key-mean norm of this head
    for (int j = tid; j < N; j += kScoreThreads) kmax = fmaxf(kmax, a.kn[bh * N + j]);
#pragma unroll
    for (int o = 16; o; o >>= 1) kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    if (lane == 0) red[warp] = kmax;
    __syncthreads();
    float kmax_all = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) kmax_all = fmaxf(kmax_all, red[w]);

    // fp32 scores: thread (warp, lane) -> rows warp + 8u (u < R / 8) x key
    // columns lane and lane + 32 of each tile.
    constexpr int rt = RT;  // = R / kWarps
    for (int t = 0; t < ntiles; ++t) {
        if (t + 1 < ntiles) {
            issue_tile(t + 1);  // buffer (t+1)&1 was released at the end of t-1
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // tile t visible to every thread
        const float* k0 = kb + (size_t)(t & 1) * kTileJ * LD + lane * LD;
        const float* k1 = k0 + 32 * LD;
        float acc[rt][2];
#pragma unroll
        for (int u = 0; u < rt; ++u) acc[u][0] = acc[u][1] = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; d += 4) {
            const float4 x0 = *reinterpret_cast<const float4*>(k0 + d);
            const float4 x1 = *reinterpret_cast<const float4*>(k1 + d);
#pragma unroll
            for (int u = 0; u < rt; ++u) {
                {
                    const float4 q = *reinterpret_cast<const float4*>(qs + (warp + kWarps * u) * LD + d);
                    acc[u][0] = fmaf(q.x, x0.x, acc[u][0]);
                    acc[u][0] = fmaf(q.y, x0.y, acc[u][0]);
                    acc[u][0] = fmaf(q.z, x0.z, acc[u][0]);
                    acc[u][0] = fmaf(q.w, x0.w, acc[u][0]);
                    acc[u][1] = fmaf(q.x, x1.x, acc[u][1]);
                    acc[u][1] = fmaf(q.y, x1.y, acc[u][1]);
                    acc[u][1] = fmaf(q.z, x1.z, acc[u][1]);
                    acc[u][1] = fmaf(q.w, x1.w, acc[u][1]);
                }
            }
        }
        const int j0 = t * kTileJ + lane;
#pragma unroll
        for (int u = 0; u < rt; ++u) {
            {
                float* row = sc + (size_t)(warp + kWarps * u) * N;
                if (j0 < N) row[j0] = a.sm_scale * acc[u][0];
                if (j0 + 32 < N) row[j0 + 32] = a.sm_scale * acc[u][1];
            }
        }
        __syncthreads();  // releases buffer t & 1 for tile t + 2
    }

    // Selection: one warp per row.
    for (int r = warp; r < R; r += kWarps) {
        const int i = i0 + r;
        if (i >= N) break;
        select_row<D, 8>(sc + (size_t)r * N, a, bh, hrow, i, qnorm[r], kmax_all, qsum_w + warp * D,
                         cand_s + warp * kCandCap, cand_j + warp * kCandCap, lane);
    }
}

// ------------------------------------------- large N: scores through memory
// When few query rows fit the fused kernel's shared memory (N above ~1100 at
// D = 128), the scores go to the workspace instead: a register-tiled fp32
// GEMM (128 x 128 score tiles, the full depth D in shared memory, each thread
// 8 x 8 scores on rows ty + 16 r and columns tx + 16 c; products accumulated
// in increasing d as in the fused kernel, so the scores are the same), then
// one warp per row runs the same selection on the row read back.
constexpr int kGemmTile = 128;

template <int D>
__global__ void __launch_bounds__(256) score_gemm_kernel(ScoreArgs a, float* __restrict__ scores) {
    constexpr int LD = D + 4;  // padded row (floats)
    extern __shared__ __align__(16) float gsm[];
    float* As = gsm;                   // [kGemmTile][LD] query means
    float* Bs = gsm + kGemmTile * LD;  // [kGemmTile][LD] key means
    const int N = a.N;
    const int i0 = blockIdx.x * kGemmTile, j0 = blockIdx.y * kGemmTile;
    const size_t bh = blockIdx.z;
    const size_t hrow = bh * (size_t)N * D;
    const int tid = threadIdx.x;
    for (int e = tid; e < kGemmTile * (D / 4); e += 256) {
        const int r = e / (D / 4), d4 = e - r * (D / 4);
        float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vb = va;
        if (i0 + r < N) va = *reinterpret_cast<const float4*>(a.qm + hrow + (size_t)(i0 + r) * D + 4 * d4);
        if (j0 + r < N) vb = *reinterpret_cast<const float4*>(a.km + hrow + (size_t)(j0 + r) * D + 4 * d4);
        *reinterpret_cast<float4*>(As + r * LD + 4 * d4) = va;
        *reinterpret_cast<float4*>(Bs + r * LD + 4 * d4) = vb;
    }
    __syncthreads();
    const int ty = tid >> 4, tx = tid & 15;
    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
#pragma unroll 2
    for (int d = 0; d < D; d += 4) {
        float4 av[8], bv[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) av[r] = *reinterpret_cast<const float4*>(As + (ty + 16 * r) * LD + d);
#pragma unroll
        for (int c = 0; c < 8; ++c) bv[c] = *reinterpret_cast<const float4*>(Bs + (tx + 16 * c) * LD + d);
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                acc[r][c] = fmaf(av[r].x, bv[c].x, acc[r][c]);
                acc[r][c] = fmaf(av[r].y, bv[c].y, acc[r][c]);
                acc[r][c] = fmaf(av[r].z, bv[c].z, acc[r][c]);
                acc[r][c] = fmaf(av[r].w, bv[c].w, acc[r][c]);
            }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int i = i0 + ty + 16 * r;
        if (i >= N) continue;
        float* dst = scores + (bh * N + i) * (size_t)N;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int j = j0 + tx + 16 * c;
            if (j < N) dst[j] = a.sm_scale * acc[r][c];
        }
    }
}

template <int D>
__global__ void __launch_bounds__(256) select_kernel(ScoreArgs a, float* __restrict__ scores) {
    __shared__ double qsum_w[8][D];
    __shared__ double cand_s[8][kCandCap];
    __shared__ int cand_j[8][kCandCap];
    __shared__ float red[8];
    const int N = a.N;
    const size_t bh = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float kmax = 0.f;  // largest key-mean norm of this head
    for (int j = tid; j < N; j += 256) kmax = fmaxf(kmax, a.kn[bh * N + j]);
#pragma unroll
    for (int o = 16; o; o >>= 1) kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    if (lane == 0) red[warp] = kmax;
    __syncthreads();
    float kmax_all = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) kmax_all = fmaxf(kmax_all, red[w]);
    const int i = blockIdx.x * 8 + warp;
    if (i >= N) return;
    select_row<D, 16>(scores + (bh * N + i) * (size_t)N, a, bh, bh * (size_t)N * D, i, a.qn[bh * N + i],
                      kmax_all, qsum_w[warp], cand_s[warp], cand_j[warp], lane);
}

// --------------------------------------------------------------- validator
constexpr int kValWarps = 4;
constexpr int kValMaxCubes = 65536;

__global__ void __launch_bounds__(kValWarps * 32) validate_kernel(const int32_t* __restrict__ idx,
                                                                  const int32_t* __restrict__ counts,
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
        int n = topk;  // entries in use: the row's count, when counts are given
        if (counts) {
            n = counts[row];
            if (n < 0 || n > topk) {
                f |= 8;
                n = n < 0 ? 0 : topk;
            }
        }
        for (int t = lane; t < n; t += 32) {
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

size_t coarse_workspace_bytes(int B, int heads, int ncubes, int D, bool split) {
    size_t bytes = (size_t)16 * B * heads * ncubes * D + (size_t)8 * B * heads * ncubes;
    if (split) bytes += (size_t)4 * B * heads * ncubes * ncubes;  // fp32 scores
    return bytes;
}

// Score-block shapes: R rows per block on 16 warps (R = 32: two rows per
// thread; R = 16: one) or on 8 warps (R = 8).
static int score_warps(int R) { return R >= 16 ? 16 : 8; }

// Rows per score block: the largest of 32, 16, 8 whose shared memory fits.
int coarse_rows_per_block(int ncubes, int D) {
    for (int R = 32; R > 8; R >>= 1)
        if (score_layout(R, ncubes, D, score_warps(R)).total <= kSmemCap) return R;
    return 8;
}

// Scores through memory (score GEMM + per-row selection) from 256 cubes, and
// whenever the fused kernel would hold fewer than 32 query rows per block.
bool coarse_split_default(int ncubes, int D) { return ncubes >= 256 || coarse_rows_per_block(ncubes, D) < 32; }

size_t coarse_smem_bytes(int N, int D, bool split) {
    if (split) return (size_t)2 * kGemmTile * (D + 4) * sizeof(float);
    const int R = coarse_rows_per_block(N, D);
    return score_layout(R, N, D, score_warps(R)).total;
}

cudaError_t launch_coarse(const void* qt, const void* kt, const int32_t* vbs, int B, int ncubes,
                          int heads, int D, int topk, float sm_scale, void* workspace,
                          int32_t* topk_idx, bool split, bool pooled, cudaStream_t stream) {
    const size_t half = (size_t)B * heads * ncubes * D;  // one [B][heads][N][D] plane
    const PoolOut po = pool_planes(workspace, B, heads, ncubes, D);
    cudaError_t e;
    if (!pooled) {
        const int row_vecs = heads * D / 8;
        dim3 pg(B * ncubes, 2);
        pool_kernel<<<pg, row_vecs < 256 ? ((row_vecs + 31) / 32) * 32 : 256, 0, stream>>>(
            static_cast<const uint4*>(qt), static_cast<const uint4*>(kt), vbs, po, B, ncubes, heads, D);
        note_launches(1);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    ScoreArgs a;
    a.qm = po.mean;
    a.km = po.mean + half;
    a.qr = po.resid;
    a.kr = po.resid + half;
    a.qn = po.norm;
    a.kn = po.norm + (size_t)B * heads * ncubes;
    a.vbs = vbs;
    a.topk_idx = topk_idx;
    a.B = B;
    a.N = ncubes;
    a.heads = heads;
    a.topk = topk;
    a.R = coarse_rows_per_block(ncubes, D);
    a.sm_scale = sm_scale;
    if (split) {
        float* scores = po.norm + 2 * (size_t)B * heads * ncubes;
        const size_t gsmem = (size_t)2 * kGemmTile * (D + 4) * sizeof(float);
        const int tiles = (ncubes + kGemmTile - 1) / kGemmTile;
        const dim3 gg(tiles, tiles, B * heads);
        auto gemm = D == 128 ? score_gemm_kernel<128> : score_gemm_kernel<64>;
        e = cudaFuncSetAttribute(gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gsmem);
        if (e != cudaSuccess) return e;
        gemm<<<gg, 256, gsmem, stream>>>(a, scores);
        auto sel = D == 128 ? select_kernel<128> : select_kernel<64>;
        sel<<<dim3((ncubes + 7) / 8, B * heads), 256, 0, stream>>>(a, scores);
        note_launches(2);
        return cudaGetLastError();
    }
    const size_t smem = coarse_smem_bytes(ncubes, D, false);
    dim3 grid((ncubes + a.R - 1) / a.R, heads, B);
    auto pick = [&](auto d) {
        constexpr int DD = decltype(d)::value;
        return a.R == 32 ? score_topk_kernel<DD, 2, 16>
                         : a.R == 16 ? score_topk_kernel<DD, 1, 16> : score_topk_kernel<DD, 1, 8>;
    };
    auto kernel = D == 128 ? pick(std::integral_constant<int, 128>()) : pick(std::integral_constant<int, 64>());
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, score_warps(a.R) * 32, smem, stream>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_validate(const int32_t* idx, const int32_t* counts, const int32_t* vbs, int rows, int ncubes,
                            int topk, int32_t* flag, cudaStream_t stream) {
    const int words = (ncubes + 31) / 32;
    const size_t smem = (size_t)kValWarps * words * 4;
    int blocks = (rows + kValWarps - 1) / kValWarps;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    cudaError_t e = cudaFuncSetAttribute(validate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    validate_kernel<<<blocks, kValWarps * 32, smem, stream>>>(idx, counts, vbs, rows, ncubes, topk, flag);
    note_launches(1);
    return cudaGetLastError();
}

int validate_max_cubes() { return kValMaxCubes; }

cudaError_t launch_debug_wait(long long limit_ns, int32_t* result, unsigned int* err,
                              cudaStream_t stream) {
    debug_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, result, err);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace vsa
