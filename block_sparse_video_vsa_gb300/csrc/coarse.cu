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
// held in registers (KPL per lane: lane l, slot q holds column l + 32 q);
// slots past N hold 0, which no candidate threshold (>= 1) counts.  The bits
// every real key shares (the common prefix of the row's largest and smallest
// keys) are taken as they are: with all keys >= that prefix, the count there
// is N >= k, so the search starts below it.  The search stops early once the
// keys still possible, [T, T + 2^rem), span at most `stop_width` as floats;
// `rem` returns the number of undecided low bits (0: T is exact).
template <int KPL>
__device__ __forceinline__ uint32_t kth_key_regs(const uint32_t (&key)[KPL], int N, int k, int lane,
                                                 float stop_width, int& rem) {
    uint32_t kmx = 0u, kmn = 0xFFFFFFFFu;
#pragma unroll
    for (int q = 0; q < KPL; ++q) {
        kmx = max(kmx, key[q]);
        if (lane + 32 * q < N) kmn = min(kmn, key[q]);
    }
    kmx = __reduce_max_sync(0xffffffffu, kmx);
    kmn = __reduce_min_sync(0xffffffffu, kmn);
    const int free_bits = 32 - __clz(kmx ^ kmn);  // bits below the common prefix
    uint32_t T = free_bits == 32 ? 0u : (kmx >> free_bits) << free_bits;
    rem = 0;
#pragma unroll 1
    for (int bit = free_bits - 1; bit >= 0; --bit) {
        // Bits bit .. 0 are open: the k-th key lies in [T, T | (2^(bit+1) - 1)].
        if (key2f(T | ((2u << bit) - 1u)) - key2f(T) <= stop_width) {
            rem = bit + 1;
            break;
        }
        const uint32_t cand = T | (1u << bit);
        int cnt[4] = {0, 0, 0, 0};  // four independent chains (latency)
#pragma unroll
        for (int q = 0; q < KPL; ++q) cnt[q & 3] += key[q] >= cand;
        const int c = __reduce_add_sync(0xffffffffu, (cnt[0] + cnt[1]) + (cnt[2] + cnt[3]));
        if (c >= k) T = cand;
    }
    return T;
}
// Same search reading the row from memory on every pass (rows longer than
// the register-held cases).
__device__ __noinline__ uint32_t kth_key_mem(const float* row, int N, int k, int lane) {
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

// Loads a score row's keys into registers (slot q of this lane: column
// lane + 32 q; 0 past N).
template <int KPL>
__device__ __forceinline__ void load_row_keys(const float* row, int N, int lane, uint32_t (&key)[KPL]) {
#pragma unroll
    for (int q = 0; q < KPL; ++q) {
        const int j = lane + 32 * q;
        key[q] = j < N ? f2key(row[j]) : 0u;
    }
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

// precise_score with the D products spread over the warp (lane l takes
// channels l, l + 32, ...; the partial sums are added in a butterfly): the
// fp64 chain per lane is D / 32 long instead of D.  The value of lane 0 is
// returned in every lane's copy only for lane 0; callers store lane 0's.
template <int D>
__device__ double precise_score_warp(const double* __restrict__ qsum, const ScoreArgs& a, size_t hrow, int j,
                                     double inv_vq, int lane) {
    const int vk = clamp_vbs(a.vbs[j]);
    const float* km = a.km + hrow + (size_t)j * D;
    const float* kr = a.kr + hrow + (size_t)j * D;
    double acc = 0.0;
#pragma unroll
    for (int d = lane; d < D; d += 32) acc = fma(qsum[d], fma((double)km[d], (double)vk, (double)kr[d]), acc);
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return vk > 0 ? (double)a.sm_scale * acc * inv_vq / (double)vk : 0.0;
}

// Top-k of one score row (one warp): the k-th largest fp32 score by bitwise
// search, then the scores within the fp32 error band of that boundary are
// re-ranked in fp64 from the exact cube sums; the selected cube ids are
// written in ascending order.  With 0 < KPL <= 32 the row's keys are in
// `key` (load_row_keys; N <= 32 * KPL) and every pass reads them there; with
// KPL > 32 they are loaded for the k-th search only (the registers they take
// are released before the other passes, which read the row from memory); with
// KPL == 0 every pass reads memory.  `row` (shared or global memory) is
// scratch: re-ranked band members are overwritten with +inf (chosen) or -inf.
__host__ __device__ constexpr bool keys_in_regs(int kpl) { return kpl > 0 && kpl <= 32; }
template <int D, int KPL>
__device__ void select_row(float* row, uint32_t (&key)[keys_in_regs(KPL) ? KPL : 1], const ScoreArgs& a,
                           size_t bh, size_t hrow, int i, float qnorm_i, float kmax_all, double* qsum, double* cs,
                           int* cj, int lane) {
    constexpr bool kRegs = keys_in_regs(KPL);
    const int N = a.N;
    const int k = a.topk;
    // Error bound of an fp32 score against the exact one (dot of rounded
    // means with fp32 accumulation, then the scale): (D + 8) u |q||k|,
    // doubled for margin (eps).  Every score within eps of the exact one, the
    // fp32 k-th largest tau within eps of the exact k-th: a score above
    // tau + 2 eps is in the exact top-k, one below tau - 2 eps is not, and the
    // ones between (the band) are re-ranked exactly.  The k-th search may stop
    // with tau known only to [tau_lo, tau_hi] (width <= eps); the band then
    // runs from tau_lo - 2 eps to tau_hi + 2 eps, which holds the exact one's.
    const float eps = 2.f * (float)(D + 8) * 5.9604645e-8f * a.sm_scale * qnorm_i * kmax_all;
    uint32_t T;
    int rem = 0;
    if constexpr (kRegs) {
        T = kth_key_regs<KPL>(key, N, k, lane, eps, rem);
    } else if constexpr (KPL > 0) {
        uint32_t kk[KPL];
        load_row_keys<KPL>(row, N, lane, kk);
        T = kth_key_regs<KPL>(kk, N, k, lane, eps, rem);
    } else {
        T = kth_key_mem(row, N, k, lane);
    }
    const float tau_lo = key2f(T);
    const float tau_hi = key2f(rem > 0 ? T | ((1u << (rem - 1)) * 2u - 1u) : T);
    const float band = 2.f * eps + 1e-30f;
    const float lo = tau_lo - band, hi = tau_hi + band;
    int cA = 0, cC = 0;
    if constexpr (kRegs) {
#pragma unroll
        for (int q = 0; q < KPL; ++q) {
            const float s = key2f(key[q]);
            const bool real = lane + 32 * q < N;
            cA += real && s > hi;
            cC += real && s >= lo && s <= hi;
        }
    } else {
        for (int j = lane; j < N; j += 32) {
            const float s = row[j];
            cA += s > hi;
            cC += (s >= lo) && (s <= hi);
        }
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
            if constexpr (kRegs) {
#pragma unroll
                for (int q = 0; q < KPL; ++q) {
                    const int j = lane + 32 * q;
                    const float s = key2f(key[q]);
                    const bool inC = j < N && s >= lo && s <= hi;
                    const unsigned m = __ballot_sync(0xffffffffu, inC);
                    if (inC) cj[pos + __popc(m & ((1u << lane) - 1u))] = j;
                    pos += __popc(m);
                }
            } else {
                for (int j0b = 0; j0b < N; j0b += 32) {
                    const int j = j0b + lane;
                    const bool inC = j < N && row[j] >= lo && row[j] <= hi;
                    const unsigned m = __ballot_sync(0xffffffffu, inC);
                    if (inC) cj[pos + __popc(m & ((1u << lane) - 1u))] = j;
                    pos += __popc(m);
                }
            }
            __syncwarp();
            for (int c = 0; c < cC; ++c) {  // warp-uniform: one candidate at a time, the warp's lanes on its channels
                const double sc = precise_score_warp<D>(qsum, a, hrow, cj[c], inv_vq, lane);
                if (lane == 0) cs[c] = sc;
            }
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
        if constexpr (kRegs) {
            // The band members' decisions (+inf / -inf) back into the keys.
#pragma unroll
            for (int q = 0; q < KPL; ++q) {
                const int j = lane + 32 * q;
                const float s = key2f(key[q]);
                if (j < N && s >= lo && s <= hi) key[q] = f2key(row[j]);
            }
        }
    }
    // Emit the selected set in ascending cube index.  After re-ranking the
    // band members hold +inf (chosen) or -inf (not chosen).
    int32_t* out = a.topk_idx + (bh * N + i) * (size_t)k;
    int pos = 0;
    const unsigned below = (1u << lane) - 1u;
    if constexpr (kRegs) {
#pragma unroll
        for (int q = 0; q < KPL; ++q) {
            const int j = lane + 32 * q;
            const float x = key2f(key[q]);
            const bool sel = j < N && (x > hi || (take_band && x >= lo));
            const unsigned m = __ballot_sync(0xffffffffu, sel);
            if (sel) out[pos + __popc(m & below)] = j;
            pos += __popc(m);
        }
    } else {
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
        float* row = sc + (size_t)r * N;
        if (N <= 256) {
            uint32_t key[8];
            load_row_keys<8>(row, N, lane, key);
            select_row<D, 8>(row, key, a, bh, hrow, i, qnorm[r], kmax_all, qsum_w + warp * D,
                             cand_s + warp * kCandCap, cand_j + warp * kCandCap, lane);
        } else {  // only when a caller without room for the score matrix takes this kernel for long rows
            uint32_t none[1];
            select_row<D, 0>(row, none, a, bh, hrow, i, qnorm[r], kmax_all, qsum_w + warp * D,
                             cand_s + warp * kCandCap, cand_j + warp * kCandCap, lane);
        }
    }
}

// ------------------------------------------- large N: scores through memory
// When few query rows fit the fused kernel's shared memory (N above ~1100 at
// D = 128), the scores go to the workspace instead: a register-tiled fp32
// GEMM of the cube means, then one warp per row runs the same selection on
// the row read back (from L2: the [B, heads, N, N] scores of a call are tens
// of MB).
//
// GEMM: 128 x 128 score tiles, 256 threads, each 8 x 8 scores (rows
// 4 ty + {0..3} and 64 + 4 ty + {0..3}, columns likewise from tx); the depth
// runs in slices of 16 channels through double-buffered shared memory, the
// next slice's global loads in flight during the current slice's FMAs.
// Slices are stored channel-major (As[k][m]), so a thread's 8 rows are two
// float4 reads; a loading thread takes 8 consecutive channels (32 bytes) of
// one row and writes them transposed, a warp's 32 rows to 32 banks.  Each
// score accumulates its D products in increasing channel order.
constexpr int kGemmTile = 128;
constexpr int kGemmK = 16;

template <int D>
__global__ void __launch_bounds__(256, 2) score_gemm_kernel(ScoreArgs a, float* __restrict__ scores) {
    constexpr int KT = D / kGemmK;
    __shared__ __align__(16) float As[2][kGemmK][kGemmTile];
    __shared__ __align__(16) float Bs[2][kGemmK][kGemmTile];
    const int N = a.N;
    const int i0 = blockIdx.x * kGemmTile, j0 = blockIdx.y * kGemmTile;
    const size_t bh = blockIdx.z;
    const float* Ag = a.qm + bh * (size_t)N * D;
    const float* Bg = a.km + bh * (size_t)N * D;
    const int tid = threadIdx.x;
    const int lrow = tid & (kGemmTile - 1);  // loader: one row, channels lk .. lk + 7 of the slice
    const int lk = (tid >> 7) * 8;
    const bool a_in = i0 + lrow < N, b_in = j0 + lrow < N;
    const float* ag = Ag + (size_t)(a_in ? i0 + lrow : 0) * D + lk;
    const float* bg = Bg + (size_t)(b_in ? j0 + lrow : 0) * D + lk;
    float4 pa[2], pb[2];
    auto gload = [&](int kt) {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        pa[0] = a_in ? *reinterpret_cast<const float4*>(ag + kt * kGemmK) : z;
        pa[1] = a_in ? *reinterpret_cast<const float4*>(ag + kt * kGemmK + 4) : z;
        pb[0] = b_in ? *reinterpret_cast<const float4*>(bg + kt * kGemmK) : z;
        pb[1] = b_in ? *reinterpret_cast<const float4*>(bg + kt * kGemmK + 4) : z;
    };
    auto sstore = [&](int buf) {
        const float av[8] = {pa[0].x, pa[0].y, pa[0].z, pa[0].w, pa[1].x, pa[1].y, pa[1].z, pa[1].w};
        const float bv[8] = {pb[0].x, pb[0].y, pb[0].z, pb[0].w, pb[1].x, pb[1].y, pb[1].z, pb[1].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            As[buf][lk + e][lrow] = av[e];
            Bs[buf][lk + e][lrow] = bv[e];
        }
    };
    const int ty = tid >> 4, tx = tid & 15;
    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
    gload(0);
    sstore(0);
    __syncthreads();
#pragma unroll 1
    for (int kt = 0; kt < KT; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < KT) gload(kt + 1);
#pragma unroll
        for (int k = 0; k < kGemmK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][4 * ty]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][64 + 4 * ty]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][4 * tx]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][64 + 4 * tx]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
        }
        if (kt + 1 < KT) sstore(buf ^ 1);  // buffer buf ^ 1 was last read before the previous barrier
        __syncthreads();
    }
    const bool vec = (N & 3) == 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int i = i0 + (r < 4 ? 4 * ty + r : 64 + 4 * ty + r - 4);
        if (i >= N) continue;
        float* dst = scores + (bh * N + i) * (size_t)N;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = j0 + 64 * h + 4 * tx;
            const float v0 = a.sm_scale * acc[r][4 * h], v1 = a.sm_scale * acc[r][4 * h + 1];
            const float v2 = a.sm_scale * acc[r][4 * h + 2], v3 = a.sm_scale * acc[r][4 * h + 3];
            if (vec && j + 3 < N) {
                *reinterpret_cast<float4*>(dst + j) = make_float4(v0, v1, v2, v3);
            } else {
                if (j < N) dst[j] = v0;
                if (j + 1 < N) dst[j + 1] = v1;
                if (j + 2 < N) dst[j + 2] = v2;
                if (j + 3 < N) dst[j + 3] = v3;
            }
        }
    }
}

// One warp per row; rows of up to 1024 scores are held in registers (KPL
// slots per lane), loaded before the block's reduction of the key norms so
// the two overlap.
template <int KPL>
constexpr int select_min_blocks() { return KPL <= 24 ? 4 : 3; }
template <int D, int KPL>
__global__ void __launch_bounds__(256, select_min_blocks<KPL>()) select_kernel(ScoreArgs a, float* __restrict__ scores) {
    __shared__ double qsum_w[8][D];
    __shared__ double cand_s[8][kCandCap];
    __shared__ int cand_j[8][kCandCap];
    __shared__ float red[8];
    const int N = a.N;
    const size_t bh = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i = blockIdx.x * 8 + warp;
    float* row = scores + (bh * N + (i < N ? i : N - 1)) * (size_t)N;
    uint32_t key[keys_in_regs(KPL) ? KPL : 1];
    if constexpr (keys_in_regs(KPL)) load_row_keys<KPL>(row, N, lane, key);
    float kmax = 0.f;  // largest key-mean norm of this head
    for (int j = tid; j < N; j += 256) kmax = fmaxf(kmax, a.kn[bh * N + j]);
#pragma unroll
    for (int o = 16; o; o >>= 1) kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    if (lane == 0) red[warp] = kmax;
    __syncthreads();
    float kmax_all = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) kmax_all = fmaxf(kmax_all, red[w]);
    if (i >= N) return;
    select_row<D, KPL>(row, key, a, bh, bh * (size_t)N * D, i, a.qn[bh * N + i], kmax_all, qsum_w[warp],
                       cand_s[warp], cand_j[warp], lane);
}

// The select_kernel instance for rows of N scores: register slots per lane
// ceil(N / 32) rounded up to a multiple of 4 up to 32 and of 8 up to 64;
// longer rows are searched in memory.
template <int D>
using SelectFn = void (*)(ScoreArgs, float*);
template <int D>
SelectFn<D> select_kernel_for(int N) {
    const int c = (N + 31) / 32;
    if (c <= 4) return select_kernel<D, 4>;
    if (c <= 8) return select_kernel<D, 8>;
    if (c <= 12) return select_kernel<D, 12>;
    if (c <= 16) return select_kernel<D, 16>;
    if (c <= 20) return select_kernel<D, 20>;
    if (c <= 24) return select_kernel<D, 24>;
    if (c <= 28) return select_kernel<D, 28>;
    if (c <= 32) return select_kernel<D, 32>;
    if (c <= 40) return select_kernel<D, 40>;
    if (c <= 48) return select_kernel<D, 48>;
    if (c <= 56) return select_kernel<D, 56>;
    if (c <= 64) return select_kernel<D, 64>;
    return select_kernel<D, 0>;
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
    if (split) return 0;  // the score GEMM and the selection use static shared memory only
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
        const int tiles = (ncubes + kGemmTile - 1) / kGemmTile;
        const dim3 gg(tiles, tiles, B * heads);
        auto gemm = D == 128 ? score_gemm_kernel<128> : score_gemm_kernel<64>;
        gemm<<<gg, 256, 0, stream>>>(a, scores);
        auto sel = D == 128 ? select_kernel_for<128>(ncubes) : select_kernel_for<64>(ncubes);
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
