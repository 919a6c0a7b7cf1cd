// Fine stage: non-causal block-sparse attention over the selected cubes.
//
// Computes, per (batch, head, query cube i) and each of its 64 query rows,
// softmax(sm_scale * q k_sel^T) v_sel over the keys of the selected cubes,
// the first vbs[j] slots of cube j only ("Wan2.2 Production Values -- VSA
// Block-Sparse Attention Inputs + Reference", Operator contract), as an
// online softmax with a running maximum and sum ("VSA: Accelerating Video
// Diffusion Inference with Sparse Attention on AMD GPUs", Kernel Architecture
// and Sparse Traversal: walk the query block's K/V block list only).
//
// sm_103a design (5th-generation tensor cores, TMEM, TMA):
//  * Work unit = one (b, head, query cube).  Persistent grid, one CTA per SM,
//    units dealt round-robin in head-major order so one head's K/V stays in L2.
//  * A step processes TWO selected key cubes (128 keys) at once in transposed
//    form, so every MMA is M = 128 with no wasted rows:
//        S^T[128 keys x 64 q]  = K_pair[128 x D] . Q^T          (tcgen05, TMEM)
//        O^T[D x 64 q]        += V_pair^T[D x 128] . P^T[128 x 64] (tcgen05, TMEM)
//    An odd last cube runs as a half step (PV over 64 keys).
//  * Warp roles (320 threads): warp 0 = TMA producer, warp 1 = MMA issuer
//    (also owns TMEM), warps 2..9 = softmax.  Each softmax thread owns one key
//    row of S^T (its TMEM lane) and 32 of the 64 query columns.
//  * Softmax per column keeps a running max m in log2 units.  The max is set
//    exactly from the first step of a unit; later steps only re-reduce (and
//    rescale O^T and the partial sums) when some logit exceeds m by more than
//    kRescaleThreshold, so the usual step needs no cross-thread reduction.
//    exp2 arguments are then <= the threshold: no overflow for logits of any
//    finite size.
//  * Padded key slots (slot >= vbs[j]) get probability 0; P^T is written as
//    bf16 into a 128-byte-swizzled shared-memory tile that is the B operand
//    of the PV MMA.
//  * Every wait is bounded; a wait that runs out raises a CTA abort flag and
//    the device error word, and each role winds down without deadlock.
#include <cuda_bf16.h>
#include <math.h>

#include "vsa_common.cuh"

namespace vsa {

namespace {

constexpr int kStages = 3;            // key/value pair stages in the TMA ring
constexpr int kThreads = 320;         // 10 warps
constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr float kRescaleThreshold = 10.0f;  // log2 units
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kIdxPerLane = 8;        // producer keeps 256 indices in registers

// Shared-memory layout (bytes from a 1024-aligned base).
constexpr int kChunkRows64 = 64 * 128;           // 64 rows x 128 B   = 8 KB
constexpr int kChunkRows128 = 128 * 128;         // 128 rows x 128 B  = 16 KB
constexpr int kOffQ = 0;                         // [2 chunks][64 q][128 B]
constexpr int kOffK = kOffQ + 2 * kChunkRows64;  // [stage][2 chunks][128 keys][128 B]
constexpr int kStageBytes = 2 * kChunkRows128;   // 32 KB per tensor per stage
constexpr int kOffV = kOffK + kStages * kStageBytes;
constexpr int kOffP = kOffV + kStages * kStageBytes;  // [128 keys][128 B]
constexpr int kOffMisc = kOffP + kChunkRows128;

struct __align__(16) Misc {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t s_full[2];
    uint64_t p_full;
    uint64_t o_done;
    uint64_t drain;
    int4 info[kStages];          // per stage: cube a, vbs a, cube b (-1 = none), vbs b
    float m[64];                 // running max per query column (log2 units)
    float mb[64];                // exp base: m, or 0 while m = -inf
    float alpha[64];             // rescale factor of the last update
    float red[kSoftmaxWarps][32];
    uint32_t tmem_base;
    int abort_flag;
    int m_neg_inf;               // some column still has m = -inf
};

constexpr int kSmemBytes = kOffMisc + (int)sizeof(Misc);
constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment

static_assert(kSmemAlloc <= 232448, "fine kernel shared memory exceeds the sm_103a limit");

struct FineParams {
    const int32_t* topk_idx;
    const int32_t* vbs;
    __nv_bfloat16* out;  // unused type-wise, raw bf16 bits written
    float* lse;
    unsigned int* err;
    int B, N, heads, D, topk, nsteps;
    int num_units;
    float scale_log2;  // sm_scale * log2(e)
};

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool named_red_or(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Reduce 32 per-thread column values over the 32 lanes of a warp; lane L
// returns the reduction of column L.
template <bool kMax>
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < off; ++j) {
            const float send = up ? v[j] : v[j + off];
            const float keep = up ? v[j + off] : v[j];
            const float recv = __shfl_xor_sync(0xffffffffu, send, off);
            v[j] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
    }
    return v[0];
}

__device__ __forceinline__ void unit_coords(int u, int N, int heads, int& b, int& h, int& i) {
    i = u % N;
    const int bh = u / N;
    h = bh % heads;
    b = bh / heads;
}

__global__ void __launch_bounds__(kThreads, 1)
    fine_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, FineParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort_flag = &ms.abort_flag;

    const int D = p.D;
    const int nchunks = D / 64;
    const int s_pad = p.N * kCubeTokens;

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&ms.kv_full[s]), 1);
            mbar_init(smem_u32(&ms.kv_empty[s]), 1);
        }
        mbar_init(smem_u32(&ms.q_full), 1);
        mbar_init(smem_u32(&ms.q_empty), 1);
        mbar_init(smem_u32(&ms.s_full[0]), 1);
        mbar_init(smem_u32(&ms.s_full[1]), 1);
        mbar_init(smem_u32(&ms.p_full), kSoftmaxWarps);
        mbar_init(smem_u32(&ms.o_done), 1);
        mbar_init(smem_u32(&ms.drain), 1);
        ms.abort_flag = 0;
        ms.m_neg_inf = 0;
        fence_barrier_init();
    }
    // Zero the K/V stages once: half steps read rows no TMA wrote, and for
    // D = 64 the second V chunk must stay zero.
    {
        int4* z = reinterpret_cast<int4*>(smem + kOffK);
        const int n16 = 2 * kStages * kStageBytes / 16;
        for (int e = threadIdx.x; e < n16; e += kThreads) z[e] = make_int4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ms.tmem_base), 256);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;

    const int nsteps = p.nsteps;
    const int k = p.topk;

    if (warp == 0) {
        // ============================================================ producer
        const uint64_t pol_kv = l2_policy_evict_last();
        const uint64_t pol_q = l2_policy_evict_first();
        uint32_t g = 0;
        int ucount = 0;
        uint32_t last_g[kStages];
        for (int s = 0; s < kStages; ++s) last_g[s] = 0xFFFFFFFFu;
        bool q_issued = false;
        bool ok = true;
        for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++ucount) {
            int b, h, i;
            unit_coords(u, p.N, p.heads, b, h, i);
            if (ucount > 0) {
                ok = mbar_wait_bounded(smem_u32(&ms.q_empty), (ucount - 1) & 1, abort_flag, p.err,
                                       kWaitLimitNs);
                if (!ok) break;
            }
            const int row0 = b * s_pad + i * kCubeTokens;
            if (lane == 0) {
                const uint32_t qbar = smem_u32(&ms.q_full);
                mbar_arrive_expect_tx(qbar, (uint32_t)(kCubeTokens * D * 2));
                for (int c = 0; c < nchunks; ++c)
                    tma_load_3d(sbase + kOffQ + c * kChunkRows64, &tm_q, qbar, c * 64, h, row0, pol_q);
            }
            q_issued = true;
            const int32_t* idx_row = p.topk_idx + (((size_t)b * p.heads + h) * p.N + i) * (size_t)k;
            int idx_reg[kIdxPerLane], vbs_reg[kIdxPerLane];
            for (int t = 0; t < nsteps && ok; ++t) {
                const int e0 = 2 * t;
                if ((e0 & (32 * kIdxPerLane - 1)) == 0) {
                    // (Re)load the next 256 indices of the row and their vbs.
#pragma unroll
                    for (int s = 0; s < kIdxPerLane; ++s) {
                        const int e = e0 + s * 32 + lane;
                        idx_reg[s] = e < k ? __ldg(idx_row + e) : -1;
                        vbs_reg[s] = idx_reg[s] >= 0 ? __ldg(p.vbs + idx_reg[s]) : 0;
                    }
                }
                const int stage = g % kStages;
                if (g >= (uint32_t)kStages) {
                    ok = mbar_wait_bounded(smem_u32(&ms.kv_empty[stage]), ((g / kStages) + 1) & 1,
                                           abort_flag, p.err, kWaitLimitNs);
                    if (!ok) break;
                }
                // Fetch entries e0 and e0 + 1 from their owner lanes.
                int ja = -1, va = 0, jb = -1, vb = 0;
                {
                    const int ea = e0 & (32 * kIdxPerLane - 1), eb = ea + 1;
                    int xa = 0, ya = 0, xb = 0, yb = 0;
#pragma unroll
                    for (int s = 0; s < kIdxPerLane; ++s) {
                        if ((ea >> 5) == s) { xa = idx_reg[s]; ya = vbs_reg[s]; }
                        if ((eb >> 5) == s) { xb = idx_reg[s]; yb = vbs_reg[s]; }
                    }
                    ja = __shfl_sync(0xffffffffu, xa, ea & 31);
                    va = __shfl_sync(0xffffffffu, ya, ea & 31);
                    jb = __shfl_sync(0xffffffffu, xb, eb & 31);
                    vb = __shfl_sync(0xffffffffu, yb, eb & 31);
                    if (e0 + 1 >= k) { jb = -1; vb = 0; }
                }
                if (lane == 0) {
                    ms.info[stage] = make_int4(ja, va, jb, vb);
                    const uint32_t fbar = smem_u32(&ms.kv_full[stage]);
                    const uint32_t bytes = (uint32_t)((jb >= 0 ? 2 : 1) * 2 * kCubeTokens * D * 2);
                    mbar_arrive_expect_tx(fbar, bytes);
                    const uint32_t kst = sbase + kOffK + stage * kStageBytes;
                    const uint32_t vst = sbase + kOffV + stage * kStageBytes;
                    const int ra = b * s_pad + ja * kCubeTokens;
                    for (int c = 0; c < nchunks; ++c) {
                        tma_load_3d(kst + c * kChunkRows128, &tm_k, fbar, c * 64, h, ra, pol_kv);
                        tma_load_3d(vst + c * kChunkRows128, &tm_v, fbar, c * 64, h, ra, pol_kv);
                    }
                    if (jb >= 0) {
                        const int rb = b * s_pad + jb * kCubeTokens;
                        for (int c = 0; c < nchunks; ++c) {
                            tma_load_3d(kst + c * kChunkRows128 + kChunkRows64, &tm_k, fbar, c * 64, h, rb,
                                        pol_kv);
                            tma_load_3d(vst + c * kChunkRows128 + kChunkRows64, &tm_v, fbar, c * 64, h, rb,
                                        pol_kv);
                        }
                    }
                }
                last_g[stage] = g;
                ++g;
            }
        }
        // Drain: every issued copy must land before the CTA exits.
        for (int s = 0; s < kStages; ++s)
            if (last_g[s] != 0xFFFFFFFFu)
                mbar_wait_bounded(smem_u32(&ms.kv_full[s]), (last_g[s] / kStages) & 1, abort_flag, p.err,
                                  kWaitLimitNs);
        if (q_issued)
            mbar_wait_bounded(smem_u32(&ms.q_full), (ucount - 1) & 1, abort_flag, p.err, kWaitLimitNs);
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 64, 0, 0);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 64, 1, 1);
        const uint32_t t_s0 = tmem;          // S^T buffers: columns [0, 64) and [64, 128)
        const uint32_t t_o = tmem + 128;     // O^T: columns [128, 192)
        uint32_t g = 0;
        int ucount = 0;
        bool ok = true;
        // Issues QK^T for global step gg (Q resident, K/V of stage landed).
        // release_q: gg is the last step of its unit, so the Q buffer is free
        // once this MMA completes.
        auto issue_qk = [&](uint32_t gg, bool release_q) {
            const int stage = gg % kStages;
            const uint32_t kst = sbase + kOffK + stage * kStageBytes;
            const uint32_t d_tmem = t_s0 + (gg & 1) * 64;
            if (lane == 0) {
                tc_fence_after();
                int n = 0;
                for (int c = 0; c < nchunks; ++c)
                    for (int kk = 0; kk < 4; ++kk, ++n) {
                        const uint64_t a = smem_desc_sw128(kst + c * kChunkRows128 + kk * 32, 16, 1024);
                        const uint64_t bq = smem_desc_sw128(sbase + kOffQ + c * kChunkRows64 + kk * 32, 16, 1024);
                        mma_ss(d_tmem, a, bq, idesc_qk, n > 0);
                    }
                mma_commit(smem_u32(&ms.s_full[gg & 1]));
                if (release_q) mma_commit(smem_u32(&ms.q_empty));
            }
            __syncwarp();
        };
        const int first_u = blockIdx.x;
        if (first_u < p.num_units) {
            ok = mbar_wait_bounded(smem_u32(&ms.q_full), 0, abort_flag, p.err, kWaitLimitNs) &&
                 mbar_wait_bounded(smem_u32(&ms.kv_full[0]), 0, abort_flag, p.err, kWaitLimitNs);
            if (ok) issue_qk(0, nsteps == 1);
        }
        for (int u = first_u; u < p.num_units && ok; u += gridDim.x, ++ucount) {
            const bool has_next_unit = u + (int)gridDim.x < p.num_units;
            for (int t = 0; t < nsteps && ok; ++t) {
                const bool last_in_unit = (t + 1 == nsteps);
                const bool next_exists = !last_in_unit || has_next_unit;
                // Within a unit the next QK^T goes first (it feeds the next
                // softmax step); at a unit boundary the PV goes first.
                if (next_exists && !last_in_unit) {
                    const uint32_t gn = g + 1;
                    ok = mbar_wait_bounded(smem_u32(&ms.kv_full[gn % kStages]), (gn / kStages) & 1,
                                           abort_flag, p.err, kWaitLimitNs);
                    if (!ok) break;
                    issue_qk(gn, t + 2 == nsteps);
                }
                ok = mbar_wait_bounded(smem_u32(&ms.p_full), g & 1, abort_flag, p.err, kWaitLimitNs);
                if (!ok) break;
                {
                    const int stage = g % kStages;
                    const uint32_t vst = sbase + kOffV + stage * kStageBytes;
                    const bool half = (2 * t + 1 >= k);
                    const int ksteps = half ? 4 : 8;
                    if (lane == 0) {
                        tc_fence_after();
                        for (int kk = 0; kk < ksteps; ++kk) {
                            const uint64_t a = smem_desc_sw128(vst + kk * 2048, kChunkRows128, 1024);
                            const uint64_t bp = smem_desc_sw128(sbase + kOffP + kk * 2048, kChunkRows128, 1024);
                            mma_ss(t_o, a, bp, idesc_pv, (t > 0 || kk > 0));
                        }
                        mma_commit(smem_u32(&ms.o_done));
                        mma_commit(smem_u32(&ms.kv_empty[stage]));
                    }
                    __syncwarp();
                }
                if (next_exists && last_in_unit) {
                    const uint32_t gn = g + 1;
                    ok = mbar_wait_bounded(smem_u32(&ms.q_full), (ucount + 1) & 1, abort_flag, p.err,
                                           kWaitLimitNs) &&
                         mbar_wait_bounded(smem_u32(&ms.kv_full[gn % kStages]), (gn / kStages) & 1,
                                           abort_flag, p.err, kWaitLimitNs);
                    if (!ok) break;
                    issue_qk(gn, nsteps == 1);
                }
                ++g;
            }
        }
        // Drain: all issued MMAs complete before TMEM is released.
        if (lane == 0) mma_commit(smem_u32(&ms.drain));
        __syncwarp();
        mbar_wait_bounded(smem_u32(&ms.drain), 0, abort_flag, p.err, kWaitLimitNs);
    } else {
        // ============================================================ softmax
        const int sw = warp - 2;            // 0..7
        const int quarter = warp & 3;       // TMEM lane quarter this warp may access
        const int half = sw >> 2;           // query columns [32*half, 32*half + 32)
        const int key = quarter * 32 + lane;  // S^T row = key slot in the pair (0..127)
        const int cube_sel = key >> 6;      // 0: first cube of the pair, 1: second
        const int slot = key & 63;
        const int col0 = half * 32;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const float c2 = p.scale_log2;
        const float ninf = -INFINITY;
        bool ok = true;
        uint32_t g = 0;
        float lpart[32];
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            int b, h, i;
            unit_coords(u, p.N, p.heads, b, h, i);
#pragma unroll
            for (int q = 0; q < 32; ++q) lpart[q] = 0.f;
            for (int t = 0; t < nsteps; ++t, ++g) {
                const int stage = g % kStages;
                const uint32_t sbuf = g & 1;
                if (ok) ok = mbar_wait_bounded(smem_u32(&ms.s_full[sbuf]), (g >> 1) & 1, abort_flag, p.err,
                                               kWaitLimitNs);
                if (ok) ok = mbar_wait_bounded(smem_u32(&ms.kv_full[stage]), (g / kStages) & 1, abort_flag,
                                               p.err, kWaitLimitNs);
                tc_fence_after();
                const int4 inf = ms.info[stage];
                const bool active = (cube_sel == 0) || (inf.z >= 0);  // warp-uniform
                const int vbm = cube_sel == 0 ? inf.y : inf.w;
                const bool real = ok && active && slot < vbm;
                float y[32];
                if (ok && active) {
                    uint32_t raw[32];
                    tmem_ld32(t_lane + sbuf * 64 + col0, raw);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 32; ++q) y[q] = __uint_as_float(raw[q]) * c2;  // log2-scaled logit
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) y[q] = 0.f;
                }
                if (!real) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) y[q] = ninf;
                }
                // Does any logit exceed its column base by more than the threshold?
                float mbr[32];
#pragma unroll
                for (int q = 0; q < 32; q += 4) {
                    const float4 m4 = *reinterpret_cast<const float4*>(&ms.mb[col0 + q]);
                    mbr[q] = m4.x; mbr[q + 1] = m4.y; mbr[q + 2] = m4.z; mbr[q + 3] = m4.w;
                }
                bool need = (t == 0);
                if (t > 0) {
                    float dmax = ninf;
#pragma unroll
                    for (int q = 0; q < 32; ++q) dmax = fmaxf(dmax, y[q] - mbr[q]);
                    bool trig = dmax > kRescaleThreshold || (real && ms.m_neg_inf);
                    need = named_red_or(1, kSoftmaxThreads, trig);
                }
                if (need) {
                    // Exact column max over the 128 keys of this step.
                    float v[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] = y[q];
                    const float cm = transpose_reduce32<true>(v, lane);
                    ms.red[sw][lane] = cm;
                    named_sync(1, kSoftmaxThreads);
                    if (sw == 0 || sw == 4) {
                        const int col = col0 + lane;
                        float mx = ms.red[sw][lane];
#pragma unroll
                        for (int w = 1; w < 4; ++w) mx = fmaxf(mx, ms.red[sw + w][lane]);
                        const float m_old = (t == 0) ? ninf : ms.m[col];
                        const float m_new = fmaxf(m_old, mx);
                        ms.alpha[col] = (m_old == ninf) ? 0.f : ex2_approx(m_old - m_new);
                        ms.m[col] = m_new;
                        ms.mb[col] = (m_new == ninf) ? 0.f : m_new;
                    }
                    named_sync(1, kSoftmaxThreads);
                    if (sw == 0 && lane == 0) {
                        int any = 0;
                        for (int c = 0; c < 64; ++c) any |= (ms.m[c] == ninf);
                        ms.m_neg_inf = any;
                    }
                    if (t > 0) {
#pragma unroll
                        for (int q = 0; q < 32; ++q) lpart[q] *= ms.alpha[col0 + q];
                        // Rescale O^T: wait for the previous PV, then scale the columns.
                        if (ok) ok = mbar_wait_bounded(smem_u32(&ms.o_done), (g - 1) & 1, abort_flag, p.err,
                                                       kWaitLimitNs);
                        if (ok) {
                            tc_fence_after();
                            uint32_t o[32];
                            tmem_ld32(t_lane + 128 + col0, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int q = 0; q < 32; ++q)
                                o[q] = __float_as_uint(__uint_as_float(o[q]) * ms.alpha[col0 + q]);
                            tmem_st32(t_lane + 128 + col0, o);
                            tmem_wait_st();
                        }
                    }
                    named_sync(1, kSoftmaxThreads);  // m_neg_inf published
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        const float4 m4 = *reinterpret_cast<const float4*>(&ms.mb[col0 + q]);
                        mbr[q] = m4.x; mbr[q + 1] = m4.y; mbr[q + 2] = m4.z; mbr[q + 3] = m4.w;
                    }
                }
                // Probabilities (exp2 relative to the column base) and partial sums.
                uint32_t pk[16];
#pragma unroll
                for (int q = 0; q < 32; q += 2) {
                    const float p0 = ex2_approx(y[q] - mbr[q]);
                    const float p1 = ex2_approx(y[q + 1] - mbr[q + 1]);
                    lpart[q] += p0;
                    lpart[q + 1] += p1;
                    pk[q >> 1] = pack_bf16x2(p0, p1);
                }
                // The single P^T buffer is free once the previous PV finished.
                if (g > 0 && ok)
                    ok = mbar_wait_bounded(smem_u32(&ms.o_done), (g - 1) & 1, abort_flag, p.err, kWaitLimitNs);
                if (ok && active) {
                    unsigned char* prow = smem + kOffP + key * 128;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int chunk = (half * 4 + cc) ^ (key & 7);
                        *reinterpret_cast<uint4*>(prow + chunk * 16) =
                            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ms.p_full));
            }
            // ------------------------------------------------ unit epilogue
            {
                float v[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = lpart[q];
                const float ls = transpose_reduce32<false>(v, lane);
                ms.red[sw][lane] = ls;
                named_sync(1, kSoftmaxThreads);
                if (sw == 0 || sw == 4) {
                    const int col = col0 + lane;
                    float l = ms.red[sw][lane];
#pragma unroll
                    for (int w = 1; w < 4; ++w) l += ms.red[sw + w][lane];
                    ms.alpha[col] = l > 0.f ? 1.f / l : 0.f;  // reused: 1 / l
                    if (p.lse && ok) {
                        const float lse = l > 0.f ? (ms.m[col] + __log2f(l)) * 0.69314718055994531f : ninf;
                        p.lse[((size_t)b * p.heads + h) * s_pad + (size_t)i * kCubeTokens + col] = lse;
                    }
                }
                named_sync(1, kSoftmaxThreads);
                if (ok) ok = mbar_wait_bounded(smem_u32(&ms.o_done), (g - 1) & 1, abort_flag, p.err, kWaitLimitNs);
                if (ok) {
                    tc_fence_after();
                    uint32_t o[32];
                    tmem_ld32(t_lane + 128 + col0, o);
                    tmem_wait_ld();
                    const int d = key;  // O^T lane = head-dim index
                    if (d < D) {
                        unsigned short* ob = reinterpret_cast<unsigned short*>(p.out);
                        const size_t rs = (size_t)p.heads * D;
                        const size_t base = ((size_t)b * s_pad + (size_t)i * kCubeTokens + col0) * rs +
                                            (size_t)h * D + d;
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            const float val = __uint_as_float(o[q]) * ms.alpha[col0 + q];
                            const __nv_bfloat16 bv = __float2bfloat16_rn(val);
                            __stcs(ob + base + (size_t)q * rs, *reinterpret_cast<const unsigned short*>(&bv));
                        }
                    }
                }
                tc_fence_before();
                named_sync(1, kSoftmaxThreads);  // 1/l and m are rewritten by the next unit
            }
        }
    }

    // ------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

}  // namespace

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 3-D map over a [B*S, heads, D] bf16 tensor with a {64, 1, 64} box.
static bool make_map(CUtensorMap* m, const void* base, int rows, int heads, int D, bool swizzle) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int fine_smem_bytes() { return kSmemAlloc; }

cudaError_t launch_fine(const void* qt, const void* kt, const void* vt, const int32_t* topk_idx,
                        const int32_t* vbs, int B, int ncubes, int heads, int D, int topk, float sm_scale,
                        void* out, float* lse, unsigned int* err, int num_sms, cudaStream_t stream) {
    CUtensorMap mq, mk, mv;
    const int rows = B * ncubes * kCubeTokens;
    if (!make_map(&mq, qt, rows, heads, D, true) || !make_map(&mk, kt, rows, heads, D, true) ||
        !make_map(&mv, vt, rows, heads, D, true))
        return cudaErrorInvalidValue;
    FineParams p;
    p.topk_idx = topk_idx;
    p.vbs = vbs;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.err = err;
    p.B = B;
    p.N = ncubes;
    p.heads = heads;
    p.D = D;
    p.topk = topk;
    p.nsteps = (topk + 1) / 2;
    p.num_units = B * heads * ncubes;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    cudaError_t e = cudaFuncSetAttribute(fine_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    const int grid = p.num_units < num_sms ? p.num_units : num_sms;
    fine_fwd_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

}  // namespace vsa
