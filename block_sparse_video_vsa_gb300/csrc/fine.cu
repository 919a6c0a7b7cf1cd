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
//  * A work unit is a PAIR of query cubes (2p, 2p+1) of one (batch, head):
//    128 query rows, one per TMEM lane.  It walks the union of the two cubes'
//    selected key cubes, two key cubes (128 keys) per step:
//        S[128 q x 128 keys]  = Q_pair . K_pair^T      (A = Q in TMEM)
//        O[128 q x D]        += P . V_pair            (A = P in TMEM)
//    Both MMAs are M = 128, N = 128 (full tensor-core rate; an M x 64 MMA runs
//    at half rate), and only the B operands (K, V) are read from shared
//    memory, which keeps shared-memory bandwidth to about half of its peak.
//    Query rows of a cube that did not select a key cube get probability 0
//    for it, so each row attends exactly its own selection.
//  * Persistent grid, one CTA per SM, units dealt round-robin in head-major
//    order so one head's K/V stays in L2.
//  * Warp roles (384 threads): warp 0 builds each unit's union list (sorted,
//    with membership bits and vbs) and is the TMA producer of K; warp 1 owns
//    TMEM and issues the Q.K^T MMAs; warp 2 is the TMA producer of V; warp 3
//    issues the P.V MMAs; warps 4..11 run the softmax and stage Q into TMEM.
//    Each MMA-issuing warp runs its loop as a whole warp and lets lane 0
//    issue, so its waits and loop state stay warp-uniform.  A query row is
//    shared by two threads (two warps on the same TMEM lane quarter), one per
//    key cube of the step; they exchange their row maxima through shared
//    memory with a 64-thread named barrier, so the running max, the sum and
//    the lazy rescale of the row's O need no wider synchronisation.
//  * TMEM (512 columns): S double buffer [0,128) [128,256); P of the current
//    step (bf16 pairs) [256,320); Q of the current unit [320,384); O
//    [384,512).  The softmax releases an S buffer as soon as it has loaded
//    it, so QK runs two steps ahead of PV; P has its own columns, rewritten
//    for step g + 1 only after PV(g) completes.
//  * Running max kept in log2 units; O and the sum are rescaled only when a
//    row's max grows by more than kRescaleThreshold, so exp2 arguments stay
//    <= the threshold and logits of any finite size are safe.
//  * Every wait is bounded; a wait that runs out raises a CTA abort flag and
//    the device error word, and each role winds down without deadlock.
#include <cuda_bf16.h>
#include <math.h>

#include "vsa_common.cuh"

namespace vsa {

namespace {

constexpr int kKStages = 3;           // K pair slots (QK operand B)
constexpr int kVStages = 3;           // V pair slots (PV operand B)
constexpr int kSoftmaxWarps = 8;
constexpr int kFirstSoftmaxWarp = 4;
constexpr int kThreads = (kFirstSoftmaxWarp + kSoftmaxWarps) * 32;  // 12 warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kMaxTopk = 512;
constexpr int kMaxUnion = 2 * kMaxTopk;
constexpr int kMaxCubes = 8192;
constexpr int kBitmapWords = kMaxCubes / 32;

// TMEM columns.
constexpr int kTmemS = 0;    // two S buffers of 128 columns
constexpr int kTmemP = 256;  // P of the current step: 128 keys as 64 columns of bf16 pairs
constexpr int kTmemQ = 320;  // Q of the current unit: D bf16 as D/2 columns of pairs
constexpr int kTmemO = 384;  // O accumulator (D columns)

// Shared-memory layout (bytes from a 1024-aligned base).
constexpr int kChunkRows64 = 64 * 128;           // 64 rows x 128 B   = 8 KB
constexpr int kChunkRows128 = 128 * 128;         // 128 rows x 128 B  = 16 KB
constexpr int kPairBytes = 2 * kChunkRows128;    // one tensor for a cube pair: 32 KB
constexpr int kOffK = 0;                         // [slot][2 chunks][128 keys][128 B]
constexpr int kOffV = kOffK + kKStages * kPairBytes;
constexpr int kOffList = kOffV + kVStages * kPairBytes;          // [2][kMaxUnion] packed entries
constexpr int kOffBitmap = kOffList + 2 * kMaxUnion * 4;         // [2][kBitmapWords]
constexpr int kOffMisc = kOffBitmap + 2 * kBitmapWords * 4;

// Union-list entry: cube id (bits 0..15), vbs (bits 16..23), membership
// (bit 24: selected by the first query cube, bit 25: by the second).
__device__ __forceinline__ int entry_cube(uint32_t e) { return (int)(e & 0xFFFFu); }
__device__ __forceinline__ int entry_vbs(uint32_t e) { return (int)((e >> 16) & 0xFFu); }
__device__ __forceinline__ uint32_t entry_mask(uint32_t e) { return (e >> 24) & 3u; }

struct __align__(16) Misc {
    uint64_t k_full[kKStages];
    uint64_t k_empty[kKStages];
    uint64_t v_full[kVStages];
    uint64_t v_empty[kVStages];
    uint64_t s_full[2];
    uint64_t s_free[2];
    uint64_t p_full;
    uint64_t pv_done;
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t list_full[2];
    uint64_t list_empty[2];
    uint64_t drain[2];  // per MMA-issuing warp
    int list_count[2];
    float xmax[2][2][128];        // [step parity][key half][row]: row maxima exchanged by thread pairs
    float xsum[2][128];           // [key half][row]: partial row sums for the epilogue
    uint32_t tmem_base;
    int abort_flag;
};

constexpr int kSmemBytes = kOffMisc + (int)sizeof(Misc);
constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment
static_assert(kSmemAlloc <= 232448, "fine kernel shared memory exceeds the sm_103a limit");

struct FineParams {
    const int32_t* topk_idx;
    const int32_t* vbs;
    const uint32_t* pairs;  // [B * heads][npairs]: i | (j << 16), j = 0xFFFF single; or null: (2u, 2u + 1)
    const int32_t* counts;  // [B * heads * N] entries of each topk_idx row in use (<= topk), or null: all
    const uint4* q;      // tiled q rows (for staging Q into TMEM)
    const float* oc;     // coarse-stage output [B * heads][N][D], or null: no gated combine
    const uint4* gc;     // gates of the coarse and fine terms, bf16 in the layout of out
    const uint4* gf;
    __nv_bfloat16* out;
    float* lse;
    unsigned int* err;
    int B, N, heads, D, topk;
    int npairs;          // ceil(N / 2)
    int num_units;       // B * heads * npairs
    float scale_log2;    // sm_scale * log2(e)
};

__device__ __forceinline__ void unit_coords(int u, const FineParams& p, int& b, int& h, int& pair) {
    pair = u % p.npairs;
    const int bh = u / p.npairs;
    h = bh % p.heads;
    b = bh / p.heads;
}

// Query cubes of unit `pair` of (b, h); -1 for none.
__device__ __forceinline__ void unit_cubes(const FineParams& p, int b, int h, int pair, int& i0, int& i1) {
    if (p.pairs) {
        const uint32_t e = __ldg(p.pairs + ((size_t)b * p.heads + h) * p.npairs + pair);
        i0 = (int)(e & 0xFFFFu);
        i1 = (int)(e >> 16);
    } else {
        i0 = 2 * pair;
        i1 = 2 * pair + 1;
    }
    if (i0 >= p.N) i0 = -1;
    if (i1 >= p.N) i1 = -1;
}

// Builds the sorted union of the two query cubes' selections (one warp).
__device__ int build_union(const FineParams& p, int u, uint32_t* list, uint32_t* bm0, uint32_t* bm1, int lane) {
    int b, h, pair;
    unit_coords(u, p, b, h, pair);
    const int N = p.N, k = p.topk;
    const int nwords = (N + 31) >> 5;
    int i0, i1;
    unit_cubes(p, b, h, pair, i0, i1);
    for (int w = lane; w < nwords; w += 32) {
        bm0[w] = 0u;
        bm1[w] = 0u;
    }
    __syncwarp();
    const int32_t* rows = p.topk_idx + ((size_t)b * p.heads + h) * N * (size_t)k;
    const int32_t* cnt = p.counts ? p.counts + ((size_t)b * p.heads + h) * N : nullptr;
    if (i0 >= 0) {
        const int32_t* r0 = rows + (size_t)i0 * k;
        const int k0 = cnt ? min(max(__ldg(cnt + i0), 0), k) : k;
        for (int e = lane; e < k0; e += 32) {
            const int j = __ldg(r0 + e);
            atomicOr(&bm0[j >> 5], 1u << (j & 31));
        }
    }
    if (i1 >= 0) {
        const int32_t* r1 = rows + (size_t)i1 * k;
        const int k1 = cnt ? min(max(__ldg(cnt + i1), 0), k) : k;
        for (int e = lane; e < k1; e += 32) {
            const int j = __ldg(r1 + e);
            atomicOr(&bm1[j >> 5], 1u << (j & 31));
        }
    }
    __syncwarp();
    int pos = 0;
    for (int w0 = 0; w0 < nwords; w0 += 32) {
        const int w = w0 + lane;
        const uint32_t a0 = w < nwords ? bm0[w] : 0u;
        const uint32_t a1 = w < nwords ? bm1[w] : 0u;
        uint32_t bits = a0 | a1;
        const int c = __popc(bits);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int q = pos + incl - c;
        while (bits) {
            const int bt = __ffs(bits) - 1;
            bits &= bits - 1u;
            const int j = w * 32 + bt;
            const uint32_t mask = ((a0 >> bt) & 1u) | (((a1 >> bt) & 1u) << 1);
            const int vb = min(max(__ldg(p.vbs + j), 0), kCubeTokens);
            list[q++] = (uint32_t)j | ((uint32_t)vb << 16) | (mask << 24);
        }
        pos += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    return pos;
}

// Issues the TMA copies of one cube pair (rows of cubes ja and jb; jb < 0:
// single cube) of tensor `tm` into a 32 KB pair slot.
__device__ __forceinline__ void load_pair(const CUtensorMap* tm, uint32_t dst, uint32_t bar, int row_a, int row_b,
                                          int h, int nchunks, int D, uint64_t policy) {
    mbar_arrive_expect_tx(bar, (uint32_t)((row_b >= 0 ? 2 : 1) * kCubeTokens * D * 2));
    for (int c = 0; c < nchunks; ++c) tma_load_3d(dst + c * kChunkRows128, tm, bar, c * 64, h, row_a, policy);
    if (row_b >= 0)
        for (int c = 0; c < nchunks; ++c)
            tma_load_3d(dst + c * kChunkRows128 + kChunkRows64, tm, bar, c * 64, h, row_b, policy);
}

// Waits (bounded, also after an abort) until the last copy issued into each
// ring slot has landed.  Called by lane 0 of the producer warp.
template <int kSlots>
__device__ __forceinline__ void drain_ring(uint64_t* full, uint32_t issued, unsigned int* err) {
    for (int s = 0; s < kSlots; ++s) {
        if ((uint32_t)s >= issued) continue;
        const uint32_t last = issued - 1 - ((issued - 1 - s) % kSlots);  // last step that used slot s
        mbar_wait_drain_1(smem_u32(&full[s]), (last / kSlots) & 1, err, kWaitLimitNs);
    }
}

// Softmax threads: copy half `hf` of this thread's Q row (or zeros) into TMEM
// Q buffer qb (D/2 elements = D/4 32-bit columns; D = 64 has one half only).
__device__ __forceinline__ void stage_q(const FineParams& p, int u, int row_in_pair, uint32_t t_lane, int hf) {
    int b, h, pair;
    unit_coords(u, p, b, h, pair);
    int i0, i1;
    unit_cubes(p, b, h, pair, i0, i1);
    const int i = (row_in_pair >> 6) ? i1 : i0;
    const int D = p.D;
    const int words = D / 2;  // 32-bit columns of a full row
    uint32_t w[32];
    for (int c0 = hf * 32; c0 < words && c0 < hf * 32 + 32; c0 += 32) {
        if (i >= 0) {
            const size_t row = (size_t)b * p.N * kCubeTokens + (size_t)i * kCubeTokens + (row_in_pair & 63);
            const uint4* src = p.q + (row * p.heads + h) * (size_t)(D / 8) + c0 / 4;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint4 x = __ldg(src + v);
                w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int v = 0; v < 32; ++v) w[v] = 0u;
        }
        tmem_st32(t_lane + kTmemQ + c0, w);
    }
    tmem_wait_st();
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <int kD, bool kGated>
__global__ void __launch_bounds__(kThreads, 1)
    fine_fwd_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    FineParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
    uint32_t* lists = reinterpret_cast<uint32_t*>(smem + kOffList);
    uint32_t* bitmaps = reinterpret_cast<uint32_t*>(smem + kOffBitmap);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort_flag = &ms.abort_flag;

    constexpr int D = kD;
    const int nchunks = D / 64;
    const int s_pad = p.N * kCubeTokens;
    const int my_units = blockIdx.x < p.num_units ? (p.num_units - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(smem_u32(&ms.k_full[s]), 1);
            mbar_init(smem_u32(&ms.k_empty[s]), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(smem_u32(&ms.v_full[s]), 1);
            mbar_init(smem_u32(&ms.v_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&ms.s_full[s]), 1);
            mbar_init(smem_u32(&ms.s_free[s]), kSoftmaxWarps);
            mbar_init(smem_u32(&ms.list_full[s]), 1);
            mbar_init(smem_u32(&ms.list_empty[s]), 1 + 1 + kSoftmaxWarps);  // V producer, MMA, softmax warps
        }
        mbar_init(smem_u32(&ms.p_full), kSoftmaxWarps);
        mbar_init(smem_u32(&ms.pv_done), 1);
        mbar_init(smem_u32(&ms.q_full), kSoftmaxWarps);
        mbar_init(smem_u32(&ms.q_empty), 1);
        mbar_init(smem_u32(&ms.drain[0]), 1);
        mbar_init(smem_u32(&ms.drain[1]), 1);
        ms.abort_flag = 0;
        fence_barrier_init();
    }
    // Zero the K/V rings once: a single-cube step's MMA reads rows no copy wrote.
    {
        int4* z = reinterpret_cast<int4*>(smem + kOffK);
        const int n16 = (kKStages + kVStages) * kPairBytes / 16;
        for (int e = threadIdx.x; e < n16; e += kThreads) z[e] = make_int4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ms.tmem_base), 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;

    if (warp == 0) {
        // ================================ union lists + TMA producer of K
        const uint64_t pol = l2_policy_evict_last();
        uint32_t g = 0;
        bool ok = true;
        for (int ul = 0; ul < my_units && ok; ++ul) {
            const int u = blockIdx.x + ul * gridDim.x;
            const int lb = ul & 1;
            if (ul >= 2)
                ok = mbar_wait_bounded(smem_u32(&ms.list_empty[lb]), ((ul >> 1) + 1) & 1, abort_flag, p.err,
                                       kWaitLimitNs);
            if (!ok) break;
            uint32_t* list = lists + lb * kMaxUnion;
            const int count = build_union(p, u, list, bitmaps, bitmaps + kBitmapWords, lane);
            if (lane == 0) {
                ms.list_count[lb] = count;
                mbar_arrive(smem_u32(&ms.list_full[lb]));
            }
            int b, h, pair;
            unit_coords(u, p, b, h, pair);
            const int nst = (count + 1) >> 1;
            for (int t = 0; t < nst; ++t, ++g) {
                const int slot = g % kKStages;
                if (g >= (uint32_t)kKStages) {
                    ok = mbar_wait_bounded(smem_u32(&ms.k_empty[slot]), ((g / kKStages) + 1) & 1, abort_flag,
                                           p.err, kWaitLimitNs);
                    if (!ok) break;
                }
                if (lane == 0) {
                    const int ra = b * s_pad + entry_cube(list[2 * t]) * kCubeTokens;
                    const int rb = 2 * t + 1 < count ? b * s_pad + entry_cube(list[2 * t + 1]) * kCubeTokens : -1;
                    load_pair(&tm_k, sbase + kOffK + slot * kPairBytes, smem_u32(&ms.k_full[slot]), ra, rb, h,
                              nchunks, D, pol);
                }
                __syncwarp();
            }
        }
        if (lane == 0) drain_ring<kKStages>(ms.k_full, g, p.err);
        __syncwarp();
    } else if (warp == 2) {
        // ========================================== TMA producer of V
        const uint64_t pol = l2_policy_evict_last();
        uint32_t g = 0;
        bool ok = true;
        for (int ul = 0; ul < my_units && ok; ++ul) {
            const int u = blockIdx.x + ul * gridDim.x;
            const int lb = ul & 1;
            ok = mbar_wait_bounded(smem_u32(&ms.list_full[lb]), (ul >> 1) & 1, abort_flag, p.err, kWaitLimitNs);
            if (!ok) break;
            const uint32_t* list = lists + lb * kMaxUnion;
            const int count = ms.list_count[lb];
            int b, h, pair;
            unit_coords(u, p, b, h, pair);
            const int nst = (count + 1) >> 1;
            for (int t = 0; t < nst; ++t, ++g) {
                const int slot = g % kVStages;
                if (g >= (uint32_t)kVStages) {
                    ok = mbar_wait_bounded(smem_u32(&ms.v_empty[slot]), ((g / kVStages) + 1) & 1, abort_flag,
                                           p.err, kWaitLimitNs);
                    if (!ok) break;
                }
                if (lane == 0) {
                    const int ra = b * s_pad + entry_cube(list[2 * t]) * kCubeTokens;
                    const int rb = 2 * t + 1 < count ? b * s_pad + entry_cube(list[2 * t + 1]) * kCubeTokens : -1;
                    load_pair(&tm_v, sbase + kOffV + slot * kPairBytes, smem_u32(&ms.v_full[slot]), ra, rb, h,
                              nchunks, D, pol);
                }
                __syncwarp();
            }
            if (lane == 0) mbar_arrive(smem_u32(&ms.list_empty[lb]));
        }
        if (lane == 0) drain_ring<kVStages>(ms.v_full, g, p.err);
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ============================================================ MMA issuers
        // Two warps issue MMAs, each warp-wide with lane 0 issuing and
        // committing: warp 1 the QK stream, warp 3 the PV stream.  The streams
        // touch disjoint TMEM (S vs P and O) and are ordered only through the
        // softmax: QK(g) writes S buffer g & 1 once the softmax has loaded
        // S(g - 2) from it (so QK runs up to two steps ahead of the softmax),
        // and PV(g) reads P(g), which the softmax writes once PV(g - 1) has
        // completed.  Descriptors are precomputed; each MMA adds a constant to
        // the start-address field of the low word (no carry: shared addresses
        // are below 256 KB).
        if (my_units > 0) {
            const uint32_t hi = (uint32_t)(smem_desc_sw128(0, 16, 1024) >> 32);  // SBO, version, swizzle
            bool ok = true;
            // Count of the list of local unit ul (waits for the list), warp-uniform.
            auto list_count = [&](int ul) -> int {
                if (!mbar_wait_bounded(smem_u32(&ms.list_full[ul & 1]), (ul >> 1) & 1, abort_flag, p.err,
                                       kWaitLimitNs))
                    return -1;
                return __shfl_sync(0xffffffffu, ms.list_count[ul & 1], 0);
            };
            if (warp == 1) {
                const uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0, 0);
                const uint32_t lo_k = (uint32_t)smem_desc_sw128(sbase + kOffK, 16, 1024);
                constexpr int ksteps_qk = D / 16;
                uint32_t gq = 0;  // QK step (global)
                for (int ul = 0; ul < my_units && ok; ++ul) {
                    const int cnt = list_count(ul);
                    if (cnt < 0) break;
                    const int nst = (cnt + 1) >> 1;
                    ok = mbar_wait_bounded(smem_u32(&ms.q_full), ul & 1, abort_flag, p.err, kWaitLimitNs);
                    for (int t = 0; t < nst && ok; ++t, ++gq) {
                        if (gq >= 2)
                            ok = mbar_wait_bounded(smem_u32(&ms.s_free[gq & 1]), ((gq >> 1) + 1) & 1, abort_flag,
                                                   p.err, kWaitLimitNs);
                        const int slot = gq % kKStages;
                        if (ok)
                            ok = mbar_wait_bounded(smem_u32(&ms.k_full[slot]), (gq / kKStages) & 1, abort_flag,
                                                   p.err, kWaitLimitNs);
                        if (!ok) break;
                        const uint32_t b0 = lo_k + ((uint32_t)(slot * kPairBytes) >> 4);
                        const uint32_t a0 = tmem + kTmemQ;
                        const uint32_t d_tmem = tmem + kTmemS + (gq & 1) * 128;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < ksteps_qk; ++kk)
                            mma_ts_warp(d_tmem, a0 + kk * 8,
                                        b0 + (((kk >> 2) * kChunkRows128 + (kk & 3) * 32) >> 4), hi, idesc_qk,
                                        kk > 0);
                        mma_commit_warp(smem_u32(&ms.s_full[gq & 1]));
                        mma_commit_warp(smem_u32(&ms.k_empty[slot]));
                    }
                    if (ok) mma_commit_warp(smem_u32(&ms.q_empty));  // the unit's Q is no longer read
                }
            } else {
                const uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
                const uint32_t lo_v = (uint32_t)smem_desc_sw128(sbase + kOffV, kChunkRows128, 1024);
                uint32_t g = 0;  // PV step (global)
                for (int ul = 0; ul < my_units && ok; ++ul) {
                    const int cnt = list_count(ul);
                    if (cnt < 0) break;
                    const int nst = (cnt + 1) >> 1;
                    for (int t = 0; t < nst && ok; ++t, ++g) {
                        const int slot = g % kVStages;
                        ok = mbar_wait_bounded(smem_u32(&ms.p_full), g & 1, abort_flag, p.err, kWaitLimitNs) &&
                             mbar_wait_bounded(smem_u32(&ms.v_full[slot]), (g / kVStages) & 1, abort_flag, p.err,
                                               kWaitLimitNs);
                        if (!ok) break;
                        const uint32_t b0 = lo_v + ((uint32_t)(slot * kPairBytes) >> 4);
                        const uint32_t a0 = tmem + kTmemP;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ts_warp(tmem + kTmemO, a0 + kk * 8, b0 + ((kk * 2048) >> 4), hi, idesc_pv,
                                        (t > 0 || kk > 0));
                        if (2 * t + 1 < cnt) {  // the second cube of the step (a single-cube step has 64 keys)
#pragma unroll
                            for (int kk = 4; kk < 8; ++kk)
                                mma_ts_warp(tmem + kTmemO, a0 + kk * 8, b0 + ((kk * 2048) >> 4), hi, idesc_pv, 1u);
                        }
                        mma_commit_warp(smem_u32(&ms.pv_done));
                        mma_commit_warp(smem_u32(&ms.v_empty[slot]));
                    }
                    // This issuer is done with the unit's list.
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ms.list_empty[ul & 1]));
                }
            }
            // Drain: every MMA this warp issued completes before TMEM is released.
            mma_commit_warp(smem_u32(&ms.drain[warp == 1 ? 0 : 1]));
            if (lane == 0) mbar_wait_drain_1(smem_u32(&ms.drain[warp == 1 ? 0 : 1]), 0, p.err, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= kFirstSoftmaxWarp) {
        // ============================================================ softmax
        const int sw = warp - kFirstSoftmaxWarp;  // 0..7
        const int quarter = warp & 3;             // TMEM lane quarter
        const int hf = sw >> 2;                   // key half of the step: cube 2t + hf
        const int r = quarter * 32 + lane;        // query row of the pair (0..127)
        const uint32_t my_bit = 1u << (r >> 6);   // membership bit of this row's cube
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const int dh = D / 2;                     // O columns this thread owns: [hf * dh, hf * dh + dh)
        const float c2 = p.scale_log2;
        const float ninf = -INFINITY;
        bool ok = true;
        uint32_t g = 0;
        if (my_units > 0) {
            stage_q(p, blockIdx.x, r, t_lane, hf);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ms.q_full));
        }
        for (int ul = 0; ul < my_units; ++ul) {
            const int u = blockIdx.x + ul * gridDim.x;
            const int lb = ul & 1;
            if constexpr (kGated) {
                // The epilogue reads this thread's half row of both gates (one
                // 128-byte line each for D = 128): start bringing them into L2.
                int b, h, pair;
                unit_coords(u, p, b, h, pair);
                int i0, i1;
                unit_cubes(p, b, h, pair, i0, i1);
                const int i = (r >> 6) ? i1 : i0;
                if (i >= 0) {
                    const size_t gi = ((size_t)(b * s_pad + i * kCubeTokens + (r & 63)) * p.heads + h) *
                                          (size_t)(D / 8) + hf * (dh / 8);
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.gc + gi));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.gf + gi));
                }
            }
            if (ok) ok = mbar_wait_bounded(smem_u32(&ms.list_full[lb]), (ul >> 1) & 1, abort_flag, p.err,
                                           kWaitLimitNs);
            const uint32_t* list = lists + lb * kMaxUnion;
            const int count = ok ? ms.list_count[lb] : 0;
            const int nst = (count + 1) >> 1;
            // Stages the next unit's Q once this unit's Q is no longer read (its
            // last QK has completed: after S of its last step, or at once for a
            // unit with an empty union, which issues no QK).
            auto stage_next_q = [&]() {
                if (ul + 1 < my_units && ok) {
                    ok = mbar_wait_bounded(smem_u32(&ms.q_empty), ul & 1, abort_flag, p.err, kWaitLimitNs);
                    if (ok) {
                        tc_fence_after();
                        stage_q(p, u + gridDim.x, r, t_lane, hf);
                        tc_fence_before();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ms.q_full));
                }
            };
            if (nst == 0) stage_next_q();
            float m = ninf, l = 0.f;
            for (int t = 0; t < nst; ++t, ++g) {
                const int e = 2 * t + hf;
                const uint32_t ent = e < count ? list[e] : 0u;
                const bool mem = (entry_mask(ent) & my_bit) != 0;  // warp-uniform (row cube)
                const int vb = entry_vbs(ent);
                const uint32_t sc = kTmemS + (g & 1) * 128;
                if (ok) ok = mbar_wait_bounded(smem_u32(&ms.s_full[g & 1]), (g >> 1) & 1, abort_flag, p.err,
                                               kWaitLimitNs);
                tc_fence_after();
                if (t + 1 == nst) stage_next_q();
                float x[64];
                if (ok && mem) {
                    tmem_ld32(t_lane + sc + hf * 64, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
                    tmem_ld32(t_lane + sc + hf * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
                    tmem_wait_ld();
                }
                // S(g) is in registers: its buffer may take S(g + 2).
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ms.s_free[g & 1]));
                // Raw row maximum of this half (keys past vbs are -inf), then log2 units.
                float lmax = ninf;
                if (ok && mem) {
                    if (vb < kCubeTokens) {
#pragma unroll
                        for (int c = 0; c < 64; ++c) x[c] = c < vb ? x[c] : ninf;
                    }
                    float mm[22];
#pragma unroll
                    for (int j = 0; j < 21; ++j) mm[j] = max3(x[3 * j], x[3 * j + 1], x[3 * j + 2]);
                    mm[21] = x[63];
#pragma unroll
                    for (int j = 0; j < 7; ++j) mm[j] = max3(mm[3 * j], mm[3 * j + 1], mm[3 * j + 2]);
                    lmax = c2 * max3(max3(mm[0], mm[1], mm[2]), max3(mm[3], mm[4], mm[5]), fmaxf(mm[6], mm[21]));
                }
                // Row max over both key cubes of the step (thread pair exchange).
                ms.xmax[g & 1][hf][r] = lmax;
                named_sync(1 + quarter, 64);
                const float rmax = fmaxf(lmax, ms.xmax[g & 1][hf ^ 1][r]);
                // Lazy running max: rescale O and l only on a jump > threshold
                // (both threads of the row take the same decision).
                float alpha = 1.f;
                if (rmax > m + kRescaleThreshold) {
                    alpha = (m == ninf) ? 0.f : ex2_approx(m - rmax);
                    m = rmax;
                    l *= alpha;
                }
                // P = exp2(x c2 - m) as bf16 pairs (this half's 32 P columns).
                uint32_t pk[32];
                if (ok && mem) {
                    const float mb = (m == ninf) ? 0.f : m;
                    // Packed two-wide fp32 FMA and add (the same roundings as the
                    // scalar forms, half the instructions).
                    const float2 c2v = make_float2(c2, c2), nmb = make_float2(-mb, -mb);
                    float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < 64; c += 4) {
                        const float2 a01 = __ffma2_rn(make_float2(x[c], x[c + 1]), c2v, nmb);
                        const float2 a23 = __ffma2_rn(make_float2(x[c + 2], x[c + 3]), c2v, nmb);
                        const float p0 = ex2_approx(a01.x), p1 = ex2_approx(a01.y);
                        const float p2 = ex2_approx(a23.x), p3 = ex2_approx(a23.y);
                        s01 = __fadd2_rn(s01, make_float2(p0, p1));
                        s23 = __fadd2_rn(s23, make_float2(p2, p3));
                        pk[c >> 1] = pack_bf16x2(p0, p1);
                        pk[(c >> 1) + 1] = pack_bf16x2(p2, p3);
                    }
                    l += (s01.x + s01.y) + (s23.x + s23.y);
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) pk[c] = 0u;
                }
                // PV(g - 1) has read the P columns and finished adding into O.
                if (g > 0 && ok)
                    ok = mbar_wait_bounded(smem_u32(&ms.pv_done), (g - 1) & 1, abort_flag, p.err, kWaitLimitNs);
                tc_fence_after();
                if (ok) tmem_st32(t_lane + kTmemP + hf * 32, pk);
                if (ok && t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // Rescale this thread's half of the O row.
#pragma unroll 1
                    for (int c0 = hf * dh; c0 < hf * dh + dh; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + kTmemO + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
                        tmem_st32(t_lane + kTmemO + c0, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ms.p_full));
            }
            if (lane == 0) mbar_arrive(smem_u32(&ms.list_empty[lb]));
            // ------------------------------------------------ unit epilogue
            int b, h, pair;
            unit_coords(u, p, b, h, pair);
            int i0, i1;
            unit_cubes(p, b, h, pair, i0, i1);
            const int i = (r >> 6) ? i1 : i0;
            ms.xsum[hf][r] = l;
            named_sync(1 + quarter, 64);
            const float lt = l + ms.xsum[hf ^ 1][r];
            const uint32_t gl = g - 1;  // last step of the unit
            // An empty union issued no PV: O holds nothing of this unit, write zeros.
            if (ok && nst > 0) ok = mbar_wait_bounded(smem_u32(&ms.pv_done), gl & 1, abort_flag, p.err, kWaitLimitNs);
            if (ok) {
                tc_fence_after();
                const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
                const size_t row = (size_t)b * s_pad + (size_t)i * kCubeTokens + (r & 63);
                uint4* dst = reinterpret_cast<uint4*>(p.out) + (row * p.heads + h) * (size_t)(D / 8);
                for (int c0 = hf * dh; c0 < hf * dh + dh; c0 += 32) {
                    uint32_t o[32];
                    if (nst > 0) {
                        tmem_ld32(t_lane + kTmemO + c0, o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int q = 0; q < 32; ++q) o[q] = 0u;
                    }
                    if (kGated && i >= 0) {
                        // Gated sum with the coarse-stage output of the row's cube.  All
                        // of the chunk's gate and coarse values are loaded before the
                        // first store (the stores could alias them for the compiler).
                        const float4* ocr = reinterpret_cast<const float4*>(
                            p.oc + (((size_t)b * p.heads + h) * p.N + i) * D + c0);
                        const size_t gi = (row * p.heads + h) * (size_t)(D / 8) + c0 / 8;
                        uint4 gcv[4], gfv[4];
                        float4 cv4[8];
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            gcv[v] = __ldcs(p.gc + gi + v);
                            gfv[v] = __ldcs(p.gf + gi + v);
                        }
#pragma unroll
                        for (int v = 0; v < 8; ++v) cv4[v] = __ldg(ocr + v);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const float cv[8] = {cv4[2 * v].x, cv4[2 * v].y, cv4[2 * v].z, cv4[2 * v].w,
                                                 cv4[2 * v + 1].x, cv4[2 * v + 1].y, cv4[2 * v + 1].z,
                                                 cv4[2 * v + 1].w};
                            const uint32_t gcw[4] = {gcv[v].x, gcv[v].y, gcv[v].z, gcv[v].w};
                            const uint32_t gfw[4] = {gfv[v].x, gfv[v].y, gfv[v].z, gfv[v].w};
                            uint32_t pw[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float f0 = __uint_as_float(o[8 * v + 2 * e]) * inv_l;
                                const float f1 = __uint_as_float(o[8 * v + 2 * e + 1]) * inv_l;
                                const float r0 = fmaf(__uint_as_float(gcw[e] << 16), cv[2 * e],
                                                      __uint_as_float(gfw[e] << 16) * f0);
                                const float r1 = fmaf(__uint_as_float(gcw[e] & 0xFFFF0000u), cv[2 * e + 1],
                                                      __uint_as_float(gfw[e] & 0xFFFF0000u) * f1);
                                pw[e] = pack_bf16x2(r0, r1);
                            }
                            __stcs(dst + c0 / 8 + v, make_uint4(pw[0], pw[1], pw[2], pw[3]));
                        }
                    } else if (i >= 0) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l);
                            w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l);
                            w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l);
                            w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l);
                            __stcs(dst + c0 / 8 + v, w);
                        }
                    }
                }
                if (p.lse && i >= 0 && hf == 0)
                    p.lse[((size_t)b * p.heads + h) * s_pad + (size_t)i * kCubeTokens + (r & 63)] =
                        lt > 0.f ? (m + __log2f(lt)) * 0.69314718055994531f : ninf;
            }
            tc_fence_before();
            named_sync(1 + quarter, 64);  // xsum is rewritten by the next unit's epilogue
        }
    }

    // ------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
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
int fine_max_topk() { return kMaxTopk; }
int fine_max_cubes() { return kMaxCubes; }

cudaError_t launch_fine(const void* qt, const void* kt, const void* vt, const int32_t* topk_idx,
                        const int32_t* counts, const int32_t* vbs, const uint32_t* pairs, int B, int ncubes,
                        int heads, int D, int topk, float sm_scale, const float* coarse_out, const void* gate_c,
                        const void* gate_f, void* out, float* lse, unsigned int* err, int num_sms,
                        cudaStream_t stream) {
    CUtensorMap mk, mv;
    const int rows = B * ncubes * kCubeTokens;
    if (!make_map(&mk, kt, rows, heads, D, true) || !make_map(&mv, vt, rows, heads, D, true))
        return cudaErrorInvalidValue;
    FineParams p;
    p.topk_idx = topk_idx;
    p.vbs = vbs;
    p.pairs = pairs;
    p.counts = counts;
    p.oc = coarse_out;
    p.gc = static_cast<const uint4*>(gate_c);
    p.gf = static_cast<const uint4*>(gate_f);
    p.q = static_cast<const uint4*>(qt);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.err = err;
    p.B = B;
    p.N = ncubes;
    p.heads = heads;
    p.D = D;
    p.topk = topk;
    p.npairs = (ncubes + 1) / 2;
    p.num_units = B * heads * p.npairs;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    auto kernel = coarse_out ? (D == 64 ? fine_fwd_kernel<64, true> : fine_fwd_kernel<128, true>)
                             : (D == 64 ? fine_fwd_kernel<64, false> : fine_fwd_kernel<128, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    const int grid = p.num_units < num_sms ? p.num_units : num_sms;
    kernel<<<grid, kThreads, kSmemAlloc, stream>>>(mk, mv, p);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace vsa
