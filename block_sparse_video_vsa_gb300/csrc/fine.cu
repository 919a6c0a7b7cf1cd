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
//  * A work unit is a PAIR of query cubes of one (batch, head): 128 query
//    rows, one per TMEM lane.  It walks the sorted union of the two cubes'
//    selected key cubes, two key cubes (128 keys) per step g:
//        S[128 q x 128 keys]  = Q_pair . K_pair(g)^T    (A = Q in TMEM)
//        O_{g&1}[128 q x D]  += P(g) . V_pair(g)        (A = P in TMEM)
//    Both MMAs are M = 128, N = 128 (full tensor-core rate; an M x 64 MMA runs
//    at half rate), and only the B operands (K, V) come from shared memory.
//    Query rows of a cube that did not select a key cube get probability 0
//    for it, so each row attends exactly its own selection.
//  * Two softmax groups of four warps (one thread per query row) take the
//    steps in turn: group 0 the even global steps, group 1 the odd ones.
//    Each group keeps its own running max and sum and accumulates into its
//    own O (O_0, O_1 in TMEM); the two partial results are merged once per
//    unit in the epilogue.  So the two groups' softmax work overlaps, and no
//    row statistics pass between steps of different groups.
//  * Two warps issue the MMAs: one the Q.K^T stream (QK(g) as soon as S is
//    free and K has landed), one the P.V stream (PV(g) as soon as P and V
//    are ready), so the tensor pipe takes each as early as it can.  Ordering
//    between the streams is explicit: per-group barriers report each P.V's
//    completion (the softmax writes P(g) once P.V(g - 1) has read P, and
//    rescales its O once P.V(g - 2) has added into it), and a per-unit
//    barrier reports that every P.V of the unit has completed (epilogue).
//  * Persistent grid, one CTA per SM, units dealt round-robin in head-major
//    order so one head's K/V stays in L2.
//  * Warp roles (384 threads): warp 0 builds each unit's union list (sorted,
//    with membership bits and vbs) and is the TMA producer of K; warp 1 owns
//    TMEM and issues Q.K^T; warp 2 is the TMA producer of V; warp 3 issues
//    P.V; warps 4..7 and 8..11 are the two softmax groups (warp w serves
//    TMEM lane quarter w % 4).  The group that takes the next unit's first
//    step stages that unit's Q into TMEM once the current unit's last Q.K^T
//    has completed.  The first warpgroup hands registers to the softmax
//    warpgroups (setmaxnreg), which hold a step's 128 logits per thread.
//  * TMEM (512 columns): S [0,128); P (bf16 pairs) [128,192); Q [192,256);
//    O_0 [256,384); O_1 [384,512).  The softmax frees S as soon as it has
//    loaded it, so Q.K^T(g + 1) runs while the softmax of step g works.
//  * Running max kept in log2 units; a group's O and sum are rescaled only
//    when a row's max grows by more than kRescaleThreshold, so exp2 arguments
//    stay <= the threshold and logits of any finite size are safe.
//  * Every wait is bounded; a wait that runs out raises a CTA abort flag and
//    the device error word, and each role winds down without deadlock.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "vsa_common.cuh"

namespace vsa {

namespace {

constexpr int kKStages = 3;           // K pair slots (QK operand B)
constexpr int kVStages = 3;           // V pair slots (PV operand B)
constexpr int kGroupWarps = 4;        // softmax warps per group (one per TMEM lane quarter)
constexpr int kFirstSoftmaxWarp = 4;
constexpr int kThreads = (kFirstSoftmaxWarp + 2 * kGroupWarps) * 32;  // 12 warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Registers per thread: the kernel is compiled for kLaunchRegs (the most 384
// threads can have); right after setup the first warpgroup (list builder,
// producers, MMA issuer) gives registers back and the two softmax
// warpgroups take them (setmaxnreg), so a softmax thread can hold a step's
// 128 logits.  The shares add up to the launch's total exactly:
// 128 * kProducerRegs + 256 * kSoftmaxRegs <= 384 * kLaunchRegs (a larger
// sum would leave setmaxnreg.inc waiting forever); the launcher checks that
// the kernel was compiled with exactly kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr int kProducerRegs = 72;
constexpr int kSoftmaxRegs = 216;
static_assert(128 * kProducerRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split exceeds the launch");
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kMaxTopk = 1024;
constexpr int kMaxUnion = 2 * kMaxTopk;
constexpr int kMaxCubes = 8192;
constexpr int kBitmapWords = kMaxCubes / 32;

// TMEM columns.
constexpr int kTmemS = 0;     // S of the current step (128 fp32 columns)
constexpr int kTmemP = 128;   // P: 128 keys as 64 columns of bf16 pairs
constexpr int kTmemQ = 192;   // Q of the current unit: D bf16 as D/2 columns of pairs
constexpr int kTmemO0 = 256;  // O of group 0 (D columns)
constexpr int kTmemO1 = 384;  // O of group 1

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
    uint64_t s_full[2];   // per softmax group: S of the group's next step is ready
    uint64_t s_free;      // S has been loaded into registers
    uint64_t p_full;      // P (and any O rescale) of the step is in TMEM
    uint64_t pv_grp[2];   // per softmax group: P.V of the group's step has completed
    uint64_t unit_done;   // every P.V of the unit has completed
    uint64_t q_full;      // the unit's Q is in TMEM
    uint64_t q_empty;     // the unit's Q.K^T MMAs have completed
    uint64_t o_free;      // the unit's O_0 and O_1 have been read by the epilogue
    uint64_t list_full[2];
    uint64_t list_empty[2];
    uint64_t drain[2];    // per MMA-issuing warp
    int list_count[2];
    int list_unit[2];     // dynamic schedule: the list's unit, or -1: no more units
    int list_next[2];     // dynamic schedule: the unit after it (whose Q the stager stages), or -1
    float xm[2][2][128];  // [unit parity][group][row]: running max at the unit's end
    float xl[2][2][128];  // [unit parity][group][row]: sum at the unit's end
    float xt[2][2][128];  // [unit parity][group][row]: exact row maximum (log2 units)
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
    const uint4* q;      // q rows (for staging Q into TMEM): tiled, or raster when tokens > 0
    const float* oc;     // coarse-stage output [B * heads][N][D], or null: no gated combine
    const uint4* gc;     // gates of the coarse and fine terms, bf16 in the layout of out
    const uint4* gf;
    __nv_bfloat16* out;
    float* lse;
    float* max_prob;     // [B * heads][S_pad] largest softmax weight of each row, or null
    unsigned int* err;
    int B, N, heads, D, topk;
    int npairs;          // ceil(N / 2)
    int num_units;       // B * heads * npairs
    int slot;            // dynamic schedule: this launch's unit counter (g_unit_next[slot])
    float scale_log2;    // sm_scale * log2(e)
    // Raster mode (tokens > 0): q is read and out written in raster token
    // order [B, tokens, heads, D] of a T x H x W grid (nh x nw cubes per
    // frame layer); lse stays cube-major.
    long long tokens;
    int gT, gH, gW, gnh, gnw;
};

// Raster token of slot s of cube c (the real tokens of the cube's clipped
// 4 x 4 x 4 sub-box fill its first slots in (t, h, w) order), or -1 for a
// padding slot.
__device__ __forceinline__ int raster_token(const FineParams& p, int c, int s) {
    const int cw = c % p.gnw;
    const int c1 = c / p.gnw;
    const int ch = c1 % p.gnh;
    const int ct = c1 / p.gnh;
    const int et = min(4, p.gT - 4 * ct), eh = min(4, p.gH - 4 * ch), ew = min(4, p.gW - 4 * cw);
    const int hw = eh * ew;
    if (s >= et * hw) return -1;
    const int lt = s / hw;
    const int rem = s - lt * hw;
    const int lh = rem / ew;
    return ((4 * ct + lt) * p.gH + 4 * ch + lh) * p.gW + 4 * cw + (rem - lh * ew);
}

// Global row (token of the [B, S, heads, D] layout) of slot s of cube i in
// batch b: tiled, or raster (-1 for a padding slot, which has no raster row).
__device__ __forceinline__ long long token_row(const FineParams& p, int b, int i, int s) {
    if (p.tokens > 0) {
        const int n = raster_token(p, i, s);
        return n < 0 ? -1 : (long long)b * p.tokens + n;
    }
    return ((long long)b * p.N + i) * kCubeTokens + s;
}

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

// Query cube of row r (0..127) of unit u, or -1.
__device__ __forceinline__ int row_cube(const FineParams& p, int u, int r, int& b, int& h) {
    int pair, i0, i1;
    unit_coords(u, p, b, h, pair);
    unit_cubes(p, b, h, pair, i0, i1);
    return (r >> 6) ? i1 : i0;
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

// Softmax thread of row r: copies its whole Q row of unit u (or zeros) into
// the TMEM Q columns of its lane.
template <int kD>
__device__ __forceinline__ void stage_q(const FineParams& p, int u, int r, uint32_t t_lane) {
    int b, h;
    const int i = row_cube(p, u, r, b, h);
    const uint4* src = nullptr;
    const long long row = i >= 0 ? token_row(p, b, i, r & 63) : -1;
    if (row >= 0) src = p.q + ((size_t)row * p.heads + h) * (size_t)(kD / 8);
#pragma unroll
    for (int c0 = 0; c0 < kD / 2; c0 += 32) {
        uint32_t w[32];
        if (src) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint4 x = __ldg(src + c0 / 4 + v);
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

// Brings row r's Q row of unit u into L2 ahead of stage_q.
template <int kD>
__device__ __forceinline__ void prefetch_q(const FineParams& p, int u, int r) {
    int b, h;
    const int i = row_cube(p, u, r, b, h);
    if (i < 0) return;
    const long long row = token_row(p, b, i, r & 63);
    if (row < 0) return;
    const uint4* src = p.q + ((size_t)row * p.heads + h) * (size_t)(kD / 8);
#pragma unroll
    for (int c = 0; c < kD * 2; c += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + c / 16));
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Maximum of x[0..63]: four running three-input max chains (few temporaries
// beside the 128 live logits of the step).
__device__ __forceinline__ float max64(const float* x) {
    float a[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
    for (int c = 4; c < 60; c += 8)  // keys 4 .. 59
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = max3(a[j], x[c + j], x[c + 4 + j]);
#pragma unroll
    for (int j = 0; j < 4; ++j) a[j] = fmaxf(a[j], x[60 + j]);  // keys 60 .. 63
    return fmaxf(max3(a[0], a[1], a[2]), a[3]);
}

// p = exp2(x * c2 - mb) for 64 keys, packed as 32 bf16 pairs; adds the
// fp32 values to l.  Packed two-wide fp32 FMA and add (the same roundings as
// the scalar forms, half the instructions).
__device__ __forceinline__ void exp64(const float* x, float c2, float mb, uint32_t* pk, float& l) {
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
}

// Unit schedules.  Static: CTA c takes units c, c + grid, c + 2 grid, ...
// Dynamic (for rows of variable length, where the static deal leaves SMs
// idle): CTA c starts with unit c, and warp 0 claims each further unit as
// gridDim.x + atomicAdd(&g_unit_next[slot], 1), one unit ahead (the softmax
// group that stages the next unit's Q needs its index), so CTAs that drew
// short units take more of them; lists then carry their unit and the next
// one, and a list with unit -1 ends every role's loop.  Each launch takes its
// own slot (a host-side ticket modulo kUnitSlots: concurrent launches on
// other streams use other slots); the last CTA to finish puts the slot's
// counters back to zero for the launch that takes it next.
constexpr int kUnitSlots = 256;
__device__ unsigned int g_unit_next[kUnitSlots];
__device__ unsigned int g_cta_done[kUnitSlots];

// A claim is drawn by lane 0 (claim_draw) and read by the warp later
// (claim_take), so the atomic's round trip overlaps other work.
__device__ __forceinline__ unsigned int claim_draw(const FineParams& p, int lane) {
    return lane == 0 ? atomicAdd(&g_unit_next[p.slot], 1u) : 0u;
}
__device__ __forceinline__ int claim_take(const FineParams& p, unsigned int drawn) {
    const int v = (int)(gridDim.x + __shfl_sync(0xffffffffu, drawn, 0));
    return v < p.num_units ? v : -1;
}

template <int kD, bool kGated, bool kPeak, bool kDyn>
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
    // Loop bound of every role: the static schedule's unit count, or for the
    // dynamic one a bound the end list always cuts short.  (Written as bounded
    // loops under a guard: open-ended loops compiled to a form that took 5-8%
    // longer at the Wan2.2 shape, measured same-box.)
    const int bound = kDyn ? p.num_units : my_units;

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
            mbar_init(smem_u32(&ms.list_full[s]), 1);
            mbar_init(smem_u32(&ms.list_empty[s]), 1 + 2 + 2 * kGroupWarps);  // V producer, MMA warps, softmax
        }
        mbar_init(smem_u32(&ms.s_free), kGroupWarps);
        mbar_init(smem_u32(&ms.p_full), kGroupWarps);
        mbar_init(smem_u32(&ms.pv_grp[0]), 1);
        mbar_init(smem_u32(&ms.pv_grp[1]), 1);
        mbar_init(smem_u32(&ms.unit_done), 1);
        mbar_init(smem_u32(&ms.q_full), kGroupWarps);
        mbar_init(smem_u32(&ms.q_empty), 1);
        mbar_init(smem_u32(&ms.o_free), 2 * kGroupWarps);
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

    if (warp < kFirstSoftmaxWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    if (warp == 0) {
        // ================================ union lists + TMA producer of K
        const uint64_t pol = l2_policy_evict_last();
        uint32_t g = 0;
        bool ok = true;
        int u_dyn = blockIdx.x;  // dynamic: grid <= units, so every CTA has a first unit
        int u_next = kDyn ? claim_take(p, claim_draw(p, lane)) : -1;
        for (int ul = 0; ul < (kDyn ? bound + 1 : bound) && ok; ++ul) {
            const int u = kDyn ? u_dyn : (int)(blockIdx.x + ul * gridDim.x);
            const int lb = ul & 1;
            if (ul >= 2)
                ok = mbar_wait_bounded(smem_u32(&ms.list_empty[lb]), ((ul >> 1) + 1) & 1, abort_flag, p.err,
                                       kWaitLimitNs);
            if (!ok) break;
            unsigned int drawn = 0u;
            if constexpr (kDyn) {
                if (u < 0) {  // no unit left: a list with unit -1 tells every role to stop
                    if (lane == 0) {
                        ms.list_count[lb] = 0;
                        ms.list_unit[lb] = -1;
                        ms.list_next[lb] = -1;
                        mbar_arrive(smem_u32(&ms.list_full[lb]));
                    }
                    break;
                }
                // The unit after u_next, drawn now and read after this unit's loads.
                if (u_next >= 0) drawn = claim_draw(p, lane);
            }
            uint32_t* list = lists + lb * kMaxUnion;
            const int count = build_union(p, u, list, bitmaps, bitmaps + kBitmapWords, lane);
            if (lane == 0) {
                ms.list_count[lb] = count;
                if constexpr (kDyn) {
                    ms.list_unit[lb] = u;
                    ms.list_next[lb] = u_next;
                }
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
            if constexpr (kDyn) {
                u_dyn = u_next;
                u_next = u_dyn >= 0 ? claim_take(p, drawn) : -1;
            }
        }
        if (lane == 0) drain_ring<kKStages>(ms.k_full, g, p.err);
        __syncwarp();
    } else if (warp == 2) {
        // ========================================== TMA producer of V
        const uint64_t pol = l2_policy_evict_last();
        uint32_t g = 0;
        bool ok = true;
        for (int ul = 0; ul < bound && ok; ++ul) {
            const int lb = ul & 1;
            ok = mbar_wait_bounded(smem_u32(&ms.list_full[lb]), (ul >> 1) & 1, abort_flag, p.err, kWaitLimitNs);
            if (!ok) break;
            const int u = kDyn ? ms.list_unit[lb] : (int)(blockIdx.x + ul * gridDim.x);
            if (kDyn && u < 0) break;
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
        // Two warps issue MMAs: warp 1 the Q.K^T stream (QK(g) as soon as S is
        // free and K has landed), warp 3 the P.V stream (PV(g) as soon as P
        // and V are ready), so the tensor pipe takes each as early as it can.
        // Each runs its loop as a whole warp and lets lane 0 issue and commit
        // (always the same thread, so its commits cover all of its MMAs).
        // The streams touch disjoint TMEM (S vs P and O) and are ordered only
        // through the softmax's barriers.  Descriptors are precomputed; each
        // MMA adds a constant to the start-address field of the low word (no
        // carry: shared addresses are below 256 KB).
        if (bound > 0) {
            const uint32_t hi = (uint32_t)(smem_desc_sw128(0, 16, 1024) >> 32);  // SBO, version, swizzle
            bool ok = true;
            // Count of the list of local unit ul (waits for the list), warp-uniform.
            auto list_count = [&](int ul) -> int {
                if (!mbar_wait_bounded(smem_u32(&ms.list_full[ul & 1]), (ul >> 1) & 1, abort_flag, p.err,
                                       kWaitLimitNs))
                    return -1;
                if constexpr (kDyn) {  // -1 also when no unit is left
                    if (__shfl_sync(0xffffffffu, ms.list_unit[ul & 1], 0) < 0) return -1;
                }
                return __shfl_sync(0xffffffffu, ms.list_count[ul & 1], 0);
            };
            uint32_t g = 0;  // global step at the start of the unit
            if (warp == 1) {
                const uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0, 0);
                const uint32_t lo_k = (uint32_t)smem_desc_sw128(sbase + kOffK, 16, 1024);
                constexpr int ksteps_qk = D / 16;
                for (int ul = 0; ul < bound && ok; ++ul) {
                    const int cnt = list_count(ul);
                    if (cnt < 0) break;
                    const int nst = (cnt + 1) >> 1;
                    ok = mbar_wait_bounded(smem_u32(&ms.q_full), ul & 1, abort_flag, p.err, kWaitLimitNs);
                    for (int t = 0; t < nst && ok; ++t) {
                        const uint32_t gs = g + t;
                        if (gs >= 1)  // S of the previous step is in registers
                            ok = mbar_wait_bounded(smem_u32(&ms.s_free), (gs - 1) & 1, abort_flag, p.err,
                                                   kWaitLimitNs);
                        const int slot = gs % kKStages;
                        if (ok)
                            ok = mbar_wait_bounded(smem_u32(&ms.k_full[slot]), (gs / kKStages) & 1, abort_flag,
                                                   p.err, kWaitLimitNs);
                        if (!ok) break;
                        const uint32_t b0 = lo_k + ((uint32_t)(slot * kPairBytes) >> 4);
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < ksteps_qk; ++kk)
                            mma_ts_warp(tmem + kTmemS, tmem + kTmemQ + kk * 8,
                                        b0 + (((kk >> 2) * kChunkRows128 + (kk & 3) * 32) >> 4), hi, idesc_qk,
                                        kk > 0);
                        mma_commit_warp(smem_u32(&ms.s_full[gs & 1]));
                        mma_commit_warp(smem_u32(&ms.k_empty[slot]));
                    }
                    if (!ok) break;
                    mma_commit_warp(smem_u32(&ms.q_empty));  // the unit's Q is no longer read
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ms.list_empty[ul & 1]));
                    g += nst;
                }
            } else {
                const uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
                const uint32_t lo_v = (uint32_t)smem_desc_sw128(sbase + kOffV, kChunkRows128, 1024);
                for (int ul = 0; ul < bound && ok; ++ul) {
                    const int cnt = list_count(ul);
                    if (cnt < 0) break;
                    const int nst = (cnt + 1) >> 1;
                    // The unit's O_0 and O_1 start over once the previous unit's
                    // epilogue has read them (an empty unit waits too, so that
                    // unit_done never runs two phases ahead of an epilogue).
                    if (ul >= 1)
                        ok = mbar_wait_bounded(smem_u32(&ms.o_free), (ul - 1) & 1, abort_flag, p.err, kWaitLimitNs);
                    for (int t = 0; t < nst && ok; ++t) {
                        const uint32_t gs = g + t;
                        const int slot = gs % kVStages;
                        ok = mbar_wait_bounded(smem_u32(&ms.p_full), gs & 1, abort_flag, p.err, kWaitLimitNs) &&
                             mbar_wait_bounded(smem_u32(&ms.v_full[slot]), (gs / kVStages) & 1, abort_flag, p.err,
                                               kWaitLimitNs);
                        if (!ok) break;
                        const uint32_t b0 = lo_v + ((uint32_t)(slot * kPairBytes) >> 4);
                        const uint32_t d_tmem = tmem + ((gs & 1) ? kTmemO1 : kTmemO0);
                        const uint32_t acc = t >= 2 ? 1u : 0u;  // a group's first step of the unit overwrites its O
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ts_warp(d_tmem, tmem + kTmemP + kk * 8, b0 + ((kk * 2048) >> 4), hi, idesc_pv,
                                        acc | (kk > 0 ? 1u : 0u));
                        if (2 * t + 1 < cnt) {  // the second cube of the step (a single-cube step has 64 keys)
#pragma unroll
                            for (int kk = 4; kk < 8; ++kk)
                                mma_ts_warp(d_tmem, tmem + kTmemP + kk * 8, b0 + ((kk * 2048) >> 4), hi, idesc_pv,
                                            1u);
                        }
                        mma_commit_warp(smem_u32(&ms.pv_grp[gs & 1]));
                        mma_commit_warp(smem_u32(&ms.v_empty[slot]));
                    }
                    if (!ok) break;
                    mma_commit_warp(smem_u32(&ms.unit_done));  // every P.V of the unit
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ms.list_empty[ul & 1]));
                    g += nst;
                }
            }
            // Drain: every MMA this warp issued completes before TMEM is released.
            const uint32_t drain = smem_u32(&ms.drain[warp == 1 ? 0 : 1]);
            mma_commit_warp(drain);
            if (lane == 0) mbar_wait_drain_1(drain, 0, p.err, kWaitLimitNs);
        }
        __syncwarp();
    }
    } else {
        // ============================================================ softmax
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
        const int G = (warp - kFirstSoftmaxWarp) / kGroupWarps;  // steps g with g % 2 == G
        const int quarter = warp & 3;                             // TMEM lane quarter
        const int r = quarter * 32 + lane;                        // query row of the pair (0..127)
        const uint32_t my_bit = 1u << (r >> 6);                   // membership bit of this row's cube
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t o_mine = t_lane + (G ? kTmemO1 : kTmemO0);
        const float c2 = p.scale_log2;
        const float ninf = -INFINITY;
        constexpr int dh = D / 2;  // output columns this thread writes: [G * dh, G * dh + dh)
        bool ok = true;
        uint32_t g = 0;   // global step at the start of the current unit
        uint32_t jg = 0;  // steps this group has taken (phase of s_full[G])
        if (G == 0 && bound > 0) {
            stage_q<D>(p, blockIdx.x, r, t_lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ms.q_full));
        }
#pragma unroll 1
        for (int ul = 0; ul < bound; ++ul) {
            const int lb = ul & 1;
            int u = (int)(blockIdx.x + ul * gridDim.x);
            if constexpr (kDyn) {
                // The unit comes with the list; it is read here and again just
                // before the list buffer is released, not held across the steps.
                if (ok) ok = mbar_wait_bounded(smem_u32(&ms.list_full[lb]), (ul >> 1) & 1, abort_flag, p.err,
                                               kWaitLimitNs);
                if (!ok || ms.list_unit[lb] < 0) break;
                u = ms.list_unit[lb];
            }
            if constexpr (kGated) {
                // The epilogue reads this thread's half row of both gates (one
                // 128-byte line each for D = 128): start bringing them into L2.
                int b, h;
                const int i = row_cube(p, u, r, b, h);
                if (i >= 0) {
                    const size_t gi = ((size_t)(b * s_pad + i * kCubeTokens + (r & 63)) * p.heads + h) *
                                          (size_t)(D / 8) + G * (dh / 8);
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.gc + gi));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.gf + gi));
                }
            }
            if constexpr (!kDyn) {
                if (ok) ok = mbar_wait_bounded(smem_u32(&ms.list_full[lb]), (ul >> 1) & 1, abort_flag, p.err,
                                               kWaitLimitNs);
            }
            const uint32_t* list = lists + lb * kMaxUnion;
            const int count = ok ? ms.list_count[lb] : 0;
            const int nst = (count + 1) >> 1;
            const uint32_t g0 = g;
            // The group that takes the next unit's first step stages its Q.
            const bool stager = (((g0 + nst) & 1) == (uint32_t)G) &&
                                (kDyn ? ms.list_next[lb] >= 0 : ul + 1 < my_units);
            if (stager) prefetch_q<D>(p, kDyn ? ms.list_next[lb] : u + (int)gridDim.x, r);
            float m = ninf, l = 0.f;
            float mx = ninf;  // exact row maximum of this group's steps (m lags it by up to the threshold)
            bool first = true;
#pragma unroll 1
            for (int t = (int)((g0 + G) & 1); t < nst; t += 2) {
                const uint32_t gs = g0 + t;
                const uint32_t e0 = list[2 * t];
                const uint32_t e1 = 2 * t + 1 < count ? list[2 * t + 1] : 0u;
                const bool mem0 = (entry_mask(e0) & my_bit) != 0;  // warp-uniform (row cube)
                const bool mem1 = (entry_mask(e1) & my_bit) != 0;
                const int vb0 = entry_vbs(e0), vb1 = entry_vbs(e1);
                if (ok) ok = mbar_wait_bounded(smem_u32(&ms.s_full[G]), jg & 1, abort_flag, p.err, kWaitLimitNs);
                ++jg;
                tc_fence_after();
                float x[128];
                // All 128 columns are loaded whatever the membership (the
                // unused half is never read; loading it keeps every value
                // defined on every path, which the register allocator needs).
#pragma unroll
                for (int c = 0; c < 128; c += 32)
                    tmem_ld32(t_lane + kTmemS + c, *reinterpret_cast<uint32_t(*)[32]>(&x[c]));
                tmem_wait_ld();
                // S(g) is in registers: the buffer may take S(g + 1).
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ms.s_free));
                // Raw row maximum over this row's keys (keys past vbs are -inf), then log2 units.
                float lmax = ninf;
                if (ok && mem0) {
                    if (vb0 < kCubeTokens) {
#pragma unroll
                        for (int c = 0; c < 64; ++c) x[c] = c < vb0 ? x[c] : ninf;
                    }
                    lmax = max64(x);
                }
                if (ok && mem1) {
                    if (vb1 < kCubeTokens) {
#pragma unroll
                        for (int c = 0; c < 64; ++c) x[64 + c] = c < vb1 ? x[64 + c] : ninf;
                    }
                    lmax = fmaxf(lmax, max64(x + 64));
                }
                lmax *= c2;
                if constexpr (kPeak) mx = fmaxf(mx, lmax);
                // Lazy running max: rescale O and l only on a jump > threshold.
                float alpha = 1.f;
                if (lmax > m + kRescaleThreshold) {
                    alpha = (m == ninf) ? 0.f : ex2_approx(m - lmax);
                    m = lmax;
                    l *= alpha;
                }
                // P = exp2(x c2 - m) as bf16 pairs: keys 0..63 in P columns
                // [0, 32), keys 64..127 in [32, 64).
                uint32_t pk[64];
                const float mb = (m == ninf) ? 0.f : m;
                if (ok && mem0) {
                    exp64(x, c2, mb, pk, l);
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) pk[c] = 0u;
                }
                if (ok && mem1) {
                    exp64(x + 64, c2, mb, pk + 32, l);
                } else {
#pragma unroll
                    for (int c = 32; c < 64; ++c) pk[c] = 0u;
                }
                // P.V(g - 1) (the other group's) has read the P columns.
                if (gs > 0 && ok)
                    ok = mbar_wait_bounded(smem_u32(&ms.pv_grp[G ^ 1]), ((gs - 1) >> 1) & 1, abort_flag, p.err,
                                           kWaitLimitNs);
                tc_fence_after();
                if (ok) {
#pragma unroll
                    for (int c = 0; c < 64; c += 16)
                        tmem_st16(t_lane + kTmemP + c, *reinterpret_cast<uint32_t(*)[16]>(&pk[c]));
                }
                if (ok && !first && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // Rescale this row of the group's O, once P.V(g - 2) -- the
                    // last one into it -- has completed.
                    ok = mbar_wait_bounded(smem_u32(&ms.pv_grp[G]), ((gs - 2) >> 1) & 1, abort_flag, p.err,
                                           kWaitLimitNs);
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(o_mine + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
                        tmem_st32(o_mine + c0, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ms.p_full));
                first = false;
            }
            if (stager) {
                // The unit's Q.K^T MMAs have completed: Q may be overwritten.
                if (ok) ok = mbar_wait_bounded(smem_u32(&ms.q_empty), ul & 1, abort_flag, p.err, kWaitLimitNs);
                if (ok) {
                    tc_fence_after();
                    stage_q<D>(p, kDyn ? *reinterpret_cast<volatile int*>(&ms.list_next[lb]) : u + (int)gridDim.x,
                               r, t_lane);
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ms.q_full));
            }
            if constexpr (kDyn) u = *reinterpret_cast<volatile int*>(&ms.list_unit[lb]);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ms.list_empty[lb]));
            // ------------------------------------------------ unit epilogue
            // Merge the two groups' partial results of each row:
            //   m = max(m_0, m_1), a_k = 2^(m_k - m), l = a_0 l_0 + a_1 l_1,
            //   out = (a_0 O_0 + a_1 O_1) / l, lse = (m + log2 l) ln 2.
            ms.xm[lb][G][r] = m;
            ms.xl[lb][G][r] = l;
            if constexpr (kPeak) ms.xt[lb][G][r] = mx;
            named_sync(1 + quarter, 2 * 32);
            const float mo = ms.xm[lb][G ^ 1][r], lo = ms.xl[lb][G ^ 1][r];
            const float m_true = kPeak ? fmaxf(mx, ms.xt[lb][G ^ 1][r]) : ninf;
            const float m0 = G ? mo : m, l0 = G ? lo : l;
            const float m1 = G ? m : mo, l1 = G ? l : lo;
            // Which group holds the unit's even steps (step t: group (g0 + t) & 1)
            // depends on the steps the CTA ran before the unit (with the dynamic
            // schedule, on the run): the merge takes the even-step group's
            // partial result first, so the bits depend on the unit alone.
            const int ge = (int)(g0 & 1u);  // group of the even steps
            const float m_e = ge ? m1 : m0, l_e = ge ? l1 : l0;
            const float m_o = ge ? m0 : m1, l_o = ge ? l0 : l1;
            // A group that took no step of this unit holds no O for it.
            const bool had_e = nst > 0, had_o = nst >= 2;
            const float mt = fmaxf(m_e, m_o);
            const float a_e = (m_e == ninf) ? 0.f : ex2_approx(m_e - mt);
            const float a_o = (m_o == ninf) ? 0.f : ex2_approx(m_o - mt);
            const float lt = __fmaf_rn(a_e, l_e, __fmul_rn(a_o, l_o));
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            const float s_e = a_e * inv, s_o = a_o * inv;
            const uint32_t o_e = ge ? kTmemO1 : kTmemO0, o_o = ge ? kTmemO0 : kTmemO1;
            int b, h;
            const int i = row_cube(p, u, r, b, h);
            const bool wr = ok && i >= 0;
            const size_t row = wr ? (size_t)b * s_pad + (size_t)i * kCubeTokens + (r & 63) : 0;
            // Output row: the tiled row, or in raster mode the slot's token
            // (padding slots have none and write nothing).
            const long long orow = wr ? token_row(p, b, i, r & 63) : -1;
            const bool wo = orow >= 0;
            uint4* dst = reinterpret_cast<uint4*>(p.out) + ((size_t)(wo ? orow : 0) * p.heads + h) * (size_t)(D / 8) +
                         G * (dh / 8);
            // Gated: the coarse term g_c * O_c of this thread's columns and the
            // fine gate g_f, loaded before the wait for the unit's last P.V.
            float ct[kGated ? dh : 1];
            uint32_t gfw[kGated ? dh / 2 : 1];
            if constexpr (kGated) {
                if (wr) {
                    const float4* ocr = reinterpret_cast<const float4*>(
                        p.oc + (((size_t)b * p.heads + h) * p.N + i) * D + G * dh);
                    const size_t gi = (row * p.heads + h) * (size_t)(D / 8) + G * (dh / 8);
#pragma unroll
                    for (int v = 0; v < dh / 8; ++v) {
                        const uint4 gc = __ldcs(p.gc + gi + v), gf = __ldcs(p.gf + gi + v);
                        const float4 ca = __ldg(ocr + 2 * v), cb = __ldg(ocr + 2 * v + 1);
                        const uint32_t gcw[4] = {gc.x, gc.y, gc.z, gc.w};
                        const float cv[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
                        gfw[4 * v] = gf.x; gfw[4 * v + 1] = gf.y; gfw[4 * v + 2] = gf.z; gfw[4 * v + 3] = gf.w;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            ct[8 * v + 2 * e] = __uint_as_float(gcw[e] << 16) * cv[2 * e];
                            ct[8 * v + 2 * e + 1] = __uint_as_float(gcw[e] & 0xFFFF0000u) * cv[2 * e + 1];
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < dh; ++c) ct[c] = 0.f;
#pragma unroll
                    for (int c = 0; c < dh / 2; ++c) gfw[c] = 0u;
                }
            }
            // Every P.V of the unit has completed.
            if (ok) ok = mbar_wait_bounded(smem_u32(&ms.unit_done), ul & 1, abort_flag, p.err, kWaitLimitNs);
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < dh; c0 += 32) {
                uint32_t oa[32], ob[32];
                // Loaded whatever had_e/had_o say (values of a group without a step
                // are never used): defined on every path, as the allocator needs.
                tmem_ld32(t_lane + o_e + G * dh + c0, oa);
                tmem_ld32(t_lane + o_o + G * dh + c0, ob);
                tmem_wait_ld();
                uint32_t pw[16];
#pragma unroll
                for (int q = 0; q < 32; q += 2) {
                    float f[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float va = (ok && had_e) ? __uint_as_float(oa[q + e]) : 0.f;
                        const float vb = (ok && had_o) ? __uint_as_float(ob[q + e]) : 0.f;
                        f[e] = __fmaf_rn(s_e, va, __fmul_rn(s_o, vb));
                    }
                    if constexpr (kGated) {
                        const uint32_t gw = gfw[(c0 + q) >> 1];
                        f[0] = fmaf(__uint_as_float(gw << 16), f[0], ct[c0 + q]);
                        f[1] = fmaf(__uint_as_float(gw & 0xFFFF0000u), f[1], ct[c0 + q + 1]);
                    }
                    pw[q >> 1] = pack_bf16x2(f[0], f[1]);
                }
                if (wo) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        __stcs(dst + c0 / 8 + v, make_uint4(pw[4 * v], pw[4 * v + 1], pw[4 * v + 2], pw[4 * v + 3]));
                }
            }
            // O_0 and O_1 have been read: the next unit's P.V may overwrite them.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ms.o_free));
            if (wr && G == 0) {
                const size_t at = ((size_t)b * p.heads + h) * s_pad + (size_t)i * kCubeTokens + (r & 63);
                const float lse2 = lt > 0.f ? mt + __log2f(lt) : ninf;  // log2 units
                if (p.lse) p.lse[at] = lt > 0.f ? lse2 * 0.69314718055994531f : ninf;
                // The largest softmax weight of the row: 2^(exact max - lse).
                if constexpr (kPeak) p.max_prob[at] = lt > 0.f ? ex2_approx(m_true - lse2) : 0.f;
            }
            g = g0 + nst;
        }
    }

    // ------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
    if (kDyn && threadIdx.x == 0) {
        // Every claim of this CTA precedes its count here; the last CTA to
        // count puts the slot back to zero for the next launch that takes it.
        __threadfence();
        if (atomicAdd(&g_cta_done[p.slot], 1u) == gridDim.x - 1) {
            g_unit_next[p.slot] = 0;
            g_cta_done[p.slot] = 0;
            __threadfence();
        }
    }
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
                        const void* gate_f, void* out, float* lse, float* max_prob, const vsa_grid* raster,
                        unsigned int* err, int num_sms, cudaStream_t stream) {
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
    p.max_prob = max_prob;
    p.err = err;
    p.B = B;
    p.N = ncubes;
    p.heads = heads;
    p.D = D;
    p.topk = topk;
    p.npairs = (ncubes + 1) / 2;
    p.num_units = B * heads * p.npairs;
    static std::atomic<unsigned int> ticket{0};
    p.slot = (int)(ticket.fetch_add(1u, std::memory_order_relaxed) % (unsigned int)kUnitSlots);
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.tokens = 0;
    p.gT = p.gH = p.gW = p.gnh = p.gnw = 1;
    if (raster) {
        if (coarse_out) return cudaErrorInvalidValue;  // gates and coarse term are laid out tiled
        p.tokens = (long long)raster->T * raster->H * raster->W;
        p.gT = raster->T;
        p.gH = raster->H;
        p.gW = raster->W;
        p.gnh = (raster->H + 3) / 4;
        p.gnw = (raster->W + 3) / 4;
    }
    // The exact row maximum behind max_prob is tracked only in the peak
    // instantiation (it costs about 1% of the ungated kernel's time); the peak
    // entry point runs ungated.
    if (max_prob && coarse_out) return cudaErrorInvalidValue;
    // Rows of variable length (counts) take the dynamic unit schedule; the
    // fixed-length call keeps the static one (no load imbalance to win back,
    // and the static form is the faster one there).
    const bool dyn = counts != nullptr && !coarse_out && !max_prob;
    auto kernel =
        coarse_out ? (D == 64 ? fine_fwd_kernel<64, true, false, false> : fine_fwd_kernel<128, true, false, false>)
        : max_prob ? (D == 64 ? fine_fwd_kernel<64, false, true, false> : fine_fwd_kernel<128, false, true, false>)
        : dyn      ? (D == 64 ? fine_fwd_kernel<64, false, false, true> : fine_fwd_kernel<128, false, false, true>)
                   : (D == 64 ? fine_fwd_kernel<64, false, false, false> : fine_fwd_kernel<128, false, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    // The setmaxnreg split is sized for a launch of exactly kLaunchRegs
    // registers per thread; any other count would leave the softmax warps'
    // setmaxnreg.inc waiting forever, so refuse to launch.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidKernelImage;
    const int grid = p.num_units < num_sms ? p.num_units : num_sms;
    kernel<<<grid, kThreads, kSmemAlloc, stream>>>(mk, mv, p);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace vsa
