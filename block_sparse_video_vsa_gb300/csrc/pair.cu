// Query-cube pairing for the fine stage.
//
// The fine kernel takes query cubes two at a time (one 128-row tensor-core
// tile) and walks the union of their selections, so a pair (i, j) costs
// ceil(|sel(i) u sel(j)| / 2) steps of 128 keys.  Pairing cubes whose
// selections overlap most makes the unions small.  The attention results do
// not depend on the pairing (each query row attends exactly its own
// selection, "Wan2.2 Production Values -- VSA Block-Sparse Attention Inputs +
// Reference", Operator contract); only the order of floating-point
// accumulation does.
//
// Deterministic and integer only, in three launches:
//  1. selection bitmaps of the N cubes of every (batch, head) (workspace);
//  2. for every cube i, the kTopC cubes j != i of sel(i) of largest overlap
//     |sel(i) & sel(j)| (popcount of the AND of two bitmaps; ties: smaller j),
//     best first, kept as int16 lists in the workspace (whole grid);
//  then one CTA per (batch, head):
//  3. kRounds1 rounds of mutual-best matching: every unpaired cube proposes to
//     its unpaired candidate of largest overlap (ties: smaller j), the first
//     unpaired entry of its list, if any; mutual proposals pair up;
//  4. the cubes still unpaired, in index order (the first kMaxLeft of them),
//     run kRounds2 more rounds in which each proposes among the kWindow list
//     entries before and after it (their overlaps computed once);
//  5. the rest pair in index order; with N odd one cube stays single.
// Units are written in order of their smaller cube index:
//   pairs[b, head, u] = i | (j << 16), j = 0xFFFF for a single cube.
#include <type_traits>

#include "vsa_common.cuh"

namespace vsa {

namespace {

constexpr int kPairThreads = 512;
constexpr int kPairWarps = kPairThreads / 32;
constexpr int kTopC = 16;  // candidates kept per cube
constexpr int kRounds1 = 4;
constexpr int kRounds2 = 4;
constexpr int kMaxLeft = 640;
constexpr int kWovStride = kMaxLeft + 2;  // window overlaps [2 kWindow][kWovStride]: conflict-free both ways
constexpr int kWindow = 64;
constexpr int kPairMaxCubes = 8192;
constexpr int kPairMaxTopk = 512;

struct PairArgs {
    const int32_t* idx;  // [B * heads][N][k]
    int N, k, Wp;        // Wp: bitmap words per cube, a multiple of 4
    int npairs;          // ceil(N / 2)
    uint32_t* bm;        // [B * heads][N][Wp]
    int16_t* cand;       // [B * heads][N][kTopC]: candidate lists, best first
    uint32_t* pairs;     // [B * heads][npairs]
};

// Ordered compaction over one chunk of kPairThreads flags: this thread's rank
// among the set flags before it, and the chunk's count in `total`.
__device__ __forceinline__ int chunk_rank(bool flag, int* wsum, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned b = __ballot_sync(0xffffffffu, flag);
    if (lane == 0) wsum[warp] = __popc(b);
    __syncthreads();
    int before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kPairWarps; ++w) {
        const int c = wsum[w];
        before += w < warp ? c : 0;
        tot += c;
    }
    __syncthreads();
    total = tot;
    return before + __popc(b & ((1u << lane) - 1u));
}

__device__ __forceinline__ int bitmap_overlap(const uint32_t* a, const uint32_t* b, int Wp) {
    const uint4* a4 = reinterpret_cast<const uint4*>(a);
    const uint4* b4 = reinterpret_cast<const uint4*>(b);
    int s = 0;
    for (int q = 0; q < Wp / 4; ++q) {
        const uint4 x = a4[q], y = b4[q];
        s += __popc(x.x & y.x) + __popc(x.y & y.y) + __popc(x.z & y.z) + __popc(x.w & y.w);
    }
    return s;
}

// 16-byte load of bitmap words, from shared memory (kShared) or global memory.
template <bool kShared>
__device__ __forceinline__ uint4 ld_words(const uint32_t* p) {
    if constexpr (kShared) {
        uint4 v;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"((uint32_t)__cvta_generic_to_shared(p)));
        return v;
    } else {
        return __ldg(reinterpret_cast<const uint4*>(p));
    }
}

// Overlaps of row a with rows b[0..3] (null: skipped, 0); the loads of the
// four rows are issued together.
template <bool kShared>
__device__ __forceinline__ void bitmap_overlap4(const uint32_t* a, const uint32_t* const (&b)[4], int Wp,
                                                int (&o)[4]) {
    int s0 = 0, s1 = 0, s2 = 0, s3 = 0;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int q = 0; q < Wp / 4; ++q) {
        const uint4 x = ld_words<kShared>(a + 4 * q);
        const uint4 y0 = b[0] ? ld_words<kShared>(b[0] + 4 * q) : z;
        const uint4 y1 = b[1] ? ld_words<kShared>(b[1] + 4 * q) : z;
        const uint4 y2 = b[2] ? ld_words<kShared>(b[2] + 4 * q) : z;
        const uint4 y3 = b[3] ? ld_words<kShared>(b[3] + 4 * q) : z;
        s0 += __popc(x.x & y0.x) + __popc(x.y & y0.y) + __popc(x.z & y0.z) + __popc(x.w & y0.w);
        s1 += __popc(x.x & y1.x) + __popc(x.y & y1.y) + __popc(x.z & y1.z) + __popc(x.w & y1.w);
        s2 += __popc(x.x & y2.x) + __popc(x.y & y2.y) + __popc(x.z & y2.z) + __popc(x.w & y2.w);
        s3 += __popc(x.x & y3.x) + __popc(x.y & y3.y) + __popc(x.z & y3.z) + __popc(x.w & y3.w);
    }
    o[0] = s0;
    o[1] = s1;
    o[2] = s2;
    o[3] = s3;
}

// 1. Selection bitmaps: one warp per (batch, head, cube) row.
__global__ void __launch_bounds__(kPairThreads) pair_bitmap_kernel(PairArgs a, size_t rows) {
    const int lane = threadIdx.x & 31;
    const size_t row = (size_t)blockIdx.x * kPairWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    uint32_t* bits = a.bm + row * a.Wp;
    for (int w = lane; w < a.Wp; w += 32) bits[w] = 0u;
    __syncwarp();
    const int32_t* sel = a.idx + row * a.k;
    for (int e = lane; e < a.k; e += 32) {
        const int j = sel[e];
        if (j >= 0 && j < a.N) atomicOr(&bits[j >> 5], 1u << (j & 31));
    }
}

// 2. Candidate lists: for every cube i, the kTopC cubes j != i of sel(i) of
// largest overlap |sel(i) & sel(j)| (ties: smaller j), best first, -1 past
// the valid entries.  Blocks (chunk, b * heads + head); one warp per cube:
// overlaps from the bitmaps (staged in shared memory when the head's fit),
// keys (ov << 16) | (0xFFFF - j) in registers, kTopC rounds of a warp max.
template <bool kStaged, int kPerLane>
__global__ void __launch_bounds__(kPairThreads) pair_candidates_kernel(PairArgs a) {
    extern __shared__ __align__(16) uint32_t dsm_c[];  // [N][Wp] bitmaps when staged
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int N = a.N, k = a.k, Wp = a.Wp;
    const size_t bh = blockIdx.y;
    const uint32_t* base = a.bm + bh * (size_t)N * Wp;
    if constexpr (kStaged) {
        uint4* dst = reinterpret_cast<uint4*>(dsm_c);
        const uint4* src = reinterpret_cast<const uint4*>(base);
        for (int t = threadIdx.x; t < N * Wp / 4; t += kPairThreads) dst[t] = src[t];
        __syncthreads();
        base = dsm_c;
    }
    const int per = (N + gridDim.x - 1) / gridDim.x;
    const int i_end = min(N, ((int)blockIdx.x + 1) * per);
    for (int i = (int)blockIdx.x * per + warp; i < i_end; i += kPairWarps) {
        const size_t row = bh * (size_t)N + i;
        const int32_t* sel = a.idx + row * k;
        uint32_t key[kPerLane];
#pragma unroll
        for (int m0 = 0; m0 < kPerLane; m0 += 4) {
            int jj[4];
            const uint32_t* rb[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int e = lane + 32 * (m0 + v);
                jj[v] = e < k ? sel[e] : -1;
                const bool ok = jj[v] >= 0 && jj[v] < N && jj[v] != i;
                if (!ok) jj[v] = -1;
                rb[v] = ok ? base + (size_t)jj[v] * Wp : nullptr;
            }
            int o[4];
            bitmap_overlap4<kStaged>(base + (size_t)i * Wp, rb, Wp, o);
#pragma unroll
            for (int v = 0; v < 4; ++v)
                key[m0 + v] = jj[v] >= 0 ? ((uint32_t)o[v] << 16) | (uint32_t)(0xFFFF - jj[v]) : 0u;
        }
        int16_t* out = a.cand + row * kTopC;
        for (int r = 0; r < kTopC; ++r) {
            uint32_t best = 0u;
#pragma unroll
            for (int m = 0; m < kPerLane; ++m) best = key[m] > best ? key[m] : best;
            best = __reduce_max_sync(0xffffffffu, best);
            if (best) {
#pragma unroll
                for (int m = 0; m < kPerLane; ++m) key[m] = key[m] == best ? 0u : key[m];
            }
            if (lane == 0) out[r] = best ? (int16_t)(0xFFFF - (best & 0xFFFFu)) : (int16_t)-1;
        }
    }
}

// 3-5. Matching and the unit list, one CTA per (batch, head).  Dynamic shared
// memory: the overlaps of each leftover cube with its window, then the
// partner, proposal and list-position arrays of N entries, the leftover list.
__global__ void __launch_bounds__(kPairThreads) pair_match_kernel(PairArgs a, int rows_cap) {
    extern __shared__ __align__(16) unsigned char dsm[];
    const int N = a.N, k = a.k, Wp = a.Wp;
    uint16_t* wov = reinterpret_cast<uint16_t*>(dsm);                   // [2 kWindow][kWovStride]
    int16_t* partner = reinterpret_cast<int16_t*>(wov + 2 * kWindow * kWovStride);  // -1 unpaired, j, or i single
    int16_t* prop = partner + N;                                        // proposals, later the rest
    int16_t* ptr = prop + N;                                            // next candidate to look at
    int16_t* left = ptr + N;                                            // [kMaxLeft]
    int16_t* lprop = left + kMaxLeft;                                   // [kMaxLeft]
    uint32_t* lrows = reinterpret_cast<uint32_t*>(dsm + (((reinterpret_cast<uintptr_t>(lprop + kMaxLeft) -
                                                          reinterpret_cast<uintptr_t>(dsm)) + 15) & ~(uintptr_t)15));
    // lrows: bitmap rows of the leftover list when nleft * Wp words fit rows_cap
    __shared__ int wsum[kPairWarps];
    __shared__ uint32_t lfree[kMaxLeft / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t bh = blockIdx.x;
    const uint32_t* bm = a.bm + bh * (size_t)N * Wp;
    const int16_t* cand = a.cand + bh * (size_t)N * kTopC;

    for (int i = tid; i < N; i += kPairThreads) {
        partner[i] = -1;
        ptr[i] = 0;
    }
    __syncthreads();

    // 3. mutual-best rounds over the own selection: the first unpaired entry of
    // the sorted candidate list (paired cubes stay paired, so the scan resumes
    // where the previous round stopped).
    for (int rd = 0; rd < kRounds1; ++rd) {
        for (int i = tid; i < N; i += kPairThreads) {
            int best = -1;
            if (partner[i] < 0) {
                const int16_t* row = cand + (size_t)i * kTopC;
                int e = ptr[i];
                for (; e < kTopC; ++e) {
                    const int j = row[e];
                    if (j < 0) {
                        e = kTopC;
                        break;
                    }
                    if (partner[j] < 0) {
                        best = j;
                        break;
                    }
                }
                ptr[i] = (int16_t)e;
            }
            prop[i] = (int16_t)best;
        }
        __syncthreads();
        for (int i = tid; i < N; i += kPairThreads) {
            const int j = prop[i];
            if (j > i && prop[j] == i) {
                partner[i] = (int16_t)j;
                partner[j] = (int16_t)i;
            }
        }
        __syncthreads();
    }

    // 4. the unpaired cubes (first kMaxLeft, index order) within a window:
    // overlaps with the kWindow list entries on each side, once (a warp per
    // leftover cube, a lane per candidate), then kRounds2 rounds.
    int nleft = 0;
    for (int base = 0; base < N; base += kPairThreads) {
        const int i = base + tid;
        const bool f = i < N && partner[i] < 0;
        int tot;
        const int r = chunk_rank(f, wsum, tot);
        if (f && nleft + r < kMaxLeft) left[nleft + r] = (int16_t)i;
        nleft += tot;
    }
    nleft = min(nleft, kMaxLeft);
    __syncthreads();
    const bool staged = nleft * Wp <= rows_cap;
    if (staged) {
        for (int t = tid; t < nleft * (Wp / 4); t += kPairThreads) {
            const int f = t / (Wp / 4), q = t - f * (Wp / 4);
            reinterpret_cast<uint4*>(lrows)[t] = reinterpret_cast<const uint4*>(bm + (size_t)left[f] * Wp)[q];
        }
        __syncthreads();
    }
    static_assert(2 * kWindow == 128, "one candidate per lane and slot of four");
    for (int f = warp; f < nleft; f += kPairWarps) {
        const uint32_t* rb[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int d = lane + 32 * v;
            const int g = d < kWindow ? f - kWindow + d : f + 1 + (d - kWindow);
            rb[v] = (g >= 0 && g < nleft) ? (staged ? lrows + (size_t)g * Wp : bm + (size_t)left[g] * Wp) : nullptr;
        }
        int o[4];
        if (staged)
            bitmap_overlap4<true>(lrows + (size_t)f * Wp, rb, Wp, o);
        else
            bitmap_overlap4<false>(bm + (size_t)left[f] * Wp, rb, Wp, o);
#pragma unroll
        for (int v = 0; v < 4; ++v) wov[(lane + 32 * v) * kWovStride + f] = (uint16_t)o[v];
    }
    __syncthreads();
    for (int rd = 0; rd < kRounds2; ++rd) {
        // Unpaired list entries as a bitmask (the list is in increasing cube
        // order, so list position breaks ties like the cube index).
        for (int g0 = warp * 32; g0 < kMaxLeft; g0 += kPairThreads) {
            const int g = g0 + lane;
            const unsigned m = __ballot_sync(0xffffffffu, g < nleft && partner[left[min(g, nleft - 1)]] < 0);
            if (lane == 0) lfree[g0 >> 5] = m;
        }
        __syncthreads();
        // A warp per leftover, a lane per four window entries; the best is the
        // largest overlap, ties to the smaller list position.
        for (int f = warp; f < nleft; f += kPairWarps) {
            uint32_t key = 0u;  // (overlap + 1) << 16 | (0xFFFF - g); 0: none
            if ((lfree[f >> 5] >> (f & 31)) & 1u) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int d = lane + 32 * v;
                    const int g = d < kWindow ? f - kWindow + d : f + 1 + (d - kWindow);
                    if (g >= 0 && g < nleft && ((lfree[g >> 5] >> (g & 31)) & 1u)) {
                        const uint32_t kk = ((uint32_t)wov[d * kWovStride + f] + 1u) << 16 | (uint32_t)(0xFFFF - g);
                        key = kk > key ? kk : key;
                    }
                }
            }
            key = __reduce_max_sync(0xffffffffu, key);
            if (lane == 0) lprop[f] = key ? (int16_t)(0xFFFF - (key & 0xFFFFu)) : (int16_t)-1;
        }
        __syncthreads();
        for (int f = tid; f < nleft; f += kPairThreads) {
            const int g = lprop[f];
            if (g > f && lprop[g] == f) {
                partner[left[f]] = left[g];
                partner[left[g]] = left[f];
            }
        }
        __syncthreads();
    }

    // 5. the rest in index order.
    int nrest = 0;
    for (int base = 0; base < N; base += kPairThreads) {
        const int i = base + tid;
        const bool f = i < N && partner[i] < 0;
        int tot;
        const int r = chunk_rank(f, wsum, tot);
        if (f) prop[nrest + r] = (int16_t)i;
        nrest += tot;
    }
    __syncthreads();
    for (int q = tid; 2 * q + 1 < nrest; q += kPairThreads) {
        const int x = prop[2 * q], y = prop[2 * q + 1];
        partner[x] = (int16_t)y;
        partner[y] = (int16_t)x;
    }
    if (tid == 0 && (nrest & 1)) partner[prop[nrest - 1]] = prop[nrest - 1];
    __syncthreads();

    // Units in order of their smaller cube index.
    uint32_t* out = a.pairs + bh * (size_t)a.npairs;
    int u0 = 0;
    for (int base = 0; base < N; base += kPairThreads) {
        const int i = base + tid;
        const bool f = i < N && partner[i] >= i;
        int tot;
        const int r = chunk_rank(f, wsum, tot);
        if (f && u0 + r < a.npairs) {
            const int j = partner[i];
            out[u0 + r] = (uint32_t)i | ((uint32_t)(j == i ? 0xFFFF : j) << 16);
        }
        u0 += tot;
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

int pair_words(int ncubes) { return ((ncubes + 31) / 32 + 3) & ~3; }

size_t pair_workspace_bytes(int B, int heads, int ncubes, int topk) {
    const size_t bh = (size_t)B * heads;
    (void)topk;
    return align256(bh * ncubes * pair_words(ncubes) * sizeof(uint32_t)) + align256(bh * ncubes * kTopC * sizeof(int16_t));
}

int pair_max_cubes() { return kPairMaxCubes; }
int pair_max_topk() { return kPairMaxTopk; }

cudaError_t launch_pair(const int32_t* topk_idx, int B, int ncubes, int heads, int topk, void* workspace,
                        uint32_t* pairs, int num_sms, int max_smem, cudaStream_t stream) {
    PairArgs a;
    a.idx = topk_idx;
    a.N = ncubes;
    a.k = topk;
    a.Wp = pair_words(ncubes);
    a.npairs = (ncubes + 1) / 2;
    const size_t bh = (size_t)B * heads;
    a.bm = static_cast<uint32_t*>(workspace);
    a.cand = reinterpret_cast<int16_t*>(static_cast<unsigned char*>(workspace) +
                                        align256(bh * ncubes * a.Wp * sizeof(uint32_t)));
    a.pairs = pairs;
    const size_t rows = bh * ncubes;
    pair_bitmap_kernel<<<(unsigned)((rows + kPairWarps - 1) / kPairWarps), kPairThreads, 0, stream>>>(a, rows);
    const size_t bm_bytes = (size_t)ncubes * a.Wp * sizeof(uint32_t);
    const bool stage_bm = bm_bytes <= (size_t)max_smem - 1024;
    const size_t dyn_c = stage_bm ? bm_bytes : 0;
    int chunks = (int)((2 * (size_t)num_sms + bh - 1) / bh);
    chunks = chunks < 1 ? 1 : chunks;
    const int max_chunks = (ncubes + kPairWarps - 1) / kPairWarps;
    chunks = chunks > max_chunks ? max_chunks : chunks;
    auto pick = [&](auto staged) -> void (*)(PairArgs) {
        constexpr bool S = decltype(staged)::value;
        if (topk <= 128) return pair_candidates_kernel<S, 4>;
        if (topk <= 256) return pair_candidates_kernel<S, 8>;
        return pair_candidates_kernel<S, 16>;
    };
    void (*cand_kernel)(PairArgs) = stage_bm ? pick(std::true_type()) : pick(std::false_type());
    cudaError_t e = cudaFuncSetAttribute(cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_c);
    if (e != cudaSuccess) return e;
    cand_kernel<<<dim3((unsigned)chunks, (unsigned)bh), kPairThreads, dyn_c, stream>>>(a);
    // Matching: window overlaps, N-entry arrays, leftover list, then as many
    // leftover bitmap rows as the rest of the shared memory holds.
    const size_t fixed = (size_t)2 * kWindow * kWovStride * sizeof(uint16_t) + 3 * (size_t)ncubes * 2 +
                         2 * (size_t)kMaxLeft * 2 + 16;
    const size_t avail = (size_t)max_smem - 1024;  // static shared memory of the kernel is below 1 KB
    if (fixed > avail) return cudaErrorInvalidValue;
    const size_t rows_bytes = avail - fixed < (size_t)kMaxLeft * a.Wp * 4 ? avail - fixed : (size_t)kMaxLeft * a.Wp * 4;
    const int rows_cap = (int)(rows_bytes / 4);
    const size_t dyn = fixed + rows_bytes;
    e = cudaFuncSetAttribute(pair_match_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
    pair_match_kernel<<<(unsigned)bh, kPairThreads, dyn, stream>>>(a, rows_cap);
    return cudaGetLastError();
}

}  // namespace vsa
