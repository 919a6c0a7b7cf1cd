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
// The procedure, per (batch, head), deterministic and integer only:
//  a. overlap(i, j) = |sel(i) & sel(j)| for j in sel(i); the candidates of i
//     are its kTopC cubes j != i of largest overlap (ties: smaller j);
//  b. kRounds1 rounds of mutual-best matching: every unpaired cube proposes to
//     its unpaired candidate of largest overlap (the first unpaired entry of
//     its list), if any; mutual proposals pair up;
//  c. the cubes still unpaired, in index order (the first kMaxLeft of them),
//     run kRounds2 more rounds in which each proposes to the unpaired cube of
//     largest overlap among the kWindow list entries before and after it
//     (ties: smaller list position, i.e. smaller cube index);
//  d. the rest pair in index order; with N odd one cube stays single.
// Units are written in order of their smaller cube index:
//   pairs[b, head, u] = i | (j << 16), j = 0xFFFF for a single cube.
//
// Five launches, each sized so that its working set sits in shared memory:
//  1. selection bitmaps (a warp per cube);
//  2. candidate lists (a): the bitmap columns are staged in chunks that fit
//     shared memory, overlaps accumulate per (cube, entry), then a warp picks
//     the kTopC best by rounds of a warp max;
//  3. rounds (b), one CTA per (batch, head), lists in shared memory; writes the
//     partner array and the leftover list;
//  4. window overlaps of (c), blocks over (leftover chunk, batch, head);
//  5. rounds (c) and (d) and the unit list, one CTA per (batch, head).
#include "vsa_common.cuh"

namespace vsa {

namespace {

constexpr int kPairThreads = 512;
constexpr int kPairWarps = kPairThreads / 32;
constexpr int kTopC = 16;        // candidates kept per cube
constexpr int kRounds1 = 4;
constexpr int kRounds2 = 4;
constexpr int kMaxLeft = 640;    // leftover list length cap
constexpr int kWindow = 64;      // list entries on each side
constexpr int kWin = 2 * kWindow;
constexpr int kWinChunk = 64;    // leftovers per window block
constexpr int kPairMaxCubes = 8192;
constexpr int kPairMaxTopk = 512;
constexpr size_t kSmemBudget = 200 * 1024;  // dynamic shared memory a pairing block plans for

struct PairArgs {
    const int32_t* idx;  // [BH][N][k]
    int N, k, Wp;        // Wp: bitmap words per cube, a multiple of 4
    int npairs;          // ceil(N / 2)
    uint32_t* bm;        // [BH][N][Wp]
    int16_t* cand;       // [BH][N][kTopC]: candidate lists, best first, -1 past the end
    int16_t* partner;    // [BH][N]: after (b); -1 unpaired
    int16_t* left;       // [BH][kMaxLeft]: leftover list
    int* nleft;          // [BH]
    uint16_t* wov;       // [BH][kMaxLeft][kWin]: window overlaps
    uint32_t* pairs;     // [BH][npairs]
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

__device__ __forceinline__ uint4 lds128(const uint32_t* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
    return v;
}

// |a & b| over `words` words (a multiple of 4) of two shared-memory rows.
__device__ __forceinline__ int smem_overlap(const uint32_t* a, const uint32_t* b, int words) {
    int s = 0;
    for (int q = 0; q < words; q += 4) {
        const uint4 x = lds128(a + q), y = lds128(b + q);
        s += __popc(x.x & y.x) + __popc(x.y & y.y) + __popc(x.z & y.z) + __popc(x.w & y.w);
    }
    return s;
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

// 2. Candidate lists.  Block (row chunk, b * heads + head) owns rows
// [i0, i0 + rb).  Shared memory: bitmap columns [N][cs] (cw words of the
// current column chunk; the row stride cs is an odd number of 16-byte quads so
// that rows at random indices spread over the banks), overlap accumulators
// [rb][k] (uint16) and the entries [rb][k] (int16, -1 for j == i or out of range).
template <int kPerLane>
__global__ void __launch_bounds__(kPairThreads) pair_candidates_kernel(PairArgs a, int rb, int cw, int cs) {
    extern __shared__ __align__(16) uint32_t dsm_c[];
    const int N = a.N, k = a.k, Wp = a.Wp;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t bh = blockIdx.y;
    const int i0 = (int)blockIdx.x * rb;
    const int rows = min(rb, N - i0);
    if (rows <= 0) return;
    uint32_t* cols = dsm_c;
    uint16_t* acc = reinterpret_cast<uint16_t*>(cols + (size_t)N * cs);
    int16_t* ids = reinterpret_cast<int16_t*>(acc + (size_t)rb * k);
    const uint32_t* bm = a.bm + bh * (size_t)N * Wp;
    const int32_t* sel = a.idx + (bh * (size_t)N + i0) * k;
    for (int t = tid; t < rows * k; t += kPairThreads) {
        const int i = i0 + t / k;
        const int j = sel[t];
        ids[t] = (j >= 0 && j < N && j != i) ? (int16_t)j : (int16_t)-1;
        acc[t] = 0;
    }
    for (int c0 = 0; c0 < Wp; c0 += cw) {
        const int w = min(cw, Wp - c0);  // a multiple of 4
        __syncthreads();                 // the previous chunk is no longer read
        for (int t = tid; t < N * (w / 4); t += kPairThreads) {
            const int n = t / (w / 4), q = t - n * (w / 4);
            reinterpret_cast<uint4*>(cols + (size_t)n * cs)[q] =
                reinterpret_cast<const uint4*>(bm + (size_t)n * Wp + c0)[q];
        }
        __syncthreads();
        for (int t = tid; t < rows * k; t += kPairThreads) {
            const int j = ids[t];
            if (j < 0) continue;
            const int i = i0 + t / k;
            acc[t] = (uint16_t)(acc[t] + smem_overlap(cols + (size_t)i * cs, cols + (size_t)j * cs, w));
        }
    }
    __syncthreads();
    // The kTopC best of each row: keys (overlap << 16) | (0xFFFF - j).
    for (int r = warp; r < rows; r += kPairWarps) {
        uint32_t key[kPerLane];
#pragma unroll
        for (int m = 0; m < kPerLane; ++m) {
            const int e = lane + 32 * m;
            const int j = e < k ? ids[r * k + e] : -1;
            key[m] = j >= 0 ? ((uint32_t)acc[r * k + e] << 16) | (uint32_t)(0xFFFF - j) : 0u;
        }
        int16_t* out = a.cand + (bh * (size_t)N + i0 + r) * kTopC;
        for (int c = 0; c < kTopC; ++c) {
            uint32_t best = 0u;
#pragma unroll
            for (int m = 0; m < kPerLane; ++m) best = key[m] > best ? key[m] : best;
            best = __reduce_max_sync(0xffffffffu, best);
            if (best) {
#pragma unroll
                for (int m = 0; m < kPerLane; ++m) key[m] = key[m] == best ? 0u : key[m];
            }
            if (lane == 0) out[c] = best ? (int16_t)(0xFFFF - (best & 0xFFFFu)) : (int16_t)-1;
        }
    }
}

// 3. Rounds (b), one CTA per (batch, head).  Shared memory: partner, proposal
// and list-position arrays [N] and, when they fit (stage_lists), the
// candidate lists [N][kTopC].
__global__ void __launch_bounds__(kPairThreads) pair_match1_kernel(PairArgs a, int stage_lists) {
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ int wsum[kPairWarps];
    const int N = a.N;
    const int tid = threadIdx.x;
    const size_t bh = blockIdx.x;
    int16_t* partner = reinterpret_cast<int16_t*>(dsm);
    int16_t* prop = partner + N;
    int16_t* ptr = prop + N;
    const int16_t* cand = a.cand + bh * (size_t)N * kTopC;
    if (stage_lists) {
        int16_t* lists = ptr + N;
        for (int t = tid; t < N * kTopC; t += kPairThreads) lists[t] = cand[t];
        cand = lists;
    }
    for (int i = tid; i < N; i += kPairThreads) {
        partner[i] = -1;
        ptr[i] = 0;
    }
    __syncthreads();
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
    // The leftover list (first kMaxLeft unpaired cubes, index order).
    int16_t* left = a.left + bh * kMaxLeft;
    int nleft = 0;
    for (int base = 0; base < N; base += kPairThreads) {
        const int i = base + tid;
        const bool f = i < N && partner[i] < 0;
        int tot;
        const int r = chunk_rank(f, wsum, tot);
        if (f && nleft + r < kMaxLeft) left[nleft + r] = (int16_t)i;
        nleft += tot;
    }
    if (tid == 0) a.nleft[bh] = min(nleft, kMaxLeft);
    int16_t* pout = a.partner + bh * (size_t)N;
    for (int i = tid; i < N; i += kPairThreads) pout[i] = partner[i];
}

// 4. Window overlaps: block (chunk of kWinChunk leftovers, b * heads + head).
// Shared memory: the bitmap rows of the list entries the chunk's windows
// reach (at most kWinChunk + kWin rows).
__global__ void __launch_bounds__(kPairThreads) pair_window_kernel(PairArgs a) {
    extern __shared__ __align__(16) uint32_t rows_s[];
    const int Wp = a.Wp;
    const size_t bh = blockIdx.y;
    const int nleft = a.nleft[bh];
    const int f0 = (int)blockIdx.x * kWinChunk;
    if (f0 >= nleft) return;
    const int f1 = min(nleft, f0 + kWinChunk);
    const int g0 = max(0, f0 - kWindow), g1 = min(nleft, f1 + kWindow);
    const int16_t* left = a.left + bh * kMaxLeft;
    const uint32_t* bm = a.bm + bh * (size_t)a.N * Wp;
    for (int t = threadIdx.x; t < (g1 - g0) * (Wp / 4); t += kPairThreads) {
        const int g = t / (Wp / 4), q = t - g * (Wp / 4);
        reinterpret_cast<uint4*>(rows_s + (size_t)g * Wp)[q] =
            reinterpret_cast<const uint4*>(bm + (size_t)left[g0 + g] * Wp)[q];
    }
    __syncthreads();
    uint16_t* wov = a.wov + bh * (size_t)kMaxLeft * kWin;
    for (int t = threadIdx.x; t < (f1 - f0) * kWin; t += kPairThreads) {
        const int f = f0 + t / kWin, d = t % kWin;
        const int g = d < kWindow ? f - kWindow + d : f + 1 + (d - kWindow);
        int o = 0;
        if (g >= 0 && g < nleft)
            o = smem_overlap(rows_s + (size_t)(f - g0) * Wp, rows_s + (size_t)(g - g0) * Wp, Wp);
        wov[(size_t)f * kWin + d] = (uint16_t)o;
    }
}

// 5. Rounds (c), (d) and the unit list, one CTA per (batch, head).  Shared
// memory: window overlaps [kMaxLeft][kWin], partner and rest arrays [N].
__global__ void __launch_bounds__(kPairThreads) pair_match2_kernel(PairArgs a) {
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ int wsum[kPairWarps];
    __shared__ uint32_t lfree[kMaxLeft / 32];
    __shared__ int16_t left[kMaxLeft];
    __shared__ int16_t lprop[kMaxLeft];
    const int N = a.N;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t bh = blockIdx.x;
    uint16_t* wov = reinterpret_cast<uint16_t*>(dsm);
    int16_t* partner = reinterpret_cast<int16_t*>(wov + (size_t)kMaxLeft * kWin);
    int16_t* rest = partner + N;
    const int nleft = a.nleft[bh];
    {
        const int16_t* pin = a.partner + bh * (size_t)N;
        for (int i = tid; i < N; i += kPairThreads) partner[i] = pin[i];
        const int16_t* lin = a.left + bh * kMaxLeft;
        for (int f = tid; f < nleft; f += kPairThreads) left[f] = lin[f];
        const uint4* win = reinterpret_cast<const uint4*>(a.wov + bh * (size_t)kMaxLeft * kWin);
        for (int t = tid; t < nleft * kWin / 8; t += kPairThreads) reinterpret_cast<uint4*>(wov)[t] = win[t];
    }
    __syncthreads();
    for (int rd = 0; rd < kRounds2; ++rd) {
        // Unpaired list entries as a bitmask.
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
                for (int v = 0; v < kWin / 32; ++v) {
                    const int d = lane + 32 * v;
                    const int g = d < kWindow ? f - kWindow + d : f + 1 + (d - kWindow);
                    if (g >= 0 && g < nleft && ((lfree[g >> 5] >> (g & 31)) & 1u)) {
                        const uint32_t kk = ((uint32_t)wov[f * kWin + d] + 1u) << 16 | (uint32_t)(0xFFFF - g);
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
    // (d) the rest in index order.
    int nrest = 0;
    for (int base = 0; base < N; base += kPairThreads) {
        const int i = base + tid;
        const bool f = i < N && partner[i] < 0;
        int tot;
        const int r = chunk_rank(f, wsum, tot);
        if (f) rest[nrest + r] = (int16_t)i;
        nrest += tot;
    }
    __syncthreads();
    for (int q = tid; 2 * q + 1 < nrest; q += kPairThreads) {
        const int x = rest[2 * q], y = rest[2 * q + 1];
        partner[x] = (int16_t)y;
        partner[y] = (int16_t)x;
    }
    if (tid == 0 && (nrest & 1)) partner[rest[nrest - 1]] = rest[nrest - 1];
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

struct PairLayout {
    size_t bm, cand, partner, left, nleft, wov, total;
};

PairLayout pair_layout(size_t bh, int ncubes, int words) {
    PairLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t r = o;
        o += align256(bytes);
        return r;
    };
    L.bm = take(bh * ncubes * words * sizeof(uint32_t));
    L.cand = take(bh * ncubes * kTopC * sizeof(int16_t));
    L.partner = take(bh * ncubes * sizeof(int16_t));
    L.left = take(bh * kMaxLeft * sizeof(int16_t));
    L.nleft = take(bh * sizeof(int));
    L.wov = take(bh * kMaxLeft * kWin * sizeof(uint16_t));
    L.total = o;
    return L;
}

}  // namespace

int pair_words(int ncubes) { return ((ncubes + 31) / 32 + 3) & ~3; }

size_t pair_workspace_bytes(int B, int heads, int ncubes, int topk) {
    (void)topk;
    return pair_layout((size_t)B * heads, ncubes, pair_words(ncubes)).total;
}

int pair_max_cubes() { return kPairMaxCubes; }
int pair_max_topk() { return kPairMaxTopk; }

cudaError_t launch_pair(const int32_t* topk_idx, int B, int ncubes, int heads, int topk, void* workspace,
                        uint32_t* pairs, int num_sms, int max_smem, cudaStream_t stream) {
    const size_t bh = (size_t)B * heads;
    const int N = ncubes, k = topk;
    PairArgs a;
    a.idx = topk_idx;
    a.N = N;
    a.k = k;
    a.Wp = pair_words(N);
    a.npairs = (N + 1) / 2;
    const PairLayout L = pair_layout(bh, N, a.Wp);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    a.bm = reinterpret_cast<uint32_t*>(ws + L.bm);
    a.cand = reinterpret_cast<int16_t*>(ws + L.cand);
    a.partner = reinterpret_cast<int16_t*>(ws + L.partner);
    a.left = reinterpret_cast<int16_t*>(ws + L.left);
    a.nleft = reinterpret_cast<int*>(ws + L.nleft);
    a.wov = reinterpret_cast<uint16_t*>(ws + L.wov);
    a.pairs = pairs;
    const size_t budget = kSmemBudget < (size_t)max_smem - 1024 ? kSmemBudget : (size_t)max_smem - 1024;
    cudaError_t e;

    // 1. bitmaps
    const size_t rows = bh * N;
    pair_bitmap_kernel<<<(unsigned)((rows + kPairWarps - 1) / kPairWarps), kPairThreads, 0, stream>>>(a, rows);
    note_launches(1);

    // 2. candidate lists: first the staged row stride cs (an odd number of
    // quads, at most ~60% of the budget, at most the padded row), then rows
    // per block (about two blocks per SM in all) within the rest.
    int cs = (int)(((budget * 3 / 5) / ((size_t)N * 4)) & ~(size_t)3);
    if (cs > 0 && ((cs / 4) & 1) == 0) cs -= 4;
    const int wp_odd = ((a.Wp / 4) & 1) ? a.Wp : a.Wp + 4;
    if (cs > wp_odd) cs = wp_odd;
    if (cs < 4) cs = 4;
    const int cw = cs > a.Wp ? a.Wp : cs;
    const size_t cols_bytes = (size_t)N * cs * 4;
    if (cols_bytes + (size_t)k * 4 > budget) return cudaErrorInvalidValue;
    int chunks = (int)((2 * (size_t)num_sms + bh - 1) / bh);
    chunks = chunks < 1 ? 1 : chunks;
    int rb = (N + chunks - 1) / chunks;
    const size_t rb_cap = (budget - cols_bytes) / ((size_t)k * 4);
    if ((size_t)rb > rb_cap) rb = (int)rb_cap;
    chunks = (N + rb - 1) / rb;
    const size_t dyn_c = cols_bytes + (size_t)rb * k * 4;
    auto cand_kernel = k <= 128 ? pair_candidates_kernel<4> : k <= 256 ? pair_candidates_kernel<8>
                                                                        : pair_candidates_kernel<16>;
    e = cudaFuncSetAttribute(cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_c);
    if (e != cudaSuccess) return e;
    cand_kernel<<<dim3((unsigned)chunks, (unsigned)bh), kPairThreads, dyn_c, stream>>>(a, rb, cw, cs);
    note_launches(1);

    // 3. rounds (b)
    const size_t arrays = 3 * (size_t)N * sizeof(int16_t);
    const size_t lists = (size_t)N * kTopC * sizeof(int16_t);
    const int stage_lists = arrays + lists <= budget ? 1 : 0;
    const size_t dyn_1 = arrays + (stage_lists ? lists : 0);
    e = cudaFuncSetAttribute(pair_match1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_1);
    if (e != cudaSuccess) return e;
    pair_match1_kernel<<<(unsigned)bh, kPairThreads, dyn_1, stream>>>(a, stage_lists);
    note_launches(1);

    // 4. window overlaps
    const size_t dyn_w = (size_t)(kWinChunk + kWin) * a.Wp * sizeof(uint32_t);
    if (dyn_w > budget) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(pair_window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_w);
    if (e != cudaSuccess) return e;
    pair_window_kernel<<<dim3(kMaxLeft / kWinChunk, (unsigned)bh), kPairThreads, dyn_w, stream>>>(a);
    note_launches(1);

    // 5. rounds (c), (d), units
    const size_t dyn_2 = (size_t)kMaxLeft * kWin * sizeof(uint16_t) + 2 * (size_t)N * sizeof(int16_t);
    if (dyn_2 > budget) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(pair_match2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_2);
    if (e != cudaSuccess) return e;
    pair_match2_kernel<<<(unsigned)bh, kPairThreads, dyn_2, stream>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace vsa
