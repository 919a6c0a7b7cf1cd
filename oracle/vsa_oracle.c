/*
 * Plain CPU oracle for the Video Sparse Attention (VSA) hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * reference that the CUDA path is checked against.  Nothing in the product
 * library links, includes or calls it; only the tests, the smoke check and
 * the benchmark's CPU-baseline leg load it.  It shares no code, header,
 * table or constant with the CUDA path.
 *
 * All arithmetic is IEEE double.  Inputs are bf16 bit patterns (uint16_t),
 * widened exactly to double.  Every loop follows the definition it cites,
 * with no blocking, fusion or reordering.
 *
 * Sources (page title, section):
 *  [VSA-AMD]  "VSA: Accelerating Video Diffusion Inference with Sparse
 *             Attention on AMD GPUs" -- Two-Stage Architecture (Pre-stage,
 *             Stage 1: Coarse Selection, Stage 2: Fine Computation),
 *             Block-Sparse Encoding, Sparse Traversal, Generating Sparsity
 *             Patterns, The Attention Bottleneck (SDPA formula).
 *  [WAN-VSA]  "Wan2.2 Production Values -- VSA Block-Sparse Attention Inputs
 *             + Reference" -- Shapes, Operator contract.
 *  [STA]      "FastVideo Guide: Sliding Tile Attention" -- Implementation
 *             (tile partition into (tile_t, tile_h, tile_w) blocks, tile
 *             index = (it*n_h + ih)*n_w + iw, inverse permutation).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - cube order: raster over the cube grid, c = (ct*nh + ch)*nw + cw, the
 *    tile index order of [STA] Implementation;
 *  - inside a cube the real tokens of its clipped sub-box come first, in
 *    raster (t, h, w) order, padding slots vbs..63 are zero ([WAN-VSA]
 *    Operator contract: a cube's attention covers only its leading vbs[c]
 *    slots of the 64);
 *  - the cube mean-pool divides by vbs[c] (real tokens only); an empty cube
 *    (vbs = 0, never produced by tiling) pools to the zero vector;
 *  - the cube score is sm_scale * (q_mean . k_mean);
 *  - top-k order: score descending, ties to the lower cube index;
 *  - a row with no unmasked key gives o = 0 and lse = -inf;
 *  - lse is the natural-log log-sum-exp of the scaled logits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define CUBE_T 4
#define CUBE_H 4
#define CUBE_W 4
#define CUBE_TOKENS 64

static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Number of 4x4x4 cubes covering a T x H x W latent grid ([WAN-VSA] Shapes:
 * Nq = ceil(T/4) * ceil(H/4) * ceil(W/4)). */
int64_t oracle_num_cubes(int64_t T, int64_t Hh, int64_t W) {
    return ceil_div(T, CUBE_T) * ceil_div(Hh, CUBE_H) * ceil_div(W, CUBE_W);
}

/*
 * Cube tiling ([VSA-AMD] Pre-stage + Stage 1 cube partition; [WAN-VSA]
 * Shapes "cube-major tiled/padded").
 *
 * x : [B, T*Hh*W, heads, D] bf16, token n = (t*Hh + h)*W + w.
 * xt: [B, ncubes*64, heads, D] bf16, written in full (pads are zero).
 * vbs: [ncubes] real-token count per cube (may be NULL).
 *
 * For each cube in raster cube order, enumerate the tokens of its clipped
 * sub-box in raster order and give them consecutive slots.
 */
void oracle_tile(int64_t B, int64_t T, int64_t Hh, int64_t W, int64_t heads, int64_t D,
                 const uint16_t* x, uint16_t* xt, int32_t* vbs) {
    const int64_t nt = ceil_div(T, CUBE_T), nh = ceil_div(Hh, CUBE_H), nw = ceil_div(W, CUBE_W);
    const int64_t N = nt * nh * nw;
    const int64_t row = heads * D; /* elements per token row */
    const int64_t S = T * Hh * W, S_pad = N * CUBE_TOKENS;
    for (int64_t b = 0; b < B; ++b) {
        memset(xt + b * S_pad * row, 0, (size_t)(S_pad * row) * sizeof(uint16_t));
        for (int64_t ct = 0; ct < nt; ++ct)
            for (int64_t ch = 0; ch < nh; ++ch)
                for (int64_t cw = 0; cw < nw; ++cw) {
                    const int64_t c = (ct * nh + ch) * nw + cw;
                    int64_t slot = 0;
                    for (int64_t t = ct * CUBE_T; t < ct * CUBE_T + CUBE_T && t < T; ++t)
                        for (int64_t h = ch * CUBE_H; h < ch * CUBE_H + CUBE_H && h < Hh; ++h)
                            for (int64_t w = cw * CUBE_W; w < cw * CUBE_W + CUBE_W && w < W; ++w) {
                                const int64_t n = (t * Hh + h) * W + w;
                                memcpy(xt + (b * S_pad + c * CUBE_TOKENS + slot) * row,
                                       x + (b * S + n) * row, (size_t)row * sizeof(uint16_t));
                                ++slot;
                            }
                    if (vbs && b == 0) vbs[c] = (int32_t)slot;
                }
    }
}

/*
 * Inverse of oracle_tile on the real slots ([STA] Implementation, inverse
 * permutation back to sequential video order); padded slots are dropped.
 */
void oracle_untile(int64_t B, int64_t T, int64_t Hh, int64_t W, int64_t heads, int64_t D,
                   const uint16_t* yt, uint16_t* y) {
    const int64_t nt = ceil_div(T, CUBE_T), nh = ceil_div(Hh, CUBE_H), nw = ceil_div(W, CUBE_W);
    const int64_t N = nt * nh * nw;
    const int64_t row = heads * D;
    const int64_t S = T * Hh * W, S_pad = N * CUBE_TOKENS;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t ct = 0; ct < nt; ++ct)
            for (int64_t ch = 0; ch < nh; ++ch)
                for (int64_t cw = 0; cw < nw; ++cw) {
                    const int64_t c = (ct * nh + ch) * nw + cw;
                    int64_t slot = 0;
                    for (int64_t t = ct * CUBE_T; t < ct * CUBE_T + CUBE_T && t < T; ++t)
                        for (int64_t h = ch * CUBE_H; h < ch * CUBE_H + CUBE_H && h < Hh; ++h)
                            for (int64_t w = cw * CUBE_W; w < cw * CUBE_W + CUBE_W && w < W; ++w) {
                                const int64_t n = (t * Hh + h) * W + w;
                                memcpy(y + (b * S + n) * row,
                                       yt + (b * S_pad + c * CUBE_TOKENS + slot) * row,
                                       (size_t)row * sizeof(uint16_t));
                                ++slot;
                            }
                }
}

/* ---------------------------------------------------------------------- */
/* Coarse stage                                                            */
/* ---------------------------------------------------------------------- */

/*
 * Cube mean-pool ([VSA-AMD] Stage 1: Coarse Selection -- the tokens of a
 * cube are averaged into a single vector that stands for the cube).  xt: [B, N*64, heads, D]; out: [B, heads, N, D].
 * The mean runs over the vbs[c] real tokens of the cube.
 */
void oracle_pool(int64_t B, int64_t N, int64_t heads, int64_t D, const uint16_t* xt,
                 const int32_t* vbs, double* out) {
    const int64_t S_pad = N * CUBE_TOKENS;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < heads; ++h)
            for (int64_t c = 0; c < N; ++c) {
                double* o = out + ((b * heads + h) * N + c) * D;
                const int64_t cnt = vbs[c];
                for (int64_t d = 0; d < D; ++d) {
                    double s = 0.0;
                    for (int64_t r = 0; r < cnt; ++r)
                        s += bf16_to_double(xt[((b * S_pad + c * CUBE_TOKENS + r) * heads + h) * D + d]);
                    o[d] = cnt > 0 ? s / (double)cnt : 0.0;
                }
            }
}

typedef struct {
    double score;
    int32_t index;
} scored_t;

/* Score descending; equal scores go to the lower cube index. */
static int cmp_scored(const void* a, const void* b) {
    const scored_t* x = (const scored_t*)a;
    const scored_t* y = (const scored_t*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->index > y->index) - (x->index < y->index);
}

/*
 * Coarse selection ([VSA-AMD] Stage 1 and Generating Sparsity Patterns:
 * pool Q and K per cube, cube-to-cube scores, Top-K key/value cubes per query
 * cube).
 *
 * qt, kt: [B, N*64, heads, D] bf16 tiled.  scores (nullable): [B, heads, N, N]
 * with scores[i][j] = sm_scale * (q_mean_i . k_mean_j).  topk_idx:
 * [B, heads, N, topk], the first topk entries of the row after a full sort by
 * (score descending, index ascending).
 */
void oracle_coarse(int64_t B, int64_t N, int64_t heads, int64_t D, const uint16_t* qt,
                   const uint16_t* kt, const int32_t* vbs, int64_t topk, double sm_scale,
                   double* scores, int32_t* topk_idx) {
    double* qm = (double*)malloc(sizeof(double) * (size_t)(B * heads * N * D));
    double* km = (double*)malloc(sizeof(double) * (size_t)(B * heads * N * D));
    scored_t* rowbuf = (scored_t*)malloc(sizeof(scored_t) * (size_t)N);
    oracle_pool(B, N, heads, D, qt, vbs, qm);
    oracle_pool(B, N, heads, D, kt, vbs, km);
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < heads; ++h)
            for (int64_t i = 0; i < N; ++i) {
                const double* qi = qm + ((b * heads + h) * N + i) * D;
                for (int64_t j = 0; j < N; ++j) {
                    const double* kj = km + ((b * heads + h) * N + j) * D;
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d) dot += qi[d] * kj[d];
                    rowbuf[j].score = sm_scale * dot;
                    rowbuf[j].index = (int32_t)j;
                    if (scores) scores[((b * heads + h) * N + i) * N + j] = sm_scale * dot;
                }
                qsort(rowbuf, (size_t)N, sizeof(scored_t), cmp_scored);
                int32_t* out = topk_idx + ((b * heads + h) * N + i) * topk;
                for (int64_t t = 0; t < topk; ++t) out[t] = rowbuf[t].index;
            }
    free(rowbuf);
    free(km);
    free(qm);
}

/* ---------------------------------------------------------------------- */
/* Fine stage                                                              */
/* ---------------------------------------------------------------------- */

typedef struct {
    int64_t B, N, heads, D, topk;
    double sm_scale;
    const uint16_t *qt, *kt, *vt;
    const int32_t* topk_idx;
    const int32_t* vbs;
    const int64_t* units; /* unit u -> flat (b*heads + h)*N + i */
    int64_t nunits;
    double* out; /* [nunits, 64, D] */
    double* lse; /* [nunits, 64] */
    int64_t next;
    pthread_mutex_t lock;
} fine_job_t;

/*
 * One query cube of the fine stage ([WAN-VSA] Operator contract:
 * out = softmax(q k_sel^T / sqrt(D)) v_sel over the selected cubes, only the
 * first vbs[c] tokens of each selected cube attended; [VSA-AMD] Sparse
 * Traversal: loop over the query block's K/V block list).
 *
 * For each of the 64 query rows: gather the logits of every attended key,
 * subtract their maximum, exponentiate, normalise, and take the weighted sum
 * of the values.  lse = max + log(sum).
 */
static void fine_unit(const fine_job_t* J, int64_t u, double* logits, double* o_acc) {
    const int64_t flat = J->units[u];
    const int64_t i = flat % J->N;
    const int64_t bh = flat / J->N;
    const int64_t h = bh % J->heads;
    const int64_t b = bh / J->heads;
    const int64_t D = J->D, heads = J->heads, S_pad = J->N * CUBE_TOKENS;
    const int32_t* sel = J->topk_idx + flat * J->topk;
    for (int64_t r = 0; r < CUBE_TOKENS; ++r) {
        const uint16_t* q = J->qt + ((b * S_pad + i * CUBE_TOKENS + r) * heads + h) * D;
        int64_t nkeys = 0;
        for (int64_t t = 0; t < J->topk; ++t) {
            const int64_t j = sel[t];
            for (int64_t s = 0; s < J->vbs[j]; ++s) {
                const uint16_t* k = J->kt + ((b * S_pad + j * CUBE_TOKENS + s) * heads + h) * D;
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(k[d]);
                logits[nkeys++] = J->sm_scale * dot;
            }
        }
        double* o = J->out + (u * CUBE_TOKENS + r) * D;
        double* lse = J->lse + u * CUBE_TOKENS + r;
        if (nkeys == 0) {
            for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            *lse = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t x = 0; x < nkeys; ++x)
            if (logits[x] > m) m = logits[x]; /* ORACLE_ROW_MAX */
        double l = 0.0;
        for (int64_t d = 0; d < D; ++d) o_acc[d] = 0.0;
        int64_t x = 0;
        for (int64_t t = 0; t < J->topk; ++t) {
            const int64_t j = sel[t];
            for (int64_t s = 0; s < J->vbs[j]; ++s, ++x) {
                const double p = exp(logits[x] - m);
                const uint16_t* v = J->vt + ((b * S_pad + j * CUBE_TOKENS + s) * heads + h) * D;
                l += p;
                for (int64_t d = 0; d < D; ++d) o_acc[d] += p * bf16_to_double(v[d]);
            }
        }
        for (int64_t d = 0; d < D; ++d) o[d] = o_acc[d] / l;
        *lse = m + log(l);
    }
}

static void* fine_worker(void* arg) {
    fine_job_t* J = (fine_job_t*)arg;
    double* logits = (double*)malloc(sizeof(double) * (size_t)(J->topk * CUBE_TOKENS + 1));
    double* o_acc = (double*)malloc(sizeof(double) * (size_t)J->D);
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t u = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (u >= J->nunits) break;
        fine_unit(J, u, logits, o_acc);
    }
    free(o_acc);
    free(logits);
    return NULL;
}

/* Threads the fine stage would use for nthreads <= 0: one per online CPU. */
int64_t oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int64_t)n : 1;
}

/*
 * Fine stage over a list of query cubes ("units"), each unit given as the flat
 * index (b*heads + h)*N + i.  out: [nunits, 64, D] fp64, lse: [nunits, 64].
 * Units are independent; nthreads <= 0 uses one worker per online CPU.
 * Returns the number of threads used.
 */
int64_t oracle_fine(int64_t B, int64_t N, int64_t heads, int64_t D, const uint16_t* qt,
                    const uint16_t* kt, const uint16_t* vt, const int32_t* topk_idx,
                    const int32_t* vbs, int64_t topk, double sm_scale, const int64_t* units,
                    int64_t nunits, double* out, double* lse, int64_t nthreads) {
    fine_job_t J;
    J.B = B; J.N = N; J.heads = heads; J.D = D; J.topk = topk; J.sm_scale = sm_scale;
    J.qt = qt; J.kt = kt; J.vt = vt; J.topk_idx = topk_idx; J.vbs = vbs;
    J.units = units; J.nunits = nunits; J.out = out; J.lse = lse; J.next = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > nunits) nthreads = nunits > 0 ? nunits : 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int64_t t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, fine_worker, &J);
    for (int64_t t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return nthreads;
}
