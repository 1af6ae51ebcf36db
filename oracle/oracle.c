/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the CTA-pipelined GEMM chain.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this file.
 * Its only users are the tests, the smoke check and the timed CPU-baseline leg of the bench.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Source of the arithmetic: "CTA-Pipelining: A Latency-Oriented Spatial Scaling Method for
 * Multi-GPU Systems" (arXiv 2607.07862).
 *   - Running example: a two-layer GEMM whose first output H is consumed directly by the
 *     second GEMM, Y = (X * A) * B  (section III, integration into CUTLASS GEMMs; section IV,
 *     tensor-parallel comparison, which writes the MLP as Y = XAB).
 *   - Precision: BF16 inputs and outputs, FP32 tensor-core accumulator (section III, protocol
 *     overhead set-up, Fig. 2).
 *   - CTA-pipelining changes only which CTA runs which tile and when; the GEMM body is left
 *     unchanged (section III-C, Fig. 2b discussion; abstract), so the values it produces are
 *     those of the plain chain below.
 *   - Dependency arrays are built from the static tile dataflow of the GEMM: a consumer CTA
 *     consumes one or more input tiles and produces one output tile (section III-A,
 *     execution model paragraph).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - fp32 accumulation runs in ascending k order; a bf16*bf16 product is exact in fp32, so
 *     only the order of the additions can differ from the GPU.
 *   - Every fp32 -> bf16 conversion rounds to nearest, ties to even; NaN stays NaN (quiet).
 *   - Chains with the GeLU option apply GeLU (tanh form) to the fp32 accumulator of every GEMM
 *     before rounding; with the residual option the last stage adds the chain input X (as fp32)
 *     to that value and rounds once.
 *   - Gated chains (the SwiGLU MLP block the paper's critique names as the test of its claim:
 *     an activation between the two matrix multiplies) compute the first stage from two weight
 *     matrices, H = SiLU(X Wg) * (X Wu), the gated linear unit with the Swish-1 gate of Shazeer,
 *     "GLU Variants Improve Transformer" (2020, eq. 6): both accumulators in fp32, SiLU and the
 *     product in double, one rounding to bf16.  Later stages are unchanged (GeLU, if asked for,
 *     applies to them only).
 *   - Dependency granularity is the whole tile: a consumer tile needs every producer tile that
 *     owns any element of the rows it reads (it reads all columns, since the next GEMM's
 *     reduction dimension is the producer's column dimension).
 *
 * Build: gcc -O2 -fPIC -shared -std=c11 -ffp-contract=off -pthread (no fast-math).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                                               */
/* ------------------------------------------------------------------------------------------ */

/* A bf16 value is the upper 16 bits of an IEEE-754 binary32 value. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest-even from binary32 to bf16: add half an ulp of the kept part, plus one if
 * the kept part is odd (so exact ties go to the even neighbour), then truncate.  NaN inputs
 * keep their sign and top payload bits and are forced quiet so truncation cannot make them
 * infinite. */
static uint16_t float_to_bf16_bits_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

uint16_t oracle_f32_to_bf16(float f) { return float_to_bf16_bits_rne(f); }
float oracle_bf16_to_f32(uint16_t b) { return bf16_bits_to_float(b); }

void oracle_round_bf16(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = float_to_bf16_bits_rne(in[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* GeLU, tanh form: 0.5 x (1 + tanh( sqrt(2/pi) (x + 0.044715 x^3) )), evaluated in double.    */
/* ------------------------------------------------------------------------------------------ */
double oracle_gelu_tanh(double x)
{
    const double pi = 3.14159265358979323846;
    const double c = sqrt(2.0 / pi);
    return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

/* ------------------------------------------------------------------------------------------ */
/* SiLU (Swish-1): x * sigmoid(x) = x / (1 + e^-x), evaluated in double.                       */
/* ------------------------------------------------------------------------------------------ */
double oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

/* ------------------------------------------------------------------------------------------ */
/* The chain, one row at a time.  Row i of every intermediate depends only on row i of X.      */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    int64_t M;
    int32_t num_gemms;
    const int64_t *dims;      /* num_gemms + 1 entries: dims[0] = K of the first GEMM        */
    const uint16_t *X;        /* M x dims[0], row-major bf16 bits                            */
    const uint16_t *const *W; /* W[s + gated]: dims[s] x dims[s+1], row-major bf16 bits      */
    int32_t gelu;             /* apply GeLU(tanh) to every (ungated) GEMM's accumulator      */
    int32_t gated;            /* first stage: H = SiLU(X W[0]) * (X W[1])                    */
    int32_t residual;         /* add X to the last stage (requires dims[last] == dims[0])    */
    const int64_t *rows;      /* rows to compute (NULL: 0..M-1)                              */
    int64_t nrows;
    uint16_t *Y;              /* nrows x dims[num_gemms]                                     */
    uint16_t *H;              /* optional: nrows x dims[1], the first intermediate           */
    int64_t row_begin, row_end; /* this worker's slice of [0, nrows)                         */
    int64_t maxdim;
    int32_t status;
} chain_job;

/* acc[n] = sum over k = 0, 1, ..., K-1 of a[k] * B[k][n], in fp32, in that order. */
static void row_times_matrix(const uint16_t *a, int64_t K, const uint16_t *B, int64_t N, float *acc)
{
    for (int64_t n = 0; n < N; ++n)
        acc[n] = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        const float ak = bf16_bits_to_float(a[k]);
        const uint16_t *brow = B + k * N;
        for (int64_t n = 0; n < N; ++n)
            acc[n] += ak * bf16_bits_to_float(brow[n]);
    }
}

static void *chain_worker(void *arg)
{
    chain_job *job = (chain_job *)arg;
    uint16_t *cur = (uint16_t *)malloc((size_t)job->maxdim * sizeof(uint16_t));
    uint16_t *nxt = (uint16_t *)malloc((size_t)job->maxdim * sizeof(uint16_t));
    float *acc = (float *)malloc((size_t)job->maxdim * sizeof(float));
    float *up = (float *)malloc((size_t)job->maxdim * sizeof(float));
    if (!cur || !nxt || !acc || !up) {
        job->status = -2;
        free(cur); free(nxt); free(acc); free(up);
        return NULL;
    }
    const int32_t S = job->num_gemms;
    const int64_t d_in = job->dims[0];
    const int64_t d_out = job->dims[S];
    for (int64_t r = job->row_begin; r < job->row_end; ++r) {
        const int64_t i = job->rows ? job->rows[r] : r;
        const uint16_t *xrow = job->X + i * d_in;
        memcpy(cur, xrow, (size_t)d_in * sizeof(uint16_t));
        for (int32_t s = 0; s < S; ++s) {
            const int64_t K = job->dims[s], N = job->dims[s + 1];
            const int gated = job->gated && s == 0;
            row_times_matrix(cur, K, job->W[s == 0 ? 0 : s + job->gated], N, acc);
            if (gated)
                row_times_matrix(cur, K, job->W[1], N, up);
            const int last = (s == S - 1);
            for (int64_t n = 0; n < N; ++n) {
                float v = acc[n];
                if (gated)
                    v = (float)(oracle_silu((double)v) * (double)up[n]);
                else if (job->gelu)
                    v = (float)oracle_gelu_tanh((double)v);
                if (last && job->residual)
                    v = v + bf16_bits_to_float(xrow[n]);
                nxt[n] = float_to_bf16_bits_rne(v);
            }
            if (s == 0 && job->H)
                memcpy(job->H + r * job->dims[1], nxt, (size_t)N * sizeof(uint16_t));
            uint16_t *t = cur; cur = nxt; nxt = t;
        }
        memcpy(job->Y + r * d_out, cur, (size_t)d_out * sizeof(uint16_t));
    }
    free(cur); free(nxt); free(acc); free(up);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments, -2 on host allocation failure. */
int oracle_chain(int64_t M, int32_t num_gemms, const int64_t *dims, const uint16_t *X,
                 const uint16_t *const *W, int32_t gelu, int32_t residual, int32_t gated,
                 const int64_t *rows, int64_t nrows, uint16_t *Y, uint16_t *H, int32_t threads)
{
    if (M < 0 || num_gemms < 1 || !dims || !X || !W || !Y)
        return -1;
    if (residual && dims[num_gemms] != dims[0])
        return -1;
    if (!rows)
        nrows = M;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M)
            return -1;
    int64_t maxdim = 0;
    for (int32_t s = 0; s <= num_gemms; ++s) {
        if (dims[s] <= 0)
            return -1;
        if (dims[s] > maxdim)
            maxdim = dims[s];
    }
    if (threads < 1)
        threads = 1;
    if (threads > 256)
        threads = 256;
    if ((int64_t)threads > nrows)
        threads = nrows > 0 ? (int32_t)nrows : 1;

    chain_job jobs[256];
    pthread_t tid[256];
    int started[256];
    for (int32_t t = 0; t < threads; ++t) {
        chain_job j = {M, num_gemms, dims, X, W, gelu, gated != 0, residual, rows, nrows, Y, H,
                       nrows * t / threads, nrows * (t + 1) / threads, maxdim, 0};
        jobs[t] = j;
        started[t] = (threads > 1) && pthread_create(&tid[t], NULL, chain_worker, &jobs[t]) == 0;
        if (!started[t])
            chain_worker(&jobs[t]);
    }
    int status = 0;
    for (int32_t t = 0; t < threads; ++t) {
        if (started[t])
            pthread_join(tid[t], NULL);
        if (jobs[t].status)
            status = jobs[t].status;
    }
    return status;
}

/* ------------------------------------------------------------------------------------------ */
/* Dependency array by brute-force tile-overlap enumeration.                                  */
/*                                                                                            */
/* Producer tiles cut the producer output (M x Nout) into BMp x BNp rectangles, numbered      */
/* row-major over the tile grid.  Consumer tiles cut the consumer output (M x Nnext) into     */
/* BMc x BNc rectangles, numbered the same way.  Consumer tile (mc, nc) reads rows            */
/* [mc*BMc, min(M, (mc+1)*BMc)) of the producer output, across all Nout columns.              */
/*                                                                                            */
/* For every element the consumer reads, the owning producer tile is found by scanning the    */
/* list of producer rectangles (the last hit is tried first, which only saves time).  Output: */
/*   prod_off[P+1], prod_tgt[nnz]: for each producer, the consumers that need it, ascending;  */
/*   init_count[C]: how many producer tiles each consumer needs.                              */
/* Returns nnz >= 0, -1 on bad arguments or too little room, -2 on allocation failure.        */
/* ------------------------------------------------------------------------------------------ */
typedef struct { int64_t r0, r1, c0, c1; } rect;

int64_t oracle_deps(int64_t M, int64_t Nout, int64_t Nnext, int32_t BMp, int32_t BNp,
                    int32_t BMc, int32_t BNc, int32_t *prod_off, int32_t *prod_tgt,
                    int64_t tgt_cap, int32_t *init_count)
{
    if (M <= 0 || Nout <= 0 || Nnext <= 0 || BMp <= 0 || BNp <= 0 || BMc <= 0 || BNc <= 0)
        return -1;
    /* list the producer rectangles by walking the output */
    int64_t P = 0;
    for (int64_t r = 0; r < M; r += BMp)
        for (int64_t c = 0; c < Nout; c += BNp)
            ++P;
    int64_t C = 0;
    for (int64_t r = 0; r < M; r += BMc)
        for (int64_t c = 0; c < Nnext; c += BNc)
            ++C;
    if (P * C > ((int64_t)1 << 28))
        return -1;
    rect *prod = (rect *)malloc((size_t)P * sizeof(rect));
    rect *cons = (rect *)malloc((size_t)C * sizeof(rect));
    unsigned char *need = (unsigned char *)calloc((size_t)(P * C), 1);
    if (!prod || !cons || !need) {
        free(prod); free(cons); free(need);
        return -2;
    }
    int64_t p = 0;
    for (int64_t r = 0; r < M; r += BMp)
        for (int64_t c = 0; c < Nout; c += BNp) {
            rect t = {r, r + BMp < M ? r + BMp : M, c, c + BNp < Nout ? c + BNp : Nout};
            prod[p++] = t;
        }
    int64_t q = 0;
    for (int64_t r = 0; r < M; r += BMc)
        for (int64_t c = 0; c < Nnext; c += BNc) {
            rect t = {r, r + BMc < M ? r + BMc : M, c, c + BNc < Nnext ? c + BNc : Nnext};
            cons[q++] = t;
        }

    for (int64_t ci = 0; ci < C; ++ci) {
        int64_t hit = 0;
        /* every element of the producer output this consumer reads */
        for (int64_t i = cons[ci].r0; i < cons[ci].r1; ++i)
            for (int64_t j = 0; j < Nout; ++j) {
                const rect *h = &prod[hit];
                if (!(i >= h->r0 && i < h->r1 && j >= h->c0 && j < h->c1)) {
                    for (hit = 0; hit < P; ++hit) {
                        h = &prod[hit];
                        if (i >= h->r0 && i < h->r1 && j >= h->c0 && j < h->c1)
                            break;
                    }
                    if (hit == P) { /* unreachable when the rectangles tile the output */
                        free(prod); free(cons); free(need);
                        return -1;
                    }
                }
                need[hit * C + ci] = 1;
            }
    }

    int64_t nnz = 0;
    for (int64_t ci = 0; ci < C; ++ci) {
        int32_t n = 0;
        for (int64_t pi = 0; pi < P; ++pi)
            n += need[pi * C + ci];
        if (init_count)
            init_count[ci] = n;
        nnz += n;
    }
    if (prod_off && prod_tgt) {
        if (nnz > tgt_cap) {
            free(prod); free(cons); free(need);
            return -1;
        }
        int64_t e = 0;
        for (int64_t pi = 0; pi < P; ++pi) {
            prod_off[pi] = (int32_t)e;
            for (int64_t ci = 0; ci < C; ++ci)
                if (need[pi * C + ci])
                    prod_tgt[e++] = (int32_t)ci;
        }
        prod_off[P] = (int32_t)e;
    }
    free(prod); free(cons); free(need);
    return nnz;
}
