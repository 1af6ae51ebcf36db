/* drive_oracle.c -- exercises the CPU oracle under AddressSanitizer / UndefinedBehaviorSanitizer:
 * plain, GeLU + residual and gated chains (all rows and a row subset, several threads) and the
 * brute-force dependency enumerator on ragged shapes.  Exit status 0 when every call succeeds
 * and the sanitizers report nothing (they abort the process otherwise). */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

int oracle_chain(int64_t M, int32_t num_gemms, const int64_t *dims, const uint16_t *X, const uint16_t *const *W,
                 int32_t gelu, int32_t residual, int32_t gated, const int64_t *rows, int64_t nrows, uint16_t *Y,
                 uint16_t *H, int32_t threads);
int64_t oracle_deps(int64_t M, int64_t n_out, int64_t n_next, int32_t bm_p, int32_t bn_p, int32_t bm_c, int32_t bn_c,
                    int32_t *prod_off, int32_t *prod_tgt, int64_t cap, int32_t *init_count);

static uint16_t *randbf(int64_t n, unsigned *seed)
{
    uint16_t *p = (uint16_t *)malloc((size_t)n * sizeof(uint16_t));
    for (int64_t i = 0; i < n; ++i) {
        *seed = *seed * 1103515245u + 12345u;
        /* small finite bf16 values: sign, exponent 120..127, random mantissa */
        p[i] = (uint16_t)(((*seed >> 31) << 15) | ((120u + ((*seed >> 20) & 7u)) << 7) | ((*seed >> 8) & 0x7fu));
    }
    return p;
}

int main(void)
{
    unsigned seed = 7;
    int fails = 0;
    const int64_t shapes[3][4] = {{37, 24, 40, 24}, {64, 64, 56, 64}, {5, 16, 8, 16}};
    for (int c = 0; c < 3; ++c) {
        const int64_t M = shapes[c][0];
        const int64_t dims[3] = {shapes[c][1], shapes[c][2], shapes[c][3]};
        uint16_t *X = randbf(M * dims[0], &seed);
        uint16_t *Wg = randbf(dims[0] * dims[1], &seed);
        uint16_t *Wu = randbf(dims[0] * dims[1], &seed);
        uint16_t *W2 = randbf(dims[1] * dims[2], &seed);
        uint16_t *Y = (uint16_t *)malloc((size_t)(M * dims[2]) * 2);
        uint16_t *H = (uint16_t *)malloc((size_t)(M * dims[1]) * 2);
        const uint16_t *plain[2] = {Wg, W2};
        const uint16_t *gated[3] = {Wg, Wu, W2};
        int64_t rows[3] = {M - 1, 0, M / 2};
        for (int threads = 1; threads <= 4; threads += 3) {
            fails += oracle_chain(M, 2, dims, X, plain, 0, 0, 0, NULL, 0, Y, H, threads) != 0;
            fails += oracle_chain(M, 2, dims, X, plain, 1, dims[2] == dims[0], 0, rows, 3, Y, H, threads) != 0;
            fails += oracle_chain(M, 2, dims, X, gated, 0, 0, 1, NULL, 0, Y, H, threads) != 0;
        }
        free(X); free(Wg); free(Wu); free(W2); free(Y); free(H);
    }
    const int64_t dshapes[3][7] = {{64, 256, 256, 64, 64, 64, 64}, {300, 384, 512, 128, 64, 128, 128}, {1, 8, 8, 128, 32, 128, 32}};
    for (int c = 0; c < 3; ++c) {
        const int64_t *d = dshapes[c];
        const int64_t P = ((d[0] + d[3] - 1) / d[3]) * ((d[1] + d[4] - 1) / d[4]);
        const int64_t C = ((d[0] + d[5] - 1) / d[5]) * ((d[2] + d[6] - 1) / d[6]);
        int32_t *init = (int32_t *)calloc((size_t)C, 4);
        const int64_t nnz = oracle_deps(d[0], d[1], d[2], (int32_t)d[3], (int32_t)d[4], (int32_t)d[5], (int32_t)d[6], NULL, NULL, 0, init);
        int32_t *off = (int32_t *)calloc((size_t)(P + 1), 4);
        int32_t *tgt = (int32_t *)calloc((size_t)(nnz > 0 ? nnz : 1), 4);
        fails += nnz < 0 || oracle_deps(d[0], d[1], d[2], (int32_t)d[3], (int32_t)d[4], (int32_t)d[5], (int32_t)d[6], off, tgt, nnz, init) != nnz;
        free(init); free(off); free(tgt);
    }
    printf("oracle driver: %d failures\n", fails);
    return fails != 0;
}
