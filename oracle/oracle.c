/*
 * Oracle for the tile-scheduled GEMM, the grid-stride int16 copy and the
 * jagged row copy.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path and is deliberately plain and slow: a sequential (i, j, k)
 * triple loop accumulating in double precision, a scalar copy loop, and a
 * round-to-nearest-even bf16 encoder written from the IEEE 754 definition.
 *
 * What the method computes (CUTLASS TS "Pipeline Groups", Overview: the GEMM
 * mainloop resource graph gmem_ab -> smem_a, smem_b -> tmem_c -> gmem_d; and
 * TS "Resources", the scale_d reset: the first MMA of a work tile overwrites
 * the accumulator, later ones accumulate) is, whatever the tile order, the
 * plain product
 *
 *     D[i][j] = sum_{k<K} a(A[i][k]) * b(B[j][k])
 *
 * with A stored [M][K] and B stored [N][K], both K-major (row i of A and row
 * j of B are contiguous along k).  a() and b() decode bf16 exactly; every
 * bf16 x bf16 product is exact in double.
 *
 * The copy follows TS "Resources", the int16 example (InputGmemResource.get_item /
 * OutputGmemResource.set_item): dst[gid] = src[gid] for every gid < n.
 *
 * The jagged row copy follows TS "Schedules": Dynamic Domain (work tile t runs
 * its loop from offsets[t] to offsets[t + 1]) and Skippable Tiles (a per-tile
 * predicate drops the copy of a tile; tiles past the row count are such tiles
 * of the oversubscribed copy queue).  Whatever the queue, the result is: every
 * row r < rows that is not skipped has dst[i] = src[i] for its i, and no
 * other element of dst changes.
 *
 * The static persistent assignment follows "Cluster Launch Control", section
 * on the limits of the static persistent scheduler: with W workers, worker w
 * takes tiles w, w + W, w + 2W, ...
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* bf16 is the upper half of an IEEE binary32: widen, then convert exactly. */
double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, binary32 exponent
 * range), ties to even.  Overflow goes to infinity, NaN stays NaN (quiet),
 * the sign of zero is kept, and results below 2^-126 are bf16 subnormals
 * (multiples of 2^-133). */
uint16_t oracle_f64_to_bf16_rne(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);           /* a in [2^(e-1), 2^e) */
    int binade = e - 1;
    int ulp_exp = binade < -126 ? -133 : binade - 7;
    double q = ldexp(a, -ulp_exp); /* exact: scaling by a power of two */
    double fl = floor(q);
    double rem = q - fl;           /* exact */
    double r = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) r = fl + 1.0;
    double y = ldexp(r, ulp_exp);
    if (y >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    float f = (float)y;            /* exact: y has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

void oracle_bf16_decode(const uint16_t *in, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f64(in[i]);
}

void oracle_bf16_encode(const double *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16_rne(in[i]);
}

/* D[i - row0][j] for rows row0 <= i < row1, all j < N.
 * A: [M][lda] bf16 bits, B: [N][ldb] bf16 bits, D: [row1 - row0][ldd] doubles.
 * `absolute` != 0 computes sum_k |a||b| instead (the scale of the error bound).
 * Rows are independent; nthreads > 1 splits them across OpenMP threads. */
void oracle_gemm_f64(const uint16_t *A, const uint16_t *B, double *D,
                     int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldd,
                     int64_t row0, int64_t row1, int absolute, int nthreads) {
    (void)M;
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t i = row0; i < row1; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = oracle_bf16_to_f64(A[i * lda + k]);
                double b = oracle_bf16_to_f64(B[j * ldb + k]);
                s += absolute ? fabs(a) * fabs(b) : a * b;
            }
            D[(i - row0) * ldd + j] = s;
        }
    }
}

/* The same sum for `count` individual entries (ii[t], jj[t]). */
void oracle_gemm_entries_f64(const uint16_t *A, const uint16_t *B,
                             int64_t K, int64_t lda, int64_t ldb,
                             const int64_t *ii, const int64_t *jj, int64_t count,
                             double *out, double *out_abs, int nthreads) {
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t t = 0; t < count; ++t) {
        double s = 0.0, sa = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = oracle_bf16_to_f64(A[ii[t] * lda + k]);
            double b = oracle_bf16_to_f64(B[jj[t] * ldb + k]);
            s += a * b;
            sa += fabs(a) * fabs(b);
        }
        out[t] = s;
        if (out_abs) out_abs[t] = sa;
    }
}

/* dst[gid] = src[gid] for gid < n, one element at a time. */
void oracle_copy_i16(const int16_t *src, int16_t *dst, int64_t n) {
    for (int64_t gid = 0; gid < n; ++gid) dst[gid] = src[gid];
}

/* For each row r < rows with skip == NULL or skip[r] == 0: dst[i] = src[i]
 * for offsets[r] <= i < offsets[r + 1].  A row whose bounds are not
 * 0 <= offsets[r] <= offsets[r + 1] <= n is left alone.  Returns the first
 * such row, or -1 if every row examined was valid. */
int64_t oracle_copy_rows_i16(const int16_t *src, int16_t *dst, int64_t n, const int64_t *offsets, int64_t rows,
                             const uint8_t *skip) {
    int64_t first_bad = -1;
    for (int64_t r = 0; r < rows; ++r) {
        if (skip && skip[r]) continue;
        const int64_t b = offsets[r], e = offsets[r + 1];
        if (b < 0 || e < b || e > n) {
            if (first_bad < 0) first_bad = r;
            continue;
        }
        for (int64_t i = b; i < e; ++i) dst[i] = src[i];
    }
    return first_bad;
}

/* owner[t] = the worker that the static grid-stride rule gives tile t. */
void oracle_static_owner(int64_t num_tiles, int64_t num_workers, int64_t *owner) {
    for (int64_t w = 0; w < num_workers; ++w)
        for (int64_t t = w; t < num_tiles; t += num_workers) owner[t] = w;
}
