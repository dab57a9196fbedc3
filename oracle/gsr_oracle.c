/*
 * gsr_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the shard-reduction GEMM computes.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load or call it; the product path (the CUDA library) never does, and the two
 * share no code, header or constant.
 *
 * What is computed (pages: "[Kimi-K3] Extend GEMM-RS to GEMM-AR", test section,
 * the reference implementation `_reference`; "[Kimi-K3] AG-GEMM for Sequence
 * Parallelism", Purpose):
 *
 *   AR  Each rank r holds an activation slice X_r (M x K_r) and the matching
 *       weight slice W_r (N x K_r), both K-major like an nn.Linear weight. Its
 *       partial product is P_r = X_r . W_r^T (the test's `torch.mm(x,
 *       weight.T)`), and the all-reduce sums the partials over the ranks:
 *       Y = sum_r P_r, an M x N result.
 *   RS  The same sum, scattered by rows: with rps = ceil(M / R) (the test pads
 *       M up to a multiple of R and gives every rank padded_M / R rows), shard s
 *       receives global rows [s*rps, min(M, (s+1)*rps)).
 *   AG  Each rank holds a row slice A_r (M_r x K) of the activation; the
 *       all-gather concatenates them and one GEMM with W (N x K) follows:
 *       Y = concat_r(A_r) . W^T. Shard r's rows start at sum_{q<r} M_q.
 *   Packed gather (page "Kimi K3 SP: pack the per-layer all-gathers into one",
 *       implementation steps 2-3 and its model.py snippet): rank r holds T
 *       states of M_r rows x H columns (its hidden state, then its auxiliary
 *       states in list order); it concatenates them along the last dimension
 *       (M_r x T*H), one all-gather stacks the ranks' packed rows in rank
 *       order, and the result keeps its first rows_out rows (the token count
 *       before sequence-parallel padding). A copy: no arithmetic.
 *
 * Arithmetic: inputs are bf16 bit patterns; each is widened exactly to double
 * (bf16 is the upper half of an IEEE binary32). Every product and sum is done in
 * fp64. A partial P_r[m,n] sums k = 0 .. K_r-1 in ascending order; the
 * cross-shard sum adds P_0, P_1, ... in ascending r. Nothing is blocked, fused
 * or reordered. Build with -ffp-contract=off so that no FMA changes the
 * rounding between machines.
 */
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> fp64: place the 16 bits above 16 zero bits to form the binary32
 * with the same sign, exponent and (shorter) mantissa, then widen. Exact. */
static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double gsr_oracle_bf16_to_f64(uint16_t bits) { return widen_bf16(bits); }

int gsr_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One rank's partial product at (m, n): sum over k < K_r of X_r[m,k] * W_r[n,k],
 * with X_r row-major M x K_r and W_r row-major N x K_r. */
static double shard_partial(const uint16_t *X_r, const uint16_t *W_r, int64_t K_r,
                            int64_t m, int64_t n)
{
    const uint16_t *x = X_r + m * K_r;
    const uint16_t *w = W_r + n * K_r;
    double p = 0.0;
    for (int64_t k = 0; k < K_r; ++k)
        p += widen_bf16(x[k]) * widen_bf16(w[k]);
    return p;
}

/* The all-reduced element Y[m,n] = P_0[m,n] + P_1[m,n] + ... + P_{R-1}[m,n]. */
static double reduced_element(int R, const int64_t *K_r, const uint16_t *const *X_r,
                              const uint16_t *const *W_r, int64_t m, int64_t n)
{
    double y = shard_partial(X_r[0], W_r[0], K_r[0], m, n);
    for (int r = 1; r < R; ++r)
        y += shard_partial(X_r[r], W_r[r], K_r[r], m, n);
    return y;
}

/* AR: Y (M x N, row-major) = sum_r X_r . W_r^T. */
void gsr_oracle_ar(int64_t M, int64_t N, int R, const int64_t *K_r,
                   const uint16_t *const *X_r, const uint16_t *const *W_r, double *Y)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            Y[m * N + n] = reduced_element(R, K_r, X_r, W_r, m, n);
}

/* AR at listed points: out[i] = Y[rows[i], cols[i]]. */
void gsr_oracle_ar_at(int64_t M, int64_t N, int R, const int64_t *K_r,
                      const uint16_t *const *X_r, const uint16_t *const *W_r,
                      int64_t count, const int64_t *rows, const int64_t *cols,
                      double *out)
{
    (void)M;
    (void)N;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        out[i] = reduced_element(R, K_r, X_r, W_r, rows[i], cols[i]);
}

/* RS row split: shard s owns global rows [first, first + count). */
void gsr_oracle_rs_rows(int64_t M, int R, int s, int64_t *first, int64_t *count)
{
    int64_t rps = (M + R - 1) / R;
    int64_t lo = (int64_t)s * rps;
    int64_t hi = lo + rps;
    if (lo > M) lo = M;
    if (hi > M) hi = M;
    *first = lo;
    *count = hi - lo;
}

/* RS: Y_s[i, n] = Y[first_s + i, n] for the rows shard s owns. Rows of Y_s past
 * its valid count are left untouched (they correspond to the reference's zero
 * padding rows, which hold no output row). */
void gsr_oracle_rs(int64_t M, int64_t N, int R, const int64_t *K_r,
                   const uint16_t *const *X_r, const uint16_t *const *W_r,
                   double *const *Y_s)
{
    for (int s = 0; s < R; ++s) {
        int64_t first, count;
        gsr_oracle_rs_rows(M, R, s, &first, &count);
        double *Ys = Y_s[s];
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t i = 0; i < count; ++i)
            for (int64_t n = 0; n < N; ++n)
                Ys[i * N + n] = reduced_element(R, K_r, X_r, W_r, first + i, n);
    }
}

/* AG element: global row g lies in shard r where sum_{q<r} M_q <= g <
 * sum_{q<=r} M_q; the element is sum_k A_r[g - offset_r, k] * W[n, k]. */
static double gathered_element(int64_t K, int R, const int64_t *M_r,
                               const uint16_t *const *A_r, const uint16_t *W,
                               int64_t g, int64_t n)
{
    int r = 0;
    int64_t offset = 0;
    while (r < R - 1 && g >= offset + M_r[r]) {
        offset += M_r[r];
        ++r;
    }
    const uint16_t *a = A_r[r] + (g - offset) * K;
    const uint16_t *w = W + n * K;
    double y = 0.0;
    for (int64_t k = 0; k < K; ++k)
        y += widen_bf16(a[k]) * widen_bf16(w[k]);
    return y;
}

/* AG: Y ((sum M_r) x N, row-major) = concat_r(A_r) . W^T. */
void gsr_oracle_ag(int64_t N, int64_t K, int R, const int64_t *M_r,
                   const uint16_t *const *A_r, const uint16_t *W, double *Y)
{
    int64_t M = 0;
    for (int r = 0; r < R; ++r)
        M += M_r[r];
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t g = 0; g < M; ++g)
        for (int64_t n = 0; n < N; ++n)
            Y[g * N + n] = gathered_element(K, R, M_r, A_r, W, g, n);
}

/* AG at listed points: out[i] = Y[rows[i], cols[i]], rows being global rows. */
void gsr_oracle_ag_at(int64_t N, int64_t K, int R, const int64_t *M_r,
                      const uint16_t *const *A_r, const uint16_t *W, int64_t count,
                      const int64_t *rows, const int64_t *cols, double *out)
{
    (void)N;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        out[i] = gathered_element(K, R, M_r, A_r, W, rows[i], cols[i]);
}

/* Packed gather: P (rows_out x T*H, row-major) with output row g, for g in rank
 * r's range offset_r <= g < offset_r + M_r (offset_r = sum_{q<r} M_q), equal to
 * the concatenation [S[r][0][g - offset_r, :], ..., S[r][T-1][g - offset_r, :]].
 * S holds R*T pointers, S[r*T + t] being rank r's state t (M_r x H, row-major).
 * The caller guarantees rows_out <= sum_r M_r. Bit patterns are copied as they are. */
void gsr_oracle_pack_gather(int R, const int64_t *M_r, int T, int64_t H,
                            const uint16_t *const *S, int64_t rows_out, uint16_t *P)
{
    (void)R;
    for (int64_t g = 0; g < rows_out; ++g) {
        int r = 0;
        int64_t offset = 0;
        while (g >= offset + M_r[r]) {
            offset += M_r[r];
            ++r;
        }
        for (int t = 0; t < T; ++t) {
            const uint16_t *src = S[r * T + t] + (g - offset) * H;
            uint16_t *dst = P + g * (T * H) + t * H;
            for (int64_t h = 0; h < H; ++h)
                dst[h] = src[h];
        }
    }
}
