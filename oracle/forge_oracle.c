/*
 * forge_oracle.c -- plain fp64 CPU oracle for the fused weight-gradient GEMM
 * with an optimizer step in its epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may link, load or call this file.  Only the test
 * suite, the smoke check and the CPU-baseline leg of the benchmark use it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Every routine is the plain definition, written out with scalar loops in
 * double precision, with no blocking, fusion or reordering beyond what the
 * definition states.  Contractions sum over the token index k in ascending
 * order, starting from 0.0, one product at a time; the file is compiled with
 * -ffp-contract=off so no multiply-add is fused.
 *
 * Sources (the FORGE assessment PR, "docs(audit): FORGE assessment +
 * residency-aware epilogue-fusion track", tessera#565):
 *   - "What's already in tree and easy to miss", first item: the weight
 *     gradient is dRhs = matmul(lhs, dy, transposeA=true), i.e. dW = X^T dY.
 *   - "What's already in tree and easy to miss", third item: K is kept whole
 *     for every output element (tessera.full_k), the legality condition of
 *     FORGE Prop. 1.
 *   - "Math verified, not asserted", P1: per-tile results are exact and do
 *     not depend on the tile partition.
 *   - "Math verified, not asserted", P5: a routed weight that received no
 *     tokens still takes the optimizer step with a zero gradient (decay).
 *   - "Math verified, not asserted", P6, and the fourth "already in tree"
 *     item (bf16 accumulate in f32 then truncf): the gradient feeds the
 *     optimizer state without the bf16 truncation.
 *   - "Claim hygiene on the source": the optimizers are AdamW and SGD.
 * Where the pages do not write a formula out (the AdamW and SGD-momentum
 * variants), this file follows PyTorch's torch.optim.AdamW (decoupled decay
 * scaled by lr, bias correction, eps added after the square root) and
 * torch.optim.SGD (momentum, no dampening, no Nesterov, weight decay added
 * to the gradient).
 *
 * Pins (tests/test_oracle.py): brute-force integer dot products on a 4x4x8
 * case, numpy fp64 X.T @ dY, one-hot token rows, tile-size independence, the
 * AdamW first-step closed form W1 = W0(1 - lr wd) - lr sign(g) at eps = 0,
 * exact beta decay at g = 0, torch CPU float64 AdamW and SGD, the SGD
 * constant-gradient closed form, all 256 e4m3 codes, bf16 decoding and
 * round-to-nearest-even ties.  The grouped routine is pinned by a one-expert
 * call equal to the dense call, zero-token experts equal to pure decay, and
 * invariance under permutation of the expert segments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element types; the numbers match the library's public enum by meaning, not
 * by shared code. */
#define OR_BF16 0
#define OR_E4M3 1
#define OR_F32 2

/* ---- decoding ------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("fn") variant: sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; largest finite
 * magnitude 448; exponent field 0 encodes subnormals 2^-6 * mant/8. */
double oracle_e4m3_to_double(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int mant = c & 0x7;
    double mag;
    if (e == 0xF && mant == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)mant / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, e - 7);
    return s ? -mag : mag;
}

float oracle_f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a double to the nearest bf16 value, ties to even, directly (no
 * intermediate rounding to binary32).  bf16 keeps 8 significant bits and the
 * binary32 exponent range: normal numbers from 2^-126, subnormal quantum
 * 2^-133, largest finite (2 - 2^-7) * 2^127. */
uint16_t oracle_double_to_bf16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    int e;
    double q, r;
    float rf;
    uint32_t u;
    if (isnan(x))
        return 0x7FC0u;
    if (isinf(x))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
    if (e - 1 < -126)
        q = ldexp(1.0, -133); /* subnormal spacing */
    else
        q = ldexp(1.0, e - 8); /* spacing of 8 significant bits */
    r = nearbyint(a / q) * q;  /* a / q is exact (power-of-two scale); RNE */
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80u);
    rf = (float)r; /* exact: r has at most 8 significant bits */
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

static double load_elem(const void* base, int dtype, int64_t i)
{
    if (dtype == OR_BF16)
        return oracle_bf16_to_double(((const uint16_t*)base)[i]);
    if (dtype == OR_E4M3)
        return oracle_e4m3_to_double(((const uint8_t*)base)[i]);
    return (double)((const float*)base)[i];
}

/* ---- fp8 quantisation ------------------------------------------------------ */

/* The e4m3fn code of the finite value nearest to x, ties to the code with an
 * even mantissa; magnitudes from 448 up saturate to 448 and NaN gives 0x7F.
 * Codes 0..126 are the non-negative finite values in increasing order (code
 * 127 is NaN), so the two neighbours of |x| are found by bisection over the
 * decoded values. */
uint8_t oracle_double_to_e4m3(double x)
{
    uint8_t sign;
    double a, vlo, vhi;
    int lo = 0, hi = 126;
    if (isnan(x))
        return 0x7F;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs(x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    while (lo < hi) { /* largest code whose value is <= a */
        int mid = (lo + hi + 1) / 2;
        if (oracle_e4m3_to_double((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    vlo = oracle_e4m3_to_double((uint8_t)lo);
    if (vlo == a)
        return (uint8_t)(sign | lo);
    vhi = oracle_e4m3_to_double((uint8_t)(lo + 1));
    if (a - vlo < vhi - a)
        return (uint8_t)(sign | lo);
    if (vhi - a < a - vlo)
        return (uint8_t)(sign | (lo + 1));
    return (uint8_t)(sign | ((lo & 1) ? lo + 1 : lo)); /* a tie: the even code */
}

/* Per-tensor e4m3 quantisation with an amax scale (the fp8 recipe, s =
 * amax / 448): amax = max |x| over the n inputs (fp32 values or bf16
 * patterns; NaN entries are skipped), s = amax / 448 divided in float (1 when
 * amax is 0), and each code is the e4m3 value nearest to the float quotient
 * x / s. */
void oracle_quantize_e4m3(const void* x, int dtype, int64_t n, uint8_t* codes, float* scale)
{
    double amax = 0.0;
    float s;
    for (int64_t i = 0; i < n; ++i) {
        const double a = fabs(load_elem(x, dtype, i));
        if (a > amax)
            amax = a;
    }
    s = amax > 0.0 ? (float)amax / 448.0f : 1.0f;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const float t = (float)load_elem(x, dtype, i) / s;
        codes[i] = oracle_double_to_e4m3((double)t);
    }
    *scale = s;
}

void oracle_decode(const void* src, int dtype, int64_t n, double* dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = load_elem(src, dtype, i);
}

void oracle_round_bf16(const double* src, int64_t n, uint16_t* dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_double_to_bf16(src[i]);
}

/* ---- the contraction ------------------------------------------------------ */

/*
 * g[n][m] = sX * sdY * sum_{k = k_begin}^{k_end - 1} X[k][n] * dY[k][m]
 *
 * X is [K_rows, N] row-major, dY is [K_rows, M] row-major, both of element
 * type in_dtype (bf16 or e4m3).  The sum over k runs in ascending order from
 * 0.0; the two per-tensor scales multiply the finished sum (they are 1 for
 * bf16).  Only the rows n listed in `rows` (nrows of them; all N rows in
 * order when rows is NULL) are produced, into G[i][m], i the position in the
 * list.  An empty range (k_begin == k_end) gives g = 0.
 */
void oracle_wgrad_rows(const void* X, const void* dY, int in_dtype,
                       int64_t M, int64_t N, int64_t k_begin, int64_t k_end,
                       double sX, double sdY, const int64_t* rows,
                       int64_t nrows, double* G)
{
    const double s = sX * sdY;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t n = rows ? rows[i] : i;
        double* g = G + i * M;
        for (int64_t m = 0; m < M; ++m)
            g[m] = 0.0;
        /* For each element the products are added in ascending k, exactly as
         * in the element-by-element definition; looping k outside m only
         * walks dY row by row. */
        for (int64_t k = k_begin; k < k_end; ++k) {
            const double x = load_elem(X, in_dtype, k * N + n);
            for (int64_t m = 0; m < M; ++m)
                g[m] += x * load_elem(dY, in_dtype, k * M + m);
        }
        for (int64_t m = 0; m < M; ++m)
            g[m] = s * g[m];
    }
}

/* The unfused lowering the fused path is measured against (P6, and "What's
 * already in tree and easy to miss": the matmul lowering accumulates bf16
 * products in f32 and then truncates to bf16).  Each product of two decoded
 * inputs is exact in float (bf16 and e4m3 significands are short enough), and
 * the products are added in ascending k into a float accumulator, one rounding
 * per addition; the sum is scaled by sX * sdY in float and, with `truncate`,
 * rounded to bf16 (nearest, ties to even).  Results are widened to double. */
void oracle_wgrad_rows_lowered(const void* X, const void* dY, int in_dtype,
                               int64_t M, int64_t N, int64_t k_begin, int64_t k_end,
                               float sX, float sdY, const int64_t* rows, int64_t nrows,
                               int truncate, double* G)
{
    const float s = sX * sdY;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t n = rows ? rows[i] : i;
        float* acc = (float*)calloc((size_t)(M > 0 ? M : 1), sizeof(float));
        double* g = G + i * M;
        for (int64_t k = k_begin; k < k_end; ++k) {
            const float x = (float)load_elem(X, in_dtype, k * N + n);
            for (int64_t m = 0; m < M; ++m) {
                const float p = x * (float)load_elem(dY, in_dtype, k * M + m);
                acc[m] = acc[m] + p;
            }
        }
        for (int64_t m = 0; m < M; ++m) {
            const float r = acc[m] * s;
            g[m] = truncate ? oracle_bf16_to_double(oracle_double_to_bf16((double)r)) : (double)r;
        }
        free(acc);
    }
}

/* The input gradient on the other side of the backward pass (the dX that
 * must read W before the in-place update, "Math verified, not asserted", P1):
 * dX[k][n] = sum over m of dY[k][m] * Wb[n][m], with dY [K, M] and the weight
 * Wb [N, M] both bf16 patterns, summed in ascending m in double, for the
 * token rows `rows` (or all K rows when rows is NULL).  G is [nrows, N]. */
void oracle_dgrad_rows(const uint16_t* dY, const uint16_t* Wb, int64_t M, int64_t N,
                       const int64_t* rows, int64_t nrows, double* G)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t k = rows ? rows[i] : i;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m)
                acc += oracle_bf16_to_double(dY[k * M + m]) * oracle_bf16_to_double(Wb[n * M + m]);
            G[i * N + n] = acc;
        }
    }
}

/* One output element, by the definition (used by the tiled pin and by the
 * sampled checks). */
double oracle_wgrad_elem(const void* X, const void* dY, int in_dtype,
                         int64_t M, int64_t N, int64_t k_begin, int64_t k_end,
                         double sX, double sdY, int64_t n, int64_t m)
{
    double acc = 0.0;
    for (int64_t k = k_begin; k < k_end; ++k)
        acc += load_elem(X, in_dtype, k * N + n) * load_elem(dY, in_dtype, k * M + m);
    return (sX * sdY) * acc;
}

/* ---- the optimizer steps -------------------------------------------------- */

static double load_state(const void* p, int state_dtype, int64_t i)
{
    if (state_dtype == OR_BF16)
        return oracle_bf16_to_double(((const uint16_t*)p)[i]);
    return (double)((const float*)p)[i];
}

static void store_state(void* p, int state_dtype, int64_t i, double x)
{
    if (state_dtype == OR_BF16)
        ((uint16_t*)p)[i] = oracle_double_to_bf16(x);
    else
        ((float*)p)[i] = (float)x; /* C conversion: round to nearest even */
}

/*
 * AdamW, PyTorch semantics, one element:
 *   W'  = W (1 - lr wd)                          decoupled weight decay
 *   m'  = b1 m + (1 - b1) g
 *   v'  = b2 v + (1 - b2) g^2
 *   bc1 = 1 - b1^t,  bc2 = 1 - b2^t               bias corrections
 *   W'' = W' - lr (m' / bc1) / (sqrt(v' / bc2) + eps)
 * W'' is rounded to binary32; m' and v' to the state type.  The update of W
 * uses the unrounded m' and v'.  The unrounded values are also returned
 * (W_exact, m_exact, v_exact may be NULL).
 */
static void adamw_elem(double g, double w, double m, double v, double lr,
                       double b1, double b2, double eps, double wd,
                       double bc1, double bc2, double* w_out, double* m_out,
                       double* v_out)
{
    double w1 = w * (1.0 - lr * wd);
    double m1 = b1 * m + (1.0 - b1) * g;
    double v1 = b2 * v + (1.0 - b2) * g * g;
    double w2 = w1 - lr * (m1 / bc1) / (sqrt(v1 / bc2) + eps);
    *w_out = w2;
    *m_out = m1;
    *v_out = v1;
}

void oracle_adamw(int64_t P, const double* G, const float* W, const void* m,
                  const void* v, int state_dtype, double lr, double b1,
                  double b2, double eps, double wd, int64_t step,
                  float* W_out, void* m_out, void* v_out, double* W_exact,
                  double* m_exact, double* v_exact)
{
    const double bc1 = 1.0 - pow(b1, (double)step);
    const double bc2 = 1.0 - pow(b2, (double)step);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < P; ++i) {
        double w2, m1, v1;
        adamw_elem(G[i], (double)W[i], load_state(m, state_dtype, i),
                   load_state(v, state_dtype, i), lr, b1, b2, eps, wd, bc1,
                   bc2, &w2, &m1, &v1);
        W_out[i] = (float)w2;
        store_state(m_out, state_dtype, i, m1);
        store_state(v_out, state_dtype, i, v1);
        if (W_exact) W_exact[i] = w2;
        if (m_exact) m_exact[i] = m1;
        if (v_exact) v_exact[i] = v1;
    }
}

/*
 * SGD with momentum, PyTorch semantics (dampening 0, no Nesterov):
 *   g'   = g + wd W
 *   buf' = mu buf + g'        (on the first step buf = 0, so buf' = g')
 *   W'   = W - lr buf'
 */
void oracle_sgdm(int64_t P, const double* G, const float* W, const void* buf,
                 int state_dtype, double lr, double mu, double wd,
                 float* W_out, void* buf_out, double* W_exact,
                 double* buf_exact)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < P; ++i) {
        double w = (double)W[i];
        double g1 = G[i] + wd * w;
        double b1 = mu * load_state(buf, state_dtype, i) + g1;
        double w1 = w - lr * b1;
        W_out[i] = (float)w1;
        store_state(buf_out, state_dtype, i, b1);
        if (W_exact) W_exact[i] = w1;
        if (buf_exact) buf_exact[i] = b1;
    }
}

/* ---- fused per tile (the partition-independence statement) ---------------- */

/*
 * dW = X^T dY followed by AdamW, evaluated tile by tile: the N x M output is
 * cut into tile_n x tile_m tiles (0 means the whole extent) and each tile's
 * gradient is formed over the whole K and consumed by the optimizer before
 * the next tile.  P1 says the result cannot depend on the tiling.
 */
void oracle_wgrad_adamw_tiled(const void* X, const void* dY, int in_dtype,
                              int64_t M, int64_t N, int64_t K, double sX,
                              double sdY, const float* W, const void* m,
                              const void* v, int state_dtype, double lr,
                              double b1, double b2, double eps, double wd,
                              int64_t step, int64_t tile_n, int64_t tile_m,
                              float* W_out, void* m_out, void* v_out)
{
    const double bc1 = 1.0 - pow(b1, (double)step);
    const double bc2 = 1.0 - pow(b2, (double)step);
    const int64_t tn = tile_n > 0 ? tile_n : N;
    const int64_t tm = tile_m > 0 ? tile_m : M;
    for (int64_t n0 = 0; n0 < N; n0 += tn)
        for (int64_t m0 = 0; m0 < M; m0 += tm)
            for (int64_t n = n0; n < n0 + tn && n < N; ++n)
                for (int64_t mm = m0; mm < m0 + tm && mm < M; ++mm) {
                    const int64_t i = n * M + mm;
                    double w2, m1, v1;
                    double g = oracle_wgrad_elem(X, dY, in_dtype, M, N, 0, K,
                                                 sX, sdY, n, mm);
                    adamw_elem(g, (double)W[i], load_state(m, state_dtype, i),
                               load_state(v, state_dtype, i), lr, b1, b2, eps,
                               wd, bc1, bc2, &w2, &m1, &v1);
                    W_out[i] = (float)w2;
                    store_state(m_out, state_dtype, i, m1);
                    store_state(v_out, state_dtype, i, v1);
                }
}

/* ---- grouped (per-expert ragged token counts) ----------------------------- */

/*
 * E experts.  Expert e owns the packed token rows [off[e], off[e+1]) of X
 * ([T, N]) and dY ([T, M]) and the parameter block e of W, m, v ([E, N, M]).
 * Each expert's gradient is its own X_e^T dY_e over its rows only; an expert
 * with no rows gets g = 0 and still takes the AdamW step (pure decay of m, v
 * and the decoupled weight decay of W).  Only the rows listed in `rows`
 * (nrows of them; all N when NULL) of every expert are produced; W_out,
 * m_out, v_out and the exact arrays are [E, nrows, M].
 */
void oracle_grouped_adamw(const void* X, const void* dY, int in_dtype,
                          const int64_t* off, int64_t E, int64_t M, int64_t N,
                          double sX, double sdY, const float* W,
                          const void* m, const void* v, int state_dtype,
                          double lr, double b1, double b2, double eps,
                          double wd, int64_t step, const int64_t* rows,
                          int64_t nrows, double* G_scratch, float* W_out,
                          void* m_out, void* v_out, double* W_exact,
                          double* m_exact, double* v_exact)
{
    const size_t esz = state_dtype == OR_BF16 ? 2 : 4;
    for (int64_t e = 0; e < E; ++e) {
        const int64_t P = nrows * M;
        /* gather this expert's selected parameter rows */
        const int64_t pbase = e * N * M;
        float* We = W_out + e * P;
        char* mo = (char*)m_out + (size_t)(e * P) * esz;
        char* vo = (char*)v_out + (size_t)(e * P) * esz;
        oracle_wgrad_rows(X, dY, in_dtype, M, N, off[e], off[e + 1], sX, sdY,
                          rows, nrows, G_scratch);
        {
            const double bc1 = 1.0 - pow(b1, (double)step);
            const double bc2 = 1.0 - pow(b2, (double)step);
            for (int64_t i = 0; i < nrows; ++i) {
                const int64_t n = rows ? rows[i] : i;
                for (int64_t mm = 0; mm < M; ++mm) {
                    const int64_t src = pbase + n * M + mm;
                    const int64_t dst = i * M + mm;
                    double w2, m1, v1;
                    adamw_elem(G_scratch[dst], (double)W[src],
                               load_state(m, state_dtype, src),
                               load_state(v, state_dtype, src), lr, b1, b2,
                               eps, wd, bc1, bc2, &w2, &m1, &v1);
                    We[dst] = (float)w2;
                    store_state(mo, state_dtype, dst, m1);
                    store_state(vo, state_dtype, dst, v1);
                    if (W_exact) W_exact[e * P + dst] = w2;
                    if (m_exact) m_exact[e * P + dst] = m1;
                    if (v_exact) v_exact[e * P + dst] = v1;
                }
            }
        }
    }
}
