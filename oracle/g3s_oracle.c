/*
 * g3s_oracle.c -- fp64 CPU oracle for fused sparse graph attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (per destination row i and head h, plain definitions in
 * double precision; inputs are read from the same stored bytes the GPU reads
 * and widened exactly):
 *
 *   Standard 3S (Fused3S abstract: "SDDMM, softmax normalization, SpMM";
 *   sciencestack.ai/paper/2505.08098, Abstract):
 *       l_j   = (sum_f q_i[h,f] * k_j[h,f]) / sqrt(d)        over in-edges j
 *       m     = max_j l_j
 *       w_j   = exp(l_j - m)
 *       O_i^h = sum_j w_j v_j[h,:] / sum_j w_j ;  O_i^h = 0 when i has no in-edge
 *   The max subtraction only guards the exponent range; the value is the plain
 *   softmax.
 *
 *   RTMScore edge-modulated variant (stondelli.it/articles/gattn-triton,
 *   section "Fusing the full graph attention", the eager torch_attn listing
 *   and the Background list), in the page's order:
 *       t     = clamp(q_i * k_j / sqrt(d), -5, 5)    elementwise over f
 *               (the elementwise clamp is skipped when elementwise_clamp == 0)
 *       u     = t * e_ij                             elementwise
 *       eout  = u                                    (the updated edge feature)
 *       l     = sum_f u
 *       s     = exp(clamp(l, -5, 5))
 *       O_i^h = sum_j s_j v_j[h,:] / (sum_j s_j + eps)
 *
 *   Weighted aggregation (the article's normalised scatter-add, section
 *   "Optimizing the scatter add in Triton" and "Using the CSC index for fast
 *   edge lookup"; the POPCORNBENCH CSR aggregation task's reference loop):
 *       O_i^h = sum_j w_ij^h x_j[h,:]                          (normalize = 0)
 *       O_i^h = sum_j w_ij^h x_j[h,:] / (sum_j w_ij^h + eps)    (normalize = 1)
 *   with the weights w given per CSR entry and head, W of shape (E, H).
 *
 * Layouts: Q, K, V, X, O are (N, H, d) row-major; E and Eout are (E, H, d)
 * row-major indexed by CSR position; W is (E, H).  row_ptr (N+1) and col_idx
 * (E) int32.
 *
 * Parallelism: OpenMP over the listed rows only; the per-row arithmetic order
 * is fixed (edges in CSR order, features in index order), so results do not
 * depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

/* IEEE 754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac + 1024), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
    return sign ? -v : v;
}

/* bfloat16 is the top half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int dtype, int64_t i)
{
    switch (dtype) {
    case OR_F32: return (double)((const float *)base)[i];
    case OR_F16: return half_bits_to_double(((const uint16_t *)base)[i]);
    default:     return bf16_bits_to_double(((const uint16_t *)base)[i]);
    }
}

static double clampd(double x, double lo, double hi)
{
    return x < lo ? lo : (x > hi ? hi : x);
}

/* Exposed so the tests can pin the widening against numpy / torch. */
int g3s_oracle_decode(int dtype, const void *src, int64_t n, double *dst)
{
    if (dtype < 0 || dtype > 2) return 1;
    for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, dtype, i);
    return 0;
}

int g3s_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Thread count of later calls (n >= 1); for timing the oracle on one core
 * and on all of them.  Results do not depend on it (fixed per-row order). */
void g3s_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Standard or RTMScore attention for the rows listed in rows[0..n_rows).
 *   O_out   : (n_rows, H, d) doubles, row k holds destination rows[k]
 *   Eout_out: (E, H, d) doubles indexed by CSR position, or NULL; only the
 *             edges of listed rows are written (RTMScore only)
 * Returns 0 on success, 1 on bad arguments, 2 on an index outside [0, N).
 */
int g3s_oracle_forward(const int32_t *row_ptr, const int32_t *col_idx, int64_t N,
                       int H, int d, int dtype, int variant,
                       const void *Q, const void *K, const void *V, const void *Eproj,
                       const int64_t *rows, int64_t n_rows,
                       double *O_out, double *Eout_out,
                       int elementwise_clamp, double eps)
{
    if (H <= 0 || d <= 0 || dtype < 0 || dtype > 2 || (variant != 0 && variant != 1))
        return 1;
    if (variant == 1 && Eproj == NULL) return 1;
    const double scale = 1.0 / sqrt((double)d);
    const int64_t HD = (int64_t)H * d;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (int64_t k = 0; k < n_rows; ++k) {
        const int64_t i = rows[k];
        double *o = O_out + k * HD;
        for (int64_t x = 0; x < HD; ++x) o[x] = 0.0;
        if (i < 0 || i >= N) { bad = 1; continue; }
        const int64_t e0 = row_ptr[i], e1 = row_ptr[i + 1];
        if (e1 <= e0) continue; /* no in-edges: O = 0 */
        for (int h = 0; h < H; ++h) {
            const int64_t qo = i * HD + (int64_t)h * d;
            if (variant == 0) {
                /* logits and their maximum */
                double m = -INFINITY;
                for (int64_t e = e0; e < e1; ++e) {
                    const int64_t j = col_idx[e];
                    if (j < 0 || j >= N) { bad = 1; continue; }
                    double dot = 0.0;
                    for (int f = 0; f < d; ++f)
                        dot += load_elem(Q, dtype, qo + f) * load_elem(K, dtype, j * HD + (int64_t)h * d + f);
                    const double l = dot * scale;
                    if (l > m) m = l;
                }
                /* softmax weights and the weighted sum of values */
                double wsum = 0.0;
                for (int64_t e = e0; e < e1; ++e) {
                    const int64_t j = col_idx[e];
                    if (j < 0 || j >= N) continue;
                    double dot = 0.0;
                    for (int f = 0; f < d; ++f)
                        dot += load_elem(Q, dtype, qo + f) * load_elem(K, dtype, j * HD + (int64_t)h * d + f);
                    const double w = exp(dot * scale - m);
                    wsum += w;
                    for (int f = 0; f < d; ++f)
                        o[(int64_t)h * d + f] += w * load_elem(V, dtype, j * HD + (int64_t)h * d + f);
                }
                for (int f = 0; f < d; ++f) o[(int64_t)h * d + f] /= wsum;
            } else {
                double ssum = 0.0;
                for (int64_t e = e0; e < e1; ++e) {
                    const int64_t j = col_idx[e];
                    if (j < 0 || j >= N) { bad = 1; continue; }
                    double l = 0.0;
                    for (int f = 0; f < d; ++f) {
                        double t = load_elem(Q, dtype, qo + f) *
                                   load_elem(K, dtype, j * HD + (int64_t)h * d + f) * scale;
                        if (elementwise_clamp) t = clampd(t, -5.0, 5.0);
                        const double u = t * load_elem(Eproj, dtype, e * HD + (int64_t)h * d + f);
                        if (Eout_out) Eout_out[e * HD + (int64_t)h * d + f] = u;
                        l += u;
                    }
                    const double s = exp(clampd(l, -5.0, 5.0));
                    ssum += s;
                    for (int f = 0; f < d; ++f)
                        o[(int64_t)h * d + f] += s * load_elem(V, dtype, j * HD + (int64_t)h * d + f);
                }
                for (int f = 0; f < d; ++f) o[(int64_t)h * d + f] /= (ssum + eps);
            }
        }
    }
    return bad ? 2 : 0;
}

/*
 * Weighted aggregation for the rows listed in rows[0..n_rows); O_out is
 * (n_rows, H, d).  Returns 0 on success, 1 on bad arguments, 2 on an index
 * outside [0, N).
 */
int g3s_oracle_aggregate(const int32_t *row_ptr, const int32_t *col_idx, int64_t N, int H, int d, int dtype,
                         const void *W, const void *X, const int64_t *rows, int64_t n_rows, double *O_out,
                         int normalize, double eps)
{
    if (H <= 0 || d <= 0 || dtype < 0 || dtype > 2 || W == NULL || X == NULL) return 1;
    const int64_t HD = (int64_t)H * d;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (int64_t k = 0; k < n_rows; ++k) {
        const int64_t i = rows[k];
        double *o = O_out + k * HD;
        for (int64_t x = 0; x < HD; ++x) o[x] = 0.0;
        if (i < 0 || i >= N) { bad = 1; continue; }
        for (int h = 0; h < H; ++h) {
            double wsum = 0.0;
            for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
                const int64_t j = col_idx[e];
                if (j < 0 || j >= N) { bad = 1; continue; }
                const double w = load_elem(W, dtype, e * H + h);
                wsum += w;
                for (int f = 0; f < d; ++f)
                    o[(int64_t)h * d + f] += w * load_elem(X, dtype, j * HD + (int64_t)h * d + f);
            }
            if (normalize)
                for (int f = 0; f < d; ++f) o[(int64_t)h * d + f] /= (wsum + eps);
        }
    }
    return bad ? 2 : 0;
}
