/*
 * oracle.c -- plain, slow, fp64 CPU reference for the batch-invariant GEMM and
 * causal GQA attention path, plus the decoder glue (RMSNorm, RoPE, SwiGLU).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
 * this file.  Its users are the tests, the smoke check and the CPU-baseline leg
 * of the benchmark.  It shares no code, header, table or constant with the CUDA
 * library: every function below is the textbook definition written out with
 * fp64 products and fp64 sums taken in natural index order, so that a reader can
 * check it against the definition by eye.  OpenMP only splits independent
 * output rows across threads; it never splits a sum.
 *
 * Source of the definitions (the "mlx-batch-invariant" README):
 *   - "Use": the op surface linear(x, w[N,K], bias), matmul(a, b[K,N]),
 *     addmm(c, a, b, alpha, beta), scaled_dot_product_attention(q,k,v,"causal").
 *   - "How the kernels work" / GEMM: the bias is added into the accumulator.
 *   - "How the kernels work" / Attention: softmax attention.
 *   - "Accuracy": the results are judged against a float64 reference; this is
 *     that reference.
 *   - "Why MLX is not invariant" / Attention: GQA (H query heads share Hkv
 *     key/value heads); "How the kernels work" / Attention: "all three mask
 *     forms" (none, causal, array); the last paragraph before "Prior art":
 *     attention sinks.
 * Readings where the page is silent (each also listed in the design notes):
 *   - causal alignment: query i sits at absolute position q_offset + i and sees
 *     key j iff j <= q_offset + i;
 *   - GQA head map: query head h reads key/value head h / (H / Hkv);
 *   - addmm: y = beta * c + alpha * (a . b), c either [M,N] or a row c[N];
 *   - RoPE: rotate-half pairing, inv_freq_i = base^(-2i/D);
 *   - SwiGLU: input [M, 2I] = [gate | up], y = silu(gate) * up;
 *   - array mask: boolean, nonzero = the key is visible;
 *   - attention sink: one extra logit per query head, in the units of the
 *     scaled scores, that joins the softmax denominator with no value;
 *   - quantized weights ("Quantized models": 2, 4 and 8-bit affine, group-wise):
 *     w[n,k] = scales[n, k/gs] * q[n,k] + biases[n, k/gs], with q the unsigned
 *     `bits`-wide field number (k mod 32/bits) of the 32-bit word k / (32/bits)
 *     of row n, fields numbered from the least significant bit.
 * Every function also returns the per-element normaliser that the tolerance
 * is stated against (the sum of the magnitudes of the terms).
 *
 * Parity status: every function here is pinned by CPU tests against exact
 * rational brute force, closed forms or independent library routines.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* linear: y[m,n] = sum_k x[m,k] * w[n,k] + bias[n]   (bias may be NULL)
 * nrm[m,n] = sum_k |x[m,k] * w[n,k]| + |bias[n]|                           */
void oracle_linear(int64_t M, int64_t N, int64_t K, const double *x, const double *w,
                   const double *bias, double *y, double *nrm)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = x[m * K + k] * w[n * K + k];
                s += t;
                a += fabs(t);
            }
            if (bias) {
                s += bias[n];
                a += fabs(bias[n]);
            }
            y[m * N + n] = s;
            if (nrm) nrm[m * N + n] = a;
        }
    }
}

/* matmul: y[m,n] = sum_k a[m,k] * b[k,n];  nrm[m,n] = sum_k |a[m,k] * b[k,n]| */
void oracle_matmul(int64_t M, int64_t N, int64_t K, const double *a, const double *b,
                   double *y, double *nrm)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0, r = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = a[m * K + k] * b[k * N + n];
                s += t;
                r += fabs(t);
            }
            y[m * N + n] = s;
            if (nrm) nrm[m * N + n] = r;
        }
    }
}

/* addmm: y[m,n] = beta * c[m,n] + alpha * sum_k a[m,k] * b[k,n]
 * c is [M,N] (c_row == 0) or a single row c[N] shared by all m (c_row != 0).
 * nrm[m,n] = |alpha| * sum_k |a b| + |beta * c|                              */
void oracle_addmm(int64_t M, int64_t N, int64_t K, const double *c, int c_row,
                  const double *a, const double *b, double alpha, double beta,
                  double *y, double *nrm)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0, r = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = a[m * K + k] * b[k * N + n];
                s += t;
                r += fabs(t);
            }
            double cv = c_row ? c[n] : c[m * N + n];
            y[m * N + n] = beta * cv + alpha * s;
            if (nrm) nrm[m * N + n] = fabs(alpha) * r + fabs(beta * cv);
        }
    }
}

/* Scaled dot-product attention with GQA.
 *   q[B,H,Lq,D], k[B,Hkv,Lkv,D], v[B,Hkv,Lkv,D], o[B,H,Lq,D]; dense row-major.
 *   kv head of query head h: h / (H / Hkv).
 *   visible keys of query i: j < Lkv and
 *     mask != NULL: mask[((b*H + h)*Lq + i)*Lkv + j] != 0   (boolean array mask)
 *     else causal:  j <= q_offset + i
 *     else:         every j.
 *   s_j = scale * <q_i, k_j>.  With sinks != NULL, head h has one more logit
 *   sinks[h] (in the units of s) that enters the softmax denominator and
 *   carries no value.  p_j = exp(s_j - mx) / (sum_visible exp(s - mx)
 *   [+ exp(sink_h - mx)]), mx the maximum of the visible s (and the sink);
 *   o_i = sum_j p_j v_j;  nrm[b,h,i,d] = sum_j p_j |v_j[d]|.
 * A query with no visible key and no sink has no defined output: NaN.      */
void oracle_sdpa_ex(int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
                    const double *q, const double *k, const double *v, double scale, int causal,
                    int64_t q_offset, const double *sinks, const unsigned char *mask, double *o,
                    double *nrm)
{
    const int64_t group = H / Hkv;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
        unsigned char *vis = (unsigned char *)malloc((size_t)(Lkv > 0 ? Lkv : 1));
#pragma omp for schedule(dynamic, 1) collapse(3)
        for (int64_t b = 0; b < B; ++b) {
            for (int64_t h = 0; h < H; ++h) {
                for (int64_t i = 0; i < Lq; ++i) {
                    const int64_t hk = h / group;
                    const double *qi = q + ((b * H + h) * Lq + i) * D;
                    const double *kb = k + (b * Hkv + hk) * Lkv * D;
                    const double *vb = v + (b * Hkv + hk) * Lkv * D;
                    double *oi = o + ((b * H + h) * Lq + i) * D;
                    double *ni = nrm ? nrm + ((b * H + h) * Lq + i) * D : 0;
                    int64_t nvis = 0;
                    for (int64_t j = 0; j < Lkv; ++j) {
                        int visible;
                        if (mask) visible = mask[((b * H + h) * Lq + i) * Lkv + j] != 0;
                        else if (causal) visible = j <= q_offset + i;
                        else visible = 1;
                        vis[j] = (unsigned char)visible;
                        nvis += visible;
                    }
                    if (nvis == 0 && !sinks) {
                        for (int64_t d = 0; d < D; ++d) {
                            oi[d] = NAN;
                            if (ni) ni[d] = NAN;
                        }
                        continue;
                    }
                    double mx = sinks ? sinks[h] : -INFINITY;
                    for (int64_t j = 0; j < Lkv; ++j) {
                        if (!vis[j]) continue;
                        double t = 0.0;
                        for (int64_t d = 0; d < D; ++d) t += qi[d] * kb[j * D + d];
                        s[j] = scale * t;
                        if (s[j] > mx) mx = s[j];
                    }
                    double den = sinks ? exp(sinks[h] - mx) : 0.0;
                    for (int64_t j = 0; j < Lkv; ++j) {
                        if (!vis[j]) continue;
                        s[j] = exp(s[j] - mx);
                        den += s[j];
                    }
                    for (int64_t d = 0; d < D; ++d) {
                        double acc = 0.0, r = 0.0;
                        for (int64_t j = 0; j < Lkv; ++j) {
                            if (!vis[j]) continue;
                            double p = s[j] / den;
                            acc += p * vb[j * D + d];
                            r += p * fabs(vb[j * D + d]);
                        }
                        oi[d] = acc;
                        if (ni) ni[d] = r;
                    }
                }
            }
        }
        free(vis);
        free(s);
    }
}

/* The plain causal / unmasked form without sinks (the README's "Use" call). */
void oracle_sdpa(int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
                 const double *q, const double *k, const double *v, double scale,
                 int causal, int64_t q_offset, double *o, double *nrm)
{
    oracle_sdpa_ex(B, H, Hkv, Lq, Lkv, D, q, k, v, scale, causal, q_offset, 0, 0, o, nrm);
}

/* Quantized linear ("mlx-batch-invariant" README, "Quantized models"):
 *   q[n,k]  = (wq[n*ldq + k/f] >> (bits * (k mod f))) & (2^bits - 1),  f = 32/bits
 *   w[n,k]  = scales[n*ldsb + k/gs] * q[n,k] + biases[n*ldsb + k/gs]
 *   y[m,n]  = sum_k x[m,k] * w[n,k]  (+ bias[n]);   nrm = sum_k |x w| (+ |bias|)
 * w is formed exactly in fp64 (no rounding to a 16-bit type).               */
void oracle_qlinear(int64_t M, int64_t N, int64_t K, const double *x, const uint32_t *wq,
                    int64_t ldq, const double *scales, const double *biases, int64_t ldsb,
                    int bits, int64_t gs, const double *bias, double *y, double *nrm)
{
    const int64_t f = 32 / bits;
    const uint32_t fmask = bits == 32 ? 0xFFFFFFFFu : ((1u << bits) - 1u);
#pragma omp parallel
    {
        double *wrow = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t k = 0; k < K; ++k) {
                const uint32_t word = wq[n * ldq + k / f];
                const uint32_t q = (word >> (bits * (k % f))) & fmask;
                wrow[k] = scales[n * ldsb + k / gs] * (double)q + biases[n * ldsb + k / gs];
            }
            for (int64_t m = 0; m < M; ++m) {
                double acc = 0.0, mag = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double t = x[m * K + k] * wrow[k];
                    acc += t;
                    mag += fabs(t);
                }
                if (bias) {
                    acc += bias[n];
                    mag += fabs(bias[n]);
                }
                y[m * N + n] = acc;
                if (nrm) nrm[m * N + n] = mag;
            }
        }
        free(wrow);
    }
}

/* RMSNorm over the last dim: y[m,n] = x[m,n] / sqrt(mean_n x[m,.]^2 + eps) * w[n] */
void oracle_rmsnorm(int64_t M, int64_t N, const double *x, const double *w, double eps,
                    double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t n = 0; n < N; ++n) ss += x[m * N + n] * x[m * N + n];
        double r = 1.0 / sqrt(ss / (double)N + eps);
        for (int64_t n = 0; n < N; ++n) y[m * N + n] = x[m * N + n] * r * w[n];
    }
}

/* Rotary position embedding, rotate-half pairing.
 *   x[T, nh, D] (one token per t), pos[t] its absolute position.
 *   half = D/2, inv_freq_i = base^(-2i/D), theta = pos * inv_freq_i,
 *   y[i]      = x[i] cos(theta) - x[i+half] sin(theta)
 *   y[i+half] = x[i+half] cos(theta) + x[i] sin(theta)                   */
void oracle_rope(int64_t T, int64_t nh, int64_t D, const double *x, const int64_t *pos,
                 double base, double *y)
{
    const int64_t half = D / 2;
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < nh; ++h) {
            const double *xi = x + (t * nh + h) * D;
            double *yi = y + (t * nh + h) * D;
            for (int64_t i = 0; i < half; ++i) {
                double inv_freq = pow(base, -2.0 * (double)i / (double)D);
                double th = (double)pos[t] * inv_freq;
                double c = cos(th), s = sin(th);
                yi[i] = xi[i] * c - xi[i + half] * s;
                yi[i + half] = xi[i + half] * c + xi[i] * s;
            }
        }
    }
}

/* SwiGLU: gu[M, 2I] = [gate | up];  y[m,i] = silu(gate) * up,  silu(g) = g / (1 + e^-g) */
void oracle_swiglu(int64_t M, int64_t I, const double *gu, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t i = 0; i < I; ++i) {
            double g = gu[m * 2 * I + i];
            double u = gu[m * 2 * I + I + i];
            y[m * I + i] = g / (1.0 + exp(-g)) * u;
        }
    }
}
