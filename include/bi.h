/*
 * bi.h -- batch-invariant GEMM and causal GQA attention for GB300 (sm_103a).
 *
 * A C ABI over device memory that the caller owns (typically PyTorch tensors)
 * and a CUDA stream the caller owns.  Every entry point:
 *   - validates its arguments on the host first; on any error it launches
 *     nothing and returns a non-zero bi_status;
 *   - allocates nothing, synchronises nothing and launches on `stream` only
 *     (so the same call is legal inside CUDA-graph capture);
 *   - chooses its kernel, tile shape and reduction order from (dtype, N, K,
 *     weight layout) for GEMMs and (dtype, head_dim, group size, mask) for
 *     attention, never from M, the batch, the query length, the context length
 *     or a pointer value.  That is the batch-invariance contract: the bits of one
 *     output row do not depend on batch size, batch neighbours, query length
 *     (decode vs chunked prefill), KV-cache length, or eager vs graph replay
 *     ("mlx-batch-invariant" README, "What batch-invariant means here").
 *     Some scheduling does follow M, and none of it changes which products are
 *     summed or in what order: the number of A rows each tensor-memory copy
 *     moves (M rounded up to 16, at most one tile), the shared-memory ring depth
 *     that those smaller copies leave room for, the GEMM pair kernel's one or two
 *     K panels per ring stage (two when every CTA pair has at least two tiles),
 *     and the grid size (never more blocks than tiles).
 *
 * Layout: row-major, the last dimension contiguous.  Leading dimensions (ld*)
 * and strides are in ELEMENTS.  dtypes: BI_F32, BI_F16, BI_BF16 -- all
 * operands and the output of one call share the dtype; accumulation is fp32.
 *
 * Alignment (16-bit dtypes; the tensor-memory-accelerator copies need it):
 * GEMM operand/attention base pointers 16-byte aligned and their leading
 * dimensions / outer strides multiples of 8 elements, else BI_ERR_ALIGNMENT.
 * fp32 GEMMs need only natural alignment.
 *
 * Errors reported by the device (a bounded wait that ran out) are recorded in
 * a library-owned device error word and read with bi_last_device_error().
 *
 * First use: the first call that reaches a kernel on a device initialises the
 * library's per-device state (kernel shared-memory attributes, the error word's
 * address, the tensor-map encoder).  Make that first call before capturing a
 * CUDA graph on the device; every later call makes only stream launches.
 */
#ifndef BI_H
#define BI_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t.  NULL is the legacy default stream. */
typedef struct CUstream_st *bi_stream_t;

typedef enum {
    BI_OK = 0,
    BI_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad stride, q_offset out of range */
    BI_ERR_UNSUPPORTED = 2, /* dtype / head_dim / group size / mask not built */
    BI_ERR_ALIGNMENT = 3,   /* pointer or stride not aligned as required */
    BI_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed */
    BI_ERR_TIMEOUT = 5      /* a device-side bounded wait ran out (see bi_last_device_error) */
} bi_status;

typedef enum { BI_F32 = 0, BI_F16 = 1, BI_BF16 = 2 } bi_dtype;

typedef enum { BI_MASK_NONE = 0, BI_MASK_CAUSAL = 1, BI_MASK_ARRAY = 2 } bi_mask;

/* ------------------------------------------------------------------ GEMMs
 * "mlx-batch-invariant" README, "Use" (the op surface) and "How the kernels
 * work" / GEMM: every output element is one reduction over K in a fixed order
 * that depends only on K (no split-K, no matrix-vector special case), with an
 * fp32 accumulator, and the epilogue rounds once to the output dtype.
 * Accumulation is fp32 for every dtype; fp32 GEMMs use a sequential fused
 * multiply-add chain over k = 0..K-1; 16-bit GEMMs use tensor-core tiles whose
 * K blocks are visited in ascending order.  M == 0 is a no-op (BI_OK).
 */

/* linear (the nn.Linear layout):  y[M,N] = x[M,K] . w[N,K]^T (+ bias[N])
 *   x    device, [M,K] with leading dimension ldx >= K
 *   w    device, [N,K] with leading dimension ldw >= K (K contiguous)
 *   bias device, [N], or NULL for no bias; added to the fp32 accumulator
 *        before the single rounding: y = round(acc + bias)
 *   y    device, [M,N] with leading dimension ldy >= N; must not overlap inputs */
bi_status bi_linear(const void *x, int64_t ldx, const void *w, int64_t ldw, const void *bias,
                    void *y, int64_t ldy, int64_t M, int64_t N, int64_t K, bi_dtype dtype,
                    bi_stream_t stream);

/* matmul:  y[M,N] = a[M,K] . b[K,N]
 *   a device [M,K] (lda >= K);  b device [K,N] (ldb >= N, N contiguous);
 *   y device [M,N] (ldy >= N).  16-bit dtypes: the tile width for this (N,K)
 *   must be a multiple of 64 columns (always true: chosen by the library). */
bi_status bi_matmul(const void *a, int64_t lda, const void *b, int64_t ldb, void *y,
                    int64_t ldy, int64_t M, int64_t N, int64_t K, bi_dtype dtype,
                    bi_stream_t stream);

/* addmm:  y[M,N] = beta * c + alpha * (a[M,K] . b[K,N])
 *   c device; ldc > 0: c is [M,N] with leading dimension ldc;
 *             ldc == 0: c is one row c[N] broadcast to every m.
 *   Epilogue in fp32, fixed order, one rounding:
 *     y = round( (alpha * acc) + (beta * float(c)) )  (two products, then the sum). */
bi_status bi_addmm(const void *c, int64_t ldc, const void *a, int64_t lda, const void *b,
                   int64_t ldb, void *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                   float alpha, float beta, bi_dtype dtype, bi_stream_t stream);

/* Batched matmul: `batch` independent problems of one shape,
 *   y_e[M,N] = a_e[M,K] . b_e,   e = 0 .. batch-1,
 * with a_e = a + e*sa, b_e = b + e*sb, y_e = y + e*sy (element offsets).
 * "mlx-batch-invariant" README, "Use": matmul is one of the routed ops, and a
 * framework matmul also takes stacked operands [..., M, K] @ [..., K, N] (a
 * reading: the page does not discuss them).  Each entry is the GEMM above.
 *   b_layout 1: b_e is [K,N] with row stride ldb (N contiguous), as bi_matmul;
 *   b_layout 0: b_e is [N,K] with row stride ldb (K contiguous), y_e = a_e . b_e^T
 *               (torch.matmul(a, w.transpose(-1, -2)) for a contiguous w).
 *   sa or sb may be 0: that operand is shared by every entry.  Entries of y must
 *   not overlap: sy >= (M-1)*ldy + N when batch > 1.  16-bit dtypes: sa, sb, sy
 *   multiples of 8 elements.  batch <= 65535.
 * The tile configuration is that of the unbatched call for (N, K, dtype,
 * b_layout), and every entry's bits equal those of bi_matmul (b_layout 1) or
 * bi_linear without bias (b_layout 0) on that entry alone: an entry's result
 * depends neither on the batch size nor on the other entries. */
bi_status bi_matmul_batched(const void *a, int64_t lda, int64_t sa, const void *b, int64_t ldb,
                            int64_t sb, int b_layout, void *y, int64_t ldy, int64_t sy,
                            int64_t batch, int64_t M, int64_t N, int64_t K, bi_dtype dtype,
                            bi_stream_t stream);

/* Quantized linear (group-wise affine weights):  y[M,N] = x[M,K] . w^T (+ bias[N])
 * "mlx-batch-invariant" README, "Quantized models": 2, 4 and 8-bit affine weights,
 * unpacked inside the K loop of one invariant kernel.  Weight format (the plain
 * affine reading):
 *   q[n,k] = field (k mod 32/bits) of word wq[n*ldq + k/(32/bits)], fields of
 *            `bits` bits counted from the least significant bit;
 *   w[n,k] = round(scales[n*ldsb + g] * q[n,k] + biases[n*ldsb + g]), g = k/group_size,
 *            formed with one rounding to the activation dtype.
 *   x       device [M,K] bf16/fp16, leading dimension ldx >= K (multiple of 8)
 *   wq      device uint32 [N, ldq], ldq >= K*bits/32 (multiple of 4), 16-byte aligned
 *   scales, biases  device [N, ldsb] in x's dtype, ldsb >= K/group_size, a multiple
 *           of 8 elements, 16-byte aligned (they are copied in 16-byte boxes)
 *   bias    device [N] or NULL; added to the fp32 accumulator, rounded once
 *   y       device [M,N], leading dimension ldy >= N
 *   bits in {2, 4, 8}; group_size in {32, 64, 128}; K a multiple of 64 and of
 *   group_size (else BI_ERR_UNSUPPORTED / BI_ERR_INVALID_ARG).
 * Each output is one fp32 reduction over K in ascending 64-wide panels for
 * every M: a row's bits do not depend on the number of rows or on the others. */
bi_status bi_qlinear(const void *x, int64_t ldx, const uint32_t *wq, int64_t ldq,
                     const void *scales, const void *biases, int64_t ldsb, const void *bias,
                     void *y, int64_t ldy, int64_t M, int64_t N, int64_t K, int bits,
                     int group_size, bi_dtype dtype, bi_stream_t stream);

/* Reports the tile configuration the GEMM entry points use for (N, K, dtype,
 * weight layout).  b_layout: 0 = linear (w[N,K]), 1 = matmul/addmm (b[K,N]).
 * Outputs (each may be NULL): block_n = output columns per tile, stages =
 * shared-memory pipeline depth.  Host only; M is deliberately not an input. */
bi_status bi_gemm_config(int64_t N, int64_t K, bi_dtype dtype, int b_layout, int *block_n,
                         int *stages);

/* ------------------------------------------------------------------ attention
 * "mlx-batch-invariant" README, "Use" (scaled_dot_product_attention(q,k,v,
 * mask="causal")) and "How the kernels work" / Attention (single pass, online
 * softmax in fp32, fixed reduction order, no split over the keys).
 *
 *   q  device [B, H,   Lq,  D]  strides qs[4] (elements; qs[3] must be 1)
 *   k  device [B, Hkv, Lkv, D]  strides ks[4]
 *   v  device [B, Hkv, Lkv, D]  strides vs[4]
 *   o  device [B, H,   Lq,  D]  strides os[4]; written, must not overlap inputs
 *   H % Hkv == 0; query head h reads key/value head h / (H / Hkv).
 *   Query i sits at absolute position q_offset + i.  q_offset < 0 selects
 *   Lkv - Lq (the last query sees the whole cache).  Requires
 *   0 <= q_offset and q_offset + Lq <= Lkv.
 *   mask BI_MASK_CAUSAL: query i sees key j iff j <= q_offset + i.
 *   mask BI_MASK_NONE:   every query sees keys 0..Lkv-1.
 *   (BI_MASK_ARRAY needs its mask: use bi_sdpa_ex; here it is BI_ERR_INVALID_ARG.)
 *   scale <= 0 selects 1/sqrt(D).
 *   Keys are visited in fixed chunks of 128 at absolute key positions
 *   (0..127, 128..255, ...) in ascending order; queries sit in tiles aligned to
 *   absolute positions; a fully masked chunk is an exact no-op.  Hence a
 *   token's output bits do not depend on Lq, B, batch neighbours, or keys
 *   appended after it.  Masked keys must hold finite values.
 *   Built: dtype BI_BF16 / BI_F16, D in {64, 96, 128, 160, 192, 224, 256} (96 and
 *   160-224 run the 128- or 256-column kernel with the columns past D zero), H/Hkv
 *   in {1,2,4,8,16}.  D up to 128 visits keys in chunks of 128, larger D in chunks
 *   of 64: the chunking is a function of D alone.
 *   Lq == 0 or B == 0 is a no-op (BI_OK). */
bi_status bi_sdpa(const void *q, const int64_t qs[4], const void *k, const int64_t ks[4],
                  const void *v, const int64_t vs[4], void *o, const int64_t os[4], int64_t B,
                  int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D, float scale,
                  bi_mask mask, int64_t q_offset, bi_dtype dtype, bi_stream_t stream);

/* Attention with the other two mask forms and attention sinks.
 * "mlx-batch-invariant" README, "How the kernels work" / Attention ("all three
 * mask forms") and the paragraph on attention sinks.  Arguments as bi_sdpa, plus:
 *   mask        BI_MASK_NONE, BI_MASK_CAUSAL, or BI_MASK_ARRAY;
 *   mask_array  BI_MASK_ARRAY only (else NULL): device uint8, nonzero = visible,
 *               element (b,h,i,j) at b*ms[0] + h*ms[1] + i*ms[2] + j (ms[3] must
 *               be 1; a stride of 0 broadcasts).  Keys j >= Lkv are never visible.
 *   sinks       device fp32 [H] or NULL: one extra logit per query head, in the
 *               units of the scaled scores, that joins the softmax denominator
 *               and carries no value; 4-byte aligned.
 * A query with no visible key and no sink gets NaN.  The mask row of a token
 * must be the same in every call for its bits to be the same in every call. */
bi_status bi_sdpa_ex(const void *q, const int64_t qs[4], const void *k, const int64_t ks[4],
                     const void *v, const int64_t vs[4], void *o, const int64_t os[4], int64_t B,
                     int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D, float scale,
                     bi_mask mask, int64_t q_offset, const float *sinks,
                     const uint8_t *mask_array, const int64_t ms[4], bi_dtype dtype,
                     bi_stream_t stream);

/* ------------------------------------------------------------------ decoder glue
 * Row-local ops that a decoder needs around the GEMMs and attention.  The
 * README ("Why MLX is not invariant", last paragraph) notes that normalisation
 * and elementwise ops are already batch-invariant in MLX; on CUDA this library
 * provides them so that their reduction order is fixed by construction.
 * All are 16-bit or fp32 in, same dtype out, fp32 arithmetic inside.
 */

/* RMSNorm: y[m,n] = round( x[m,n] * r_m * w[n] ),  r_m = 1 / sqrt(mean_n x[m,n]^2 + eps)
 *   x, y device [M,N] with leading dimensions ldx, ldy; w device [N].
 *   The sum of squares of one row is reduced by one block in a fixed tree. */
bi_status bi_rmsnorm(const void *x, int64_t ldx, const void *w, void *y, int64_t ldy, int64_t M,
                     int64_t N, float eps, bi_dtype dtype, bi_stream_t stream);

/* Rotary position embedding (rotate-half pairing) on x viewed as [B, L, nh, D]:
 *   position of (b, l) = pos0 + l;  half = D/2;  inv_freq_i = base^(-2i/D);
 *   y[i] = x[i] cos - x[i+half] sin,  y[i+half] = x[i+half] cos + x[i] sin.
 *   xs[4], ys[4]: element strides of x and y over (b, l, head, d); the d
 *   strides must be 1.  y may be a slice of a KV cache (e.g. [B,Hkv,Lmax,D]
 *   viewed through strides).  In-place (x == y with equal strides) is allowed. */
bi_status bi_rope(const void *x, const int64_t xs[4], void *y, const int64_t ys[4], int64_t B,
                  int64_t L, int64_t nh, int64_t D, int64_t pos0, float base, bi_dtype dtype,
                  bi_stream_t stream);

/* SwiGLU: gu[M, 2I] = [gate | up] (row stride ldgu), y[M, I] (row stride ldy):
 *   y = round( silu(gate) * up ),  silu(g) = g / (1 + exp(-g)). */
bi_status bi_swiglu(const void *gu, int64_t ldgu, void *y, int64_t ldy, int64_t M, int64_t I,
                    bi_dtype dtype, bi_stream_t stream);

/* Elementwise sum of two contiguous vectors of n elements: y = round(a + b).
 * y may alias a or b. */
bi_status bi_add(const void *a, const void *b, void *y, int64_t n, bi_dtype dtype,
                 bi_stream_t stream);

/* Embedding gather: y[t, :] = table[ids[t], :] for t < n_ids.
 *   ids device int64 [n_ids], each in [0, vocab) (out-of-range ids produce a
 *   zero row and set the device error word); table device [vocab, dim] with
 *   row stride ldt; y device [n_ids, dim] with row stride ldy. */
bi_status bi_embedding(const int64_t *ids, int64_t n_ids, const void *table, int64_t ldt,
                       int64_t vocab, void *y, int64_t ldy, int64_t dim, bi_dtype dtype,
                       bi_stream_t stream);

/* Strided 4-D copy: dst[i0,i1,i2,i3] = src[i0,i1,i2,i3] over sizes n[4];
 * ss[4], ds[4] element strides (the last must be 1).  Used to write new
 * keys/values into a KV cache. */
bi_status bi_copy4d(const void *src, const int64_t ss[4], void *dst, const int64_t ds[4],
                    const int64_t n[4], bi_dtype dtype, bi_stream_t stream);

/* ------------------------------------------------------------------ status
 */

/* A static, human-readable name for a status code. */
const char *bi_status_string(bi_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int bi_version(void);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device.  BI_OK if no kernel recorded an error since the last call;
 * BI_ERR_TIMEOUT if a bounded wait ran out (the kernel stopped early and its
 * outputs are undefined); BI_ERR_INVALID_ARG for a device-detected bad index.
 * *code (may be NULL) receives the raw word. */
bi_status bi_last_device_error(bi_stream_t stream, uint32_t *code);

/* Number of kernels this library has launched in this process (host counter). */
int64_t bi_launch_count(void);

/* Test hook for the bounded-wait machinery: launches one block that waits on
 * a shared-memory barrier that nothing will ever complete, for at most
 * `limit_us` microseconds (1 .. 2,000,000).  The wait must run out; the kernel
 * then records BI_ERR_TIMEOUT in the device error word and returns.  Nothing
 * else runs, nothing is written but the error word. */
bi_status bi_debug_wait_probe(int64_t limit_us, bi_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BI_H */
