/*
 * coda.h -- C ABI of libcoda: the non-attention part of a Transformer block
 * run as GEMM-plus-epilogue programs on sm_103a (tcgen05 + TMEM + TMA).
 *
 * Sources (page title, section):
 *   [pith]   "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
 *            (pith.science summary of arXiv 2605.19269): Fig. 3, 4, 5 and 7
 *            captions, Appendix A.1 "Tile-wise Epilogue", Listing 2 "Kernel
 *            Example".
 *   [notes]  "Reading notes on CODA" (jianyuh.github.io): s1 "The Epilogue
 *            Concept", s2 "Forward-Pass Reparameterizations", s3 "The Backward
 *            Pass: Reverse Fusion".
 *   [thread] digg thread on CODA: Patterns 1-3.
 *
 * Conventions for every entry point:
 *   - Tensor arguments are DEVICE pointers owned by the caller. The library
 *     never allocates, frees or keeps them; it reads inputs and writes
 *     outputs only during the asynchronous work it enqueues.
 *   - Tensors are dense row-major. "bf16" = IEEE bfloat16 (uint16 storage),
 *     vectors and partials are fp32, targets are int32. Rows are contiguous;
 *     the only strided entry point is coda_gemm (lda/ldb/ldc in elements).
 *   - Every pointer must be 16-byte aligned and every row length (in bytes)
 *     a multiple of 16 (bf16: a multiple of 8 elements), because all tiles
 *     move through TMA.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; 0 = legacy default
 *     stream) and thread-safe.
 *   - Return value: CODA_OK, or
 *       CODA_ERR_INVALID_VALUE  null/misaligned pointer, non-positive or
 *                               inconsistent size (checked before launch,
 *                               nothing is enqueued);
 *       CODA_ERR_UNSUPPORTED    device is not sm_100-family / shape beyond
 *                               the supported range;
 *       CODA_ERR_LAUNCH         a CUDA error at launch (text from
 *                               coda_last_error_string()).
 *     Device-side failures (a bounded wait that ran out, an out-of-range CE
 *     target, a value beyond the fp16 range in a saved fp16 copy) are
 *     recorded in a device error word and reported by
 *     coda_get_device_error() (CODA_ERR_TIMEOUT, CODA_ERR_INVALID_VALUE,
 *     CODA_ERR_RANGE).
 *   - Partial buffers: the GEMM epilogues write tile-local partials that a
 *     small auxiliary kernel reduces ([pith] Fig. 4 caption). Their shapes
 *     use coda_col_tiles(N) = ceil(N / 128) (one partial per 128 columns,
 *     whatever tile width a kernel runs) and coda_row_tiles32(M) =
 *     ceil(M / 32).
 */
#ifndef CODA_H_
#define CODA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CODA_OK = 0,
  CODA_ERR_INVALID_VALUE = 1,
  CODA_ERR_UNSUPPORTED = 2,
  CODA_ERR_LAUNCH = 3,
  CODA_ERR_TIMEOUT = 4,
  CODA_ERR_RANGE = 5
} coda_status_t;

/* Opaque CUDA stream (identical to cudaStream_t). */
typedef struct CUstream_st* coda_stream_t;

/* Library version (major * 10000 + minor * 100 + patch). */
int coda_version(void);

/* Number of row partials per row written by the *_stats / *_bwd GEMMs for an
 * output of N columns: ceil(N / 128), one per 128-column group. */
int coda_col_tiles(int N);
/* Number of per-32-row partials per column of the RMSNorm weight gradient:
 * ceil(M / 32). */
int coda_row_tiles32(int M);

/* Bound, in milliseconds, on every wait inside the kernels (default 2000).
 * A wait that runs out records CODA_ERR_TIMEOUT and the kernel returns. */
void coda_set_timeout_ms(int ms);

/* For tests of failure detection only; never set in normal use (default -1,
 * off). With kb >= 0, every later GEMM launch leaves k-block kb of the first
 * tile of each CTA pair unloaded, so the MMA issuer's bounded wait for it
 * runs out (and with it the waits of the other roles): the kernel records
 * CODA_ERR_TIMEOUT in the device error word, stops its loads, frees its
 * TMEM and returns, and coda_get_device_error reports the timeout. Nothing
 * faults and the context stays usable. kb < 0 switches it off. The setting
 * is process-wide. */
void coda_debug_skip_kblock(int kb);

/* Synchronises `stream`, then returns and clears the device error word:
 * CODA_OK, CODA_ERR_TIMEOUT (a bounded wait ran out),
 * CODA_ERR_INVALID_VALUE (a CE target outside [0, V)) or CODA_ERR_RANGE (a
 * value beyond the fp16 range in a saved fp16 copy). There is one error word
 * per device, shared by every stream and thread: it holds the first error
 * recorded since it was last read, and reading it clears it, so callers that
 * launch on several streams of one device should read it from one place. */
coda_status_t coda_get_device_error(coda_stream_t stream);

/* Text of the last error seen by this thread (never NULL). With the
 * environment variable CODA_DEBUG set to anything but "0" when the library
 * first records an error, every host-side error message is also written to
 * stderr, prefixed "libcoda: ", as it is recorded. */
const char* coda_last_error_string(void);

/* ------------------------------------------------------------------ GEMM */

/* Plain GEMM with an optional residual and row-statistic epilogue
 * ([notes] s1: the fixed mainloop with tile-local epilogue primitives).
 *   C[M, N] = op(A) op(B) (+ resid)
 *   transA = 0: A is [M, K] (lda >= K); 1: A is stored [K, M] (lda >= M).
 *   transB = 0: B is [K, N] (ldb >= N); 1: B is stored [N, K] (ldb >= K).
 *   resid (nullable, [M, N] of C's type, row stride ldc) is added in fp32
 *   before rounding; rowsq_part (nullable, fp32 [coda_col_tiles(N), M]) receives
 *   the sum over each 128-column group of the fp32 result squared.
 *   c_fp32 = 1: C is fp32 (e.g. weight gradients), else bf16.
 *   rowsq_part requires transA = 0, transB = 0, c_fp32 = 0. resid requires
 *   transA = 0; with c_fp32 = 0 it is bf16 and needs transB = 0, with
 *   c_fp32 = 1 it is fp32 (and may be C itself: C += op(A) op(B)). */
coda_status_t coda_gemm(const void* A, int lda, int transA, const void* B, int ldb, int transB,
                        const void* resid, float* rowsq_part, void* C, int ldc, int c_fp32,
                        int M, int N, int K, coda_stream_t stream);

/* GEMM 1 of GEMM-RMSNorm-GEMM ([notes] s2 "GEMM -> Residual -> RMSNorm ->
 * GEMM"; [pith] Listing 2: residual, block mean of squares of the unscaled
 * output, RMSNorm-weight side output):
 *   h  = x W0 + z             (bf16 [M, N], the residual stream)
 *   hg = h * gamma[n]         (bf16 [M, N], input of the next GEMM)
 *   part[t, m] = sum over columns 128 t .. 128 t + 127 of h[m, n]^2 (fp32,
 *                before rounding h), part is [coda_col_tiles(N), M]
 * x bf16 [M, K]; W0 bf16 [K, N]; z bf16 [M, N]; gamma bf16 [N]. */
coda_status_t coda_gemm_resid_norm_stats(const void* x, const void* W0, const void* z,
                                         const void* gamma, void* h, void* hg, float* part,
                                         int M, int N, int K, coda_stream_t stream);

/* Auxiliary row reduction ([pith] Fig. 5: r = 1/sqrt(reduce(r_hat) + eps)):
 *   r[m] = 1 / sqrt(sum_j part[j, m] / d + eps)
 * part fp32 [nparts, M]; r fp32 [M]; d = hidden width (> 0). */
coda_status_t coda_row_rms(const float* part, int nparts, int M, int d, float eps, float* r,
                           coda_stream_t stream);

/* GEMM 2 with the delayed row scale and the pairwise SwiGLU map ([notes] s2:
 * y = r (h2 W1); [pith] Fig. 7: SwiGLU combines gate and value streams):
 *   y = r[m] * (hg W1)   (columns 2k = gate g_k, 2k+1 = up u_k)
 *   a[m, k] = silu(g_k) * u_k          (bf16 [M, two_f / 2])
 *   y_save (nullable): fp16 [M, two_f], the scaled y kept for the backward.
 *   Not bf16: the relocated RMSNorm statistic of the backward sums 2f
 *   products of y with heavy cancellation, and bf16 storage of y alone moves
 *   it by ~1e-3..5e-3 relative; fp16 (11-bit significand) keeps it near
 *   1e-4 at half the bytes of fp32. A y of magnitude >= 65520 (or NaN) is
 *   stored as inf/NaN and raises CODA_ERR_RANGE in coda_get_device_error();
 *   a and the other outputs are still written.
 * hg bf16 [M, K]; W1 bf16 [K, two_f]; r fp32 [M]; two_f even. */
coda_status_t coda_gemm_rowscale_swiglu(const void* hg, const void* W1, const float* r, void* a,
                                        void* y_save, int M, int two_f, int K,
                                        coda_stream_t stream);

/* Row scale and pairwise RoPE epilogue ([pith] Fig. 7: RoPE rotates each
 * feature pair and returns two outputs):
 *   v = r[m] * (A W)   (r nullable: no scale)
 *   for n < n_rope_cols, inside each head_dim-wide head, pair (2i, 2i+1):
 *     v'_2i = v_2i c - v_2i+1 s,  v'_2i+1 = v_2i s + v_2i+1 c,
 *     (c, s) = cos_sin[m mod seq_len, i]
 *   out bf16 [M, N]; out_f16 (nullable) fp16 [M, N], the same values kept
 *   with a longer significand for the backward's relocated RMSNorm statistic
 *   (coda_gemm_rope_bwd); range errors as for y_save of
 *   coda_gemm_rowscale_swiglu. A bf16 [M, K]; W bf16 [K, N];
 *   cos_sin fp32 [seq_len, head_dim/2, 2] (see coda_rope_table).
 *   head_dim % 32 == 0, n_rope_cols % head_dim == 0, n_rope_cols <= N. */
coda_status_t coda_gemm_rope(const void* A, const void* W, const float* r, const float* cos_sin,
                             int seq_len, int head_dim, int n_rope_cols, void* out, void* out_f16,
                             int M, int N, int K, coda_stream_t stream);

/* Fills cos_sin[p, i] = (cos(p t_i), sin(p t_i)), t_i = theta^(-2i/head_dim),
 * computed in fp64 on the device and rounded to fp32.
 * cos_sin fp32 [seq_len, head_dim/2, 2]. */
coda_status_t coda_rope_table(float* cos_sin, int seq_len, int head_dim, double theta,
                              coda_stream_t stream);

/* Bytes of scratch that coda_lmhead_ce needs for M rows and V classes. */
size_t coda_lmhead_ce_workspace_size(int M, int V);

/* LM head + cross-entropy without writing the logits ([notes] s2
 * "Cross-entropy loss": l_i = -h_{i,y_i} + log sum_k exp h_{i,k}; [thread]
 * Pattern 3). The GEMM epilogue keeps a running max and sum-exp per row and
 * column tile and picks the target logit by index; an auxiliary kernel
 * combines the tiles:
 *   lse[m]  = log sum_v exp(logit[m, v])       (fp32 [M])
 *   loss[m] = lse[m] - logit[m, targets[m]]    (fp32 [M])
 * hidden bf16 [M, d]; W bf16 [d, V]; targets int32 [M] in [0, V) (a target
 * out of range gives loss NaN and CODA_ERR_INVALID_VALUE from
 * coda_get_device_error); ws: caller-owned device scratch of at least
 * coda_lmhead_ce_workspace_size(M, V) bytes. */
coda_status_t coda_lmhead_ce(const void* hidden, const void* W, const int32_t* targets, float* lse,
                             float* loss, void* ws, size_t ws_bytes, int M, int V, int d,
                             coda_stream_t stream);

/* LM head + cross-entropy without any scratch from the caller (the pages
 * have no counterpart: this is a convenience of this library). Same inputs,
 * outputs and results as coda_lmhead_ce; the scratch comes from an array of
 * coda_lmhead_ce_noalloc_capacity() bytes (16 MiB) that the library keeps in
 * the memory of every GPU that loads it, until the process exits.
 * For callers that may not allocate device memory: e.g. an operator hook
 * that receives only its inputs and outputs while a host framework's
 * allocator owns the rest of the device, or a loop where cudaMalloc /
 * cudaFree (which can synchronise the device) are not allowed.
 *   - M, V and d must be positive (else CODA_ERR_INVALID_VALUE, before any
 *     device call), and M and V must satisfy
 *     coda_lmhead_ce_workspace_size(M, V) <= coda_lmhead_ce_noalloc_capacity()
 *     (about 4100 rows at V = 128256); larger requests return
 *     CODA_ERR_INVALID_VALUE with an explanation. The remaining argument
 *     checks are those of coda_lmhead_ce.
 *   - Every call looks the array's device address up on the current device
 *     (cudaGetSymbolAddress, a host-side query) and keeps nothing, so the
 *     call stays valid after a cudaDeviceReset. The first call on a device
 *     may load the library's module there: make it before any stream
 *     capture.
 *   - All calls share the array: calls whose work overlaps on the GPU (e.g.
 *     on two streams at once) race and give wrong results. Each call
 *     rewrites every entry it reads, so no clearing is needed.
 *   - Allocates nothing (no cudaMalloc, cudaFree or allocating library call). */
size_t coda_lmhead_ce_noalloc_capacity(void);
coda_status_t coda_lmhead_ce_noalloc(const void* hidden, const void* W, const int32_t* targets,
                                     float* lse, float* loss, int M, int V, int d,
                                     coda_stream_t stream);

/* Bytes of scratch that coda_lmhead_ce_bwd is designed for with M rows and V
 * classes: one bf16 gradient chunk of M x min(V rounded up to 256, 16384)
 * (268 MB at M = 8192). A smaller workspace (at least M * 256 * 2 bytes)
 * gives narrower chunks; a larger one wider chunks, up to 32768 columns. */
size_t coda_lmhead_ce_bwd_workspace_size(int M, int V);

/* LM-head cross-entropy backward without materialising the logits
 * ([notes] s2 "Cross-entropy loss"; [thread] Pattern 3, "as in Cut Cross
 * Entropy"; the pages give no backward, this is the reading): for
 * L = sum_m dloss[m] * loss[m],
 *   G = dloss[m] (softmax(hidden W)[m] - onehot(targets[m]))
 *   dhidden = G W^T (fp32 [M, d]),  dW = hidden^T G (fp32 [d, V])
 * The vocabulary is processed in chunks: per chunk, a GEMM recomputes the
 * logit tile and its epilogue writes G (bf16) into ws; a second GEMM adds
 * G W_chunk^T into dhidden; a third writes dW's columns of the chunk.
 * lse: fp32 [M] from coda_lmhead_ce. ws: caller-owned scratch; its size
 * sets the chunk width (at least M * 256 * 2 bytes; see
 * coda_lmhead_ce_bwd_workspace_size). Other arguments as in coda_lmhead_ce. */
coda_status_t coda_lmhead_ce_bwd(const void* hidden, const void* W, const int32_t* targets,
                                 const float* lse, const float* dloss, float* dhidden, float* dW,
                                 void* ws, size_t ws_bytes, int M, int V, int d,
                                 coda_stream_t stream);

/* ------------------------------------------------------------ backward */

/* Reverse-fused SwiGLU backward ([notes] s3 "Reverse Fusion": f'(h)
 * multiplies into the GEMM that produces the gradient of f's output; [pith]
 * Fig. 7: one incoming gradient, two outgoing; [notes] s3 "Eliminating the
 * RMSNorm backward kernel": the statistic is accumulated here):
 *   da = dout W2^T ; (g, u) = y_save pair ; sg = sigmoid(g)
 *   dg = da u sg (1 + g (1 - sg)) ; du = da g sg
 *   dyhat[m, 2k..2k+1] = r[m] (dg, du)            (bf16 [M, 2f])
 *   spart[t, m] = sum of dg g + du u over da columns 128 t .. 128 t + 127
 *                                                 (fp32 [coda_col_tiles(f), M])
 * dout bf16 [M, d]; W2 bf16 [f, d]; y fp16 [M, 2f] (as saved by
 * coda_gemm_rowscale_swiglu); r fp32 [M]. */
coda_status_t coda_gemm_rowscale_swiglu_bwd(const void* dout, const void* W2, const void* y,
                                            const float* r, void* dyhat, float* spart, int M,
                                            int f, int d, coda_stream_t stream);

/* s[m] = (1/d) sum_j spart[j, m]  ([notes] s3: s = sumcols(dy * y) / d). */
coda_status_t coda_row_rms_bwd(const float* spart, int nparts, int M, int d, float* s,
                               coda_stream_t stream);

/* RMSNorm backward fused into the GEMM P = dyhat W1^T ([notes] s3):
 *   dh = gamma[n] P - r[m]^2 s[m] h (+ dresid)     (bf16 [M, d])
 *   dgamma_part[j, n] = sum over rows 32j..32j+31 of P h
 *                       (fp32 [coda_row_tiles32(M), d])
 * dyhat bf16 [M, two_f]; W1 bf16 [d, two_f]; h bf16 [M, d]; gamma bf16 [d];
 * r, s fp32 [M]; dresid nullable bf16 [M, d]. */
coda_status_t coda_gemm_resid_norm_stats_bwd(const void* dyhat, const void* W1, const void* h,
                                             const void* gamma, const float* r, const float* s,
                                             const void* dresid, void* dh, float* dgamma_part,
                                             int M, int d, int two_f, coda_stream_t stream);

/* out[n] = sum_j part[j, n]; part fp32 [nparts, N] (e.g. dgamma). */
coda_status_t coda_col_reduce(const float* part, int nparts, int N, float* out,
                              coda_stream_t stream);

/* RoPE backward with the delayed row scale and the relocated statistic
 * ([pith] Fig. 7; [notes] s3): the GEMM that produces this gradient
 * (attention backward) is outside this library, so the pairwise map runs as
 * its own bandwidth-bound kernel:
 *   dqkv_hat = r[m] R(pos)^T dqkv_rot           (bf16 [M, N])
 *   s[m] = (1/d) sum_n dqkv_rot[m, n] qkv_rot[m, n]   (fp32 [M])
 * dqkv_rot bf16 [M, N]; qkv_rot fp16 [M, N] (the out_f16 copy saved by
 * coda_gemm_rope); r fp32 [M] (nullable: no scale); cos_sin as in
 * coda_gemm_rope; d = width of the normalised input of the QKV GEMM. */
coda_status_t coda_gemm_rope_bwd(const void* dqkv_rot, const void* qkv_rot, const float* r,
                                 const float* cos_sin, int seq_len, int head_dim, int n_rope_cols,
                                 void* dqkv_hat, float* s, int M, int N, int d,
                                 coda_stream_t stream);

/* ------------------------------------------------- LayerNorm variant */
/* The pages promise a LayerNorm composition without working it; this is the
 * library's reading, built the same way as the RMSNorm path ([notes] s2-s3):
 * with mu, r = 1/sqrt(var + eps) per row and the n-vectors w1 = gamma W1,
 * b1 = beta W1 (fp32 [2f], e.g. two M=1 calls of coda_gemm),
 *   ((h - mu) r gamma + beta) W1 = r (hg W1) - (r mu) w1 + b1,
 * and the two LayerNorm-backward statistics relocate into the epilogue of
 * the GEMM producing dy: s_a = (1/d) sum dy w1, s_b = (1/d)(sum dy y -
 * sum dy b1). */

/* GEMM 1: h = x W0 + z, hg = h * gamma (bf16), per-tile partials
 * part_sq[t, m] = sum h^2 and part_sum[t, m] = sum h (fp32
 * [coda_col_tiles(N), M]). Otherwise as coda_gemm_resid_norm_stats. */
coda_status_t coda_gemm_resid_ln_stats(const void* x, const void* W0, const void* z,
                                       const void* gamma, void* h, void* hg, float* part_sq,
                                       float* part_sum, int M, int N, int K, coda_stream_t stream);

/* mu[m] = sum_j part_sum[j, m] / d ;
 * r[m] = 1 / sqrt(max(sum_j part_sq[j, m] / d - mu^2, 0) + eps). */
coda_status_t coda_row_ln(const float* part_sq, const float* part_sum, int nparts, int M, int d,
                          float eps, float* r, float* mu, coda_stream_t stream);

/* GEMM 2: y = r[m] (hg W1) - (r mu)[m] w1[n] + b1[n]; a = SwiGLU(y) (bf16
 * [M, two_f/2]); y_save (nullable) fp16 [M, two_f] (as for
 * coda_gemm_rowscale_swiglu). */
coda_status_t coda_gemm_ln_rowscale_swiglu(const void* hg, const void* W1, const float* r,
                                           const float* mu, const float* w1, const float* b1,
                                           void* a, void* y_save, int M, int two_f, int K,
                                           coda_stream_t stream);

/* SwiGLU backward as coda_gemm_rowscale_swiglu_bwd, plus the row partials
 * spart_w = sum dy w1 and spart_b = sum dy b1 (fp32 [coda_col_tiles(f), M]). */
coda_status_t coda_gemm_ln_rowscale_swiglu_bwd(const void* dout, const void* W2, const void* y,
                                               const float* r, const float* w1, const float* b1,
                                               void* dyhat, float* spart, float* spart_w,
                                               float* spart_b, int M, int f, int d,
                                               coda_stream_t stream);

/* s_a[m] = sum_j spart_w[j, m] / d ; s_b[m] = (sum_j spart[j, m] -
 * sum_j spart_b[j, m]) / d. */
coda_status_t coda_row_ln_bwd(const float* spart, const float* spart_w, const float* spart_b,
                              int nparts, int M, int d, float* s_a, float* s_b,
                              coda_stream_t stream);

/* LayerNorm backward fused into P = dyhat W1^T:
 *   dh = gamma P - r s_a - r^2 s_b (h - mu) (+ dresid)        (bf16 [M, d])
 *   dgamma_part[j, n] = sum over rows 32j.. of P (h - mu)      (fp32)
 *   dbeta_part[j, n]  = sum over rows 32j.. of P / r           (fp32)
 *   hhat (nullable) = (h - mu) gamma + beta / r  (bf16 [M, d]): the operand
 *   of the W1 gradient, dW1 = hhat^T dyhat.
 * beta bf16 [d]; partial shapes [coda_row_tiles32(M), d]. */
coda_status_t coda_gemm_resid_ln_stats_bwd(const void* dyhat, const void* W1, const void* h,
                                           const void* gamma, const void* beta, const float* r,
                                           const float* mu, const float* s_a, const float* s_b,
                                           const void* dresid, void* dh, void* hhat,
                                           float* dgamma_part, float* dbeta_part, int M, int d,
                                           int two_f, coda_stream_t stream);

/* Test hook for the bounded waits: launches one tiny kernel whose only wait
 * is on an mbarrier that nothing arrives at, bounded by timeout_ms. The wait
 * gives up, records CODA_ERR_TIMEOUT in the device error word and the kernel
 * returns normally (no trap, no fault). Synchronises the stream and returns
 * what coda_get_device_error() reports: CODA_ERR_TIMEOUT when the bound
 * worked. */
coda_status_t coda_selftest_bounded_wait(int timeout_ms, coda_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* CODA_H_ */
