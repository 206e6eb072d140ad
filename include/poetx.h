/*
 * poetx.h -- C ABI of the POET-X transformed-linear library for B300 (sm_103a).
 *
 * The layer: a linear map whose effective weight is the orthogonal
 * equivalence transform W = R . W0 . P of a frozen W0, applied input-centric
 * as y = R (W0 (P x)) so that R . W0 . P is never formed.  R and P are
 * block-diagonal orthogonal matrices conjugated by index-only permutations;
 * each b x b block is built from b(b-1)/2 packed skew parameters by the
 * Cayley-Neumann parameterisation.
 *
 * Source: the page "POET-X: Memory-efficient LLM Training by Scaling
 * Orthogonal Transformation" (gist.science technical summary), section 2:
 *   §2.A input-centric implementation      §2.B permutations as index maps,
 *   §2.C batched block-diagonal blocks          merged into W0 (4 -> 2)
 *   §2.D Cayley-Neumann parameterisation   §2.E POET-Xfast / POET-Xmem
 *
 * Conventions (the page fixes none; these are the library's definitions):
 *   - every matrix and activation is row-major; activations are token-major,
 *     x [T, d_in], y [T, d_out]; W0 is [d_out, d_in] and y = x W^T;
 *   - a permutation is an int32 array perm[d] holding each of 0..d-1 once;
 *     applying it gathers, (Pi v)_i = v[perm[i]]; inv[perm[i]] = i;
 *   - P = Pi_P^T B_P Pi_P and R = Pi_R^T B_R Pi_R with
 *     B = blockdiag(Q_0, .., Q_{d/b-1}); perm_in belongs to P, perm_out to R;
 *   - packed skew parameters theta [nb, b(b-1)/2] fp32 fill each block's
 *     strict upper triangle row by row, (0,1),(0,2),..,(0,b-1),(1,2),..;
 *     K[i][k] = theta, K[k][i] = -theta;
 *   - Cayley-Neumann with n terms: Q = (I + K)(I + K + K^2 + ... + K^n)
 *     (the Cayley map with (I - K)^{-1} replaced by its Neumann series).
 *
 * Memory and streams: every pointer argument is a DEVICE pointer unless its
 * description says otherwise, aligned to 16 bytes.  The caller owns every
 * buffer; the library allocates no device memory (scratch comes in through
 * `workspace`, sized by poetx_workspace_bytes).  Every call is asynchronous
 * on `stream`.  Argument errors are detected on the host and returned before
 * anything is launched; nothing throws across this ABI.  Errors raised while
 * kernels run surface as POETX_ERR_CUDA from a later call or from
 * poetx_stream_status().  Kernels that wait on the tensor-core pipeline use
 * bounded waits: on expiry they set a device error word instead of hanging,
 * read back by poetx_stream_status() as POETX_ERR_TIMEOUT; a kernel that meets
 * a value outside the range it computes in sets POETX_ERR_RANGE there.
 */
#ifndef POETX_H
#define POETX_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  POETX_OK = 0,
  POETX_ERR_INVALID_ARG = 1,     /* null pointer, misaligned pointer, bad enum, n < 1 */
  POETX_ERR_SHAPE = 2,           /* d % b != 0, negative sizes, workspace too small */
  POETX_ERR_UNSUPPORTED = 3,     /* block size outside the supported set */
  POETX_ERR_NOT_PERMUTATION = 4, /* poetx_check_perm: an index repeats or is out of range */
  POETX_ERR_CUDA = 5,            /* a CUDA runtime call or a launch failed */
  POETX_ERR_TIMEOUT = 6,         /* a bounded device-side wait expired */
  POETX_ERR_RANGE = 7            /* a value left the range a kernel computes in */
} poetx_status;

typedef enum { POETX_F32 = 0, POETX_BF16 = 1 } poetx_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *poetx_status_string(poetx_status s);

/* Library version as 10000*major + 100*minor + patch. */
int poetx_version(void);

/* Block sizes: any power of two 2 <= b <= 256 for POETX_F32; the bf16
 * tensor-core path takes b in {32, 64, 128, 256}. */

/* ------------------------------------------------------------------------ */
/* Cayley-Neumann parameterisation [POET-X §2.D]                            */
/* ------------------------------------------------------------------------ */

/* Batched CNP: Q_j = (I + K_j)(I + K_j + ... + K_j^n) for j < nb.
 *   theta  [nb, b(b-1)/2] fp32, packed as above (read only)
 *   Q      [nb, b, b] in out_dtype (fp32 or bf16; written)
 *   n >= 1 is the highest Neumann power.  nb == 0 is a no-op.
 * fp32 Q at b in {32, 64, 128, 256} (at b = 256: nb <= 65535) runs on the
 * tensor cores with each chain value held as two fp16 parts: an intermediate
 * power sum of magnitude 65504 or more (far outside the series' convergent
 * range) leaves Q undefined and sets POETX_ERR_RANGE for
 * poetx_stream_status(). */
poetx_status poetx_cayley_neumann(const float *theta, int nb, int b, int n, void *Q,
                                  poetx_dtype out_dtype, cudaStream_t stream);

/* Both factors of one layer, Q_P from theta_P and Q_R from theta_R, with the
 * same n [§2.C: all blocks are processed as one batch]: identical results to
 * two poetx_cayley_neumann calls, in a single launch when b_P == b_R (bf16
 * output).  Arguments as poetx_cayley_neumann, per factor; nb_P or nb_R may be
 * 0 (that factor is skipped and its pointers are not read). */
poetx_status poetx_cayley_neumann_pair(const float *theta_P, int nb_P, int b_P,
                                       const float *theta_R, int nb_R, int b_R, int n, void *Q_P,
                                       void *Q_R, poetx_dtype out_dtype, cudaStream_t stream);

/* Backward of poetx_cayley_neumann (not on the page, which only says
 * "autograd" [§2.E]; this is the chain rule of the forward):
 *   dK = sum_{m=1}^{n+1} c_m sum_{a=0}^{m-1} (K^a)^T dQ (K^{m-1-a})^T,
 *   c_m = 2 for m <= n, c_{n+1} = 1;  dtheta_(i,k) = dK[i][k] - dK[k][i].
 *   dQ      [nb, b, b] fp32 (read only), dL/dQ of each block
 *   dtheta  [nb, b(b-1)/2] fp32, overwritten. */
poetx_status poetx_cayley_neumann_backward(const float *theta, const float *dQ, int nb, int b,
                                           int n, float *dtheta, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Permutations as index maps [POET-X §2.B]                                 */
/* ------------------------------------------------------------------------ */

/* inv[perm[i]] = i for i < d (bit-exact integer work).  perm must be a
 * permutation (see poetx_check_perm); otherwise inv is unspecified. */
poetx_status poetx_invert_perm(const int32_t *perm, int32_t *inv, int d, cudaStream_t stream);

/* Validator: returns POETX_OK if perm holds each of 0..d-1 exactly once and,
 * when inv is not NULL, inv[perm[i]] == i for all i; POETX_ERR_NOT_PERMUTATION
 * otherwise.  Synchronises `stream` (it returns a verdict).  `scratch` is a
 * device buffer of at least d + 1 int32 (overwritten). */
poetx_status poetx_check_perm(const int32_t *perm, const int32_t *inv, int d, int32_t *scratch,
                              cudaStream_t stream);

/* Merge the two inner permutations into the frozen weight, once per inner
 * loop [§2.B "4 -> 2 permutations per step"]:
 *   W0m[i][k] = W0[perm_out[i]][perm_in[k]],  i.e. W0m = Pi_R W0 Pi_P^T.
 * W0, W0m [d_out, d_in] in `dtype` (must not alias). */
poetx_status poetx_merge_w0(const void *W0, void *W0m, int d_out, int d_in, poetx_dtype dtype,
                            const int32_t *perm_out, const int32_t *perm_in,
                            cudaStream_t stream);

/* End of an inner loop [§2.B: the permutations are fixed for an inner loop
 * and merged into the weight; the learned rotations are then folded into the
 * frozen weight before new permutations are drawn]: the effective weight in
 * the original coordinates,
 *   W0_new = R W0 P = Pi_R^T B_R W0m B_P Pi_P,
 * from the merged W0m = Pi_R W0 Pi_P^T of poetx_merge_w0 and the current
 * blocks Q_P, Q_R (poetx_cayley_neumann of the current theta).  The caller
 * then resets theta (to zero: Q = I), draws new permutations and merges
 * W0_new with them (poetx_merge_w0).
 * Arguments (device, `dtype` unless stated): W0m [d_out, d_in],
 *   Q_P [d_in/b_in, b_in, b_in], Q_R [d_out/b_out, b_out, b_out],
 *   perm_in int32 [d_in], perm_out int32 [d_out] (the permutations W0m was
 *   merged with), W0_new [d_out, d_in] written (may be W0m itself: the fold
 *   can run in place), workspace of ws_bytes >= poetx_fold_workspace_bytes.
 * Two scattered block applies (on the rows of W0m, then on the rows of its
 * transpose) and two transposes; bf16 runs the applies on the tensor cores
 * with fp32 accumulation and one bf16 rounding of the intermediate. */
size_t poetx_fold_workspace_bytes(int d_out, int d_in, int b_in, int b_out, poetx_dtype dtype);
poetx_status poetx_fold_w0(const void *W0m, const void *Q_P, const void *Q_R,
                           const int32_t *perm_in, const int32_t *perm_out, int d_out, int d_in,
                           int b_in, int b_out, poetx_dtype dtype, void *W0_new, void *workspace,
                           size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* The transformed linear [POET-X §2.A-§2.C, §2.E]                          */
/* ------------------------------------------------------------------------ */

/* Bytes of `workspace` that poetx_forward / poetx_backward need for these
 * sizes (the larger of the two, including the recompute of z when the
 * backward is called without a saved z).  Returns 0 for invalid sizes. */
size_t poetx_workspace_bytes(int T, int d_in, int d_out, int b_in, int b_out, poetx_dtype dtype);

/* Forward, y = Pi_R^T B_R W0m B_P Pi_P x with W0m from poetx_merge_w0:
 *   u = gather(x, perm_in) . blockdiag(Q_P)^T      (permutation on the load)
 *   z = u . W0m^T                                   (the frozen weight)
 *   y = scatter(z . blockdiag(Q_R)^T, perm_out)     (permutation on the store)
 * Arguments (all device, act_dtype unless stated):
 *   x [T, d_in], W0m [d_out, d_in], Q_P [d_in/b_in, b_in, b_in],
 *   Q_R [d_out/b_out, b_out, b_out], perm_in/inv_in int32 [d_in],
 *   perm_out/inv_out int32 [d_out]  (inv = poetx_invert_perm(perm)),
 *   y [T, d_out] written,
 *   z_save [T, d_out] written with z when not NULL (POET-Xfast keeps it for
 *          the backward; NULL = POET-Xmem, the backward recomputes it),
 *   workspace of ws_bytes >= poetx_workspace_bytes(...).
 * T == 0 is a no-op. */
poetx_status poetx_forward(const void *x, const void *W0m, const void *Q_P, const void *Q_R,
                           const int32_t *perm_in, const int32_t *inv_in,
                           const int32_t *perm_out, const int32_t *inv_out, int T, int d_in,
                           int d_out, int b_in, int b_out, poetx_dtype act_dtype, void *y,
                           void *z_save, void *workspace, size_t ws_bytes,
                           cudaStream_t stream);

/* Backward for an upstream gradient dy [T, d_out] (act_dtype):
 *   g_r = gather(dy, perm_out);  g_z = g_r . blockdiag(Q_R)
 *   dQ_R,j = sum_t g_r,j^T z_j;  g_u = g_z . W0m
 *   dQ_P,j = sum_t g_u,j^T gather(x, perm_in)_j
 *   dX = scatter(g_u . blockdiag(Q_P), perm_in)
 *   dtheta_P, dtheta_R = poetx_cayley_neumann_backward(theta, dQ, n)
 * Arguments as poetx_forward, plus theta_P [d_in/b_in, b_in(b_in-1)/2] and
 * theta_R fp32 (the parameters Q_P, Q_R were made from, with the same n),
 * z_saved = the z_save of the forward, or NULL to recompute it (POET-Xmem);
 * outputs dX [T, d_in] (act_dtype), dtheta_P, dtheta_R fp32 packed,
 * all overwritten.  W0 is frozen: there is no dW0. */
poetx_status poetx_backward(const void *x, const void *dy, const void *W0m, const float *theta_P,
                            const float *theta_R, int n, const void *Q_P, const void *Q_R,
                            const void *z_saved, const int32_t *perm_in, const int32_t *inv_in,
                            const int32_t *perm_out, const int32_t *inv_out, int T, int d_in,
                            int d_out, int b_in, int b_out, poetx_dtype act_dtype, void *dX,
                            float *dtheta_P, float *dtheta_R, void *workspace, size_t ws_bytes,
                            cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Forward for callers that cannot allocate device memory                   */
/* (this entry point has no counterpart in the paper)                       */
/* ------------------------------------------------------------------------ */

/* Size of the library's own static device array that serves as the
 * workspace of poetx_forward_noalloc: 32 MiB, held by every device that
 * loads the library until the process exits. */
#define POETX_NOALLOC_WORKSPACE_BYTES ((size_t)32 << 20)

/* poetx_forward for callers that cannot call cudaMalloc (for instance a host
 * framework that owns all device memory through its own pool, or a loop in
 * which allocating is forbidden after start-up).  Same arguments and result
 * as poetx_forward, without `workspace`: the scratch is a file-scope static
 * device array of POETX_NOALLOC_WORKSPACE_BYTES inside the library.  The
 * caller still owns x, the weights, y and z_save.  This call allocates no
 * device memory.
 *   - Sizes whose forward scratch (the forward's part of
 *     poetx_workspace_bytes(T, d_in, d_out, b_in, b_out, act_dtype)) exceeds
 *     POETX_NOALLOC_WORKSPACE_BYTES are rejected with POETX_ERR_SHAPE before
 *     anything is launched (e.g. T up to about 2600 tokens for
 *     d_in = d_out = 2048 in bf16).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.  The cached address belongs
 *     to the device's current context: calls must not span a
 *     cudaDeviceReset (which may reload the library's device code elsewhere).
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents; calls that overlap on the GPU (on streams with no
 *     ordering between them) race on it and must be serialised by the
 *     caller. */
poetx_status poetx_forward_noalloc(const void *x, const void *W0m, const void *Q_P,
                                   const void *Q_R, const int32_t *perm_in, const int32_t *inv_in,
                                   const int32_t *perm_out, const int32_t *inv_out, int T,
                                   int d_in, int d_out, int b_in, int b_out,
                                   poetx_dtype act_dtype, void *y, void *z_save,
                                   cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* POET-XQ [POET-X §2.E]: the frozen weight stored in INT8                   */
/* ------------------------------------------------------------------------ */
/* The page stores the base weight in INT8 and dequantises it on the fly; it
 * gives no scale granularity.  Reading: one fp32 scale per row, symmetric,
 * codes in [-127, 127]:
 *   scale[i] = max_k |W0[i][k]| / 127              (fp32 division)
 *   W0q[i][k] = rint(W0[i][k] / scale[i])          (fp32 division, ties to even;
 *                                                   a zero row: scale 0, codes 0)
 *   dequantised W0[i][k] = W0q[i][k] * scale[i]    (fp32 product, rounded to dtype)
 * Quantise the merged weight (poetx_merge_w0's output): permuting rows or
 * columns commutes with this quantiser.
 *
 * poetx_quantize_w0: W0 [d_out, d_in] in `dtype` -> W0q int8 [d_out, d_in],
 *   scale fp32 [d_out].  d_in % 4 == 0.
 * poetx_dequantize_w0: the inverse map, W0 [d_out, d_in] in `dtype` written.
 * poetx_forward_xq / poetx_backward_xq: poetx_forward / poetx_backward with
 *   the weight given as (W0q, scale) of the merged weight; every call first
 *   dequantises it into the head of `workspace` (read back by the
 *   tensor-core products while it is still in L2), so only the INT8 codes
 *   and the scales stay resident.  `workspace` of ws_bytes >=
 *   poetx_workspace_bytes_xq(...) = d_out * d_in * sizeof(act) rounded up to
 *   256 bytes + poetx_workspace_bytes(...).  Other arguments, results and
 *   errors as in poetx_forward / poetx_backward. */
poetx_status poetx_quantize_w0(const void *W0, int d_out, int d_in, poetx_dtype dtype,
                               int8_t *W0q, float *scale, cudaStream_t stream);
poetx_status poetx_dequantize_w0(const int8_t *W0q, const float *scale, int d_out, int d_in,
                                 poetx_dtype dtype, void *W0, cudaStream_t stream);
size_t poetx_workspace_bytes_xq(int T, int d_in, int d_out, int b_in, int b_out,
                                poetx_dtype dtype);
poetx_status poetx_forward_xq(const void *x, const int8_t *W0q, const float *scale,
                              const void *Q_P, const void *Q_R, const int32_t *perm_in,
                              const int32_t *inv_in, const int32_t *perm_out,
                              const int32_t *inv_out, int T, int d_in, int d_out, int b_in,
                              int b_out, poetx_dtype act_dtype, void *y, void *z_save,
                              void *workspace, size_t ws_bytes, cudaStream_t stream);
poetx_status poetx_backward_xq(const void *x, const void *dy, const int8_t *W0q,
                               const float *scale, const float *theta_P, const float *theta_R,
                               int n, const void *Q_P, const void *Q_R, const void *z_saved,
                               const int32_t *perm_in, const int32_t *inv_in,
                               const int32_t *perm_out, const int32_t *inv_out, int T, int d_in,
                               int d_out, int b_in, int b_out, poetx_dtype act_dtype, void *dX,
                               float *dtheta_P, float *dtheta_R, void *workspace,
                               size_t ws_bytes, cudaStream_t stream);

/* Diagnostic of the failure path (no counterpart on the page): launches one
 * thread that waits, through the same bounded wait as every tensor-core
 * kernel, on an mbarrier in its own shared memory that nothing arrives on.
 * After `polls` polls (1 <= polls <= 2^20; cluster_scope 0 = the CTA-scope
 * wait, 1 = the cluster-scope wait) it gives up and records
 * POETX_ERR_TIMEOUT in the device error word, which the next
 * poetx_stream_status() on `stream` returns (and clears).  Nothing else is
 * touched: the context stays usable.  Returns POETX_ERR_INVALID_ARG for
 * arguments out of range, else the launch status. */
poetx_status poetx_diag_expire_wait(int cluster_scope, unsigned polls, cudaStream_t stream);

/* Synchronises `stream` and reports the first error since the last call:
 * a CUDA error (POETX_ERR_CUDA) or an expired device-side wait
 * (POETX_ERR_TIMEOUT).  Clears the device error word. */
poetx_status poetx_stream_status(cudaStream_t stream);


/* ------------------------------------------------------------------------ */
/* Measurement (host-side; off by default)                                  */
/* ------------------------------------------------------------------------ */

/* Number of kernels this library has launched since it was loaded. */
unsigned long long poetx_launch_count(void);

/* While enabled, every kernel launch of the library is bracketed by a pair of
 * CUDA events recorded on the launch's own stream (no device memory is
 * allocated; events are recycled).  Returns POETX_OK. */
poetx_status poetx_profile_enable(int enable);

/* Waits for the recorded events and writes one line per kernel name,
 * "<name> <launches> <total_ms>\n", into buf (host memory, NUL-terminated,
 * truncated to len); then forgets them.  Returns the full report length, or
 * -1 if an event could not be read. */
int poetx_profile_report(char *buf, size_t len);

#ifdef __cplusplus
}
#endif

#endif /* POETX_H */
