// tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) path for sm_103a: host-side entry points.
#pragma once

#include "poetx.h"

namespace poetx {

// Cayley-Neumann forward on the tensor cores.
bool tc_cnp_supported(int b, poetx_dtype out_dtype);
poetx_status tc_cnp_fwd(const float* theta, int nb, int b, int n, void* Q, poetx_dtype out_dtype,
                        cudaStream_t s);

// Transformed linear (bf16 activations, fp32 accumulation) on the tensor cores.
bool tc_linear_supported(int d_in, int d_out, int b_in, int b_out, poetx_dtype dt);
size_t tc_workspace_bytes(int T, int d_in, int d_out, int b_in, int b_out, poetx_dtype dt,
                          bool backward);
size_t tc_cnp_ws_offset(int T, int d_in, int d_out, int b_in, int b_out);
// Partial-sum slots the tensor-core dQ would use for a side (1 off that path).
int tc_dq_slots(int T, int d, int b, poetx_dtype dt);
poetx_status tc_forward(const void* x, const void* W0m, const void* Q_P, const void* Q_R,
                        const int32_t* perm_in, const int32_t* inv_in, const int32_t* perm_out,
                        const int32_t* inv_out, int T, int d_in, int d_out, int b_in, int b_out,
                        void* u, void* z, void* y, void* ws, cudaStream_t s);
// One scattered block apply of bf16 rows on the fastest kernel that takes the
// shape: out[t][scat(jb + i)] = sum_k Qop_j[i][k] in[t][jb + k], Qop = Q or
// (transpose_q) Q^T.  `ws` holds tc_scatter_apply_bytes(T, d, b).
size_t tc_scatter_apply_bytes(int T, int d, int b);
poetx_status tc_scatter_apply(const void* in, void* out, const void* Q, int T, int d, int b,
                              const int32_t* scat, bool transpose_q, void* ws, cudaStream_t s);
// The Cayley-Neumann backward of both sides, when tc_backward runs it too.
struct TcCnpBwd {
  const float* theta_P;
  const float* theta_R;
  int n;
  float* dtheta_P;
  float* dtheta_R;
  void* ws;   // cnp_bwd_workspace_bytes(d_in, b_in, d_out, b_out)
};
// With `cnp`, the R side's block backward runs on a library stream as soon as
// dQ_R is summed, next to the g_u GEMM, and joins `s` before the call returns.
poetx_status tc_backward(const void* x, const void* dy, const void* W0m, const void* Q_P,
                         const void* Q_R, const void* z, const int32_t* perm_in,
                         const int32_t* inv_in, const int32_t* perm_out, const int32_t* inv_out,
                         int T, int d_in, int d_out, int b_in, int b_out, void* dX, void* gz,
                         void* gu, float* dqp, int slots_p, float* dqr, int slots_r, void* ws,
                         const TcCnpBwd* cnp, cudaStream_t s);

namespace tc {
// C[M,N] (bf16) = A[M,K] . B^T with A [M,K] and B [N,K] (b_mn == false) or
// B [K,N] (b_mn == true), all bf16 row-major, fp32 accumulation (tcgen05).
bool gemm_supported(int N, int K);
// reserve_sms: SMs to leave to kernels on another stream (where that adds no
// round of output tiles).
poetx_status gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, bool b_mn,
                       cudaStream_t s, int reserve_sms = 0);

// Permuted block-diagonal apply, bf16 in/out, fp32 accumulation (tcgen05):
//   scatter == false: out[t][jb+i] = sum_k Qop_j[i][k] in[t][perm[jb+k]]
//   scatter == true:  out[t][perm[jb+i]] = sum_k Qop_j[i][k] in[t][jb+k]
// with Qop_j = Q_j, or Q_j^T when transpose_q.  b in {128, 256}.
bool blockapply_supported(int d, int b);
poetx_status blockapply_bf16(const void* in, void* out, const void* Q, const int32_t* perm, int T,
                             int d, int b, bool transpose_q, bool scatter, cudaStream_t s);

// The same permuted block apply over a thread-block cluster: the permutation
// travels between the CTAs' shared memories and each CTA keeps its blocks'
// Qop in tensor memory.  `inv` is the inverse of `perm` (gather form only).
// Scratch: a small exchange ring in `ws` (cluster_apply_workspace_bytes).
bool cluster_apply_supported(int d, int b, bool scatter);
size_t cluster_apply_workspace_bytes(int T, int d, int b, bool scatter);
int cluster_apply_clusters(int T, int d, int b, bool scatter);
// max_clusters > 0 caps the clusters of the launch (SMs left to another stream).
poetx_status cluster_apply_bf16(const void* in, void* out, const void* Q, const int32_t* perm,
                                const int32_t* inv, int T, int d, int b, bool transpose_q,
                                bool scatter, void* ws, size_t ws_bytes, cudaStream_t s, int max_clusters = 0);

// Unpermuted block apply, bf16 in/out, fp32 accumulation (tcgen05), one CTA
// per (block, token stripe) with the block's Qop resident in tensor memory:
//   out[t][jb+i] = sum_k Qop_j[i][k] in[t][jb+k],  Qop_j = Q_j or Q_j^T.
// b in {128, 256}.  With a column permutation before or after it, the
// permuted applies of the shapes the cluster form does not take.
bool plain_apply_supported(int d, int b);
poetx_status plain_apply_bf16(const void* in, void* out, const void* Q, int T, int d, int b,
                              bool transpose_q, cudaStream_t s);

// dQ_j[i][k] = sum_t G[t][jb+i] V[t][jb+k] (both operands already gathered),
// as n_split partial sums over token ranges: part [n_split][d/b, b, b] fp32,
// every slot written (the sum over slots is dQ).  dq_splits gives the count
// that keeps the GPU busy.
bool dq_supported(int d, int b);
// The same sums with the permuted operand gathered in flight through a
// thread-block cluster (no permuted copy in HBM): P is the activation to be
// gathered (natural layout), inv the inverse of its gather permutation, Vc the
// unpermuted operand; gather_a: P gives the rows i (dQ_R), else the columns k
// (dQ_P).  part: cluster_dq_splits(T, d, b) slots (min(that, max_clusters) when
// max_clusters > 0), every one written; T > 0.
bool cluster_dq_supported(int d, int b);
int cluster_dq_splits(int T, int d, int b);
size_t cluster_dq_workspace_bytes(int T, int d, int b);
poetx_status cluster_dq_bf16(const void* P, const void* Vc, const int32_t* inv, int T, int d, int b,
                             bool gather_a, float* part, void* ws, size_t ws_bytes, cudaStream_t s,
                             int max_clusters = 0);
int dq_splits(int T, int d, int b);
poetx_status dq_bf16(const void* G, const void* V, int T, int d, int b, int n_split, float* part,
                     cudaStream_t s);

// out[t][c] = in[t][perm[c]] for bf16 token-major [T, d] (one pass over HBM).
bool permute_supported(int d);
poetx_status permute_cols_bf16(const void* in, void* out, const int32_t* perm, int T, int d,
                               cudaStream_t s);

// Cayley-Neumann forward for b in {32, 64, 128}: the parameters unpacked in
// shared memory, 128 / b blocks per 128-row tile (block-diagonal), bf16 Q
// from bf16 operands or fp32 Q from a three-term split of every operand
// into fp16 parts; both factors of a layer in one launch (nb0 or nb1 may be
// 0).  Any block count.
bool cnp_tile_supported(int b);
poetx_status cnp_tile_fwd(const float* theta0, int nb0, const float* theta1, int nb1, int b, int n,
                          void* Q0, void* Q1, bool out_f32, cudaStream_t s);

// Cayley-Neumann forward / backward with bf16 operands and fp32 accumulation
// (tcgen05), b in {128, 256}; the forward also gives fp32 Q at b = 256 (each
// product as three products of the operands' fp16 parts).  The backward
// overwrites dtheta.
bool cnp_supported(int b);
poetx_status cnp_fwd_bf16ops(const float* theta, int nb, int b, int n, void* Q, bool out_f32,
                             cudaStream_t s);
// Both factors of a layer (same b) in one launch.
poetx_status cnp_fwd_pair_bf16ops(const float* theta0, int nb0, const float* theta1, int nb1,
                                  int b, int n, void* Q0, void* Q1, bool out_f32, cudaStream_t s);
// Backward of both sides of a layer in one launch (after a prep kernel that
// writes dense bf16 K and G into `ws`, cnp_bwd_workspace_bytes of it).
size_t cnp_bwd_workspace_bytes(int d_in, int b_in, int d_out, int b_out);
// One side alone (its workspace part: 10 * nb * b * b bytes, the P side's at
// the start of the CNP backward workspace, the R side's after it); the chain
// kernel runs one cluster of (b/128) * (b/64) CTAs per block, and
// with `narrow` two CTAs per block that stream K and G through a ring (for
// running beside a kernel that holds most SMs: cnp_bwd_ctas(nb, b) = nb * b /
// 128 is the count of SMs that kernel leaves free).  parts (bit flags): 1 =
// dense bf16 K and K^T from theta (needs only theta: may run early), 2 = the
// summed dQ as bf16 G, 4 = the chain (after both); 7 = all three.
poetx_status cnp_bwd_side(const float* theta, const float* dQ, int splits, int nb, int b, int n,
                          float* dtheta, void* ws, cudaStream_t s, int parts = 7,
                          bool narrow = false);
int cnp_bwd_ctas(int nb, int b);
// dQ_P / dQ_R come as `splits_P` / `splits_R` partial-sum slots [splits][nb, b, b].
poetx_status cnp_bwd_layer(const float* theta_P, const float* dQ_P, int splits_P, int nb_P, int b_P,
                           const float* theta_R, const float* dQ_R, int splits_R, int nb_R, int b_R,
                           int n, float* dtheta_P, float* dtheta_R, void* ws, cudaStream_t s);
}  // namespace tc

}  // namespace poetx
