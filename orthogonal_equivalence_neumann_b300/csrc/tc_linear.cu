// tc_linear.cu -- the bf16 transformed linear on the tensor-core path.
//
// [POET-X §2.A-§2.C] ("POET-X: Memory-efficient LLM Training by Scaling
// Orthogonal Transformation", gist.science summary): the chain
//   u = gather(x, perm_in) . B_P^T,  z = u . W0m^T,  y = scatter(z . B_R^T, perm_out)
// and its backward.  The frozen-weight products run on tcgen05 (tc_gemm.cu),
// so do the permuted block-diagonal applies (tc_blockapply.cu) for b in
// {128, 256}, and so do the dQ token sums (tc_dq.cu); other block sizes use
// the CUDA-core kernels.
#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace poetx {

#define TC_TRY(expr)                 \
  do {                               \
    poetx_status _st = (expr);       \
    if (_st != POETX_OK) return _st; \
  } while (0)

// bf16 Q: tensor-core chain with bf16 operands (the fp32 path stays exact on the CUDA cores).
bool tc_cnp_supported(int b, poetx_dtype out_dtype) {
  return out_dtype == POETX_BF16 && tc::cnp_supported(b);
}
poetx_status tc_cnp_fwd(const float* theta, int nb, int b, int n, void* Q, poetx_dtype out_dtype,
                        cudaStream_t s) {
  return tc::cnp_fwd_bf16ops(theta, nb, b, n, Q, out_dtype == POETX_F32, s);
}

bool tc_linear_supported(int d_in, int d_out, int b_in, int b_out, poetx_dtype dt) {
  (void)b_in;
  (void)b_out;
  return dt == POETX_BF16 && tc::gemm_supported(d_out, d_in) && tc::gemm_supported(d_in, d_out);
}

// Tensor-core scratch.  Forward: the exchange ring of the cluster block
// applies.  Backward: one region that serves, in turn, the exchange ring of
// the block applies and the gathered activation [T, max(d_in, d_out)] of the
// dQ token sums (dy by perm_out, then x by perm_in); after it, the dense bf16
// K and G of every block (CNP backward).
static bool dq_tc(int d, int b) { return tc::dq_supported(d, b) && tc::permute_supported(d); }

static size_t ring_bytes(int d, int b, bool scatter) {
  return tc::cluster_apply_supported(d, b, scatter) ? tc::cluster_apply_workspace_bytes(d, b, scatter)
                                                    : 0;
}

static size_t shared_region_bytes(int T, int d_in, int d_out, int b_in, int b_out, bool backward) {
  // the backward may also run the forward applies (z recomputed without a saved copy)
  size_t bytes = 0;
  const size_t rings[4] = {ring_bytes(d_in, b_in, false), ring_bytes(d_out, b_out, true),
                           backward ? ring_bytes(d_out, b_out, false) : 0,
                           backward ? ring_bytes(d_in, b_in, true) : 0};
  for (size_t r : rings)
    if (r > bytes) bytes = r;
  if (backward && (dq_tc(d_in, b_in) || dq_tc(d_out, b_out))) {
    const size_t g = (size_t)T * (d_in > d_out ? d_in : d_out) * 2;
    if (g > bytes) bytes = g;
  }
  return round_up(bytes, 256);
}

size_t tc_workspace_bytes(int T, int d_in, int d_out, int b_in, int b_out, poetx_dtype dt,
                          bool backward) {
  if (dt != POETX_BF16) return 0;
  size_t bytes = shared_region_bytes(T, d_in, d_out, b_in, b_out, backward);
  if (backward && tc::cnp_supported(b_in) && tc::cnp_supported(b_out))
    bytes += tc::cnp_bwd_workspace_bytes(d_in, b_in, d_out, b_out);
  return bytes;
}

int tc_dq_slots(int T, int d, int b, poetx_dtype dt) {
  return (dt == POETX_BF16 && dq_tc(d, b)) ? tc::dq_splits(T, d, b) : 1;
}

// Offset of the CNP backward's part of the tensor-core scratch.
size_t tc_cnp_ws_offset(int T, int d_in, int d_out, int b_in, int b_out) {
  return shared_region_bytes(T, d_in, d_out, b_in, b_out, true);
}

// Permuted block apply: a thread-block cluster when the shape allows, else one
// CTA per token slab on the tensor cores, else the CUDA cores.  `inv` is the
// inverse of the gather permutation.
static poetx_status block_apply(const void* in, void* out, const void* Q, int T, int d, int b,
                                const int32_t* gath, const int32_t* inv, const int32_t* scat,
                                bool transpose_q, void* ws, cudaStream_t s) {
  const bool scatter = scat != nullptr;
  if (tc::cluster_apply_supported(d, b, scatter))
    return tc::cluster_apply_bf16(in, out, Q, scatter ? scat : gath, inv, T, d, b, transpose_q,
                                  scatter, ws, tc::cluster_apply_workspace_bytes(d, b, scatter), s);
  if (tc::blockapply_supported(d, b))
    return tc::blockapply_bf16(in, out, Q, gath ? gath : scat, T, d, b, transpose_q, scatter, s);
  return launch_block_apply_simt(in, out, Q, T, d, b, gath, scat, transpose_q, POETX_BF16, s);
}

// dQ token sums: gather once, then tensor cores, when the shape allows; CUDA cores otherwise.
// `slots` partial sums on the tensor-core path (each written whole), one plain sum otherwise.
static poetx_status dq(const void* G, const void* V, int T, int d, int b, const int32_t* gG,
                       const int32_t* gV, float* out, int slots, void* gbuf, cudaStream_t s) {
  if (dq_tc(d, b)) {
    if (gG) {
      TC_TRY(tc::permute_cols_bf16(G, gbuf, gG, T, d, s));
      return tc::dq_bf16(gbuf, V, T, d, b, slots, out, s);
    }
    TC_TRY(tc::permute_cols_bf16(V, gbuf, gV, T, d, s));
    return tc::dq_bf16(G, gbuf, T, d, b, slots, out, s);
  }
  return launch_dq_simt(G, V, T, d, b, gG, gV, out, POETX_BF16, s);
}

poetx_status tc_forward(const void* x, const void* W0m, const void* Q_P, const void* Q_R,
                        const int32_t* perm_in, const int32_t* inv_in, const int32_t* perm_out,
                        const int32_t* inv_out, int T, int d_in, int d_out, int b_in, int b_out,
                        void* u, void* z, void* y, void* ws, cudaStream_t s) {
  TC_TRY(block_apply(x, u, Q_P, T, d_in, b_in, perm_in, inv_in, nullptr, false, ws, s));
  TC_TRY(tc::gemm_bf16(u, W0m, z, T, d_out, d_in, false, s));
  if (y) TC_TRY(block_apply(z, y, Q_R, T, d_out, b_out, nullptr, nullptr, perm_out, false, ws, s));
  return POETX_OK;
}

poetx_status tc_backward(const void* x, const void* dy, const void* W0m, const void* Q_P,
                         const void* Q_R, const void* z, const int32_t* perm_in,
                         const int32_t* inv_in, const int32_t* perm_out, const int32_t* inv_out,
                         int T, int d_in, int d_out, int b_in, int b_out, void* dX, void* gz,
                         void* gu, float* dqp, int slots_p, float* dqr, int slots_r, void* ws,
                         cudaStream_t s) {
  TC_TRY(block_apply(dy, gz, Q_R, T, d_out, b_out, perm_out, inv_out, nullptr, true, ws, s));
  TC_TRY(dq(dy, z, T, d_out, b_out, perm_out, nullptr, dqr, slots_r, ws, s));
  TC_TRY(tc::gemm_bf16(gz, W0m, gu, T, d_in, d_out, true, s));
  TC_TRY(block_apply(gu, dX, Q_P, T, d_in, b_in, nullptr, nullptr, perm_in, true, ws, s));
  TC_TRY(dq(gu, x, T, d_in, b_in, nullptr, perm_in, dqp, slots_p, ws, s));
  return POETX_OK;
}

}  // namespace poetx
