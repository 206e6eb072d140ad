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

// The backward's tensor-core scratch: dense bf16 K and G of every block (CNP backward).
size_t tc_workspace_bytes(int T, int d_in, int d_out, int b_in, int b_out, poetx_dtype dt,
                          bool backward) {
  (void)T;
  if (!backward || dt != POETX_BF16 || !tc::cnp_supported(b_in) || !tc::cnp_supported(b_out))
    return 0;
  return tc::cnp_bwd_workspace_bytes(d_in, b_in, d_out, b_out);
}

// Permuted block apply: tensor cores when the shape allows, CUDA cores otherwise.
static poetx_status block_apply(const void* in, void* out, const void* Q, int T, int d, int b,
                                const int32_t* gath, const int32_t* scat, bool transpose_q,
                                cudaStream_t s) {
  if (tc::blockapply_supported(d, b))
    return tc::blockapply_bf16(in, out, Q, gath ? gath : scat, T, d, b, transpose_q,
                               scat != nullptr, s);
  return launch_block_apply_simt(in, out, Q, T, d, b, gath, scat, transpose_q, POETX_BF16, s);
}

// dQ token sums: tensor cores when the shape allows, CUDA cores otherwise.
static poetx_status dq(const void* G, const void* V, int T, int d, int b, const int32_t* gG,
                       const int32_t* gV, float* out, cudaStream_t s) {
  if (tc::dq_supported(d, b)) return tc::dq_bf16(G, V, T, d, b, gG, gV, out, s);
  return launch_dq_simt(G, V, T, d, b, gG, gV, out, POETX_BF16, s);
}

poetx_status tc_forward(const void* x, const void* W0m, const void* Q_P, const void* Q_R,
                        const int32_t* perm_in, const int32_t* inv_in, const int32_t* perm_out,
                        const int32_t* inv_out, int T, int d_in, int d_out, int b_in, int b_out,
                        void* u, void* z, void* y, void* ws, cudaStream_t s) {
  (void)inv_in;
  (void)inv_out;
  (void)ws;
  TC_TRY(block_apply(x, u, Q_P, T, d_in, b_in, perm_in, nullptr, false, s));
  TC_TRY(tc::gemm_bf16(u, W0m, z, T, d_out, d_in, false, s));
  if (y) TC_TRY(block_apply(z, y, Q_R, T, d_out, b_out, nullptr, perm_out, false, s));
  return POETX_OK;
}

poetx_status tc_backward(const void* x, const void* dy, const void* W0m, const void* Q_P,
                         const void* Q_R, const void* z, const int32_t* perm_in,
                         const int32_t* inv_in, const int32_t* perm_out, const int32_t* inv_out,
                         int T, int d_in, int d_out, int b_in, int b_out, void* dX, void* gz,
                         void* gu, float* dqp, float* dqr, void* ws, cudaStream_t s) {
  (void)inv_in;
  (void)inv_out;
  (void)ws;
  TC_TRY(block_apply(dy, gz, Q_R, T, d_out, b_out, perm_out, nullptr, true, s));
  TC_TRY(dq(dy, z, T, d_out, b_out, perm_out, nullptr, dqr, s));
  TC_TRY(tc::gemm_bf16(gz, W0m, gu, T, d_in, d_out, true, s));
  TC_TRY(block_apply(gu, dX, Q_P, T, d_in, b_in, nullptr, perm_in, true, s));
  TC_TRY(dq(gu, x, T, d_in, b_in, nullptr, perm_in, dqp, s));
  return POETX_OK;
}

}  // namespace poetx
