// api.cu -- the C ABI (include/poetx.h): argument checks and dispatch.
//
// Every entry point validates on the host and returns before any launch on a
// bad argument; kernels then run asynchronously on the caller's stream.
#include <string.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace poetx {

// The library's device error word (one per device that loads the library).
__device__ int g_poetx_error = 0;

int* device_error_word() {
  int* p = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_poetx_error) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return p;
}

poetx_status check_launch() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? POETX_OK : POETX_ERR_CUDA;
}

namespace {

bool valid_dtype(poetx_dtype d) { return d == POETX_F32 || d == POETX_BF16; }

bool valid_block(int b) { return is_pow2(b) && b >= 2 && b <= 256; }

// Byte layout of the caller's workspace (each region 256-byte aligned).  The
// forward and the backward each lay out their own regions from offset 0.
struct Workspace {
  // forward
  size_t f_u = 0;      // u = B_P Pi_P x                          [T, d_in]  act
  size_t f_z = 0;      // z when the caller keeps no copy          [T, d_out] act
  size_t f_tc = 0;     // tensor-core path scratch
  size_t fwd_bytes = 0;
  // backward
  size_t gz = 0;       // g_z                                      [T, d_out] act
  size_t gu = 0;       // g_u (also u while z is recomputed)       [T, d_in]  act
  size_t dqp = 0;      // dQ_P partial sums                 [slots][d_in * b_in]  f32
  size_t dqr = 0;      // dQ_R partial sums                 [slots][d_out * b_out] f32
  size_t z = 0;        // recomputed z when none was saved         [T, d_out] act
  size_t tc = 0;       // tensor-core path scratch
  size_t bwd_bytes = 0;
  int slots_p = 1;     // dQ_P / dQ_R partial-sum slot counts
  int slots_r = 1;
};

// Whether the backward runs the Cayley-Neumann blocks on the tensor cores.
bool tc_cnp_backward(int d_in, int d_out, int b_in, int b_out, poetx_dtype dt) {
  return dt == POETX_BF16 && tc::cnp_supported(b_in) && tc::cnp_supported(b_out) &&
         d_in / b_in + d_out / b_out <= 65535;
}

// dQ partial-sum slots of one side: the tensor-core dQ writes several (the
// block backward adds them in slot order), the CUDA-core dQ one.
int dq_slots(int T, int d_in, int d_out, int b_in, int b_out, poetx_dtype dt, bool in_side) {
  if (!tc_linear_supported(d_in, d_out, b_in, b_out, dt)) return 1;
  return in_side ? tc_dq_slots(T, d_in, b_in, dt) : tc_dq_slots(T, d_out, b_out, dt);
}

Workspace layout(int T, int d_in, int d_out, int b_in, int b_out, poetx_dtype dt) {
  Workspace w;
  const size_t es = dtype_size(dt);
  const size_t A = 256;
  size_t off = 0;
  w.f_u = off;  off += round_up((size_t)T * d_in * es, A);
  w.f_z = off;  off += round_up((size_t)T * d_out * es, A);
  w.f_tc = off; off += round_up(tc_workspace_bytes(T, d_in, d_out, b_in, b_out, dt, false), A);
  w.fwd_bytes = off;
  off = 0;
  w.gz = off;  off += round_up((size_t)T * d_out * es, A);
  w.gu = off;  off += round_up((size_t)T * d_in * es, A);
  w.slots_p = dq_slots(T, d_in, d_out, b_in, b_out, dt, true);
  w.slots_r = dq_slots(T, d_in, d_out, b_in, b_out, dt, false);
  w.dqp = off; off += round_up((size_t)w.slots_p * d_in * b_in * 4, A);
  w.dqr = off; off += round_up((size_t)w.slots_r * d_out * b_out * 4, A);
  w.z = off;   off += round_up((size_t)T * d_out * es, A);
  w.tc = off;  off += round_up(tc_workspace_bytes(T, d_in, d_out, b_in, b_out, dt, true), A);
  w.bwd_bytes = off;
  return w;
}

bool sizes_ok(int T, int d_in, int d_out, int b_in, int b_out) {
  return T >= 0 && d_in > 0 && d_out > 0 && valid_block(b_in) && valid_block(b_out) &&
         d_in % b_in == 0 && d_out % b_out == 0;
}

poetx_status check_linear_args(int T, int d_in, int d_out, int b_in, int b_out, poetx_dtype dt,
                               std::initializer_list<const void*> required) {
  if (!valid_dtype(dt)) return POETX_ERR_INVALID_ARG;
  if (T < 0 || d_in <= 0 || d_out <= 0) return POETX_ERR_SHAPE;
  if (!is_pow2(b_in) || !is_pow2(b_out) || b_in > 256 || b_out > 256 || b_in < 2 || b_out < 2)
    return POETX_ERR_UNSUPPORTED;
  if (d_in % b_in || d_out % b_out) return POETX_ERR_SHAPE;
  for (const void* p : required) {
    if (p == nullptr) return POETX_ERR_INVALID_ARG;
    if (!aligned16(p)) return POETX_ERR_INVALID_ARG;
  }
  return POETX_OK;
}

#define POETX_TRY(expr)                  \
  do {                                   \
    poetx_status _st = (expr);           \
    if (_st != POETX_OK) return _st;     \
  } while (0)

}  // namespace
}  // namespace poetx

using namespace poetx;

extern "C" {

const char* poetx_status_string(poetx_status s) {
  switch (s) {
    case POETX_OK: return "POETX_OK";
    case POETX_ERR_INVALID_ARG: return "POETX_ERR_INVALID_ARG";
    case POETX_ERR_SHAPE: return "POETX_ERR_SHAPE";
    case POETX_ERR_UNSUPPORTED: return "POETX_ERR_UNSUPPORTED";
    case POETX_ERR_NOT_PERMUTATION: return "POETX_ERR_NOT_PERMUTATION";
    case POETX_ERR_CUDA: return "POETX_ERR_CUDA";
    case POETX_ERR_TIMEOUT: return "POETX_ERR_TIMEOUT";
    case POETX_ERR_RANGE: return "POETX_ERR_RANGE";
  }
  return "POETX_ERR_UNKNOWN";
}

int poetx_version(void) { return 100; }

poetx_status poetx_cayley_neumann(const float* theta, int nb, int b, int n, void* Q,
                                  poetx_dtype out_dtype, cudaStream_t stream) {
  if (!valid_dtype(out_dtype) || n < 1) return POETX_ERR_INVALID_ARG;
  if (nb < 0) return POETX_ERR_SHAPE;
  if (!valid_block(b)) return POETX_ERR_UNSUPPORTED;
  if (nb == 0) return POETX_OK;
  if (!theta || !Q || !aligned16(theta) || !aligned16(Q)) return POETX_ERR_INVALID_ARG;
  if (tc::cnp_tile_supported(b))
    return tc::cnp_tile_fwd(theta, nb, theta, 0, b, n, Q, Q, out_dtype == POETX_F32, stream);
  if (tc_cnp_supported(b, out_dtype) && nb <= 65535)
    return tc_cnp_fwd(theta, nb, b, n, Q, out_dtype, stream);
  return launch_cnp_fwd_simt(theta, nb, b, n, Q, out_dtype, stream);
}

poetx_status poetx_cayley_neumann_pair(const float* theta_P, int nb_P, int b_P,
                                       const float* theta_R, int nb_R, int b_R, int n, void* Q_P,
                                       void* Q_R, poetx_dtype out_dtype, cudaStream_t stream) {
  if (!valid_dtype(out_dtype) || n < 1) return POETX_ERR_INVALID_ARG;
  if (nb_P < 0 || nb_R < 0) return POETX_ERR_SHAPE;
  if (!valid_block(b_P) || !valid_block(b_R)) return POETX_ERR_UNSUPPORTED;
  if ((nb_P > 0 && (!theta_P || !Q_P || !aligned16(theta_P) || !aligned16(Q_P))) ||
      (nb_R > 0 && (!theta_R || !Q_R || !aligned16(theta_R) || !aligned16(Q_R))))
    return POETX_ERR_INVALID_ARG;
  if (b_P == b_R && tc::cnp_tile_supported(b_P))
    return tc::cnp_tile_fwd(theta_P, nb_P, theta_R, nb_R, b_P, n, Q_P, Q_R,
                            out_dtype == POETX_F32, stream);
  if (b_P == b_R && tc_cnp_supported(b_P, out_dtype) && nb_P + nb_R <= 65535)
    return tc::cnp_fwd_pair_bf16ops(theta_P, nb_P, theta_R, nb_R, b_P, n, Q_P, Q_R,
                                    out_dtype == POETX_F32, stream);
  POETX_TRY(poetx_cayley_neumann(theta_P, nb_P, b_P, n, Q_P, out_dtype, stream));
  return poetx_cayley_neumann(theta_R, nb_R, b_R, n, Q_R, out_dtype, stream);
}

poetx_status poetx_cayley_neumann_backward(const float* theta, const float* dQ, int nb, int b,
                                           int n, float* dtheta, cudaStream_t stream) {
  if (n < 1) return POETX_ERR_INVALID_ARG;
  if (nb < 0) return POETX_ERR_SHAPE;
  if (!valid_block(b)) return POETX_ERR_UNSUPPORTED;
  if (nb == 0) return POETX_OK;
  if (!theta || !dQ || !dtheta || !aligned16(theta) || !aligned16(dQ) || !aligned16(dtheta))
    return POETX_ERR_INVALID_ARG;
  return launch_cnp_bwd_simt(theta, dQ, nb, b, n, dtheta, stream);
}

poetx_status poetx_invert_perm(const int32_t* perm, int32_t* inv, int d, cudaStream_t stream) {
  if (d < 0) return POETX_ERR_SHAPE;
  if (d == 0) return POETX_OK;
  if (!perm || !inv) return POETX_ERR_INVALID_ARG;
  return launch_invert_perm(perm, inv, d, stream);
}

poetx_status poetx_check_perm(const int32_t* perm, const int32_t* inv, int d, int32_t* scratch,
                              cudaStream_t stream) {
  if (d < 0) return POETX_ERR_SHAPE;
  if (d == 0) return POETX_OK;
  if (!perm || !scratch) return POETX_ERR_INVALID_ARG;
  int32_t flag = 0;
  POETX_TRY(launch_check_perm(perm, inv, d, scratch, &flag, stream));
  return flag ? POETX_ERR_NOT_PERMUTATION : POETX_OK;
}

poetx_status poetx_merge_w0(const void* W0, void* W0m, int d_out, int d_in, poetx_dtype dtype,
                            const int32_t* perm_out, const int32_t* perm_in,
                            cudaStream_t stream) {
  if (!valid_dtype(dtype)) return POETX_ERR_INVALID_ARG;
  if (d_out <= 0 || d_in <= 0) return POETX_ERR_SHAPE;
  if (!W0 || !W0m || !perm_out || !perm_in || W0 == W0m) return POETX_ERR_INVALID_ARG;
  return launch_merge_w0(W0, W0m, d_out, d_in, dtype, perm_out, perm_in, stream);
}

// [§2.B] fold at the end of an inner loop: W0_new = Pi_R^T B_R W0m B_P Pi_P.
// Workspace: one [d_out, d_in] matrix, then (bf16) the exchange ring of the
// larger of the two scattered applies.
static size_t fold_ring_bytes(int d_out, int d_in, int b_in, int b_out, poetx_dtype dtype) {
  if (dtype != POETX_BF16) return 0;
  const size_t a = tc_scatter_apply_bytes(d_out, d_in, b_in);
  const size_t b = tc_scatter_apply_bytes(d_in, d_out, b_out);
  return a > b ? a : b;
}

size_t poetx_fold_workspace_bytes(int d_out, int d_in, int b_in, int b_out, poetx_dtype dtype) {
  if (!valid_dtype(dtype) || !sizes_ok(0, d_in, d_out, b_in, b_out)) return 0;
  return round_up((size_t)d_out * d_in * dtype_size(dtype), 256) +
         round_up(fold_ring_bytes(d_out, d_in, b_in, b_out, dtype), 256);
}

poetx_status poetx_fold_w0(const void* W0m, const void* Q_P, const void* Q_R,
                           const int32_t* perm_in, const int32_t* perm_out, int d_out, int d_in,
                           int b_in, int b_out, poetx_dtype dtype, void* W0_new, void* workspace,
                           size_t ws_bytes, cudaStream_t stream) {
  POETX_TRY(check_linear_args(0, d_in, d_out, b_in, b_out, dtype,
                              {W0m, Q_P, Q_R, perm_in, perm_out, W0_new, workspace}));
  if (ws_bytes < poetx_fold_workspace_bytes(d_out, d_in, b_in, b_out, dtype))
    return POETX_ERR_SHAPE;
  char* ws = static_cast<char*>(workspace);
  void* M = ws;   // [d_out, d_in], then [d_in, d_out]
  void* ring = ws + round_up((size_t)d_out * d_in * dtype_size(dtype), 256);
  auto scatter_apply = [&](const void* in, void* out, const void* Q, int T, int d, int b,
                           const int32_t* scat, bool transpose_q) {
    if (dtype == POETX_BF16)
      return tc_scatter_apply(in, out, Q, T, d, b, scat, transpose_q, ring, stream);
    return launch_block_apply_simt(in, out, Q, T, d, b, nullptr, scat, transpose_q, dtype, stream);
  };
  // rows of W0m times B_P, columns scattered by perm_in:  M = W0m B_P Pi_P
  POETX_TRY(scatter_apply(W0m, M, Q_P, d_out, d_in, b_in, perm_in, true));
  // M^T [d_in, d_out] into W0_new's storage (W0m is no longer read)
  POETX_TRY(launch_transpose(M, W0_new, d_out, d_in, dtype, stream));
  // rows of M^T times B_R^T, scattered by perm_out:  (Pi_R^T B_R M)^T = M^T B_R^T Pi_R
  POETX_TRY(scatter_apply(W0_new, M, Q_R, d_in, d_out, b_out, perm_out, false));
  // back to [d_out, d_in]
  return launch_transpose(M, W0_new, d_in, d_out, dtype, stream);
}

size_t poetx_workspace_bytes(int T, int d_in, int d_out, int b_in, int b_out, poetx_dtype dtype) {
  if (!valid_dtype(dtype) || !sizes_ok(T, d_in, d_out, b_in, b_out)) return 0;
  const Workspace w = layout(T, d_in, d_out, b_in, b_out, dtype);
  return w.fwd_bytes > w.bwd_bytes ? w.fwd_bytes : w.bwd_bytes;
}

}  // extern "C"

namespace poetx {
size_t forward_workspace_bytes(int T, int d_in, int d_out, int b_in, int b_out, poetx_dtype dtype) {
  if (!valid_dtype(dtype) || !sizes_ok(T, d_in, d_out, b_in, b_out)) return 0;
  return layout(T, d_in, d_out, b_in, b_out, dtype).fwd_bytes;
}
}  // namespace poetx

extern "C" {

// Forward chain into caller buffers; `u` and `z` may live in the workspace.
static poetx_status forward_chain(const void* x, const void* W0m, const void* Q_P,
                                  const void* Q_R, const int32_t* perm_in, const int32_t* inv_in,
                                  const int32_t* perm_out, const int32_t* inv_out, int T, int d_in,
                                  int d_out, int b_in, int b_out, poetx_dtype dt, void* u, void* z,
                                  void* y, void* tc_ws, cudaStream_t s) {
  if (tc_linear_supported(d_in, d_out, b_in, b_out, dt))
    return tc_forward(x, W0m, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out, T, d_in, d_out, b_in,
                      b_out, u, z, y, tc_ws, s);
  // u = gather(x, perm_in) . B_P^T
  POETX_TRY(launch_block_apply_simt(x, u, Q_P, T, d_in, b_in, perm_in, nullptr, false, dt, s));
  // z = u . W0m^T
  POETX_TRY(launch_gemm_simt(u, W0m, z, T, d_out, d_in, true, dt, s));
  // y = scatter(z . B_R^T, perm_out)
  if (y) POETX_TRY(launch_block_apply_simt(z, y, Q_R, T, d_out, b_out, nullptr, perm_out, false, dt, s));
  return POETX_OK;
}

poetx_status poetx_forward(const void* x, const void* W0m, const void* Q_P, const void* Q_R,
                           const int32_t* perm_in, const int32_t* inv_in,
                           const int32_t* perm_out, const int32_t* inv_out, int T, int d_in,
                           int d_out, int b_in, int b_out, poetx_dtype act_dtype, void* y,
                           void* z_save, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  POETX_TRY(check_linear_args(T, d_in, d_out, b_in, b_out, act_dtype,
                              {W0m, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out}));
  if (T == 0) return POETX_OK;
  POETX_TRY(check_linear_args(T, d_in, d_out, b_in, b_out, act_dtype, {x, y, workspace}));
  if (z_save && !aligned16(z_save)) return POETX_ERR_INVALID_ARG;
  const Workspace w = layout(T, d_in, d_out, b_in, b_out, act_dtype);
  if (ws_bytes < w.fwd_bytes) return POETX_ERR_SHAPE;
  char* ws = static_cast<char*>(workspace);
  void* u = ws + w.f_u;
  void* tc_ws = ws + w.f_tc;
  void* z = z_save ? z_save : ws + w.f_z;
  return forward_chain(x, W0m, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out, T, d_in, d_out, b_in,
                       b_out, act_dtype, u, z, y, tc_ws, stream);
}

poetx_status poetx_backward(const void* x, const void* dy, const void* W0m, const float* theta_P,
                            const float* theta_R, int n, const void* Q_P, const void* Q_R,
                            const void* z_saved, const int32_t* perm_in, const int32_t* inv_in,
                            const int32_t* perm_out, const int32_t* inv_out, int T, int d_in,
                            int d_out, int b_in, int b_out, poetx_dtype act_dtype, void* dX,
                            float* dtheta_P, float* dtheta_R, void* workspace, size_t ws_bytes,
                            cudaStream_t stream) {
  if (n < 1) return POETX_ERR_INVALID_ARG;
  POETX_TRY(check_linear_args(T, d_in, d_out, b_in, b_out, act_dtype,
                              {W0m, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out, theta_P,
                               theta_R, dtheta_P, dtheta_R}));
  const int nb_in = d_in / b_in, nb_out = d_out / b_out;
  if (T == 0) {
    // no tokens: every gradient is zero
    if (cudaMemsetAsync(dtheta_P, 0, sizeof(float) * nb_in * (size_t)(b_in * (b_in - 1) / 2),
                        stream) != cudaSuccess ||
        cudaMemsetAsync(dtheta_R, 0, sizeof(float) * nb_out * (size_t)(b_out * (b_out - 1) / 2),
                        stream) != cudaSuccess)
      return POETX_ERR_CUDA;
    return POETX_OK;
  }
  POETX_TRY(check_linear_args(T, d_in, d_out, b_in, b_out, act_dtype, {x, dy, dX, workspace}));
  if (z_saved && !aligned16(z_saved)) return POETX_ERR_INVALID_ARG;
  const Workspace w = layout(T, d_in, d_out, b_in, b_out, act_dtype);
  if (ws_bytes < w.bwd_bytes) return POETX_ERR_SHAPE;
  char* ws = static_cast<char*>(workspace);
  void* gz = ws + w.gz;
  void* gu = ws + w.gu;
  float* dqp = reinterpret_cast<float*>(ws + w.dqp);
  float* dqr = reinterpret_cast<float*>(ws + w.dqr);
  void* tc_ws = ws + w.tc;
  const void* z = z_saved;
  if (!z) {
    // POET-Xmem [§2.E]: recompute z (u lives in the g_u region until g_u is made)
    void* zr = ws + w.z;
    POETX_TRY(forward_chain(x, W0m, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out, T, d_in, d_out,
                            b_in, b_out, act_dtype, gu, zr, nullptr, tc_ws, stream));
    z = zr;
  }
  const poetx_dtype dt = act_dtype;
  // [§2.D] backward of the Cayley-Neumann blocks: on the bf16 tensor-core path
  // it runs inside tc_backward (bf16 operands; the R side overlapping the g_u
  // GEMM); the fp32 layer uses the exact CUDA-core kernel per side
  const bool tc_cnp = tc_cnp_backward(d_in, d_out, b_in, b_out, dt);
  if (tc_linear_supported(d_in, d_out, b_in, b_out, dt)) {
    TcCnpBwd cnp{theta_P, theta_R, n, dtheta_P, dtheta_R,
                     static_cast<char*>(tc_ws) + tc_cnp_ws_offset(T, d_in, d_out, b_in, b_out)};
    POETX_TRY(tc_backward(x, dy, W0m, Q_P, Q_R, z, perm_in, inv_in, perm_out, inv_out, T, d_in,
                          d_out, b_in, b_out, dX, gz, gu, dqp, w.slots_p, dqr, w.slots_r, tc_ws,
                          tc_cnp ? &cnp : nullptr, stream));
    if (tc_cnp) return POETX_OK;
  } else {
    // g_z = gather(dy, perm_out) . B_R
    POETX_TRY(launch_block_apply_simt(dy, gz, Q_R, T, d_out, b_out, perm_out, nullptr, true, dt, stream));
    // dQ_R,j = sum_t gather(dy)_j^T z_j
    POETX_TRY(launch_dq_simt(dy, z, T, d_out, b_out, perm_out, nullptr, dqr, dt, stream));
    // g_u = g_z . W0m
    POETX_TRY(launch_gemm_simt(gz, W0m, gu, T, d_in, d_out, false, dt, stream));
    // dX = scatter(g_u . B_P, perm_in)
    POETX_TRY(launch_block_apply_simt(gu, dX, Q_P, T, d_in, b_in, nullptr, perm_in, true, dt, stream));
    // dQ_P,j = sum_t g_u,j^T gather(x)_j
    POETX_TRY(launch_dq_simt(gu, x, T, d_in, b_in, nullptr, perm_in, dqp, dt, stream));
  }
  if (tc_cnp) {
    POETX_TRY(tc::cnp_bwd_layer(theta_P, dqp, w.slots_p, nb_in, b_in, theta_R, dqr, w.slots_r,
                                nb_out, b_out, n, dtheta_P, dtheta_R,
                                static_cast<char*>(tc_ws) +
                                    tc_cnp_ws_offset(T, d_in, d_out, b_in, b_out),
                                stream));
  } else {
    POETX_TRY(launch_sum_slots(dqp, w.slots_p, (size_t)d_in * b_in, stream));
    POETX_TRY(launch_sum_slots(dqr, w.slots_r, (size_t)d_out * b_out, stream));
    POETX_TRY(launch_cnp_bwd_simt(theta_P, dqp, nb_in, b_in, n, dtheta_P, stream));
    POETX_TRY(launch_cnp_bwd_simt(theta_R, dqr, nb_out, b_out, n, dtheta_R, stream));
  }
  return POETX_OK;
}

// ---- POET-XQ [§2.E]: INT8 frozen weight, dequantised per call -----------------

poetx_status poetx_quantize_w0(const void* W0, int d_out, int d_in, poetx_dtype dtype,
                               int8_t* W0q, float* scale, cudaStream_t stream) {
  if (!valid_dtype(dtype)) return POETX_ERR_INVALID_ARG;
  if (d_out <= 0 || d_in <= 0 || d_in % 4) return POETX_ERR_SHAPE;
  if (!W0 || !W0q || !scale || !aligned16(W0) || !aligned16(W0q) || !aligned16(scale))
    return POETX_ERR_INVALID_ARG;
  return launch_quantize_w0(W0, d_out, d_in, dtype, W0q, scale, stream);
}

poetx_status poetx_dequantize_w0(const int8_t* W0q, const float* scale, int d_out, int d_in,
                                 poetx_dtype dtype, void* W0, cudaStream_t stream) {
  if (!valid_dtype(dtype)) return POETX_ERR_INVALID_ARG;
  if (d_out <= 0 || d_in <= 0 || d_in % 4) return POETX_ERR_SHAPE;
  if (!W0 || !W0q || !scale || !aligned16(W0) || !aligned16(W0q) || !aligned16(scale))
    return POETX_ERR_INVALID_ARG;
  return launch_dequantize_w0(W0q, scale, d_out, d_in, dtype, W0, stream);
}

// The dequantised weight's region, at the head of the XQ workspace.
static size_t xq_weight_bytes(int d_in, int d_out, poetx_dtype dtype) {
  return round_up((size_t)d_out * d_in * dtype_size(dtype), 256);
}

size_t poetx_workspace_bytes_xq(int T, int d_in, int d_out, int b_in, int b_out,
                                poetx_dtype dtype) {
  const size_t rest = poetx_workspace_bytes(T, d_in, d_out, b_in, b_out, dtype);
  if (rest == 0 || d_in % 4) return 0;
  return xq_weight_bytes(d_in, d_out, dtype) + rest;
}

poetx_status poetx_forward_xq(const void* x, const int8_t* W0q, const float* scale,
                              const void* Q_P, const void* Q_R, const int32_t* perm_in,
                              const int32_t* inv_in, const int32_t* perm_out,
                              const int32_t* inv_out, int T, int d_in, int d_out, int b_in,
                              int b_out, poetx_dtype act_dtype, void* y, void* z_save,
                              void* workspace, size_t ws_bytes, cudaStream_t stream) {
  POETX_TRY(check_linear_args(T, d_in, d_out, b_in, b_out, act_dtype, {W0q, scale, workspace}));
  if (d_in % 4) return POETX_ERR_SHAPE;
  if (ws_bytes < poetx_workspace_bytes_xq(T, d_in, d_out, b_in, b_out, act_dtype))
    return POETX_ERR_SHAPE;
  const size_t head = xq_weight_bytes(d_in, d_out, act_dtype);
  void* W0m = workspace;
  POETX_TRY(launch_dequantize_w0(W0q, scale, d_out, d_in, act_dtype, W0m, stream));
  return poetx_forward(x, W0m, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out, T, d_in, d_out, b_in,
                       b_out, act_dtype, y, z_save, static_cast<char*>(workspace) + head,
                       ws_bytes - head, stream);
}

poetx_status poetx_backward_xq(const void* x, const void* dy, const int8_t* W0q,
                               const float* scale, const float* theta_P, const float* theta_R,
                               int n, const void* Q_P, const void* Q_R, const void* z_saved,
                               const int32_t* perm_in, const int32_t* inv_in,
                               const int32_t* perm_out, const int32_t* inv_out, int T, int d_in,
                               int d_out, int b_in, int b_out, poetx_dtype act_dtype, void* dX,
                               float* dtheta_P, float* dtheta_R, void* workspace,
                               size_t ws_bytes, cudaStream_t stream) {
  POETX_TRY(check_linear_args(T, d_in, d_out, b_in, b_out, act_dtype, {W0q, scale, workspace}));
  if (d_in % 4) return POETX_ERR_SHAPE;
  if (ws_bytes < poetx_workspace_bytes_xq(T, d_in, d_out, b_in, b_out, act_dtype))
    return POETX_ERR_SHAPE;
  const size_t head = xq_weight_bytes(d_in, d_out, act_dtype);
  void* W0m = workspace;
  POETX_TRY(launch_dequantize_w0(W0q, scale, d_out, d_in, act_dtype, W0m, stream));
  return poetx_backward(x, dy, W0m, theta_P, theta_R, n, Q_P, Q_R, z_saved, perm_in, inv_in,
                        perm_out, inv_out, T, d_in, d_out, b_in, b_out, act_dtype, dX, dtheta_P,
                        dtheta_R, static_cast<char*>(workspace) + head, ws_bytes - head, stream);
}

poetx_status poetx_stream_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return POETX_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return POETX_ERR_CUDA;
  int err = 0;
  if (cudaMemcpyFromSymbol(&err, g_poetx_error, sizeof(int)) != cudaSuccess) return POETX_ERR_CUDA;
  if (err) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_poetx_error, &zero, sizeof(int));
    return (poetx_status)err;
  }
  return POETX_OK;
}

}  // extern "C"
