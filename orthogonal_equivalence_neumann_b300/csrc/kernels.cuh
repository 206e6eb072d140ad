// kernels.cuh -- internal launchers behind the C ABI (host-side declarations).
#pragma once

#include "poetx.h"

namespace poetx {

// ---- CUDA-core (fp32 FFMA) kernels: the exact-fp32 path ------------------------
poetx_status launch_cnp_fwd_simt(const float* theta, int nb, int b, int n, void* Q,
                                 poetx_dtype out_dtype, cudaStream_t s);
poetx_status launch_cnp_bwd_simt(const float* theta, const float* dQ, int nb, int b, int n,
                                 float* dtheta, cudaStream_t s);
// part[i] = sum over s < slots of part[s*n + i], added in slot order (dQ partial sums -> dQ).
poetx_status launch_sum_slots(float* part, int slots, size_t n, cudaStream_t s);
size_t cnp_fwd_simt_smem(int b);
size_t cnp_bwd_simt_smem(int b);

poetx_status launch_block_apply_simt(const void* in, void* out, const void* Qs, int T, int d,
                                     int b, const int32_t* gath, const int32_t* scat,
                                     bool transpose_q, poetx_dtype dt, cudaStream_t s);
poetx_status launch_gemm_simt(const void* A, const void* B, void* C, int M, int N, int K,
                              bool b_kmajor, poetx_dtype dt, cudaStream_t s);
poetx_status launch_dq_simt(const void* G, const void* V, int T, int d, int b, const int32_t* gG,
                            const int32_t* gV, float* dQ, poetx_dtype dt, cudaStream_t s);

// Scratch of poetx_forward alone (poetx_workspace_bytes covers the backward too).
size_t forward_workspace_bytes(int T, int d_in, int d_out, int b_in, int b_out, poetx_dtype dtype);

// ---- index maps ------------------------------------------------------------------
poetx_status launch_invert_perm(const int32_t* perm, int32_t* inv, int d, cudaStream_t s);
poetx_status launch_check_perm(const int32_t* perm, const int32_t* inv, int d, int32_t* scratch,
                               int32_t* flag_host, cudaStream_t s);
// out [cols][rows] = in [rows][cols]^T (activation dtype).
poetx_status launch_transpose(const void* in, void* out, int rows, int cols, poetx_dtype dt,
                              cudaStream_t s);
poetx_status launch_merge_w0(const void* W0, void* W0m, int d_out, int d_in, poetx_dtype dt,
                             const int32_t* po, const int32_t* pi, cudaStream_t s);

// ---- POET-XQ: per-row INT8 codes of the frozen weight --------------------------
poetx_status launch_quantize_w0(const void* W, int d_out, int d_in, poetx_dtype dt, int8_t* q,
                                float* scale, cudaStream_t s);
poetx_status launch_dequantize_w0(const int8_t* q, const float* scale, int d_out, int d_in,
                                  poetx_dtype dt, void* W, cudaStream_t s);

}  // namespace poetx
