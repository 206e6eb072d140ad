// tc_linear.cu -- the bf16 transformed linear on the tensor-core path.
//
// [POET-X §2.A-§2.C] ("POET-X: Memory-efficient LLM Training by Scaling
// Orthogonal Transformation", gist.science summary): the chain
//   u = gather(x, perm_in) . B_P^T,  z = u . W0m^T,  y = scatter(z . B_R^T, perm_out)
// and its backward.  The frozen-weight products run on tcgen05 (tc_gemm.cu),
// so do the permuted block-diagonal applies (tc_blockapply.cu) for b in
// {128, 256}, and so do the dQ token sums (tc_cluster_dq.cu, which gathers
// the permuted operand in flight; tc_permute.cu + tc_dq.cu where the cluster
// form does not fit); other block sizes use the CUDA-core kernels.  Where the
// cluster applies do not fit (a CTA's share of the blocks exceeds its tensor
// memory), a permuted apply is a column permutation through the scratch and
// the unpermuted block apply (tc_plain_apply.cu).
#include <mutex>

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
  // bf16 Q at b in {128, 256}; fp32 Q at b = 256 (three-term split)
  return tc::cnp_supported(b) && (out_dtype == POETX_BF16 || b == 256);
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
// applies.  Backward: one region that serves, in turn, the exchange rings of
// the block applies and of the dQ token sums (or, where the cluster dQ does
// not fit, a gathered activation [T, max(d_in, d_out)]); after it, the dense
// bf16 K and G of every block (CNP backward).
static bool dq_cluster(int T, int d, int b) {
  return tc::cluster_dq_supported(d, b) && tc::cluster_dq_splits(T, d, b) > 0;
}
static bool dq_tc(int T, int d, int b) {
  return dq_cluster(T, d, b) || (tc::dq_supported(d, b) && tc::permute_supported(d));
}

static size_t ring_bytes(int T, int d, int b, bool scatter) {
  return tc::cluster_apply_supported(d, b, scatter) ? tc::cluster_apply_workspace_bytes(T, d, b, scatter)
                                                    : 0;
}

// A permuted apply the cluster form does not take: permutation of the
// columns through a [T, d] bf16 copy in the scratch plus the unpermuted apply.
static bool apply_staged(int d, int b, bool scatter) {
  return !tc::cluster_apply_supported(d, b, scatter) && tc::plain_apply_supported(d, b) &&
         tc::permute_supported(d);
}

// Scratch of one permuted apply: the exchange ring, or the staged copy.
static size_t apply_bytes(int T, int d, int b, bool scatter) {
  if (tc::cluster_apply_supported(d, b, scatter)) return ring_bytes(T, d, b, scatter);
  return apply_staged(d, b, scatter) ? (size_t)T * d * 2 : 0;
}

// Scratch of the block applies (forward, and the backward's g_z and dX).
static size_t apply_region_bytes(int T, int d_in, int d_out, int b_in, int b_out, bool backward) {
  // the backward may also run the forward applies (z recomputed without a saved copy)
  size_t bytes = 0;
  const size_t rings[4] = {apply_bytes(T, d_in, b_in, false), apply_bytes(T, d_out, b_out, true),
                           backward ? apply_bytes(T, d_out, b_out, false) : 0,
                           backward ? apply_bytes(T, d_in, b_in, true) : 0};
  for (size_t r : rings)
    if (r > bytes) bytes = r;
  return round_up(bytes, 256);
}

// The dQ sums' scratch (their exchange ring, or a gathered activation), apart
// from the applies' so that a dQ sum can run beside an apply.
static size_t dq_region_bytes(int T, int d_in, int d_out, int b_in, int b_out) {
  size_t bytes = 0;
  const int ds[2] = {d_in, d_out}, bs[2] = {b_in, b_out};
  for (int i = 0; i < 2; ++i) {
    size_t need = 0;
    if (dq_cluster(T, ds[i], bs[i]))
      need = tc::cluster_dq_workspace_bytes(T, ds[i], bs[i]);
    else if (dq_tc(T, ds[i], bs[i]))
      need = (size_t)T * ds[i] * 2;
    if (need > bytes) bytes = need;
  }
  return round_up(bytes, 256);
}

static size_t shared_region_bytes(int T, int d_in, int d_out, int b_in, int b_out, bool backward) {
  return apply_region_bytes(T, d_in, d_out, b_in, b_out, backward) +
         (backward ? dq_region_bytes(T, d_in, d_out, b_in, b_out) : 0);
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
  if (dt != POETX_BF16 || !dq_tc(T, d, b)) return 1;
  return dq_cluster(T, d, b) ? tc::cluster_dq_splits(T, d, b) : tc::dq_splits(T, d, b);
}

// Offset of the CNP backward's part of the tensor-core scratch.
size_t tc_cnp_ws_offset(int T, int d_in, int d_out, int b_in, int b_out) {
  return shared_region_bytes(T, d_in, d_out, b_in, b_out, true);
}

// Permuted block apply: a thread-block cluster when the shape allows, else a
// column permutation through the scratch (`ws`, apply_bytes of it) and the
// unpermuted apply, else one CTA per token slab on the tensor cores, else the
// CUDA cores.  `inv` is the inverse of the permutation (gath or scat) in use;
// a scatter without it takes the slab form where the cluster form does not fit.
static poetx_status block_apply(const void* in, void* out, const void* Q, int T, int d, int b,
                                const int32_t* gath, const int32_t* inv, const int32_t* scat,
                                bool transpose_q, void* ws, cudaStream_t s, int max_clusters = 0) {
  const bool scatter = scat != nullptr;
  if (tc::cluster_apply_supported(d, b, scatter))
    return tc::cluster_apply_bf16(in, out, Q, scatter ? scat : gath, inv, T, d, b, transpose_q,
                                  scatter, ws, tc::cluster_apply_workspace_bytes(T, d, b, scatter), s,
                                  max_clusters);
  if (apply_staged(d, b, scatter) && ws && (!scatter || inv)) {
    if (!scatter) {   // out = apply(in[:, gath])
      TC_TRY(tc::permute_cols_bf16(in, ws, gath, T, d, s));
      return tc::plain_apply_bf16(ws, out, Q, T, d, b, transpose_q, s);
    }
    // out[:, scat[c]] = apply(in)[:, c], i.e. out = apply(in)[:, inv]
    TC_TRY(tc::plain_apply_bf16(in, ws, Q, T, d, b, transpose_q, s));
    return tc::permute_cols_bf16(ws, out, inv, T, d, s);
  }
  if (tc::blockapply_supported(d, b))
    return tc::blockapply_bf16(in, out, Q, gath ? gath : scat, T, d, b, transpose_q, scatter, s);
  return launch_block_apply_simt(in, out, Q, T, d, b, gath, scat, transpose_q, POETX_BF16, s);
}

// dQ token sums as `slots` partial sums on the tensor cores (the permuted
// operand gathered through the cluster exchange, or gathered once into the
// scratch where that does not fit); one plain sum on the CUDA cores otherwise.
// gG / gV: the gather permutation of G or V (one of them), iG / iV its inverse.
// max_clusters > 0 caps the cluster form's clusters, and with them its slots.
static poetx_status dq(const void* G, const void* V, int T, int d, int b, const int32_t* gG,
                       const int32_t* iG, const int32_t* gV, const int32_t* iV, float* out,
                       int slots, void* ws, size_t ws_bytes, cudaStream_t s, int max_clusters = 0) {
  if (dq_cluster(T, d, b)) {
    if (gG) return tc::cluster_dq_bf16(G, V, iG, T, d, b, true, out, ws, ws_bytes, s, max_clusters);
    return tc::cluster_dq_bf16(V, G, iV, T, d, b, false, out, ws, ws_bytes, s, max_clusters);
  }
  if (dq_tc(T, d, b)) {
    if (gG) {
      TC_TRY(tc::permute_cols_bf16(G, ws, gG, T, d, s));
      return tc::dq_bf16(ws, V, T, d, b, slots, out, s);
    }
    TC_TRY(tc::permute_cols_bf16(V, ws, gV, T, d, s));
    return tc::dq_bf16(G, ws, T, d, b, slots, out, s);
  }
  return launch_dq_simt(G, V, T, d, b, gG, gV, out, POETX_BF16, s);
}

poetx_status tc_forward(const void* x, const void* W0m, const void* Q_P, const void* Q_R,
                        const int32_t* perm_in, const int32_t* inv_in, const int32_t* perm_out,
                        const int32_t* inv_out, int T, int d_in, int d_out, int b_in, int b_out,
                        void* u, void* z, void* y, void* ws, cudaStream_t s) {
  TC_TRY(block_apply(x, u, Q_P, T, d_in, b_in, perm_in, inv_in, nullptr, false, ws, s));
  TC_TRY(tc::gemm_bf16(u, W0m, z, T, d_out, d_in, false, s));
  if (y) TC_TRY(block_apply(z, y, Q_R, T, d_out, b_out, nullptr, inv_out, perm_out, false, ws, s));
  return POETX_OK;
}

size_t tc_scatter_apply_bytes(int T, int d, int b) { return ring_bytes(T, d, b, true); }

poetx_status tc_scatter_apply(const void* in, void* out, const void* Q, int T, int d, int b,
                              const int32_t* scat, bool transpose_q, void* ws, cudaStream_t s) {
  return block_apply(in, out, Q, T, d, b, nullptr, nullptr, scat, transpose_q, ws, s);
}

// A second stream per device for work that overlaps the main chain, with the
// two events of a fork and a join; calls that use it hold the mutex while they
// enqueue, so forks and joins of concurrent callers do not interleave.
namespace {
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxSideDevices = 64;
std::mutex g_side_mu;
SideStream g_side[kMaxSideDevices];

SideStream* side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) {
    cudaGetLastError();
    return nullptr;
  }
  SideStream& ss = g_side[dev];
  if (!ss.stream) {
    if (cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      ss = SideStream{};
      return nullptr;
    }
  }
  return &ss;
}
}  // namespace

poetx_status tc_backward(const void* x, const void* dy, const void* W0m, const void* Q_P,
                         const void* Q_R, const void* z, const int32_t* perm_in,
                         const int32_t* inv_in, const int32_t* perm_out, const int32_t* inv_out,
                         int T, int d_in, int d_out, int b_in, int b_out, void* dX, void* gz,
                         void* gu, float* dqp, int slots_p, float* dqr, int slots_r, void* ws,
                         const TcCnpBwd* cnp, cudaStream_t s) {
  // the applies' exchange rings first, the dQ sums' scratch after them
  const size_t apply_bytes = apply_region_bytes(T, d_in, d_out, b_in, b_out, true);
  const size_t dq_bytes = dq_region_bytes(T, d_in, d_out, b_in, b_out);
  void* ws_dq = static_cast<uint8_t*>(ws) + apply_bytes;
  const int nb_in = d_in / b_in, nb_out = d_out / b_out;
  // the R side's g_z apply and dQ_R sums
  auto r_side = [&](cudaStream_t st) -> poetx_status {
    if (apply_staged(d_out, b_out, false) && !dq_cluster(T, d_out, b_out) && dq_tc(T, d_out, b_out)) {
      // dy gathered once, for both g_z and the dQ_R sums
      TC_TRY(tc::permute_cols_bf16(dy, ws_dq, perm_out, T, d_out, st));
      TC_TRY(tc::plain_apply_bf16(ws_dq, gz, Q_R, T, d_out, b_out, true, st));
      return tc::dq_bf16(ws_dq, z, T, d_out, b_out, slots_r, dqr, st);
    }
    TC_TRY(block_apply(dy, gz, Q_R, T, d_out, b_out, perm_out, inv_out, nullptr, true, ws, st));
    return dq(dy, z, T, d_out, b_out, perm_out, inv_out, nullptr, nullptr, dqr, slots_r, ws_dq,
              dq_bytes, st);
  };
  auto p_dq = [&](cudaStream_t st) -> poetx_status {
    return dq(gu, x, T, d_in, b_in, nullptr, nullptr, perm_in, inv_in, dqp, slots_p, ws_dq, dq_bytes, st);
  };
  auto p_apply = [&](cudaStream_t st) -> poetx_status {
    return block_apply(gu, dX, Q_P, T, d_in, b_in, nullptr, inv_in, perm_in, true, ws, st);
  };
  auto sequential = [&](cudaStream_t st) -> poetx_status {
    TC_TRY(r_side(st));
    TC_TRY(tc::gemm_bf16(gz, W0m, gu, T, d_in, d_out, true, st));
    TC_TRY(p_apply(st));
    return p_dq(st);
  };
  if (!cnp) return sequential(s);
  uint8_t* cnp_ws = static_cast<uint8_t*>(cnp->ws);
  uint8_t* cnp_ws_r = cnp_ws + 10 * (size_t)d_in * b_in;
  const int ctas_r = tc::cnp_bwd_ctas(nb_out, b_out), ctas_p = tc::cnp_bwd_ctas(nb_in, b_in);
  const int sms = device_sm_count();
  // Clusters of the two concurrent pairs (g_z beside dQ_R, dX beside dQ_P):
  // the applies' clusters split between the two kernels of a pair.
  const int cl_r = tc::cluster_apply_clusters(T, d_out, b_out, false);
  const int cl_p = tc::cluster_apply_clusters(T, d_in, b_in, true);
  const bool dq_r = dq_cluster(T, d_out, b_out), dq_p = dq_cluster(T, d_in, b_in);
  std::unique_lock<std::mutex> lk(g_side_mu);
  SideStream* side = side_stream();
  if (!side || 2 * ctas_r > sms || 2 * ctas_p > sms) {
    // no overlap: everything in order on `s`
    lk.unlock();
    TC_TRY(sequential(s));
    TC_TRY(tc::cnp_bwd_side(cnp->theta_R, dqr, slots_r, nb_out, b_out, cnp->n, cnp->dtheta_R,
                            cnp_ws_r, s));
    return tc::cnp_bwd_side(cnp->theta_P, dqp, slots_p, nb_in, b_in, cnp->n, cnp->dtheta_P, cnp_ws, s);
  }
  auto fork = [&]() -> poetx_status {
    if (cudaEventRecord(side->fork, s) != cudaSuccess ||
        cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)
      return check_launch();
    return POETX_OK;
  };
  // Schedule (main = `s`, side = the library stream):
  //   main: g_z apply                | g_u GEMM (leaves the chain's SMs) | dX apply
  //   side: dQ_R, R prep + chain, P's K                                 | dQ_P, P's G + chain
  // A side whose apply and dQ sums both take the cluster form runs them side
  // by side on a split of the exchange clusters; their partial slots are as
  // many as the dQ kernel's clusters.  On the P side the dQ sums take the
  // larger half: the P chain waits for them, not for dX, so finishing them
  // first lets the chain run beside the end of the dX apply (measured at the
  // square 2048 layer: 15 clusters as 7 + 8 gave 0.379 ms per step, 8 + 7
  // 0.384, 6 + 9 0.380).  A side without the cluster form (its blocks need
  // more tensor memory than 8 CTAs hold) runs its apply and dQ sums as whole-
  // GPU kernels on the two streams; when both read dy gathered by perm_out it
  // is gathered once, before the fork.  The R chain runs in its narrow form
  // (two CTAs per block: the GEMM beside it leaves few SMs free, where the
  // cluster form's 8 CTAs per block would need several waves and delay dQ_P);
  // the P chain in the cluster form where the dX apply beside it runs on
  // half the clusters.
  const bool split_r = cl_r >= 2 && dq_r, split_p = cl_p >= 2 && dq_p;
  const int main_r = split_r ? (cl_r + 1) / 2 : 0, side_r = split_r ? cl_r - main_r : 0;
  const int main_p = split_p ? cl_p / 2 : 0, side_p = split_p ? cl_p - main_p : 0;
  auto used = [&](bool cl, int cap, int splits, int slots) {
    if (!cl) return slots;
    return cap > 0 && cap < splits ? cap : splits;
  };
  const int used_r = used(dq_r, side_r, dq_r ? tc::cluster_dq_splits(T, d_out, b_out) : 0, slots_r);
  const int used_p = used(dq_p, side_p, dq_p ? tc::cluster_dq_splits(T, d_in, b_in) : 0, slots_p);
  const bool share_dy = apply_staged(d_out, b_out, false) && !dq_r && dq_tc(T, d_out, b_out);
  poetx_status st = POETX_OK;
  if (share_dy) st = tc::permute_cols_bf16(dy, ws_dq, perm_out, T, d_out, s);   // dy[:, perm_out]
  if (st == POETX_OK) st = fork();
  if (st == POETX_OK)
    st = share_dy ? tc::dq_bf16(ws_dq, z, T, d_out, b_out, slots_r, dqr, side->stream)
                  : dq(dy, z, T, d_out, b_out, perm_out, inv_out, nullptr, nullptr, dqr, slots_r, ws_dq,
                       dq_bytes, side->stream, side_r);
  if (st == POETX_OK)
    st = tc::cnp_bwd_side(cnp->theta_R, dqr, used_r, nb_out, b_out, cnp->n, cnp->dtheta_R, cnp_ws_r,
                          side->stream, 7, true);
  // the P side's dense K and K^T need only theta: made here, beside the GEMM,
  // so that after the dQ_P sums only their sum and the chain remain
  if (st == POETX_OK)
    st = tc::cnp_bwd_side(cnp->theta_P, dqp, used_p, nb_in, b_in, cnp->n, cnp->dtheta_P, cnp_ws,
                          side->stream, 1);
  if (st == POETX_OK)
    st = share_dy ? tc::plain_apply_bf16(ws_dq, gz, Q_R, T, d_out, b_out, true, s)
                  : block_apply(dy, gz, Q_R, T, d_out, b_out, perm_out, inv_out, nullptr, true, ws, s,
                                main_r);
  if (st == POETX_OK) st = tc::gemm_bf16(gz, W0m, gu, T, d_in, d_out, true, s, ctas_r);
  if (st == POETX_OK) st = fork();
  if (st == POETX_OK)
    st = dq(gu, x, T, d_in, b_in, nullptr, nullptr, perm_in, inv_in, dqp, slots_p, ws_dq, dq_bytes,
            side->stream, side_p);
  if (st == POETX_OK)
    st = tc::cnp_bwd_side(cnp->theta_P, dqp, used_p, nb_in, b_in, cnp->n, cnp->dtheta_P, cnp_ws,
                          side->stream, 2 | 4, !split_p);
  if (st == POETX_OK && cudaEventRecord(side->join, side->stream) != cudaSuccess) st = check_launch();
  if (st == POETX_OK)
    st = block_apply(gu, dX, Q_P, T, d_in, b_in, nullptr, inv_in, perm_in, true, ws, s, main_p);
  if (cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess && st == POETX_OK) st = check_launch();
  return st;
}

}  // namespace poetx
