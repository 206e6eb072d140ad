// noalloc.cu -- poetx_forward_noalloc: the forward with its scratch memory in a
// fixed device array owned by the library, for callers that cannot allocate.
//
// Some callers of this library cannot call cudaMalloc: a host framework that
// owns all device memory through its own pool and hands out only the tensors
// it manages, or a latency-critical loop in which allocation (which may
// synchronise the device) is forbidden after start-up.  Such callers still
// own x, the weights, y and z_save; only the forward's scratch (the
// workspace of poetx_forward) comes from the array below instead of from
// the caller.
//
// The array is a file-scope static __device__ object: every device that
// loads the library holds POETX_NOALLOC_WORKSPACE_BYTES of it until the
// process exits.  Host code cannot use the array's name as a device address
// (on the host it names a shadow object), so the device address is looked up
// with cudaGetSymbolAddress, once per device, with that device current, and
// cached.  All calls on a device share the one array: calls that overlap on
// the GPU (different streams, no ordering between them) race on it.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_workspace[POETX_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the array on the current device (set-up on first use).
poetx_status noalloc_workspace(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return POETX_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return POETX_ERR_CUDA;
    }
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return POETX_OK;
}

}  // namespace

extern "C" poetx_status poetx_forward_noalloc(const void* x, const void* W0m, const void* Q_P,
                                              const void* Q_R, const int32_t* perm_in,
                                              const int32_t* inv_in, const int32_t* perm_out,
                                              const int32_t* inv_out, int T, int d_in, int d_out,
                                              int b_in, int b_out, poetx_dtype act_dtype, void* y,
                                              void* z_save, cudaStream_t stream) {
  const size_t need = poetx::forward_workspace_bytes(T, d_in, d_out, b_in, b_out, act_dtype);
  if (need == 0)  // invalid sizes or dtype: let the forward name the error
    return poetx_forward(x, W0m, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out, T, d_in, d_out,
                         b_in, b_out, act_dtype, y, z_save, nullptr, 0, stream);
  if (need > POETX_NOALLOC_WORKSPACE_BYTES) return POETX_ERR_SHAPE;
  void* ws = nullptr;
  const poetx_status st = noalloc_workspace(&ws);
  if (st != POETX_OK) return st;
  // The forward writes every byte of scratch it reads, so the array's
  // previous contents (the last call's) need no clearing.
  return poetx_forward(x, W0m, Q_P, Q_R, perm_in, inv_in, perm_out, inv_out, T, d_in, d_out, b_in,
                       b_out, act_dtype, y, z_save, ws, POETX_NOALLOC_WORKSPACE_BYTES, stream);
}
