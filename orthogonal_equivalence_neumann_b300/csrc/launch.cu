// launch.cu -- launch set-up done once per device and kernel.
//
// The per-call host cost of a launch is kept to the launch itself: device
// properties, kernel attributes and occupancy answers do not change while the
// process runs, so they are looked up once and remembered (small tables under
// a mutex; a library process drives few kernels on few devices).
#include <mutex>
#include <vector>

#include "common.cuh"

namespace poetx {

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;

struct SmemEntry {
  int dev;
  const void* kernel;
  int bytes;
};
std::vector<SmemEntry> g_smem;

struct OccEntry {
  int dev;
  const void* kernel;
  unsigned grid, block, cluster;
  size_t smem;
  int active;
};
std::vector<OccEntry> g_occ;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return dev;
}

}  // namespace

int device_sm_count() {
  static int sms[kMaxDevices] = {0};
  const int dev = current_device();
  if (dev >= 0 && dev < kMaxDevices && sms[dev] > 0) return sms[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 148;
  }
  if (dev >= 0 && dev < kMaxDevices) sms[dev] = n;
  return n;
}

cudaError_t set_max_dynamic_smem(const void* kernel, int bytes) {
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  for (const SmemEntry& e : g_smem)
    if (e.dev == dev && e.kernel == kernel && e.bytes >= bytes) return cudaSuccess;
  const cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (r != cudaSuccess) return r;
  for (SmemEntry& e : g_smem)
    if (e.dev == dev && e.kernel == kernel) {
      e.bytes = bytes;
      return r;
    }
  g_smem.push_back(SmemEntry{dev, kernel, bytes});
  return r;
}

int max_active_clusters(const void* kernel, const cudaLaunchConfig_t& cfg) {
  unsigned cluster = 1;
  for (unsigned i = 0; i < cfg.numAttrs; ++i)
    if (cfg.attrs[i].id == cudaLaunchAttributeClusterDimension) cluster = cfg.attrs[i].val.clusterDim.x;
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  for (const OccEntry& e : g_occ)
    if (e.dev == dev && e.kernel == kernel && e.grid == cfg.gridDim.x && e.block == cfg.blockDim.x &&
        e.cluster == cluster && e.smem == cfg.dynamicSmemBytes)
      return e.active;
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  g_occ.push_back(OccEntry{dev, kernel, cfg.gridDim.x, cfg.blockDim.x, cluster, cfg.dynamicSmemBytes, active});
  return active;
}

}  // namespace poetx
