// profile.cu -- launch accounting and optional per-kernel CUDA-event timing.
//
// Every kernel launch of the library goes through a KernelScope: it counts
// the launch and, while profiling is enabled, brackets the launch with a pair
// of CUDA events recorded on the launch's own stream.  poetx_profile_report()
// waits for those events and returns, per kernel name, the launch count and
// the summed device time.  Off by default; events are recycled, no device
// memory is allocated.  Launches captured into a CUDA graph carry their event
// pair into the graph; a report after a replay gives that replay's times.
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "profile.cuh"

namespace poetx {

namespace {

std::atomic<unsigned long long> g_launches{0};
std::atomic<bool> g_profiling{false};
std::mutex g_mu;

struct Pending {
  std::string name;
  cudaEvent_t begin, end;
};
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free;

cudaEvent_t take_event() {
  if (!g_free.empty()) {
    cudaEvent_t e = g_free.back();
    g_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Records `e` on `s`.  While `s` is being captured into a CUDA graph the
// record becomes a node of the graph (an external event record), so every
// replay re-records the pair around the kernel's node.
void record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

}  // namespace

KernelScope::KernelScope(const char* name, cudaStream_t s) : name_(name), stream_(s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_profiling.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  begin_ = take_event();
  end_ = take_event();
  if (begin_ && end_) record(begin_, stream_);
}

KernelScope::~KernelScope() {
  if (!begin_ || !end_) return;
  record(end_, stream_);
  std::lock_guard<std::mutex> lk(g_mu);
  g_pending.push_back(Pending{name_, begin_, end_});
}

}  // namespace poetx

using namespace poetx;

extern "C" {

unsigned long long poetx_launch_count(void) { return g_launches.load(); }

poetx_status poetx_profile_enable(int enable) {
  g_profiling.store(enable != 0);
  return POETX_OK;
}

int poetx_profile_report(char* buf, size_t len) {
  std::map<std::string, std::pair<long, double>> agg;
  std::vector<Pending> pend;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    pend.swap(g_pending);
  }
  int bad = 0;
  for (auto& p : pend) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.end) != cudaSuccess || cudaEventElapsedTime(&ms, p.begin, p.end) != cudaSuccess) {
      bad = 1;
      cudaGetLastError();
    }
    auto& a = agg[p.name];
    a.first += 1;
    a.second += ms;
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& p : pend) {
      g_free.push_back(p.begin);
      g_free.push_back(p.end);
    }
  }
  std::string out;
  char line[256];
  for (auto& kv : agg) {
    snprintf(line, sizeof line, "%s %ld %.6f\n", kv.first.c_str(), kv.second.first, kv.second.second);
    out += line;
  }
  if (buf && len) {
    strncpy(buf, out.c_str(), len - 1);
    buf[len - 1] = 0;
  }
  return bad ? -1 : (int)out.size();
}

}  // extern "C"
