// Launch profiler: counts every kernel launch of the library and, when
// enabled, brackets each with CUDA events on the launching stream together
// with the launch's algorithmic work (FLOPs and HBM bytes), so a caller can
// measure per-kernel time and roofline fractions inside a timed region.
#include <string.h>

#include <mutex>
#include <vector>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

struct Rec {
  const char* name;
  int ev;  // index of the start event; stop is ev + 1
  double flops;
  double bytes;
};

constexpr int MAX_EVENTS = 1 << 16;

struct Profiler {
  std::mutex mu;
  bool on = false;
  uint64_t launches = 0;
  std::vector<cudaEvent_t> events;
  std::vector<Rec> recs;
  int next = 0;
  int device = -1;
};

Profiler& prof() {
  static Profiler p;
  return p;
}

}  // namespace

ProfScope::ProfScope(const char* name, cudaStream_t st, double flops, double bytes) : st_(st), ev_(-1) {
  Profiler& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  ++p.launches;
  if (!p.on || p.next + 2 > MAX_EVENTS) return;
  while (static_cast<int>(p.events.size()) < p.next + 2) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return;
    p.events.push_back(e);
  }
  ev_ = p.next;
  p.next += 2;
  p.recs.push_back({name, ev_, flops, bytes});
  cudaEventRecord(p.events[ev_], st_);
}

ProfScope::~ProfScope() {
  if (ev_ < 0) return;
  Profiler& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  cudaEventRecord(p.events[ev_ + 1], st_);
}

bool profiling_on() {
  Profiler& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  return p.on;
}

}  // namespace kl

using namespace kl;

extern "C" {

kl_status kl_profile_enable(int32_t on) {
  Profiler& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  p.on = on != 0;
  p.recs.clear();
  p.next = 0;
  return KL_OK;
}

uint64_t kl_launch_count(void) {
  Profiler& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  return p.launches;
}

int32_t kl_profile_read(kl_prof_entry* out, int32_t max_entries) {
  Profiler& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  if (p.next > 0 && cudaEventSynchronize(p.events[p.next - 1]) != cudaSuccess) {
    set_error(KL_ERR_CUDA, "profile: event synchronise failed");
    return -1;
  }
  int n = 0;
  for (const Rec& r : p.recs) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.events[r.ev], p.events[r.ev + 1]) != cudaSuccess) continue;
    int i = 0;
    while (i < n && strncmp(out[i].name, r.name, sizeof(out[i].name)) != 0) ++i;
    if (i == n) {
      if (n >= max_entries) continue;
      memset(&out[n], 0, sizeof(out[n]));
      strncpy(out[n].name, r.name, sizeof(out[n].name) - 1);
      ++n;
    }
    out[i].launches += 1;
    out[i].ms += ms;
    out[i].flops += r.flops;
    out[i].bytes += r.bytes;
  }
  return n;
}

}  // extern "C"
