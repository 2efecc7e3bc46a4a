// Per-kernel CUDA-event timing of the library's launches (see msa_profile.h).
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "msa_internal.cuh"
#include "msa_profile.h"

namespace msa {
namespace {

struct Record {
  const char* name;
  cudaEvent_t start, stop;
};

std::mutex g_mu;
bool g_on = false;
std::atomic<int> g_inject_timeout{0};
std::vector<Record> g_records;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

bool debug_inject_timeout() { return g_inject_timeout.load() != 0; }

ProfScope::ProfScope(const char* name, cudaStream_t stream) : name_(name), stream_(stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on) return;
  start_ = take_event();
  if (start_ && cudaEventRecord(start_, stream_) != cudaSuccess) {
    g_pool.push_back(start_);
    start_ = nullptr;
  }
}

ProfScope::~ProfScope() {
  if (!start_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t stop = take_event();
  if (!stop || cudaEventRecord(stop, stream_) != cudaSuccess) {
    g_pool.push_back(start_);
    if (stop) g_pool.push_back(stop);
    return;
  }
  g_records.push_back({name_, start_, stop});
}

}  // namespace msa

extern "C" int msa_profile_begin(void) {
  std::lock_guard<std::mutex> lk(msa::g_mu);
  for (auto& r : msa::g_records) {
    msa::g_pool.push_back(r.start);
    msa::g_pool.push_back(r.stop);
  }
  msa::g_records.clear();
  msa::g_on = true;
  return 0;
}

extern "C" int msa_profile_end(msa_kernel_time_t* out, int max_entries) {
  std::lock_guard<std::mutex> lk(msa::g_mu);
  msa::g_on = false;
  std::vector<msa_kernel_time_t> agg;
  int rc = 0;
  for (auto& r : msa::g_records) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      rc = -1;
    size_t k = 0;
    while (k < agg.size() && std::strcmp(agg[k].name, r.name) != 0) ++k;
    if (k == agg.size()) agg.push_back({r.name, 0, 0.0});
    agg[k].launches += 1;
    agg[k].total_ms += ms;
    msa::g_pool.push_back(r.start);
    msa::g_pool.push_back(r.stop);
  }
  msa::g_records.clear();
  if (rc != 0) return -1;
  for (size_t k = 0; k < agg.size() && int(k) < max_entries; ++k) out[k] = agg[k];
  return int(agg.size());
}

extern "C" int msa_debug_inject_timeout(int enable) { return msa::g_inject_timeout.exchange(enable ? 1 : 0); }
