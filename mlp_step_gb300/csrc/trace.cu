// Launch counter and per-kernel CUDA-event timing (see trace.cuh).
#include <atomic>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "trace.cuh"

namespace mlp {

namespace {

std::atomic<unsigned long long> g_launches{0};
std::atomic<bool> g_timing{false};
std::mutex g_mu;

struct Record {
  std::string name;
  cudaEvent_t start = nullptr, stop = nullptr;
};
std::vector<Record> g_records;
size_t g_used = 0;

bool capturing(cudaStream_t st) {
  cudaStreamCaptureStatus s = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &s) != cudaSuccess) return true;
  return s != cudaStreamCaptureStatusNone;
}

}  // namespace

LaunchScope::LaunchScope(const char* what, cudaStream_t st, long long a, long long b, long long c)
    : st_(st), slot_(-1) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_timing.load(std::memory_order_relaxed) || capturing(st)) return;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_used == g_records.size()) {
    Record r;
    if (cudaEventCreate(&r.start) != cudaSuccess || cudaEventCreate(&r.stop) != cudaSuccess)
      return;
    g_records.push_back(r);
  }
  char buf[160];
  if (a || b || c) snprintf(buf, sizeof buf, "%s[%lld,%lld,%lld]", what, a, b, c);
  else snprintf(buf, sizeof buf, "%s", what);
  Record& r = g_records[g_used];
  r.name = buf;
  if (cudaEventRecord(r.start, st) != cudaSuccess) return;
  slot_ = (int)g_used++;
}

LaunchScope::~LaunchScope() {
  if (slot_ < 0) return;
  std::lock_guard<std::mutex> lock(g_mu);
  cudaEventRecord(g_records[slot_].stop, st_);
}

}  // namespace mlp

extern "C" {

unsigned long long mlp_launch_count(void) {
  return mlp::g_launches.load(std::memory_order_relaxed);
}

mlp_status mlp_timing_enable(int on) {
  std::lock_guard<std::mutex> lock(mlp::g_mu);
  if (on) mlp::g_used = 0;
  mlp::g_timing.store(on != 0);
  return MLP_OK;
}

size_t mlp_timing_report(char* buf, size_t cap) {
  std::lock_guard<std::mutex> lock(mlp::g_mu);
  std::map<std::string, std::pair<long long, double>> agg;
  for (size_t i = 0; i < mlp::g_used; ++i) {
    auto& r = mlp::g_records[i];
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess) continue;
    if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) continue;
    auto& e = agg[r.name];
    e.first += 1;
    e.second += ms;
  }
  std::string out = "{";
  bool first = true;
  for (auto& kv : agg) {
    char tmp[256];
    snprintf(tmp, sizeof tmp, "%s\"%s\": [%lld, %.6f]", first ? "" : ", ", kv.first.c_str(),
             kv.second.first, kv.second.second);
    out += tmp;
    first = false;
  }
  out += "}";
  if (buf && cap > 0) {
    size_t n = out.size() < cap - 1 ? out.size() : cap - 1;
    memcpy(buf, out.data(), n);
    buf[n] = 0;
  }
  return out.size() + 1;
}

}  // extern "C"
