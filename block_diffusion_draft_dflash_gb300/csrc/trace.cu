// Launch tracing (see trace.h and dflash_trace_enable in include/dflash.h).
#include <string.h>

#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/dflash.h"
#include "trace.h"

namespace df {
namespace {
struct Rec {
  std::string tag;
  cudaEvent_t a, b;
};
std::mutex mu;
bool enabled = false;
std::vector<Rec> recs;
std::vector<cudaEvent_t> pool;
std::vector<std::string> open_tags;

cudaEvent_t get_event() {
  if (!pool.empty()) {
    cudaEvent_t e = pool.back();
    pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

bool trace_on() { return enabled; }

void trace_begin(const char* tag, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
  std::lock_guard<std::mutex> g(mu);
  Rec r{tag, get_event(), get_event()};
  cudaEventRecord(r.a, st);
  recs.push_back(r);
}

void trace_end(cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
  std::lock_guard<std::mutex> g(mu);
  if (!recs.empty()) cudaEventRecord(recs.back().b, st);
}
}  // namespace df

extern "C" int dflash_trace_enable(int on) {
  std::lock_guard<std::mutex> g(df::mu);
  df::enabled = on != 0;
  return DF_OK;
}

extern "C" int dflash_trace_read(int max_entries, char* names, double* total_ms, int* count) {
  std::lock_guard<std::mutex> g(df::mu);
  std::map<std::string, std::pair<double, int>> agg;
  for (auto& r : df::recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return DF_ERR_CUDA;
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    auto& e = agg[r.tag];
    e.first += ms;
    e.second += 1;
    df::pool.push_back(r.a);
    df::pool.push_back(r.b);
  }
  df::recs.clear();
  int n = 0;
  for (auto& kv : agg) {
    if (n >= max_entries) break;
    if (names) {
      strncpy(names + 64 * n, kv.first.c_str(), 63);
      names[64 * n + 63] = 0;
    }
    if (total_ms) total_ms[n] = kv.second.first;
    if (count) count[n] = kv.second.second;
    ++n;
  }
  return n;
}
