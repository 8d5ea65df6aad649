// Kernel trace for benchmarks: CUDA event pairs around every library launch,
// recorded on the launch's stream, with the kernel class and algorithmic work.
#include <mutex>
#include <vector>

#include "dash_internal.h"
#include "dashroot.h"

namespace dash {
namespace {

struct Record {
  cudaEvent_t begin = nullptr, end = nullptr;
  int kind = 0;
  double flops = 0.0, bytes = 0.0;
};

std::mutex g_mu;
std::vector<Record> g_rec;
int g_used = 0;
bool g_active = false;

}  // namespace

int trace_begin(cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_active || g_used >= static_cast<int>(g_rec.size())) return -1;
  const int i = g_used++;
  cudaEventRecord(g_rec[i].begin, st);
  return i;
}

void trace_end(int rec, cudaStream_t st, int kind, double flops, double bytes) {
  if (rec < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (rec >= static_cast<int>(g_rec.size())) return;
  cudaEventRecord(g_rec[rec].end, st);
  g_rec[rec].kind = kind;
  g_rec[rec].flops = flops;
  g_rec[rec].bytes = bytes;
}

}  // namespace dash

using namespace dash;

extern "C" {

dash_status dash_trace_start(int capacity) {
  if (capacity < 0 || capacity > (1 << 22)) return DASH_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  while (static_cast<int>(g_rec.size()) < capacity) {
    Record r;
    if (cudaEventCreate(&r.begin) != cudaSuccess) return DASH_ERR_CUDA;
    if (cudaEventCreate(&r.end) != cudaSuccess) return DASH_ERR_CUDA;
    g_rec.push_back(r);
  }
  g_used = 0;
  g_active = true;
  return DASH_OK;
}

int dash_trace_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_used;
}

dash_status dash_trace_read(int i, int* kind, double* flops, double* bytes, float* ms) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (i < 0 || i >= g_used) return DASH_ERR_INVALID_ARG;
  Record& r = g_rec[i];
  if (cudaEventSynchronize(r.end) != cudaSuccess) return DASH_ERR_CUDA;
  float t = 0.0f;
  if (cudaEventElapsedTime(&t, r.begin, r.end) != cudaSuccess) return DASH_ERR_CUDA;
  if (kind) *kind = r.kind;
  if (flops) *flops = r.flops;
  if (bytes) *bytes = r.bytes;
  if (ms) *ms = t;
  return DASH_OK;
}

dash_status dash_trace_stop(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_active = false;
  return DASH_OK;
}

}  // extern "C"
