// profile.cu -- optional kernel timing and launch counting for libslimspec.
//
// When enabled (ss_profile_start), every kernel launch of the library is
// bracketed by two CUDA events recorded on the launching stream; the
// benchmark reads per-kernel launch counts and summed durations back with
// ss_profile_read.  Events recorded while a stream is captured become graph
// nodes; each replay re-records them, so reading with `keep` after every
// replay accumulates per-replay kernel times.  A launch counter runs whether
// or not timing is enabled.
// Disabled, the cost is one relaxed atomic increment per launch.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "../../include/slimspec.h"
#include "ss_internal.h"

namespace ss {

static const char* const kKindNames[kKindCount] = {
    "k_down_proj",   "k_head_stream", "k_head_finish", "k_verify_rows", "k_verify_decide",
    "k_verify_resid", "k_verify_finish", "k_topk",      "k_gather_logits", "k_cand_finish",
    "k_head_mma",    "k_verify_first", "k_verify_qrow", "k_down_reduce"};

namespace {
struct Rec {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_mu;
std::atomic<bool> g_on{false};
std::atomic<long long> g_launches{0};
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
// While `st` is being captured, the record must become an event-record node
// of the graph (cudaEventRecordExternal) so that each replay re-records it.
void record(cudaEvent_t e, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
  else
    cudaEventRecord(e, st);
}
}  // namespace

cudaError_t set_smem_once(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  // every kernel of the head asks for the same (largest) shared-memory split,
  // so that the next kernel's CTAs can join an SM without reconfiguring it
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

int resident_blocks(const void* kernel, int threads, size_t smem) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> seen;
  static std::vector<std::pair<std::pair<const void*, int>, int>> values;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& kv : values)
    if (kv.first.first == kernel && kv.first.second == dev) return kv.second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1)
    n = 1;
  values.push_back({{kernel, dev}, n});
  return n;
}

ProfScope::ProfScope(int kind, cudaStream_t st) : slot(-1), stream(st) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  Rec r{kind, take_event(), take_event()};
  if (!r.a || !r.b) return;
  record(r.a, st);
  g_recs.push_back(r);
  slot = (int)g_recs.size() - 1;
}

ProfScope::~ProfScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (slot < (int)g_recs.size()) record(g_recs[slot].b, stream);
}

}  // namespace ss

using namespace ss;

extern "C" {

int ss_profile_start(void) {
  g_on.store(true);
  return SS_OK;
}

int ss_profile_stop(void) {
  g_on.store(false);
  return SS_OK;
}

long long ss_launch_count(void) { return g_launches.load(); }

int ss_profile_read(int* launches, double* total_ms, int n_kinds, int keep) {
  if (!launches || !total_ms || n_kinds < 1) return SS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int k = 0; k < n_kinds; ++k) { launches[k] = 0; total_ms[k] = 0.0; }
  int status = SS_OK;
  for (const Rec& r : g_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) { status = SS_ERR_CUDA; continue; }
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) { status = SS_ERR_CUDA; continue; }
    if (r.kind < n_kinds) { launches[r.kind] += 1; total_ms[r.kind] += ms; }
  }
  if (!keep) {
    for (const Rec& r : g_recs) { g_pool.push_back(r.a); g_pool.push_back(r.b); }
    g_recs.clear();
  }
  return status;
}

const char* ss_profile_kind_name(int kind) {
  return (kind >= 0 && kind < kKindCount) ? kKindNames[kind] : "unknown";
}

}  // extern "C"
