// timeline.cpp -- device start and end times of every kernel a process runs,
// from CUPTI's activity API (concurrent-kernel records).  Built as its own
// small library (libsstimeline.so, linked against libcupti) for the
// benchmark: it times the kernels of a captured CUDA graph as they run in the
// replayed schedule, dependent launches and overlaps included, instead of
// bracketing each launch with events (which would serialise them).  Records
// hold GPU timestamps in nanoseconds; tracing costs about one percent of a
// replayed speculative round.
#include <cupti.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

namespace {

struct Rec {
  uint64_t start, end;
  uint32_t stream;
  std::string name;
};

std::mutex g_mu;
std::vector<Rec> g_recs;
bool g_registered = false;
constexpr size_t kBufBytes = 16u << 20;

void CUPTIAPI on_buffer_requested(uint8_t** buf, size_t* size, size_t* max_records) {
  *buf = static_cast<uint8_t*>(aligned_alloc(8, kBufBytes));
  *size = *buf != nullptr ? kBufBytes : 0;
  *max_records = 0;
}

void CUPTIAPI on_buffer_completed(CUcontext, uint32_t, uint8_t* buf, size_t, size_t valid) {
  CUpti_Activity* r = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    while (cuptiActivityGetNextRecord(buf, valid, &r) == CUPTI_SUCCESS) {
      if (r->kind != CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL && r->kind != CUPTI_ACTIVITY_KIND_KERNEL)
        continue;
      const auto* k = reinterpret_cast<const CUpti_ActivityKernel10*>(r);
      g_recs.push_back({k->start, k->end, k->streamId, k->name != nullptr ? k->name : ""});
    }
  }
  free(buf);
}

}  // namespace

extern "C" {

// Starts recording kernel activity (0 on success).
int sstl_start(void) {
  if (!g_registered) {
    if (cuptiActivityRegisterCallbacks(on_buffer_requested, on_buffer_completed) != CUPTI_SUCCESS)
      return 1;
    g_registered = true;
  }
  return cuptiActivityEnable(CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL) == CUPTI_SUCCESS ? 0 : 2;
}

// Stops recording and delivers every pending record (0 on success).
int sstl_stop(void) {
  const bool flushed = cuptiActivityFlushAll(1) == CUPTI_SUCCESS;
  const bool off = cuptiActivityDisable(CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL) == CUPTI_SUCCESS;
  return flushed && off ? 0 : 3;
}

int sstl_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return static_cast<int>(g_recs.size());
}

// Record i: start and end (ns, device clock), stream id, mangled kernel name.
int sstl_get(int i, uint64_t* start, uint64_t* end, uint32_t* stream, char* name, int cap) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (i < 0 || i >= static_cast<int>(g_recs.size()) || cap < 1) return 1;
  *start = g_recs[i].start;
  *end = g_recs[i].end;
  *stream = g_recs[i].stream;
  std::strncpy(name, g_recs[i].name.c_str(), static_cast<size_t>(cap) - 1);
  name[cap - 1] = '\0';
  return 0;
}

void sstl_clear(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_recs.clear();
}

}  // extern "C"
