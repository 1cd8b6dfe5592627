// Kernel-time recorder for the bench: the GPU start and end timestamps of
// every kernel launched while recording, from CUPTI's activity API.
//
// "SASS-Level Kernel Generation for Blackwell", section "How we measured",
// times each call as the GPU time of its kernels, from CUPTI, and reports the
// median over the last calls. Events around a launch also count the launch
// latency; these records hold the kernel's own start and end on the GPU.
//
// CONCURRENT_KERNEL records are used, so kernels are not serialised by the
// recording. Measurement tooling only: the GEMM library does not link it.
//
// C ABI (all return 0 on success, else the CUPTI result code, > 0):
//   wkt_start()   register the buffer callbacks (once) and enable recording
//   wkt_stop()    flush every buffer and disable recording
//   wkt_flush()   hand every completed record to the store
//   wkt_count()   records stored
//   wkt_get(i, &start_ns, &end_ns, &stream, name, cap)   record i
//   wkt_clear()   drop the stored records
//   wkt_dropped() records CUPTI dropped (buffers full)
//   wkt_error_string(code)
#include <cupti.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

namespace {

struct Record {
  uint64_t start, end;
  uint32_t stream;
  std::string name;
};

std::mutex g_mu;
std::vector<Record> g_records;
uint64_t g_dropped = 0;
bool g_registered = false;
constexpr size_t kBufferBytes = size_t(8) << 20;

void CUPTIAPI on_request(uint8_t** buffer, size_t* size, size_t* max_records) {
  void* p = nullptr;
  if (posix_memalign(&p, 8, kBufferBytes) != 0) p = nullptr;
  *buffer = static_cast<uint8_t*>(p);
  *size = p ? kBufferBytes : 0;
  *max_records = 0;  // as many as fit
}

void CUPTIAPI on_complete(CUcontext ctx, uint32_t stream_id, uint8_t* buffer, size_t,
                          size_t valid) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    CUpti_Activity* r = nullptr;
    while (valid > 0 && cuptiActivityGetNextRecord(buffer, valid, &r) == CUPTI_SUCCESS) {
      if (r->kind != CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL && r->kind != CUPTI_ACTIVITY_KIND_KERNEL)
        continue;
      const auto* k = reinterpret_cast<const CUpti_ActivityKernel10*>(r);
      g_records.push_back({k->start, k->end, k->streamId, k->name ? k->name : ""});
    }
    size_t dropped = 0;
    if (cuptiActivityGetNumDroppedRecords(ctx, stream_id, &dropped) == CUPTI_SUCCESS)
      g_dropped += dropped;
  }
  std::free(buffer);
}

}  // namespace

extern "C" {

int wkt_start(void) {
  if (!g_registered) {
    const CUptiResult r = cuptiActivityRegisterCallbacks(on_request, on_complete);
    if (r != CUPTI_SUCCESS) return (int)r;
    g_registered = true;
  }
  return (int)cuptiActivityEnable(CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL);
}

int wkt_flush(void) { return (int)cuptiActivityFlushAll(CUPTI_ACTIVITY_FLAG_FLUSH_FORCED); }

int wkt_stop(void) {
  const int f = wkt_flush();
  const int d = (int)cuptiActivityDisable(CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL);
  return f != 0 ? f : d;
}

long long wkt_count(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  return (long long)g_records.size();
}

int wkt_get(long long i, unsigned long long* start_ns, unsigned long long* end_ns,
            unsigned* stream, char* name, int name_cap) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (i < 0 || i >= (long long)g_records.size()) return -1;
  const Record& r = g_records[(size_t)i];
  if (start_ns) *start_ns = r.start;
  if (end_ns) *end_ns = r.end;
  if (stream) *stream = r.stream;
  if (name && name_cap > 0) {
    std::strncpy(name, r.name.c_str(), (size_t)name_cap - 1);
    name[name_cap - 1] = '\0';
  }
  return 0;
}

void wkt_clear(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_records.clear();
}

unsigned long long wkt_dropped(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  return g_dropped;
}

const char* wkt_error_string(int code) {
  const char* s = nullptr;
  if (cuptiGetResultString((CUptiResult)code, &s) != CUPTI_SUCCESS || !s) return "unknown";
  return s;
}

}  // extern "C"
