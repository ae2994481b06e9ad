// Per-launch timing of the tensor-core GEMM launches (fkl_trace_* in include/fkl.h).
//
// While a trace is active on a thread, fkl_forward / fkl_backward record a CUDA event pair on
// the caller's stream around every GEMM launch they make.  The events belong to the library
// and are created when the trace starts; no device memory is allocated.
#include <mutex>
#include <vector>

#include "../../include/fkl.h"
#include "fkl_internal.h"

namespace fkl {

namespace {
struct TraceState {
  std::vector<cudaEvent_t> begin, end;
  std::vector<int32_t> kind;
  std::vector<double> flops;
  int32_t capacity = 0;
  int32_t count = 0;
  bool active = false;

  void release() {
    for (cudaEvent_t e : begin) cudaEventDestroy(e);
    for (cudaEvent_t e : end) cudaEventDestroy(e);
    begin.clear();
    end.clear();
    kind.clear();
    flops.clear();
    capacity = count = 0;
    active = false;
  }
  ~TraceState() { release(); }
};
thread_local TraceState g_trace;
}  // namespace

void trace_launch_begin(cudaStream_t st) {
  TraceState& t = g_trace;
  if (!t.active || t.count >= t.capacity) return;
  cudaEventRecord(t.begin[t.count], st);
}

void trace_launch_end(cudaStream_t st, int kind, double flops) {
  TraceState& t = g_trace;
  if (!t.active || t.count >= t.capacity) return;
  cudaEventRecord(t.end[t.count], st);
  t.kind[t.count] = kind;
  t.flops[t.count] = flops;
  ++t.count;
}

}  // namespace fkl

using namespace fkl;

extern "C" {

fkl_status fkl_trace_start(int32_t capacity) {
  set_last_error_message("");
  if (capacity < 1 || capacity > 65536) {
    set_last_error_message("trace capacity must be in [1, 65536]");
    return FKL_ERR_INVALID_ARG;
  }
  TraceState& t = g_trace;
  t.release();
  t.begin.resize(capacity);
  t.end.resize(capacity);
  t.kind.assign(capacity, -1);
  t.flops.assign(capacity, 0.0);
  for (int32_t i = 0; i < capacity; ++i) {
    if (cudaEventCreate(&t.begin[i]) != cudaSuccess || cudaEventCreate(&t.end[i]) != cudaSuccess) {
      t.begin.resize(i);
      t.end.resize(i);
      t.release();
      set_last_error_message("cudaEventCreate failed");
      return FKL_ERR_CUDA;
    }
  }
  t.capacity = capacity;
  t.count = 0;
  t.active = true;
  return FKL_OK;
}

fkl_status fkl_trace_stop(void) {
  g_trace.active = false;
  return FKL_OK;
}

int32_t fkl_trace_read(float* ms, int32_t* kind, double* flops, int32_t capacity) {
  TraceState& t = g_trace;
  const int32_t n = t.count < capacity ? t.count : capacity;
  for (int32_t i = 0; i < n; ++i) {
    float v = 0.f;
    if (cudaEventSynchronize(t.end[i]) != cudaSuccess ||
        cudaEventElapsedTime(&v, t.begin[i], t.end[i]) != cudaSuccess) {
      set_last_error_message("reading trace events failed");
      return -1;
    }
    if (ms) ms[i] = v;
    if (kind) kind[i] = t.kind[i];
    if (flops) flops[i] = t.flops[i];
  }
  return n;
}

}  // extern "C"
