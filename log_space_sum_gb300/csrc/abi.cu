// Library-wide entry points and host helpers: version, status strings, the
// thread-local error detail, the device status word and TMA tensor-map encoding.
#include <cstring>
#include <atomic>
#include <mutex>

#include "pc_device.cuh"
#include "pc_host.h"

namespace {

thread_local char g_last_error[512] = "";

// Word 0: set by kernels that give up a bounded wait (bits pc::kErrTimeout*). Words 2..3:
// the contraction kernel's first-wait limit in ns (pc::first_wait_limit; 0 = default).
__device__ __align__(16) unsigned g_device_status[4] = {0u, 0u, 0u, 0u};

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;
cudaStream_t g_side[kMaxDevices] = {};
std::mutex g_side_mu;

// Records an event on `from` and makes `to` wait for it (the event is released once it
// has completed).
pc_status_t stream_after(cudaStream_t to, cudaStream_t from) {
  cudaEvent_t ev = nullptr;
  PC_CUDA(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
  const cudaError_t e1 = cudaEventRecord(ev, from);
  const cudaError_t e2 = e1 == cudaSuccess ? cudaStreamWaitEvent(to, ev, 0) : e1;
  cudaEventDestroy(ev);
  if (e2 != cudaSuccess) return pc::set_error(PC_ERR_CUDA, "side stream event: %s", cudaGetErrorString(e2));
  return PC_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

// Event pairs of the contraction profiler: one per launch, or one per group of launches.
struct Profiler {
  std::mutex mu;
  bool active = false;
  bool group_open = false;  // inside profile_group_begin .. _end: launches add no record
  int capacity = 0, count = 0;
  cudaEvent_t* begin = nullptr;
  cudaEvent_t* end = nullptr;
  int* kind = nullptr;
  long long* flops = nullptr;
  int* launches = nullptr;
  void release() {
    for (int i = 0; i < capacity; ++i) {
      if (begin && begin[i]) cudaEventDestroy(begin[i]);
      if (end && end[i]) cudaEventDestroy(end[i]);
    }
    delete[] begin;
    delete[] end;
    delete[] kind;
    delete[] flops;
    delete[] launches;
    begin = end = nullptr;
    kind = nullptr;
    flops = nullptr;
    launches = nullptr;
    capacity = count = 0;
    active = false;
    group_open = false;
  }
} g_prof;

}  // namespace

namespace pc {

int profile_begin(cudaStream_t s) {
  if (!g_prof.active || g_prof.group_open) return -1;
  std::lock_guard<std::mutex> lock(g_prof.mu);
  if (!g_prof.active || g_prof.count >= g_prof.capacity) return -1;
  const int i = g_prof.count++;
  if (cudaEventRecord(g_prof.begin[i], s) != cudaSuccess) return -1;
  return i;
}

void profile_end(int i, cudaStream_t s, int kind, long long flops) {
  if (i < 0) return;
  g_prof.kind[i] = kind;
  g_prof.flops[i] = flops;
  g_prof.launches[i] = 1;
  cudaEventRecord(g_prof.end[i], s);
}

int profile_group_begin(cudaStream_t s) {
  const int i = profile_begin(s);
  if (i >= 0) g_prof.group_open = true;
  return i;
}

void profile_group_end(int i, cudaStream_t s, int kind, long long flops, int launches) {
  if (i < 0) return;
  g_prof.group_open = false;
  profile_end(i, s, kind, flops);
  g_prof.launches[i] = launches;
}

pc_status_t set_error(pc_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_last_error[0] = '\0'; }

std::atomic<unsigned long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

unsigned* device_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

int num_sms() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 148;
  }
  const int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 148;
  }
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

pc_status_t SideStream::fork(cudaStream_t main) {
  int dev = 0;
  PC_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return set_error(PC_ERR_CUDA, "device index %d out of range", dev);
  {
    std::lock_guard<std::mutex> lock(g_side_mu);
    if (!g_side[dev]) PC_CUDA(cudaStreamCreateWithFlags(&g_side[dev], cudaStreamNonBlocking));
    s = g_side[dev];
  }
  return stream_after(s, main);
}

pc_status_t SideStream::join(cudaStream_t main) { return stream_after(main, s); }

pc_status_t encode_operand_map(CUtensorMap* map, const Operand& op, pc_precision_t p,
                               int box_rows, int part, bool swizzle, long long group_stride) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (!g_encode) return set_error(PC_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const int es = operand_elem_bytes(p);
  uint8_t* base = static_cast<uint8_t*>(op.ptr) + (part ? op.lo_elems * size_t(es) : 0);
  const cuuint64_t dims[3] = {cuuint64_t(op.cols), cuuint64_t(op.rows), cuuint64_t(op.groups)};
  const cuuint64_t strides[2] = {cuuint64_t(op.ld) * es,
                                 cuuint64_t(group_stride > 0 ? group_stride : op.ld * op.rows) * es};
  const cuuint32_t box[3] = {cuuint32_t(128 / es), cuuint32_t(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = p == PC_PREC_AUTO  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : p == kPrecFp8Ops ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUresult r = g_encode(map, dt,
                              3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(PC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %lldx%lldx%lld operand",
                     int(r), op.groups, op.rows, op.cols);
  return PC_OK;
}

}  // namespace pc

extern "C" {

const char* pc_version(void) { return "pcsum 0.1 sm_103a"; }

const char* pc_status_string(pc_status_t s) {
  switch (s) {
    case PC_OK: return "PC_OK";
    case PC_ERR_NULL: return "PC_ERR_NULL";
    case PC_ERR_SHAPE: return "PC_ERR_SHAPE";
    case PC_ERR_ALIGNMENT: return "PC_ERR_ALIGNMENT";
    case PC_ERR_UNKNOWN_PRECISION: return "PC_ERR_UNKNOWN_PRECISION";
    case PC_ERR_WORKSPACE: return "PC_ERR_WORKSPACE";
    case PC_ERR_UNSUPPORTED: return "PC_ERR_UNSUPPORTED";
    case PC_ERR_CUDA: return "PC_ERR_CUDA";
    case PC_ERR_TIMEOUT: return "PC_ERR_TIMEOUT";
    case PC_ERR_RANGE: return "PC_ERR_RANGE";
  }
  return "PC_ERR_UNKNOWN_STATUS";
}

const char* pc_last_error(void) { return g_last_error; }

unsigned long long pc_launch_count(void) { return pc::g_launches.load(std::memory_order_relaxed); }

pc_status_t pc_device_status(pc_stream_t stream) {
  pc::clear_error();
  unsigned* word = pc::device_status_word();
  if (!word) return pc::set_error(PC_ERR_CUDA, "device status word unavailable");
  unsigned v = 0;
  PC_CUDA(cudaStreamSynchronize(stream));
  PC_CUDA(cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost));
  if (v) {
    const unsigned zero = 0;
    PC_CUDA(cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice));
    if (v & pc::kErrTimeoutBits)
      return pc::set_error(PC_ERR_TIMEOUT, "a kernel gave up a bounded wait (status bits 0x%x)", v);
    return pc::set_error(PC_ERR_RANGE,
                         "an HMM sample left the range its per-layer scaling keeps exact: its ll is NaN and it "
                         "passed no flow (status bits 0x%x)", v);
  }
  return PC_OK;
}

pc_status_t pc_set_wait_limit_ns(unsigned long long ns) {
  pc::clear_error();
  unsigned* word = pc::device_status_word();
  if (!word) return pc::set_error(PC_ERR_CUDA, "device status word unavailable");
  PC_CUDA(cudaMemcpy(word + 2, &ns, sizeof(ns), cudaMemcpyHostToDevice));
  return PC_OK;
}

pc_status_t pc_profile_start(int capacity) {
  pc::clear_error();
  PC_CHECK(capacity >= 1 && capacity <= (1 << 20), PC_ERR_SHAPE, "capacity must be in [1, 2^20]");
  std::lock_guard<std::mutex> lock(g_prof.mu);
  g_prof.release();
  g_prof.begin = new cudaEvent_t[capacity]();
  g_prof.end = new cudaEvent_t[capacity]();
  g_prof.kind = new int[capacity]();
  g_prof.flops = new long long[capacity]();
  g_prof.launches = new int[capacity]();
  g_prof.capacity = capacity;
  for (int i = 0; i < capacity; ++i) {
    if (cudaEventCreate(&g_prof.begin[i]) != cudaSuccess || cudaEventCreate(&g_prof.end[i]) != cudaSuccess) {
      g_prof.release();
      return pc::set_error(PC_ERR_CUDA, "cudaEventCreate failed");
    }
  }
  g_prof.active = true;
  return PC_OK;
}

pc_status_t pc_profile_stop(int* count, float* ms, int* kind, long long* flops, int* launches, int capacity) {
  pc::clear_error();
  PC_CHECK(count != nullptr, PC_ERR_NULL, "count is NULL");
  std::lock_guard<std::mutex> lock(g_prof.mu);
  g_prof.active = false;
  PC_CUDA(cudaDeviceSynchronize());
  const int n = g_prof.count < capacity ? g_prof.count : capacity;
  for (int i = 0; i < n; ++i) {
    float t = 0.f;
    PC_CUDA(cudaEventElapsedTime(&t, g_prof.begin[i], g_prof.end[i]));
    if (ms) ms[i] = t;
    if (kind) kind[i] = g_prof.kind[i];
    if (flops) flops[i] = g_prof.flops[i];
    if (launches) launches[i] = g_prof.launches[i];
  }
  *count = n;
  g_prof.release();
  return PC_OK;
}

}  // extern "C"
