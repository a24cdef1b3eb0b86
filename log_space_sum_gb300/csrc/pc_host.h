// Host-side helpers shared by the entry points: error reporting, argument checks,
// workspace carving, TMA tensor-map encoding and GEMM launches.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstddef>
#include <cstdint>
#include <cstdio>

#include "pcsum.h"

namespace pc {

// ------------------------------------------------------------------ errors
pc_status_t set_error(pc_status_t st, const char* fmt, ...);
void clear_error();

// Device status word of the current device (a __device__ variable; its address is
// looked up once per device).
unsigned* device_status_word();

// Streaming multiprocessors of the current device (cached per device; 148 if the device
// cannot be queried). The planners size grids and K-range splits by it.
int num_sms();

// A library-owned stream of the current device for work that runs beside the caller's
// stream within one call: fork() makes it wait for everything issued on `main` so far,
// join() makes `main` wait for everything issued on it since. Both are event waits, so a
// call stays asynchronous and can be captured into a CUDA graph.
struct SideStream {
  cudaStream_t s = nullptr;
  pc_status_t fork(cudaStream_t main);
  pc_status_t join(cudaStream_t main);
};

// Contraction profiler hooks (no-ops unless pc_profile_start is active).
int profile_begin(cudaStream_t s);
void profile_end(int slot, cudaStream_t s, int kind, long long flops);
// One record for a run of `launches` consecutive launches of one kind on stream s (no
// record of their own): events between them would serialise their programmatic overlap.
int profile_group_begin(cudaStream_t s);
void profile_group_end(int slot, cudaStream_t s, int kind, long long flops, int launches);

// One profiler record around the memory-bound launches of a scope (none unless
// pc_profile_start is active): `bytes` = their algorithmic bytes.
struct ProfileScope {
  int slot;
  cudaStream_t s;
  int kind;
  long long bytes;
  ProfileScope(cudaStream_t s_, int kind_, long long bytes_) : slot(profile_begin(s_)), s(s_), kind(kind_), bytes(bytes_) {}
  ~ProfileScope() { profile_end(slot, s, kind, bytes); }
  ProfileScope(const ProfileScope&) = delete;
  ProfileScope& operator=(const ProfileScope&) = delete;
};

#define PC_CHECK(cond, st, ...)                 \
  do {                                          \
    if (!(cond)) return ::pc::set_error(st, __VA_ARGS__); \
  } while (0)

#define PC_CUDA(call)                                                                     \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess)                                                                \
      return ::pc::set_error(PC_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

// Counts every kernel the library launches (pc_launch_count) after checking the launch.
void count_launch();
#define PC_LAUNCH_CHECK()         \
  do {                            \
    PC_CUDA(cudaGetLastError());  \
    ::pc::count_launch();         \
  } while (0)

inline pc_status_t check_precision(pc_precision_t p) {
  if (p != PC_PREC_AUTO && p != PC_PREC_TF32 && p != PC_PREC_FP32)
    return set_error(PC_ERR_UNKNOWN_PRECISION,
                     "unknown precision %d; valid modes are PC_PREC_AUTO (0, bf16 products), "
                     "PC_PREC_TF32 (1) and PC_PREC_FP32 (2, 3xTF32)",
                     static_cast<int>(p));
  return PC_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline long long round_up(long long v, long long m) { return (v + m - 1) / m * m; }

// Bytes of one stored operand element, and the number of stored parts (hi, lo).
// Internal operand format of the opt-in fp8 flow contractions (not a public mode: the
// public calls reject it): e4m3, one byte per element.
constexpr pc_precision_t kPrecFp8Ops = static_cast<pc_precision_t>(3);
inline int operand_elem_bytes(pc_precision_t p) { return p == PC_PREC_AUTO ? 2 : (p == kPrecFp8Ops ? 1 : 4); }
inline int operand_parts(pc_precision_t p) { return p == PC_PREC_FP32 ? 2 : 1; }

// An operand matrix [groups][rows][ld] in a precision's storage format. For 3xTF32
// the lo part follows the hi part at +lo_elems elements.
struct Operand {
  void* ptr = nullptr;
  long long rows = 0, cols = 0, ld = 0, groups = 1;
  size_t lo_elems = 0;
  static size_t bytes(pc_precision_t p, long long groups, long long rows, long long cols, int parts = 0) {
    const long long ld = round_up(cols > 0 ? cols : 1, 64);
    return size_t(groups) * rows * ld * operand_elem_bytes(p) * (parts > 0 ? parts : operand_parts(p));
  }
};

// Bump allocator over the caller's workspace (256-byte granules).
struct Carver {
  uint8_t* base;
  size_t used = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t n) {
    used = static_cast<size_t>(round_up(static_cast<long long>(used), 256));
    void* p = base ? base + used : nullptr;
    used += n;
    return p;
  }
  // parts = 2 gives a bf16 or TF32 operand a lo part (hi + lo, as 3xTF32 always has)
  Operand operand(pc_precision_t p, long long groups, long long rows, long long cols, int parts = 0) {
    Operand o;
    o.groups = groups;
    o.rows = rows;
    o.cols = cols;
    o.ld = round_up(cols > 0 ? cols : 1, 64);
    const int np = parts > 0 ? parts : operand_parts(p);
    const size_t part = size_t(groups) * rows * o.ld;
    o.lo_elems = np == 2 ? part : 0;
    o.ptr = take(Operand::bytes(p, groups, rows, cols, np));
    return o;
  }
};

// 3-D tensor map over an Operand: dims {cols (K), rows, groups}, box {128 bytes of K,
// box_rows, 1}, 128-byte swizzle (or none), zero fill outside the tensor. part 1 = the lo
// half. group_stride: elements between groups (0: rows x ld); a K-split view takes
// groups that are consecutive K ranges of the same rows (op.cols = the range's length,
// group_stride = op.cols).
pc_status_t encode_operand_map(CUtensorMap* map, const Operand& op, pc_precision_t p,
                               int box_rows, int part, bool swizzle = true, long long group_stride = 0);

}  // namespace pc
