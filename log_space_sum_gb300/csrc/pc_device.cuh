// Device-side primitives for sm_103a: mbarriers with bounded waits, TMA tile loads,
// tcgen05 (TMEM allocation, UMMA descriptors, MMA issue/commit, TMEM loads) and the
// operand formats of the three precision modes. Inline PTX written from the public
// PTX ISA; no library code.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pc {

// ----------------------------------------------------------------- device status
// Bits of the device status word a kernel sets when it gives up a bounded wait.
enum : unsigned { kErrTimeoutProducer = 1u, kErrTimeoutMma = 2u, kErrTimeoutEpilogue = 4u,
                  kErrTimeoutDrain = 8u, kErrRange = 16u };
constexpr unsigned kErrTimeoutBits = 15u;

// 2 s of wall time: three orders of magnitude above the longest legitimate wait here
// (an epilogue waiting for the full K loop of its tile).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// The status word is the first of four: words 2..3 hold the limit, in ns, of the
// contraction kernel's first waits (the producer's wait for a free ring slot, the MMA
// issuer's waits for a filled slot or a free accumulator, the epilogue's wait for the
// accumulator), set by pc_set_wait_limit_ns; 0 means kWaitLimitNs. Waits for work
// already issued (copies landing, MMAs completing before TMEM is freed) always take
// kWaitLimitNs, so a kernel that gives up early never exits with work in flight.
__device__ __forceinline__ unsigned long long first_wait_limit(const unsigned* status) {
  if (!status) return kWaitLimitNs;
  const unsigned long long v = *reinterpret_cast<const volatile unsigned long long*>(status + 2);
  return v ? v : kWaitLimitNs;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// -------------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Gives up after limit_ns,
// sets `code` in the status word and returns false. (A limit below the default is
// checked on every iteration.)
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* status,
                                          unsigned code, unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  const bool short_limit = limit_ns < kWaitLimitNs;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (((it & 63u) == 0 || short_limit) && globaltimer_ns() - t0 > limit_ns) {
      if (status) atomicOr(status, code);
      return false;
    }
  }
}

// --------------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load (coordinates innermost first) into shared memory; completion is
// reported as transaction bytes on `bar`. x * element size is always a multiple of
// 16 bytes here (x is a multiple of the 128-byte box width).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// --------------------------------------------------- programmatic dependent launch
// Wait until the previous kernel in the stream has completed and its memory is visible
// (a no-op when the launch did not allow overlap).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next kernel in the stream to start its prologue once every CTA of this grid
// has signalled (or exited).
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------- thread-block clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of every CTA of the cluster: arrive (release) and wait (acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of this shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t caddr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(caddr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// ------------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole warp: allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row core groups 1024 bytes apart (stride
// byte offset), leading byte offset unused for this layout, descriptor version 1,
// layout type 2 = SWIZZLE_128B. The tile base is 1024-byte aligned; a K step inside
// the 128-byte row is taken by advancing the start address.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;             // leading byte offset (16 B, unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;     // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;             // descriptor version
  d |= static_cast<uint64_t>(2) << 61;             // SWIZZLE_128B
  return d;
}

// Instruction descriptor for dense kind::f16 / kind::tf32 with an f32 accumulator,
// both operands K-major. fmt: 1 = bf16 (kind::f16), 2 = tf32 (kind::tf32).
__host__ __device__ constexpr uint32_t umma_idesc(uint32_t fmt, uint32_t M, uint32_t N) {
  return (1u << 4)            // D format: f32
         | (fmt << 7)         // A format
         | (fmt << 10)        // B format
         | ((N >> 3) << 17)   // N / 8
         | ((M >> 4) << 24);  // M / 16
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// e4m3 x e4m3 products (instruction descriptor formats 0), K = 32 per instruction.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives TMEM lane
// (lane field of taddr) + t, columns col .. col+31.
__device__ __forceinline__ void tmem_ld_32x32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  // the registers are read only after the wait (see tmem_wait_ld)
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i])::"memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The same load without the wait, so that several loads are in flight; complete them
// with tmem_wait_ld before the registers are read.
__device__ __forceinline__ void tmem_ld_32x32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// The wait, then an empty volatile statement that rewrites the loaded registers, so that
// every later use of them depends on a point after the wait (the load's own statement
// names them as outputs and nothing else would keep their uses behind the wait).
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// Packed float32 pairs (sm_100 family): a += b and a += b + h * k, two lanes per instruction.
__device__ __forceinline__ void add2(float& a0, float& a1, uint32_t b0, uint32_t b1) {
  asm("{\n\t.reg .b64 a, b;\n\t"
      "mov.b64 a, {%0, %1};\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "add.rn.f32x2 a, a, b;\n\t"
      "mov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "r"(b0), "r"(b1));
}
// a += b + (b's exponent and sign bits) * k: b plus half an ulp of b (see half_ulp) for
// k = 2^-24 (bit pattern 0x33800000), or a multiple of it.
__device__ __forceinline__ void add2_half_ulp(float& a0, float& a1, uint32_t b0, uint32_t b1,
                                              uint32_t kbits = 0x33800000u) {
  asm("{\n\t.reg .b64 a, b, h, k;\n\t.reg .b32 h0, h1;\n\t"
      "and.b32 h0, %2, 0xFF800000;\n\t"
      "and.b32 h1, %3, 0xFF800000;\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "mov.b64 h, {h0, h1};\n\t"
      "mov.b64 k, {%4, %4};\n\t"
      "fma.rn.f32x2 b, h, k, b;\n\t"
      "mov.b64 a, {%0, %1};\n\t"
      "add.rn.f32x2 a, a, b;\n\t"
      "mov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "r"(b0), "r"(b1), "r"(kbits));
}

// --------------------------------------------------------------- operand formats
// Precision modes of the contractions (pyjuice PR #62, Summary 1 table).
// kFP8: e4m3 operands (kind::f8f6f4), used internally by the opt-in fp8 flow contractions.
enum Prec : int { kBF16 = 0, kTF32 = 1, kTF32x3 = 2, kFP8 = 3 };

__device__ __forceinline__ float tf32_rna(float v) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
  return __uint_as_float(r);
}

// Operand storage: bf16 for kBF16; float32 holding a TF32 value for kTF32; two
// float32 arrays (hi, then lo at +lo_stride elements) for kTF32x3.
template <int P>
__device__ __forceinline__ void store_operand(void* base, size_t idx, size_t lo_stride, float v) {
  if constexpr (P == kBF16) {
    reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
  } else if constexpr (P == kTF32) {
    reinterpret_cast<float*>(base)[idx] = tf32_rna(v);
  } else {
    const float hi = tf32_rna(v);
    const float lo = tf32_rna(v - hi);
    reinterpret_cast<float*>(base)[idx] = hi;
    reinterpret_cast<float*>(base)[idx + lo_stride] = lo;
  }
}

// A bf16 or TF32 operand stored as hi + lo: hi = the mode's rounding of v, lo = that of
// v - hi (for kTF32x3, the same as store_operand). Read by contractions whose B operand
// has a lo part (EpiBLo).
template <int P>
__device__ __forceinline__ float round_operand(float v) {
  if constexpr (P == kBF16) return __bfloat162float(__float2bfloat16_rn(v));
  else return tf32_rna(v);
}
template <int P>
__device__ __forceinline__ void store_operand_hilo(void* base, size_t idx, size_t lo_stride, float v) {
  if constexpr (P == kBF16) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    reinterpret_cast<__nv_bfloat16*>(base)[idx] = hi;
    reinterpret_cast<__nv_bfloat16*>(base)[idx + lo_stride] = __float2bfloat16_rn(v - __bfloat162float(hi));
  } else {
    const float hi = tf32_rna(v);
    reinterpret_cast<float*>(base)[idx] = hi;
    reinterpret_cast<float*>(base)[idx + lo_stride] = tf32_rna(v - hi);
  }
}

// Operand value as the tensor cores see it (hi + lo for kTF32x3).
template <int P>
__device__ __forceinline__ float load_operand(const void* base, size_t idx, size_t lo_stride) {
  if constexpr (P == kBF16) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  } else if constexpr (P == kTF32) {
    return reinterpret_cast<const float*>(base)[idx];
  } else {
    return reinterpret_cast<const float*>(base)[idx] +
           reinterpret_cast<const float*>(base)[idx + lo_stride];
  }
}

template <int P>
constexpr int operand_bytes() { return P == kBF16 ? 2 : (P == kFP8 ? 1 : 4); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// A thread's run of n <= 32 consecutive operand values starting at element idx:
// 16-byte vector accesses when the run is full and aligned, scalar ones otherwise.
template <int P>
__device__ __forceinline__ void store_operand_run(void* base, size_t idx, size_t lo,
                                                  const float (&v)[32], int n) {
  constexpr int kVec = P == kBF16 ? 8 : 4;
  if (n == 32 && (idx % kVec) == 0) {
    if constexpr (P == kBF16) {
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + idx);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        dst[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                            pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
    } else {
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx);
      float4* dlo = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx + lo);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 h = make_float4(tf32_rna(v[4 * q]), tf32_rna(v[4 * q + 1]), tf32_rna(v[4 * q + 2]),
                                     tf32_rna(v[4 * q + 3]));
        dst[q] = h;
        if constexpr (P == kTF32x3)
          dlo[q] = make_float4(tf32_rna(v[4 * q] - h.x), tf32_rna(v[4 * q + 1] - h.y),
                               tf32_rna(v[4 * q + 2] - h.z), tf32_rna(v[4 * q + 3] - h.w));
      }
    }
  } else {
    // unrolled with a predicate: a runtime index would place v in local memory
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < n) store_operand<P>(base, idx + i, lo, v[i]);
  }
}

template <int P>
__device__ __forceinline__ void load_operand_run(const void* base, size_t idx, size_t lo,
                                                 float (&v)[32], int n) {
  constexpr int kVec = P == kBF16 ? 8 : 4;
  if (n == 32 && (idx % kVec) == 0) {
    if constexpr (P == kBF16) {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + idx);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = src[q];
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          v[8 * q + 2 * r] = __uint_as_float(ww[r] << 16);
          v[8 * q + 2 * r + 1] = __uint_as_float(ww[r] & 0xFFFF0000u);
        }
      }
    } else {
      const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx);
      const float4* slo = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx + lo);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 h = src[q];
        if constexpr (P == kTF32x3) {
          const float4 l = slo[q];
          h.x += l.x;
          h.y += l.y;
          h.z += l.z;
          h.w += l.w;
        }
        v[4 * q] = h.x;
        v[4 * q + 1] = h.y;
        v[4 * q + 2] = h.z;
        v[4 * q + 3] = h.w;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = i < n ? load_operand<P>(base, idx + i, lo) : 0.f;
  }
}

// Non-negative floats order like their bit patterns: atomicMax on the bits.
__device__ __forceinline__ void atomic_max_nonneg(float* addr, float v) {
  atomicMax(reinterpret_cast<unsigned*>(addr), __float_as_uint(v));
}

}  // namespace pc
