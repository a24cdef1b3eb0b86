// One warp-specialised tensor-core contraction, used by every sum-layer pass:
//
//   D[m, n] = sum_k Aop[g][m][k] * Bop[g][n][k]        (both operands K-major)
//
// followed by a pass-specific epilogue on the float32 accumulator. A CTA owns one
// 128 x BN tile of D for group g = blockIdx.z:
//   warp 0     TMA producer (one thread): 128-byte-swizzled K-slices of A and B into a
//              STAGES-deep shared-memory ring, completion counted in transaction bytes
//   warp 1     MMA issuer (one thread): tcgen05.mma (kind::f16 or kind::tf32, M = 128,
//              N = BN) into a TMEM accumulator; tcgen05.commit frees each ring slot
//   warps 2-9  epilogue: tcgen05.ld of the accumulator, one TMEM lane (row of D) per
//              thread, 32 columns at a time, into the pass's epilogue functor
// Launched as a programmatic dependent of the previous kernel in the stream: everything
// up to the first global access (barrier set-up, TMEM allocation, and with a_early the
// first ring slots' A tiles) overlaps that kernel's tail; griddepcontrol.wait precedes
// every other global access.
// Precision kTF32x3 forms each product from three TF32 MMAs (lo*hi + hi*lo + hi*hi)
// into the same accumulator (pyjuice PR #62, Summary 3, "tf32x3").
//
// Every wait is bounded (pc::mbar_wait); on a timeout the kernel records the reason
// in the device status word, lets the producer drain its in-flight copies, frees its
// TMEM and returns.
#pragma once

#include <type_traits>

#include "pc_device.cuh"

namespace pc {

// Epi::kPrefetchTile (optional, default false): after the K loop the epilogue fetches a
// per-tile input into the idle ring (Epi::prefetch<BN>) and applies from there
// (Epi::apply_prefetched<BN>).
template <class E, class = void>
struct EpiPrefetch : std::false_type {};
template <class E>
struct EpiPrefetch<E, std::void_t<decltype(E::kPrefetchTile)>> : std::bool_constant<E::kPrefetchTile> {};

// Epi::kSliceTF32 (optional, default kSliceK1): the TF32 accumulation slice in k-steps
// (0 = one accumulation over all of K, as the split-K chain tiles need).
template <class E, class = void>
struct EpiSliceTF32 : std::integral_constant<int, 8> {};
template <class E>
struct EpiSliceTF32<E, std::void_t<decltype(E::kSliceTF32)>> : std::integral_constant<int, E::kSliceTF32> {};

// Epi::kBLo (optional, default false; bf16 and TF32 only): the B operand (the layer's
// children) is stored as hi + lo, hi = the mode's rounding of the value and lo = that of
// the remainder, and every k-step adds A * B_lo into a separate TMEM accumulator that
// spans all of K (its entries are 2^-9 / 2^-12 of the main ones, so its truncation is
// negligible); the epilogue adds it to the sliced sum. For children that sit within a
// rounding step of one another (every latent of an HCLT node near its maximum) a single
// rounding would move them all the same way.
template <class E, class = void>
struct EpiBLo : std::false_type {};
template <class E>
struct EpiBLo<E, std::void_t<decltype(E::kBLo)>> : std::bool_constant<E::kBLo> {};

// Epi::kLoadAhead (optional, persistent tiles only): the epilogue's global operand of a
// chunk (a 32 x 32 float block: theta, or node values) goes through a ring of
// Epi::kAheadBufs 4 KB shared-memory buffers per epilogue warp. Epi::issue(p, g, m0, n0,
// q, col0, buf) starts its asynchronous copy (cp.async, no registers held) kAheadBufs - 1
// chunks ahead, across tile boundaries and before the accumulator of that chunk is
// waited for; Epi::apply_buf(p, g, m0, n0, row, col0, v, buf) consumes it. A warp keeps
// up to kAheadBufs - 1 blocks in flight through its stores, TMEM loads and waits: what a
// memory-bound epilogue needs to run near the HBM rate.
template <class E, class = void>
struct EpiLoadAhead : std::false_type {};
template <class E>
struct EpiLoadAhead<E, std::void_t<decltype(E::kLoadAhead)>> : std::bool_constant<E::kLoadAhead> {};

// Warp 0: TMA producer; warp 1: MMA issuer; then the epilogue warps, kEpiWarps / 4 per
// TMEM lane quarter, each taking every (kEpiWarps / 4)-th 32-column chunk of the tile.
// Epi::kEpiWarps (optional) sets the count for one instantiation: 16 for the sliced
// 3xTF32 tiles, whose accumulator slices arrive every k-step (more warps hide the TMEM
// load latency, one chunk per warp leaves registers to keep the next slice's load in
// flight); epilogues that opt in stride their own loops by their count.
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kGemmThreads = 64 + kEpiThreads;
template <class E, class = void>
struct EpiWarps : std::integral_constant<int, kEpiWarps> {};
template <class E>
struct EpiWarps<E, std::void_t<decltype(E::kEpiWarps)>> : std::integral_constant<int, E::kEpiWarps> {};
// (Ten warps place three on some SM sub-partitions, whose 16K registers then allow 168
// per thread; the launch bounds let the compiler plan for that.)
constexpr int kBM = 128;

template <int P, int BN, bool kBLo = false>
struct GemmShape {
  static constexpr int kElem = operand_bytes<P>();
  static constexpr int kBK = 128 / kElem;                 // K elements per 128-byte row
  static constexpr int kAParts = (P == kTF32x3) ? 2 : 1;  // hi (+ lo)
  static constexpr int kBParts = (P == kTF32x3 || kBLo) ? 2 : 1;
  static constexpr uint32_t kABytes = kBM * 128;
  static constexpr uint32_t kBBytes = BN * 128;
  static constexpr uint32_t kStageBytes = kAParts * kABytes + kBParts * kBBytes;
  static constexpr uint32_t kUmmaK = (P == kBF16) ? 16 : (P == kFP8 ? 32 : 8);  // K per MMA instruction
  static constexpr uint32_t kKSteps = kBK / kUmmaK;          // MMAs per ring slot (4)
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN: two epilogue warps split the 32-column chunks");
};

// Accumulation slices, in MMA k-steps (1 or 2, or a multiple of the k-steps of one ring
// slot); see k_umma_gemm. The bf16 mode slices only where the epilogue asks for it
// (Epi::kSliceBF16 k-steps; 0 = one accumulation over all of K). 3xTF32 slices one k-step
// at a time unless the epilogue asks for more (Epi::kSlice3x: 2, or 4 = a ring slot):
// fewer slices (HMM 4096 step 14.6, 10.8, 9.4 ms with 1, 2, 4), but every hi*hi product
// after the slice's first adds a truncation at the partial sum's own magnitude, whose
// expected size depends on the data; the correction for it (kCorrBits) leaves a residual
// bias per contraction of up to ~2.5e-8 of the sum with two k-steps (the HCLT-768 LL, 767
// chained edges, moved by 8e-6, and by 1.9e-5 on uniform emissions): fine for a chain of
// tens of layers, not for hundreds.
constexpr int kSliceK3x = 1;
template <class E, class = void>
struct EpiSlice3x : std::integral_constant<int, kSliceK3x> {};
template <class E>
struct EpiSlice3x<E, std::void_t<decltype(E::kSlice3x)>> : std::integral_constant<int, E::kSlice3x> {};
constexpr int kSliceK1 = 8;  // the TF32 default (EpiSliceTF32)

// The tensor core's float32 accumulator truncates toward zero. A slice of one 3xTF32
// k-step ends in one such truncation at the slice's own magnitude, which drops the bits
// below one ulp of the result: on average half an ulp when the dropped fraction is
// uniform. half_ulp(v) = sign(v) 2^e 2^-24 for v = m 2^e (1 <= m < 2), the exponent and
// sign bits of v scaled by 2^-24 (0 for zero and subnormal v).
__device__ __forceinline__ float half_ulp(float v) {
  return __uint_as_float(__float_as_uint(v) & 0xFF800000u) * 5.9604644775390625e-8f;
}

// Per epilogue warp: a padded 32 x 33 float tile for warp_transpose32.
constexpr int kTBufFloats = 32 * 33;

constexpr size_t kSmemPerCta = 232448;  // opt-in maximum dynamic shared memory per CTA

// Shared-memory plan of one instantiation: the ring gets what the epilogue leaves.
template <int P, int BN, class Epi>
struct GemmPlan {
  using S = GemmShape<P, BN, EpiBLo<Epi>::value && P != kTF32x3>;
  static constexpr size_t kTBufBytes = Epi::kTranspose ? EpiWarps<Epi>::value * kTBufFloats * sizeof(float) : 0;
  static constexpr size_t kEpiBytes = ((Epi::kSmemBytes + 15) / 16) * 16;
  static constexpr size_t kFixed = 1024 /* alignment slack */ + 256 /* barriers */ + kTBufBytes + kEpiBytes;
  static constexpr int kFit = static_cast<int>((kSmemPerCta - kFixed) / S::kStageBytes);
  static constexpr int kStages = kFit < 8 ? kFit : 8;
  static constexpr size_t kBytes = kFixed + size_t(kStages) * S::kStageBytes;
  static_assert(kStages >= 2, "the epilogue leaves room for fewer than two ring slots");
};

template <int P, int BN, class Epi>
constexpr size_t gemm_smem_bytes() {
  return GemmPlan<P, BN, Epi>::kBytes;
}

// The warp holds a 32 x 32 tile one row per lane (v[c] = tile[lane][c]); returns it one
// column per lane (w[r] = tile[r][lane]) through the warp's padded shared buffer, so
// that row-major global data can then be read and written a whole row per instruction.
__device__ __forceinline__ void warp_transpose32(const float (&v)[32], float (&w)[32], float* buf) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < 32; ++c) buf[lane * 33 + c] = v[c];
  __syncwarp();
#pragma unroll
  for (int r = 0; r < 32; ++r) w[r] = buf[r * 33 + lane];
  __syncwarp();
}

template <int N = kEpiThreads>
__device__ __forceinline__ void epilogue_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// Named barrier of the epilogue threads that also ANDs a predicate over them.
template <int N = kEpiThreads>
__device__ __forceinline__ bool epilogue_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(N)
      : "memory");
  return r != 0;
}

// Staged bf16 tiles of 128 rows x 128 values in shared memory (row pitch `pitch` bytes,
// a multiple of 16), moved to and from a row-major global matrix by all epilogue
// threads: two 256-byte row segments per warp instruction instead of one scattered
// 16-byte run per lane. Only rows < nrows and columns < ncols touch global memory; a
// row whose start is not 16-byte aligned goes element by element.
constexpr int kStageTileRows = 128;
constexpr int kStageChunks = 16;  // 16-byte chunks of a 128-value bf16 row
constexpr int kStageIters = kStageTileRows * kStageChunks / kEpiThreads;

__device__ __forceinline__ void stage_tile_store_bf16(const uint8_t* tile, int pitch, __nv_bfloat16* dst,
                                                      long long ld, int nrows, int ncols, int et) {
#pragma unroll 4
  for (int it = 0; it < kStageIters; ++it) {
    const int i = et + it * kEpiThreads;
    const int r = i / kStageChunks, c0 = (i % kStageChunks) * 8;
    if (r >= nrows || c0 >= ncols) continue;
    const uint4 v = *reinterpret_cast<const uint4*>(tile + r * pitch + c0 * 2);
    __nv_bfloat16* g = dst + r * ld + c0;
    if (c0 + 8 <= ncols && (reinterpret_cast<uintptr_t>(g) & 15) == 0) {
      *reinterpret_cast<uint4*>(g) = v;
    } else {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c0 + j < ncols) g[j] = __ushort_as_bfloat16(static_cast<unsigned short>(w[j >> 1] >> (16 * (j & 1))));
    }
  }
}

// The inverse, global rows into the staged tile (zero outside nrows x ncols), issued as
// asynchronous copies (cp.async) so that it overlaps other work; the issuing thread
// completes them with cp_async_wait_all before a barrier that publishes the tile. Rows
// whose start is not 16-byte aligned are loaded element by element on the spot.
__device__ __forceinline__ void cp_async_16(uint8_t* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void stage_tile_load_bf16_async(uint8_t* tile, int pitch, const __nv_bfloat16* src,
                                                           long long ld, int nrows, int ncols, int et) {
#pragma unroll
  for (int it = 0; it < kStageIters; ++it) {
    const int i = et + it * kEpiThreads;
    const int r = i / kStageChunks, c0 = (i % kStageChunks) * 8;
    uint8_t* dst = tile + r * pitch + c0 * 2;
    const int n = (r < nrows && c0 < ncols) ? min(8, ncols - c0) : 0;
    if (n == 0) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const __nv_bfloat16* g = src + r * ld + c0;
    if ((reinterpret_cast<uintptr_t>(g) & 15) == 0) {
      cp_async_16(dst, g, static_cast<uint32_t>(n * 2));  // zero-fills beyond n values
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < n) w[j >> 1] |= static_cast<uint32_t>(__bfloat16_as_ushort(g[j])) << (16 * (j & 1));
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// kSplit: a 2-CTA cluster (consecutive blockIdx.x) computes one 128 x BN tile with
// BN-wide MMAs, each CTA over half of K; after both K loops each CTA sends the partial
// sums of the other half of the columns to its partner through distributed shared memory
// and finishes its own 128 x BN/2 sub-tile. (A 128 x 128 MMA leaves half of the tensor
// core's width idle; at batch 512 there are too few 128 x 256 tiles to fill the GPU
// without splitting K. Where even those are too few, 128 x 128 or 128 x 64 tiles split the
// same way trade MMA width for more CTAs and a smaller exchange.)
template <int P, int BN, class Epi, bool kSplit = false>
__global__ void __launch_bounds__(64 + EpiWarps<Epi>::value * 32, 1)
    k_umma_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA_lo,
                const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB_lo,
                int num_kb_total, unsigned* status, const typename Epi::Params ep, int a_early) {
  // B_lo products in their own accumulator (EpiBLo); 3xTF32 has its own lo terms
  constexpr bool kBLo = EpiBLo<Epi>::value && P != kTF32x3;
  static_assert(!kBLo || P == kBF16 || P == kTF32, "a B lo part in bf16 or TF32");
  using S = GemmShape<P, BN, kBLo>;
  constexpr int kEW = EpiWarps<Epi>::value;  // epilogue warps
  constexpr int kET = kEW * 32;
  constexpr int kWPQ = kEW / 4;              // epilogue warps per TMEM lane quarter
  static_assert(kEW % 4 == 0 && (kEW == kEpiWarps || P == kTF32x3), "more epilogue warps: sliced 3xTF32 only");
  constexpr int kStages = GemmPlan<P, BN, Epi>::kStages;
  // Sliced modes: every K slice (kSliceK k-steps of the MMA) is accumulated from zero in
  // one of kAccBufs TMEM buffers and added into registers by the epilogue with round-to-
  // nearest adds. The tensor-core accumulator truncates on every accumulation, so its
  // bias grows with the number of MMAs summed into one value; slicing bounds that number
  // whatever K is. A slice of one k-step (3xTF32: lo*hi, hi*lo, then hi*hi) ends in a
  // single truncation at the slice's own magnitude, whose expected loss (half_ulp of the
  // slice) the epilogue adds back to each slice.
  constexpr int kSliceK =
      (P == kTF32x3) ? EpiSlice3x<Epi>::value : (P == kTF32 ? EpiSliceTF32<Epi>::value : Epi::kSliceBF16);
  constexpr bool kSliced = kSliceK > 0;
  constexpr bool kStepSliced = kSliced && kSliceK < static_cast<int>(S::kKSteps);
  static_assert(!kSliced || (kStepSliced ? S::kKSteps % kSliceK == 0 && (kSliceK == 1 || P == kTF32x3)
                                           : kSliceK % S::kKSteps == 0),
                "slices are k-steps that divide a ring slot (several: 3xTF32) or whole ring slots");
  // four slice buffers where TMEM holds them (k-step slices; 3xTF32 slot slices), else two
  constexpr int kAccBufs = !kSliced ? 1 : ((kStepSliced || P == kTF32x3) && 4 * BN <= 512 ? 4 : 2);
  static_assert(!kBLo || (kSliced && !kStepSliced), "B lo parts with slot-granular slices");
  constexpr uint32_t kLoCol = kAccBufs * BN;  // the B_lo accumulator's first column
  constexpr uint32_t kTmemUsed = kAccBufs * BN + (kBLo ? BN : 0);
  // tcgen05.alloc takes a power of two
  constexpr uint32_t kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
                                 : kTmemUsed <= 256 ? 256 : 512;
  static_assert(kTmemUsed <= 512, "TMEM columns");
  constexpr bool kHalfUlp = kSliced && P == kTF32x3;
  static_assert(!kHalfUlp || kSliceK <= 4, "the truncation correction is that of slices of up to one ring slot");
  // every fourth slice adds 4 half ulps (one-k-step slices: one truncation at the slice's
  // magnitude), 6 (two k-steps: that one plus one at about half of it) or 12 (a slot of
  // four k-steps, hi*hi after the slot's cross terms: truncations at about a quarter, half,
  // three quarters and all of the slice; 12 measured the least biased on the HMM chains,
  // with a mean LL error of -3e-7 and -6e-7 on the 4096 x 32 and 1024 x 64 workloads,
  // against -1.0e-6 / -2.0e-6 with 10 and -1.7e-6 / -3.3e-6 with 8)
  constexpr uint32_t kCorrBits = kSliceK == 1 ? 0x34800000u : kSliceK == 2 ? 0x34C00000u : 0x35400000u;
  // split K: the idle ring holds the exchange buffer (128 x BN/2 floats), then the
  // epilogue's staged tiles
  constexpr int kXchgBytes = kBM * (BN / 2) * 4;
  if constexpr (kSplit)
    static_assert(!kSliced && (BN == 256 || BN == 128 || BN == 64) &&
                      kStages * S::kStageBytes >= kXchgBytes + Epi::kSplitStageBytes &&
                      Epi::kSplitScratchOffset + kEW * 4096 <= Epi::kSplitStageBytes,
                  "split K: unsliced 128 x 256, 128 x 128 or 128 x 64 tiles, the ring holds the exchange buffer "
                  "and the staged tiles");
  constexpr int kEpiBN = kSplit ? BN / 2 : BN;  // columns this CTA's epilogue finishes
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * S::kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;  // [4]
  uint64_t* acc_empty = acc_full + 4;    // [4]
  uint64_t* mma_done = acc_empty + 4;    // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  float* tbuf_base = reinterpret_cast<float*>(smem + kStages * S::kStageBytes + 256);
  uint8_t* epi_smem = reinterpret_cast<uint8_t*>(tbuf_base) + GemmPlan<P, BN, Epi>::kTBufBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = kSplit ? static_cast<int>(cluster_ctarank()) : 0;
  const unsigned long long wl = first_wait_limit(status);  // the first waits' limit
  const int m0 = (kSplit ? blockIdx.x >> 1 : blockIdx.x) * kBM;
  const int n0 = blockIdx.y * BN;
  const int g = blockIdx.z;
  // this CTA's share of K (in ring blocks) and the first columns of its epilogue
  const int kb_first = kSplit && rank == 1 ? (num_kb_total + 1) / 2 : 0;
  const int num_kb = kSplit ? (rank == 1 ? num_kb_total - kb_first : (num_kb_total + 1) / 2) : num_kb_total;
  const int n0_epi = n0 + rank * kEpiBN;

  auto a_tile = [&](int s, int part) { return smem + s * S::kStageBytes + part * S::kABytes; };
  auto b_tile = [&](int s, int part) {
    return smem + s * S::kStageBytes + S::kAParts * S::kABytes + part * S::kBBytes;
  };

  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int b = 0; b < 4; ++b) {
        mbar_init(&acc_full[b], 1);
        mbar_init(&acc_empty[b], kSliced ? kEW : 1);  // sliced: every epilogue warp releases
      }
      mbar_init(mma_done, 1);
      fence_barrier_init();
      tma_prefetch_map(&tmA);
      tma_prefetch_map(&tmB);
      if constexpr (P == kTF32x3) tma_prefetch_map(&tmA_lo);
      if constexpr (S::kBParts == 2) tma_prefetch_map(&tmB_lo);
    }
    __syncwarp();
    tmem_alloc(tmem_slot, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      // a_early: the A operand was complete before the previous kernel started, so the
      // first (still empty) ring slots' A tiles are fetched before waiting for it.
      const int early = a_early ? (num_kb < kStages ? num_kb : kStages) : 0;
      for (int kb = 0; kb < early; ++kb) {
        const int kx = (kb_first + kb) * S::kBK;
        mbar_arrive_expect_tx(&full[kb], S::kStageBytes);
        tma_load_3d(a_tile(kb, 0), &tmA, &full[kb], kx, m0, g);
        if constexpr (P == kTF32x3) tma_load_3d(a_tile(kb, 1), &tmA_lo, &full[kb], kx, m0, g);
      }
      grid_dependency_wait();
      grid_dependents_launch();
      int issued = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = (kb / kStages) & 1;
        const int kx = (kb_first + kb) * S::kBK;
        if (kb >= early) {
          if (!mbar_wait(&empty[s], ph ^ 1, status, kErrTimeoutProducer, wl)) break;
          mbar_arrive_expect_tx(&full[s], S::kStageBytes);
          tma_load_3d(a_tile(s, 0), &tmA, &full[s], kx, m0, g);
          if constexpr (P == kTF32x3) tma_load_3d(a_tile(s, 1), &tmA_lo, &full[s], kx, m0, g);
        }
        tma_load_3d(b_tile(s, 0), &tmB, &full[s], kx, n0, g);
        if constexpr (S::kBParts == 2) tma_load_3d(b_tile(s, 1), &tmB_lo, &full[s], kx, n0, g);
        issued = kb + 1;
      }
      // Drain: every slot's most recent fill must have landed before the CTA exits.
      for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb) {
        mbar_wait(&full[kb % kStages], (kb / kStages) & 1, status, kErrTimeoutDrain);
      }
    }
    if constexpr (kSplit) {  // the epilogue's two cluster barriers
      __syncwarp();
      cluster_sync();
      cluster_sync();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = umma_idesc(P == kBF16 ? 1u : (P == kFP8 ? 0u : 2u), kBM, BN);
      const int total_q = num_kb * static_cast<int>(S::kKSteps);
      int q = 0;  // k-steps issued so far
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = (kb / kStages) & 1;
        // slot-granular slices: wait for this slice's buffer before the slot
        const int slice = kSliced && !kStepSliced ? q / kSliceK : 0;
        const bool first = kSliced ? (q % (kSliceK > 0 ? kSliceK : 1)) == 0 : kb == 0;
        const bool last = kSliced && !kStepSliced &&
                          ((q + static_cast<int>(S::kKSteps)) % (kSliceK > 0 ? kSliceK : 1) == 0 ||
                           q + static_cast<int>(S::kKSteps) == total_q);
        uint32_t d = tmem;
        if constexpr (kSliced && !kStepSliced) {
          const int buf = slice % kAccBufs;
          if (first && !mbar_wait(&acc_empty[buf], ((slice / kAccBufs) & 1) ^ 1, status, kErrTimeoutMma, wl)) break;
          d = tmem + static_cast<uint32_t>(buf * BN);
        }
        if (!mbar_wait(&full[s], ph, status, kErrTimeoutMma, wl)) break;
        tc_fence_after();
        const uint32_t a0 = smem_addr(a_tile(s, 0));
        const uint32_t b0 = smem_addr(b_tile(s, 0));
        const uint32_t a1 = smem_addr(a_tile(s, P == kTF32x3 ? 1 : 0));
        const uint32_t b1 = smem_addr(b_tile(s, S::kBParts == 2 ? 1 : 0));
        bool timed_out = false;
        if constexpr (kStepSliced) {
          // one slice per kSliceK k-steps, each into the next of kAccBufs buffers; in
          // 3xTF32 the small cross terms of the slice's k-steps first, then hi*hi
#pragma unroll
          for (uint32_t k0 = 0; k0 < S::kKSteps; k0 += kSliceK) {
            const int sl = (q + static_cast<int>(k0)) / kSliceK;
            const int buf = sl % kAccBufs;
            if (!mbar_wait(&acc_empty[buf], ((sl / kAccBufs) & 1) ^ 1, status, kErrTimeoutMma, wl)) {
              timed_out = true;
              break;
            }
            tc_fence_after();
            const uint32_t ds = tmem + static_cast<uint32_t>(buf * BN);
            if constexpr (P == kTF32x3) {
#pragma unroll
              for (uint32_t kk = k0; kk < k0 + kSliceK; ++kk) {
                const uint32_t off = kk * 32;
                umma_tf32(ds, umma_desc_sw128(a1 + off), umma_desc_sw128(b0 + off), idesc, kk == k0 ? 0u : 1u);
                umma_tf32(ds, umma_desc_sw128(a0 + off), umma_desc_sw128(b1 + off), idesc, 1u);
              }
#pragma unroll
              for (uint32_t kk = k0; kk < k0 + kSliceK; ++kk)
                umma_tf32(ds, umma_desc_sw128(a0 + kk * 32), umma_desc_sw128(b0 + kk * 32), idesc, 1u);
            } else {
              umma_tf32(ds, umma_desc_sw128(a0 + k0 * 32), umma_desc_sw128(b0 + k0 * 32), idesc, 0u);
            }
            umma_commit(&acc_full[buf]);
          }
        } else if constexpr (P == kTF32x3) {
          // the small cross terms of the slot first, then hi*hi
#pragma unroll
          for (uint32_t kk = 0; kk < S::kKSteps; ++kk) {
            const uint32_t off = kk * 32;
            umma_tf32(d, umma_desc_sw128(a1 + off), umma_desc_sw128(b0 + off), idesc,
                      (first && kk == 0) ? 0u : 1u);
            umma_tf32(d, umma_desc_sw128(a0 + off), umma_desc_sw128(b1 + off), idesc, 1u);
          }
#pragma unroll
          for (uint32_t kk = 0; kk < S::kKSteps; ++kk) {
            const uint32_t off = kk * 32;
            umma_tf32(d, umma_desc_sw128(a0 + off), umma_desc_sw128(b0 + off), idesc, 1u);
          }
        } else {
#pragma unroll
          for (uint32_t kk = 0; kk < S::kKSteps; ++kk) {
            const uint32_t off = kk * 32;  // 32 bytes of K per MMA
            const uint32_t acc = (first && kk == 0) ? 0u : 1u;
            if constexpr (kBLo) {  // A * B_lo into the lo accumulator, over all of K
              const uint32_t lacc = (kb == 0 && kk == 0) ? 0u : 1u;
              if constexpr (P == kBF16)
                umma_bf16(tmem + kLoCol, umma_desc_sw128(a0 + off), umma_desc_sw128(b1 + off), idesc, lacc);
              else
                umma_tf32(tmem + kLoCol, umma_desc_sw128(a0 + off), umma_desc_sw128(b1 + off), idesc, lacc);
            }
            if constexpr (P == kBF16) {
              umma_bf16(d, umma_desc_sw128(a0 + off), umma_desc_sw128(b0 + off), idesc, acc);
            } else if constexpr (P == kFP8) {
              umma_f8(d, umma_desc_sw128(a0 + off), umma_desc_sw128(b0 + off), idesc, acc);
            } else {
              umma_tf32(d, umma_desc_sw128(a0 + off), umma_desc_sw128(b0 + off), idesc, acc);
            }
          }
        }
        umma_commit(&empty[s]);
        if (timed_out) break;
        if (last) umma_commit(&acc_full[slice % kAccBufs]);
        q += static_cast<int>(S::kKSteps);
      }
      // also on a timeout: the epilogue must not wait forever
      if constexpr (!kSliced) umma_commit(&acc_full[0]);
      // TMEM is freed (and, split, the ring handed to the partner) only once every MMA
      // issued has completed, whether or not a wait gave up
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, status, kErrTimeoutDrain);
    }
    if constexpr (kSplit) {  // the epilogue's two cluster barriers
      __syncwarp();
      cluster_sync();
      cluster_sync();
    }
  } else {
    // ------------------------------------------------------------------- epilogue
    const int et = threadIdx.x - 64;  // 0 .. kET-1
    const int ew = warp - 2;          // epilogue warp 0 .. kEW-1
    grid_dependency_wait();           // the epilogue reads and writes global memory
    Epi::prepare(ep, g, m0, n0_epi, et, epi_smem);
    epilogue_bar_sync<kET>();
    const int q = warp & 3;       // TMEM lane quarter this warp may access
    const int part = ew >> 2;     // the warp takes the chunks c with c % kWPQ == part
    const int row = q * 32 + lane;
    float* tbuf = Epi::kTranspose ? tbuf_base + ew * kTBufFloats : nullptr;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    constexpr int kChunks = kEpiBN / (32 * kWPQ);  // 32-column chunks per epilogue warp (sliced path)
    auto chunk_col = [&](int c) { return (kWPQ * c + part) * 32; };
    bool ok = true;
    if constexpr (kSliced) {
      static_assert(kChunks >= 1 && kEpiBN % (32 * kWPQ) == 0, "whole chunks per epilogue warp");
      float acc[kChunks][32];
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[c][i] = 0.f;
      const int total_q = num_kb * static_cast<int>(S::kKSteps);
      const int num_slices = (total_q + kSliceK - 1) / kSliceK;
      // Each warp takes its slices on its own and releases a slice's buffer to the MMA
      // issuer as soon as its loads have landed (acc_empty counts the epilogue warps), so
      // no block-wide barrier sits between a slice's arrival and its release.
      // The truncation correction (kHalfUlp) is sampled: every fourth slice adds four
      // times its own half ulp. Its expectation is that of adding each slice's half ulp
      // (the slices' magnitudes do not depend on their index modulo 4), its extra noise is
      // of the order of 2^-24 / sqrt(slices) of the sum, and the epilogue's arithmetic per
      // slice drops to about one packed add per two values.
      auto add_slice = [&](float (&a)[32], const uint32_t (&v)[32], bool corr) {
        if (kHalfUlp && corr) {
#pragma unroll
          for (int i = 0; i < 32; i += 2) add2_half_ulp(a[i], a[i + 1], v[i], v[i + 1], kCorrBits);
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 2) add2(a[i], a[i + 1], v[i], v[i + 1]);
        }
      };
      auto wait_slice = [&](int sl) {
        return __all_sync(0xffffffffu, mbar_wait(&acc_full[sl % kAccBufs], (sl / kAccBufs) & 1, status,
                                                  kErrTimeoutEpilogue, wl));
      };
      auto release = [&](int sl) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[sl % kAccBufs]);
      };
      {
        constexpr int kGroup = kChunks < 2 ? kChunks : 2;  // loads in flight at a time
        // (with kEpiWarps = 16 a warp holds one chunk: four warps per SM sub-partition
        // overlap one another's TMEM load latency)
        for (int sl = 0; sl < num_slices; ++sl) {
          const int buf = sl % kAccBufs;
          ok = wait_slice(sl);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < kChunks; c0 += kGroup) {
            uint32_t v[kGroup][32];
#pragma unroll
            for (int c = 0; c < kGroup; ++c)
              tmem_ld_32x32_async(lane_base + static_cast<uint32_t>(buf * BN + chunk_col(c0 + c)), v[c]);
#pragma unroll
            for (int c = 0; c < kGroup; ++c) tmem_wait_ld(v[c]);
            if (c0 + kGroup == kChunks) release(sl);
#pragma unroll
            for (int c = 0; c < kGroup; ++c) add_slice(acc[c0 + c], v[c], (sl & 3) == 0);
          }
        }
      }
      ok = epilogue_bar_and<kET>(ok);  // every epilogue thread takes the same branch below
      if constexpr (kBLo) {
        // the last slice's commit covered every MMA, the B_lo ones included
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            float v[32];
            tmem_ld_32x32(lane_base + static_cast<uint32_t>(kLoCol + chunk_col(c)), v);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[c][i] += v[i];
          }
        }
      }
      if (ok) {
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          Epi::apply(ep, g, m0, n0_epi, row, chunk_col(c), acc[c], epi_smem, tbuf);
        }
      }
    } else {
      ok = epilogue_bar_and<kET>(mbar_wait(&acc_full[0], 0, status, kErrTimeoutEpilogue, wl));
      tc_fence_after();
      if constexpr (kSplit) {
        // the MMAs are complete: this CTA's ring is idle; inputs of the epilogue are
        // staged behind the exchange buffer while the partner finishes
        if (ok) Epi::after_mma(ep, g, m0, n0_epi, et, epi_smem, smem + kXchgBytes);
        // Exchange buffer: 128 rows x BN/2 floats in the (now idle) ring, stored by 32-column
        // chunk, then row, then 16-byte piece (swizzled by the row so that 32 rows' reads of
        // one piece spread over the banks). A warp's 32 x 32 block is contiguous, so each
        // remote store instruction writes 512 consecutive bytes: the block is first turned
        // around in a 4 KB per-warp scratch buffer that the epilogue leaves free until
        // apply_staged (Epi::kSplitScratchOffset).
        auto xoff = [&](int chunk, int r, int piece) {
          return static_cast<uint32_t>(((chunk * 128 + r) * 8 + (piece ^ (r & 7))) * 16);
        };
        uint8_t* scratch = smem + kXchgBytes + Epi::kSplitScratchOffset + ew * 4096;
        cluster_sync();  // both accumulators are final and both rings idle
        if (ok) {
          const uint32_t peer = cluster_map(smem_addr(smem), static_cast<uint32_t>(rank ^ 1));
#pragma unroll 1
          for (int c = part * 32; c < kEpiBN; c += 32 * kWPQ) {
            float v[32];
            tmem_ld_32x32(lane_base + static_cast<uint32_t>((rank ^ 1) * kEpiBN + c), v);
            if (num_kb == 0) {  // a share of no k-blocks: the accumulator was never written
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<float4*>(scratch + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                  make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {  // rows 4i .. 4i+3 of the block, 8 pieces each
              const int r = i * 4 + (lane >> 3), piece = lane & 7;
              const float4 x = *reinterpret_cast<const float4*>(scratch + r * 128 + ((piece ^ (r & 7)) << 4));
              st_cluster_v4(peer + xoff(c >> 5, q * 32 + r, piece), x.x, x.y, x.z, x.w);
            }
            __syncwarp();
          }
        }
        cp_async_wait_all();  // this thread's share of after_mma's staged inputs
        cluster_sync();  // the partner's partial sums of this CTA's columns have landed
        if (ok) {
#pragma unroll 1
          for (int c = part * 32; c < kEpiBN; c += 32 * kWPQ) {
            float v[32];
            tmem_ld_32x32(lane_base + static_cast<uint32_t>(rank * kEpiBN + c), v);
            if (num_kb == 0) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 x = *reinterpret_cast<const float4*>(smem + xoff(c >> 5, row, j));
              v[4 * j] += x.x;
              v[4 * j + 1] += x.y;
              v[4 * j + 2] += x.z;
              v[4 * j + 3] += x.w;
            }
            Epi::apply_staged(ep, g, m0, n0_epi, row, c, v, epi_smem, smem + kXchgBytes);
          }
        }
      } else {
        constexpr bool kPre = EpiPrefetch<Epi>::value;
        if constexpr (kPre) {
          static_assert(kStages * S::kStageBytes >= static_cast<uint32_t>(kBM) * BN * 4, "the ring holds the tile");
          ok = epilogue_bar_and<kET>(ok);  // every epilogue thread takes the same branch
          if (ok) {
            Epi::template prefetch<BN>(ep, g, m0, n0_epi, et, smem);  // the MMAs are done: the ring is idle
            cp_async_wait_all();
          }
          epilogue_bar_sync<kET>();
        }
        if (ok) {
#pragma unroll 1
          for (int c = part * 32; c < BN; c += 32 * kWPQ) {
            float v[32];
            tmem_ld_32x32(lane_base + static_cast<uint32_t>(c), v);
            if constexpr (kPre)
              Epi::template apply_prefetched<BN>(ep, g, m0, n0_epi, row, c, v, smem, tbuf);
            else
              Epi::apply(ep, g, m0, n0_epi, row, c, v, epi_smem, tbuf);
          }
        }
      }
    }
    tc_fence_before();
    ok = epilogue_bar_and<kET>(ok);
    if constexpr (kSplit) {
      if (ok) Epi::store_staged(ep, g, m0, n0_epi, et, smem + kXchgBytes);
    }
    if (ok) Epi::finish(ep, g, m0, n0_epi, et, epi_smem);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------
// Persistent form for many short tiles (the HCLT's per-edge contractions: K = H or B, tens
// of thousands of tiles per step): one CTA per SM takes the tiles t = blockIdx.x,
// blockIdx.x + gridDim.x, ... (t = (g * tiles_m + m) * tiles_n + n, so a CTA's consecutive
// tiles share A's row panel), the producer's ring runs on across tile boundaries, and the
// accumulator alternates between two TMEM buffers, so that one tile's epilogue runs while
// the next tile's K loop does. Unsliced bf16 or TF32, no split, no prefetched tile (the
// ring is never idle); Epi::prepare runs per tile (the epilogue warps own their shared
// memory between tiles). Waits and drains as in k_umma_gemm.
// Split tail (split_from < the tile count; epilogues with apply_add / accumulating load-
// ahead only): the tiles from split_from on are taken as two units each, over the first
// and the second half of K, whose epilogues add their partial products into the output
// with one reduction per element. When the tiles leave a last partial wave of at most
// half the CTAs, halving its tiles halves its length.
template <class E, class = void>
struct EpiHasAdd : std::false_type {};
template <class E>
struct EpiHasAdd<E, std::void_t<decltype(&E::apply_add)>> : std::true_type {};
template <int P, int BN, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_umma_gemm_persist(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA_lo,
                        const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB_lo,
                        int num_kb, int tiles_m, int tiles_n, int groups, int split_from, unsigned* status,
                        const typename Epi::Params ep) {
  static_assert(P == kBF16 || P == kTF32, "persistent tiles: bf16 or TF32");
  static_assert(EpiWarps<Epi>::value == kEpiWarps && !EpiPrefetch<Epi>::value,
                "persistent tiles: default epilogue warps, no prefetched tile");
  // B lo part (EpiBLo): A * B_lo accumulates beside A * B_hi, in the same TMEM buffer's
  // upper BN columns, and the epilogue adds the two
  constexpr bool kBLo = EpiBLo<Epi>::value;
  using S = GemmShape<P, BN, kBLo>;
  constexpr int kStages = GemmPlan<P, BN, Epi>::kStages;
  constexpr int kSliceK = (P == kTF32 ? EpiSliceTF32<Epi>::value : Epi::kSliceBF16);
  static_assert(kSliceK == 0, "persistent tiles accumulate unsliced");
  constexpr uint32_t kAccCols = kBLo ? 2 * BN : BN;  // one accumulator buffer
  static_assert(2 * kAccCols <= 512, "two accumulator buffers in TMEM");
  constexpr uint32_t kTmemCols = 2 * kAccCols <= 256 ? 256 : 512;
  constexpr int kWPQ = kEpiWarps / 4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * S::kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;    // [2]
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  float* tbuf_base = reinterpret_cast<float*>(smem + kStages * S::kStageBytes + 256);
  uint8_t* epi_smem = reinterpret_cast<uint8_t*>(tbuf_base) + GemmPlan<P, BN, Epi>::kTBufBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long wl = first_wait_limit(status);
  const int num_tiles = tiles_m * tiles_n * groups;
  auto tile_coords = [&](int t, int& m0, int& n0, int& g) {
    const int mn = tiles_m * tiles_n;
    g = t / mn;
    const int r = t - g * mn;
    m0 = (r / tiles_n) * kBM;
    n0 = (r % tiles_n) * BN;
  };
  // work units: the tiles before split_from whole, then two K halves of each later tile
  const int num_units = split_from + 2 * (num_tiles - split_from);
  auto unit_info = [&](int u, int& t, int& kb0, int& kb1) {  // returns the tile's K-block range
    if (u < split_from) {
      t = u;
      kb0 = 0;
      kb1 = num_kb;
    } else {
      const int j = u - split_from;
      t = split_from + j / 2;
      kb0 = (j & 1) ? num_kb / 2 : 0;
      kb1 = (j & 1) ? num_kb : num_kb / 2;
    }
    return u >= split_from;  // a partial product: the epilogue adds
  };
  auto a_tile = [&](int s) { return smem + s * S::kStageBytes; };
  auto b_tile = [&](int s, int part) { return smem + s * S::kStageBytes + S::kABytes + part * S::kBBytes; };

  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(&acc_full[b], 1);
        mbar_init(&acc_empty[b], kEpiWarps);
      }
      mbar_init(mma_done, 1);
      fence_barrier_init();
      tma_prefetch_map(&tmA);
      tma_prefetch_map(&tmB);
      if constexpr (kBLo) tma_prefetch_map(&tmB_lo);
    }
    __syncwarp();
    tmem_alloc(tmem_slot, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      grid_dependency_wait();
      grid_dependents_launch();
      int it = 0, issued = 0;  // k-blocks issued over all tiles
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        int t, kb0, kb1, m0, n0, g;
        unit_info(u, t, kb0, kb1);
        tile_coords(t, m0, n0, g);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, status, kErrTimeoutProducer, wl)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], S::kStageBytes);
          tma_load_3d(a_tile(s), &tmA, &full[s], kb * S::kBK, m0, g);
          tma_load_3d(b_tile(s, 0), &tmB, &full[s], kb * S::kBK, n0, g);
          if constexpr (kBLo) tma_load_3d(b_tile(s, 1), &tmB_lo, &full[s], kb * S::kBK, n0, g);
          issued = it + 1;
        }
      }
      for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
        mbar_wait(&full[k % kStages], (k / kStages) & 1, status, kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = umma_idesc(P == kBF16 ? 1u : 2u, kBM, BN);
      int it = 0, local = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x, ++local) {
        int t, kb0, kb1;
        unit_info(u, t, kb0, kb1);
        const int a = local & 1;
        if (!mbar_wait(&acc_empty[a], ((local >> 1) & 1) ^ 1, status, kErrTimeoutMma, wl)) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(a * kAccCols);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&full[s], (it / kStages) & 1, status, kErrTimeoutMma, wl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_addr(a_tile(s)), b0 = smem_addr(b_tile(s, 0)), b1 = smem_addr(b_tile(s, 1));
#pragma unroll
          for (uint32_t kk = 0; kk < S::kKSteps; ++kk) {
            const uint32_t off = kk * 32;
            const uint32_t acc = (kb == kb0 && kk == 0) ? 0u : 1u;
            if constexpr (P == kBF16) {
              umma_bf16(d, umma_desc_sw128(a0 + off), umma_desc_sw128(b0 + off), idesc, acc);
              if constexpr (kBLo) umma_bf16(d + BN, umma_desc_sw128(a0 + off), umma_desc_sw128(b1 + off), idesc, acc);
            } else {
              umma_tf32(d, umma_desc_sw128(a0 + off), umma_desc_sw128(b0 + off), idesc, acc);
              if constexpr (kBLo) umma_tf32(d + BN, umma_desc_sw128(a0 + off), umma_desc_sw128(b1 + off), idesc, acc);
            }
          }
          umma_commit(&empty[s]);
        }
        umma_commit(&acc_full[a]);  // also on a timeout: the epilogue must not wait forever
      }
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, status, kErrTimeoutDrain);
    }
  } else {
    // ------------------------------------------------------------------- epilogue
    const int et = threadIdx.x - 64;
    const int ew = warp - 2;
    const int q = warp & 3, part = ew >> 2;
    const int row = q * 32 + lane;
    float* tbuf = Epi::kTranspose ? tbuf_base + ew * kTBufFloats : nullptr;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    // chunk c of accumulator buffer a (+ its B lo part)
    auto load_acc = [&](int a, int c, float (&v)[32]) {
      tmem_ld_32x32(lane_base + static_cast<uint32_t>(a * kAccCols + c), v);
      if constexpr (kBLo) {
        float lo[32];
        tmem_ld_32x32(lane_base + static_cast<uint32_t>(a * kAccCols + BN + c), lo);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += lo[i];
      }
    };
    grid_dependency_wait();
    bool ok = true;
    int local = 0;
    if constexpr (EpiLoadAhead<Epi>::value) {
      constexpr int kNB = Epi::kAheadBufs;
      constexpr int kCPT = BN / (32 * kWPQ);  // chunks of one tile per warp
      static_assert(kNB >= 2 && Epi::kSmemBytes >= kEpiWarps * kNB * 4096, "a ring of 4 KB blocks per warp");
      float* ring = reinterpret_cast<float*>(epi_smem) + ew * kNB * 1024;
      const int my_units =
          static_cast<int>(blockIdx.x) < num_units ? (num_units - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
      const int items = my_units * kCPT;  // (unit, chunk) items of this warp, in order
      auto item_unit = [&](int i) { return static_cast<int>(blockIdx.x) + (i / kCPT) * static_cast<int>(gridDim.x); };
      auto item_col = [&](int i) { return part * 32 + (i % kCPT) * 32 * kWPQ; };
      auto item_tile = [&](int i, bool& add) {
        int t, kb0, kb1;
        add = unit_info(item_unit(i), t, kb0, kb1);
        return t;
      };
      auto issue = [&](int i) {
        if (i < items) {
          int m0, n0, g;
          bool add;
          tile_coords(item_tile(i, add), m0, n0, g);
          Epi::issue(ep, g, m0, n0, q, item_col(i), ring + (i % kNB) * 1024);
        }
        cp_async_commit();  // (an empty group past the end keeps the counting uniform)
      };
      for (int i = 0; i < kNB - 1; ++i) issue(i);
      for (int i = 0; i < items; ++i) {
        issue(i + kNB - 1);  // into the buffer item i - 1 left
        int m0, n0, g;
        bool add;
        tile_coords(item_tile(i, add), m0, n0, g);
        const int local_i = i / kCPT, a = local_i & 1, c = item_col(i);
        if (i % kCPT == 0) {
          ok = epilogue_bar_and(ok && mbar_wait(&acc_full[a], (local_i >> 1) & 1, status, kErrTimeoutEpilogue, wl));
          if (!ok) break;
          tc_fence_after();
        }
        cp_async_wait_group<kNB - 1>();  // item i's block has landed (this thread's share)
        __syncwarp();                    // ... and every lane's
        float v[32];
        load_acc(a, c, v);
        if (i % kCPT == kCPT - 1) {  // this warp's last chunk of the tile: the buffer is free
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[a]);
        }
        if constexpr (EpiHasAdd<Epi>::value) {
          if (add) {
            typename Epi::Params pa = ep;
            pa.accumulate = 1;  // a K half: added with one reduction per element
            Epi::apply_buf(pa, g, m0, n0, row, c, v, ring + (i % kNB) * 1024);
          } else {
            Epi::apply_buf(ep, g, m0, n0, row, c, v, ring + (i % kNB) * 1024);
          }
        } else {
          Epi::apply_buf(ep, g, m0, n0, row, c, v, ring + (i % kNB) * 1024);
        }
        __syncwarp();  // every lane is done with the block before it is refilled
      }
      cp_async_wait_all();  // no copy may land after the CTA has left
    } else {
      for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++local) {
        int t, kb0, kb1, m0, n0, g;
        const bool add = unit_info(u, t, kb0, kb1);
        tile_coords(t, m0, n0, g);
        Epi::prepare(ep, g, m0, n0, et, epi_smem);
        epilogue_bar_sync();
        const int a = local & 1;
        ok = epilogue_bar_and(ok && mbar_wait(&acc_full[a], (local >> 1) & 1, status, kErrTimeoutEpilogue, wl));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = part * 32; c < BN; c += 32 * kWPQ) {
          float v[32];
          load_acc(a, c, v);
          if (c + 32 * kWPQ >= BN) {  // this warp's last chunk of the tile: the buffer is free
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[a]);
          }
          if constexpr (EpiHasAdd<Epi>::value) {
            if (add)
              Epi::apply_add(ep, g, m0, n0, row, c, v, epi_smem, tbuf);
            else
              Epi::apply(ep, g, m0, n0, row, c, v, epi_smem, tbuf);
          } else {
            Epi::apply(ep, g, m0, n0, row, c, v, epi_smem, tbuf);
          }
        }
        Epi::finish(ep, g, m0, n0, et, epi_smem);
        epilogue_bar_sync();  // prepare of the next tile rewrites the epilogue's shared memory
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Default hooks for epilogues that need no per-CTA set-up or reduction.
struct EpiNoHooks {
  static constexpr int kSmemBytes = 0;
  static constexpr int kSliceBF16 = 0;       // bf16 accumulation slice in k-steps (0 = none)
  static constexpr bool kTranspose = false;  // true: apply() uses warp_transpose32
  template <class Params>
  __device__ static void prepare(const Params&, int, int, int, int, uint8_t*) {}
  template <class Params>
  __device__ static void finish(const Params&, int, int, int, int, uint8_t*) {}
};

}  // namespace pc
