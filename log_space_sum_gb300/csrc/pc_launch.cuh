// Launch helpers: the tensor-core contraction and the small elementwise kernels that
// build its operands.
#pragma once

#include "pc_gemm.cuh"
#include "pc_host.h"

namespace pc {

// a_early: the A operand was written before the previous kernel in the stream started.
// kSplit: grid.x counts CTAs (two per 128-row tile), launched as 2-CTA clusters.
template <int P, int BN, class Epi, bool kSplit = false>
pc_status_t launch_gemm(dim3 grid, const CUtensorMap& a, const CUtensorMap& a_lo,
                        const CUtensorMap& b, const CUtensorMap& b_lo, int num_kb,
                        const typename Epi::Params& ep, cudaStream_t stream, int kind,
                        long long flops, bool a_early = false) {
  constexpr size_t smem = gemm_smem_bytes<P, BN, Epi>();
  static_assert(smem <= 232448, "shared memory per CTA");
  static bool attr_set[64] = {};
  int dev = 0;
  PC_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return set_error(PC_ERR_CUDA, "device index %d out of range", dev);
  if (!attr_set[dev]) {
    PC_CUDA(cudaFuncSetAttribute(k_umma_gemm<P, BN, Epi, kSplit>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
    attr_set[dev] = true;
  }
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return PC_OK;
  const int slot = profile_begin(stream);
  // A programmatic dependent of the previous kernel in the stream (see k_umma_gemm).
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kSplit ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(64 + EpiWarps<Epi>::value * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = kSplit ? 2 : 1;
  PC_CUDA(cudaLaunchKernelEx(&cfg, k_umma_gemm<P, BN, Epi, kSplit>, a, a_lo, b, b_lo, num_kb, device_status_word(),
                             ep, a_early ? 1 : 0));
  PC_LAUNCH_CHECK();
  profile_end(slot, stream, kind, flops);
  return PC_OK;
}

// The persistent contraction over tiles_m x tiles_n x groups tiles (k_umma_gemm_persist):
// one CTA per SM, or fewer when there are fewer tiles.
// split_tail: the last tiles taken as two K halves each (EpiHasAdd epilogues; the caller
// zeroes their output first unless the epilogue accumulates).
template <int P, int BN, class Epi>
pc_status_t launch_gemm_persist(int tiles_m, int tiles_n, int groups, const CUtensorMap& a, const CUtensorMap& a_lo,
                                const CUtensorMap& b, const CUtensorMap& b_lo, int num_kb,
                                const typename Epi::Params& ep, cudaStream_t stream, int kind, long long flops,
                                int split_tail = 0) {
  constexpr size_t smem = gemm_smem_bytes<P, BN, Epi>();
  static_assert(smem <= 232448, "shared memory per CTA");
  static bool attr_set[64] = {};
  int dev = 0;
  PC_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return set_error(PC_ERR_CUDA, "device index %d out of range", dev);
  if (!attr_set[dev]) {
    PC_CUDA(cudaFuncSetAttribute(k_umma_gemm_persist<P, BN, Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)));
    attr_set[dev] = true;
  }
  const long long tiles = static_cast<long long>(tiles_m) * tiles_n * groups;
  if (tiles == 0) return PC_OK;
  if (split_tail < 0 || split_tail > tiles || (split_tail > 0 && (!EpiHasAdd<Epi>::value || num_kb < 2)))
    return set_error(PC_ERR_UNSUPPORTED, "split tail of %d tiles not supported here", split_tail);
  const long long units = tiles + split_tail;
  const int slot = profile_begin(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units < num_sms() ? units : num_sms()));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  PC_CUDA(cudaLaunchKernelEx(&cfg, k_umma_gemm_persist<P, BN, Epi>, a, a_lo, b, b_lo, num_kb, tiles_m, tiles_n,
                             groups, static_cast<int>(tiles - split_tail), device_status_word(), ep));
  PC_LAUNCH_CHECK();
  profile_end(slot, stream, kind, flops);
  return PC_OK;
}

// Tensor maps of an operand's hi and (3xTF32) lo parts.
struct OperandMaps {
  CUtensorMap hi, lo;
};

inline pc_status_t encode_maps(OperandMaps* m, const Operand& op, pc_precision_t p, int box_rows) {
  pc_status_t st = encode_operand_map(&m->hi, op, p, box_rows, 0);
  if (st != PC_OK) return st;
  if (p == PC_PREC_FP32) return encode_operand_map(&m->lo, op, p, box_rows, 1);
  m->lo = m->hi;
  return PC_OK;
}

// Both parts of an operand that has a lo part (Carver::operand with parts = 2).
inline pc_status_t encode_maps_hilo(OperandMaps* m, const Operand& op, pc_precision_t p, int box_rows) {
  if (op.lo_elems == 0) return set_error(PC_ERR_CUDA, "operand has no lo part");
  pc_status_t st = encode_operand_map(&m->hi, op, p, box_rows, 0);
  if (st != PC_OK) return st;
  return encode_operand_map(&m->lo, op, p, box_rows, 1);
}

inline int num_k_blocks(long long K, pc_precision_t p) {
  const int bk = 128 / operand_elem_bytes(p);
  return static_cast<int>((K + bk - 1) / bk);
}

inline unsigned cdiv(long long a, long long b) { return static_cast<unsigned>((a + b - 1) / b); }

// ---------------------------------------------------------------------------------
// Operand builders.

// dst[g][r][c] = op(src[g][r][c]); src row stride src_ld, group stride src_gs.
template <int P>
__global__ void k_rows_to_operand(const float* __restrict__ src, long long src_ld,
                                  long long src_gs, int G, int R, int C, void* dst,
                                  long long dst_ld, size_t lo, const int* gmap) {
  const long long total = static_cast<long long>(G) * R * C;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long c = idx % C;
    const long long gr = idx / C;
    const long long r = gr % R;
    const long long g = gr / R;
    const float v = src[(gmap ? gmap[g] : g) * src_gs + r * src_ld + c];
    store_operand<P>(dst, static_cast<size_t>((g * R + r) * dst_ld + c), lo, v);
  }
}

// Four consecutive columns per thread, blockIdx.x = matrix row (16-byte loads).
template <int P>
__global__ void k_rows_to_operand4(const float* __restrict__ src, long long src_ld, long long src_gs, int R,
                                   int C, void* dst, long long dst_ld, size_t lo, const int* gmap) {
  const long long gr = blockIdx.x;
  const long long g = gr / R, r = gr % R;
  const int c = 4 * (blockIdx.y * blockDim.x + threadIdx.x);
  if (c >= C) return;
  const float4 v = *reinterpret_cast<const float4*>(src + (gmap ? gmap[g] : g) * src_gs + r * src_ld + c);
  const size_t idx = static_cast<size_t>(gr * dst_ld + c);
  if constexpr (P == kBF16) {
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(dst) + idx) =
        make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  } else {
    const float4 h = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(dst) + idx) = h;
    if constexpr (P == kTF32x3)
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(dst) + idx + lo) =
          make_float4(tf32_rna(v.x - h.x), tf32_rna(v.y - h.y), tf32_rna(v.z - h.z), tf32_rna(v.w - h.w));
  }
}

template <int P>
pc_status_t rows_to_operand(const float* src, long long src_ld, long long src_gs, int G, int R,
                            int C, const Operand& dst, cudaStream_t s, const int* gmap = nullptr) {
  const long long total = static_cast<long long>(G) * R * C;
  if (total == 0) return PC_OK;
  const bool vec = (C % 4 == 0) && (src_ld % 4 == 0) && (src_gs % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(src) & 15) == 0 && static_cast<long long>(G) * R < (1ll << 31) &&
                   (C / 4 + 255) / 256 < 65536;
  if (vec) {
    const dim3 grid(static_cast<unsigned>(static_cast<long long>(G) * R), cdiv(C / 4, 256));
    k_rows_to_operand4<P><<<grid, 256, 0, s>>>(src, src_ld, src_gs, R, C, dst.ptr, dst.ld, dst.lo_elems, gmap);
  } else {
    const unsigned blocks = static_cast<unsigned>((total + 255) / 256 < 16ll * num_sms() ? (total + 255) / 256 : 16ll * num_sms());
    k_rows_to_operand<P><<<blocks, 256, 0, s>>>(src, src_ld, src_gs, G, R, C, dst.ptr, dst.ld, dst.lo_elems, gmap);
  }
  PC_LAUNCH_CHECK();
  return PC_OK;
}

// ---------------------------------------------------------------- transposes
// dst(g, c, r) = src(g, r, c) over 64 x 64 tiles, 256 threads: the loads are 16-byte row
// segments of src (c contiguous), the stores are runs of 8 consecutive r of one output
// row per thread (16 or 32 bytes), both through a padded shared tile.
// Store functors write n <= 8 values v[0 .. n) at (g, c, r .. r+n-1).
template <int P>
struct StoreOperand {  // an operand matrix [g][c][ld] in precision P
  void* dst;
  long long ld;
  size_t lo;
  __device__ void operator()(int g, int c, int r, const float (&v)[8], int n) const {
    const size_t idx = static_cast<size_t>((static_cast<long long>(g) * rows_per_group + c) * ld + r);
    if (n == 8) {
      if constexpr (P == kBF16) {
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(dst) + idx) =
            make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                       pack_bf16x2(v[6], v[7]));
      } else {
        float* d = reinterpret_cast<float*>(dst) + idx;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float4 x = make_float4(tf32_rna(v[4 * h]), tf32_rna(v[4 * h + 1]), tf32_rna(v[4 * h + 2]),
                                       tf32_rna(v[4 * h + 3]));
          *reinterpret_cast<float4*>(d + 4 * h) = x;
          if constexpr (P == kTF32x3)
            *reinterpret_cast<float4*>(d + lo + 4 * h) =
                make_float4(tf32_rna(v[4 * h] - x.x), tf32_rna(v[4 * h + 1] - x.y), tf32_rna(v[4 * h + 2] - x.z),
                            tf32_rna(v[4 * h + 3] - x.w));
        }
      }
    } else {
      for (int k = 0; k < n; ++k) store_operand<P>(dst, idx + k, lo, v[k]);
    }
  }
  long long rows_per_group;
};

// The untransposed copy (k_transpose64's Direct): the operand [g][r][ld] of the tile's own
// rows, four consecutive columns per call (n <= 4 valid).
template <int P>
struct StoreOperandRows {
  void* dst;
  long long ld;
  size_t lo;
  long long rows_per_group;
  __device__ void operator()(int g, int r, int c, const float4& v, int n) const {
    const size_t idx = static_cast<size_t>((static_cast<long long>(g) * rows_per_group + r) * ld + c);
    if (n == 4) {
      if constexpr (P == kBF16) {
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(dst) + idx) =
            make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
      } else {
        const float4 h = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(dst) + idx) = h;
        if constexpr (P == kTF32x3)
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(dst) + idx + lo) =
              make_float4(tf32_rna(v.x - h.x), tf32_rna(v.y - h.y), tf32_rna(v.z - h.z), tf32_rna(v.w - h.w));
      }
    } else {
      const float x[4] = {v.x, v.y, v.z, v.w};
      for (int k = 0; k < n; ++k) store_operand<P>(dst, idx + k, lo, x[k]);
    }
  }
};
struct NoDirect {
  __device__ void operator()(int, int, int, const float4&, int) const {}
};

struct StoreF32 {  // a float32 matrix [g][c][ld], overwritten or accumulated into
  float* dst;
  long long ld, rows_per_group;
  int accumulate;
  __device__ void operator()(int g, int c, int r, const float (&v)[8], int n) const {
    float* d = dst + (static_cast<long long>(g) * rows_per_group + c) * ld + r;
    if (n == 8 && (reinterpret_cast<uintptr_t>(d) & 15) == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float4 x = make_float4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]);
        if (accumulate) {
          const float4 o = *reinterpret_cast<const float4*>(d + 4 * h);
          x.x += o.x;
          x.y += o.y;
          x.z += o.z;
          x.w += o.w;
        }
        *reinterpret_cast<float4*>(d + 4 * h) = x;
      }
    } else {
      for (int k = 0; k < n; ++k) d[k] = accumulate ? d[k] + v[k] : v[k];
    }
  }
};

// Source elements: float32, or bf16 bit patterns (uint16_t, widened exactly).
__device__ __forceinline__ float src_value(const float* p) { return *p; }
__device__ __forceinline__ float src_value(const uint16_t* p) { return __uint_as_float(static_cast<uint32_t>(*p) << 16); }
__device__ __forceinline__ float4 src_value4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 src_value4(const uint16_t* p) {
  const uint2 x = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(x.x << 16), __uint_as_float(x.x & 0xFFFF0000u), __uint_as_float(x.y << 16),
                     __uint_as_float(x.y & 0xFFFF0000u));
}

template <class Store, class Direct = NoDirect, class T = float>
__global__ void __launch_bounds__(256) k_transpose64(const T* __restrict__ src, long long src_ld,
                                                      long long src_gs, int R, int C, const int* gmap, Store st,
                                                      Direct direct = {}) {
  __shared__ float tile[64][65];
  const int g = blockIdx.z;
  const long long gs = gmap ? gmap[g] : g;
  const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64;
  const T* s = src + gs * src_gs;
  const int t = threadIdx.x;
  const bool vec = (src_ld & 3) == 0 && (reinterpret_cast<uintptr_t>(s) & (4 * sizeof(T) - 1)) == 0;
#pragma unroll
  for (int i = t; i < 64 * 16; i += 256) {
    const int rr = i >> 4, cq = (i & 15) * 4;
    const int r = r0 + rr, c = c0 + cq;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < R) {
      const T* p = s + static_cast<long long>(r) * src_ld + c;
      if (vec && c + 3 < C) {
        v = src_value4(p);
      } else {
        if (c < C) v.x = src_value(p);
        if (c + 1 < C) v.y = src_value(p + 1);
        if (c + 2 < C) v.z = src_value(p + 2);
        if (c + 3 < C) v.w = src_value(p + 3);
      }
      if (c < C) direct(g, r, c, v, min(4, C - c));
    }
    tile[rr][cq] = v.x;
    tile[rr][cq + 1] = v.y;
    tile[rr][cq + 2] = v.z;
    tile[rr][cq + 3] = v.w;
  }
  __syncthreads();
#pragma unroll
  for (int i = t; i < 64 * 8; i += 256) {
    const int cc = i >> 3, rq = (i & 7) * 8;
    const int c = c0 + cc, r = r0 + rq;
    if (c >= C || r >= R) continue;
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = tile[rq + k][cc];
    st(g, c, r, v, min(8, R - r));
  }
}

template <class Store>
pc_status_t launch_transpose64(const float* src, long long src_ld, long long src_gs, int G, int R, int C,
                               const int* gmap, const Store& st, cudaStream_t s) {
  if (G == 0 || R == 0 || C == 0) return PC_OK;
  k_transpose64<Store><<<dim3(cdiv(C, 64), cdiv(R, 64), G), 256, 0, s>>>(src, src_ld, src_gs, R, C, gmap, st);
  PC_LAUNCH_CHECK();
  return PC_OK;
}

// The same from a bf16 source (bit patterns): exact for a bf16 operand.
inline pc_status_t transpose_bf16_to_operand(const uint16_t* src, long long src_ld, long long src_gs, int G, int R,
                                             int C, const Operand& dst, cudaStream_t s) {
  if (G == 0 || R == 0 || C == 0) return PC_OK;
  k_transpose64<StoreOperand<kBF16>, NoDirect, uint16_t><<<dim3(cdiv(C, 64), cdiv(R, 64), G), 256, 0, s>>>(
      src, src_ld, src_gs, R, C, nullptr,
      StoreOperand<kBF16>{dst.ptr, dst.ld, dst.lo_elems, static_cast<long long>(C)});
  PC_LAUNCH_CHECK();
  return PC_OK;
}

template <int P>
pc_status_t transpose_to_operand(const float* src, long long src_ld, long long src_gs, int G,
                                 int R, int C, const Operand& dst, cudaStream_t s, const int* gmap = nullptr) {
  // operand rows are 64-element aligned, so full runs of 8 are 16-byte aligned
  return launch_transpose64(src, src_ld, src_gs, G, R, C, gmap,
                            StoreOperand<P>{dst.ptr, dst.ld, dst.lo_elems, static_cast<long long>(C)}, s);
}

// Both operand copies of src in one pass over it: rows (dst[g][r][c], as rows_to_operand)
// and transposed (dstT[g][c][r], as transpose_to_operand).
template <int P>
pc_status_t operand_and_transpose(const float* src, long long src_ld, long long src_gs, int G, int R, int C,
                                  const Operand& dst, const Operand& dstT, cudaStream_t s, const int* gmap = nullptr) {
  if (G == 0 || R == 0 || C == 0) return PC_OK;
  k_transpose64<StoreOperand<P>, StoreOperandRows<P>><<<dim3(cdiv(C, 64), cdiv(R, 64), G), 256, 0, s>>>(
      src, src_ld, src_gs, R, C, gmap, StoreOperand<P>{dstT.ptr, dstT.ld, dstT.lo_elems, static_cast<long long>(C)},
      StoreOperandRows<P>{dst.ptr, dst.ld, dst.lo_elems, static_cast<long long>(R)});
  PC_LAUNCH_CHECK();
  return PC_OK;
}

// dst[g][c][r] (+)= src[g][r][c] in float32, dst rows ld apart.
inline pc_status_t transpose_f32(const float* src, long long src_ld, long long src_gs, int G, int R, int C,
                                 float* dst, long long dst_ld, int accumulate, cudaStream_t s) {
  return launch_transpose64(src, src_ld, src_gs, G, R, C, nullptr,
                            StoreF32{dst, dst_ld, static_cast<long long>(C), accumulate}, s);
}

// w[r] (rows i0 + r of column j, one lane per column) *= rs[i0 + r] * cs[j] (NULL: 1).
__device__ __forceinline__ void scale_rows(const float* rs, const float* cs, int i0, int j, int M,
                                           float (&w)[32]) {
  const float c = cs ? cs[j] : 1.f;
#pragma unroll
  for (int r = 0; r < 32; ++r) w[r] *= (rs && i0 + r < M) ? rs[i0 + r] * c : c;
}

// Shared with the circuits: F[g][i][j] (+)= theta[g][i][j] * D[i,j].
struct EpiThetaScale : EpiNoHooks {
  static constexpr bool kTranspose = true;
  // TF32 accumulates unsliced: a parameter-flow entry is one contraction, not a chain of
  // them, and its truncation bias (at most ~4e-5 of the value at K = 15872) is far below
  // the mode's rounding; 256-wide tiles would not hold sliced sums in registers.
  static constexpr int kSliceTF32 = 0;
  // Unsliced contractions fetch the tile's theta block into the idle ring with
  // asynchronous copies (32 in flight per thread) once the MMAs are done, instead of 16
  // dependent-free global loads at a time per thread in apply.
  static constexpr bool kPrefetchTile = true;
  struct Params {
    float* F;
    const float* theta;
    int M, N, accumulate;
    const int* gmap;  // group g reads theta / writes F at matrix gmap[g] (NULL: g)
    // D is scaled by rscale[i] * cscale[j] (NULL: 1): the inverse operand row scales of
    // the fp8 flow contractions
    const float* rscale = nullptr;
    const float* cscale = nullptr;
  };
  // Transposed so that lane l owns column col0 + l of the warp's 32 rows: every theta
  // load and F store of the warp covers one contiguous row segment. All loads of the
  // chunk are issued before the first store.
  __device__ static void apply(const Params& p, int g, int m0, int n0, int row, int col0,
                               float (&v)[32], uint8_t*, float* tbuf) {
    float w[32];
    warp_transpose32(v, w, tbuf);
    const int lane = threadIdx.x & 31;
    const int i0 = m0 + row - lane;
    const int j = n0 + col0 + lane;
    if (j >= p.N) return;
    const long long ld = p.N;
    const long long gm = p.gmap ? p.gmap[g] : g;
    const float* tp = p.theta + (gm * p.M + i0) * ld + j;
    float* Fp = p.F + (gm * p.M + i0) * ld + j;
    if (p.rscale || p.cscale) scale_rows(p.rscale, p.cscale, i0, j, p.M, w);
    // two halves of 16 rows keep the loads-before-stores batch within the register budget
#pragma unroll
    for (int h = 0; h < 32; h += 16) {
      float t[16], f[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const bool in = i0 + h + r < p.M;
        t[r] = in ? tp[(h + r) * ld] : 0.f;
        f[r] = (in && p.accumulate) ? Fp[(h + r) * ld] : 0.f;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (i0 + h + r < p.M) Fp[(h + r) * ld] = f[r] + t[r] * w[h + r];
    }
  }

  // apply for a partial product (a K half of a split tile, k_umma_gemm_persist): F +=
  // theta * D by one reduction per element, whatever accumulate says (F holds the other
  // half's share, or zeros the caller wrote).
  __device__ static void apply_add(const Params& p, int g, int m0, int n0, int row, int col0, float (&v)[32],
                                   uint8_t*, float* tbuf) {
    float w[32];
    warp_transpose32(v, w, tbuf);
    const int lane = threadIdx.x & 31;
    const int i0 = m0 + row - lane;
    const int j = n0 + col0 + lane;
    if (j >= p.N) return;
    const long long ld = p.N;
    const long long gm = p.gmap ? p.gmap[g] : g;
    const float* tp = p.theta + (gm * p.M + i0) * ld + j;
    float* Fp = p.F + (gm * p.M + i0) * ld + j;
    if (p.rscale || p.cscale) scale_rows(p.rscale, p.cscale, i0, j, p.M, w);
#pragma unroll
    for (int h = 0; h < 32; h += 16) {
      float t[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) t[r] = i0 + h + r < p.M ? tp[(h + r) * ld] : 0.f;
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (i0 + h + r < p.M) atomicAdd(Fp + (h + r) * ld, t[r] * w[h + r]);
    }
  }

  // theta block [kBM][BN] of the tile, float32 row-major in `stage` (0 outside theta).
  template <int BN>
  __device__ static void prefetch(const Params& p, int g, int m0, int n0, int et, uint8_t* stage) {
    constexpr int kPieces = BN / 4;  // 16-byte pieces of a tile row
    const long long gm = p.gmap ? p.gmap[g] : g;
    const float* src = p.theta + (gm * p.M + m0) * static_cast<long long>(p.N) + n0;
    const int nrows = min(kBM, p.M - m0), ncols = min(BN, p.N - n0);
#pragma unroll 4
    for (int i = et; i < kBM * kPieces; i += kEpiThreads) {
      const int r = i / kPieces, c0 = (i % kPieces) * 4;
      uint8_t* dst = stage + (static_cast<long long>(r) * BN + c0) * 4;
      const int n = (r < nrows && c0 < ncols) ? min(4, ncols - c0) : 0;
      if (n == 0) {
        *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const float* gp = src + static_cast<long long>(r) * p.N + c0;
      if ((reinterpret_cast<uintptr_t>(gp) & 15) == 0) {
        cp_async_16(dst, gp, static_cast<uint32_t>(n * 4));  // zero-fills beyond n values
      } else {
        float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (k < n) x[k] = gp[k];
        *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
      }
    }
  }

  template <int BN>
  __device__ static void apply_prefetched(const Params& p, int g, int m0, int n0, int row, int col0,
                                          float (&v)[32], const uint8_t* stage, float* tbuf) {
    float w[32];
    warp_transpose32(v, w, tbuf);
    const int lane = threadIdx.x & 31;
    const int i0 = m0 + row - lane;  // the warp's first row
    const int j = n0 + col0 + lane;
    if (j >= p.N) return;
    const long long ld = p.N;
    const long long gm = p.gmap ? p.gmap[g] : g;
    const float* ts = reinterpret_cast<const float*>(stage) + static_cast<long long>(i0 - m0) * BN + col0 + lane;
    float* Fp = p.F + (gm * p.M + i0) * ld + j;
    if (p.rscale || p.cscale) scale_rows(p.rscale, p.cscale, i0, j, p.M, w);
#pragma unroll
    for (int h = 0; h < 32; h += 16) {
      float f[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) f[r] = (i0 + h + r < p.M && p.accumulate) ? Fp[(h + r) * ld] : 0.f;
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (i0 + h + r < p.M) Fp[(h + r) * ld] = f[r] + ts[(h + r) * BN] * w[h + r];
    }
  }
};

// EpiThetaScale reading theta directly in apply (the persistent contraction's ring is never
// idle, so no tile is prefetched into it).
struct EpiThetaScaleDirect : EpiThetaScale {
  static constexpr bool kPrefetchTile = false;
};

// EpiThetaScale on persistent tiles (kLoadAhead): the theta block of a chunk (32 rows x
// 32 columns) comes through the warp's ring of shared-memory buffers, its 16-byte pieces
// swizzled by the row; the product theta * D is formed one row per lane, written back in
// place and read out one column per lane, so that each global store of the warp is one
// contiguous 128-byte row segment (the buffer doubles as the transpose). Flows are written
// with streaming stores, or added by one reduction per element when accumulating (each
// element of F has one writer per call). Needs N % 4 == 0 and a 16-byte aligned theta.
struct EpiThetaScaleAhead : EpiThetaScale {
  static constexpr bool kTranspose = false;
  static constexpr bool kPrefetchTile = false;
  static constexpr bool kLoadAhead = true;
  // two blocks (one in flight while the other is consumed): deeper rings cost the
  // contraction a ring stage, and measured slower (HCLT 768: 10.16 ms per step with two,
  // 10.49 with three, 10.54 with four)
  static constexpr int kAheadBufs = 2;
  static constexpr int kSmemBytes = kEpiWarps * kAheadBufs * 4096;
  __device__ static int piece(int r, int p) { return r * 32 + ((p ^ (r & 7)) << 2); }
  __device__ static void issue(const Params& p, int g, int m0, int n0, int q, int col0, float* buf) {
    const int lane = threadIdx.x & 31;
    const long long gm = p.gmap ? p.gmap[g] : g;
    const int pc = lane & 7;
    const int j = n0 + col0 + 4 * pc;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = 4 * k + (lane >> 3);
      const int i = m0 + q * 32 + r;
      const int n = (i < p.M && j < p.N) ? min(4, p.N - j) : 0;
      const float* src = n ? p.theta + (gm * p.M + i) * static_cast<long long>(p.N) + j : p.theta;
      cp_async_16(reinterpret_cast<uint8_t*>(buf + piece(r, pc)), src, static_cast<uint32_t>(n * 4));
    }
  }
  __device__ static void apply_buf(const Params& p, int g, int m0, int n0, int row, int col0, float (&v)[32],
                                   float* buf) {
    const int lane = threadIdx.x & 31;
    const int i = m0 + row;
    if (p.rscale || p.cscale) {
      const float rs = (p.rscale && i < p.M) ? p.rscale[i] : 1.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int j = n0 + col0 + c;
        v[c] *= rs * ((p.cscale && j < p.N) ? p.cscale[j] : 1.f);
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {  // row lane: theta * D, in place
      float4* t = reinterpret_cast<float4*>(buf + piece(lane, k));
      const float4 x = *t;
      *t = make_float4(x.x * v[4 * k], x.y * v[4 * k + 1], x.z * v[4 * k + 2], x.w * v[4 * k + 3]);
    }
    __syncwarp();
    const int i0 = m0 + row - lane;
    const int j = n0 + col0 + lane;
    if (j >= p.N) return;
    const long long gm = p.gmap ? p.gmap[g] : g;
    const long long ld = p.N;
    float* Fp = p.F + (gm * p.M + i0) * ld + j;
    const int pl = lane >> 2, wl = lane & 3;
    if (p.accumulate) {
#pragma unroll
      for (int r = 0; r < 32; ++r)
        if (i0 + r < p.M) atomicAdd(Fp + r * ld, buf[piece(r, pl) + wl]);
    } else {
#pragma unroll
      for (int r = 0; r < 32; ++r)
        if (i0 + r < p.M) __stcs(Fp + r * ld, buf[piece(r, pl) + wl]);
    }
  }
};

// D[i][j] (+)= the accumulator: the contraction's result as a float32 matrix (rows ld
// apart, M x N valid). Transposed per warp as EpiThetaScale, so that each store of the
// warp is one contiguous row segment.
struct EpiStoreF32 : EpiNoHooks {
  static constexpr bool kTranspose = true;
  static constexpr int kSliceTF32 = 0;  // as EpiThetaScale
  struct Params {
    float* D;
    long long ld;
    int M, N, accumulate;
    const float* rscale = nullptr;  // as EpiThetaScale's
    const float* cscale = nullptr;
    long long gstride = 0;          // elements between the outputs of groups (blockIdx.z)
  };
  __device__ static void apply(const Params& p, int g, int m0, int n0, int row, int col0, float (&v)[32], uint8_t*,
                               float* tbuf) {
    float w[32];
    warp_transpose32(v, w, tbuf);
    const int lane = threadIdx.x & 31;
    const int i0 = m0 + row - lane;
    const int j = n0 + col0 + lane;
    if (j >= p.N) return;
    float* Dp = p.D + g * p.gstride + static_cast<long long>(i0) * p.ld + j;
    if (p.rscale || p.cscale) scale_rows(p.rscale, p.cscale, i0, j, p.M, w);
#pragma unroll
    for (int h = 0; h < 32; h += 16) {
      float f[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) f[r] = (i0 + h + r < p.M && p.accumulate) ? Dp[(h + r) * p.ld] : 0.f;
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (i0 + h + r < p.M) Dp[(h + r) * p.ld] = f[r] + w[h + r];
    }
  }
};

}  // namespace pc
