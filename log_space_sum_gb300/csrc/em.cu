// EM M-step (pyjuice LowRank API doc, Training): every node's parameters become its
// statistic normalized over its children,
//
//   theta[i][j] = r[i][j] / sum_j r[i][j],   r = F   or   r = F / W (0 where W <= 0),
//
// the plain normalize(F) of a sum layer's parameter flows, or the LowRank conditional
// update normalize(theta * F+ / F-) with F- = theta * W. A row whose r sums to zero or to
// a non-finite value keeps its parameters.
//
// Memory-bound: one CTA per row reads F (and W) once and writes theta once, 8 (12 with
// W) bytes per parameter. Rows of up to 8192 aligned values are held in registers
// (every load of a thread issued before the first use); longer or unaligned rows are
// summed in a first pass and re-read (from L1/L2) in a second.
#include "pc_device.cuh"
#include "pc_host.h"

namespace pc {
namespace {

constexpr int kEmThreads = 256;

__device__ __forceinline__ float em_ratio(float f, float w) { return w > 0.f ? f / w : 0.f; }

// Sum over the CTA (all threads receive it).
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kEmThreads / 32; ++w) s += red[w];
  return s;
}

// kVec: rows start 16-byte aligned and N % 4 == 0 (float4 accesses).
template <bool kRatio, bool kVec>
__global__ void __launch_bounds__(kEmThreads) k_em_normalize(int N, const float* __restrict__ F,
                                                             const float* __restrict__ W,
                                                             float* __restrict__ theta) {
  __shared__ float red[kEmThreads / 32];
  const long long row0 = static_cast<long long>(blockIdx.x) * N;
  const float* f = F + row0;
  const float* w = kRatio ? W + row0 : nullptr;
  float* th = theta + row0;
  float acc = 0.f;
  if constexpr (kVec) {
    const int n4 = N >> 2;
    for (int i = threadIdx.x; i < n4; i += kEmThreads) {
      const float4 a = reinterpret_cast<const float4*>(f)[i];
      if constexpr (kRatio) {
        const float4 b = reinterpret_cast<const float4*>(w)[i];
        acc += (em_ratio(a.x, b.x) + em_ratio(a.y, b.y)) + (em_ratio(a.z, b.z) + em_ratio(a.w, b.w));
      } else {
        acc += (a.x + a.y) + (a.z + a.w);
      }
    }
  } else {
    for (int i = threadIdx.x; i < N; i += kEmThreads) acc += kRatio ? em_ratio(f[i], w[i]) : f[i];
  }
  const float s = block_sum(acc, red);
  if (!(s > 0.f) || !isfinite(s)) return;  // no flow reached the node: it keeps theta
  if constexpr (kVec) {
    const int n4 = N >> 2;
    for (int i = threadIdx.x; i < n4; i += kEmThreads) {
      float4 a = reinterpret_cast<const float4*>(f)[i];
      if constexpr (kRatio) {
        const float4 b = reinterpret_cast<const float4*>(w)[i];
        a = make_float4(em_ratio(a.x, b.x), em_ratio(a.y, b.y), em_ratio(a.z, b.z), em_ratio(a.w, b.w));
      }
      reinterpret_cast<float4*>(th)[i] = make_float4(a.x / s, a.y / s, a.z / s, a.w / s);
    }
  } else {
    for (int i = threadIdx.x; i < N; i += kEmThreads) th[i] = (kRatio ? em_ratio(f[i], w[i]) : f[i]) / s;
  }
}

// Register-resident rows: N % 4 == 0, 16-byte aligned, N <= 4 * kItems * kEmThreads.
template <bool kRatio, int kItems>
__global__ void __launch_bounds__(kEmThreads) k_em_normalize_reg(int N, const float* __restrict__ F,
                                                                 const float* __restrict__ W,
                                                                 float* __restrict__ theta) {
  __shared__ float red[kEmThreads / 32];
  const long long row0 = static_cast<long long>(blockIdx.x) * N;
  const float4* f = reinterpret_cast<const float4*>(F + row0);
  const float4* w = kRatio ? reinterpret_cast<const float4*>(W + row0) : nullptr;
  const int n4 = N >> 2;
  float4 r[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int i = threadIdx.x + k * kEmThreads;
    r[k] = i < n4 ? f[i] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if constexpr (kRatio) {
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int i = threadIdx.x + k * kEmThreads;
      const float4 b = i < n4 ? w[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      r[k] = make_float4(em_ratio(r[k].x, b.x), em_ratio(r[k].y, b.y), em_ratio(r[k].z, b.z), em_ratio(r[k].w, b.w));
    }
  }
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < kItems; ++k) acc += (r[k].x + r[k].y) + (r[k].z + r[k].w);
  const float s = block_sum(acc, red);
  if (!(s > 0.f) || !isfinite(s)) return;  // no flow reached the node: it keeps theta
  const float inv = 1.f / s;                // r * (1 / s): within 1.5 ulp of r / s
  float4* th = reinterpret_cast<float4*>(theta + row0);
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int i = threadIdx.x + k * kEmThreads;
    if (i < n4) th[i] = make_float4(r[k].x * inv, r[k].y * inv, r[k].z * inv, r[k].w * inv);
  }
}

template <bool kRatio>
void launch_em(int rows, int N, const float* F, const float* W, float* theta, bool vec, cudaStream_t s) {
  const int items = vec ? (N / 4 + kEmThreads - 1) / kEmThreads : 0;
  if (vec && items <= 1)
    k_em_normalize_reg<kRatio, 1><<<rows, kEmThreads, 0, s>>>(N, F, W, theta);
  else if (vec && items <= 2)
    k_em_normalize_reg<kRatio, 2><<<rows, kEmThreads, 0, s>>>(N, F, W, theta);
  else if (vec && items <= 4)
    k_em_normalize_reg<kRatio, 4><<<rows, kEmThreads, 0, s>>>(N, F, W, theta);
  else if (vec && items <= 8)
    k_em_normalize_reg<kRatio, 8><<<rows, kEmThreads, 0, s>>>(N, F, W, theta);
  else if (vec)
    k_em_normalize<kRatio, true><<<rows, kEmThreads, 0, s>>>(N, F, W, theta);
  else
    k_em_normalize<kRatio, false><<<rows, kEmThreads, 0, s>>>(N, F, W, theta);
}

}  // namespace
}  // namespace pc

extern "C" {

pc_status_t pc_em_normalize(int G, int M, int N, const float* F, const float* W, float* theta,
                            cudaStream_t stream) {
  pc::clear_error();
  PC_CHECK(F && theta, PC_ERR_NULL, "F and theta must not be NULL");
  PC_CHECK(G >= 1 && M >= 1 && N >= 1, PC_ERR_SHAPE, "G, M, N must be >= 1 (got %d, %d, %d)", G, M, N);
  const long long rows = static_cast<long long>(G) * M;
  PC_CHECK(rows < (1ll << 31), PC_ERR_SHAPE, "G * M must be < 2^31");
  const bool vec = N % 4 == 0 && pc::aligned16(F) && pc::aligned16(theta) && (!W || pc::aligned16(W));
  const int slot = pc::profile_begin(stream);
  if (W)
    pc::launch_em<true>(static_cast<int>(rows), N, F, W, theta, vec, stream);
  else
    pc::launch_em<false>(static_cast<int>(rows), N, F, W, theta, vec, stream);
  PC_LAUNCH_CHECK();
  pc::profile_end(slot, stream, PC_KIND_EM_MSTEP, rows * N * (W ? 12ll : 8ll));
  return PC_OK;
}

}  // extern "C"
