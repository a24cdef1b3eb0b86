// Whole HMM circuit, forward + backward, on the tensor-core contraction.
//
// The circuit (pyjuice PR #62, Results table: "HMM, 4096 latents, 32 positions";
// Summary 2, first bullet: the HMM's sum layers share their children) is built from
// the last position back, with positions t = 0..T-1:
//   P_{T-1}(k) = E[k, x_{T-1}]
//   S_t(k)     = sum_l A[k,l] P_{t+1}(l)            tied H x H sum layer, shared children
//   P_t(k)     = E[k, x_t] S_t(k)                    product (emission) layer
//   LL         = log sum_k pi[k] P_0(k)              root sum layer
//
// Each sum layer's log-space form out = m + log sum_l A exp(x - m) is evaluated with
// the exponentials of its children kept from the layer below: the epilogue of S_t
// writes the next layer's shifted children u_t = exp(x_t - shift_t) directly as
//   u_t[k,b] = E[k, x_{t,b}] * D_t[k,b] * c_{t,b},   D_t = sum_l A[k,l] u_{t+1}[l,b]
// (the log of the epilogue and the exp of the next prologue cancel), where
//   c_{t,b} = 1 / (max_l u_{t+1}[l,b] * max_k E[k, x_{t,b}] sum_l A[k,l])
// bounds every u_t by 1. max_l u_{t+1} is the exact column maximum of the layer
// below (reduced by that layer's epilogue), so the bound's slack never accumulates
// over positions. The per-sample log-scales accumulate in double:
//   LL_b = log sum_k pi[k] u_0[k,b] - sum_t log c_{t,b}.
//
// Backward (root flow 1 per sample; product nodes pass flows to their children):
//   r_b        = 1 / sum_k pi[k] u_0[k,b]
//   f_0[k,b]   = pi[k] u_0[k,b] r_b                   flows of P_0 (posteriors)
//   w_t[k,b]   = f_t / D_t = E[k,x_t] c_t s_t          sum-layer flow / its value,
//                (w_0 = pi[k] r_b E[k,x_0] c_0)        the contraction's right factor
//   s_{t+1}[j,b] = sum_i A[i,j] w_t[i,b]               element-flow contraction
//   f_{t+1}    = u_{t+1} s_{t+1}                       element flows = posteriors
//   dA[i,j]    = A[i,j] sum_{t,b} w_t[i,b] u_{t+1}[j,b] parameter flows, all T-1 tied
//                                                       layers in one contraction of
//                                                       depth (T-1) B
//   dE[k,v]    = sum_{t,b: x_{t,b}=v} f_t[k,b],  dpi[k] = sum_b f_0[k,b]
#include <cmath>

#include "pc_launch.cuh"
#include "pc_tokens.cuh"

namespace pc {
namespace {

constexpr int kChainBN = 128;

// ------------------------------------------------------------------ set-up

// rs[k] = sum_l A[k,l], one warp per row (float: it only feeds an upper bound).
__global__ void k_rowsum(const float* __restrict__ A, int H, float* __restrict__ rs) {
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= H) return;
  const float* a = A + static_cast<long long>(row) * H;
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  if ((H & 3) == 0 && (reinterpret_cast<uintptr_t>(a) & 15) == 0) {
    const float4* a4 = reinterpret_cast<const float4*>(a);
    for (int l = lane; l < H / 4; l += 32) {
      const float4 v = a4[l];
      s += (v.x + v.y) + (v.z + v.w);
    }
  } else {
    for (int l = lane; l < H; l += 32) s += a[l];
  }
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) rs[row] = s;
}

// The transition operand and the row sums in one pass over A: one block per row, the
// row read once with 16-byte loads (H % 4 == 0, A 16-byte aligned), its operand copy
// written and its sum reduced in a fixed order (float: it only feeds an upper bound).
template <int P>
__global__ void __launch_bounds__(256) k_transition_operand(const float* __restrict__ A, int H, void* op,
                                                            long long op_ld, size_t op_lo, float* __restrict__ rs) {
  __shared__ float red[8];
  const int row = blockIdx.x;
  const float4* a4 = reinterpret_cast<const float4*>(A + static_cast<long long>(row) * H);
  float sum = 0.f;
  for (int q = threadIdx.x; q < H / 4; q += blockDim.x) {
    const float4 v = a4[q];
    sum += (v.x + v.y) + (v.z + v.w);
    const size_t idx = static_cast<size_t>(row * op_ld + 4 * q);
    if constexpr (P == kBF16) {
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(op) + idx) =
          make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    } else {
      const float4 h = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
      *reinterpret_cast<float4*>(static_cast<float*>(op) + idx) = h;
      if constexpr (P == kTF32x3)
        *reinterpret_cast<float4*>(static_cast<float*>(op) + idx + op_lo) =
            make_float4(tf32_rna(v.x - h.x), tf32_rna(v.y - h.y), tf32_rna(v.z - h.z), tf32_rna(v.w - h.w));
    }
  }
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += red[w];
    rs[row] = t;
  }
}

// Et[v][k] = E[k][v] over 64 x 64 tiles, and the emission bounds of every token from the
// same tile: emax[v] = max_k E[k,v], emax_rs[v] = max_k E[k,v] * rs[k], reduced over the
// tiles with atomic maxima on the bit patterns (non-negative values; zeroed beforehand;
// the result does not depend on the order).
__global__ void __launch_bounds__(256) k_emission_transpose(const float* __restrict__ E, int H, int V,
                                                            const float* __restrict__ rs, float* __restrict__ Et,
                                                            float* __restrict__ emax, float* __restrict__ emax_rs) {
  __shared__ float tile[64][65];
  __shared__ float rsk[64];
  const int v0 = blockIdx.x * 64, k0 = blockIdx.y * 64;
  const int t = threadIdx.x;
  if (t < 64) rsk[t] = k0 + t < H ? rs[k0 + t] : 0.f;
  for (int i = t; i < 64 * 64; i += 256) {
    const int kk = i >> 6, vv = i & 63;
    const int k = k0 + kk, v = v0 + vv;
    tile[kk][vv] = (k < H && v < V) ? E[static_cast<long long>(k) * V + v] : 0.f;
  }
  __syncthreads();
  for (int i = t; i < 64 * 64; i += 256) {
    const int vv = i >> 6, kk = i & 63;
    const int k = k0 + kk, v = v0 + vv;
    if (k < H && v < V) Et[static_cast<long long>(v) * H + k] = tile[kk][vv];
  }
  // bounds: four threads per token, 16 of the tile's states each
  const int vv = t >> 2, part = t & 3;
  float m0 = 0.f, m1 = 0.f;
  for (int kk = part * 16; kk < part * 16 + 16; ++kk) {
    const float e = tile[kk][vv];
    m0 = fmaxf(m0, e);
    m1 = fmaxf(m1, e * rsk[kk]);
  }
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
  if (part == 0 && v0 + vv < V) {
    atomic_max_nonneg(&emax[v0 + vv], m0);
    atomic_max_nonneg(&emax_rs[v0 + vv], m1);
  }
}


// The per-sample scale of a layer, 1 / (the bound of its values): clamped at 2^100, where
// it is still exact as a power-of-two shift of the column, so that the products below
// never overflow and a denormal emission is scaled into the normal range before it is
// multiplied. A column whose largest value then falls below kRangeFloor (the bound was
// looser than e^-55 at some position; values that matter would lose precision in the
// operand formats) is reported by the root instead of giving a silently wrong LL.
constexpr float kScaleMax = 0x1p100f;
constexpr float kRangeFloor = 0x1p-80f;
constexpr float kUnderflowMark = 0x1p-149f;  // column max of a column whose nonzero products underflowed
// The bound of a chain layer is a product a * b (the previous maximum and the emission
// bound), whose float32 product can underflow for a denormal b: the scale is formed as
// (1/a)(1/b), where an overflow only meets the clamp. (Float only: this GPU's FP64 pipe is
// narrow.)
__device__ __forceinline__ float layer_scale(float bound) { return bound > 0.f ? fminf(1.f / bound, kScaleMax) : 0.f; }
__device__ __forceinline__ float layer_scale2(float a, float b) {
  return (a > 0.f && b > 0.f) ? fminf((1.f / a) * (1.f / b), kScaleMax) : 0.f;
}

__device__ __forceinline__ void write_scale(float c, float* cf, double* logc, long long idx) {
  cf[idx] = c;
  logc[idx] = c > 0.f ? log(static_cast<double>(c)) : static_cast<double>(INFINITY);
}

// The last position: u_{T-1}[k,b] = E[k, x_{T-1,b}] / max_k E[k, x_{T-1,b}].
// Tile of 32 states (lanes) x 32 samples; writes the next forward operand
// (batch-major), the parameter-flow operand (node-major, column block T-2), or
// u_0 in float32 when T = 1; and the column maximum.
template <int P>
__global__ void k_hmm_leaf(int H, int B, int T, const int* __restrict__ tokens,
                           const float* __restrict__ Et, const float* __restrict__ emax,
                           void* ubm, long long ubm_ld, size_t ubm_lo, void* un, long long un_ld,
                           size_t un_lo, long long un_col, float* U0, float* umax, float* cf,
                           double* logc) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.x * 32, b0 = blockIdx.y * 32;
  const int k = k0 + threadIdx.x;
  const int t = T - 1;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int b = b0 + i;
    float u = 0.f;
    if (b < B) {
      const int tok = tokens[static_cast<long long>(b) * T + t];
      const float em = emax[tok];
      const float c = layer_scale(em);
      if (k < H) {
        u = Et[static_cast<long long>(tok) * H + k] * c;
        if (ubm) store_operand<P>(ubm, static_cast<size_t>(b * ubm_ld + k), ubm_lo, u);
        if (U0) U0[static_cast<long long>(b) * H + k] = u;
      }
      // the column maximum is em * c exactly (rounding is monotone): no reduction needed
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        write_scale(c, cf, logc, static_cast<long long>(t) * B + b);
        umax[static_cast<long long>(t) * B + b] = em * c;
      }
    }
    tile[i][threadIdx.x] = u;
  }
  if (!un) return;
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int kk = k0 + i, b = b0 + threadIdx.x;
    if (kk < H && b < B)
      store_operand<P>(un, static_cast<size_t>(kk * un_ld + un_col + b), un_lo, tile[threadIdx.x][i]);
  }
}

// The staged emission block holds row r (a state) as Pitch floats whose 16-byte pieces
// are swizzled by r: an epilogue thread reads its row's 32 columns with 8 vector loads,
// and the 32 rows of a warp spread over all banks.
template <int Pitch = kChainBN>
__device__ __forceinline__ int es_index(int r, int c) { return r * Pitch + (((c >> 2) ^ (r & 7)) << 2) + (c & 3); }
template <int Pitch = kChainBN>
__device__ __forceinline__ void es_run(const float* Es, int row, int col0, float (&e)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 x = *reinterpret_cast<const float4*>(Es + es_index<Pitch>(row, col0 + 4 * j));
    e[4 * j] = x.x;
    e[4 * j + 1] = x.y;
    e[4 * j + 2] = x.z;
    e[4 * j + 3] = x.w;
  }
}
// The per-column factors c_s[col0 .. col0+31] (the same for every thread: broadcast loads).
__device__ __forceinline__ void cs_run(const float* c_s, int col0, float (&cv)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 x = *reinterpret_cast<const float4*>(c_s + col0 + 4 * j);
    cv[4 * j] = x.x;
    cv[4 * j + 1] = x.y;
    cv[4 * j + 2] = x.z;
    cv[4 * j + 3] = x.w;
  }
}

// Stages the CTA's emission block Es(r, c) = E[m0 + r, x_{t,b}] (b = n0 + c) into shared
// memory (es_index layout): rows and columns outside the problem read 0. The epilogue
// warps do this while the contraction's K loop runs, so the gathers are off the critical
// path. The block is W columns wide (W <= kChainBN); each epilogue warp owns
// W / kEpiWarps of them and issues 8 columns x 4 rows of loads per batch.
template <int W, int Pitch = kChainBN>
__device__ __forceinline__ void stage_emissions(const float* __restrict__ Et, int H, int B, int m0, int n0,
                                                const int* tok_s, float* Es, int et) {
  constexpr int kCols = W / kEpiWarps;  // columns staged by one epilogue warp
  constexpr int kBatch = kCols < 8 ? kCols : 8;
  static_assert(W <= kChainBN && W % kEpiWarps == 0 && kCols % kBatch == 0, "whole batches of columns per warp");
  const int lane = et & 31;
  const int c_begin = (et >> 5) * kCols;
#pragma unroll 1
  for (int cb = c_begin; cb < c_begin + kCols; cb += kBatch) {
    float vals[kBatch][4];
#pragma unroll
    for (int c = 0; c < kBatch; ++c) {
      const bool bin = n0 + cb + c < B;
      const float* src = Et + static_cast<long long>(tok_s[cb + c]) * H + m0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        vals[c][i] = (bin && m0 + r < H) ? src[r] : 0.f;
      }
    }
#pragma unroll
    for (int c = 0; c < kBatch; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) Es[es_index<Pitch>(lane + 32 * i, cb + c)] = vals[c][i];
  }
}

// The same block gathered with asynchronous 4-byte copies (zero-filled outside the
// problem), which the issuing thread completes with cp_async_wait_all before a barrier.
__device__ __forceinline__ void cp_async_4(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
template <int W, int Pitch>
__device__ __forceinline__ void stage_emissions_async(const float* __restrict__ Et, int H, int B, int m0, int n0,
                                                      const int* tok_s, float* Es, int et) {
  static_assert(W % kEpiWarps == 0, "whole columns per warp");
  constexpr int kCols = W / kEpiWarps;
  const int lane = et & 31;
  const int c_begin = (et >> 5) * kCols;
#pragma unroll 1
  for (int c = c_begin; c < c_begin + kCols; ++c) {
    const bool bin = n0 + c < B;
    const float* src = Et + static_cast<long long>(tok_s[c]) * H + m0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane + 32 * i;
      const bool in = bin && m0 + r < H;
      cp_async_4(Es + es_index<Pitch>(r, c), in ? src + r : Et, in ? 4u : 0u);
    }
  }
}

// The wide bf16 split-K tiles (128 x 256, epilogue width kChainBN) stage only the first
// kEsLoCols columns of the emission block before the K loop, so that the ring keeps four
// stages; the other columns are gathered into the idle ring behind the staged tiles
// while the partial sums are exchanged.
constexpr int kEsLoCols = kChainBN / 2;
constexpr int kEsHiBytes = (kChainBN - kEsLoCols) * kBM * 4;

// Column maxima of the warp's 32 x 32 block of non-negative values (thread = row, v[c] =
// column c): lane l returns the maximum of column l. Non-negative floats order like
// their bit patterns, so each column is one integer warp reduction.
__device__ __forceinline__ float warp_column_max(const float (&v)[32]) {
  const int lane = threadIdx.x & 31;
  unsigned mx = 0;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(v[c]) & 0x7FFFFFFFu);  // -0 as +0
    if (lane == c) mx = m;
  }
  return __uint_as_float(mx);
}

// Columns whose product u = e (D c) is 0 although e, D and the column's scale c are
// positive (the product underflowed).
__device__ __forceinline__ uint32_t underflow_mask(const float (&u)[32], const float (&e)[32], const float (&d)[32],
                                                   const float* c_s, int col0, int nvalid) {
  uint32_t m = 0;
#pragma unroll
  for (int c = 0; c < 32; ++c)
    if (c < nvalid && u[c] == 0.f && e[c] > 0.f && d[c] > 0.f && c_s[col0 + c] > 0.f) m |= 1u << c;
  return m;
}

// After the values are stored: a column whose nonzero product underflowed to 0 takes the
// smallest positive float into its maximum, so that the root can tell it from a column of
// exact zeros (a sequence of probability 0).
__device__ __forceinline__ void mark_underflow(float (&v)[32], uint32_t under) {
  if (under) {
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if ((under >> c) & 1u) v[c] = kUnderflowMark;
  }
}

// Split-K chain epilogues (bf16) stage their node-major tile [k][b] (row pitch 272
// bytes: the 16-byte runs of 32 consecutive rows spread over all banks) and their
// batch-major tile [b][k] in the idle ring; store_staged then writes both out with
// coalesced 16-byte accesses (stage_tile_store_bf16).
constexpr int kNodePitch = 272;
constexpr int kBatchPitch = 256;
constexpr int kNodeTileBytes = kBM * kNodePitch;
constexpr int kBatchTileBytes = kChainBN * kBatchPitch;

__device__ __forceinline__ void stage_node_run(uint8_t* stage, int row, int col0, const float (&v)[32]) {
  uint4* nt = reinterpret_cast<uint4*>(stage + row * kNodePitch + col0 * 2);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    nt[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                       pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
}

__device__ __forceinline__ void stage_batch_col(uint8_t* stage, int row, int col0, const float (&v)[32]) {
  __nv_bfloat16* bt = reinterpret_cast<__nv_bfloat16*>(stage + kNodeTileBytes);
#pragma unroll
  for (int c = 0; c < 32; ++c) bt[(col0 + c) * (kBatchPitch / 2) + row] = __float2bfloat16_rn(v[c]);
}

// ----------------------------------------------------------- forward epilogue
struct HmmFwdParams {
    int H, B, T, t;
    const int* tokens;
    const float* Et;
    const float* emax_rs;
    const float* umax_prev;  // column maxima of u_{t+1}
    float* umax_cur;         // column maxima of u_t (atomic max, zeroed beforehand)
    float* cf;
    double* logc;
    void* ubm;               // u_t batch-major for S_{t-1} (NULL at t = 0)
    long long ubm_ld;
    size_t ubm_lo;
    void* un;                // u_t node-major, column (t-1) B, for dA (NULL if not needed)
    long long un_ld;
    size_t un_lo;
    float* U0;               // u_0 float32 [B][H] (t = 0 only)
};

// W: the columns one CTA's epilogue finishes (kChainBN, or half of it for 128-wide
// split-K tiles).
template <int P, int W = kChainBN>
struct EpiHmmFwd {
  using Params = HmmFwdParams;
  static constexpr bool kTranspose = false;
  // sliced 3xTF32 tiles: 16 epilogue warps (prepare strides by 256 threads and needs no
  // more; apply takes one chunk per warp)
  static constexpr int kEpiWarps = P == kTF32x3 ? 16 : 8;
  static constexpr int kSliceBF16 = 0;
  static constexpr int kSliceTF32 = 0;  // the TF32 chain runs as split-K pairs: one accumulation
  // 3xTF32: slices of a whole ring slot (4 k-steps; see EpiSlice3x): the chain has T - 1
  // layers, whose residual truncation bias stays far below the fp32 mode's 1e-5 (LL
  // errors 4.4e-7 and 8.6e-7 on the 4096 x 32 and 1024 x 64 workloads)
  static constexpr int kSlice3x = 4;
  // the 3xTF32 ring needs the room: it gathers emissions directly instead
  static constexpr bool kStageE = P != kTF32x3;
  static constexpr bool kEsSplit = P != kTF32x3 && W == kChainBN;  // see kEsLoCols
  // split-K pairs stage their bf16 output tiles in the idle ring; TF32 values (4 bytes)
  // would not fit beside the exchange buffer and go to global memory from registers
  static constexpr bool kStageOut = P == kBF16;
  static constexpr int kEsLo = kEsSplit ? kEsLoCols : W;         // columns staged before the K loop
  static constexpr int kEsPitch = kEsSplit ? kEsLoCols : kChainBN;
  static constexpr int kSmemBytes = kChainBN * 4 * 2 + (kStageE ? kEsPitch * kBM * 4 : 0);

  __device__ static void prepare(const Params& p, int, int m0, int n0, int et, uint8_t* smem) {
    int* tok_s = reinterpret_cast<int*>(smem);
    float* c_s = reinterpret_cast<float*>(smem) + kChainBN;
    for (int c = et; c < W; c += kEpiThreads) {
      const int b = n0 + c;
      int tok = 0;
      float cv = 0.f;
      if (b < p.B) {
        tok = p.tokens[static_cast<long long>(b) * p.T + p.t];
        cv = layer_scale2(p.umax_prev[b], p.emax_rs[tok]);
        if (m0 == 0) write_scale(cv, p.cf, p.logc, static_cast<long long>(p.t) * p.B + b);
      }
      tok_s[c] = tok;
      c_s[c] = cv;
    }
    if constexpr (kStageE) {
      epilogue_bar_sync();
      stage_emissions<kEsLo, kEsPitch>(p.Et, p.H, p.B, m0, n0, tok_s, reinterpret_cast<float*>(smem) + 2 * kChainBN,
                                       et);
    }
  }

  // Thread = state k (TMEM lane), registers = 32 consecutive samples.
  __device__ static void apply(const Params& p, int, int m0, int n0, int row, int col0,
                               float (&v)[32], uint8_t* smem, float*) {
    const int* tok_s = reinterpret_cast<const int*>(smem);
    const float* c_s = reinterpret_cast<const float*>(smem) + kChainBN;
    const float* Es = reinterpret_cast<const float*>(smem) + 2 * kChainBN;
    const int k = m0 + row;
    const bool kin = k < p.H;
    const int nvalid = kin ? min(32, p.B - (n0 + col0)) : 0;
    static_assert(!kEsSplit, "the split emission block is read by apply_staged");
    float e[32], cv[32];
    if constexpr (kStageE) {
      es_run(Es, row, col0, e);
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) e[c] = c < nvalid ? p.Et[static_cast<long long>(tok_s[col0 + c]) * p.H + k] : 0.f;
    }
    cs_run(c_s, col0, cv);
    // u = e (D c) into e; v keeps D for the rare check below
#pragma unroll
    for (int c = 0; c < 32; ++c) e[c] = c < nvalid ? e[c] * (v[c] * cv[c]) : 0.f;
    if (p.ubm) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c < nvalid)
          store_operand<P>(p.ubm, static_cast<size_t>((n0 + col0 + c) * p.ubm_ld + k), p.ubm_lo, e[c]);
    }
    if (p.U0) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c < nvalid) p.U0[static_cast<long long>(n0 + col0 + c) * p.H + k] = e[c];
    }
    if (p.un && nvalid > 0)
      store_operand_run<P>(p.un, static_cast<size_t>(k * p.un_ld + static_cast<long long>(p.t - 1) * p.B + n0 + col0),
                           p.un_lo, e, nvalid);
    const int b = n0 + col0 + (threadIdx.x & 31);
    float mx = warp_column_max(e);
    if (__any_sync(0xffffffffu, mx == 0.f && b < p.B)) {
      // a column of this warp's 32 states is all zero: tell an exact zero from products
      // that underflowed (the emissions are gathered again into cv)
      if constexpr (kStageE) {
        es_run(Es, row, col0, cv);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          cv[c] = c < nvalid ? p.Et[static_cast<long long>(tok_s[col0 + c]) * p.H + k] : 0.f;
      }
      mark_underflow(e, underflow_mask(e, cv, v, c_s, col0, nvalid));
      mx = warp_column_max(e);
    }
    if (b < p.B) atomic_max_nonneg(&p.umax_cur[b], mx);
  }

  // Split-K form of apply: u_t goes to the staged tiles (bf16) or straight to global memory.
  static constexpr int kOutBytes = kStageOut ? kNodeTileBytes + kBatchTileBytes : kEpiWarps * 4096;
  static constexpr int kSplitStageBytes = kOutBytes + (kEsSplit ? kEsHiBytes : 0);
  static_assert(kSplitStageBytes % 16 == 0, "16-byte staged rows");
  // the batch-major tile is written only in apply_staged: the exchange's scratch until then
  static constexpr int kSplitScratchOffset = kStageOut ? kNodeTileBytes : 0;
  static_assert(kSplitScratchOffset % 16 == 0, "16-byte scratch rows");
  __device__ static float* es_hi(uint8_t* stage) { return reinterpret_cast<float*>(stage + kOutBytes); }
  __device__ static void after_mma(const Params& p, int, int m0, int n0, int et, uint8_t* smem, uint8_t* stage) {
    if constexpr (kEsSplit)
      stage_emissions_async<kChainBN - kEsLoCols, kEsLoCols>(p.Et, p.H, p.B, m0, n0 + kEsLoCols,
                                                             reinterpret_cast<const int*>(smem) + kEsLoCols,
                                                             es_hi(stage), et);
  }
  __device__ static void apply_staged(const Params& p, int, int m0, int n0, int row, int col0,
                                      float (&v)[32], uint8_t* smem, uint8_t* stage) {
    static_assert(P != kTF32x3 && kStageE, "split-K chain tiles in bf16 or TF32");
    const float* c_s = reinterpret_cast<const float*>(smem) + kChainBN;
    const float* Es = reinterpret_cast<const float*>(smem) + 2 * kChainBN;
    const int k = m0 + row;
    const int nvalid = k < p.H ? min(32, p.B - (n0 + col0)) : 0;
    float e[32], cv[32];
    if (col0 < kEsLo)
      es_run<kEsPitch>(Es, row, col0, e);
    else
      es_run<kEsLoCols>(es_hi(stage), row, col0 - kEsLoCols, e);
    cs_run(c_s, col0, cv);
    // u = e (D c) into e; v keeps D for the rare check below
#pragma unroll
    for (int c = 0; c < 32; ++c) e[c] = c < nvalid ? e[c] * (v[c] * cv[c]) : 0.f;
    if constexpr (kStageOut) {
      if (p.ubm) stage_batch_col(stage, row, col0, e);
    } else if (p.ubm) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c < nvalid)
          store_operand<P>(p.ubm, static_cast<size_t>((n0 + col0 + c) * p.ubm_ld + k), p.ubm_lo, e[c]);
    }
    if (p.U0) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c < nvalid) p.U0[static_cast<long long>(n0 + col0 + c) * p.H + k] = e[c];
    }
    if constexpr (kStageOut) {
      if (p.un) stage_node_run(stage, row, col0, e);
    } else if (p.un && nvalid > 0) {
      store_operand_run<P>(p.un, static_cast<size_t>(k * p.un_ld + static_cast<long long>(p.t - 1) * p.B + n0 + col0),
                           p.un_lo, e, nvalid);
    }
    const int b = n0 + col0 + (threadIdx.x & 31);
    float mx = warp_column_max(e);
    if (__any_sync(0xffffffffu, mx == 0.f && b < p.B)) {  // as in apply
      if (col0 < kEsLo)
        es_run<kEsPitch>(Es, row, col0, cv);
      else
        es_run<kEsLoCols>(es_hi(stage), row, col0 - kEsLoCols, cv);
      mark_underflow(e, underflow_mask(e, cv, v, c_s, col0, nvalid));
      mx = warp_column_max(e);
    }
    if (b < p.B) atomic_max_nonneg(&p.umax_cur[b], mx);
  }
  __device__ static void store_staged(const Params& p, int, int m0, int n0, int et, uint8_t* stage) {
    if constexpr (!kStageOut) return;
    const int nr = min(kBM, p.H - m0), nc = min(W, p.B - n0);
    if (p.ubm)
      stage_tile_store_bf16(stage + kNodeTileBytes, kBatchPitch,
                            static_cast<__nv_bfloat16*>(p.ubm) + static_cast<long long>(n0) * p.ubm_ld + m0,
                            p.ubm_ld, nc, nr, et);
    if (p.un)
      stage_tile_store_bf16(stage, kNodePitch,
                            static_cast<__nv_bfloat16*>(p.un) + static_cast<long long>(m0) * p.un_ld +
                                static_cast<long long>(p.t - 1) * p.B + n0,
                            p.un_ld, nr, nc, et);
  }

  __device__ static void finish(const Params&, int, int, int, int, uint8_t*) {}
};

// ------------------------------------------------------------------- root
// ll[b] = log sum_k pi[k] u_0[k,b] - sum_t log c_{t,b};  r[b] = 1 / sum_k pi u_0.
// A sample whose column maximum fell into (0, kRangeFloor) at some position left the
// range the per-layer shift keeps exact: its LL is NaN, it passes no flow (r = 0) and the
// device status word records kErrRange. One warp per sample (16-byte loads when H % 4 == 0
// and the rows are aligned): each run of four products is summed in float and the runs in
// double (one FP64 add per four values: this GPU's FP64 pipe is narrow).
__global__ void __launch_bounds__(128) k_hmm_root(int H, int B, int T, const float* __restrict__ pi,
                                                  const float* __restrict__ U0, const double* __restrict__ logc,
                                                  const float* __restrict__ umax, double* __restrict__ ll,
                                                  float* __restrict__ rroot, unsigned* status) {
  const int b = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (b >= B) return;
  const int lane = threadIdx.x & 31;
  const float* u = U0 + static_cast<long long>(b) * H;
  double s = 0.0;
  if ((H & 3) == 0 && ((reinterpret_cast<uintptr_t>(u) | reinterpret_cast<uintptr_t>(pi)) & 15) == 0) {
    const float4* u4 = reinterpret_cast<const float4*>(u);
    const float4* p4 = reinterpret_cast<const float4*>(pi);
    for (int q = lane; q < H / 4; q += 32) {
      const float4 x = u4[q], y = p4[q];
      s += static_cast<double>(fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, x.w * y.w))));
    }
  } else {
    for (int k = lane; k < H; k += 32) s += static_cast<double>(pi[k]) * u[k];
  }
  double off = 0.0;
  bool out_of_range = false;
  for (int t = lane; t < T; t += 32) {
    off += logc[static_cast<long long>(t) * B + b];
    const float m = umax[static_cast<long long>(t) * B + b];
    out_of_range |= m > 0.f && m < kRangeFloor;
  }
  for (int o = 16; o; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    off += __shfl_xor_sync(0xffffffffu, off, o);
  }
  out_of_range = __any_sync(0xffffffffu, out_of_range);
  if (lane != 0) return;
  const bool zero = !(s > 0.0) || !(off < INFINITY);
  if (out_of_range) {
    ll[b] = NAN;
    rroot[b] = 0.f;
    if (status) atomicOr(status, kErrRange);
  } else {
    ll[b] = zero ? -INFINITY : log(s) - off;
    rroot[b] = zero ? 0.f : static_cast<float>(1.0 / s);
  }
}

// Root flows: f_0 = pi u_0 r (stored batch-major for dE), w_0 = pi r E[., x_0] c_0; dpi.
template <int P>
__global__ void k_hmm_root_flows(int H, int B, int T, const int* __restrict__ tokens,
                                 const float* __restrict__ pi, const float* __restrict__ U0,
                                 const float* __restrict__ Et, const float* __restrict__ cf,
                                 const float* __restrict__ rroot, void* wbm, long long wbm_ld,
                                 size_t wbm_lo, void* wn, long long wn_ld, size_t wn_lo,
                                 float* fbm, float* dpi) {
  __shared__ float tile[32][33];
  __shared__ float fsum[8][32];
  const int k0 = blockIdx.x * 32, b0 = blockIdx.y * 32;
  const int k = k0 + threadIdx.x;
  const float pk = k < H ? pi[k] : 0.f;
  float facc = 0.f;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int b = b0 + i;
    float w = 0.f;
    if (b < B && k < H) {
      const int tok = tokens[static_cast<long long>(b) * T];
      const float r = rroot[b];
      const float f = pk * U0[static_cast<long long>(b) * H + k] * r;
      w = pk * r * Et[static_cast<long long>(tok) * H + k] * cf[b];
      facc += f;
      if (fbm) fbm[static_cast<long long>(b) * H + k] = f;
      if (wbm) store_operand<P>(wbm, static_cast<size_t>(b * wbm_ld + k), wbm_lo, w);
    }
    tile[i][threadIdx.x] = w;
  }
  fsum[threadIdx.y][threadIdx.x] = facc;
  __syncthreads();
  if (dpi && threadIdx.y == 0 && k < H) {
    float s = 0.f;
    for (int y = 0; y < 8; ++y) s += fsum[y][threadIdx.x];
    atomicAdd(&dpi[k], s);
  }
  if (!wn) return;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int kk = k0 + i, b = b0 + threadIdx.x;
    if (kk < H && b < B) store_operand<P>(wn, static_cast<size_t>(kk * wn_ld + b), wn_lo, tile[threadIdx.x][i]);
  }
}

// ---------------------------------------------------------- backward epilogue
struct HmmBwdParams {
    int H, B, T, t;
    const int* tokens;
    const float* Et;
    const float* cf;
    const void* un;          // u_{t+1} node-major at column t B
    long long un_ld;
    size_t un_lo;
    float* fbm;              // flows f_{t+1} batch-major [B][H] for dE, or NULL
    void* wbm;               // w_{t+1} batch-major for the next step (NULL at the end)
    long long wbm_ld;
    size_t wbm_lo;
    void* wn;                // w_{t+1} node-major at column (t+1) B for dA (NULL if unused)
    long long wn_ld;
    size_t wn_lo;
};

// W as in EpiHmmFwd.
template <int P, int W = kChainBN>
struct EpiHmmBwd : EpiNoHooks {
  using Params = HmmBwdParams;
  static constexpr int kEpiWarps = P == kTF32x3 ? 16 : 8;  // as EpiHmmFwd
  static constexpr int kSliceTF32 = 0;  // as EpiHmmFwd
  static constexpr int kSlice3x = 4;  // as EpiHmmFwd
  static constexpr bool kStageE = P != kTF32x3;
  static constexpr bool kEsSplit = P != kTF32x3 && W == kChainBN;  // see kEsLoCols
  static constexpr bool kStageOut = P == kBF16;                    // as EpiHmmFwd
  static constexpr int kEsLo = kEsSplit ? kEsLoCols : W;
  static constexpr int kEsPitch = kEsSplit ? kEsLoCols : kChainBN;
  static constexpr int kSmemBytes = kChainBN * 8 + (kStageE ? kEsPitch * kBM * 4 : 0);

  __device__ static void prepare(const Params& p, int, int m0, int n0, int et, uint8_t* smem) {
    int* tok_s = reinterpret_cast<int*>(smem);
    float* c_s = reinterpret_cast<float*>(smem) + kChainBN;
    for (int c = et; c < W; c += kEpiThreads) {
      const int b = n0 + c;
      tok_s[c] = b < p.B ? p.tokens[static_cast<long long>(b) * p.T + p.t + 1] : 0;
      c_s[c] = b < p.B ? p.cf[static_cast<long long>(p.t + 1) * p.B + b] : 0.f;
    }
    if constexpr (kStageE) {
      if (p.wbm) {
        epilogue_bar_sync();
        stage_emissions<kEsLo, kEsPitch>(p.Et, p.H, p.B, m0, n0, tok_s,
                                         reinterpret_cast<float*>(smem) + 2 * kChainBN, et);
      }
    }
  }

  // Thread = state j, registers = 32 consecutive samples; the u_{t+1} run is loaded
  // before the first atomic or store.
  __device__ static void apply(const Params& p, int, int m0, int n0, int row, int col0,
                               float (&v)[32], uint8_t* smem, float*) {
    const int* tok_s = reinterpret_cast<const int*>(smem);
    const float* c_s = reinterpret_cast<const float*>(smem) + kChainBN;
    const float* Es = reinterpret_cast<const float*>(smem) + 2 * kChainBN;
    const int j = m0 + row;
    if (j >= p.H) return;
    const int nvalid = min(32, p.B - (n0 + col0));
    if (nvalid <= 0) return;
    float u[32], e[32];
    if (p.fbm)
      load_operand_run<P>(p.un, static_cast<size_t>(j * p.un_ld + static_cast<long long>(p.t) * p.B + n0 + col0),
                          p.un_lo, u, nvalid);
    static_assert(!kEsSplit, "the split emission block is read by apply_staged");
    if (p.wbm) {
      if constexpr (kStageE) {
        es_run(Es, row, col0, e);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) e[c] = c < nvalid ? p.Et[static_cast<long long>(tok_s[col0 + c]) * p.H + j] : 0.f;
      }
    }
    if (p.fbm) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c < nvalid) p.fbm[static_cast<long long>(n0 + col0 + c) * p.H + j] = u[c] * v[c];
    }
    if (!p.wbm) return;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float w = c < nvalid ? e[c] * c_s[col0 + c] * v[c] : 0.f;
      if (c < nvalid) store_operand<P>(p.wbm, static_cast<size_t>((n0 + col0 + c) * p.wbm_ld + j), p.wbm_lo, w);
      v[c] = w;
    }
    if (p.wn)
      store_operand_run<P>(p.wn, static_cast<size_t>(j * p.wn_ld + static_cast<long long>(p.t + 1) * p.B + n0 + col0),
                           p.wn_lo, v, nvalid);
  }

  // Split-K form of apply: in bf16, u_{t+1} is staged (coalesced, asynchronous: the copies
  // complete while the partial sums are exchanged) and w_{t+1} goes to the staged tiles, the
  // node-major one in place of u; TF32 reads and writes global memory from registers.
  static constexpr int kOutBytes = kStageOut ? kNodeTileBytes + kBatchTileBytes : kEpiWarps * 4096;
  static constexpr int kSplitStageBytes = kOutBytes + (kEsSplit ? kEsHiBytes : 0);
  static_assert(kSplitStageBytes % 16 == 0, "16-byte staged rows");
  // the batch-major tile is written only in apply_staged: the exchange's scratch until then
  static constexpr int kSplitScratchOffset = kStageOut ? kNodeTileBytes : 0;
  static_assert(kSplitScratchOffset % 16 == 0, "16-byte scratch rows");
  __device__ static float* es_hi(uint8_t* stage) { return reinterpret_cast<float*>(stage + kOutBytes); }
  __device__ static void after_mma(const Params& p, int, int m0, int n0, int et, uint8_t* smem, uint8_t* stage) {
    if constexpr (kEsSplit)
      if (p.wbm)
        stage_emissions_async<kChainBN - kEsLoCols, kEsLoCols>(p.Et, p.H, p.B, m0, n0 + kEsLoCols,
                                                               reinterpret_cast<const int*>(smem) + kEsLoCols,
                                                               es_hi(stage), et);
    if (kStageOut && p.fbm)
      stage_tile_load_bf16_async(stage, kNodePitch,
                           static_cast<const __nv_bfloat16*>(p.un) + static_cast<long long>(m0) * p.un_ld +
                               static_cast<long long>(p.t) * p.B + n0,
                           p.un_ld, min(kBM, p.H - m0), min(W, p.B - n0), et);
  }
  __device__ static void apply_staged(const Params& p, int, int m0, int n0, int row, int col0,
                                      float (&v)[32], uint8_t* smem, uint8_t* stage) {
    static_assert(P != kTF32x3 && kStageE, "split-K chain tiles in bf16 or TF32");
    const float* c_s = reinterpret_cast<const float*>(smem) + kChainBN;
    const float* Es = reinterpret_cast<const float*>(smem) + 2 * kChainBN;
    const int j = m0 + row;
    const int nvalid = j < p.H ? min(32, p.B - (n0 + col0)) : 0;
    if (p.fbm) {
      float u[32];
      if constexpr (kStageOut) {
        const uint4* nt = reinterpret_cast<const uint4*>(stage + row * kNodePitch + col0 * 2);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w = nt[q];
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            u[8 * q + 2 * r] = __uint_as_float(ww[r] << 16);
            u[8 * q + 2 * r + 1] = __uint_as_float(ww[r] & 0xFFFF0000u);
          }
        }
      } else if (nvalid > 0) {
        load_operand_run<P>(p.un, static_cast<size_t>(j * p.un_ld + static_cast<long long>(p.t) * p.B + n0 + col0),
                            p.un_lo, u, nvalid);
      }
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c < nvalid) p.fbm[static_cast<long long>(n0 + col0 + c) * p.H + j] = u[c] * v[c];
    }
    if (!p.wbm) return;
    float e[32], cv[32];
    if (col0 < kEsLo)
      es_run<kEsPitch>(Es, row, col0, e);
    else
      es_run<kEsLoCols>(es_hi(stage), row, col0 - kEsLoCols, e);
    cs_run(c_s, col0, cv);
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] = c < nvalid ? e[c] * cv[c] * v[c] : 0.f;
    if constexpr (kStageOut) {
      stage_batch_col(stage, row, col0, v);
      if (p.wn) stage_node_run(stage, row, col0, v);
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c < nvalid) store_operand<P>(p.wbm, static_cast<size_t>((n0 + col0 + c) * p.wbm_ld + j), p.wbm_lo, v[c]);
      if (p.wn && nvalid > 0)
        store_operand_run<P>(p.wn,
                             static_cast<size_t>(j * p.wn_ld + static_cast<long long>(p.t + 1) * p.B + n0 + col0),
                             p.wn_lo, v, nvalid);
    }
  }
  __device__ static void store_staged(const Params& p, int, int m0, int n0, int et, uint8_t* stage) {
    if constexpr (!kStageOut) return;
    if (!p.wbm) return;
    const int nr = min(kBM, p.H - m0), nc = min(W, p.B - n0);
    stage_tile_store_bf16(stage + kNodeTileBytes, kBatchPitch,
                          static_cast<__nv_bfloat16*>(p.wbm) + static_cast<long long>(n0) * p.wbm_ld + m0,
                          p.wbm_ld, nc, nr, et);
    if (p.wn)
      stage_tile_store_bf16(stage, kNodePitch,
                            static_cast<__nv_bfloat16*>(p.wn) + static_cast<long long>(m0) * p.wn_ld +
                                static_cast<long long>(p.t + 1) * p.B + n0,
                            p.wn_ld, nr, nc, et);
  }
};

// ------------------------------------------------------- dA over K ranges
// The stacked dA contraction has K = (T-1) B but only cdiv(H,128) x cdiv(H,BN) output
// tiles: for a small H too few CTAs for the GPU. It then runs over S consecutive K ranges
// (blockIdx.z; the operands' tensor maps take the ranges as groups) into S float32
// partial products, which k_dA_reduce adds in range order and scales by A.
constexpr int kParamSplitMax = 4;

int param_split(int H, int T, int B, pc_precision_t prec) {
  if (T < 2) return 1;
  const long long K = static_cast<long long>(T - 1) * B;
  const int kb = 128 / operand_elem_bytes(prec);  // K elements per ring block
  const long long tiles = static_cast<long long>(cdiv(H, kBM)) * cdiv(H, prec == PC_PREC_FP32 ? 128 : 256);
  for (int S = kParamSplitMax; S >= 2; S /= 2)
    if (tiles * S <= num_sms() && K % (static_cast<long long>(S) * kb) == 0 && K / S >= 8ll * kb) return S;
  return 1;
}

// dA[i] = (accumulate ? dA[i] : 0) + A[i] (part[0][i] + part[1][i] + ...), float4 runs
// where n is a multiple of 4 and the caller's A and dA are 16-byte aligned.
__global__ void k_dA_reduce(int S, long long n, const float* __restrict__ part, const float* __restrict__ A,
                            float* __restrict__ dA, int accumulate) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const bool vec = (n & 3) == 0 && ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(dA)) & 15) == 0;
  if (vec) {
    const long long n4 = n >> 2;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
      float4 sum = reinterpret_cast<const float4*>(part)[i];
      for (int g = 1; g < S; ++g) {
        const float4 x = reinterpret_cast<const float4*>(part + g * n)[i];
        sum.x += x.x;
        sum.y += x.y;
        sum.z += x.z;
        sum.w += x.w;
      }
      const float4 a = reinterpret_cast<const float4*>(A)[i];
      float4 r = make_float4(a.x * sum.x, a.y * sum.y, a.z * sum.z, a.w * sum.w);
      if (accumulate) {
        const float4 d = reinterpret_cast<const float4*>(dA)[i];
        r = make_float4(d.x + r.x, d.y + r.y, d.z + r.z, d.w + r.w);
      }
      reinterpret_cast<float4*>(dA)[i] = r;
    }
  } else {
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
      float sum = part[i];
      for (int g = 1; g < S; ++g) sum += part[g * n + i];
      dA[i] = (accumulate ? dA[i] : 0.f) + A[i] * sum;
    }
  }
}

// -------------------------------------------------------------- workspace
struct HmmWs {
  Operand Aop, Atop, ubm[2], wbm[2], un, wn;
  float *Et, *rs, *emax, *emax_rs, *U0, *umax, *cf, *rroot, *dEt, *fbm;
  int *tok_count, *tok_offset, *tok_order;
  double* logc;
  float* dA_part;  // param_split > 1: the K ranges' partial products [S][H][H]
};

size_t carve_hmm(void* base, pc_precision_t p, int H, int T, int V, int B, bool flows, bool chain,
                 bool want_dE, HmmWs* w) {
  Carver c(base);
  *w = HmmWs{};
  w->Aop = c.operand(p, 1, H, H);
  w->ubm[0] = c.operand(p, 1, B, H);
  w->ubm[1] = c.operand(p, 1, B, H);
  w->Et = static_cast<float*>(c.take(size_t(V) * H * 4));
  w->rs = static_cast<float*>(c.take(size_t(H) * 4));
  w->emax = static_cast<float*>(c.take(size_t(V) * 8));  // emax, then emax_rs (cleared together)
  w->emax_rs = w->emax + V;
  w->U0 = static_cast<float*>(c.take(size_t(B) * H * 4));
  w->umax = static_cast<float*>(c.take(size_t(T) * B * 4));
  w->cf = static_cast<float*>(c.take(size_t(T) * B * 4));
  w->logc = static_cast<double*>(c.take(size_t(T) * B * 8));
  w->rroot = static_cast<float*>(c.take(size_t(B) * 4));
  if (flows && chain) {
    w->Atop = c.operand(p, 1, H, H);
    w->wbm[0] = c.operand(p, 1, B, H);
    w->wbm[1] = c.operand(p, 1, B, H);
    w->un = c.operand(p, 1, H, static_cast<long long>(T - 1) * B);
    w->wn = c.operand(p, 1, H, static_cast<long long>(T - 1) * B);
    const int S = param_split(H, T, B, p);
    if (S > 1) w->dA_part = static_cast<float*>(c.take(size_t(S) * H * H * 4));
  }
  if (flows && want_dE) {
    w->dEt = static_cast<float*>(c.take(size_t(V) * H * 4));
    w->fbm = static_cast<float*>(c.take(size_t(T) * B * H * 4));
    w->tok_count = static_cast<int*>(c.take(size_t(V + 1) * 4));
    w->tok_offset = static_cast<int*>(c.take(size_t(V + 1) * 4));
    w->tok_order = static_cast<int*>(c.take(size_t(T) * B * 4));
  }
  return c.used;
}

size_t hmm_ws_bytes(pc_precision_t p, int H, int T, int V, int B) {
  HmmWs w;
  return carve_hmm(nullptr, p, H, T, V, B, true, T >= 2, true, &w) + 256;
}

pc_status_t check_hmm_shape(int H, int T, int V, int B) {
  PC_CHECK(H >= 1 && T >= 1 && V >= 1 && B >= 1, PC_ERR_SHAPE,
           "H, T, V, B must be >= 1 (got %d, %d, %d, %d)", H, T, V, B);
  PC_CHECK(H <= 16384 && T <= 4096 && V <= 65536 && B <= 65536, PC_ERR_SHAPE,
           "sizes out of range (H <= 16384, T <= 4096, V <= 65536, B <= 65536)");
  PC_CHECK(static_cast<long long>(T) * B < (1ll << 31), PC_ERR_SHAPE, "T * B must be < 2^31");
  return PC_OK;
}

// The stacked dA contraction (one contraction over K = (T - 1) B, not a chain): in 3xTF32
// it accumulates slices of one ring slot (4 k-steps, corrected as every 3xTF32 slice), at a
// quarter of the one-k-step slices' round trips.
struct EpiThetaScaleStacked : EpiThetaScale {
  static constexpr int kSlice3x = 4;
};
struct EpiStoreF32Stacked : EpiStoreF32 {
  static constexpr int kSlice3x = 4;
};

template <int P>
pc_status_t hmm_run(int H, int T, int V, int B, const int32_t* tokens, const float* pi, const float* A,
                    const float* E, double* ll, float* dpi, float* dA, float* dE, int accumulate,
                    pc_precision_t prec, void* ws, cudaStream_t s) {
  constexpr int kParamBN = (P == kTF32x3) ? 128 : 256;  // 3xTF32 (sliced) holds BN sums per thread
  const bool flows = dpi || dA || dE;
  const bool chain = flows && (dA || dE) && T >= 2;
  HmmWs w;
  void* base = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
  carve_hmm(base, prec, H, T, V, B, flows, T >= 2, dE != nullptr, &w);
  pc_status_t st;

  PC_CUDA(cudaMemsetAsync(w.umax, 0, size_t(T) * B * 4, s));
  // algorithmic bytes of the memory-bound launches (profiler records, PC_KIND_HMM_MEM)
  const long long eb = operand_elem_bytes(prec) * operand_parts(prec);  // stored bytes per operand value
  const long long HH = static_cast<long long>(H) * H, BH = static_cast<long long>(B) * H;
  const long long TB = static_cast<long long>(T) * B, VH = static_cast<long long>(V) * H;
  // Work off the forward chain's path (the token buckets for dE, the transposed A operand
  // of the backward chain) runs on a side stream, beside the forward contractions, which
  // leave some SMs free; it joins the caller's stream before the backward chain.
  SideStream side;
  const bool use_side = w.dEt || chain;
  if (use_side && (st = side.fork(s)) != PC_OK) return st;
  const cudaStream_t sa = use_side ? side.s : s;
  if (w.dEt) {
    // token buckets of every (position, sample): dE is then a per-token gather-sum
    PC_CUDA(cudaMemsetAsync(w.tok_count, 0, size_t(V + 1) * 4, sa));
    {
      ProfileScope ps(sa, PC_KIND_HMM_MEM, TB * 4 + (V + 1) * 4ll);
      k_token_hist<<<cdiv(static_cast<long long>(T) * B, 256), 256, 0, sa>>>(tokens, T * B, V, w.tok_count);
      PC_LAUNCH_CHECK();
    }
    {
      ProfileScope ps(sa, PC_KIND_HMM_MEM, (V + 1) * 8ll);
      k_exclusive_scan<<<1, 1024, 0, sa>>>(w.tok_count, V, w.tok_offset);
      PC_LAUNCH_CHECK();
    }
    {
      ProfileScope ps(sa, PC_KIND_HMM_MEM, TB * 8 + (V + 1) * 4ll);
      k_token_bucket<<<cdiv(V, kBucketSpan), 256, 0, sa>>>(tokens, T, B, V, w.tok_offset, w.tok_order);
      PC_LAUNCH_CHECK();
    }
  }
  if (chain) {
    ProfileScope ps(sa, PC_KIND_HMM_MEM, HH * (4 + eb));
    if ((st = transpose_to_operand<P>(A, H, 0, 1, H, H, w.Atop, sa)) != PC_OK) return st;
  }
  if (dpi && !accumulate) PC_CUDA(cudaMemsetAsync(dpi, 0, size_t(H) * 4, s));
  if (dA && !accumulate && T < 2) PC_CUDA(cudaMemsetAsync(dA, 0, size_t(H) * H * 4, s));

  // set-up: row sums of A with its operand copy, E transposed with the emission bounds
  const bool fused_a = T >= 2 && (H & 3) == 0 && aligned16(A);
  if (fused_a) {
    ProfileScope ps(s, PC_KIND_HMM_MEM, HH * (4 + eb) + H * 4ll);
    k_transition_operand<P><<<H, 256, 0, s>>>(A, H, w.Aop.ptr, w.Aop.ld, w.Aop.lo_elems, w.rs);
    PC_LAUNCH_CHECK();
  } else {
    {
      ProfileScope ps(s, PC_KIND_HMM_MEM, HH * 4 + H * 4ll);
      k_rowsum<<<cdiv(H, 8), 256, 0, s>>>(A, H, w.rs);
      PC_LAUNCH_CHECK();
    }
    if (T >= 2) {
      ProfileScope ps(s, PC_KIND_HMM_MEM, HH * (4 + eb));
      if ((st = rows_to_operand<P>(A, H, 0, 1, H, H, w.Aop, s)) != PC_OK) return st;
    }
  }
  PC_CUDA(cudaMemsetAsync(w.emax, 0, size_t(V) * 8, s));  // emax and emax_rs are adjacent
  {
    ProfileScope ps(s, PC_KIND_HMM_MEM, 2 * VH * 4 + H * 4ll + V * 8ll);
    k_emission_transpose<<<dim3(cdiv(V, 64), cdiv(H, 64)), 256, 0, s>>>(E, H, V, w.rs, w.Et, w.emax, w.emax_rs);
    PC_LAUNCH_CHECK();
  }

  // leaf (position T-1)
  {
    const int t = T - 1;
    const bool has_next = T >= 2;
    const Operand& ub = w.ubm[t & 1];
    ProfileScope ps(s, PC_KIND_HMM_MEM,
                    B * 4ll + V * 4ll + BH * 4 + (has_next ? BH * eb : 0) + (chain ? BH * eb : 0) + (T == 1 ? BH * 4 : 0));
    k_hmm_leaf<P><<<dim3(cdiv(H, 32), cdiv(B, 32)), dim3(32, 8), 0, s>>>(
        H, B, T, tokens, w.Et, w.emax, has_next ? ub.ptr : nullptr, ub.ld, ub.lo_elems,
        chain ? w.un.ptr : nullptr, w.un.ld, w.un.lo_elems, static_cast<long long>(T - 2) * B,
        T == 1 ? w.U0 : nullptr, w.umax, w.cf, w.logc);
    PC_LAUNCH_CHECK();
  }

  // The bf16 chain contractions run as split-K pairs of 128 x 256 tiles (k_umma_gemm,
  // kSplit); each CTA's epilogue still finishes 128 x kChainBN. Where that gives fewer
  // than kNarrowBelow CTAs (a small H: short K loops, the fixed costs dominate), the
  // pairs take 128 x 128 (or 128 x 64) tiles instead: twice (four times) the CTAs, a half
  // (a quarter) of the exchange and epilogue per CTA.
  constexpr bool kSplitChain = P != kTF32x3;
  constexpr int kTileBN = kSplitChain ? 2 * kChainBN : kChainBN;
  constexpr long long kNarrowBelow = 96;
  // split-K tiles 128 x 256, else 128 x 128, else 128 x 64: the widest with enough CTAs
  int tile_bn = kTileBN;
  if (kSplitChain)
    while (tile_bn > 64 && 2ll * cdiv(H, kBM) * cdiv(B, tile_bn) < kNarrowBelow) tile_bn /= 2;
  const dim3 chain_grid((kSplitChain ? 2 : 1) * cdiv(H, kBM), cdiv(B, tile_bn), 1);

  // forward chain: S_t for t = T-2 .. 0
  if (T >= 2) {
    OperandMaps ma, mb[2];
    if ((st = encode_maps(&ma, w.Aop, prec, kBM)) != PC_OK) return st;
    for (int i = 0; i < 2; ++i)
      if ((st = encode_maps(&mb[i], w.ubm[i], prec, tile_bn)) != PC_OK) return st;
    const dim3 grid = chain_grid;
    const int nkb = num_k_blocks(H, prec);
    // the chain is one profiler record: events between its launches would break their overlap
    const int prof = profile_group_begin(s);
    for (int t = T - 2; t >= 0; --t) {
      typename EpiHmmFwd<P>::Params ep{};
      ep.H = H; ep.B = B; ep.T = T; ep.t = t;
      ep.tokens = tokens; ep.Et = w.Et; ep.emax_rs = w.emax_rs;
      ep.umax_prev = w.umax + static_cast<long long>(t + 1) * B;
      ep.umax_cur = w.umax + static_cast<long long>(t) * B;
      ep.cf = w.cf; ep.logc = w.logc;
      if (t >= 1) {
        ep.ubm = w.ubm[t & 1].ptr; ep.ubm_ld = w.ubm[t & 1].ld; ep.ubm_lo = w.ubm[t & 1].lo_elems;
        if (chain) { ep.un = w.un.ptr; ep.un_ld = w.un.ld; ep.un_lo = w.un.lo_elems; }
      } else {
        ep.U0 = w.U0;
      }
      const OperandMaps& b = mb[(t + 1) & 1];
      // a_early: the A operand was converted before k_hmm_leaf, the kernel that precedes
      // the first layer, so no kernel still running when a layer starts writes it.
      if constexpr (kSplitChain) {
        if (tile_bn == kChainBN / 2)
          st = launch_gemm<P, kChainBN / 2, EpiHmmFwd<P, kChainBN / 4>, true>(grid, ma.hi, ma.lo, b.hi, b.lo, nkb, ep,
                                                                              s, PC_KIND_HMM_FWD, 2ll * H * H * B,
                                                                              true);
        else if (tile_bn == kChainBN)
          st = launch_gemm<P, kChainBN, EpiHmmFwd<P, kChainBN / 2>, true>(grid, ma.hi, ma.lo, b.hi, b.lo, nkb, ep, s,
                                                                          PC_KIND_HMM_FWD, 2ll * H * H * B, true);
        else
          st = launch_gemm<P, kTileBN, EpiHmmFwd<P>, true>(grid, ma.hi, ma.lo, b.hi, b.lo, nkb, ep, s,
                                                            PC_KIND_HMM_FWD, 2ll * H * H * B, true);
      } else {
        st = launch_gemm<P, kTileBN, EpiHmmFwd<P>, false>(grid, ma.hi, ma.lo, b.hi, b.lo, nkb, ep, s,
                                                           PC_KIND_HMM_FWD, 2ll * H * H * B, true);
      }
      if (st != PC_OK) return st;
    }
    profile_group_end(prof, s, PC_KIND_HMM_FWD, 2ll * H * H * B * (T - 1), T - 1);
  }

  {
    ProfileScope ps(s, PC_KIND_HMM_MEM, BH * 4 + H * 4ll + TB * 8 + B * 12ll);
    k_hmm_root<<<cdiv(B, 4), 128, 0, s>>>(H, B, T, pi, w.U0, w.logc, w.umax, ll, w.rroot, device_status_word());
    PC_LAUNCH_CHECK();
  }
  if (use_side && (st = side.join(s)) != PC_OK) return st;
  if (!flows) return PC_OK;

  {
  ProfileScope ps(s, PC_KIND_HMM_MEM,
                  2 * BH * 4 + H * 4ll + (w.fbm ? BH * 4 : 0) + (chain ? BH * eb : 0) + (chain && dA ? BH * eb : 0));
  k_hmm_root_flows<P><<<dim3(cdiv(H, 32), cdiv(B, 32)), dim3(32, 8), 0, s>>>(
      H, B, T, tokens, pi, w.U0, w.Et, w.cf, w.rroot, chain ? w.wbm[0].ptr : nullptr, w.wbm[0].ld,
      w.wbm[0].lo_elems, (chain && dA) ? w.wn.ptr : nullptr, w.wn.ld, w.wn.lo_elems, w.fbm, dpi);
  PC_LAUNCH_CHECK();
  }

  if (chain) {
    OperandMaps ma, mb[2];
    if ((st = encode_maps(&ma, w.Atop, prec, kBM)) != PC_OK) return st;
    for (int i = 0; i < 2; ++i)
      if ((st = encode_maps(&mb[i], w.wbm[i], prec, tile_bn)) != PC_OK) return st;
    const dim3 grid = chain_grid;
    const int nkb = num_k_blocks(H, prec);
    const int prof = profile_group_begin(s);
    for (int t = 0; t <= T - 2; ++t) {
      typename EpiHmmBwd<P>::Params ep{};
      ep.H = H; ep.B = B; ep.T = T; ep.t = t;
      ep.tokens = tokens; ep.Et = w.Et; ep.cf = w.cf;
      ep.un = w.un.ptr; ep.un_ld = w.un.ld; ep.un_lo = w.un.lo_elems;
      ep.fbm = w.fbm ? w.fbm + static_cast<long long>(t + 1) * B * H : nullptr;
      if (t + 1 <= T - 2) {
        const Operand& nb = w.wbm[(t + 1) & 1];
        ep.wbm = nb.ptr; ep.wbm_ld = nb.ld; ep.wbm_lo = nb.lo_elems;
        if (dA) { ep.wn = w.wn.ptr; ep.wn_ld = w.wn.ld; ep.wn_lo = w.wn.lo_elems; }
      }
      const OperandMaps& b = mb[t & 1];
      // a_early: the transposed A operand was converted before the forward chain
      if constexpr (kSplitChain) {
        if (tile_bn == kChainBN / 2)
          st = launch_gemm<P, kChainBN / 2, EpiHmmBwd<P, kChainBN / 4>, true>(grid, ma.hi, ma.lo, b.hi, b.lo, nkb, ep,
                                                                              s, PC_KIND_HMM_ELEM, 2ll * H * H * B,
                                                                              true);
        else if (tile_bn == kChainBN)
          st = launch_gemm<P, kChainBN, EpiHmmBwd<P, kChainBN / 2>, true>(grid, ma.hi, ma.lo, b.hi, b.lo, nkb, ep, s,
                                                                          PC_KIND_HMM_ELEM, 2ll * H * H * B, true);
        else
          st = launch_gemm<P, kTileBN, EpiHmmBwd<P>, true>(grid, ma.hi, ma.lo, b.hi, b.lo, nkb, ep, s,
                                                            PC_KIND_HMM_ELEM, 2ll * H * H * B, true);
      } else {
        st = launch_gemm<P, kTileBN, EpiHmmBwd<P>, false>(grid, ma.hi, ma.lo, b.hi, b.lo, nkb, ep, s,
                                                           PC_KIND_HMM_ELEM, 2ll * H * H * B, true);
      }
      if (st != PC_OK) return st;
    }
    profile_group_end(prof, s, PC_KIND_HMM_ELEM, 2ll * H * H * B * (T - 1), T - 1);
    // dE's gather reads the flows of every position: it runs on the side stream beside
    // the stacked dA contraction (which is bound by the tensor cores)
    if (dE) {
      if ((st = side.fork(s)) != PC_OK) return st;
      {
        ProfileScope ps(side.s, PC_KIND_HMM_MEM, TB * H * 4 + TB * 4 + VH * 4);
        k_dE_gather<<<dim3(V, cdiv(H, 256)), 256, 0, side.s>>>(w.fbm, H, w.tok_offset, w.tok_order, w.dEt);
        PC_LAUNCH_CHECK();
      }
      {
        ProfileScope ps(side.s, PC_KIND_HMM_MEM, (accumulate ? 3 : 2) * VH * 4);
        if ((st = transpose_f32(w.dEt, H, 0, 1, V, H, dE, V, accumulate, side.s)) != PC_OK) return st;
      }
    }
    if (dA) {
      OperandMaps pa, pb;
      if ((st = encode_maps(&pa, w.wn, prec, kBM)) != PC_OK) return st;
      if ((st = encode_maps(&pb, w.un, prec, kParamBN)) != PC_OK) return st;
      const int S = param_split(H, T, B, prec);
      const long long K = static_cast<long long>(T - 1) * B;
      if (S > 1) {
        // K-range views of the two operands: S groups of K/S columns, K/S elements apart
        OperandMaps va, vb;
        Operand oa = w.wn, ob = w.un;
        oa.cols = ob.cols = K / S;
        oa.groups = ob.groups = S;
        for (int part = 0; part < (prec == PC_PREC_FP32 ? 2 : 1); ++part) {
          if ((st = encode_operand_map(part ? &va.lo : &va.hi, oa, prec, kBM, part, true, K / S)) != PC_OK) return st;
          if ((st = encode_operand_map(part ? &vb.lo : &vb.hi, ob, prec, kParamBN, part, true, K / S)) != PC_OK)
            return st;
        }
        if (prec != PC_PREC_FP32) {
          va.lo = va.hi;
          vb.lo = vb.hi;
        }
        EpiStoreF32::Params ep{w.dA_part, H, H, H, 0, nullptr, nullptr, static_cast<long long>(H) * H};
        if ((st = launch_gemm<P, kParamBN, EpiStoreF32Stacked>(dim3(cdiv(H, kBM), cdiv(H, kParamBN), S), va.hi,
                                                               va.lo, vb.hi, vb.lo, num_k_blocks(K / S, prec), ep, s,
                                                               PC_KIND_HMM_PARAM, 2ll * H * H * K)) != PC_OK)
          return st;
        const long long n = static_cast<long long>(H) * H;
        ProfileScope ps(s, PC_KIND_HMM_MEM, (S + 2 + (accumulate ? 1 : 0)) * n * 4);
        k_dA_reduce<<<static_cast<unsigned>(std::min<long long>(cdiv(n, 4 * 256), 4ll * num_sms())), 256, 0, s>>>(
            S, n, w.dA_part, A, dA, accumulate);
        PC_LAUNCH_CHECK();
      } else {
        EpiThetaScale::Params ep{dA, A, H, H, accumulate};
        bool persist = false;
        if constexpr (P != kTF32x3) {
          // bf16 / TF32: persistent tiles (each tile's theta and dA traffic under the next
          // tile's K loop); a last partial wave of at most half the SMs is split into K
          // halves added into dA (zeroed first), which halves its length: 512 tiles on
          // 152 SMs take 3.5 tile times instead of 4
          const int tm = static_cast<int>(cdiv(H, kBM)), tn = static_cast<int>(cdiv(H, kParamBN));
          const int tail = (tm * tn) % num_sms();
          const int split =
              (!accumulate && tail > 0 && 2 * tail <= num_sms() && num_k_blocks(K, prec) >= 2) ? tail : 0;
          if (split) {
            const long long row0 = static_cast<long long>((tm * tn - split) / tn) * kBM;
            PC_CUDA(cudaMemsetAsync(dA + row0 * H, 0, size_t(H - row0) * H * 4, s));
          }
          persist = true;
          st = launch_gemm_persist<P, kParamBN, EpiThetaScaleDirect>(tm, tn, 1, pa.hi, pa.lo, pb.hi, pb.lo,
                                                                     num_k_blocks(K, prec), ep, s, PC_KIND_HMM_PARAM,
                                                                     2ll * H * H * K, split);
        }
        if (!persist)
          st = launch_gemm<P, kParamBN, EpiThetaScaleStacked>(dim3(cdiv(H, kBM), cdiv(H, kParamBN), 1), pa.hi, pa.lo,
                                                              pb.hi, pb.lo, num_k_blocks(K, prec), ep, s,
                                                              PC_KIND_HMM_PARAM, 2ll * H * H * K);
        if (st != PC_OK) return st;
      }
    }
    if (dE && (st = side.join(s)) != PC_OK) return st;
  } else {
    if (dA && !accumulate && T >= 2) PC_CUDA(cudaMemsetAsync(dA, 0, size_t(H) * H * 4, s));
    if (dE) {
      {
        ProfileScope ps(s, PC_KIND_HMM_MEM, TB * H * 4 + TB * 4 + VH * 4);
        k_dE_gather<<<dim3(V, cdiv(H, 256)), 256, 0, s>>>(w.fbm, H, w.tok_offset, w.tok_order, w.dEt);
        PC_LAUNCH_CHECK();
      }
      ProfileScope ps(s, PC_KIND_HMM_MEM, (accumulate ? 3 : 2) * VH * 4);
      if ((st = transpose_f32(w.dEt, H, 0, 1, V, H, dE, V, accumulate, s)) != PC_OK) return st;
    }
  }
  return PC_OK;
}

}  // namespace
}  // namespace pc

extern "C" {

pc_status_t pc_hmm_workspace(int H, int T, int V, int B, pc_precision_t prec, size_t* bytes) {
  pc::clear_error();
  PC_CHECK(bytes != nullptr, PC_ERR_NULL, "bytes is NULL");
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_hmm_shape(H, T, V, B)) != PC_OK) return st;
  *bytes = pc::hmm_ws_bytes(prec, H, T, V, B);
  return PC_OK;
}

pc_status_t pc_hmm_fwd_bwd(int H, int T, int V, int B, const int32_t* tokens, const float* pi,
                           const float* A, const float* E, double* ll, float* dpi, float* dA,
                           float* dE, int accumulate, pc_precision_t prec, void* ws,
                           size_t ws_bytes, pc_stream_t stream) {
  pc::clear_error();
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_hmm_shape(H, T, V, B)) != PC_OK) return st;
  PC_CHECK(tokens && pi && A && E && ll, PC_ERR_NULL, "tokens, pi, A, E and ll must not be NULL");
  PC_CHECK(ws, PC_ERR_WORKSPACE, "workspace is NULL");
  const size_t need = pc::hmm_ws_bytes(prec, H, T, V, B);
  PC_CHECK(ws_bytes >= need, PC_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", ws_bytes, need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (prec) {
    case PC_PREC_AUTO:
      return pc::hmm_run<pc::kBF16>(H, T, V, B, tokens, pi, A, E, ll, dpi, dA, dE, accumulate, prec, ws, s);
    case PC_PREC_TF32:
      return pc::hmm_run<pc::kTF32>(H, T, V, B, tokens, pi, A, E, ll, dpi, dA, dE, accumulate, prec, ws, s);
    default:
      return pc::hmm_run<pc::kTF32x3>(H, T, V, B, tokens, pi, A, E, ll, dpi, dA, dE, accumulate, prec, ws, s);
  }
}

}  // extern "C"
