// Whole HCLT circuit, forward + backward, on the tensor-core contraction.
//
// The circuit (pyjuice PR #62, Results table: "HCLT, 1024 latents, 768 variables, 512
// categories"; Summary 2, second bullet: its layers run as batched GEMMs over evenly
// strided child groups) is a latent tree over the variables, variable 0 the root,
// parent[i] in [0, i):
//   n_v(z) = E_v[z, x_v] * prod_{c : parent[c] = v} s_c(z)      product layer
//   s_c(z) = sum_{z'} W_c[z, z'] n_c(z')                         sum layer per edge
//   LL     = log sum_z pi[z] n_0(z)                              root sum layer
//
// Schedule. Nodes are renumbered into "slots" ordered by height (leaves first, the root
// last), so the edges whose child has height L form one contiguous run of slots: one
// grouped contraction per level, the groups evenly strided in every operand.
//
// Values. Every node keeps u_v[b][z] = n_v(z) / max_z n_v(z) (so max_z u_v = 1) and its
// own log max as an integer exponent and a float32 log-mantissa. Each edge's sum layer
//   D_c[b][z] = sum_{z'} W_c[z,z'] u_c[b][z']
// is kept linear, and the product layer multiplies in float32 with an exact power-of-two
// exponent carried beside every running product, so a node with many children cannot
// underflow and no rounding but the multiplies' own round-to-nearest enters:
//   n'_v[b][z] = E_v[z, x_v] * prod_c D_c[b][z] = m_z 2^{e_z}   (m_z in [1/2, 1)),
//   u_v = n'_v / max_z n'_v,
//   LL_b = sum over all nodes v of log max_z n'_v[b]  +  log sum_z pi[z] u_0[b][z]
// (every node lies under the root), summed in double once per sample at the end.
// (Taking logs instead would round every y = log E + sum log D to float32 at |y| of
// several nats, an error of ~1e-7 per node that a 768-node tree accumulates.)
// Backward (root flow 1; product nodes pass their flow to every child):
//   f_0 = pi u_0 / sum_z pi u_0,     g_c = f_parent(c) / D_c      (the layer's scaled flow)
//   f_c[b][z'] = u_c[b][z'] sum_z W_c[z,z'] g_c[b][z]             element flows
//   dW_c[z,z'] = W_c[z,z'] sum_b g_c[b][z] u_c[b][z']            parameter flows
//   dE_v[z,k]  = sum_{b : x_{v,b} = k} f_v[b][z],  dpi = sum_b f_0.
// Per-node data is batch-major [slot][b][z] (z contiguous): the operands of the forward
// and element contractions are then plain row copies.
#include <algorithm>
#include <cmath>
#include <vector>

#include "pc_launch.cuh"

namespace pc {
namespace {

constexpr int kHcltBN = 128;

// ------------------------------------------------------------------ set-up

// m 2^e with m in [1/2, 1) and the exponent added to e, for p >= 0 (0 stays 0). Normal
// values by their bit fields; zero and subnormal products through frexpf.
__device__ __forceinline__ float renorm(float p, int& e) {
  const uint32_t bits = __float_as_uint(p);
  const uint32_t f = bits >> 23;
  if (f == 0u) {
    if (bits == 0u) return 0.f;
    int k;
    const float r = frexpf(p, &k);
    e += k;
    return r;
  }
  e += static_cast<int>(f) - 126;
  return __uint_as_float((bits & 0x007FFFFFu) | (126u << 23));
}

// 2^d for d <= 0 (0 below the subnormal range).
__device__ __forceinline__ float pow2_nonpos(int d) {
  if (d >= -126) return __uint_as_float(static_cast<uint32_t>(d + 127) << 23);
  return d >= -149 ? ldexpf(1.f, d) : 0.f;
}

// Four operand values at idx (idx % 4 == 0, rows 64-element aligned).
template <int P>
__device__ __forceinline__ void store_operand4(void* base, size_t idx, size_t lo, float4 v) {
  if constexpr (P == kBF16) {
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(base) + idx) =
        make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  } else {
    const float4 h = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx) = h;
    if constexpr (P == kTF32x3)
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx + lo) =
          make_float4(tf32_rna(v.x - h.x), tf32_rna(v.y - h.y), tf32_rna(v.z - h.z), tf32_rna(v.w - h.w));
  }
}

// The forward contraction's children operand: hi + lo in every mode (3xTF32's own pair,
// or EpiHcltFwd::kBLo's for bf16 and TF32).
template <int P>
__device__ __forceinline__ void store_child4(void* base, size_t idx, size_t lo, float4 v) {
  if constexpr (P == kTF32x3) {
    store_operand4<P>(base, idx, lo, v);
  } else if constexpr (P == kBF16) {
    const float4 h = make_float4(round_operand<P>(v.x), round_operand<P>(v.y), round_operand<P>(v.z),
                                 round_operand<P>(v.w));
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(base) + idx) =
        make_uint2(pack_bf16x2(h.x, h.y), pack_bf16x2(h.z, h.w));
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(base) + idx + lo) =
        make_uint2(pack_bf16x2(v.x - h.x, v.y - h.y), pack_bf16x2(v.z - h.z, v.w - h.w));
  } else {
    const float4 h = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx) = h;
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx + lo) =
        make_float4(tf32_rna(v.x - h.x), tf32_rna(v.y - h.y), tf32_rna(v.z - h.z), tf32_rna(v.w - h.w));
  }
}
template <int P>
__device__ __forceinline__ void store_child(void* base, size_t idx, size_t lo, float v) {
  if constexpr (P == kTF32x3) store_operand<P>(base, idx, lo, v);
  else store_operand_hilo<P>(base, idx, lo, v);
}

// Product layer of the nodes in slots [s0, s0 + gridDim.x), one block per (node, sample):
// n' = E_v[., x_v] * prod_children D as float32 mantissas in [1/2, 1) with int exponents,
// u = n' / max n' (float32 and operand copies), and the node's own log max n' as its
// exponent Ex and float32 log-mantissa Lm; for the root also sum_z pi u (rdot). Each
// thread takes runs of four latents: 16-byte loads and stores when H % 4 == 0 (kVec),
// element by element otherwise. No double-precision arithmetic: this GPU's FP64 pipe is
// narrow, and the log-likelihood's double sum is formed once per sample (k_hclt_ll).
template <bool kVec>
__device__ __forceinline__ float4 load_run4(const float* row, int q, int H) {
  if constexpr (kVec) return reinterpret_cast<const float4*>(row)[q];
  const int z = 4 * q;
  return make_float4(row[z], z + 1 < H ? row[z + 1] : 0.f, z + 2 < H ? row[z + 2] : 0.f, z + 3 < H ? row[z + 3] : 0.f);
}

template <int P, bool kVec>
__global__ void __launch_bounds__(256) k_hclt_product(
    int s0, int root_slot, int nvars, int H, int B, const int* __restrict__ data, const int* __restrict__ var_of_slot,
    const int* __restrict__ child_ptr, const int* __restrict__ child_slots, const float* __restrict__ Et,
    const float* __restrict__ D, int C, float* __restrict__ U32, long long u32_off, void* uop, long long uop_ld,
    size_t uop_lo,
    int* __restrict__ Ex, float* __restrict__ Lm, const float* __restrict__ pi, float* __restrict__ rdot) {
  extern __shared__ float4 mant4[];  // ceil(H/4) mantissa runs, then as many exponent runs
  const int H4 = (H + 3) / 4;
  int4* expo4 = reinterpret_cast<int4*>(mant4 + H4);
  __shared__ long long red[32];
  __shared__ float redf[32];
  constexpr long long kNone = -0x7fffffffffffffffLL - 1;  // key of a zero product
  const int s = s0 + blockIdx.x;
  const int b = blockIdx.y;
  const int v = var_of_slot[s];
  const int x = data[static_cast<long long>(b) * nvars + v];
  const bool xin = x >= 0 && x < C;  // a category outside [0, C) has emission 0
  const int c0 = child_ptr[s], c1 = child_ptr[s + 1];
  const float* er = Et + (static_cast<long long>(v) * C + (xin ? x : 0)) * H;
  // key = e * 2^32 + bits(m) orders the nonzero products m 2^e (m in [1/2, 1)) by value
  long long best = kNone;
  for (int q = threadIdx.x; q < H4; q += blockDim.x) {
    const float4 ev = xin ? load_run4<kVec>(er, q, H) : make_float4(0.f, 0.f, 0.f, 0.f);
    float m[4] = {ev.x, ev.y, ev.z, ev.w};
    int e[4] = {0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = renorm(m[k], e[k]);
    for (int c = c0; c < c1; ++c) {
      const float4 d = load_run4<kVec>(D + (static_cast<long long>(child_slots[c]) * B + b) * H, q, H);
      m[0] = renorm(m[0] * d.x, e[0]);
      m[1] = renorm(m[1] * d.y, e[1]);
      m[2] = renorm(m[2] * d.z, e[2]);
      m[3] = renorm(m[3] * d.w, e[3]);
    }
    mant4[q] = make_float4(m[0], m[1], m[2], m[3]);
    expo4[q] = make_int4(e[0], e[1], e[2], e[3]);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (m[k] > 0.f) best = max(best, static_cast<long long>(e[k]) * 4294967296LL + __float_as_uint(m[k]));
  }
  for (int o = 16; o; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x < 32) {
    long long mx = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : kNone;
    for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (threadIdx.x == 0) red[0] = mx;
  }
  __syncthreads();
  best = red[0];
  const bool live = best != kNone;
  const unsigned mbits = static_cast<unsigned>(best & 0xffffffffLL);
  const int emax = live ? static_cast<int>((best - static_cast<long long>(mbits)) / 4294967296LL) : 0;
  const float mmax = live ? __uint_as_float(mbits) : 1.f;
  const float rinv = 1.f / mmax;
  const long long row = static_cast<long long>(s) * B + b;
  float* u32 = U32 ? U32 + row * H - u32_off : nullptr;  // NULL: the bf16 operand parts carry u
  float dot = 0.f;
  for (int q = threadIdx.x; q < H4; q += blockDim.x) {
    const float4 m = mant4[q];
    const int4 e = expo4[q];
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
      u.x = m.x > 0.f ? (m.x * rinv) * pow2_nonpos(e.x - emax) : 0.f;
      u.y = m.y > 0.f ? (m.y * rinv) * pow2_nonpos(e.y - emax) : 0.f;
      u.z = m.z > 0.f ? (m.z * rinv) * pow2_nonpos(e.z - emax) : 0.f;
      u.w = m.w > 0.f ? (m.w * rinv) * pow2_nonpos(e.w - emax) : 0.f;
    }
    const int z = 4 * q;
    if constexpr (kVec) {
      if (u32) reinterpret_cast<float4*>(u32)[q] = u;
      if (uop) store_child4<P>(uop, static_cast<size_t>(row * uop_ld + z), uop_lo, u);
    } else {
      const float uu[4] = {u.x, u.y, u.z, u.w};
      for (int k = 0; k < 4 && z + k < H; ++k) {
        if (u32) u32[z + k] = uu[k];
        if (uop) store_child<P>(uop, static_cast<size_t>(row * uop_ld + z + k), uop_lo, uu[k]);
      }
    }
    if (s == root_slot) {
      const float4 pz = load_run4<kVec>(pi, q, H);  // zero beyond H, where u is zero too
      dot += (pz.x * u.x + pz.y * u.y) + (pz.z * u.z + pz.w * u.w);
    }
  }
  if (threadIdx.x == 0) {
    Ex[row] = live ? emax : 0;
    Lm[row] = live ? logf(mmax) : -INFINITY;
  }
  if (s != root_slot) return;
  for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  if ((threadIdx.x & 31) == 0) redf[threadIdx.x >> 5] = dot;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tt = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tt += redf[w];
    rdot[b] = tt;
  }
}

// The same product layer with one warp per (node, sample) for H <= 1024: every lane keeps
// its runs of four latents in registers (eight runs at most), the maximum is a warp
// reduction, and a lane's loads of one child row are independent, so they are all in
// flight together. Warp w of the launch takes node s0 + w / B, sample w % B.
constexpr int kWarpRuns = 8;  // runs of four latents per lane: H <= 4 * 32 * 8
// kLeaf: nodes without children below the root (height 0), where n' = E_v[., x_v] itself:
// its maximum is taken on the values and u = n' * (1 / max n'), the same bits as the
// exponent-tracked path gives while u is a normal float (a power-of-two scale of a
// product rounds the same way), with a third of its work per latent.
template <int P, bool kVec, bool kLeaf = false>
__global__ void __launch_bounds__(256) k_hclt_product_warp(
    int s0, int G, int root_slot, int nvars, int H, int B, const int* __restrict__ data,
    const int* __restrict__ var_of_slot, const int* __restrict__ child_ptr, const int* __restrict__ child_slots,
    const float* __restrict__ Et, const float* __restrict__ D, int C, float* __restrict__ U32, long long u32_off,
    void* uop, long long uop_ld, size_t uop_lo, int* __restrict__ Ex, float* __restrict__ Lm, const float* __restrict__ pi,
    float* __restrict__ rdot) {
  constexpr long long kNone = -0x7fffffffffffffffLL - 1;
  const long long wid = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (wid >= static_cast<long long>(G) * B) return;  // the whole warp leaves together
  const int lane = threadIdx.x & 31;
  const int s = s0 + static_cast<int>(wid / B);
  const int b = static_cast<int>(wid % B);
  const int v = var_of_slot[s];
  const int x = data[static_cast<long long>(b) * nvars + v];
  const bool xin = x >= 0 && x < C;
  const int c0 = child_ptr[s], c1 = child_ptr[s + 1];
  const float* er = Et + (static_cast<long long>(v) * C + (xin ? x : 0)) * H;
  const long long row = static_cast<long long>(s) * B + b;
  if constexpr (kLeaf) {
    float ev[kWarpRuns][4];
    float mx = 0.f;
#pragma unroll
    for (int r = 0; r < kWarpRuns; ++r) {
      const int q = lane + 32 * r;
      const float4 x4 = (xin && 4 * q < H) ? load_run4<kVec>(er, q, H) : make_float4(0.f, 0.f, 0.f, 0.f);
      ev[r][0] = x4.x;
      ev[r][1] = x4.y;
      ev[r][2] = x4.z;
      ev[r][3] = x4.w;
      mx = fmaxf(mx, fmaxf(fmaxf(x4.x, x4.y), fmaxf(x4.z, x4.w)));
    }
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const bool live = mx > 0.f;
    int emax = 0;
    const float mmax = live ? renorm(mx, emax) : 1.f;
    const float rinv = live ? 1.f / mx : 0.f;
    float* u32 = U32 ? U32 + row * H - u32_off : nullptr;
#pragma unroll
    for (int r = 0; r < kWarpRuns; ++r) {
      const int q = lane + 32 * r;
      const int z = 4 * q;
      if (z >= H) continue;
      float uu[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) uu[k] = ev[r][k] > 0.f ? ev[r][k] * rinv : 0.f;
      const float4 u = make_float4(uu[0], uu[1], uu[2], uu[3]);
      if constexpr (kVec) {
        if (u32) reinterpret_cast<float4*>(u32)[q] = u;
        store_child4<P>(uop, static_cast<size_t>(row * uop_ld + z), uop_lo, u);
      } else {
        for (int k = 0; k < 4 && z + k < H; ++k) {
          if (u32) u32[z + k] = uu[k];
          store_child<P>(uop, static_cast<size_t>(row * uop_ld + z + k), uop_lo, uu[k]);
        }
      }
    }
    if (lane == 0) {
      Ex[row] = live ? emax : 0;
      Lm[row] = live ? logf(mmax) : -INFINITY;
    }
    return;
  }
  float m[kWarpRuns][4];
  int e[kWarpRuns][4];
  float4 d[kWarpRuns];
#pragma unroll
  for (int r = 0; r < kWarpRuns; ++r) {
    const int q = lane + 32 * r;
    const float4 ev = (xin && 4 * q < H) ? load_run4<kVec>(er, q, H) : make_float4(0.f, 0.f, 0.f, 0.f);
    m[r][0] = ev.x;
    m[r][1] = ev.y;
    m[r][2] = ev.z;
    m[r][3] = ev.w;
  }
  auto load_child = [&](int c) {
    const float* drow = D + (static_cast<long long>(child_slots[c]) * B + b) * H;
#pragma unroll
    for (int r = 0; r < kWarpRuns; ++r) {
      const int q = lane + 32 * r;
      d[r] = 4 * q < H ? load_run4<kVec>(drow, q, H) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  // the first child's row goes out together with the emission row: one memory round
  // trip fewer per (node, sample)
  if (c0 < c1) load_child(c0);
#pragma unroll
  for (int r = 0; r < kWarpRuns; ++r)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      e[r][k] = 0;
      m[r][k] = renorm(m[r][k], e[r][k]);
    }
  for (int c = c0; c < c1; ++c) {
    if (c > c0) load_child(c);
#pragma unroll
    for (int r = 0; r < kWarpRuns; ++r) {
      m[r][0] = renorm(m[r][0] * d[r].x, e[r][0]);
      m[r][1] = renorm(m[r][1] * d[r].y, e[r][1]);
      m[r][2] = renorm(m[r][2] * d[r].z, e[r][2]);
      m[r][3] = renorm(m[r][3] * d[r].w, e[r][3]);
    }
  }
  long long best = kNone;
#pragma unroll
  for (int r = 0; r < kWarpRuns; ++r)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (m[r][k] > 0.f) best = max(best, static_cast<long long>(e[r][k]) * 4294967296LL + __float_as_uint(m[r][k]));
  for (int o = 16; o; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  const bool live = best != kNone;
  const unsigned mbits = static_cast<unsigned>(best & 0xffffffffLL);
  const int emax = live ? static_cast<int>((best - static_cast<long long>(mbits)) / 4294967296LL) : 0;
  const float mmax = live ? __uint_as_float(mbits) : 1.f;
  const float rinv = 1.f / mmax;
  float* u32 = U32 ? U32 + row * H - u32_off : nullptr;  // NULL: the bf16 operand parts carry u
  float dot = 0.f;
#pragma unroll
  for (int r = 0; r < kWarpRuns; ++r) {
    const int q = lane + 32 * r;
    const int z = 4 * q;
    if (z >= H) continue;
    float uu[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      uu[k] = (live && m[r][k] > 0.f) ? (m[r][k] * rinv) * pow2_nonpos(e[r][k] - emax) : 0.f;
    const float4 u = make_float4(uu[0], uu[1], uu[2], uu[3]);
    if constexpr (kVec) {
      if (u32) reinterpret_cast<float4*>(u32)[q] = u;
      if (uop) store_child4<P>(uop, static_cast<size_t>(row * uop_ld + z), uop_lo, u);
    } else {
      for (int k = 0; k < 4 && z + k < H; ++k) {
        if (u32) u32[z + k] = uu[k];
        if (uop) store_child<P>(uop, static_cast<size_t>(row * uop_ld + z + k), uop_lo, uu[k]);
      }
    }
    if (s == root_slot) {
      const float4 pz = load_run4<kVec>(pi, q, H);
      dot += (pz.x * u.x + pz.y * u.y) + (pz.z * u.z + pz.w * u.w);
    }
  }
  if (lane == 0) {
    Ex[row] = live ? emax : 0;
    Lm[row] = live ? logf(mmax) : -INFINITY;
  }
  if (s != root_slot) return;
  for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  if (lane == 0) rdot[b] = dot;
}

// The log-likelihood. Every node lies under the root, so the root's offset is the sum over
// all nodes of their own log max: LL_b = ln 2 sum_v e_v[b] + sum_v log m_v[b] +
// log sum_z pi u_0[b][z], summed in double (the exponents exactly, as integers); also
// 1 / sum_z pi u_0 for the root flows. A block per 32 samples, one per lane: warp w sums
// the nodes w, w + 8, ... (128-byte loads, independent of one another), and the eight
// partial sums are combined in warp order.
constexpr int kLlWarps = 8;
__global__ void __launch_bounds__(kLlWarps * 32) k_hclt_ll(int nslots, int B, const int* __restrict__ Ex,
                                                          const float* __restrict__ Lm,
                                                          const float* __restrict__ rdot, double* __restrict__ ll,
                                                          float* __restrict__ rroot) {
  __shared__ long long esum_w[kLlWarps][32];
  __shared__ double lsum_w[kLlWarps][32];
  __shared__ int live_w[kLlWarps][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int b = blockIdx.x * 32 + lane;
  long long esum = 0;
  double lsum = 0.0;
  bool live = true;
  if (b < B) {
#pragma unroll 4
    for (int s = w; s < nslots; s += kLlWarps) {
      const long long idx = static_cast<long long>(s) * B + b;
      const float l = Lm[idx];
      live = live && l > -INFINITY;
      esum += Ex[idx];
      lsum += static_cast<double>(l);
    }
  }
  esum_w[w][lane] = esum;
  lsum_w[w][lane] = lsum;
  live_w[w][lane] = live;
  __syncthreads();
  if (w != 0 || b >= B) return;
  for (int k = 1; k < kLlWarps; ++k) {
    esum += esum_w[k][lane];
    lsum += lsum_w[k][lane];
    live = live && live_w[k][lane];
  }
  const float dot = rdot[b];
  live = live && dot > 0.f;
  ll[b] = live ? static_cast<double>(esum) * 0.69314718055994530942 + lsum + log(static_cast<double>(dot))
               : -static_cast<double>(INFINITY);
  rroot[b] = live ? 1.f / dot : 0.f;
}

// Root flows f_0[b][z] = pi[z] u_0[b][z] / sum_z pi u_0 (batch-major) and dpi += sum_b f_0.
__global__ void k_hclt_root_flows(int root_slot, int H, int B, const float* __restrict__ pi,
                                  const float* __restrict__ U32, long long u32_off, const float* __restrict__ rroot,
                                  float* __restrict__ F32, float* dpi) {
  const int z = blockIdx.x * blockDim.x + threadIdx.x;
  if (z >= H) return;
  const float pz = pi[z];
  float acc = 0.f;
  const int b0 = blockIdx.y * 32;
  for (int b = b0; b < b0 + 32 && b < B; ++b) {
    const long long idx = (static_cast<long long>(root_slot) * B + b) * H + z;
    const float f = pz * U32[idx - u32_off] * rroot[b];
    F32[idx] = f;
    acc += f;
  }
  if (dpi) atomicAdd(&dpi[z], acc);
}

// The layer's scaled flows of the edges in slots [s0, s0 + G): g[b][z] = f_parent[b][z] /
// D[b][z] (0 where D = 0), written batch-major (element contraction operand) and
// node-major (parameter contraction operand) through a 64 x 64 shared-memory tile; runs of
// four latents per load (16-byte accesses when kVec), runs of eight samples per
// node-major store.
template <int P, bool kVec>
__global__ void __launch_bounds__(256) k_hclt_scaled_flows(int s0, int H, int B, const int* __restrict__ parent_slot,
                                                           const float* __restrict__ F32, const float* __restrict__ D,
                                                           void* gbm, long long gbm_ld, size_t gbm_lo, void* gnm,
                                                           long long gnm_ld, size_t gnm_lo) {
  __shared__ float tile[64][65];
  const int g = blockIdx.z;
  const int s = s0 + g;
  const int ps = parent_slot[s];
  const int z0 = blockIdx.x * 64, b0 = blockIdx.y * 64;
  for (int i = threadIdx.x; i < 64 * 16; i += 256) {
    const int bb = i >> 4, zq = (i & 15) * 4;
    const int b = b0 + bb, z = z0 + zq;
    float w[4] = {0.f, 0.f, 0.f, 0.f};
    if (b < B && z < H) {
      const float4 d = load_run4<kVec>(D + (static_cast<long long>(s) * B + b) * H, z >> 2, H);
      const float4 f = load_run4<kVec>(F32 + (static_cast<long long>(ps) * B + b) * H, z >> 2, H);
      w[0] = d.x > 0.f ? f.x / d.x : 0.f;
      w[1] = d.y > 0.f ? f.y / d.y : 0.f;
      w[2] = d.z > 0.f ? f.z / d.z : 0.f;
      w[3] = d.w > 0.f ? f.w / d.w : 0.f;
      const size_t idx = static_cast<size_t>((static_cast<long long>(g) * B + b) * gbm_ld + z);
      if constexpr (kVec) {
        store_operand4<P>(gbm, idx, gbm_lo, make_float4(w[0], w[1], w[2], w[3]));
      } else {
        for (int k = 0; k < 4 && z + k < H; ++k) store_operand<P>(gbm, idx + k, gbm_lo, w[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) tile[bb][zq + k] = w[k];
  }
  __syncthreads();
  const StoreOperand<P> st{gnm, gnm_ld, gnm_lo, static_cast<long long>(H)};
  for (int i = threadIdx.x; i < 64 * 8; i += 256) {
    const int zz = i >> 3, bq = (i & 7) * 8;
    const int z = z0 + zz, b = b0 + bq;
    if (z >= H || b >= B) continue;
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = tile[bq + k][zz];
    st(g, z, b, v, min(8, B - b));
  }
}

// Stable per-node bucketing of the samples by category: order[s][..] lists the samples
// of node s grouped by x_{v,b} (increasing b inside a category), off[s][k] the start of
// category k. One warp per node; categories outside [0, C) are ignored.
__global__ void k_hclt_cat_bucket(int nvars, int B, int C, const int* __restrict__ data,
                                  const int* __restrict__ var_of_slot, int* __restrict__ order,
                                  int* __restrict__ off) {
  extern __shared__ int cnt[];  // C + 1
  const int s = blockIdx.x;
  const int v = var_of_slot[s];
  const int lane = threadIdx.x;
  for (int k = lane; k <= C; k += 32) cnt[k] = 0;
  __syncwarp();
  for (int b = lane; b < B; b += 32) {
    const int x = data[static_cast<long long>(b) * nvars + v];
    if (x >= 0 && x < C) atomicAdd(&cnt[x], 1);
  }
  __syncwarp();
  if (lane == 0) {  // exclusive scan, kept in cnt (running cursor) and written to off
    int run = 0;
    for (int k = 0; k < C; ++k) {
      const int c = cnt[k];
      cnt[k] = run;
      off[static_cast<long long>(s) * (C + 1) + k] = run;
      run += c;
    }
    off[static_cast<long long>(s) * (C + 1) + C] = run;
  }
  __syncwarp();
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    const int x = b < B ? data[static_cast<long long>(b) * nvars + v] : -1;
    const bool ok = x >= 0 && x < C;
    const unsigned same = __match_any_sync(0xffffffffu, ok ? x : -1);
    const int rank = __popc(same & ((1u << lane) - 1u));
    const int base = ok ? cnt[x] : 0;
    __syncwarp();
    if (ok) order[static_cast<long long>(s) * B + base + rank] = b;
    if (ok && rank == 0) cnt[x] = base + __popc(same);
    __syncwarp();
  }
}

// dE[v][z][k] (+)= sum over the samples of node s with category k of f[s][b][z], written
// in dE's own [H][C] layout in one pass. A block takes 32 categories and 256 latents of
// one node: each warp sums its categories' sample rows (bucket order, so the sums are
// deterministic; lane l takes latents l, l + 32, ..., 128-byte loads per row) into a
// shared-memory tile, and the block then writes the tile out latent by latent, the 32
// categories of a latent (128 contiguous bytes) per warp store. f is read once and dE
// written once, with no category-major copy between them.
constexpr int kDETileC = 32;   // categories per block (one per lane on the way out)
constexpr int kDETileZ = 256;  // latents per block
constexpr int kDEWarps = 8;
__global__ void __launch_bounds__(kDEWarps * 32) k_hclt_dE_tiles(int n, int H, int B, int C, int accumulate,
                                                                const int* __restrict__ var_of_slot,
                                                                const int* __restrict__ order,
                                                                const int* __restrict__ off,
                                                                const float* __restrict__ F32,
                                                                float* __restrict__ dE) {
  __shared__ float tile[kDETileC][kDETileZ + 1];  // odd row length: both phases conflict-free
  __shared__ int bounds[kDETileC + 1];
  constexpr int kRuns = kDETileZ / 32;
  const long long zt = (H + kDETileZ - 1) / kDETileZ, ct = (C + kDETileC - 1) / kDETileC;
  const long long blk = blockIdx.x;
  const int z0 = static_cast<int>(blk % zt) * kDETileZ;
  const int k0 = static_cast<int>((blk / zt) % ct) * kDETileC;
  const int s = static_cast<int>(blk / (zt * ct));
  if (s >= n) return;  // the whole block leaves together
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long ob = static_cast<long long>(s) * (C + 1);
  if (threadIdx.x <= kDETileC) bounds[threadIdx.x] = off[ob + min(k0 + static_cast<int>(threadIdx.x), C)];
  __syncthreads();
  const int* ord = order + static_cast<long long>(s) * B;
  const float* fs = F32 + static_cast<long long>(s) * B * H + z0;
  const int zn = min(kDETileZ, H - z0);
  for (int c = warp; c < kDETileC; c += kDEWarps) {
    float acc[kRuns];
#pragma unroll
    for (int r = 0; r < kRuns; ++r) acc[r] = 0.f;
    const int e1 = bounds[c + 1];
    for (int e = bounds[c]; e < e1; ++e) {
      const float* row = fs + static_cast<long long>(ord[e]) * H;
      float x[kRuns];
#pragma unroll
      for (int r = 0; r < kRuns; ++r) x[r] = lane + 32 * r < zn ? row[lane + 32 * r] : 0.f;
#pragma unroll
      for (int r = 0; r < kRuns; ++r) acc[r] += x[r];
    }
#pragma unroll
    for (int r = 0; r < kRuns; ++r) tile[c][lane + 32 * r] = acc[r];
  }
  __syncthreads();
  const int k = k0 + lane;
  if (k >= C) return;
  float* out = dE + static_cast<long long>(var_of_slot[s]) * H * C + static_cast<long long>(z0) * C + k;
  for (int z = warp; z < zn; z += kDEWarps) {
    const float v = tile[lane][z];
    float* p = out + static_cast<long long>(z) * C;
    *p = accumulate ? *p + v : v;
  }
}


// Copies a 128 x 128 block rows[n0 + c][m0 + r] of a row-major [B][H] array into
// shared memory as S[c][r] (0 outside), so an epilogue thread owning row r reads its 32
// columns without touching global memory. Runs in the epilogue warps during the K loop.
__device__ __forceinline__ void stage_block(const float* __restrict__ src, int H, int B, int m0, int n0,
                                            float* S, int et) {
  constexpr int kCols = kBM / kEpiWarps;  // columns staged by one epilogue warp
  const int lane = et & 31;
  const int c_begin = (et >> 5) * kCols;
#pragma unroll 1
  for (int cb = c_begin; cb < c_begin + kCols; cb += 8) {
    float vals[8][4];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const bool bin = n0 + cb + c < B;
      const float* row = src + static_cast<long long>(n0 + cb + c) * H + m0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        vals[c][i] = (bin && m0 + r < H) ? row[r] : 0.f;
      }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) S[(cb + c) * kBM + lane + 32 * i] = vals[c][i];
  }
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// stage_block of u given as the children operand's bf16 hi and lo parts (rows ld apart,
// the lo part lo elements after the hi part): S[c][r] = hi + lo.
__device__ __forceinline__ void stage_block_hilo(const uint16_t* __restrict__ src, long long ld, size_t lo, int H,
                                                 int B, int m0, int n0, float* S, int et) {
  constexpr int kCols = kBM / kEpiWarps;
  const int lane = et & 31;
  const int c_begin = (et >> 5) * kCols;
#pragma unroll 1
  for (int cb = c_begin; cb < c_begin + kCols; cb += 8) {
    float vals[8][4];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const bool bin = n0 + cb + c < B;
      const uint16_t* row = src + static_cast<long long>(n0 + cb + c) * ld + m0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        vals[c][i] = (bin && m0 + r < H) ? bf16_bits_to_float(row[r]) + bf16_bits_to_float(row[r + lo]) : 0.f;
      }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) S[(cb + c) * kBM + lane + 32 * i] = vals[c][i];
  }
}

// Forward epilogue: D[g][b][z], the edge's sum layer kept linear; thread = parent latent z.
// The bf16 forward runs on persistent tiles with one accumulation over K (= H) per tile:
// the accumulator's truncation costs an edge at most H / 16 half ulps of D (K = 1024:
// < 4e-6 of D, far inside the bf16 mode's rounding), and one tile's stores run under the
// next tile's MMAs. (The TF32 mode slices K, EpiSliceTF32.)
struct EpiHcltFwd : EpiNoHooks {
  static constexpr int kSliceBF16 = 0;
  // With uniform emissions every latent of a node is within a rounding step of the node's
  // maximum, where one bf16 / TF32 rounding would take them all to exactly 1 and each
  // edge would gain its largest row sum error instead of an average: the children
  // operand keeps a lo part (EpiBLo).
  static constexpr bool kBLo = true;
  struct Params {
    float* D;  // at the level's first slot, [G][B][H]
    int H, B;
  };
  __device__ static void apply(const Params& p, int g, int m0, int n0, int row, int col0,
                               float (&v)[32], uint8_t*, float*) {
    const int z = m0 + row;
    if (z >= p.H) return;
    float* dst = p.D + (static_cast<long long>(g) * p.B + n0 + col0) * p.H + z;
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if (n0 + col0 + c < p.B) dst[static_cast<long long>(c) * p.H] = v[c];
  }
};

// Element-flow epilogue: f[g][b][z'] = u[g][b][z'] * D[z', b]; thread = child latent z'.
// For 128-wide tiles the u block is staged in shared memory during the K loop (not in
// 3xTF32, whose ring needs the room); 256-wide tiles read it directly (a 128 KB block
// would leave the ring two slots).
struct HcltElemParams {
  const float* U32;  // at the level's first slot, [G][B][H] (TF32 modes)
  float* F32;        // idem
  int H, B;
  // bf16 mode: u as the children operand's hi and lo parts (the forward's B operand; no
  // float32 copy of u is kept below the root): [G][B][ld] at the level's first slot
  const uint16_t* Uh;
  long long uld;
  size_t ulo;
};
template <int P, int BN = kHcltBN>
struct EpiHcltElem : EpiNoHooks {
  using Params = HcltElemParams;
  static constexpr bool kStage = P != kTF32x3 && BN == kHcltBN;
  static constexpr bool kLoadAhead = BN == 2 * kHcltBN;  // the persistent 256-wide form, see issue
  static constexpr int kAheadBufs = 2;  // as EpiThetaScaleAhead
  static constexpr int kSmemBytes = kStage ? kHcltBN * kBM * 4 : (kLoadAhead ? kEpiWarps * kAheadBufs * 4096 : 0);

  __device__ static void prepare(const Params& p, int g, int m0, int n0, int et, uint8_t* smem) {
    if constexpr (kStage && P == kBF16)
      stage_block_hilo(p.Uh + static_cast<long long>(g) * p.B * p.uld, p.uld, p.ulo, p.H, p.B, m0, n0,
                       reinterpret_cast<float*>(smem), et);
    else if constexpr (kStage)
      stage_block(p.U32 + static_cast<long long>(g) * p.B * p.H, p.H, p.B, m0, n0, reinterpret_cast<float*>(smem),
                  et);
  }

  __device__ static void apply(const Params& p, int g, int m0, int n0, int row, int col0,
                               float (&v)[32], uint8_t* smem, float*) {
    const int z = m0 + row;
    if (z >= p.H) return;
    const long long base = (static_cast<long long>(g) * p.B + n0 + col0) * p.H + z;
    float u[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      if constexpr (kStage) {
        u[c] = reinterpret_cast<const float*>(smem)[(col0 + c) * kBM + row];
      } else if constexpr (P == kBF16) {
        const long long i = (static_cast<long long>(g) * p.B + n0 + col0 + c) * p.uld + z;
        u[c] = n0 + col0 + c < p.B ? bf16_bits_to_float(p.Uh[i]) + bf16_bits_to_float(p.Uh[i + p.ulo]) : 0.f;
      } else {
        u[c] = n0 + col0 + c < p.B ? p.U32[base + static_cast<long long>(c) * p.H] : 0.f;
      }
    }
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if (n0 + col0 + c < p.B) p.F32[base + static_cast<long long>(c) * p.H] = u[c] * v[c];
  }

  // persistent tiles (kLoadAhead, bf16): the chunk's node values u[b][z] (32 samples x 32
  // latents, as 128-byte rows of 32 hi then 32 lo parts) come through the warp's ring of
  // shared-memory buffers; lane = latent z reads them conflict-free. Needs H % 8 == 0
  // (16-byte pieces of bf16 rows).
  __device__ static void issue(const Params& p, int g, int m0, int n0, int q, int col0, float* buf) {
    static_assert(P == kBF16, "the persistent element-flow tiles are bf16");
    const int lane = threadIdx.x & 31;
    const int pc = lane & 7;  // pieces 0-3: hi, 4-7: lo
    const int z = m0 + q * 32 + 8 * (pc & 3);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = 4 * k + (lane >> 3);
      const int b = n0 + col0 + c;
      const int n = (b < p.B && z < p.H) ? min(8, p.H - z) : 0;
      const uint16_t* src =
          n ? p.Uh + (pc >= 4 ? p.ulo : 0) + (static_cast<long long>(g) * p.B + b) * p.uld + z : p.Uh;
      cp_async_16(reinterpret_cast<uint8_t*>(buf) + c * 128 + pc * 16, src, static_cast<uint32_t>(n * 2));
    }
  }
  __device__ static void apply_buf(const Params& p, int g, int m0, int n0, int row, int col0, float (&v)[32],
                                   float* buf) {
    const int z = m0 + row;
    if (z >= p.H) return;
    const int lane = threadIdx.x & 31;
    const uint16_t* hb = reinterpret_cast<const uint16_t*>(buf);
    const long long base = (static_cast<long long>(g) * p.B + n0 + col0) * p.H + z;
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if (n0 + col0 + c < p.B)
        p.F32[base + static_cast<long long>(c) * p.H] =
            (bf16_bits_to_float(hb[c * 64 + lane]) + bf16_bits_to_float(hb[c * 64 + 32 + lane])) * v[c];
  }
};

// The host plan reaches the device inside kernel arguments (by value, up to kPlanChunk
// ints per launch), so that a call issues no host-to-device copy from pageable memory and
// can be captured into a CUDA graph: the graph keeps the arguments.
constexpr int kPlanChunk = 6144;  // 24 KB of kernel parameters (the limit is 32 KB)
struct PlanChunk {
  int n;
  int v[kPlanChunk];
};
__global__ void k_write_plan(int* __restrict__ dst, const __grid_constant__ PlanChunk c) {
  for (int i = threadIdx.x; i < c.n; i += blockDim.x) dst[i] = c.v[i];
}

// ---------------------------------------------------------------- host plan
struct HcltPlan {
  int n = 0, E = 0, maxh = 0;
  std::vector<int> var_of_slot, child_ptr, child_slots, parent_slot, level_start;
  std::vector<int> blob;  // var_of_slot | child_ptr | child_slots | parent_slot
  int off_var = 0, off_cptr = 0, off_cslots = 0, off_pslot = 0;
};

pc_status_t make_plan(int n, const int32_t* parent, HcltPlan* pl) {
  PC_CHECK(parent[0] == -1, PC_ERR_SHAPE, "parent[0] must be -1 (variable 0 is the root)");
  for (int i = 1; i < n; ++i)
    PC_CHECK(parent[i] >= 0 && parent[i] < i, PC_ERR_SHAPE, "parent[%d] = %d is not in [0, %d)", i, parent[i], i);
  std::vector<int> height(n, 0);
  for (int v = n - 1; v >= 1; --v) height[parent[v]] = std::max(height[parent[v]], height[v] + 1);
  pl->n = n;
  pl->E = n - 1;
  pl->maxh = height[0];
  std::vector<int> edges(n - 1);
  for (int i = 0; i < n - 1; ++i) edges[i] = i + 1;
  std::stable_sort(edges.begin(), edges.end(), [&](int a, int b) { return height[a] < height[b]; });
  pl->var_of_slot.assign(n, 0);
  std::vector<int> slot_of_var(n, 0);
  for (int s = 0; s < n - 1; ++s) {
    pl->var_of_slot[s] = edges[s];
    slot_of_var[edges[s]] = s;
  }
  pl->var_of_slot[n - 1] = 0;
  slot_of_var[0] = n - 1;
  pl->level_start.assign(pl->maxh + 2, 0);
  for (int L = 0; L <= pl->maxh + 1; ++L) {
    int s = 0;
    while (s < n && height[pl->var_of_slot[s]] < L) ++s;
    pl->level_start[L] = s;
  }
  std::vector<std::vector<int>> kids(n);
  for (int c = 1; c < n; ++c) kids[parent[c]].push_back(slot_of_var[c]);
  pl->child_ptr.assign(n + 1, 0);
  pl->child_slots.clear();
  for (int s = 0; s < n; ++s) {
    const int v = pl->var_of_slot[s];
    pl->child_ptr[s] = static_cast<int>(pl->child_slots.size());
    for (int cs : kids[v]) pl->child_slots.push_back(cs);
  }
  pl->child_ptr[n] = static_cast<int>(pl->child_slots.size());
  if (pl->child_slots.empty()) pl->child_slots.push_back(0);
  pl->parent_slot.assign(n, -1);
  for (int s = 0; s < n - 1; ++s) pl->parent_slot[s] = slot_of_var[parent[pl->var_of_slot[s]]];
  pl->blob.clear();
  pl->off_var = 0;
  pl->blob.insert(pl->blob.end(), pl->var_of_slot.begin(), pl->var_of_slot.end());
  pl->off_cptr = static_cast<int>(pl->blob.size());
  pl->blob.insert(pl->blob.end(), pl->child_ptr.begin(), pl->child_ptr.end());
  pl->off_cslots = static_cast<int>(pl->blob.size());
  pl->blob.insert(pl->blob.end(), pl->child_slots.begin(), pl->child_slots.end());
  pl->off_pslot = static_cast<int>(pl->blob.size());
  pl->blob.insert(pl->blob.end(), pl->parent_slot.begin(), pl->parent_slot.end());
  return PC_OK;
}

// Operand view of groups [first, first + count) of an operand array.
Operand operand_view(const Operand& op, pc_precision_t p, long long first, long long count) {
  Operand v = op;
  v.ptr = static_cast<uint8_t*>(op.ptr) + size_t(first) * op.rows * op.ld * operand_elem_bytes(p);
  v.groups = count;
  return v;
}

struct HcltWs {
  int* plan;
  Operand Wop, WopT, Uop, Gbm, Gnm, Unm;
  float *Et, *U32, *D, *rroot, *rdot, *Lm, *F32;
  long long u32_off = 0;  // elements between U32 and the first stored slot row
  int* Ex;
  int *cat_order, *cat_off;
};

// The parameters in the contractions' formats, prepared once for many calls (pc_hclt_prepare):
// the slot order of the edges, W's per-edge operand copies in slot order (rows z_parent,
// K = z_child) and transposed (rows z_child), and E transposed per variable [v][k][z].
struct HcltPrep {
  int* var_of_slot;
  Operand Wop, WopT;
  float* Et;
};

size_t carve_prep(void* base, pc_precision_t p, int n, int H, int C, HcltPrep* w) {
  Carver c(base);
  *w = HcltPrep{};
  const long long E1 = n > 1 ? n - 1 : 1;
  w->var_of_slot = static_cast<int*>(c.take(size_t(n) * 4));
  w->Wop = c.operand(p, E1, H, H);
  w->WopT = c.operand(p, E1, H, H);
  w->Et = static_cast<float*>(c.take(size_t(n) * C * H * 4));
  return c.used;
}

size_t hclt_prep_bytes(pc_precision_t p, int n, int H, int C) {
  HcltPrep w;
  return carve_prep(nullptr, p, n, H, C, &w) + 256;
}

// prepared = true: W's operand copies and E transposed come from a prepared buffer.
size_t carve_hclt(void* base, pc_precision_t p, int n, int H, int C, int B, bool flows, bool want_dE, HcltWs* w,
                  bool prepared = false) {
  Carver c(base);
  *w = HcltWs{};
  const long long E1 = n > 1 ? n - 1 : 1;
  w->plan = static_cast<int*>(c.take(size_t(4 * n + 2) * 4));
  if (!prepared) {
    w->Wop = c.operand(p, E1, H, H);
    w->Et = static_cast<float*>(c.take(size_t(n) * C * H * 4));
  }
  // bf16: u is kept in float32 for the root alone (below it the children operand's hi
  // and lo parts carry it); U32 then holds the root's rows and u32_off shifts slot rows
  const bool u32_root_only = p == PC_PREC_AUTO;
  w->u32_off = u32_root_only ? static_cast<long long>(n - 1) * B * H : 0;
  w->U32 = static_cast<float*>(c.take(size_t(u32_root_only ? 1 : n) * B * H * 4));
  w->Uop = c.operand(p, E1, B, H, 2);  // hi + lo in every mode (EpiHcltFwd::kBLo)
  w->D = static_cast<float*>(c.take(size_t(E1) * B * H * 4));
  w->Ex = static_cast<int*>(c.take(size_t(n) * B * 4));
  w->Lm = static_cast<float*>(c.take(size_t(n) * B * 4));
  w->rroot = static_cast<float*>(c.take(size_t(B) * 4));
  w->rdot = static_cast<float*>(c.take(size_t(B) * 4));
  if (flows) {
    if (!prepared) w->WopT = c.operand(p, E1, H, H);
    w->F32 = static_cast<float*>(c.take(size_t(n) * B * H * 4));
    w->Gbm = c.operand(p, E1, B, H);
    w->Gnm = c.operand(p, E1, H, B);
    w->Unm = c.operand(p, E1, H, B);
    if (want_dE) {
      w->cat_order = static_cast<int*>(c.take(size_t(n) * B * 4));
      w->cat_off = static_cast<int*>(c.take(size_t(n) * (C + 1) * 4));
    }
  }
  return c.used;
}

size_t hclt_ws_bytes(pc_precision_t p, int n, int H, int C, int B, bool prepared = false) {
  HcltWs w;
  return carve_hclt(nullptr, p, n, H, C, B, true, true, &w, prepared) + 256;
}

pc_status_t check_hclt_shape(int n, int H, int C, int B) {
  PC_CHECK(n >= 1 && H >= 1 && C >= 1 && B >= 1, PC_ERR_SHAPE,
           "nvars, H, C, B must be >= 1 (got %d, %d, %d, %d)", n, H, C, B);
  PC_CHECK(n <= 65535 && H <= 8192 && C <= 8192 && B <= 65535, PC_ERR_SHAPE,
           "sizes out of range (nvars <= 65535, H <= 8192, C <= 8192, B <= 65535)");
  PC_CHECK(static_cast<long long>(n) * B * H < (1ll << 40) && static_cast<long long>(n) * C * H < (1ll << 40),
           PC_ERR_SHAPE, "problem too large");
  return PC_OK;
}

void* align256(const void* p) {
  return reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(p) + 255) & ~uintptr_t(255));
}

// W's operand copies (slot order of the tree) and E transposed, into a prepared buffer.
template <int P>
pc_status_t hclt_prepare(int n, int H, int C, const int32_t* parent, const float* W, const float* Em,
                         pc_precision_t prec, void* prep, cudaStream_t s) {
  HcltPlan pl;
  pc_status_t st;
  if ((st = make_plan(n, parent, &pl)) != PC_OK) return st;
  HcltPrep w;
  carve_prep(align256(prep), prec, n, H, C, &w);
  for (int off = 0; off < n; off += kPlanChunk) {
    PlanChunk ch;
    ch.n = std::min(kPlanChunk, n - off);
    std::copy(pl.var_of_slot.begin() + off, pl.var_of_slot.begin() + off + ch.n, ch.v);
    k_write_plan<<<1, 256, 0, s>>>(w.var_of_slot + off, ch);
    PC_LAUNCH_CHECK();
  }
  if ((st = transpose_f32(Em, C, static_cast<long long>(H) * C, n, H, C, w.Et, H, 0, s)) != PC_OK) return st;
  const int E = n - 1;
  if (E > 0 &&
      (st = operand_and_transpose<P>(W, H, static_cast<long long>(H) * H, E, H, H, w.Wop, w.WopT, s, w.var_of_slot)) !=
          PC_OK)
    return st;
  return PC_OK;
}

// prep: NULL, or a buffer written by hclt_prepare for the same tree, sizes and precision.
template <int P>
pc_status_t hclt_run(int n, int H, int C, int B, const int32_t* parent, const int32_t* data, const float* pi,
                     const float* W, const float* Em, double* ll, float* dpi, float* dW, float* dE, int accumulate,
                     pc_precision_t prec, void* ws, cudaStream_t s, const void* prep = nullptr) {
  constexpr int kParamBN = (P == kBF16) ? 256 : 128;
  HcltPlan pl;
  pc_status_t st;
  if ((st = make_plan(n, parent, &pl)) != PC_OK) return st;
  const bool flows = dpi || dW || dE;
  const bool down = flows && (dW || dE) && n >= 2;  // flows below the root are needed
  HcltWs w;
  carve_hclt(align256(ws), prec, n, H, C, B, flows, dE != nullptr, &w, prep != nullptr);
  if (prep) {
    HcltPrep pw;
    carve_prep(align256(prep), prec, n, H, C, &pw);
    w.Wop = pw.Wop;
    w.WopT = pw.WopT;
    w.Et = pw.Et;
  }
  const int E = n - 1;
  const int root = n - 1;
  const int* d_var = w.plan + pl.off_var;
  const int* d_cptr = w.plan + pl.off_cptr;
  const int* d_cslots = w.plan + pl.off_cslots;
  const int* d_pslot = w.plan + pl.off_pslot;

  // algorithmic bytes of the memory-bound launches (profiler records, PC_KIND_HCLT_MEM)
  const long long eb = operand_elem_bytes(prec) * operand_parts(prec);  // stored bytes per operand value
  const long long eb2 = 2ll * operand_elem_bytes(prec);                  // the children operand's hi + lo
  const long long HH = static_cast<long long>(H) * H, BH = static_cast<long long>(B) * H;
  const long long CH = static_cast<long long>(C) * H;
  // the tree plan (a few KB of host data) travels in kernel arguments
  for (size_t off = 0; off < pl.blob.size(); off += kPlanChunk) {
    PlanChunk ch;
    ch.n = static_cast<int>(std::min<size_t>(kPlanChunk, pl.blob.size() - off));
    std::copy(pl.blob.begin() + off, pl.blob.begin() + off + ch.n, ch.v);
    k_write_plan<<<1, 256, 0, s>>>(w.plan + off, ch);
    PC_LAUNCH_CHECK();
  }
  if (dpi && !accumulate) PC_CUDA(cudaMemsetAsync(dpi, 0, size_t(H) * 4, s));
  if (dW && !accumulate) PC_CUDA(cudaMemsetAsync(dW, 0, size_t(H) * H * 4, s));  // W[0] has no edge

  // Et[v][k][z] = E[v][z][k]: the emissions of one category are a contiguous row
  if (!prep) {
    ProfileScope ps(s, PC_KIND_HCLT_MEM, 2ll * n * CH * 4);
    if ((st = transpose_f32(Em, C, static_cast<long long>(H) * C, n, H, C, w.Et, H, 0, s)) != PC_OK) return st;
  }
  if (E > 0 && !prep) {
    // W's two operand copies (Wᵀ's for the element flows) in one pass over W
    ProfileScope ps(s, PC_KIND_HCLT_MEM, E * HH * (4 + (down ? 2 : 1) * eb));
    if ((st = down ? operand_and_transpose<P>(W, H, HH, E, H, H, w.Wop, w.WopT, s, d_var)
                   : rows_to_operand<P>(W, H, HH, E, H, H, w.Wop, s, d_var)) != PC_OK)
      return st;
  }

  // -------------------------------------------------------------- forward
  const size_t prod_smem = size_t((H + 3) / 4) * 32;  // mantissa and exponent runs, up to 64 KB
  const bool prod_vec = H % 4 == 0 && aligned16(pi);
  if (prod_smem > 48 * 1024) {
    PC_CUDA(cudaFuncSetAttribute(k_hclt_product<P, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(prod_smem)));
    PC_CUDA(cudaFuncSetAttribute(k_hclt_product<P, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(prod_smem)));
  }
  OperandMaps ma, mb;
  for (int L = 0; L <= pl.maxh; ++L) {
    const int sA = pl.level_start[L], sB = pl.level_start[L + 1];
    const int G = sB - sA;
    if (G <= 0) continue;
    const bool edges = L < pl.maxh;
    const long long kids = pl.child_ptr[sB] - pl.child_ptr[sA];
    // bf16: below the root u lives only in the children operand's hi and lo parts
    float* u32_out = (P == kBF16 && edges) ? nullptr : w.U32;
    ProfileScope ps(s, PC_KIND_HCLT_MEM,
                    G * B * 4ll + G * BH * 4 + (u32_out ? G * BH * 4 : 0) + kids * BH * 4 +
                        (edges ? G * BH * eb2 : H * 4ll + B * 4ll));
    if (H <= 4 * 32 * kWarpRuns) {
      const unsigned blocks = static_cast<unsigned>(cdiv(static_cast<long long>(G) * B, 8));
      // height 0 below the root: nodes without children (the leaf kernel)
      const bool leaf = L == 0 && edges;
      (leaf ? (prod_vec ? k_hclt_product_warp<P, true, true> : k_hclt_product_warp<P, false, true>)
            : (prod_vec ? k_hclt_product_warp<P, true> : k_hclt_product_warp<P, false>))<<<blocks, 256, 0, s>>>(
          sA, G, root, n, H, B, data, d_var, d_cptr, d_cslots, w.Et, w.D, C, u32_out, w.u32_off, edges ? w.Uop.ptr : nullptr,
          w.Uop.ld, w.Uop.lo_elems, w.Ex, w.Lm, pi, w.rdot);
    } else {
      (prod_vec ? k_hclt_product<P, true> : k_hclt_product<P, false>)<<<dim3(G, B), 256, prod_smem, s>>>(
          sA, root, n, H, B, data, d_var, d_cptr, d_cslots, w.Et, w.D, C, u32_out, w.u32_off, edges ? w.Uop.ptr : nullptr,
          w.Uop.ld, w.Uop.lo_elems, w.Ex, w.Lm, pi, w.rdot);
    }
    PC_LAUNCH_CHECK();
    if (!edges) continue;
    if ((st = encode_maps(&ma, operand_view(w.Wop, prec, sA, G), prec, kBM)) != PC_OK) return st;
    if ((st = encode_maps_hilo(&mb, operand_view(w.Uop, prec, sA, G), prec, kHcltBN)) != PC_OK) return st;
    EpiHcltFwd::Params ep{w.D + static_cast<long long>(sA) * B * H, H, B};
    // a_early: W's operand copy was written before the first product layer
    if constexpr (P == kBF16)
      st = launch_gemm_persist<P, kHcltBN, EpiHcltFwd>(cdiv(H, kBM), cdiv(B, kHcltBN), G, ma.hi, ma.lo, mb.hi, mb.lo,
                                                       num_k_blocks(H, prec), ep, s, PC_KIND_HCLT_FWD,
                                                       2ll * G * H * H * B);
    else
      st = launch_gemm<P, kHcltBN, EpiHcltFwd>(dim3(cdiv(H, kBM), cdiv(B, kHcltBN), G), ma.hi, ma.lo, mb.hi, mb.lo,
                                               num_k_blocks(H, prec), ep, s, PC_KIND_HCLT_FWD, 2ll * G * H * H * B,
                                               true);
    if (st != PC_OK) return st;
  }
  {
    ProfileScope ps(s, PC_KIND_HCLT_MEM, n * B * 8ll + B * 16ll);
    k_hclt_ll<<<cdiv(B, 32), kLlWarps * 32, 0, s>>>(n, B, w.Ex, w.Lm, w.rdot, ll, w.rroot);
    PC_LAUNCH_CHECK();
  }
  if (!flows) return PC_OK;

  // ------------------------------------------------------------- backward
  {
    ProfileScope ps(s, PC_KIND_HCLT_MEM, 2 * BH * 4 + H * 4ll + B * 4ll);
    k_hclt_root_flows<<<dim3(cdiv(H, 256), cdiv(B, 32)), 256, 0, s>>>(root, H, B, pi, w.U32, w.u32_off, w.rroot,
                                                                       w.F32, dpi);
    PC_LAUNCH_CHECK();
  }
  if (down) {
    for (int L = pl.maxh - 1; L >= 0; --L) {
      const int sA = pl.level_start[L], sB = pl.level_start[L + 1];
      const int G = sB - sA;
      if (G <= 0) continue;
      {
        ProfileScope ps(s, PC_KIND_HCLT_MEM, G * BH * (8 + 2 * eb));
        (prod_vec ? k_hclt_scaled_flows<P, true> : k_hclt_scaled_flows<P, false>)<<<dim3(cdiv(H, 64), cdiv(B, 64), G),
                                                                                   256, 0, s>>>(
            sA, H, B, d_pslot, w.F32, w.D, w.Gbm.ptr, w.Gbm.ld, w.Gbm.lo_elems, w.Gnm.ptr, w.Gnm.ld,
            w.Gnm.lo_elems);
        PC_LAUNCH_CHECK();
      }
      // element flows of the level's children; 256-wide tiles (full-rate MMAs) where the
      // level has enough of them to fill the GPU
      if ((st = encode_maps(&ma, operand_view(w.WopT, prec, sA, G), prec, kBM)) != PC_OK) return st;
      const bool wide = P == kBF16 && H % 8 == 0 &&
                        static_cast<long long>(cdiv(H, kBM)) * cdiv(B, 2 * kHcltBN) * G >= num_sms();
      const int ebn = wide ? 2 * kHcltBN : kHcltBN;
      if ((st = encode_maps(&mb, operand_view(w.Gbm, prec, 0, G), prec, ebn)) != PC_OK) return st;
      HcltElemParams ee{w.U32 + static_cast<long long>(sA) * B * H, w.F32 + static_cast<long long>(sA) * B * H, H,
                        B, static_cast<const uint16_t*>(w.Uop.ptr) + static_cast<long long>(sA) * B * w.Uop.ld,
                        w.Uop.ld, w.Uop.lo_elems};
      // a_early: Wᵀ's operand copy was written before the first scaled-flow kernel. Levels with
      // more tiles than SMs run persistent (bf16: one tile's epilogue under the next's K loop).
      if constexpr (P == kBF16) {
        if (wide)
          st = launch_gemm_persist<P, 2 * kHcltBN, EpiHcltElem<P, 2 * kHcltBN>>(
              cdiv(H, kBM), cdiv(B, 2 * kHcltBN), G, ma.hi, ma.lo, mb.hi, mb.lo, num_k_blocks(H, prec), ee, s,
              PC_KIND_HCLT_ELEM, 2ll * G * H * H * B);
      }
      if (!wide)
        st = launch_gemm<P, kHcltBN, EpiHcltElem<P>>(dim3(cdiv(H, kBM), cdiv(B, kHcltBN), G), ma.hi, ma.lo, mb.hi,
                                                     mb.lo, num_k_blocks(H, prec), ee, s, PC_KIND_HCLT_ELEM,
                                                     2ll * G * H * H * B, true);
      if (st != PC_OK) return st;
      if (!dW) continue;
      // parameter flows of the level's edges
      if constexpr (P == kBF16) {  // u's bf16 operand is its hi part
        ProfileScope ps(s, PC_KIND_HCLT_MEM, G * BH * 4);
        if ((st = transpose_bf16_to_operand(
                 static_cast<const uint16_t*>(w.Uop.ptr) + static_cast<long long>(sA) * B * w.Uop.ld, w.Uop.ld,
                 static_cast<long long>(B) * w.Uop.ld, G, B, H, w.Unm, s)) != PC_OK)
          return st;
      } else {
        ProfileScope ps(s, PC_KIND_HCLT_MEM, G * BH * (4 + eb));
        if ((st = transpose_to_operand<P>(w.U32 + static_cast<long long>(sA) * B * H, H,
                                          static_cast<long long>(B) * H, G, B, H, w.Unm, s)) != PC_OK)
          return st;
      }
      if ((st = encode_maps(&ma, operand_view(w.Gnm, prec, 0, G), prec, kBM)) != PC_OK) return st;
      if ((st = encode_maps(&mb, operand_view(w.Unm, prec, 0, G), prec, kParamBN)) != PC_OK) return st;
      EpiThetaScale::Params ep{dW, W, H, H, accumulate, d_var + sA};
      // short K (= B) and a theta block per tile: persistent (bf16, TF32), so the epilogue's
      // theta reads and dW writes overlap the next tile's K loop
      // (the theta blocks travel as 16-byte pieces: H % 4 == 0 and an aligned W)
      bool persist = false;
      if constexpr (P != kTF32x3) {
        if (H % 4 == 0 && aligned16(W)) {
          persist = true;
          st = launch_gemm_persist<P, kParamBN, EpiThetaScaleAhead>(cdiv(H, kBM), cdiv(H, kParamBN), G, ma.hi, ma.lo,
                                                                    mb.hi, mb.lo, num_k_blocks(B, prec), ep, s,
                                                                    PC_KIND_HCLT_PARAM, 2ll * G * H * H * B);
        }
      }
      if (!persist)
        st = launch_gemm<P, kParamBN, EpiThetaScale>(dim3(cdiv(H, kBM), cdiv(H, kParamBN), G), ma.hi, ma.lo, mb.hi,
                                                     mb.lo, num_k_blocks(B, prec), ep, s, PC_KIND_HCLT_PARAM,
                                                     2ll * G * H * H * B);
      if (st != PC_OK) return st;
    }
  }
  if (dE) {
    {
      ProfileScope ps(s, PC_KIND_HCLT_MEM, n * B * 8ll + n * (C + 1) * 4ll);
      k_hclt_cat_bucket<<<n, 32, size_t(C + 1) * 4, s>>>(n, B, C, data, d_var, w.cat_order, w.cat_off);
      PC_LAUNCH_CHECK();
    }
    ProfileScope ps(s, PC_KIND_HCLT_MEM, n * BH * 4 + n * B * 4ll + (accumulate ? 2ll : 1ll) * n * CH * 4);
    // at most 65535 x 256 x 32 blocks (the shape limits)
    const long long blocks = static_cast<long long>(n) * cdiv(C, kDETileC) * cdiv(H, kDETileZ);
    k_hclt_dE_tiles<<<static_cast<unsigned>(blocks), kDEWarps * 32, 0, s>>>(n, H, B, C, accumulate, d_var,
                                                                            w.cat_order, w.cat_off, w.F32, dE);
    PC_LAUNCH_CHECK();
  }
  return PC_OK;
}

}  // namespace
}  // namespace pc

extern "C" {

pc_status_t pc_hclt_workspace(int nvars, int H, int C, int B, pc_precision_t prec, size_t* bytes) {
  pc::clear_error();
  PC_CHECK(bytes != nullptr, PC_ERR_NULL, "bytes is NULL");
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_hclt_shape(nvars, H, C, B)) != PC_OK) return st;
  *bytes = pc::hclt_ws_bytes(prec, nvars, H, C, B);
  return PC_OK;
}

pc_status_t pc_hclt_fwd_bwd(int nvars, int H, int C, int B, const int32_t* parent, const int32_t* data,
                            const float* pi, const float* W, const float* E, double* ll, float* dpi, float* dW,
                            float* dE, int accumulate, pc_precision_t prec, void* ws, size_t ws_bytes,
                            pc_stream_t stream) {
  pc::clear_error();
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_hclt_shape(nvars, H, C, B)) != PC_OK) return st;
  PC_CHECK(parent && data && pi && W && E && ll, PC_ERR_NULL, "parent, data, pi, W, E and ll must not be NULL");
  PC_CHECK(ws, PC_ERR_WORKSPACE, "workspace is NULL");
  const size_t need = pc::hclt_ws_bytes(prec, nvars, H, C, B);
  PC_CHECK(ws_bytes >= need, PC_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", ws_bytes, need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (prec) {
    case PC_PREC_AUTO:
      return pc::hclt_run<pc::kBF16>(nvars, H, C, B, parent, data, pi, W, E, ll, dpi, dW, dE, accumulate, prec, ws, s);
    case PC_PREC_TF32:
      return pc::hclt_run<pc::kTF32>(nvars, H, C, B, parent, data, pi, W, E, ll, dpi, dW, dE, accumulate, prec, ws, s);
    default:
      return pc::hclt_run<pc::kTF32x3>(nvars, H, C, B, parent, data, pi, W, E, ll, dpi, dW, dE, accumulate, prec, ws,
                                       s);
  }
}

pc_status_t pc_hclt_prepare_bytes(int nvars, int H, int C, pc_precision_t prec, size_t* bytes) {
  pc::clear_error();
  PC_CHECK(bytes != nullptr, PC_ERR_NULL, "bytes is NULL");
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_hclt_shape(nvars, H, C, 1)) != PC_OK) return st;
  *bytes = pc::hclt_prep_bytes(prec, nvars, H, C);
  return PC_OK;
}

pc_status_t pc_hclt_prepare(int nvars, int H, int C, const int32_t* parent, const float* W, const float* E,
                            pc_precision_t prec, void* prep, size_t prep_bytes, pc_stream_t stream) {
  pc::clear_error();
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_hclt_shape(nvars, H, C, 1)) != PC_OK) return st;
  PC_CHECK(parent && W && E, PC_ERR_NULL, "parent, W and E must not be NULL");
  PC_CHECK(prep, PC_ERR_WORKSPACE, "prepared buffer is NULL");
  const size_t need = pc::hclt_prep_bytes(prec, nvars, H, C);
  PC_CHECK(prep_bytes >= need, PC_ERR_WORKSPACE, "prepared buffer of %zu bytes < %zu required", prep_bytes, need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (prec) {
    case PC_PREC_AUTO: return pc::hclt_prepare<pc::kBF16>(nvars, H, C, parent, W, E, prec, prep, s);
    case PC_PREC_TF32: return pc::hclt_prepare<pc::kTF32>(nvars, H, C, parent, W, E, prec, prep, s);
    default: return pc::hclt_prepare<pc::kTF32x3>(nvars, H, C, parent, W, E, prec, prep, s);
  }
}

pc_status_t pc_hclt_prepared_workspace(int nvars, int H, int C, int B, pc_precision_t prec, size_t* bytes) {
  pc::clear_error();
  PC_CHECK(bytes != nullptr, PC_ERR_NULL, "bytes is NULL");
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_hclt_shape(nvars, H, C, B)) != PC_OK) return st;
  *bytes = pc::hclt_ws_bytes(prec, nvars, H, C, B, true);
  return PC_OK;
}

pc_status_t pc_hclt_fwd_bwd_prepared(int nvars, int H, int C, int B, const int32_t* parent, const int32_t* data,
                                     const float* pi, const float* W, const void* prep, size_t prep_bytes, double* ll,
                                     float* dpi, float* dW, float* dE, int accumulate, pc_precision_t prec, void* ws,
                                     size_t ws_bytes, pc_stream_t stream) {
  pc::clear_error();
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_hclt_shape(nvars, H, C, B)) != PC_OK) return st;
  PC_CHECK(parent && data && pi && W && ll, PC_ERR_NULL, "parent, data, pi, W and ll must not be NULL");
  PC_CHECK(prep, PC_ERR_WORKSPACE, "prepared buffer is NULL");
  PC_CHECK(prep_bytes >= pc::hclt_prep_bytes(prec, nvars, H, C), PC_ERR_WORKSPACE,
           "prepared buffer of %zu bytes is smaller than pc_hclt_prepare_bytes reports", prep_bytes);
  PC_CHECK(ws, PC_ERR_WORKSPACE, "workspace is NULL");
  const size_t need = pc::hclt_ws_bytes(prec, nvars, H, C, B, true);
  PC_CHECK(ws_bytes >= need, PC_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", ws_bytes, need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (prec) {
    case PC_PREC_AUTO:
      return pc::hclt_run<pc::kBF16>(nvars, H, C, B, parent, data, pi, W, nullptr, ll, dpi, dW, dE, accumulate, prec,
                                     ws, s, prep);
    case PC_PREC_TF32:
      return pc::hclt_run<pc::kTF32>(nvars, H, C, B, parent, data, pi, W, nullptr, ll, dpi, dW, dE, accumulate, prec,
                                     ws, s, prep);
    default:
      return pc::hclt_run<pc::kTF32x3>(nvars, H, C, B, parent, data, pi, W, nullptr, ll, dpi, dW, dE, accumulate,
                                       prec, ws, s, prep);
  }
}

}  // extern "C"
