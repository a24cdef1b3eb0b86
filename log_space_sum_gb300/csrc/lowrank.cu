// LowRank "exp_sum" per-sample scale on a dense sum layer, forward and backward.
//
// pyjuice LowRank API doc (intro formulas; Tensor layout; Training): per sample b, with
// A_b [M,K] and B_b [K,N] (K = rank <= 64),
//   S_b = A_b B_b,   g_b = exp(S_b),   Z_b[i] = sum_j theta[i,j] g_b[i,j],
//   theta_b = theta g_b / Z_b,         out[i,b] = log sum_j theta_b[i,j] exp(x[j,b]).
// Backward for node flows f [M,B], with q = theta_b and p = theta_b exp(x_j - out_i):
//   D = f (p - q),  dA_b = D B_b^T,  dB_b = A_b^T D,  e[j,b] = sum_i f p,
//   F+[i,j] = sum_b f p,  W[i,j] = sum_b f g_b / Z_b.
// The doc's Note: the scale is made tile by tile on tensor cores and used where it is
// made, never stored; the factors' products in bf16 hi + lo under the default precision
// (the gradients' products one bf16 term), three-term TF32 under "fp32". The tf32 mode
// (which the doc does not name for this path) takes S in three-term TF32 and the
// gradients' products in one TF32 term.
//
// GB300 design. Every pass is one kernel over 128-row tiles of an "own" dimension with a
// 32-column sweep over the other; S for a 128 x 32 chunk is one tcgen05 MMA group into
// TMEM, read back by the thread that owns the row, exponentiated and consumed in
// registers. Shifts: the forward keeps a running row maximum of S (exact rescaling of
// its two sums); the backward uses the saved log Z (theta exp(S - log Z) = theta_b <= 1).
//   forward  own i, sweep j:  Z and sum_j theta g u_j online           -> out, logZ
//   grad A   own i, sweep j:  D row-tile to shared memory, dA += D B^T (TMEM accumulator)
//   grad B   own j, sweep i:  S^T = B^T A^T, D^T row-tile, dB^T += D^T A, e_j in registers
//   stats    own i, fixed 32 columns, sweep the samples: F+ and W in registers
// No pass needs an atomic: every output element is written by exactly one thread.
#include <algorithm>
#include <cmath>

#include "pc_launch.cuh"

namespace pc {
namespace {

constexpr int kLrRows = 128;   // own rows per CTA (TMEM lanes)
constexpr int kLrChunk = 32;   // sweep columns per MMA group
constexpr int kLrMaxRank = 64;
constexpr int kGradAccs = 4;   // TMEM accumulators of the gradient contractions

enum LrMode : int { kLrFwd = 0, kLrGradA = 1, kLrGradB = 2 };

// Operand formats of one tile: element bytes, parts (hi, lo) and MMA kind.
enum LrFmt : int { kFmtBF16 = 0, kFmtBF16x2 = 1, kFmtTF32 = 2, kFmtTF32x2 = 3 };
__host__ __device__ constexpr int fmt_bytes(int f) { return f <= kFmtBF16x2 ? 2 : 4; }
__host__ __device__ constexpr int fmt_parts(int f) { return (f == kFmtBF16x2 || f == kFmtTF32x2) ? 2 : 1; }
__host__ __device__ constexpr int fmt_kstep(int f) { return f <= kFmtBF16x2 ? 16 : 8; }  // K per MMA
// S = A B: bf16 hi + lo (auto), TF32 hi + lo (tf32 and fp32). exp turns an absolute
// error of S into a relative error of the scale, so S takes the split form in every
// mode; the modes differ in the gradients' products.
__host__ __device__ constexpr int s_fmt(int P) { return P == kBF16 ? kFmtBF16x2 : kFmtTF32x2; }
// The gradients' products: one bf16 term (auto), one TF32 pass, 3xTF32.
__host__ __device__ constexpr int g_fmt(int P) { return P == kBF16 ? kFmtBF16 : (P == kTF32 ? kFmtTF32 : kFmtTF32x2); }

// Geometry of a K-major SWIZZLE_128B operand tile of R rows (R % 8 == 0) holding K
// columns of format F: k-steps of fmt_kstep(F), 128-byte k-blocks of R rows each, the lo
// part after all hi blocks.
struct TileGeo {
  int rows, ksteps, kblocks;
  __host__ __device__ int bytes_part() const { return kblocks * rows * 128; }
};
__host__ __device__ inline TileGeo tile_geo(int F, int rows, int K) {
  TileGeo g;
  g.rows = rows;
  g.ksteps = (K + fmt_kstep(F) - 1) / fmt_kstep(F);
  const int bytes = g.ksteps * 32;  // every k-step covers 32 bytes of a row
  g.kblocks = (bytes + 127) / 128;
  return g;
}
__host__ __device__ inline int tile_bytes(int F, int rows, int K) {
  const TileGeo g = tile_geo(F, rows, K);
  return fmt_parts(F) * g.bytes_part();
}
// A split-format operand of K columns is "packed" when its hi and lo parts fit one
// 128-byte row together and K fills whole k-steps (rank 16 or 32 in bf16, 8 or 16 in
// TF32): the row holds the hi k-steps, then the lo k-steps, and no padding lies between.
// Its copy is one [rows][2K] array and its tile one part; otherwise the lo part follows
// all hi k-blocks.
__host__ __device__ constexpr bool lr_packed(int F, int K) {
  return fmt_parts(F) == 2 && K % fmt_kstep(F) == 0 && 2 * K * fmt_bytes(F) <= 128;
}
// The S operands' tiles: the parts loaded (each kblocks x rows x 128 bytes), the lo
// part's byte offset inside the tile and the tile's bytes.
struct STile {
  TileGeo g;
  int parts, lo_off, bytes;
};
__host__ __device__ inline STile s_tile(int F, int rows, int K) {
  STile t;
  t.g = tile_geo(F, rows, K);
  const bool packed = lr_packed(F, K);
  t.parts = packed ? 1 : fmt_parts(F);
  t.lo_off = packed ? K * fmt_bytes(F) : t.g.bytes_part();
  t.bytes = t.parts * t.g.bytes_part();
  return t;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Issues D(tmem) (+)= A(tile a, M = 128 rows) * B(tile b, N rows)^T over the k-steps of
// the tiles, in format F: split formats take lo*hi, hi*lo, then hi*hi per k-step, the lo
// parts a_lo and b_lo bytes after the hi parts.
template <int F>
__device__ __forceinline__ void lr_mma(uint32_t d, const uint8_t* a, const TileGeo& ga, const uint8_t* b,
                                       const TileGeo& gb, int n, bool accumulate, uint32_t a_lo, uint32_t b_lo) {
  constexpr uint32_t kind = F <= kFmtBF16x2 ? 1u : 2u;
  const uint32_t idesc = umma_idesc(kind, kLrRows, static_cast<uint32_t>(n));
  const uint32_t a0 = smem_addr(a), b0 = smem_addr(b);
  const uint32_t a1 = a0 + (fmt_parts(F) == 2 ? a_lo : 0);
  const uint32_t b1 = b0 + (fmt_parts(F) == 2 ? b_lo : 0);
  uint32_t acc = accumulate ? 1u : 0u;
  for (int kk = 0; kk < ga.ksteps; ++kk) {
    const uint32_t oa = (kk >> 2) * ga.rows * 128 + (kk & 3) * 32;
    const uint32_t ob = (kk >> 2) * gb.rows * 128 + (kk & 3) * 32;
    if constexpr (fmt_parts(F) == 2) {
      if constexpr (kind == 1u) {
        umma_bf16(d, umma_desc_sw128(a1 + oa), umma_desc_sw128(b0 + ob), idesc, acc);
        umma_bf16(d, umma_desc_sw128(a0 + oa), umma_desc_sw128(b1 + ob), idesc, 1u);
        umma_bf16(d, umma_desc_sw128(a0 + oa), umma_desc_sw128(b0 + ob), idesc, 1u);
      } else {
        umma_tf32(d, umma_desc_sw128(a1 + oa), umma_desc_sw128(b0 + ob), idesc, acc);
        umma_tf32(d, umma_desc_sw128(a0 + oa), umma_desc_sw128(b1 + ob), idesc, 1u);
        umma_tf32(d, umma_desc_sw128(a0 + oa), umma_desc_sw128(b0 + ob), idesc, 1u);
      }
    } else if constexpr (kind == 1u) {
      umma_bf16(d, umma_desc_sw128(a0 + oa), umma_desc_sw128(b0 + ob), idesc, acc);
    } else {
      umma_tf32(d, umma_desc_sw128(a0 + oa), umma_desc_sw128(b0 + ob), idesc, acc);
    }
    acc = 1u;
  }
}

// ------------------------------------------------------------------ set-up kernels
// Per sample b: m_b = max_j x[j,b] and u[b][j] = exp(x[j,b] - m_b) (sample-major, rows
// ldu apart). One block per sample.
__global__ void k_lr_colmax_u(int N, int B, const float* __restrict__ x, float* __restrict__ m,
                              float* __restrict__ u, long long ldu) {
  __shared__ float red[32];
  const int b = blockIdx.x;
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < N; j += blockDim.x) mx = fmaxf(mx, x[static_cast<long long>(j) * B + b]);
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : -INFINITY;
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  mx = red[0];
  if (threadIdx.x == 0) m[b] = mx;
  for (int j = threadIdx.x; j < N; j += blockDim.x)
    u[static_cast<long long>(b) * ldu + j] =
        mx > -INFINITY ? expf(x[static_cast<long long>(j) * B + b] - mx) : 0.f;
}

// Plain float32 copy of theta [M][N] (or its transpose) into a row-padded buffer that a
// tensor map can address (rows 16-byte aligned).
__global__ void k_lr_theta_copy(int M, int N, const float* __restrict__ theta, float* __restrict__ dst,
                                long long ld, int transpose) {
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;  // tile of theta: rows r0.., cols c0..
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (r < M && c < N) ? theta[static_cast<long long>(r) * N + c] : 0.f;
  }
  __syncthreads();
  if (!transpose) {
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + threadIdx.x;
      if (r < M && c < N) dst[static_cast<long long>(r) * ld + c] = tile[i][threadIdx.x];
    }
  } else {
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int c = c0 + i, r = r0 + threadIdx.x;
      if (r < M && c < N) dst[static_cast<long long>(c) * ld + r] = tile[threadIdx.x][i];
    }
  }
}

// Per (b, i): the backward's row factors lz = log Z_b[i], f_i and fc = f_i exp(m_b - out_i)
// (0 where out or log Z is -inf: such a node passes no flow), sample-major [B][ldm].
__global__ void k_lr_row_factors(int M, int B, const float* __restrict__ out, const float* __restrict__ f,
                                 const float* __restrict__ logZ, const float* __restrict__ m,
                                 float* __restrict__ rf_lz, float* __restrict__ rf_f, float* __restrict__ rf_fc,
                                 long long ldm) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(M) * B) return;
  const int b = static_cast<int>(idx / M), i = static_cast<int>(idx % M);
  const float o = out[static_cast<long long>(i) * B + b];
  const float lz = logZ[idx];
  const float fi = f[static_cast<long long>(i) * B + b];
  const bool live = o > -INFINITY && lz > -INFINITY && m[b] > -INFINITY;
  const long long dst = static_cast<long long>(b) * ldm + i;
  rf_lz[dst] = lz;
  rf_f[dst] = live ? fi : 0.f;
  rf_fc[dst] = live ? fi * expf(m[b] - o) : 0.f;
}

// Operand copy in format F: dst[g][r][c] (rows ld elements apart) = src[g*sg + r*sr +
// c*sc] for c < C, rounded to bf16 / TF32 (hi, and lo = the rounded remainder). The row
// padding [C, ld) is left unwritten: the operand's tensor maps end at C, so the TMA fills
// those columns of a tile with zeros and never reads them. One row (g, r) per warp row of
// the block: the row's index is split once per row, not per element.
template <int F>
__global__ void k_lr_to_op(const float* __restrict__ src, long long sg, long long sr, long long sc, int G, int R,
                           int C, void* __restrict__ hi, void* __restrict__ lo, long long ld) {
  const long long rows = static_cast<long long>(G) * R;
  for (long long gr = static_cast<long long>(blockIdx.x) * blockDim.y + threadIdx.y; gr < rows;
       gr += static_cast<long long>(gridDim.x) * blockDim.y) {
    const long long g = gr / R, r = gr - g * R;
    const float* s0 = src + g * sg + r * sr;
    for (long long c = threadIdx.x; c < C; c += blockDim.x) {
      const long long idx = gr * ld + c;
      const float v = s0[c * sc];
      if constexpr (F == kFmtBF16 || F == kFmtBF16x2) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        static_cast<__nv_bfloat16*>(hi)[idx] = h;
        if constexpr (F == kFmtBF16x2) static_cast<__nv_bfloat16*>(lo)[idx] = __float2bfloat16_rn(v - __bfloat162float(h));
      } else {
        const float h = tf32_rna(v);
        static_cast<float*>(hi)[idx] = h;
        if constexpr (F == kFmtTF32x2) static_cast<float*>(lo)[idx] = tf32_rna(v - h);
      }
    }
  }
}

// The same copy for a source contiguous along c (sc = 1) with C, sr and sg multiples of
// four and a 16-byte aligned base: four columns per thread (16-byte loads, 8- or 16-byte
// stores), so a rank-16 row takes four threads rather than half a warp of scalar loads.
// Rounds each value exactly as the element-wise copy does.
template <int F>
__global__ void k_lr_to_op4(const float* __restrict__ src, long long sg, long long sr, int R, int C4, long long rows,
                            void* __restrict__ hi, void* __restrict__ lo, long long ld) {
  const long long total = rows * C4;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long gr = i / C4;
    const int q = static_cast<int>(i - gr * C4);
    const long long g = gr / R, r = gr - g * R;
    const float4 v4 = *reinterpret_cast<const float4*>(src + g * sg + r * sr + 4 * q);
    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
    const long long idx = gr * ld + 4 * q;
    if constexpr (F == kFmtBF16 || F == kFmtBF16x2) {
      uint32_t h[4], l[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat16 b = __float2bfloat16_rn(v[k]);
        h[k] = __bfloat16_as_ushort(b);
        l[k] = __bfloat16_as_ushort(__float2bfloat16_rn(v[k] - __bfloat162float(b)));
      }
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(hi) + idx) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
      if constexpr (F == kFmtBF16x2)
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(lo) + idx) = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
    } else {
      const float4 h = make_float4(tf32_rna(v[0]), tf32_rna(v[1]), tf32_rna(v[2]), tf32_rna(v[3]));
      *reinterpret_cast<float4*>(static_cast<float*>(hi) + idx) = h;
      if constexpr (F == kFmtTF32x2)
        *reinterpret_cast<float4*>(static_cast<float*>(lo) + idx) =
            make_float4(tf32_rna(v[0] - h.x), tf32_rna(v[1] - h.y), tf32_rna(v[2] - h.z), tf32_rna(v[3] - h.w));
    }
  }
}

// The same copy where the source is contiguous along r (sr = 1) and strided along c: a
// 32 x 32 tile goes through shared memory, so that both the reads (along r) and the
// writes (along c) are coalesced.
template <int F>
__global__ void k_lr_to_op_t(const float* __restrict__ src, long long sg, long long sc, int G, int R, int C,
                             void* __restrict__ hi, void* __restrict__ lo, long long ld) {
  __shared__ float tile[32][33];
  const int g = blockIdx.z;
  const int r0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  const float* s0 = src + g * sg;
  for (int i = threadIdx.y; i < 32; i += 8) {  // i: column c0 + i, lane: row r0 + lane
    const int r = r0 + threadIdx.x, c = c0 + i;
    tile[i][threadIdx.x] = (r < R && c < C) ? s0[r + c * sc] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {  // i: row r0 + i, lane: column c0 + lane
    const int r = r0 + i;
    const long long c = c0 + threadIdx.x;
    if (r >= R || c >= C) continue;
    const long long idx = (static_cast<long long>(g) * R + r) * ld + c;
    const float v = tile[threadIdx.x][i];
    if constexpr (F == kFmtBF16 || F == kFmtBF16x2) {
      const __nv_bfloat16 h = __float2bfloat16_rn(v);
      static_cast<__nv_bfloat16*>(hi)[idx] = h;
      if constexpr (F == kFmtBF16x2) static_cast<__nv_bfloat16*>(lo)[idx] = __float2bfloat16_rn(v - __bfloat162float(h));
    } else {
      const float h = tf32_rna(v);
      static_cast<float*>(hi)[idx] = h;
      if constexpr (F == kFmtTF32x2) static_cast<float*>(lo)[idx] = tf32_rna(v - h);
    }
  }
}

// ------------------------------------------------------------------ shared memory plan
enum : int { kLrStats = 3 };
constexpr int kThetaTileBytes = kLrRows * 128;  // 128 rows x 32 floats
constexpr int kLrWarps = 8;                      // consumers: two warps per TMEM lane quarter
constexpr int kLrThreadsFused = (kLrWarps + 2) * 32;  // + a TMA producer warp and an MMA warp
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ constexpr int lr_stages(int mode) { return mode == kLrFwd ? 3 : 4; }
__host__ __device__ constexpr int lr_nvec(int mode) { return mode == kLrGradB ? 3 : 1; }

// Byte offsets inside the (1024-aligned) dynamic shared memory. Every TMA destination
// and every operand tile starts on a 1024-byte boundary.
struct LrSmem {
  int own, own_bytes;              // resident own tile (not the statistics pass)
  int stage, stage_bytes, nstage;  // ring of TMA stages
  int sw_off, th_off, vec_off;
  int sw_bytes, tx_bytes;
  int gbr, gb_bytes, ngb;          // ring of ngb gradient B-operand tiles (gradient passes)
  int d, d_bytes, nd;              // ring of nd D tiles (gradient passes)
  int bars, total;
};
constexpr int kGbSlots = 4;  // gradient B-operand tiles in flight at most
__host__ __device__ inline int up1024(int v) { return (v + 1023) & ~1023; }
__host__ __device__ inline LrSmem lr_smem_plan(int P, int mode, int K, int nstage, int nd, int ngb) {
  const int SF = s_fmt(P), GF = g_fmt(P);
  const int Kp = (K + 15) & ~15;
  const bool grad = mode == kLrGradA || mode == kLrGradB;
  LrSmem s;
  s.own_bytes = s_tile(SF, kLrRows, K).bytes;
  s.sw_bytes = s_tile(SF, kLrChunk, K).bytes;
  s.gb_bytes = grad ? fmt_parts(GF) * Kp * 128 : 0;
  s.nstage = nstage;
  s.nd = nd;
  s.ngb = grad ? ngb : 0;
  int off = 0;
  if (mode == kLrStats) off += s.own_bytes;  // the sample's own tile travels with its stage
  s.sw_off = off;
  off += s.sw_bytes;
  s.th_off = off;
  if (mode != kLrStats) off += kThetaTileBytes;
  s.vec_off = off;
  off += up1024(lr_nvec(mode) * 128);
  s.stage_bytes = up1024(off);
  s.tx_bytes = (mode == kLrStats ? s.own_bytes : 0) + s.sw_bytes + (mode != kLrStats ? kThetaTileBytes : 0) +
               lr_nvec(mode) * 128;
  off = 0;
  s.own = off;
  if (mode != kLrStats) off += s.own_bytes;
  s.stage = off;
  off += s.nstage * s.stage_bytes;
  s.gbr = off;  // gb_bytes is a multiple of 2048
  off += s.ngb * s.gb_bytes;
  s.d_bytes = grad ? tile_bytes(GF, kLrRows, kLrChunk) : 0;
  s.d = off;
  // bf16 D tiles fill half of each 128-byte row: two share one tile (d_pair)
  off += (GF == kFmtBF16 && nd == 2 ? 1 : nd) * s.d_bytes;
  s.bars = off;
  off += 2048;  // barriers, the TMEM slot and the end-of-pass merge buffers
  s.total = off + 1024;  // alignment slack
  return s;
}
constexpr int kLrSmemLimit = 232448;
constexpr int kLrSmemHalf = 113 * 1024;  // two CTAs per SM
// The backward passes run two CTAs per SM (their consumer warps are latency-bound, so a
// second CTA's warps fill the issue slots) when a ring of two or more stages fits half the
// shared memory; otherwise, and for the forward pass, the deepest ring (and two D tiles)
// that fits the shared memory of one CTA: large ranks in the TF32 formats take two
// 128-byte k-blocks per operand row.
__host__ __device__ inline LrSmem lr_smem(int P, int mode, int K) {
  if (mode != kLrFwd)
    for (int ns = 4; ns >= 2; --ns)
      for (int d = 2; d >= 1; --d) {
        const LrSmem h = lr_smem_plan(P, mode, K, ns, d, kGbSlots);
        if (h.total <= kLrSmemHalf) return h;
      }
  int nstage = lr_stages(mode), nd = 2, ngb = kGbSlots;
  LrSmem s = lr_smem_plan(P, mode, K, nstage, nd, ngb);
  while (s.total > kLrSmemLimit && nstage > 2) s = lr_smem_plan(P, mode, K, --nstage, nd, ngb);
  if (s.total > kLrSmemLimit) s = lr_smem_plan(P, mode, K, nstage, nd = 1, ngb);
  while (s.total > kLrSmemLimit && ngb > 1) s = lr_smem_plan(P, mode, K, nstage, nd, ngb /= 2);
  return s;
}

// Tensor maps of one pass: the own and sweep operand tiles (hi, lo), the gradient
// B-operand (hi, lo), theta (or its transpose) and up to three 32-float vectors.
struct LrMaps {
  CUtensorMap own[2], sw[2], gb[2], th, vec[3];
};

struct LrArgs {
  int M, N, K, B;
  const float* rf_lz;  // [B][ldm]  backward row factors (padded rows)
  const float* rf_f;
  const float* rf_fc;
  long long ldm;
  const float* theta_ld;  // row-padded theta copy (statistics pass)
  long long theta_ld_stride;
  const float* m;  // [B]
  const float* u;  // [B][ldu]  exp(x - m_b) (grad B's own-row constant)
  long long ldu;
  float* out;   // [M][B]
  float* logZ;  // [B][M]
  float* dA;    // [B][M][K]
  float* dB;    // [B][K][N]
  float* e;     // [N][B] or null
  float* Fp;    // [M][N] or null
  float* W;     // [M][N] or null
  int accumulate;
  unsigned* status;
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_ld_32x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive floats of row `row` of a 128-byte-swizzled tile of 32-float rows
// (theta tiles): four 16-byte loads.
__device__ __forceinline__ void tile_row16_f32(const uint8_t* tile, int row, int col0, float (&v)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int chunk = (col0 >> 2) + q;
    const float4 x =
        *reinterpret_cast<const float4*>(tile + row * 128 + (((chunk ^ (row & 7)) & 7) << 4));
    v[4 * q] = x.x;
    v[4 * q + 1] = x.y;
    v[4 * q + 2] = x.z;
    v[4 * q + 3] = x.w;
  }
}

// Writes 16 values at (row, col0 .. col0+15) of a one-k-block operand tile of format F
// with 16-byte stores (col0 a multiple of 16; the row's bytes fit one 128-byte block).
template <int F>
__device__ __forceinline__ void tile_put_row16(uint8_t* tile, const TileGeo& g, int row, int col0,
                                               const float (&v)[16]) {
  uint8_t* base = tile + (row >> 3) * 1024 + (row & 7) * 128;
  if constexpr (F == kFmtBF16) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int chunk = (col0 >> 3) + q;
      *reinterpret_cast<uint4*>(base + (((chunk ^ (row & 7)) & 7) << 4)) =
          make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                     pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int chunk = (col0 >> 2) + q;
      const uint32_t off = (((chunk ^ (row & 7)) & 7) << 4);
      const float4 h = make_float4(tf32_rna(v[4 * q]), tf32_rna(v[4 * q + 1]), tf32_rna(v[4 * q + 2]),
                                   tf32_rna(v[4 * q + 3]));
      *reinterpret_cast<float4*>(base + off) = h;
      if constexpr (F == kFmtTF32x2)
        *reinterpret_cast<float4*>(base + g.bytes_part() + off) =
            make_float4(tf32_rna(v[4 * q] - h.x), tf32_rna(v[4 * q + 1] - h.y), tf32_rna(v[4 * q + 2] - h.z),
                        tf32_rna(v[4 * q + 3] - h.w));
    }
  }
}

// One pass (forward, grad A or grad B) over the tile of 128 own rows of sample
// blockIdx.y; see the file comment. Warp specialised, with mbarrier hand-offs only:
//   warp 8, one thread: the TMA loads (a ring of R chunk stages), ahead of the MMAs;
//   warp 9, one thread: every MMA;
//   warps 0..7: consumers; warp w reads TMEM lane quarter w & 3 and handles columns
//   16 (w >> 2) .. +15 of every 32-column chunk.
// (With one thread doing both, each chunk's copy was issued only after the previous
// chunk's MMA and then waited for at once: copy, MMA and hand-off ran in series, and the
// consumers sat idle half of every chunk.)
// Barriers: mbT[stage] chunk landed; mbE[stage] the consumers are done with the stage;
// mbGT / mbGE[slot] a gradient B-operand tile landed / read by its MMA; mbS[c & 1] S of
// chunk c in TMEM; mbF[c & 1] all eight consumer warps are done with chunk c's S slot;
// mbDf[c & 1] chunk c's D tile is written; mbG[c & 1] the gradient MMA of chunk c is done.
// (The forward's shared memory leaves room for two CTAs per SM; its launch bounds ask the
// compiler for registers that allow two as well.)
template <int P, int Mode>
__global__ void __launch_bounds__(kLrThreadsFused, 2)
    k_lowrank(const __grid_constant__ LrMaps maps, const LrArgs a) {
  constexpr int SF = s_fmt(P), GF = g_fmt(P);
  constexpr bool kGrad = Mode != kLrFwd;
  constexpr int kNvec = lr_nvec(Mode);
  constexpr int esS = fmt_bytes(SF);
  const int K = a.K;
  const int Kp = (K + 15) & ~15;
  const int own_n = Mode == kLrGradB ? a.N : a.M;
  const int sw_n = Mode == kLrGradB ? a.M : a.N;
  const int b = blockIdx.y;
  const int o0 = blockIdx.x * kLrRows;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int quarter = warp & 3, half = (warp >> 2) & 1;
  const int row = quarter * 32 + lane;  // own row in the tile (TMEM lane)
  const int col0 = half * 16;           // this thread's columns of a chunk
  const int own = o0 + row;
  const STile so = s_tile(SF, kLrRows, K), ss = s_tile(SF, kLrChunk, K);
  const TileGeo go = so.g, gs = ss.g;
  const TileGeo gd = tile_geo(GF, kLrRows, kLrChunk), gg = tile_geo(GF, Kp, kLrChunk);
  const LrSmem L = lr_smem(P, Mode, K);
  const int R = L.nstage, ND = L.nd, NG = L.ngb;
  // TMEM: two 32-column S slots, then (gradients) kGradAccs accumulators of gstride
  // columns that the chunks take in turn: each sums a quarter of the sweep, which keeps
  // the accumulator's truncations to a quarter; the epilogue adds them up.
  const int gstride = (Kp + 31) & ~31;
  const uint32_t tcols = !kGrad ? 64u : (64 + kGradAccs * gstride <= 128 ? 128u
                                         : (64 + kGradAccs * gstride <= 256 ? 256u : 512u));

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* own_tile = smem + L.own;
  uint64_t* mbT = reinterpret_cast<uint64_t*>(smem + L.bars);  // [R <= 4]
  uint64_t* mbS = mbT + 4;                                      // [2]
  uint64_t* mbF = mbS + 2;                                      // [2]
  uint64_t* mbDf = mbF + 2;                                     // [2]
  uint64_t* mbG = mbDf + 2;                                     // [2]
  uint64_t* mbO = mbG + 2;                                      // own tile landed
  uint64_t* mbE = mbO + 1;                                      // [R <= 4] stage free
  uint64_t* mbGT = mbE + 4;                                     // [NG <= 4] B-operand tile landed
  uint64_t* mbGE = mbGT + 4;                                    // [NG <= 4] B-operand tile free
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mbGE + 4);
  float* merge = reinterpret_cast<float*>(smem + L.bars + 256);  // [3][128]
  auto stage = [&](int c) { return smem + L.stage + (c % R) * L.stage_bytes; };
  // A bf16 D tile is 32 columns = 64 bytes of each 128-byte row: with two slots, slot 1
  // takes the second half of the rows of the same tile (its k-steps 2 and 3), which the
  // consumers address as columns 32 .. 63 and the MMA by a 64-byte start offset.
  constexpr bool kDPair = GF == kFmtBF16;
  auto d_tile = [&](int c) {
    return kDPair ? smem + L.d + (c % ND) * 64 : smem + L.d + (c % ND) * L.d_bytes;
  };
  auto d_col = [&](int c) { return kDPair ? (c % ND) * 32 : 0; };
  auto gb_tile = [&](int c) { return smem + L.gbr + (c % NG) * L.gb_bytes; };

  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < 4; ++i) {
        mbar_init(&mbT[i], 1);
        mbar_init(&mbE[i], kLrWarps);
        mbar_init(&mbGT[i], 1);
        mbar_init(&mbGE[i], 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&mbS[i], 1);
        mbar_init(&mbF[i], kLrWarps);
        mbar_init(&mbDf[i], kLrWarps);
        mbar_init(&mbG[i], 1);
      }
      mbar_init(mbO, 1);
      fence_barrier_init();
    }
    __syncwarp();
    tmem_alloc(tslot, tcols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const int nch = (sw_n + kLrChunk - 1) / kLrChunk;
  bool ok = true;

  // Each barrier below has one waiter role, and no role can fall two phases behind on a
  // barrier it waits on (the phase after the one it waits for needs the waiter's own next
  // step), so a parity wait never aliases onto a later phase.
  if (warp == kLrWarps) {
    // -------------------------------------------------------------- TMA producer
    // Runs ahead of the MMAs as far as the rings allow: chunk c's stage is refilled as
    // soon as the consumers of chunk c - R have released it (mbE), and its gradient
    // B-operand tile, which only the gradient MMA reads, travels in a ring of its own
    // (mbGT landed, mbGE read), so a stage never waits for a gradient MMA.
    if (lane == 0) {
      int issued = -1, gb_issued = -1;
      auto issue_tma = [&](int c) {
        uint8_t* st = stage(c);
        uint64_t* bar = &mbT[c % R];
        const int w0 = c * kLrChunk;
        mbar_arrive_expect_tx(bar, L.tx_bytes);
        for (int part = 0; part < ss.parts; ++part)
          for (int kb = 0; kb < gs.kblocks; ++kb)
            tma_load_3d(st + L.sw_off + part * gs.bytes_part() + kb * kLrChunk * 128, &maps.sw[part], bar,
                        kb * (128 / esS), w0, b);
        tma_load_3d(st + L.th_off, &maps.th, bar, w0, o0, 0);
        for (int v = 0; v < kNvec; ++v) tma_load_3d(st + L.vec_off + v * 128, &maps.vec[v], bar, w0, b, 0);
        issued = c;
      };
      auto issue_gb = [&](int c) {
        uint64_t* bar = &mbGT[c % NG];
        mbar_arrive_expect_tx(bar, L.gb_bytes);
        for (int part = 0; part < fmt_parts(GF); ++part)
          tma_load_3d(gb_tile(c) + part * gg.bytes_part(), &maps.gb[part], bar, c * kLrChunk, 0, b);
        gb_issued = c;
      };
      mbar_arrive_expect_tx(mbO, L.own_bytes);
      for (int part = 0; part < so.parts; ++part)
        for (int kb = 0; kb < go.kblocks; ++kb)
          tma_load_3d(own_tile + part * go.bytes_part() + kb * kLrRows * 128, &maps.own[part], mbO,
                      kb * (128 / esS), o0, b);
      for (int c = 0; c < nch; ++c) {
        if (c >= R) ok = mbar_wait(&mbE[c % R], ((c / R) - 1) & 1, a.status, kErrTimeoutMma);
        if (!ok) break;
        issue_tma(c);
        if constexpr (kGrad) {
          if (c >= NG) ok = mbar_wait(&mbGE[c % NG], ((c / NG) - 1) & 1, a.status, kErrTimeoutMma);
          if (!ok) break;
          issue_gb(c);
        }
      }
      if (!ok) {
        // a wait gave up: let the copies in flight land before the block exits
        mbar_wait(mbO, 0, a.status, kErrTimeoutDrain);
        for (int c = issued; c >= 0 && c > issued - R; --c)
          mbar_wait(&mbT[c % R], (c / R) & 1, a.status, kErrTimeoutDrain);
        for (int c = gb_issued; c >= 0 && c > gb_issued - NG; --c)
          mbar_wait(&mbGT[c % NG], (c / NG) & 1, a.status, kErrTimeoutDrain);
      }
    }
    ok = __all_sync(0xffffffffu, ok);
  } else if (warp == kLrWarps + 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int s_issued = -1, g_issued = -1;
      auto issue_grad = [&](int c) {  // the D tile of chunk c is written, its B-operand landed
        ok = ok && mbar_wait(&mbDf[c & 1], (c >> 1) & 1, a.status, kErrTimeoutMma) &&
             mbar_wait(&mbGT[c % NG], (c / NG) & 1, a.status, kErrTimeoutMma);
        if (!ok) return;
        tc_fence_after();
        lr_mma<GF>(tmem + static_cast<uint32_t>(64 + (c % kGradAccs) * gstride), d_tile(c), gd, gb_tile(c), gg, Kp,
                   c >= kGradAccs, gd.bytes_part(), gg.bytes_part());
        umma_commit(&mbG[c & 1]);
        umma_commit(&mbGE[c % NG]);  // the B-operand tile has been read
        g_issued = c;
      };
      ok = mbar_wait(mbO, 0, a.status, kErrTimeoutMma);
      for (int c = 0; c < nch && ok; ++c) {
        ok = mbar_wait(&mbT[c % R], (c / R) & 1, a.status, kErrTimeoutMma);
        // the TMEM slot of chunk c - 2 is free once its consumers are done
        if (ok && c >= 2) ok = mbar_wait(&mbF[c & 1], ((c - 2) >> 1) & 1, a.status, kErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        lr_mma<SF>(tmem + static_cast<uint32_t>((c & 1) * kLrChunk), own_tile, go, stage(c) + L.sw_off, gs, kLrChunk,
                   false, so.lo_off, ss.lo_off);
        umma_commit(&mbS[c & 1]);
        s_issued = c;
        if constexpr (kGrad) {
          if (c >= 1) issue_grad(c - 1);
        }
      }
      if (kGrad && ok && nch > 0) issue_grad(nch - 1);
      if (!ok) {
        // a wait gave up: let the MMAs in flight finish before TMEM is freed
        if (s_issued >= 0) mbar_wait(&mbS[s_issued & 1], (s_issued >> 1) & 1, a.status, kErrTimeoutDrain);
        if (g_issued >= 0) mbar_wait(&mbG[g_issued & 1], (g_issued >> 1) & 1, a.status, kErrTimeoutDrain);
      }
    }
    ok = __all_sync(0xffffffffu, ok);
  } else {
    // ---------------------------------------------------------------- consumers
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float lz = 0.f, fi = 0.f, fc = 0.f, uj = 0.f;
    if constexpr (Mode == kLrGradB) uj = own < a.N ? a.u[static_cast<long long>(b) * a.ldu + own] : 0.f;
    if constexpr (Mode == kLrGradA) {
      if (own < a.M) {
        const long long r = static_cast<long long>(b) * a.ldm + own;
        lz = a.rf_lz[r];
        fi = a.rf_f[r];
        fc = a.rf_fc[r];
      }
    }
    const bool row_live = lz > -INFINITY;
    float run = -INFINITY, Z = 0.f, num = 0.f;  // forward
    float e_acc = 0.f;                          // grad B
    for (int c = 0; c < nch; ++c) {
      bool w = mbar_wait(&mbS[c & 1], (c >> 1) & 1, a.status, kErrTimeoutEpilogue) &&
               mbar_wait(&mbT[c % R], (c / R) & 1, a.status, kErrTimeoutEpilogue);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[16], th[16], va[16], vb[16], vc[16];
      tmem_ld_32x16(lane_base + static_cast<uint32_t>((c & 1) * kLrChunk + col0), v);
      const uint8_t* st = stage(c);
      tile_row16_f32(st + L.th_off, row, col0, th);
      const float* vec = reinterpret_cast<const float*>(st + L.vec_off);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        va[jj] = vec[col0 + jj];
        if constexpr (Mode == kLrGradB) {
          vb[jj] = vec[32 + col0 + jj];
          vc[jj] = vec[64 + col0 + jj];
        }
      }
      // Chunk c's S slot and stage are released (mbF) only after the values read from them
      // have been used: the stage's next fill is an async-proxy write, which the arrival
      // alone does not order after these generic-proxy reads.
      auto release_chunk = [&]() {
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&mbF[c & 1]);
          mbar_arrive(&mbE[c % R]);
        }
      };
      const int w0 = c * kLrChunk + col0;
      if constexpr (Mode == kLrFwd) {
        float cm = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          if (w0 + jj < a.N) cm = fmaxf(cm, v[jj]);
        if (cm > run) {
          const float sc = run > -INFINITY ? ex2_approx((run - cm) * kLog2e) : 0.f;
          Z *= sc;
          num *= sc;
          run = cm;
        }
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const float tg = w0 + jj < a.N ? th[jj] * ex2_approx((v[jj] - run) * kLog2e) : 0.f;
          Z += tg;
          num = fmaf(tg, va[jj], num);
        }
        release_chunk();
      } else {
        float dv[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          if constexpr (Mode == kLrGradA) {
            const float q = (row_live && th[jj] > 0.f) ? th[jj] * ex2_approx((v[jj] - lz) * kLog2e) : 0.f;
            dv[jj] = q * fmaf(va[jj], fc, -fi);
          } else {
            const float lzi = va[jj];
            const float q = (lzi > -INFINITY && th[jj] > 0.f) ? th[jj] * ex2_approx((v[jj] - lzi) * kLog2e) : 0.f;
            const float pf = q * uj * vc[jj];
            e_acc += pf;
            dv[jj] = pf - q * vb[jj];
          }
          if (own >= own_n) dv[jj] = 0.f;
        }
        release_chunk();
        // the D slot was read by the gradient MMA of chunk c - ND
        if (c >= ND) {
          const int pc = c - ND;
          w = __all_sync(0xffffffffu, mbar_wait(&mbG[pc & 1], (pc >> 1) & 1, a.status, kErrTimeoutEpilogue));
          if (!w) {
            ok = false;
            break;
          }
        }
        tile_put_row16<GF>(smem + L.d + (kDPair ? 0 : (c % ND) * L.d_bytes), gd, row, col0 + d_col(c), dv);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&mbDf[c & 1]);
      }
    }
    if (ok && kGrad && nch > 0) {
      const int lc = nch - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&mbG[lc & 1], (lc >> 1) & 1, a.status, kErrTimeoutEpilogue));
    }
    // merge the two column halves of each row (consumer warps only)
    if (half == 1) {
      merge[row] = run;
      merge[128 + row] = Z;
      merge[256 + row] = Mode == kLrGradB ? e_acc : num;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kLrWarps * 32) : "memory");
    if (ok && half == 0) {
      if constexpr (Mode == kLrFwd) {
        if (own < a.M) {
          const float r1 = merge[row], z1 = merge[128 + row], n1 = merge[256 + row];
          const float r = fmaxf(run, r1);
          float zt = 0.f, nt = 0.f;
          if (r > -INFINITY) {
            const float s0 = run > -INFINITY ? ex2_approx((run - r) * kLog2e) : 0.f;
            const float s1 = r1 > -INFINITY ? ex2_approx((r1 - r) * kLog2e) : 0.f;
            zt = Z * s0 + z1 * s1;
            nt = num * s0 + n1 * s1;
          }
          const float mb = a.m[b];
          const bool live = zt > 0.f && nt > 0.f && mb > -INFINITY;
          a.out[static_cast<long long>(own) * a.B + b] = live ? mb + logf(nt / zt) : -INFINITY;
          a.logZ[static_cast<long long>(b) * a.M + own] = zt > 0.f ? logf(zt) + r : -INFINITY;
        }
      } else {
        tc_fence_after();
        float acc[64];  // static indices only: kept in registers
#pragma unroll
        for (int r = 0; r < 64; ++r) acc[r] = 0.f;
        for (int q = 0; q < kGradAccs && q < nch; ++q) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            if (h2 * 32 < Kp) {
              float v[32];
              tmem_ld_32x32(lane_base + static_cast<uint32_t>(64 + q * gstride + h2 * 32), v);
#pragma unroll
              for (int r = 0; r < 32; ++r) acc[h2 * 32 + r] += v[r];
            }
          }
        }
        if (own < own_n) {
          if constexpr (Mode == kLrGradA) {
            float* dst = a.dA + (static_cast<long long>(b) * a.M + own) * K;
#pragma unroll
            for (int r = 0; r < 64; ++r)
              if (r < K) dst[r] = a.accumulate ? dst[r] + acc[r] : acc[r];
          } else {
            if (a.dB) {
#pragma unroll
              for (int r = 0; r < 64; ++r) {
                if (r < K) {
                  float* dst = a.dB + (static_cast<long long>(b) * K + r) * a.N + own;
                  *dst = a.accumulate ? *dst + acc[r] : acc[r];
                }
              }
            }
            if (a.e) {
              const float ev = e_acc + merge[256 + row];
              float* de = a.e + static_cast<long long>(own) * a.B + b;
              *de = a.accumulate ? *de + ev : ev;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

// Parameter-flow statistics F+ and W over all samples for the 128 x 32 tile (blockIdx.x,
// blockIdx.y) of [M, N]: own rows i, the 32 columns j fixed, a sweep over the samples.
// Each stage of the TMA ring holds one sample's A_b tile, its B_b^T chunk and u_b. Warp
// specialised as k_lowrank: warp 8 issues the copies, warp 9 the MMAs, warps 0..7 consume.
template <int P>
__global__ void __launch_bounds__(kLrThreadsFused, 2)
    k_lowrank_stats(const __grid_constant__ LrMaps maps, const LrArgs a) {
  constexpr int SF = s_fmt(P);
  constexpr int esS = fmt_bytes(SF);
  const int K = a.K;
  const int i0 = blockIdx.x * kLrRows, j0 = blockIdx.y * kLrChunk;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int quarter = warp & 3, half = (warp >> 2) & 1;
  const int row = quarter * 32 + lane;
  const int col0 = half * 16;
  const int i = i0 + row;
  const STile so = s_tile(SF, kLrRows, K), ss = s_tile(SF, kLrChunk, K);
  const TileGeo go = so.g, gs = ss.g;
  const LrSmem L = lr_smem(P, kLrStats, K);
  const int R = L.nstage;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* mbT = reinterpret_cast<uint64_t*>(smem + L.bars);  // [R <= 4]
  uint64_t* mbS = mbT + 4;                                      // [2]
  uint64_t* mbF = mbS + 2;                                      // [2]
  uint64_t* mbE = mbF + 2;                                      // [R <= 4] stage free
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mbE + 4);
  auto stage = [&](int b) { return smem + L.stage + (b % R) * L.stage_bytes; };

  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < 4; ++s) {
        mbar_init(&mbT[s], 1);
        mbar_init(&mbE[s], kLrWarps);
      }
      for (int s = 0; s < 2; ++s) {
        mbar_init(&mbS[s], 1);
        mbar_init(&mbF[s], kLrWarps);
      }
      fence_barrier_init();
    }
    __syncwarp();
    tmem_alloc(tslot, 64);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = true;

  // The same roles as k_lowrank: a TMA producer that refills a stage as soon as its
  // consumers release it (mbE), and an MMA warp.
  if (warp == kLrWarps) {
    if (lane == 0) {
      int issued = -1;
      auto issue_tma = [&](int b) {
        uint8_t* st = stage(b);
        uint64_t* bar = &mbT[b % R];
        mbar_arrive_expect_tx(bar, L.tx_bytes);
        for (int part = 0; part < so.parts; ++part) {  // so.parts == ss.parts
          for (int kb = 0; kb < go.kblocks; ++kb)
            tma_load_3d(st + part * go.bytes_part() + kb * kLrRows * 128, &maps.own[part], bar, kb * (128 / esS), i0,
                        b);
          for (int kb = 0; kb < gs.kblocks; ++kb)
            tma_load_3d(st + L.sw_off + part * gs.bytes_part() + kb * kLrChunk * 128, &maps.sw[part], bar,
                        kb * (128 / esS), j0, b);
        }
        tma_load_3d(st + L.vec_off, &maps.vec[0], bar, j0, b, 0);
        issued = b;
      };
      for (int b = 0; b < a.B; ++b) {
        if (b >= R) ok = mbar_wait(&mbE[b % R], ((b / R) - 1) & 1, a.status, kErrTimeoutMma);
        if (!ok) break;
        issue_tma(b);
      }
      if (!ok)
        for (int b = issued; b >= 0 && b > issued - R; --b)
          mbar_wait(&mbT[b % R], (b / R) & 1, a.status, kErrTimeoutDrain);
    }
    ok = __all_sync(0xffffffffu, ok);
  } else if (warp == kLrWarps + 1) {
    if (lane == 0) {
      int s_issued = -1;
      for (int b = 0; b < a.B && ok; ++b) {
        ok = mbar_wait(&mbT[b % R], (b / R) & 1, a.status, kErrTimeoutMma);
        // the TMEM slot of sample b - 2 is free once its consumers are done
        if (ok && b >= 2) ok = mbar_wait(&mbF[b & 1], ((b - 2) >> 1) & 1, a.status, kErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        lr_mma<SF>(tmem + static_cast<uint32_t>((b & 1) * kLrChunk), stage(b), go, stage(b) + L.sw_off, gs,
                   kLrChunk, false, so.lo_off, ss.lo_off);
        umma_commit(&mbS[b & 1]);
        s_issued = b;
      }
      if (!ok && s_issued >= 0) mbar_wait(&mbS[s_issued & 1], (s_issued >> 1) & 1, a.status, kErrTimeoutDrain);
    }
    ok = __all_sync(0xffffffffu, ok);
  } else {
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    // theta[i][j0 + col0 .. +15] in registers, from the row-padded copy
    float th[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const int j = j0 + col0 + jj;
      th[jj] = (i < a.M && j < a.N) ? a.theta_ld[static_cast<long long>(i) * a.theta_ld_stride + j] : 0.f;
    }
    float fp[16], wst[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) fp[jj] = wst[jj] = 0.f;
    auto row_factors = [&](int b, float& lz, float& fi, float& fc) {
      lz = -INFINITY;
      fi = fc = 0.f;
      if (i < a.M && b < a.B) {
        const long long r = static_cast<long long>(b) * a.ldm + i;
        lz = a.rf_lz[r];
        fi = a.rf_f[r];
        fc = a.rf_fc[r];
      }
    };
    float lz, fi, fc;
    row_factors(0, lz, fi, fc);
    for (int b = 0; b < a.B; ++b) {
      float nlz, nfi, nfc;  // the next sample's row factors, loaded while this one computes
      row_factors(b + 1, nlz, nfi, nfc);
      const bool w = __all_sync(0xffffffffu, mbar_wait(&mbS[b & 1], (b >> 1) & 1, a.status, kErrTimeoutEpilogue) &&
                                                 mbar_wait(&mbT[b % R], (b / R) & 1, a.status, kErrTimeoutEpilogue));
      if (!w) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[16], us[16];
      tmem_ld_32x16(lane_base + static_cast<uint32_t>((b & 1) * kLrChunk + col0), v);
      const float* uv = reinterpret_cast<const float*>(stage(b) + L.vec_off) + col0;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) us[jj] = uv[jj];
      if (lz > -INFINITY) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const float gz = ex2_approx((v[jj] - lz) * kLog2e);  // g_b / Z_b
          fp[jj] = fmaf(th[jj] * gz, us[jj] * fc, fp[jj]);
          wst[jj] = fmaf(fi, gz, wst[jj]);
        }
      }
      // the stage and S slot are released after their values are used (see k_lowrank)
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&mbF[b & 1]);
        mbar_arrive(&mbE[b % R]);
      }
      lz = nlz;
      fi = nfi;
      fc = nfc;
    }
    if (ok && i < a.M) {
      for (int jj = 0; jj < 16; ++jj) {
        const int j = j0 + col0 + jj;
        if (j >= a.N) break;
        const long long idx = static_cast<long long>(i) * a.N + j;
        if (a.Fp) a.Fp[idx] = a.accumulate ? a.Fp[idx] + fp[jj] : fp[jj];
        if (a.W) a.W[idx] = a.accumulate ? a.W[idx] + wst[jj] : wst[jj];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// ------------------------------------------------------------------------ host side
__global__ void k_lr_fill(float* __restrict__ p, long long n, float v) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}

// An operand matrix in format F: one Operand per part (hi, lo), element type bf16 or fp32.
struct LrOp {
  Operand part[2];
  int parts = 0;
  pc_precision_t ety = PC_PREC_TF32;
  long long packed_lo = 0;  // packed (lr_packed): the lo values start this many elements into a row
};
// pack: an S operand (K = cols), which may take the packed layout
LrOp carve_op(Carver& c, int F, long long groups, long long rows, long long cols, bool pack = false) {
  LrOp o;
  o.ety = fmt_bytes(F) == 2 ? PC_PREC_AUTO : PC_PREC_TF32;
  if (pack && lr_packed(F, static_cast<int>(cols))) {  // one array of rows [hi | lo]
    o.parts = 1;
    o.packed_lo = cols;
    o.part[0] = c.operand(o.ety, groups, rows, 2 * cols);
    return o;
  }
  o.parts = fmt_parts(F);
  for (int p = 0; p < o.parts; ++p) o.part[p] = c.operand(o.ety, groups, rows, cols);
  return o;
}
void* op_lo(const LrOp& o) {
  if (o.packed_lo)
    return static_cast<uint8_t*>(o.part[0].ptr) + o.packed_lo * (o.ety == PC_PREC_AUTO ? 2 : 4);
  return o.parts > 1 ? o.part[1].ptr : nullptr;
}

struct LrWs {
  float* m;
  Operand u;                            // [B][N] exp(x - m_b), padded rows
  Operand theta, thetaT;                // float32 theta (the caller's rows when 16-byte aligned,
                                        // else a padded copy) and a padded transposed copy
  Operand rf_lz, rf_f, rf_fc;           // [B][M] backward row factors
  LrOp Aop, BTop;                       // A_b rows, B_b^T rows (format of S)
  LrOp Bg, AgT;                         // B_b rows, A_b^T rows (format of the gradients)
};

size_t carve_lr(void* base, pc_precision_t prec, int M, int N, int K, int B, bool bwd, LrWs* w) {
  const int P = prec == PC_PREC_AUTO ? kBF16 : (prec == PC_PREC_TF32 ? kTF32 : kTF32x3);
  Carver c(base);
  *w = LrWs{};
  w->m = static_cast<float*>(c.take(size_t(B) * 4));
  w->u = c.operand(PC_PREC_TF32, 1, B, N);
  w->theta = c.operand(PC_PREC_TF32, 1, M, N);
  w->Aop = carve_op(c, s_fmt(P), B, M, K, true);
  w->BTop = carve_op(c, s_fmt(P), B, N, K, true);
  if (bwd) {
    w->thetaT = c.operand(PC_PREC_TF32, 1, N, M);
    w->rf_lz = c.operand(PC_PREC_TF32, 1, B, M);
    w->rf_f = c.operand(PC_PREC_TF32, 1, B, M);
    w->rf_fc = c.operand(PC_PREC_TF32, 1, B, M);
    w->Bg = carve_op(c, g_fmt(P), B, K, N);
    w->AgT = carve_op(c, g_fmt(P), B, K, M);
  }
  return c.used + 256;
}

pc_status_t check_lr_shape(int M, int N, int K, int B, pc_precision_t prec) {
  pc_status_t st = check_precision(prec);
  if (st != PC_OK) return st;
  PC_CHECK(M >= 0 && N >= 0 && B >= 0, PC_ERR_SHAPE, "negative size (M=%d N=%d B=%d)", M, N, B);
  PC_CHECK(K >= 1, PC_ERR_SHAPE, "rank K=%d must be at least 1", K);
  PC_CHECK(K <= kLrMaxRank, PC_ERR_UNSUPPORTED, "rank K=%d exceeds the fused kernels' limit of %d", K,
           kLrMaxRank);
  PC_CHECK(B <= 65535, PC_ERR_SHAPE, "batch B=%d exceeds 65535", B);
  PC_CHECK(static_cast<long long>(N) <= 65535LL * kLrChunk, PC_ERR_SHAPE, "N=%d too large", N);
  return PC_OK;
}

template <class Kern>
pc_status_t lr_attr(Kern kern, int smem) {
  PC_CHECK(smem <= 232448, PC_ERR_UNSUPPORTED, "LowRank kernel needs %d bytes of shared memory", smem);
  PC_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  return PC_OK;
}

template <int F>
pc_status_t to_op(const float* src, long long sg, long long sr, long long sc, int G, int R, int C, const LrOp& o,
                  cudaStream_t s) {
  if (sr == 1 && sc != 1 && G <= 65535) {  // a transpose: tiled through shared memory
    const dim3 grid(cdiv(R, 32), cdiv(C, 32), G);
    k_lr_to_op_t<F><<<grid, dim3(32, 8), 0, s>>>(src, sg, sc, G, R, C, o.part[0].ptr,
                                                 op_lo(o), o.part[0].ld);
    PC_LAUNCH_CHECK();
    return PC_OK;
  }
  const long long rows = static_cast<long long>(G) * R;
  if (sc == 1 && C % 4 == 0 && sr % 4 == 0 && sg % 4 == 0 && aligned16(src) && o.part[0].ld % 4 == 0) {
    const int blocks = static_cast<int>(std::min<long long>(cdiv(rows * (C / 4), 256), 65535));
    k_lr_to_op4<F><<<blocks, 256, 0, s>>>(src, sg, sr, R, C / 4, rows, o.part[0].ptr,
                                          op_lo(o), o.part[0].ld);
    PC_LAUNCH_CHECK();
    return PC_OK;
  }
  const int blocks = static_cast<int>(std::min<long long>(cdiv(rows, 8), 8192));
  k_lr_to_op<F><<<blocks, dim3(32, 8), 0, s>>>(src, sg, sr, sc, G, R, C, o.part[0].ptr,
                                               op_lo(o), o.part[0].ld);
  PC_LAUNCH_CHECK();
  return PC_OK;
}

pc_status_t encode_op(CUtensorMap (&maps)[2], const LrOp& o, int box_rows) {
  for (int p = 0; p < o.parts; ++p) {
    const pc_status_t st = encode_operand_map(&maps[p], o.part[p], o.ety, box_rows, 0);
    if (st != PC_OK) return st;
  }
  if (o.parts == 1) maps[1] = maps[0];
  return PC_OK;
}

// Set-up shared by both passes: m, u, theta's tensor-map rows (and its transposed copy) and
// the operand copies of A, B.
template <int P>
pc_status_t lr_prepare(const float* theta, const float* A, const float* Bm, const float* x, int M, int N, int K,
                       int B, bool bwd, LrWs& w, cudaStream_t s) {
  k_lr_colmax_u<<<B, 256, 0, s>>>(N, B, x, w.m, static_cast<float*>(w.u.ptr), w.u.ld);
  PC_LAUNCH_CHECK();
  const dim3 g(cdiv(N, 32), cdiv(M, 32));
  if (N % 4 == 0 && aligned16(theta)) {  // theta's own rows are a tensor map's rows: no copy
    w.theta.ptr = const_cast<float*>(theta);
    w.theta.ld = N;
  } else {
    k_lr_theta_copy<<<g, dim3(32, 8), 0, s>>>(M, N, theta, static_cast<float*>(w.theta.ptr), w.theta.ld, 0);
    PC_LAUNCH_CHECK();
  }
  const long long MK = static_cast<long long>(M) * K, KN = static_cast<long long>(K) * N;
  pc_status_t st;
  if ((st = to_op<s_fmt(P)>(A, MK, K, 1, B, M, K, w.Aop, s)) != PC_OK) return st;    // A_b[i][k]
  if ((st = to_op<s_fmt(P)>(Bm, KN, 1, N, B, N, K, w.BTop, s)) != PC_OK) return st;  // B_b[k][j] as [j][k]
  if (bwd) {
    k_lr_theta_copy<<<g, dim3(32, 8), 0, s>>>(M, N, theta, static_cast<float*>(w.thetaT.ptr), w.thetaT.ld, 1);
    PC_LAUNCH_CHECK();
    if ((st = to_op<g_fmt(P)>(Bm, KN, N, 1, B, K, N, w.Bg, s)) != PC_OK) return st;   // B_b[k][j]
    if ((st = to_op<g_fmt(P)>(A, MK, 1, K, B, K, M, w.AgT, s)) != PC_OK) return st;   // A_b[i][k] as [k][i]
  }
  return PC_OK;
}

template <int P>
pc_status_t lr_fwd(int M, int N, int K, int B, const float* theta, const float* A, const float* Bm, const float* x,
                   float* out, float* logZ, void* ws, cudaStream_t s) {
  LrWs w;
  carve_lr(ws, static_cast<pc_precision_t>(P == kBF16 ? PC_PREC_AUTO : (P == kTF32 ? PC_PREC_TF32 : PC_PREC_FP32)),
           M, N, K, B, false, &w);
  if (M == 0 || B == 0) return PC_OK;
  if (N == 0) {  // no children: every node's sum is empty
    k_lr_fill<<<cdiv(static_cast<long long>(M) * B, 256), 256, 0, s>>>(out, static_cast<long long>(M) * B, -INFINITY);
    PC_LAUNCH_CHECK();
    k_lr_fill<<<cdiv(static_cast<long long>(M) * B, 256), 256, 0, s>>>(logZ, static_cast<long long>(M) * B, -INFINITY);
    PC_LAUNCH_CHECK();
    return PC_OK;
  }
  pc_status_t st = lr_prepare<P>(theta, A, Bm, x, M, N, K, B, false, w, s);
  if (st != PC_OK) return st;
  LrMaps maps;
  if ((st = encode_op(maps.own, w.Aop, kLrRows)) != PC_OK) return st;
  if ((st = encode_op(maps.sw, w.BTop, kLrChunk)) != PC_OK) return st;
  maps.gb[0] = maps.gb[1] = maps.sw[0];  // unused
  if ((st = encode_operand_map(&maps.th, w.theta, PC_PREC_TF32, kLrRows, 0)) != PC_OK) return st;
  if ((st = encode_operand_map(&maps.vec[0], w.u, PC_PREC_TF32, 1, 0, false)) != PC_OK) return st;
  maps.vec[1] = maps.vec[2] = maps.vec[0];
  LrArgs a{};
  a.M = M; a.N = N; a.K = K; a.B = B;
  a.m = w.m;
  a.out = out; a.logZ = logZ;
  a.status = device_status_word();
  const int smem = lr_smem(P, kLrFwd, K).total;
  if ((st = lr_attr(k_lowrank<P, kLrFwd>, smem)) != PC_OK) return st;
  const int slot = profile_begin(s);
  k_lowrank<P, kLrFwd><<<dim3(cdiv(M, kLrRows), B), kLrThreadsFused, smem, s>>>(maps, a);
  PC_LAUNCH_CHECK();
  profile_end(slot, s, PC_KIND_LOWRANK_FWD, 2LL * M * N * K * B);
  return PC_OK;
}

template <int P>
pc_status_t lr_bwd(int M, int N, int K, int B, const float* theta, const float* A, const float* Bm, const float* x,
                   const float* out, const float* logZ, const float* f, float* dA, float* dB, float* e, float* Fp,
                   float* W, int accumulate, void* ws, cudaStream_t s) {
  LrWs w;
  carve_lr(ws, static_cast<pc_precision_t>(P == kBF16 ? PC_PREC_AUTO : (P == kTF32 ? PC_PREC_TF32 : PC_PREC_FP32)),
           M, N, K, B, true, &w);
  if (!accumulate) {  // outputs that no pass writes when a size is zero
    if (dA && N == 0) PC_CUDA(cudaMemsetAsync(dA, 0, size_t(B) * M * K * 4, s));
    if (dB && M == 0) PC_CUDA(cudaMemsetAsync(dB, 0, size_t(B) * K * N * 4, s));
    if (e && M == 0) PC_CUDA(cudaMemsetAsync(e, 0, size_t(N) * B * 4, s));
    if (Fp && B == 0) PC_CUDA(cudaMemsetAsync(Fp, 0, size_t(M) * N * 4, s));
    if (W && B == 0) PC_CUDA(cudaMemsetAsync(W, 0, size_t(M) * N * 4, s));
  }
  if (M == 0 || N == 0 || B == 0) return PC_OK;
  pc_status_t st = lr_prepare<P>(theta, A, Bm, x, M, N, K, B, true, w, s);
  if (st != PC_OK) return st;
  k_lr_row_factors<<<cdiv(static_cast<long long>(M) * B, 256), 256, 0, s>>>(
      M, B, out, f, logZ, w.m, static_cast<float*>(w.rf_lz.ptr), static_cast<float*>(w.rf_f.ptr),
      static_cast<float*>(w.rf_fc.ptr), w.rf_lz.ld);
  PC_LAUNCH_CHECK();
  LrArgs a{};
  a.M = M; a.N = N; a.K = K; a.B = B;
  a.m = w.m;
  a.rf_lz = static_cast<const float*>(w.rf_lz.ptr);
  a.rf_f = static_cast<const float*>(w.rf_f.ptr);
  a.rf_fc = static_cast<const float*>(w.rf_fc.ptr);
  a.ldm = w.rf_lz.ld;
  a.theta_ld = static_cast<const float*>(w.theta.ptr);
  a.theta_ld_stride = w.theta.ld;
  a.u = static_cast<const float*>(w.u.ptr);
  a.ldu = w.u.ld;
  a.dA = dA; a.dB = dB; a.e = e; a.Fp = Fp; a.W = W;
  a.accumulate = accumulate;
  a.status = device_status_word();
  const long long flops = 2LL * M * N * K * B;
  const int Kp = (K + 15) & ~15;
  if (dA) {
    LrMaps maps;
    if ((st = encode_op(maps.own, w.Aop, kLrRows)) != PC_OK) return st;
    if ((st = encode_op(maps.sw, w.BTop, kLrChunk)) != PC_OK) return st;
    if ((st = encode_op(maps.gb, w.Bg, Kp)) != PC_OK) return st;
    if ((st = encode_operand_map(&maps.th, w.theta, PC_PREC_TF32, kLrRows, 0)) != PC_OK) return st;
    if ((st = encode_operand_map(&maps.vec[0], w.u, PC_PREC_TF32, 1, 0, false)) != PC_OK) return st;
    maps.vec[1] = maps.vec[2] = maps.vec[0];
    const int smem = lr_smem(P, kLrGradA, K).total;
    if ((st = lr_attr(k_lowrank<P, kLrGradA>, smem)) != PC_OK) return st;
    const int slot = profile_begin(s);
    k_lowrank<P, kLrGradA><<<dim3(cdiv(M, kLrRows), B), kLrThreadsFused, smem, s>>>(maps, a);
    PC_LAUNCH_CHECK();
    profile_end(slot, s, PC_KIND_LOWRANK_BWD, 2 * flops);
  }
  if (dB || e) {
    LrMaps maps;
    if ((st = encode_op(maps.own, w.BTop, kLrRows)) != PC_OK) return st;
    if ((st = encode_op(maps.sw, w.Aop, kLrChunk)) != PC_OK) return st;
    if ((st = encode_op(maps.gb, w.AgT, Kp)) != PC_OK) return st;
    if ((st = encode_operand_map(&maps.th, w.thetaT, PC_PREC_TF32, kLrRows, 0)) != PC_OK) return st;
    if ((st = encode_operand_map(&maps.vec[0], w.rf_lz, PC_PREC_TF32, 1, 0, false)) != PC_OK) return st;
    if ((st = encode_operand_map(&maps.vec[1], w.rf_f, PC_PREC_TF32, 1, 0, false)) != PC_OK) return st;
    if ((st = encode_operand_map(&maps.vec[2], w.rf_fc, PC_PREC_TF32, 1, 0, false)) != PC_OK) return st;
    const int smem = lr_smem(P, kLrGradB, K).total;
    if ((st = lr_attr(k_lowrank<P, kLrGradB>, smem)) != PC_OK) return st;
    const int slot = profile_begin(s);
    k_lowrank<P, kLrGradB><<<dim3(cdiv(N, kLrRows), B), kLrThreadsFused, smem, s>>>(maps, a);
    PC_LAUNCH_CHECK();
    profile_end(slot, s, PC_KIND_LOWRANK_BWD, 2 * flops);
  }
  if (Fp || W) {
    LrMaps maps;
    if ((st = encode_op(maps.own, w.Aop, kLrRows)) != PC_OK) return st;
    if ((st = encode_op(maps.sw, w.BTop, kLrChunk)) != PC_OK) return st;
    maps.gb[0] = maps.gb[1] = maps.th = maps.sw[0];  // unused
    if ((st = encode_operand_map(&maps.vec[0], w.u, PC_PREC_TF32, 1, 0, false)) != PC_OK) return st;
    maps.vec[1] = maps.vec[2] = maps.vec[0];
    const int smem = lr_smem(P, kLrStats, K).total;
    if ((st = lr_attr(k_lowrank_stats<P>, smem)) != PC_OK) return st;
    const int slot = profile_begin(s);
    k_lowrank_stats<P><<<dim3(cdiv(M, kLrRows), cdiv(N, kLrChunk)), kLrThreadsFused, smem, s>>>(maps, a);
    PC_LAUNCH_CHECK();
    profile_end(slot, s, PC_KIND_LOWRANK_BWD, flops);
  }
  return PC_OK;
}

}  // namespace
}  // namespace pc

using namespace pc;

extern "C" {

pc_status_t pc_lowrank_exp_sum_workspace(int M, int N, int K, int B, int with_backward, pc_precision_t prec,
                                         size_t* bytes) {
  clear_error();
  PC_CHECK(bytes, PC_ERR_NULL, "bytes is NULL");
  pc_status_t st = check_lr_shape(M, N, K, B, prec);
  if (st != PC_OK) return st;
  LrWs w;
  *bytes = carve_lr(nullptr, prec, M, N, K, B, with_backward != 0, &w);
  return PC_OK;
}

pc_status_t pc_lowrank_exp_sum_fwd(int M, int N, int K, int B, const float* theta, const float* A, const float* Bm,
                                   const float* x, float* out, float* logZ, pc_precision_t prec, void* ws,
                                   size_t ws_bytes, pc_stream_t stream) {
  clear_error();
  pc_status_t st = check_lr_shape(M, N, K, B, prec);
  if (st != PC_OK) return st;
  const bool work = M > 0 && B > 0;
  PC_CHECK(!work || (out && logZ), PC_ERR_NULL, "out and logZ are required");
  PC_CHECK(!work || N == 0 || (theta && A && Bm && x), PC_ERR_NULL, "theta, A, B and x are required");
  PC_CHECK(ws || !work, PC_ERR_NULL, "workspace is NULL");
  PC_CHECK(!ws || aligned16(ws), PC_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  LrWs w;
  const size_t need = carve_lr(nullptr, prec, M, N, K, B, false, &w);
  PC_CHECK(!work || ws_bytes >= need, PC_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (prec) {
    case PC_PREC_AUTO: return lr_fwd<kBF16>(M, N, K, B, theta, A, Bm, x, out, logZ, ws, s);
    case PC_PREC_TF32: return lr_fwd<kTF32>(M, N, K, B, theta, A, Bm, x, out, logZ, ws, s);
    default: return lr_fwd<kTF32x3>(M, N, K, B, theta, A, Bm, x, out, logZ, ws, s);
  }
}

pc_status_t pc_lowrank_exp_sum_bwd(int M, int N, int K, int B, const float* theta, const float* A, const float* Bm,
                                   const float* x, const float* out, const float* logZ, const float* f, float* dA,
                                   float* dB, float* e, float* Fplus, float* Wstat, int accumulate,
                                   pc_precision_t prec, void* ws, size_t ws_bytes, pc_stream_t stream) {
  clear_error();
  pc_status_t st = check_lr_shape(M, N, K, B, prec);
  if (st != PC_OK) return st;
  const bool work = M > 0 && N > 0 && B > 0;
  PC_CHECK(!work || (theta && A && Bm && x && out && logZ && f), PC_ERR_NULL,
           "theta, A, B, x, out, logZ and f are required");
  PC_CHECK(ws || !work, PC_ERR_NULL, "workspace is NULL");
  PC_CHECK(!ws || aligned16(ws), PC_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  LrWs w;
  const size_t need = carve_lr(nullptr, prec, M, N, K, B, true, &w);
  PC_CHECK(!work || ws_bytes >= need, PC_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (prec) {
    case PC_PREC_AUTO:
      return lr_bwd<kBF16>(M, N, K, B, theta, A, Bm, x, out, logZ, f, dA, dB, e, Fplus, Wstat, accumulate, ws, s);
    case PC_PREC_TF32:
      return lr_bwd<kTF32>(M, N, K, B, theta, A, Bm, x, out, logZ, f, dA, dB, e, Fplus, Wstat, accumulate, ws, s);
    default:
      return lr_bwd<kTF32x3>(M, N, K, B, theta, A, Bm, x, out, logZ, f, dA, dB, e, Fplus, Wstat, accumulate, ws, s);
  }
}

}  // extern "C"
