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
#include <cmath>

#include "pc_launch.cuh"

namespace pc {
namespace {

constexpr int kLrRows = 128;   // own rows per CTA (TMEM lanes)
constexpr int kLrChunk = 32;   // sweep columns per MMA group
constexpr int kLrThreads = 128;
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

// Byte offset of element (row, k) inside one part of a tile: 128-byte swizzle of the
// 16-byte chunk index by the row within its 8-row core group.
__device__ __forceinline__ uint32_t tile_off(const TileGeo& g, int es, int row, int k) {
  const int byte = k * es;
  const int blk = byte >> 7;
  const int in = byte & 127;
  return static_cast<uint32_t>(blk * g.rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
                               ((((in >> 4) ^ (row & 7)) & 7) << 4) + (in & 15));
}

// Writes v at (row, k) in format F (both parts for the split formats).
template <int F>
__device__ __forceinline__ void tile_put(uint8_t* tile, const TileGeo& g, int row, int k, float v) {
  constexpr int es = fmt_bytes(F);
  const uint32_t off = tile_off(g, es, row, k);
  if constexpr (F == kFmtBF16 || F == kFmtBF16x2) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    *reinterpret_cast<__nv_bfloat16*>(tile + off) = hi;
    if constexpr (F == kFmtBF16x2)
      *reinterpret_cast<__nv_bfloat16*>(tile + g.bytes_part() + off) =
          __float2bfloat16_rn(v - __bfloat162float(hi));
  } else {
    const float hi = tf32_rna(v);
    *reinterpret_cast<float*>(tile + off) = hi;
    if constexpr (F == kFmtTF32x2) *reinterpret_cast<float*>(tile + g.bytes_part() + off) = tf32_rna(v - hi);
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Issues D(tmem) (+)= A(tile a, M = 128 rows) * B(tile b, N rows)^T over the k-steps of
// the tiles, in format F: split formats take lo*hi, hi*lo, then hi*hi per k-step.
template <int F>
__device__ __forceinline__ void lr_mma(uint32_t d, const uint8_t* a, const TileGeo& ga, const uint8_t* b,
                                       const TileGeo& gb, int n, bool accumulate) {
  constexpr uint32_t kind = F <= kFmtBF16x2 ? 1u : 2u;
  const uint32_t idesc = umma_idesc(kind, kLrRows, static_cast<uint32_t>(n));
  const uint32_t a0 = smem_addr(a), b0 = smem_addr(b);
  const uint32_t a1 = a0 + (fmt_parts(F) == 2 ? ga.bytes_part() : 0);
  const uint32_t b1 = b0 + (fmt_parts(F) == 2 ? gb.bytes_part() : 0);
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
// Per sample b: m_b = max_j x[j,b] and u[b][j] = exp(x[j,b] - m_b) (sample-major). One
// block per sample.
__global__ void k_lr_colmax_u(int N, int B, const float* __restrict__ x, float* __restrict__ m,
                              float* __restrict__ u) {
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
    u[static_cast<long long>(b) * N + j] =
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
// (0 where out or log Z is -inf: such a node passes no flow), sample-major [B][M].
__global__ void k_lr_row_factors(int M, int B, const float* __restrict__ out, const float* __restrict__ f,
                                 const float* __restrict__ logZ, const float* __restrict__ m,
                                 float* __restrict__ rf_lz, float* __restrict__ rf_f, float* __restrict__ rf_fc) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(M) * B) return;
  const int b = static_cast<int>(idx / M), i = static_cast<int>(idx % M);
  const float o = out[static_cast<long long>(i) * B + b];
  const float lz = logZ[idx];
  const float fi = f[static_cast<long long>(i) * B + b];
  const bool live = o > -INFINITY && lz > -INFINITY && m[b] > -INFINITY;
  rf_lz[idx] = lz;
  rf_f[idx] = live ? fi : 0.f;
  rf_fc[idx] = live ? fi * expf(m[b] - o) : 0.f;
}

// ------------------------------------------------------------------ shared memory plan
// Byte offsets inside the (1024-aligned) dynamic shared memory of the LowRank kernels.
struct LrSmem {
  int own, sw, sw_bytes, theta, d, d_bytes, gb, gb_bytes, small, total;
};
constexpr int kThetaTileBytes = kLrRows * 128;  // 128 rows x 32 floats
__host__ __device__ inline LrSmem lr_smem(int P, bool grad, int K, int own_bufs) {
  const int SF = s_fmt(P), GF = g_fmt(P);
  const int Kp = (K + 15) & ~15;
  LrSmem s;
  int off = 0;
  s.own = off;
  off += own_bufs * tile_bytes(SF, kLrRows, K);
  s.sw_bytes = tile_bytes(SF, kLrChunk, K);
  s.sw = off;
  off += 2 * s.sw_bytes;
  s.theta = off;
  off += 2 * kThetaTileBytes;
  s.d_bytes = grad ? tile_bytes(GF, kLrRows, kLrChunk) : 0;
  s.d = off;
  off += 2 * s.d_bytes;
  s.gb_bytes = grad ? tile_bytes(GF, Kp, kLrChunk) : 0;
  s.gb = off;
  off += 2 * s.gb_bytes;
  s.small = off;        // [0,256) staged u, [256,1024) staged row factors, then barriers
  off += 2048;
  s.total = off + 1024;  // alignment slack
  return s;
}

struct LrArgs {
  int M, N, K, B;
  const float* A;      // [B][M][K]
  const float* Bm;     // [B][K][N]
  const float* u;      // [B][N]  exp(x - m_b)
  const float* m;      // [B]
  const float* rf_lz;  // [B][M]  backward row factors
  const float* rf_f;
  const float* rf_fc;
  const float* theta_ld;  // row-padded theta copy (stats pass)
  long long theta_ld_stride;
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

__device__ __forceinline__ float theta_at(const uint8_t* tile, int row, int col) {
  return *reinterpret_cast<const float*>(tile + row * 128 + ((((col >> 2) ^ (row & 7)) & 7) << 4) + (col & 3) * 4);
}

// One pass (forward, grad A or grad B) over the tile of 128 own rows of sample
// blockIdx.y; see the file comment.
template <int P, int Mode>
__global__ void __launch_bounds__(kLrThreads, 1)
    k_lowrank(const __grid_constant__ CUtensorMap tmTheta, const LrArgs a) {
  constexpr int SF = s_fmt(P), GF = g_fmt(P);
  constexpr bool kGrad = Mode != kLrFwd;
  const int K = a.K;
  const int Kp = (K + 15) & ~15;
  const int own_n = Mode == kLrGradB ? a.N : a.M;
  const int sw_n = Mode == kLrGradB ? a.M : a.N;
  const int b = blockIdx.y;
  const int o0 = blockIdx.x * kLrRows;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int own = o0 + t;
  const TileGeo go = tile_geo(SF, kLrRows, K), gs = tile_geo(SF, kLrChunk, K);
  const TileGeo gd = tile_geo(GF, kLrRows, kLrChunk), gg = tile_geo(GF, Kp, kLrChunk);
  const int kf = go.ksteps * fmt_kstep(SF);  // K padded to whole k-steps (zeros)
  const LrSmem L = lr_smem(P, kGrad, K, 1);
  // TMEM: two 32-column S slots, then (gradients) kGradAccs accumulators of gstride
  // columns that the chunks take in turn: each sums a quarter of the sweep, which keeps
  // the accumulator's truncations to a quarter; the epilogue adds them up.
  const int gstride = (Kp + 31) & ~31;
  const uint32_t tcols = !kGrad ? 64u : (64 + kGradAccs * gstride <= 128 ? 128u
                                         : (64 + kGradAccs * gstride <= 256 ? 256u : 512u));

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* own_tile = smem + L.own;
  float* uS = reinterpret_cast<float*>(smem + L.small);  // [2][32]
  float* rfS = uS + 64;                                    // [2][3][32]
  uint64_t* mbS = reinterpret_cast<uint64_t*>(smem + L.small + 1024);
  uint64_t* mbT = mbS + 2;
  uint64_t* mbG = mbS + 4;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mbS + 6);
  auto sw_tile = [&](int s) { return smem + L.sw + s * L.sw_bytes; };
  auto th_tile = [&](int s) { return smem + L.theta + s * kThetaTileBytes; };
  auto d_tile = [&](int s) { return smem + L.d + s * L.d_bytes; };
  auto gb_tile = [&](int s) { return smem + L.gb + s * L.gb_bytes; };

  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(&mbS[i], 1);
        mbar_init(&mbT[i], 1);
        mbar_init(&mbG[i], 1);
      }
      fence_barrier_init();
      tma_prefetch_map(&tmTheta);
    }
    __syncwarp();
    tmem_alloc(tslot, tcols);
  }
  // own operand: A_b rows (forward, grad A) or B_b^T rows (grad B)
  for (int idx = t; idx < kLrRows * kf; idx += kLrThreads) {
    int o, k;
    if constexpr (Mode == kLrGradB) {
      o = idx % kLrRows;
      k = idx / kLrRows;
    } else {
      k = idx % kf;
      o = idx / kf;
    }
    const int gi = o0 + o;
    float v = 0.f;
    if (gi < own_n && k < K)
      v = Mode == kLrGradB ? a.Bm[(static_cast<long long>(b) * K + k) * a.N + gi]
                           : a.A[(static_cast<long long>(b) * a.M + gi) * K + k];
    tile_put<SF>(own_tile, go, o, k, v);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);

  // per-row constants
  float lz = 0.f, fi = 0.f, fc = 0.f, uj = 0.f;
  if constexpr (Mode == kLrGradA) {
    if (own < a.M) {
      const long long r = static_cast<long long>(b) * a.M + own;
      lz = a.rf_lz[r];
      fi = a.rf_f[r];
      fc = a.rf_fc[r];
    }
  }
  if constexpr (Mode == kLrGradB) uj = own < a.N ? a.u[static_cast<long long>(b) * a.N + own] : 0.f;
  const bool row_live = lz > -INFINITY;
  const float mb = a.m[b];

  // fills of chunk c (all threads)
  auto stage = [&](int c) {
    const int sl = c & 1, w0 = c * kLrChunk;
    uint8_t* st = sw_tile(sl);
    for (int idx = t; idx < kLrChunk * kf; idx += kLrThreads) {
      int w, k;
      if constexpr (Mode == kLrGradB) {
        k = idx % kf;
        w = idx / kf;
      } else {
        w = idx % kLrChunk;
        k = idx / kLrChunk;
      }
      const int gw = w0 + w;
      float v = 0.f;
      if (gw < sw_n && k < K)
        v = Mode == kLrGradB ? a.A[(static_cast<long long>(b) * a.M + gw) * K + k]
                             : a.Bm[(static_cast<long long>(b) * K + k) * a.N + gw];
      tile_put<SF>(st, gs, w, k, v);
    }
    if constexpr (kGrad) {
      uint8_t* gt = gb_tile(sl);
      for (int idx = t; idx < Kp * kLrChunk; idx += kLrThreads) {
        int r, kk;
        if constexpr (Mode == kLrGradA) {
          kk = idx % kLrChunk;
          r = idx / kLrChunk;
        } else {
          r = idx % Kp;
          kk = idx / Kp;
        }
        const int gw = w0 + kk;
        float v = 0.f;
        if (r < K && gw < sw_n)
          v = Mode == kLrGradA ? a.Bm[(static_cast<long long>(b) * K + r) * a.N + gw]
                               : a.A[(static_cast<long long>(b) * a.M + gw) * K + r];
        tile_put<GF>(gt, gg, r, kk, v);
      }
    }
    if (t < kLrChunk) {
      const int gw = w0 + t;
      if constexpr (Mode == kLrGradB) {
        const long long r = static_cast<long long>(b) * a.M + gw;
        rfS[(sl * 3 + 0) * 32 + t] = gw < a.M ? a.rf_lz[r] : -INFINITY;
        rfS[(sl * 3 + 1) * 32 + t] = gw < a.M ? a.rf_f[r] : 0.f;
        rfS[(sl * 3 + 2) * 32 + t] = gw < a.M ? a.rf_fc[r] : 0.f;
      } else {
        uS[sl * 32 + t] = gw < a.N ? a.u[static_cast<long long>(b) * a.N + gw] : 0.f;
      }
    }
    fence_proxy_async_smem();
  };
  // theta tile and S = own * sweep^T of chunk c (thread 0, after the fills are visible)
  auto issue = [&](int c) {
    const int sl = c & 1;
    mbar_arrive_expect_tx(&mbT[sl], kThetaTileBytes);
    tma_load_3d(th_tile(sl), &tmTheta, &mbT[sl], c * kLrChunk, o0, 0);
    tc_fence_after();
    lr_mma<SF>(tmem + static_cast<uint32_t>(sl * kLrChunk), own_tile, go, sw_tile(sl), gs, kLrChunk, false);
    umma_commit(&mbS[sl]);
  };

  const int nch = (sw_n + kLrChunk - 1) / kLrChunk;
  bool ok = true;
  int issued = -1, consumed = -1, g_issued = -1;  // chunk indices (thread 0's view)
  float run = -INFINITY, Z = 0.f, num = 0.f;       // forward
  float e_acc = 0.f;                               // grad B
  stage(0);
  __syncthreads();
  if (t == 0) {
    issue(0);
    issued = 0;
  }
  for (int c = 0; c < nch; ++c) {
    const int sl = c & 1;
    const uint32_t ph = (c >> 1) & 1;
    if (c + 1 < nch) {
      // the grad B-operand slot of chunk c+1 was read by the grad MMA of chunk c-1
      if (kGrad && c >= 1) ok = ok && mbar_wait(&mbG[(c - 1) & 1], ((c - 1) >> 1) & 1, a.status, kErrTimeoutMma);
      stage(c + 1);
    }
    ok = __syncthreads_and(ok);
    if (!ok) break;
    if (t == 0 && c + 1 < nch) {
      issue(c + 1);
      issued = c + 1;
    }
    bool w = mbar_wait(&mbS[sl], ph, a.status, kErrTimeoutEpilogue) &&
             mbar_wait(&mbT[sl], ph, a.status, kErrTimeoutEpilogue);
    w = __all_sync(0xffffffffu, w);
    consumed = c;
    tc_fence_after();
    float v[32];
    if (w) {
      tmem_ld_32x32(lane_base + static_cast<uint32_t>(sl * kLrChunk), v);
      const uint8_t* th = th_tile(sl);
      const int w0 = c * kLrChunk;
      if constexpr (Mode == kLrFwd) {
        float cm = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj)
          if (w0 + jj < a.N) cm = fmaxf(cm, v[jj]);
        if (cm > run) {
          const float sc = run > -INFINITY ? expf(run - cm) : 0.f;
          Z *= sc;
          num *= sc;
          run = cm;
        }
        const float* us = uS + sl * 32;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const float tg = w0 + jj < a.N ? theta_at(th, t, jj) * expf(v[jj] - run) : 0.f;
          Z += tg;
          num = fmaf(tg, us[jj], num);
        }
      } else {
        // D (grad A: row i over columns j; grad B: row j over columns i)
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          float q, dv;
          if constexpr (Mode == kLrGradA) {
            const float tj = theta_at(th, t, jj);
            q = (row_live && tj > 0.f) ? tj * expf(v[jj] - lz) : 0.f;
            dv = q * fmaf(uS[sl * 32 + jj], fc, -fi);
          } else {
            const float lzi = rfS[(sl * 3 + 0) * 32 + jj];
            const float fci = rfS[(sl * 3 + 2) * 32 + jj];
            const float tj = theta_at(th, t, jj);
            q = (lzi > -INFINITY && tj > 0.f) ? tj * expf(v[jj] - lzi) : 0.f;
            const float pf = q * uj * fci;
            e_acc += pf;
            dv = pf - q * rfS[(sl * 3 + 1) * 32 + jj];
          }
          v[jj] = own < own_n ? dv : 0.f;
        }
        // the D slot was read by the grad MMA of chunk c-2
        if (c >= 2) w = w && mbar_wait(&mbG[sl], ((c - 2) >> 1) & 1, a.status, kErrTimeoutMma);
        uint8_t* dt = d_tile(sl);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) tile_put<GF>(dt, gd, t, jj, v[jj]);
        fence_proxy_async_smem();
      }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok && w);
    if (!ok) break;
    if (kGrad && t == 0) {
      tc_fence_after();
      lr_mma<GF>(tmem + static_cast<uint32_t>(64 + (c % kGradAccs) * gstride), d_tile(sl), gd, gb_tile(sl), gg,
                 Kp, c >= kGradAccs);
      umma_commit(&mbG[sl]);
      g_issued = c;
    }
  }

  if (ok && kGrad && nch > 0) {
    bool w = mbar_wait(&mbG[(nch - 1) & 1], ((nch - 1) >> 1) & 1, a.status, kErrTimeoutEpilogue);
    ok = __syncthreads_and(w);
  }
  if (ok) {
    if constexpr (Mode == kLrFwd) {
      if (own < a.M) {
        const bool live = Z > 0.f && num > 0.f && mb > -INFINITY;
        const float o = live ? mb + logf(num / Z) : -INFINITY;
        const float lzv = Z > 0.f ? logf(Z) + run : -INFINITY;
        a.out[static_cast<long long>(own) * a.B + b] = o;
        a.logZ[static_cast<long long>(b) * a.M + own] = lzv;
      }
    } else {
      tc_fence_after();
      float acc[64];
      for (int r = 0; r < 64; ++r) acc[r] = 0.f;
      for (int q = 0; q < kGradAccs && q < nch; ++q) {
        for (int c0 = 0; c0 < Kp; c0 += 32) {
          float v[32];
          tmem_ld_32x32(lane_base + static_cast<uint32_t>(64 + q * gstride + c0), v);
#pragma unroll
          for (int r = 0; r < 32; ++r) acc[c0 + r] += v[r];
        }
      }
      if (own < own_n) {
        if constexpr (Mode == kLrGradA) {
          float* dst = a.dA + (static_cast<long long>(b) * a.M + own) * K;
          for (int r = 0; r < K; ++r) dst[r] = a.accumulate ? dst[r] + acc[r] : acc[r];
        } else {
          if (a.dB) {
            for (int r = 0; r < K; ++r) {
              float* dst = a.dB + (static_cast<long long>(b) * K + r) * a.N + own;
              *dst = a.accumulate ? *dst + acc[r] : acc[r];
            }
          }
          if (a.e) {
            float* de = a.e + static_cast<long long>(own) * a.B + b;
            *de = a.accumulate ? *de + e_acc : e_acc;
          }
        }
      }
    }
  } else if (t == 0) {
    // a wait gave up: let the copies and MMAs in flight finish before TMEM is freed
    for (int c = consumed + 1; c <= issued; ++c) {
      mbar_wait(&mbT[c & 1], (c >> 1) & 1, a.status, kErrTimeoutDrain);
      mbar_wait(&mbS[c & 1], (c >> 1) & 1, a.status, kErrTimeoutDrain);
    }
    if (g_issued >= 0) mbar_wait(&mbG[g_issued & 1], (g_issued >> 1) & 1, a.status, kErrTimeoutDrain);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

// Parameter-flow statistics F+ and W over all samples for the 128 x 32 tile (blockIdx.x,
// blockIdx.y) of [M, N]: own rows i, the 32 columns j fixed, a sweep over the samples;
// each sample's S chunk is one MMA group, its own A_b tile double-buffered.
template <int P>
__global__ void __launch_bounds__(kLrThreads, 1)
    k_lowrank_stats(const LrArgs a) {
  constexpr int SF = s_fmt(P);
  const int K = a.K;
  const int i0 = blockIdx.x * kLrRows, j0 = blockIdx.y * kLrChunk;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int i = i0 + t;
  const TileGeo go = tile_geo(SF, kLrRows, K), gs = tile_geo(SF, kLrChunk, K);
  const int kf = go.ksteps * fmt_kstep(SF);
  const LrSmem L = lr_smem(P, false, K, 2);
  const int own_bytes = tile_bytes(SF, kLrRows, K);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* uS = reinterpret_cast<float*>(smem + L.small);  // [2][32]
  uint64_t* mbS = reinterpret_cast<uint64_t*>(smem + L.small + 1024);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mbS + 2);
  auto own_tile = [&](int s) { return smem + L.own + s * own_bytes; };
  auto sw_tile = [&](int s) { return smem + L.sw + s * L.sw_bytes; };

  if (warp == 0) {
    if (lane == 0) {
      mbar_init(&mbS[0], 1);
      mbar_init(&mbS[1], 1);
      fence_barrier_init();
    }
    __syncwarp();
    tmem_alloc(tslot, 64);
  }
  // theta[i][j0 .. j0+31] in registers, from the row-padded copy
  float th[32];
#pragma unroll
  for (int jj = 0; jj < 32; ++jj)
    th[jj] = (i < a.M && j0 + jj < a.N) ? a.theta_ld[static_cast<long long>(i) * a.theta_ld_stride + j0 + jj] : 0.f;

  auto stage = [&](int b) {
    const int sl = b & 1;
    uint8_t* ot = own_tile(sl);
    for (int idx = t; idx < kLrRows * kf; idx += kLrThreads) {
      const int k = idx % kf, o = idx / kf;
      const int gi = i0 + o;
      const float v = (gi < a.M && k < K) ? a.A[(static_cast<long long>(b) * a.M + gi) * K + k] : 0.f;
      tile_put<SF>(ot, go, o, k, v);
    }
    uint8_t* st = sw_tile(sl);
    for (int idx = t; idx < kLrChunk * kf; idx += kLrThreads) {
      const int w = idx % kLrChunk, k = idx / kLrChunk;
      const int gj = j0 + w;
      const float v = (gj < a.N && k < K) ? a.Bm[(static_cast<long long>(b) * K + k) * a.N + gj] : 0.f;
      tile_put<SF>(st, gs, w, k, v);
    }
    if (t < kLrChunk) uS[sl * 32 + t] = j0 + t < a.N ? a.u[static_cast<long long>(b) * a.N + j0 + t] : 0.f;
    fence_proxy_async_smem();
  };

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  float fp[32], wst[32];
#pragma unroll
  for (int jj = 0; jj < 32; ++jj) fp[jj] = wst[jj] = 0.f;

  bool ok = true;
  int issued = -1, consumed = -1;
  stage(0);
  __syncthreads();
  if (t == 0) {
    tc_fence_after();
    lr_mma<SF>(tmem, own_tile(0), go, sw_tile(0), gs, kLrChunk, false);
    umma_commit(&mbS[0]);
    issued = 0;
  }
  for (int b = 0; b < a.B; ++b) {
    const int sl = b & 1;
    if (b + 1 < a.B) stage(b + 1);  // slot (b+1)&1 was read by the MMA of sample b-1 (waited)
    ok = __syncthreads_and(ok);
    if (!ok) break;
    if (t == 0 && b + 1 < a.B) {
      tc_fence_after();
      lr_mma<SF>(tmem + static_cast<uint32_t>(((b + 1) & 1) * kLrChunk), own_tile((b + 1) & 1), go,
                 sw_tile((b + 1) & 1), gs, kLrChunk, false);
      umma_commit(&mbS[(b + 1) & 1]);
      issued = b + 1;
    }
    // row factors of sample b
    float lz = -INFINITY, fi = 0.f, fc = 0.f;
    if (i < a.M) {
      const long long r = static_cast<long long>(b) * a.M + i;
      lz = a.rf_lz[r];
      fi = a.rf_f[r];
      fc = a.rf_fc[r];
    }
    bool w = __all_sync(0xffffffffu, mbar_wait(&mbS[sl], (b >> 1) & 1, a.status, kErrTimeoutEpilogue));
    consumed = b;
    tc_fence_after();
    if (w) {
      float v[32];
      tmem_ld_32x32(lane_base + static_cast<uint32_t>(sl * kLrChunk), v);
      if (lz > -INFINITY) {
        const float* us = uS + sl * 32;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const float gz = expf(v[jj] - lz);  // g_b / Z_b
          fp[jj] = fmaf(th[jj] * gz, us[jj] * fc, fp[jj]);
          wst[jj] = fmaf(fi, gz, wst[jj]);
        }
      }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok && w);
    if (!ok) break;
  }
  if (ok) {
    if (i < a.M) {
      for (int jj = 0; jj < 32; ++jj) {
        const int j = j0 + jj;
        if (j >= a.N) break;
        const long long idx = static_cast<long long>(i) * a.N + j;
        if (a.Fp) a.Fp[idx] = a.accumulate ? a.Fp[idx] + fp[jj] : fp[jj];
        if (a.W) a.W[idx] = a.accumulate ? a.W[idx] + wst[jj] : wst[jj];
      }
    }
  } else if (t == 0) {
    for (int b = consumed + 1; b <= issued; ++b) mbar_wait(&mbS[b & 1], (b >> 1) & 1, a.status, kErrTimeoutDrain);
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

struct LrWs {
  float *m, *u, *rf_lz, *rf_f, *rf_fc;
  Operand theta, thetaT;  // plain float32 copies, rows padded to 64 elements
};

size_t carve_lr(void* base, int M, int N, int B, bool bwd, LrWs* w) {
  Carver c(base);
  *w = LrWs{};
  w->m = static_cast<float*>(c.take(size_t(B) * 4));
  w->u = static_cast<float*>(c.take(size_t(B) * N * 4));
  w->theta = c.operand(PC_PREC_TF32, 1, M, N);
  if (bwd) {
    w->thetaT = c.operand(PC_PREC_TF32, 1, N, M);
    w->rf_lz = static_cast<float*>(c.take(size_t(B) * M * 4));
    w->rf_f = static_cast<float*>(c.take(size_t(B) * M * 4));
    w->rf_fc = static_cast<float*>(c.take(size_t(B) * M * 4));
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

pc_status_t lr_prepare(const float* theta, const float* x, int M, int N, int B, bool bwd, LrWs& w,
                       cudaStream_t s) {
  if (B > 0 && N > 0) {
    k_lr_colmax_u<<<B, 256, 0, s>>>(N, B, x, w.m, w.u);
    PC_LAUNCH_CHECK();
  }
  if (M > 0 && N > 0) {
    const dim3 g(cdiv(N, 32), cdiv(M, 32));
    k_lr_theta_copy<<<g, dim3(32, 8), 0, s>>>(M, N, theta, static_cast<float*>(w.theta.ptr), w.theta.ld, 0);
    PC_LAUNCH_CHECK();
    if (bwd) {
      k_lr_theta_copy<<<g, dim3(32, 8), 0, s>>>(M, N, theta, static_cast<float*>(w.thetaT.ptr), w.thetaT.ld, 1);
      PC_LAUNCH_CHECK();
    }
  }
  return PC_OK;
}

template <int P>
pc_status_t lr_fwd(int M, int N, int K, int B, const float* theta, const float* A, const float* Bm, const float* x,
                   float* out, float* logZ, void* ws, cudaStream_t s) {
  LrWs w;
  carve_lr(ws, M, N, B, false, &w);
  if (M == 0 || B == 0) return PC_OK;
  if (N == 0) {  // no children: every node's sum is empty
    k_lr_fill<<<cdiv(static_cast<long long>(M) * B, 256), 256, 0, s>>>(out, static_cast<long long>(M) * B, -INFINITY);
    PC_LAUNCH_CHECK();
    k_lr_fill<<<cdiv(static_cast<long long>(M) * B, 256), 256, 0, s>>>(logZ, static_cast<long long>(M) * B, -INFINITY);
    PC_LAUNCH_CHECK();
    return PC_OK;
  }
  pc_status_t st = lr_prepare(theta, x, M, N, B, false, w, s);
  if (st != PC_OK) return st;
  CUtensorMap tm;
  if ((st = encode_operand_map(&tm, w.theta, PC_PREC_TF32, kLrRows, 0)) != PC_OK) return st;
  LrArgs a{};
  a.M = M; a.N = N; a.K = K; a.B = B;
  a.A = A; a.Bm = Bm; a.u = w.u; a.m = w.m;
  a.out = out; a.logZ = logZ;
  a.status = device_status_word();
  const int smem = lr_smem(P, false, K, 1).total;
  if ((st = lr_attr(k_lowrank<P, kLrFwd>, smem)) != PC_OK) return st;
  const int slot = profile_begin(s);
  k_lowrank<P, kLrFwd><<<dim3(cdiv(M, kLrRows), B), kLrThreads, smem, s>>>(tm, a);
  PC_LAUNCH_CHECK();
  profile_end(slot, s, PC_KIND_LOWRANK_FWD, 2LL * M * N * K * B);
  return PC_OK;
}

template <int P>
pc_status_t lr_bwd(int M, int N, int K, int B, const float* theta, const float* A, const float* Bm, const float* x,
                   const float* out, const float* logZ, const float* f, float* dA, float* dB, float* e, float* Fp,
                   float* W, int accumulate, void* ws, cudaStream_t s) {
  LrWs w;
  carve_lr(ws, M, N, B, true, &w);
  if (!accumulate) {  // outputs that no pass writes when a size is zero
    if (dA && N == 0) PC_CUDA(cudaMemsetAsync(dA, 0, size_t(B) * M * K * 4, s));
    if (dB && M == 0) PC_CUDA(cudaMemsetAsync(dB, 0, size_t(B) * K * N * 4, s));
    if (e && M == 0) PC_CUDA(cudaMemsetAsync(e, 0, size_t(N) * B * 4, s));
    if (Fp && B == 0) PC_CUDA(cudaMemsetAsync(Fp, 0, size_t(M) * N * 4, s));
    if (W && B == 0) PC_CUDA(cudaMemsetAsync(W, 0, size_t(M) * N * 4, s));
  }
  if (M == 0 || N == 0 || B == 0) return PC_OK;
  pc_status_t st = lr_prepare(theta, x, M, N, B, true, w, s);
  if (st != PC_OK) return st;
  k_lr_row_factors<<<cdiv(static_cast<long long>(M) * B, 256), 256, 0, s>>>(M, B, out, f, logZ, w.m, w.rf_lz,
                                                                             w.rf_f, w.rf_fc);
  PC_LAUNCH_CHECK();
  LrArgs a{};
  a.M = M; a.N = N; a.K = K; a.B = B;
  a.A = A; a.Bm = Bm; a.u = w.u; a.m = w.m;
  a.rf_lz = w.rf_lz; a.rf_f = w.rf_f; a.rf_fc = w.rf_fc;
  a.theta_ld = static_cast<const float*>(w.theta.ptr);
  a.theta_ld_stride = w.theta.ld;
  a.dA = dA; a.dB = dB; a.e = e; a.Fp = Fp; a.W = W;
  a.accumulate = accumulate;
  a.status = device_status_word();
  const long long flops = 2LL * M * N * K * B;
  if (dA) {
    CUtensorMap tm;
    if ((st = encode_operand_map(&tm, w.theta, PC_PREC_TF32, kLrRows, 0)) != PC_OK) return st;
    const int smem = lr_smem(P, true, K, 1).total;
    if ((st = lr_attr(k_lowrank<P, kLrGradA>, smem)) != PC_OK) return st;
    const int slot = profile_begin(s);
    k_lowrank<P, kLrGradA><<<dim3(cdiv(M, kLrRows), B), kLrThreads, smem, s>>>(tm, a);
    PC_LAUNCH_CHECK();
    profile_end(slot, s, PC_KIND_LOWRANK_BWD, 2 * flops);
  }
  if (dB || e) {
    CUtensorMap tm;
    if ((st = encode_operand_map(&tm, w.thetaT, PC_PREC_TF32, kLrRows, 0)) != PC_OK) return st;
    const int smem = lr_smem(P, true, K, 1).total;
    if ((st = lr_attr(k_lowrank<P, kLrGradB>, smem)) != PC_OK) return st;
    const int slot = profile_begin(s);
    k_lowrank<P, kLrGradB><<<dim3(cdiv(N, kLrRows), B), kLrThreads, smem, s>>>(tm, a);
    PC_LAUNCH_CHECK();
    profile_end(slot, s, PC_KIND_LOWRANK_BWD, 2 * flops);
  }
  if (Fp || W) {
    const int smem = lr_smem(P, false, K, 2).total;
    if ((st = lr_attr(k_lowrank_stats<P>, smem)) != PC_OK) return st;
    const int slot = profile_begin(s);
    k_lowrank_stats<P><<<dim3(cdiv(M, kLrRows), cdiv(N, kLrChunk)), kLrThreads, smem, s>>>(a);
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
  *bytes = carve_lr(nullptr, M, N, B, with_backward != 0, &w);
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
  const size_t need = carve_lr(nullptr, M, N, B, false, &w);
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
  const size_t need = carve_lr(nullptr, M, N, B, true, &w);
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
