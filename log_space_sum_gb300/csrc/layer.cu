// Dense log-space sum layer, G groups: forward and EM flows (pyjuice PR #62,
// Summary 2 and 3). Each pass is
//   1. a prologue kernel that reduces the per-group column maximum m_b over the
//      group's children and writes the exponentiated, shifted operand once for all
//      nodes of the group (the children are shared by every node of a group),
//   2. the tcgen05 contraction (pc_gemm.cuh) with the pass's epilogue in registers:
//        forward    D[i,b] = sum_j theta[i,j] u[j,b],   u = exp(x - m_b)
//                   out    = m_b + log D
//        element    D[j,b] = sum_i theta[i,j] w[i,b],   w = f exp(m_b - out)
//                   e      = exp(x - m_b) * D
//        parameter  D[i,j] = sum_b w[i,b] u[j,b]
//                   F      = theta * D
#include <algorithm>
#include <cmath>
#include <mutex>

#include "pc_launch.cuh"

namespace pc {
namespace {

// ------------------------------------------------------------------ prologue
// colmax[g][b] = max over the group's N children of x[g*cs + j][b].
__global__ void k_colmax(const float* __restrict__ x, long long cs, int N, int B,
                         float* __restrict__ colmax) {
  __shared__ float red[16][33];
  const int g = blockIdx.y;
  const int b = blockIdx.x * 32 + threadIdx.x;
  float m = -INFINITY;
  if (b < B) {
    const float* xg = x + static_cast<long long>(g) * cs * B + b;
    for (int j = threadIdx.y; j < N; j += 16) m = fmaxf(m, xg[static_cast<long long>(j) * B]);
  }
  red[threadIdx.y][threadIdx.x] = m;
  __syncthreads();
  if (threadIdx.y == 0 && b < B) {
    for (int k = 1; k < 16; ++k) m = fmaxf(m, red[k][threadIdx.x]);
    colmax[static_cast<long long>(g) * B + b] = m;
  }
}

// Value sources of the operand builder.
struct ExpChildren {            // u[g][j][b] = exp(x[g*cs+j][b] - m[g][b])
  const float* x;
  const float* colmax;
  long long cs;
  int B;
  __device__ float operator()(int g, int j, int b) const {
    const float m = colmax[static_cast<long long>(g) * B + b];
    if (!(m > -INFINITY)) return 0.f;
    return expf(x[(static_cast<long long>(g) * cs + j) * B + b] - m);
  }
};

struct ScaledFlow {             // w[g][i][b] = f exp(m[g][b] - out)
  const float* f;
  const float* out;
  const float* colmax;
  int M, B;
  __device__ float operator()(int g, int i, int b) const {
    const long long idx = (static_cast<long long>(g) * M + i) * B + b;
    const float o = out[idx];
    if (!(o > -INFINITY)) return 0.f;
    return f[idx] * expf(colmax[static_cast<long long>(g) * B + b] - o);
  }
};

// Writes the operand value v(g, r, b) for r < R, b < B node-major nm[g][r][b] and/or
// batch-major bm[g][b][r] (transposed through a shared-memory tile).
template <int P, class Src>
__global__ void k_make_operands(Src src, int R, int B, void* nm, long long nm_ld, size_t nm_lo,
                                void* bm, long long bm_ld, size_t bm_lo) {
  __shared__ float tile[32][33];
  const int g = blockIdx.z;
  const int b0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int k = ty; k < 32; k += 8) {
    const int r = r0 + k, b = b0 + tx;
    float v = 0.f;
    if (r < R && b < B) {
      v = src(g, r, b);
      if (nm) store_operand<P>(nm, static_cast<size_t>((static_cast<long long>(g) * R + r) * nm_ld + b), nm_lo, v);
    }
    tile[k][tx] = v;
  }
  if (!bm) return;
  __syncthreads();
  for (int k = ty; k < 32; k += 8) {
    const int b = b0 + k, r = r0 + tx;
    if (r < R && b < B)
      store_operand<P>(bm, static_cast<size_t>((static_cast<long long>(g) * B + b) * bm_ld + r), bm_lo,
                       tile[tx][k]);
  }
}

template <int P, class Src>
pc_status_t make_operands(const Src& src, int G, int R, int B, const Operand* nm, const Operand* bm,
                          cudaStream_t s) {
  dim3 grid(cdiv(B, 32), cdiv(R, 32), G);
  k_make_operands<P, Src><<<grid, dim3(32, 8), 0, s>>>(
      src, R, B, nm ? nm->ptr : nullptr, nm ? nm->ld : 0, nm ? nm->lo_elems : 0,
      bm ? bm->ptr : nullptr, bm ? bm->ld : 0, bm ? bm->lo_elems : 0);
  PC_LAUNCH_CHECK();
  return PC_OK;
}

// ----------------------------------------------------------------- epilogues
struct EpiLayerFwd : EpiNoHooks {
  static constexpr bool kTranspose = true;
  struct Params {
    float* out;
    const float* colmax;
    int M, B;
  };
  // Transposed: lane l owns sample column b = n0 + col0 + l of the warp's 32 node rows,
  // so each store instruction writes one contiguous row segment of out.
  __device__ static void apply(const Params& p, int g, int m0, int n0, int row, int col0,
                               float (&v)[32], uint8_t*, float* tbuf) {
    float w[32];
    warp_transpose32(v, w, tbuf);
    const int lane = threadIdx.x & 31;
    const int i0 = m0 + row - lane;
    const int b = n0 + col0 + lane;
    if (b >= p.B) return;
    const float m = p.colmax[static_cast<long long>(g) * p.B + b];
    float* o = p.out + (static_cast<long long>(g) * p.M + i0) * p.B + b;
#pragma unroll
    for (int r = 0; r < 32; ++r)
      if (i0 + r < p.M)
        o[static_cast<long long>(r) * p.B] = (m > -INFINITY && w[r] > 0.f) ? m + logf(w[r]) : -INFINITY;
  }
};

struct EpiLayerElem : EpiNoHooks {
  static constexpr bool kTranspose = true;
  struct Params {
    float* e;
    const float* x;
    const float* colmax;
    long long cs;
    int N, B, accumulate;
  };
  // Transposed like EpiLayerFwd; x (and e when accumulating) are loaded for the whole
  // chunk before the first store.
  __device__ static void apply(const Params& p, int g, int m0, int n0, int row, int col0,
                               float (&v)[32], uint8_t*, float* tbuf) {
    float w[32];
    warp_transpose32(v, w, tbuf);
    const int lane = threadIdx.x & 31;
    const int j0 = m0 + row - lane;
    const int b = n0 + col0 + lane;
    if (b >= p.B) return;
    const float m = p.colmax[static_cast<long long>(g) * p.B + b];
    const long long ld = p.B;
    const long long base = (static_cast<long long>(g) * p.cs + j0) * ld + b;
    const float* xp = p.x + base;
    float* ep = p.e + base;
#pragma unroll
    for (int h = 0; h < 32; h += 16) {
      float xv[16], ev[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const bool in = j0 + h + r < p.N;
        xv[r] = in ? xp[(h + r) * ld] : -INFINITY;
        ev[r] = (in && p.accumulate) ? ep[(h + r) * ld] : 0.f;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        if (j0 + h + r < p.N) {
          const float u = (m > -INFINITY) ? expf(xv[r] - m) : 0.f;
          ep[(h + r) * ld] = ev[r] + u * w[h + r];
        }
      }
    }
  }
};

constexpr int kLayerBN = 128;

// ------------------------------------------------- contraction over K ranges
// A single group's forward and element-flow contractions have cdiv(rows,128) x
// cdiv(B,128) output tiles: at M = N = 1024, B = 128 eight CTAs, each over all of K. They
// then run over S consecutive K ranges (blockIdx.z; the operands' tensor maps take the
// ranges as groups) into S float32 partial sums, and the pass's elementwise epilogue
// runs in a reduction kernel that adds them in range order.
constexpr int kLayerSplitMax = 8;

int layer_split(int G, int rows, int K, int B, pc_precision_t prec) {
  if (G != 1) return 1;
  const int kb = 128 / operand_elem_bytes(prec);  // K elements per ring block
  const long long tiles = static_cast<long long>(cdiv(rows, kBM)) * cdiv(B, kLayerBN);
  if (tiles * B > (1ll << 24)) return 1;
  for (int S = kLayerSplitMax; S >= 2; S /= 2)
    if (tiles * S <= num_sms() && K % (S * kb) == 0 && K / S >= 2 * kb) return S;
  return 1;
}

// Tensor maps of an operand's K-range view: S groups of K/S columns, K/S elements apart.
pc_status_t encode_krange_maps(OperandMaps* m, const Operand& op, pc_precision_t p, int box_rows, int S) {
  Operand v = op;
  v.cols = op.cols / S;
  v.groups = S;
  pc_status_t st = encode_operand_map(&m->hi, v, p, box_rows, 0, true, v.cols);
  if (st != PC_OK) return st;
  if (p == PC_PREC_FP32) return encode_operand_map(&m->lo, v, p, box_rows, 1, true, v.cols);
  m->lo = m->hi;
  return PC_OK;
}

// out[i][b] = m_b + log(sum_s part[s][i][b]) (-inf where m_b is -inf or the sum is 0).
__global__ void k_layer_fwd_reduce(int S, int M, int B, const float* __restrict__ part,
                                   const float* __restrict__ colmax, float* __restrict__ out) {
  const int n = M * B;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += gridDim.x * blockDim.x) {
    float sum = part[idx];
    for (int k = 1; k < S; ++k) sum += part[static_cast<long long>(k) * n + idx];
    const float m = colmax[idx % B];
    out[idx] = (m > -INFINITY && sum > 0.f) ? m + logf(sum) : -INFINITY;
  }
}

// e[j][b] = (accumulate ? e : 0) + exp(x[j][b] - m_b) sum_s part[s][j][b].
__global__ void k_layer_elem_reduce(int S, int N, int B, const float* __restrict__ part, const float* __restrict__ x,
                                    const float* __restrict__ colmax, float* __restrict__ e, int accumulate) {
  const int n = N * B;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += gridDim.x * blockDim.x) {
    float sum = part[idx];
    for (int k = 1; k < S; ++k) sum += part[static_cast<long long>(k) * n + idx];
    const float m = colmax[idx % B];
    const float u = m > -INFINITY ? expf(x[idx] - m) : 0.f;
    e[idx] = (accumulate ? e[idx] : 0.f) + u * sum;
  }
}

struct LayerFwdWs {
  float* colmax;
  Operand th, ubm;
  float* part;  // layer_split > 1: the K ranges' partial sums
};
struct LayerBwdWs {
  float* colmax;
  Operand thT, gbm, gnm, unm;
  float* part;
};

size_t carve_fwd(void* base, pc_precision_t p, int G, int M, int N, int B, LayerFwdWs* w) {
  Carver c(base);
  w->colmax = static_cast<float*>(c.take(size_t(G) * B * sizeof(float)));
  w->th = c.operand(p, G, M, N);
  w->ubm = c.operand(p, G, B, N);
  const int S = layer_split(G, M, N, B, p);
  w->part = S > 1 ? static_cast<float*>(c.take(size_t(S) * M * B * sizeof(float))) : nullptr;
  return c.used;
}

size_t carve_bwd(void* base, pc_precision_t p, int G, int M, int N, int B, LayerBwdWs* w) {
  Carver c(base);
  w->colmax = static_cast<float*>(c.take(size_t(G) * B * sizeof(float)));
  w->thT = c.operand(p, G, N, M);
  w->gbm = c.operand(p, G, B, M);
  w->gnm = c.operand(p, G, M, B);
  w->unm = c.operand(p, G, N, B);
  const int S = layer_split(G, N, M, B, p);
  w->part = S > 1 ? static_cast<float*>(c.take(size_t(S) * N * B * sizeof(float))) : nullptr;
  return c.used;
}

size_t layer_ws_bytes(pc_precision_t p, int G, int M, int N, int B) {
  LayerFwdWs f;
  LayerBwdWs b;
  const size_t a = carve_fwd(nullptr, p, G, M, N, B, &f);
  const size_t c = carve_bwd(nullptr, p, G, M, N, B, &b);
  return (a > c ? a : c) + 256;
}

void* align256(void* p) {
  return reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(p) + 255) & ~uintptr_t(255));
}

pc_status_t check_layer_shape(int G, int M, int N, int B, long long cs) {
  PC_CHECK(G >= 1 && M >= 1 && N >= 1 && B >= 1, PC_ERR_SHAPE,
           "G, M, N, B must be >= 1 (got %d, %d, %d, %d)", G, M, N, B);
  PC_CHECK(M < (1 << 24) && N < (1 << 24) && B < (1 << 24) && G <= 65535, PC_ERR_SHAPE,
           "sizes out of range (M, N, B < 2^24, G <= 65535)");
  PC_CHECK(cs >= 0, PC_ERR_SHAPE, "child_stride must be >= 0 (got %lld)", cs);
  PC_CHECK(G == 1 || cs >= N, PC_ERR_SHAPE,
           "with G > 1 groups the child groups must not overlap: child_stride %lld < N %d", cs, N);
  PC_CHECK((static_cast<long long>(G) - 1) * cs + N < (1ll << 31), PC_ERR_SHAPE,
           "x has more than 2^31 rows");
  return PC_OK;
}

template <int P>
pc_status_t layer_fwd(int G, int M, int N, int B, const float* theta, const float* x, long long cs,
                      float* out, pc_precision_t prec, void* ws, cudaStream_t s) {
  LayerFwdWs w;
  carve_fwd(align256(ws), prec, G, M, N, B, &w);
  pc_status_t st;
  k_colmax<<<dim3(cdiv(B, 32), G), dim3(32, 16), 0, s>>>(x, cs, N, B, w.colmax);
  PC_LAUNCH_CHECK();
  if ((st = rows_to_operand<P>(theta, N, static_cast<long long>(M) * N, G, M, N, w.th, s)) != PC_OK) return st;
  if ((st = make_operands<P>(ExpChildren{x, w.colmax, cs, B}, G, N, B, nullptr, &w.ubm, s)) != PC_OK) return st;
  OperandMaps ma, mb;
  const int S = layer_split(G, M, N, B, prec);
  if (S > 1) {
    if ((st = encode_krange_maps(&ma, w.th, prec, kBM, S)) != PC_OK) return st;
    if ((st = encode_krange_maps(&mb, w.ubm, prec, kLayerBN, S)) != PC_OK) return st;
    EpiStoreF32::Params ep{w.part, B, M, B, 0, nullptr, nullptr, static_cast<long long>(M) * B};
    if ((st = launch_gemm<P, kLayerBN, EpiStoreF32>(dim3(cdiv(M, kBM), cdiv(B, kLayerBN), S), ma.hi, ma.lo, mb.hi,
                                                    mb.lo, num_k_blocks(N / S, prec), ep, s, PC_KIND_LAYER_FWD,
                                                    2ll * M * N * B)) != PC_OK)
      return st;
    k_layer_fwd_reduce<<<static_cast<unsigned>(std::min<long long>(cdiv(static_cast<long long>(M) * B, 256), 1184)),
                         256, 0, s>>>(S, M, B, w.part, w.colmax, out);
    PC_LAUNCH_CHECK();
    return PC_OK;
  }
  if ((st = encode_maps(&ma, w.th, prec, kBM)) != PC_OK) return st;
  if ((st = encode_maps(&mb, w.ubm, prec, kLayerBN)) != PC_OK) return st;
  EpiLayerFwd::Params ep{out, w.colmax, M, B};
  return launch_gemm<P, kLayerBN, EpiLayerFwd>(dim3(cdiv(M, kBM), cdiv(B, kLayerBN), G), ma.hi,
                                               ma.lo, mb.hi, mb.lo, num_k_blocks(N, prec), ep, s,
                                               PC_KIND_LAYER_FWD, 2ll * G * M * N * B);
}

template <int P>
pc_status_t layer_bwd(int G, int M, int N, int B, const float* theta, const float* x, long long cs,
                      const float* out, const float* f, float* e, float* F, int accumulate,
                      pc_precision_t prec, void* ws, cudaStream_t s) {
  LayerBwdWs w;
  carve_bwd(align256(ws), prec, G, M, N, B, &w);
  pc_status_t st;
  k_colmax<<<dim3(cdiv(B, 32), G), dim3(32, 16), 0, s>>>(x, cs, N, B, w.colmax);
  PC_LAUNCH_CHECK();
  if ((st = make_operands<P>(ScaledFlow{f, out, w.colmax, M, B}, G, M, B, F ? &w.gnm : nullptr,
                             e ? &w.gbm : nullptr, s)) != PC_OK)
    return st;
  if (e) {
    if ((st = transpose_to_operand<P>(theta, N, static_cast<long long>(M) * N, G, M, N, w.thT, s)) != PC_OK) return st;
    OperandMaps ma, mb;
    const int S = layer_split(G, N, M, B, prec);
    if (S > 1) {
      if ((st = encode_krange_maps(&ma, w.thT, prec, kBM, S)) != PC_OK) return st;
      if ((st = encode_krange_maps(&mb, w.gbm, prec, kLayerBN, S)) != PC_OK) return st;
      EpiStoreF32::Params ep{w.part, B, N, B, 0, nullptr, nullptr, static_cast<long long>(N) * B};
      if ((st = launch_gemm<P, kLayerBN, EpiStoreF32>(dim3(cdiv(N, kBM), cdiv(B, kLayerBN), S), ma.hi, ma.lo, mb.hi,
                                                      mb.lo, num_k_blocks(M / S, prec), ep, s, PC_KIND_LAYER_ELEM,
                                                      2ll * M * N * B)) != PC_OK)
        return st;
      k_layer_elem_reduce<<<static_cast<unsigned>(std::min<long long>(cdiv(static_cast<long long>(N) * B, 256), 1184)),
                            256, 0, s>>>(S, N, B, w.part, x, w.colmax, e, accumulate);
      PC_LAUNCH_CHECK();
    } else {
      if ((st = encode_maps(&ma, w.thT, prec, kBM)) != PC_OK) return st;
      if ((st = encode_maps(&mb, w.gbm, prec, kLayerBN)) != PC_OK) return st;
      EpiLayerElem::Params ep{e, x, w.colmax, cs, N, B, accumulate};
      if ((st = launch_gemm<P, kLayerBN, EpiLayerElem>(dim3(cdiv(N, kBM), cdiv(B, kLayerBN), G), ma.hi,
                                                       ma.lo, mb.hi, mb.lo, num_k_blocks(M, prec), ep,
                                                       s, PC_KIND_LAYER_ELEM, 2ll * G * M * N * B)) != PC_OK)
        return st;
    }
  }
  if (F) {
    if ((st = make_operands<P>(ExpChildren{x, w.colmax, cs, B}, G, N, B, &w.unm, nullptr, s)) != PC_OK) return st;
    OperandMaps ma, mb;
    if ((st = encode_maps(&ma, w.gnm, prec, kBM)) != PC_OK) return st;
    if ((st = encode_maps(&mb, w.unm, prec, kLayerBN)) != PC_OK) return st;
    EpiThetaScale::Params ep{F, theta, M, N, accumulate};
    if ((st = launch_gemm<P, kLayerBN, EpiThetaScale>(dim3(cdiv(M, kBM), cdiv(N, kLayerBN), G), ma.hi,
                                                      ma.lo, mb.hi, mb.lo, num_k_blocks(B, prec), ep,
                                                      s, PC_KIND_LAYER_PARAM, 2ll * G * M * N * B)) != PC_OK)
      return st;
  }
  return PC_OK;
}

}  // namespace
}  // namespace pc

extern "C" {

pc_status_t pc_sum_layer_workspace(int G, int M, int N, int B, pc_precision_t prec, size_t* bytes) {
  pc::clear_error();
  PC_CHECK(bytes != nullptr, PC_ERR_NULL, "bytes is NULL");
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_layer_shape(G, M, N, B, G == 1 ? 0 : N)) != PC_OK) return st;
  *bytes = pc::layer_ws_bytes(prec, G, M, N, B);
  return PC_OK;
}

pc_status_t pc_sum_layer_fwd(int G, int M, int N, int B, const float* theta, const float* x,
                             long long child_stride, float* out, pc_precision_t prec, void* ws,
                             size_t ws_bytes, pc_stream_t stream) {
  pc::clear_error();
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_layer_shape(G, M, N, B, child_stride)) != PC_OK) return st;
  PC_CHECK(theta && x && out, PC_ERR_NULL, "theta, x and out must not be NULL");
  PC_CHECK(ws, PC_ERR_WORKSPACE, "workspace is NULL");
  const size_t need = pc::layer_ws_bytes(prec, G, M, N, B);
  PC_CHECK(ws_bytes >= need, PC_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", ws_bytes, need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (prec) {
    case PC_PREC_AUTO: return pc::layer_fwd<pc::kBF16>(G, M, N, B, theta, x, child_stride, out, prec, ws, s);
    case PC_PREC_TF32: return pc::layer_fwd<pc::kTF32>(G, M, N, B, theta, x, child_stride, out, prec, ws, s);
    default: return pc::layer_fwd<pc::kTF32x3>(G, M, N, B, theta, x, child_stride, out, prec, ws, s);
  }
}

pc_status_t pc_sum_layer_bwd(int G, int M, int N, int B, const float* theta, const float* x,
                             long long child_stride, const float* out, const float* f, float* e,
                             float* F, int accumulate, pc_precision_t prec, void* ws,
                             size_t ws_bytes, pc_stream_t stream) {
  pc::clear_error();
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_layer_shape(G, M, N, B, child_stride)) != PC_OK) return st;
  PC_CHECK(theta && x && out && f, PC_ERR_NULL, "theta, x, out and f must not be NULL");
  if (!e && !F) return PC_OK;
  PC_CHECK(ws, PC_ERR_WORKSPACE, "workspace is NULL");
  const size_t need = pc::layer_ws_bytes(prec, G, M, N, B);
  PC_CHECK(ws_bytes >= need, PC_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", ws_bytes, need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (prec) {
    case PC_PREC_AUTO:
      return pc::layer_bwd<pc::kBF16>(G, M, N, B, theta, x, child_stride, out, f, e, F, accumulate, prec, ws, s);
    case PC_PREC_TF32:
      return pc::layer_bwd<pc::kTF32>(G, M, N, B, theta, x, child_stride, out, f, e, F, accumulate, prec, ws, s);
    default:
      return pc::layer_bwd<pc::kTF32x3>(G, M, N, B, theta, x, child_stride, out, f, e, F, accumulate, prec, ws, s);
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// Forward without a caller workspace. Some callers cannot allocate device memory at
// all: a plugin whose host framework owns every device allocation and hands it no
// allocator, or a hot path where cudaMalloc (and the synchronisation it implies) is
// not allowed. For them the scratch lives in this file-scope device array, which every
// GPU that loads the library holds until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device, looked up once per device
// (host code may not use the symbol itself: it is only a host-side stand-in).
pc_status_t noalloc_scratch(void** ptr) {
  int dev = 0;
  PC_CUDA(cudaGetDevice(&dev));
  PC_CHECK(dev >= 0 && dev < 64, PC_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return pc::set_error(PC_ERR_CUDA, "cudaGetSymbolAddress of the built-in scratch failed: %s",
                           cudaGetErrorString(e));
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return PC_OK;
}

}  // namespace

extern "C" {

pc_status_t pc_sum_layer_fwd_noalloc(int G, int M, int N, int B, const float* theta, const float* x,
                                     long long child_stride, float* out, pc_precision_t prec,
                                     pc_stream_t stream) {
  pc::clear_error();
  pc_status_t st;
  if ((st = pc::check_precision(prec)) != PC_OK) return st;
  if ((st = pc::check_layer_shape(G, M, N, B, child_stride)) != PC_OK) return st;
  PC_CHECK(theta && x && out, PC_ERR_NULL, "theta, x and out must not be NULL");
  const size_t need = pc::layer_ws_bytes(prec, G, M, N, B);
  PC_CHECK(need <= kNoAllocScratchBytes, PC_ERR_UNSUPPORTED,
           "this layer needs %zu bytes of scratch but the built-in scratch holds %zu; call "
           "pc_sum_layer_fwd with a workspace instead",
           need, kNoAllocScratchBytes);
  void* ws = nullptr;
  if ((st = noalloc_scratch(&ws)) != PC_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Every value the forward reads from the scratch is written earlier in the same call,
  // so nothing has to be cleared between calls.
  switch (prec) {
    case PC_PREC_AUTO: return pc::layer_fwd<pc::kBF16>(G, M, N, B, theta, x, child_stride, out, prec, ws, s);
    case PC_PREC_TF32: return pc::layer_fwd<pc::kTF32>(G, M, N, B, theta, x, child_stride, out, prec, ws, s);
    default: return pc::layer_fwd<pc::kTF32x3>(G, M, N, B, theta, x, child_stride, out, prec, ws, s);
  }
}

}  // extern "C"
