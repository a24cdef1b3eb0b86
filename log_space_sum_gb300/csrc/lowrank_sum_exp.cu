// LowRank "sum_exp" scale (pyjuice LowRank API doc, intro formulas): per sample b,
//
//   g_b[i,j] = sum_r exp(A_b[i,r]) exp(B_b[r,j]),   Z_b[i] = sum_j theta[i,j] g_b[i,j],
//   theta_b  = theta g_b / Z_b,                     out[i,b] = log sum_j theta_b[i,j] e^x[j,b].
//
// As the doc says of this form, it is k matmuls with the shared parameters: every pass is
// a dense contraction over a virtual batch of the B*K (sample, rank) pairs, run by the
// same tcgen05 contraction as the plain sum layers (k_umma_gemm), with the exponentials
// and the reductions over the rank in small element-wise kernels around it. With the row
// maxima beta_{b,r} = max_j B_b[r,j], m_b = max_j x[j,b], alpha_{b,i} = max_r (A_b[i,r] +
// beta_{b,r}) and
//
//   c[b,r,j] = exp(B_b[r,j] - beta_{b,r})            <= 1
//   v[j,b]   = exp(x[j,b] - m_b)                     <= 1
//   a[b,i,r] = exp(A_b[i,r] + beta_{b,r} - alpha_{b,i})   <= 1
//
// (the shifts cancel in theta_b), the forward is
//
//   P[i,(b,r)] = sum_j theta[i,j] c[b,r,j] v[j,b],   Q[i,(b,r)] = sum_j theta[i,j] c[b,r,j]
//   num = sum_r a P,  Z' = sum_r a Q,  out = m_b + log num - log Z',  log Z = alpha + log Z'
//
// and, with s = f / num and t = f / Z' per (node, sample), the backward (the chain rule
// through d(sum f out)/dg = f (p - q) / g, in which g cancels):
//
//   dA[b,i,r]  = a (s P - t Q)
//   U[j,(b,r)] = sum_i theta[i,j] a[b,i,r] s[i,b]   (and U' with t in place of s)
//   dB[b,r,j]  = c v U - c U',    e[j,b] = v sum_r c U
//   F+[i,j]    = theta[i,j] sum_(b,r) (a s)[i,(b,r)] (c v)[j,(b,r)]
//   W[i,j]     = sum_(b,r) (a t)[i,(b,r)] c[j,(b,r)].
//
// Contractions: P|Q (M x 2BK x N), U|U' (N x 2BK x M), F+ and W (M x N x BK).
//
// Opt-in fp8 flow products (the doc's flow_precision "fp8", precision auto only): the two
// flow contractions take e4m3 operands, each operand row scaled by a power of two that
// brings its largest magnitude within the e4m3 range (448), accumulated in float32; the
// epilogue multiplies by the inverse row scales of both operands.
#include <cuda_fp8.h>

#include "pc_launch.cuh"

namespace pc {
namespace {

constexpr int kSeBN = 128;  // column tile of the contractions

// out[r] = max over the row of src (rows ld apart, n values); -inf for an empty row.
__global__ void k_se_rowmax(const float* __restrict__ src, long long ld, int rows, int n, float* __restrict__ out) {
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* p = src + static_cast<long long>(row) * ld;
  float m = -INFINITY;
  for (int j = lane; j < n; j += 32) m = fmaxf(m, p[j]);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) out[row] = m;
}

// The virtual batch's child factors, float32 [2][B*K][N]: CV[0][(b,r)][j] = c v and
// CV[1][(b,r)][j] = c. xT is x transposed, [B][N].
__global__ void k_se_child_factors(const float* __restrict__ Bm, const float* __restrict__ xT,
                                   const float* __restrict__ beta, const float* __restrict__ m, int N, int K,
                                   long long V, float* __restrict__ CV) {
  const long long vr = blockIdx.x;  // (b, r) = b * K + r
  const int b = static_cast<int>(vr / K);
  const int j = blockIdx.y * blockDim.x + threadIdx.x;
  if (j >= N) return;
  const float c = expf(Bm[vr * N + j] - beta[vr]);
  const float mb = m[b];
  const float v = mb == -INFINITY ? 0.f : expf(xT[static_cast<long long>(b) * N + j] - mb);
  CV[vr * N + j] = c * v;
  CV[(V + vr) * N + j] = c;
}

// Per (node i, sample b): alpha, num and Z' from the contraction P|Q ([M][2V], columns
// (kind, b, r)). Forward: out and log Z. Backward: dA, and the node-side factors of the
// flow contractions, L[kind][(b,r)][i] = a s (kind 0) and a t (kind 1), float32.
template <bool kBwd>
__global__ void k_se_nodes(int M, int K, int B, const float* __restrict__ A, const float* __restrict__ beta,
                           const float* __restrict__ m, const float* __restrict__ PQ, long long V,
                           const float* __restrict__ f, float* __restrict__ out, float* __restrict__ logZ,
                           float* __restrict__ dA, int accumulate, float* __restrict__ L) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(M) * B) return;
  const int i = static_cast<int>(idx % M), b = static_cast<int>(idx / M);
  const float* a_row = A + (static_cast<long long>(b) * M + i) * K;
  const float* bt = beta + static_cast<long long>(b) * K;
  float alpha = -INFINITY;
  for (int r = 0; r < K; ++r) alpha = fmaxf(alpha, a_row[r] + bt[r]);
  const float* P = PQ + static_cast<long long>(i) * 2 * V + static_cast<long long>(b) * K;
  const float* Q = P + V;
  float num = 0.f, zp = 0.f;
  for (int r = 0; r < K; ++r) {
    const float a = expf(a_row[r] + bt[r] - alpha);
    num += a * P[r];
    zp += a * Q[r];
  }
  const bool live = num > 0.f && zp > 0.f && m[b] > -INFINITY;  // otherwise out = -inf, no flow
  if constexpr (!kBwd) {
    out[static_cast<long long>(i) * B + b] = live ? m[b] + logf(num) - logf(zp) : -INFINITY;
    logZ[static_cast<long long>(b) * M + i] = zp > 0.f ? alpha + logf(zp) : -INFINITY;
  } else {
    const float fb = f[static_cast<long long>(i) * B + b];
    const float s = live ? fb / num : 0.f;
    const float t = live ? fb / zp : 0.f;
    float* dA_row = dA ? dA + (static_cast<long long>(b) * M + i) * K : nullptr;
    for (int r = 0; r < K; ++r) {
      const float a = expf(a_row[r] + bt[r] - alpha);
      if (dA_row) dA_row[r] = (accumulate ? dA_row[r] : 0.f) + a * (s * P[r] - t * Q[r]);
      const long long vr = static_cast<long long>(b) * K + r;
      L[vr * M + i] = a * s;
      L[(V + vr) * M + i] = a * t;
    }
  }
}

// dB[b][r][j] (+)= CV0 U - CV1 U' and e[j][b] (+)= sum_r CV0 U, from U|U' ([N][2V]).
__global__ void k_se_children(int N, int K, int B, long long V, const float* __restrict__ CV,
                              const float* __restrict__ U, float* __restrict__ dB, float* __restrict__ e,
                              int accumulate) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int b = blockIdx.y;
  if (j >= N) return;
  const float* u = U + static_cast<long long>(j) * 2 * V + static_cast<long long>(b) * K;
  float acc = 0.f;
  for (int r = 0; r < K; ++r) {
    const long long vr = static_cast<long long>(b) * K + r;
    const float cv = CV[vr * N + j], c = CV[(V + vr) * N + j];
    acc += cv * u[r];
    if (dB) {
      float* d = dB + vr * N + j;
      *d = (accumulate ? *d : 0.f) + cv * u[r] - c * u[V + r];
    }
  }
  if (e) {
    float* d = e + static_cast<long long>(j) * B + b;
    *d = (accumulate ? *d : 0.f) + acc;
  }
}

// dst[r][c] = e4m3(src[r][c] * 2^e_r) with 2^e_r the largest power of two for which the
// row's largest magnitude stays within 448; inv[r] = 2^-e_r. One block per row.
__global__ void k_se_rows_to_fp8(const float* __restrict__ src, long long ld_src, int C, uint8_t* __restrict__ dst,
                                 long long ld_dst, float* __restrict__ inv) {
  __shared__ float red[32];
  const long long r = blockIdx.x;
  const float* row = src + r * ld_src;
  float m = 0.f;
  for (int c = threadIdx.x; c < C; c += blockDim.x) m = fmaxf(m, fabsf(row[c]));
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = m;
  __syncthreads();
  m = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x / 32); ++w) m = fmaxf(m, red[w]);
  int k = 0;
  if (m > 0.f) frexpf(448.f / m, &k);  // 448 / m = f 2^k, f in [0.5, 1): floor(log2) = k - 1
  const float sc = m > 0.f ? ldexpf(1.f, k - 1) : 1.f;
  uint8_t* out = dst + r * ld_dst;
  for (int c = threadIdx.x; c < C; c += blockDim.x) out[c] = __nv_fp8_e4m3(row[c] * sc).__x;
  if (threadIdx.x == 0) inv[r] = 1.f / sc;
}

__global__ void k_se_fill(float* __restrict__ p, long long n, float v) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}

struct SeWs {
  float *xT, *m, *beta, *CV, *PQ, *L, *U;
  Operand th, thT, Vop, Lop, LsT, LtT, RvT, RcT;
  float *T8a, *T8b, *inv_a, *inv_b;  // fp8 flow products: float32 transposes, inverse row scales
  Operand A8, B8;                     // and the e4m3 operands
};

size_t carve_se(void* base, pc_precision_t p, int M, int N, int K, int B, bool bwd, SeWs* w) {
  Carver c(base);
  *w = SeWs{};
  const long long V = static_cast<long long>(B) * K;
  w->xT = static_cast<float*>(c.take(size_t(B) * N * 4));
  w->m = static_cast<float*>(c.take(size_t(B) * 4));
  w->beta = static_cast<float*>(c.take(size_t(V) * 4));
  w->CV = static_cast<float*>(c.take(size_t(2 * V) * N * 4));
  w->PQ = static_cast<float*>(c.take(size_t(M) * 2 * V * 4));
  w->th = c.operand(p, 1, M, N);
  w->Vop = c.operand(p, 1, 2 * V, N);
  if (bwd) {
    w->L = static_cast<float*>(c.take(size_t(2 * V) * M * 4));
    w->U = static_cast<float*>(c.take(size_t(N) * 2 * V * 4));
    w->thT = c.operand(p, 1, N, M);
    w->Lop = c.operand(p, 1, 2 * V, M);
    w->LsT = c.operand(p, 1, M, V);
    w->LtT = c.operand(p, 1, M, V);
    w->RvT = c.operand(p, 1, N, V);
    w->RcT = c.operand(p, 1, N, V);
    if (p == PC_PREC_AUTO) {
      w->T8a = static_cast<float*>(c.take(size_t(M) * V * 4));
      w->T8b = static_cast<float*>(c.take(size_t(N) * V * 4));
      w->inv_a = static_cast<float*>(c.take(size_t(M) * 4));
      w->inv_b = static_cast<float*>(c.take(size_t(N) * 4));
      w->A8 = c.operand(kPrecFp8Ops, 1, M, V);
      w->B8 = c.operand(kPrecFp8Ops, 1, N, V);
    }
  }
  return c.used + 256;
}

pc_status_t check_se_shape(int M, int N, int K, int B, pc_precision_t prec) {
  pc_status_t st = check_precision(prec);
  if (st != PC_OK) return st;
  PC_CHECK(M >= 0 && N >= 0 && B >= 0, PC_ERR_SHAPE, "negative size (M=%d N=%d B=%d)", M, N, B);
  PC_CHECK(K >= 1, PC_ERR_SHAPE, "rank K=%d must be at least 1", K);
  PC_CHECK(B <= 65535, PC_ERR_SHAPE, "batch B=%d exceeds 65535", B);
  PC_CHECK(static_cast<long long>(B) * K <= (1ll << 22), PC_ERR_SHAPE, "B*K=%lld exceeds 2^22",
           static_cast<long long>(B) * K);
  PC_CHECK(N <= (1 << 24) && M <= (1 << 24), PC_ERR_SHAPE, "M, N must be <= 2^24");
  return PC_OK;
}

// The shared part of both passes: the row maxima, the child factors and P|Q.
template <int P>
pc_status_t se_core(int M, int N, int K, int B, const float* theta, const float* Bm, const float* x,
                    pc_precision_t prec, int kind, const SeWs& w, cudaStream_t s) {
  const long long V = static_cast<long long>(B) * K;
  pc_status_t st;
  if ((st = transpose_f32(x, B, 0, 1, N, B, w.xT, N, 0, s)) != PC_OK) return st;  // xT[b][j] = x[j][b]
  k_se_rowmax<<<cdiv(B, 8), 256, 0, s>>>(w.xT, N, B, N, w.m);
  PC_LAUNCH_CHECK();
  k_se_rowmax<<<cdiv(V, 8), 256, 0, s>>>(Bm, N, static_cast<int>(V), N, w.beta);
  PC_LAUNCH_CHECK();
  k_se_child_factors<<<dim3(static_cast<unsigned>(V), cdiv(N, 256)), 256, 0, s>>>(Bm, w.xT, w.beta, w.m, N, K, V,
                                                                                 w.CV);
  PC_LAUNCH_CHECK();
  if ((st = rows_to_operand<P>(theta, N, 0, 1, M, N, w.th, s)) != PC_OK) return st;
  if ((st = rows_to_operand<P>(w.CV, N, 0, 1, static_cast<int>(2 * V), N, w.Vop, s)) != PC_OK) return st;
  OperandMaps ma, mb;
  if ((st = encode_maps(&ma, w.th, prec, kBM)) != PC_OK) return st;
  if ((st = encode_maps(&mb, w.Vop, prec, kSeBN)) != PC_OK) return st;
  EpiStoreF32::Params ep{w.PQ, 2 * V, M, static_cast<int>(2 * V), 0};
  return launch_gemm<P, kSeBN, EpiStoreF32>(dim3(cdiv(M, kBM), cdiv(2 * V, kSeBN), 1), ma.hi, ma.lo, mb.hi, mb.lo,
                                            num_k_blocks(N, prec), ep, s, kind, 2ll * M * 2 * V * N);
}

template <int P>
pc_status_t se_fwd(int M, int N, int K, int B, const float* theta, const float* A, const float* Bm, const float* x,
                   float* out, float* logZ, pc_precision_t prec, void* ws, cudaStream_t s) {
  if (M == 0 || B == 0) return PC_OK;
  const long long MB = static_cast<long long>(M) * B;
  if (N == 0) {  // no children: every node's sum is empty
    k_se_fill<<<cdiv(MB, 256), 256, 0, s>>>(out, MB, -INFINITY);
    PC_LAUNCH_CHECK();
    k_se_fill<<<cdiv(MB, 256), 256, 0, s>>>(logZ, MB, -INFINITY);
    PC_LAUNCH_CHECK();
    return PC_OK;
  }
  SeWs w;
  carve_se(ws, prec, M, N, K, B, false, &w);
  pc_status_t st = se_core<P>(M, N, K, B, theta, Bm, x, prec, PC_KIND_LOWRANK_FWD, w, s);
  if (st != PC_OK) return st;
  k_se_nodes<false><<<cdiv(MB, 256), 256, 0, s>>>(M, K, B, A, w.beta, w.m, w.PQ, static_cast<long long>(B) * K,
                                                  nullptr, out, logZ, nullptr, 0, nullptr);
  PC_LAUNCH_CHECK();
  return PC_OK;
}

template <int P>
pc_status_t se_bwd(int M, int N, int K, int B, const float* theta, const float* A, const float* Bm, const float* x,
                   const float* f, float* dA, float* dB, float* e, float* Fp, float* W, int accumulate,
                   bool flow_fp8, pc_precision_t prec, void* ws, cudaStream_t s) {
  if (!accumulate) {  // outputs that no pass writes when a size is zero
    if (dA && N == 0) PC_CUDA(cudaMemsetAsync(dA, 0, size_t(B) * M * K * 4, s));
    if (dB && M == 0) PC_CUDA(cudaMemsetAsync(dB, 0, size_t(B) * K * N * 4, s));
    if (e && M == 0) PC_CUDA(cudaMemsetAsync(e, 0, size_t(N) * B * 4, s));
    if (Fp && B == 0) PC_CUDA(cudaMemsetAsync(Fp, 0, size_t(M) * N * 4, s));
    if (W && B == 0) PC_CUDA(cudaMemsetAsync(W, 0, size_t(M) * N * 4, s));
  }
  if (M == 0 || N == 0 || B == 0) return PC_OK;
  const long long V = static_cast<long long>(B) * K;
  SeWs w;
  carve_se(ws, prec, M, N, K, B, true, &w);
  pc_status_t st = se_core<P>(M, N, K, B, theta, Bm, x, prec, PC_KIND_LOWRANK_BWD, w, s);
  if (st != PC_OK) return st;
  k_se_nodes<true><<<cdiv(static_cast<long long>(M) * B, 256), 256, 0, s>>>(M, K, B, A, w.beta, w.m, w.PQ, V, f,
                                                                            nullptr, nullptr, dA, accumulate, w.L);
  PC_LAUNCH_CHECK();
  if (dB || e) {  // U|U' = theta^T [a s | a t], then dB and e
    if ((st = transpose_to_operand<P>(theta, N, 0, 1, M, N, w.thT, s)) != PC_OK) return st;
    if ((st = rows_to_operand<P>(w.L, M, 0, 1, static_cast<int>(2 * V), M, w.Lop, s)) != PC_OK) return st;
    OperandMaps ma, mb;
    if ((st = encode_maps(&ma, w.thT, prec, kBM)) != PC_OK) return st;
    if ((st = encode_maps(&mb, w.Lop, prec, kSeBN)) != PC_OK) return st;
    EpiStoreF32::Params ep{w.U, 2 * V, N, static_cast<int>(2 * V), 0};
    if ((st = launch_gemm<P, kSeBN, EpiStoreF32>(dim3(cdiv(N, kBM), cdiv(2 * V, kSeBN), 1), ma.hi, ma.lo, mb.hi,
                                                 mb.lo, num_k_blocks(M, prec), ep, s, PC_KIND_LOWRANK_BWD,
                                                 2ll * N * 2 * V * M)) != PC_OK)
      return st;
    k_se_children<<<dim3(cdiv(N, 256), B), 256, 0, s>>>(N, K, B, V, w.CV, w.U, dB, e, accumulate);
    PC_LAUNCH_CHECK();
  }
  if constexpr (P == kBF16) {
    if (flow_fp8) {  // both flow contractions on e4m3 operands
      for (int kind = 0; kind < 2; ++kind) {
        float* out = kind == 0 ? Fp : W;
        if (!out) continue;
        if ((st = transpose_f32(w.L + kind * V * M, M, 0, 1, static_cast<int>(V), M, w.T8a, V, 0, s)) != PC_OK)
          return st;
        if ((st = transpose_f32(w.CV + kind * V * N, N, 0, 1, static_cast<int>(V), N, w.T8b, V, 0, s)) != PC_OK)
          return st;
        k_se_rows_to_fp8<<<M, 256, 0, s>>>(w.T8a, V, static_cast<int>(V), static_cast<uint8_t*>(w.A8.ptr), w.A8.ld,
                                           w.inv_a);
        PC_LAUNCH_CHECK();
        k_se_rows_to_fp8<<<N, 256, 0, s>>>(w.T8b, V, static_cast<int>(V), static_cast<uint8_t*>(w.B8.ptr), w.B8.ld,
                                           w.inv_b);
        PC_LAUNCH_CHECK();
        OperandMaps ma, mb;
        if ((st = encode_maps(&ma, w.A8, kPrecFp8Ops, kBM)) != PC_OK) return st;
        if ((st = encode_maps(&mb, w.B8, kPrecFp8Ops, kSeBN)) != PC_OK) return st;
        const dim3 grid(cdiv(M, kBM), cdiv(N, kSeBN), 1);
        const int nkb = num_k_blocks(V, kPrecFp8Ops);
        if (kind == 0) {
          EpiThetaScale::Params ep{Fp, theta, M, N, accumulate, nullptr, w.inv_a, w.inv_b};
          st = launch_gemm<kFP8, kSeBN, EpiThetaScale>(grid, ma.hi, ma.lo, mb.hi, mb.lo, nkb, ep, s,
                                                        PC_KIND_LOWRANK_BWD, 2ll * M * N * V);
        } else {
          EpiStoreF32::Params ep{W, N, M, N, accumulate, w.inv_a, w.inv_b};
          st = launch_gemm<kFP8, kSeBN, EpiStoreF32>(grid, ma.hi, ma.lo, mb.hi, mb.lo, nkb, ep, s,
                                                      PC_KIND_LOWRANK_BWD, 2ll * M * N * V);
        }
        if (st != PC_OK) return st;
      }
      return PC_OK;
    }
  }
  if (Fp) {  // F+ = theta * ((a s) (c v)^T) over the virtual batch
    if ((st = transpose_to_operand<P>(w.L, M, 0, 1, static_cast<int>(V), M, w.LsT, s)) != PC_OK) return st;
    if ((st = transpose_to_operand<P>(w.CV, N, 0, 1, static_cast<int>(V), N, w.RvT, s)) != PC_OK) return st;
    OperandMaps ma, mb;
    if ((st = encode_maps(&ma, w.LsT, prec, kBM)) != PC_OK) return st;
    if ((st = encode_maps(&mb, w.RvT, prec, kSeBN)) != PC_OK) return st;
    EpiThetaScale::Params ep{Fp, theta, M, N, accumulate, nullptr};
    if ((st = launch_gemm<P, kSeBN, EpiThetaScale>(dim3(cdiv(M, kBM), cdiv(N, kSeBN), 1), ma.hi, ma.lo, mb.hi, mb.lo,
                                                   num_k_blocks(V, prec), ep, s, PC_KIND_LOWRANK_BWD,
                                                   2ll * M * N * V)) != PC_OK)
      return st;
  }
  if (W) {  // W = (a t) c^T over the virtual batch
    if ((st = transpose_to_operand<P>(w.L + V * M, M, 0, 1, static_cast<int>(V), M, w.LtT, s)) != PC_OK) return st;
    if ((st = transpose_to_operand<P>(w.CV + V * N, N, 0, 1, static_cast<int>(V), N, w.RcT, s)) != PC_OK) return st;
    OperandMaps ma, mb;
    if ((st = encode_maps(&ma, w.LtT, prec, kBM)) != PC_OK) return st;
    if ((st = encode_maps(&mb, w.RcT, prec, kSeBN)) != PC_OK) return st;
    EpiStoreF32::Params ep{W, N, M, N, accumulate};
    if ((st = launch_gemm<P, kSeBN, EpiStoreF32>(dim3(cdiv(M, kBM), cdiv(N, kSeBN), 1), ma.hi, ma.lo, mb.hi, mb.lo,
                                                 num_k_blocks(V, prec), ep, s, PC_KIND_LOWRANK_BWD,
                                                 2ll * M * N * V)) != PC_OK)
      return st;
  }
  return PC_OK;
}

}  // namespace
}  // namespace pc

using namespace pc;

extern "C" {

pc_status_t pc_lowrank_sum_exp_workspace(int M, int N, int K, int B, int with_backward, pc_precision_t prec,
                                         size_t* bytes) {
  clear_error();
  PC_CHECK(bytes, PC_ERR_NULL, "bytes is NULL");
  pc_status_t st = check_se_shape(M, N, K, B, prec);
  if (st != PC_OK) return st;
  SeWs w;
  *bytes = carve_se(nullptr, prec, M, N, K, B, with_backward != 0, &w);
  return PC_OK;
}

pc_status_t pc_lowrank_sum_exp_fwd(int M, int N, int K, int B, const float* theta, const float* A, const float* Bm,
                                   const float* x, float* out, float* logZ, pc_precision_t prec, void* ws,
                                   size_t ws_bytes, pc_stream_t stream) {
  clear_error();
  pc_status_t st = check_se_shape(M, N, K, B, prec);
  if (st != PC_OK) return st;
  const bool work = M > 0 && B > 0;
  PC_CHECK(!work || (out && logZ), PC_ERR_NULL, "out and logZ are required");
  PC_CHECK(!work || N == 0 || (theta && A && Bm && x), PC_ERR_NULL, "theta, A, B and x are required");
  PC_CHECK(ws || !work, PC_ERR_NULL, "workspace is NULL");
  PC_CHECK(!ws || aligned16(ws), PC_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  SeWs w;
  const size_t need = carve_se(nullptr, prec, M, N, K, B, false, &w);
  PC_CHECK(!work || ws_bytes >= need, PC_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (prec) {
    case PC_PREC_AUTO: return se_fwd<kBF16>(M, N, K, B, theta, A, Bm, x, out, logZ, prec, ws, s);
    case PC_PREC_TF32: return se_fwd<kTF32>(M, N, K, B, theta, A, Bm, x, out, logZ, prec, ws, s);
    default: return se_fwd<kTF32x3>(M, N, K, B, theta, A, Bm, x, out, logZ, prec, ws, s);
  }
}

pc_status_t pc_lowrank_sum_exp_bwd(int M, int N, int K, int B, const float* theta, const float* A, const float* Bm,
                                   const float* x, const float* f, float* dA, float* dB, float* e, float* Fplus,
                                   float* Wstat, int accumulate, int flow_fp8, pc_precision_t prec, void* ws,
                                   size_t ws_bytes, pc_stream_t stream) {
  clear_error();
  pc_status_t st = check_se_shape(M, N, K, B, prec);
  if (st != PC_OK) return st;
  const bool work = M > 0 && N > 0 && B > 0;
  PC_CHECK(!work || (theta && A && Bm && x && f), PC_ERR_NULL, "theta, A, B, x and f are required");
  PC_CHECK(ws || !work, PC_ERR_NULL, "workspace is NULL");
  PC_CHECK(!ws || aligned16(ws), PC_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  SeWs w;
  const size_t need = carve_se(nullptr, prec, M, N, K, B, true, &w);
  PC_CHECK(!work || ws_bytes >= need, PC_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (prec) {
    case PC_PREC_AUTO:
      return se_bwd<kBF16>(M, N, K, B, theta, A, Bm, x, f, dA, dB, e, Fplus, Wstat, accumulate, flow_fp8 != 0, prec,
                           ws, s);
    case PC_PREC_TF32:
      return se_bwd<kTF32>(M, N, K, B, theta, A, Bm, x, f, dA, dB, e, Fplus, Wstat, accumulate, false, prec, ws, s);
    default:
      return se_bwd<kTF32x3>(M, N, K, B, theta, A, Bm, x, f, dA, dB, e, Fplus, Wstat, accumulate, false, prec, ws,
                             s);
  }
}

}  // extern "C"
