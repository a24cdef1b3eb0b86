// HMM circuit whose transition layers carry the LowRank "exp_sum" per-sample scale
// (pyjuice LowRank API doc: intro formulas; Parameters, tie_external off: one pair of
// factor tensors per copy of the tied node vector). Position t's transition layer
// (t = 0 .. T-2) uses factors FA[t] [B][H][K], FB[t] [B][K][H]:
//
//   A_b^(t) = A exp(FA[t][b] FB[t][b]) / Z_b^(t),   S_t = A_b^(t) P_{t+1},
//   P_t = E[., x_t] S_t,   P_{T-1} = E[., x_{T-1}],   LL = log sum_k pi_k P_0(k).
//
// Every transition layer is the fused exp_sum layer (pc_lowrank_exp_sum_fwd / _bwd, the
// scale made tile by tile on the tensor cores and never stored), on the log-values
// log P_{t+1}; the emission products, the root and the flow glue are small kernels here.
// The tied A's statistics are the copies' sums (F+ and W accumulate over t); dE is the
// deterministic per-token gather of the emission flows (pc_tokens.cuh).
//
// The log-values handed from layer to layer are shifted per sample so that their column
// maximum is 0, the shifts summed in double (c_t[b]): unshifted, log P_t reaches hundreds
// of nats, where one float32 ulp is already ~1e-5. Every layer and every flow is
// invariant to such a per-sample shift of its children.
#include "pc_launch.cuh"
#include "pc_tokens.cuh"

namespace pc {
namespace {

// logP[k][b] = S[k][b] (0 if S is NULL) + log E[k][x_{t,b}]: the product with the emission.
__global__ void k_hl_emit(int H, int B, int T, int V, int t, const int* __restrict__ tokens,
                          const float* __restrict__ E, const float* __restrict__ S, float* __restrict__ logP) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(H) * B) return;
  const int k = static_cast<int>(i / B), b = static_cast<int>(i % B);
  const int tok = tokens[static_cast<long long>(b) * T + t];
  const float e = (tok >= 0 && tok < V) ? E[static_cast<long long>(k) * V + tok] : 0.f;
  const float le = e > 0.f ? logf(e) : -INFINITY;
  logP[i] = (S ? S[i] : 0.f) + le;
}

// Shifts column b of logP (node-major [H][B]) to a maximum of 0 and adds the shift to
// c[b] (double; set rather than added for the first position). One block per sample.
__global__ void k_hl_shift(int H, int B, float* __restrict__ logP, double* __restrict__ c, int first) {
  __shared__ float red[32];
  const int b = blockIdx.x;
  float m = -INFINITY;
  for (int k = threadIdx.x; k < H; k += blockDim.x) m = fmaxf(m, logP[static_cast<long long>(k) * B + b]);
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = m;
  __syncthreads();
  m = -INFINITY;
  for (int w = 0; w < static_cast<int>(blockDim.x / 32); ++w) m = fmaxf(m, red[w]);
  if (m == -INFINITY) {  // a sample of zero likelihood: nothing to shift
    if (threadIdx.x == 0) c[b] = -INFINITY;
    return;
  }
  for (int k = threadIdx.x; k < H; k += blockDim.x) logP[static_cast<long long>(k) * B + b] -= m;
  if (threadIdx.x == 0) c[b] = (first ? 0.0 : c[b]) + static_cast<double>(m);
}

// ll[b] = c[b] + log sum_k pi_k exp(logP0[k][b]), in double; one block per sample.
__global__ void k_hl_root(int H, int B, const float* __restrict__ pi, const float* __restrict__ logP0,
                          const double* __restrict__ c, double* __restrict__ ll) {
  __shared__ double red[32];
  const int b = blockIdx.x;
  float m = -INFINITY;
  for (int k = threadIdx.x; k < H; k += blockDim.x)
    if (pi[k] > 0.f) m = fmaxf(m, logf(pi[k]) + logP0[static_cast<long long>(k) * B + b]);
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = m;
  __syncthreads();
  for (int w = 0; w < static_cast<int>(blockDim.x / 32); ++w) m = fmaxf(m, static_cast<float>(red[w]));
  __syncthreads();
  double s = 0.0;
  if (m > -INFINITY)
    for (int k = threadIdx.x; k < H; k += blockDim.x)
      if (pi[k] > 0.f) s += exp(static_cast<double>(logf(pi[k]) + logP0[static_cast<long long>(k) * B + b]) - m);
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < static_cast<int>(blockDim.x / 32); ++w) t += red[w];
    ll[b] = (m > -INFINITY && t > 0.0 && c[b] > -INFINITY) ? c[b] + m + log(t) : -INFINITY;
  }
}

// Root flows: f0[k][b] = pi_k P_0(k) / P(x_b) (0 for a sample of zero likelihood), and
// dpi[k] (+)= sum_b f0[k][b] summed by one thread per k. logP0 is shifted by c (ll holds
// the shift).
__global__ void k_hl_root_flows(int H, int B, const float* __restrict__ pi, const float* __restrict__ logP0,
                                const double* __restrict__ c, const double* __restrict__ ll,
                                float* __restrict__ f0, float* __restrict__ dpi, int accumulate) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= H) return;
  const float lp = pi[k] > 0.f ? logf(pi[k]) : -INFINITY;
  double acc = 0.0;
  for (int b = 0; b < B; ++b) {
    const double l = ll[b] - c[b];  // log P(x_b) relative to the shift of logP0
    const float x = logP0[static_cast<long long>(k) * B + b];
    const float f = (l > -INFINITY && lp > -INFINITY && x > -INFINITY) ? static_cast<float>(exp(lp + x - l)) : 0.f;
    f0[static_cast<long long>(k) * B + b] = f;
    acc += f;
  }
  if (dpi) dpi[k] = (accumulate ? dpi[k] : 0.f) + static_cast<float>(acc);
}

struct HlWs {
  float *logP, *outs, *logZ, *f[2], *fbm, *dEt;
  double* shift;
  int *tok_count, *tok_offset, *tok_order;
  void* lr;
  size_t lr_bytes;
};

size_t carve_hl(void* base, pc_precision_t p, int H, int T, int V, int B, int K, HlWs* w) {
  Carver c(base);
  *w = HlWs{};
  const size_t HB = size_t(H) * B;
  w->logP = static_cast<float*>(c.take(size_t(T) * HB * 4));
  w->shift = static_cast<double*>(c.take(size_t(B) * 8));
  w->outs = static_cast<float*>(c.take(size_t(T > 1 ? T - 1 : 0) * HB * 4));
  w->logZ = static_cast<float*>(c.take(size_t(T > 1 ? T - 1 : 0) * HB * 4));
  w->f[0] = static_cast<float*>(c.take(HB * 4));
  w->f[1] = static_cast<float*>(c.take(HB * 4));
  w->fbm = static_cast<float*>(c.take(size_t(T) * HB * 4));
  w->dEt = static_cast<float*>(c.take(size_t(V) * H * 4));
  w->tok_count = static_cast<int*>(c.take(size_t(V + 1) * 4));
  w->tok_offset = static_cast<int*>(c.take(size_t(V + 1) * 4));
  w->tok_order = static_cast<int*>(c.take(size_t(T) * B * 4));
  size_t lr = 0;
  if (T > 1 && pc_lowrank_exp_sum_workspace(H, H, K, B, 1, p, &lr) != PC_OK) lr = 0;
  w->lr_bytes = lr;
  w->lr = c.take(lr + 256);
  return c.used + 256;
}

pc_status_t check_hl_shape(int H, int T, int V, int B, int K, pc_precision_t prec) {
  pc_status_t st = check_precision(prec);
  if (st != PC_OK) return st;
  PC_CHECK(H >= 1 && T >= 1 && V >= 1 && B >= 1, PC_ERR_SHAPE, "H, T, V, B must be >= 1 (got %d, %d, %d, %d)", H,
           T, V, B);
  PC_CHECK(K >= 1, PC_ERR_SHAPE, "rank K=%d must be at least 1", K);
  PC_CHECK(K <= 64, PC_ERR_UNSUPPORTED, "rank K=%d exceeds the fused layer's limit of 64", K);
  PC_CHECK(H <= 16384 && T <= 4096 && V <= 65536 && B <= 65535, PC_ERR_SHAPE,
           "sizes out of range (H <= 16384, T <= 4096, V <= 65536, B <= 65535)");
  PC_CHECK(static_cast<long long>(T) * B < (1ll << 31), PC_ERR_SHAPE, "T * B must be < 2^31");
  return PC_OK;
}

pc_status_t hl_run(int H, int T, int V, int B, int K, const int32_t* tokens, const float* pi, const float* A,
                   const float* E, const float* FA, const float* FB, double* ll, float* dpi, float* dA, float* Wst,
                   float* dE, float* dFA, float* dFB, int accumulate, pc_precision_t prec, void* ws, cudaStream_t s) {
  HlWs w;
  void* base = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
  carve_hl(base, prec, H, T, V, B, K, &w);
  const long long HB = static_cast<long long>(H) * B;
  const unsigned gHB = cdiv(HB, 256);
  const size_t fa_layer = size_t(B) * H * K;  // one copy's factors (FA and FB alike)
  pc_status_t st;

  // forward: P_{T-1}, then S_t and P_t for t = T-2 .. 0
  k_hl_emit<<<gHB, 256, 0, s>>>(H, B, T, V, T - 1, tokens, E, nullptr, w.logP + (T - 1) * HB);
  PC_LAUNCH_CHECK();
  k_hl_shift<<<B, 256, 0, s>>>(H, B, w.logP + (T - 1) * HB, w.shift, 1);
  PC_LAUNCH_CHECK();
  for (int t = T - 2; t >= 0; --t) {
    if ((st = pc_lowrank_exp_sum_fwd(H, H, K, B, A, FA + t * fa_layer, FB + t * fa_layer, w.logP + (t + 1) * HB,
                                     w.outs + t * HB, w.logZ + t * HB, prec, w.lr, w.lr_bytes, s)) != PC_OK)
      return st;
    k_hl_emit<<<gHB, 256, 0, s>>>(H, B, T, V, t, tokens, E, w.outs + t * HB, w.logP + t * HB);
    PC_LAUNCH_CHECK();
    k_hl_shift<<<B, 256, 0, s>>>(H, B, w.logP + t * HB, w.shift, 0);
    PC_LAUNCH_CHECK();
  }
  k_hl_root<<<B, 256, 0, s>>>(H, B, pi, w.logP, w.shift, ll);
  PC_LAUNCH_CHECK();
  const bool flows = dpi || dA || Wst || dE || dFA || dFB;
  if (!flows) return PC_OK;

  // backward: the flow of S_t is P_t's; the layer's element flows are P_{t+1}'s
  if (!accumulate) {
    if (dA) PC_CUDA(cudaMemsetAsync(dA, 0, size_t(H) * H * 4, s));
    if (Wst) PC_CUDA(cudaMemsetAsync(Wst, 0, size_t(H) * H * 4, s));
    if (dFA && T > 1) PC_CUDA(cudaMemsetAsync(dFA, 0, size_t(T - 1) * fa_layer * 4, s));
    if (dFB && T > 1) PC_CUDA(cudaMemsetAsync(dFB, 0, size_t(T - 1) * fa_layer * 4, s));
  }
  k_hl_root_flows<<<cdiv(H, 256), 256, 0, s>>>(H, B, pi, w.logP, w.shift, ll, w.f[0], dpi, accumulate);
  PC_LAUNCH_CHECK();
  for (int t = 0; t < T; ++t) {
    const float* f = w.f[t & 1];
    if (dE && (st = transpose_f32(f, B, 0, 1, H, B, w.fbm + t * HB, H, 0, s)) != PC_OK) return st;  // [b][k]
    if (t == T - 1) break;
    float* e = w.f[(t + 1) & 1];
    PC_CUDA(cudaMemsetAsync(e, 0, size_t(HB) * 4, s));
    if ((st = pc_lowrank_exp_sum_bwd(H, H, K, B, A, FA + t * fa_layer, FB + t * fa_layer, w.logP + (t + 1) * HB,
                                     w.outs + t * HB, w.logZ + t * HB, f, dFA ? dFA + t * fa_layer : nullptr,
                                     dFB ? dFB + t * fa_layer : nullptr, e, dA, Wst, 1, prec, w.lr, w.lr_bytes,
                                     s)) != PC_OK)
      return st;
  }
  if (dE) {
    PC_CUDA(cudaMemsetAsync(w.tok_count, 0, size_t(V + 1) * 4, s));
    k_token_hist<<<cdiv(static_cast<long long>(T) * B, 256), 256, 0, s>>>(tokens, T * B, V, w.tok_count);
    PC_LAUNCH_CHECK();
    k_exclusive_scan<<<1, 1024, 0, s>>>(w.tok_count, V, w.tok_offset);
    PC_LAUNCH_CHECK();
    k_token_bucket<<<cdiv(V, kBucketSpan), 256, 0, s>>>(tokens, T, B, V, w.tok_offset, w.tok_order);
    PC_LAUNCH_CHECK();
    k_dE_gather<<<dim3(V, cdiv(H, 256)), 256, 0, s>>>(w.fbm, H, w.tok_offset, w.tok_order, w.dEt);
    PC_LAUNCH_CHECK();
    if ((st = transpose_f32(w.dEt, H, 0, 1, V, H, dE, V, accumulate, s)) != PC_OK) return st;
  }
  return PC_OK;
}

}  // namespace
}  // namespace pc

using namespace pc;

extern "C" {

pc_status_t pc_hmm_lowrank_workspace(int H, int T, int V, int B, int K, pc_precision_t prec, size_t* bytes) {
  clear_error();
  PC_CHECK(bytes, PC_ERR_NULL, "bytes is NULL");
  pc_status_t st = check_hl_shape(H, T, V, B, K, prec);
  if (st != PC_OK) return st;
  HlWs w;
  *bytes = carve_hl(nullptr, prec, H, T, V, B, K, &w) + 256;
  return PC_OK;
}

pc_status_t pc_hmm_lowrank_fwd_bwd(int H, int T, int V, int B, int K, const int32_t* tokens, const float* pi,
                                   const float* A, const float* E, const float* FA, const float* FB, double* ll,
                                   float* dpi, float* dA, float* Wstat, float* dE, float* dFA, float* dFB,
                                   int accumulate, pc_precision_t prec, void* ws, size_t ws_bytes,
                                   pc_stream_t stream) {
  clear_error();
  pc_status_t st = check_hl_shape(H, T, V, B, K, prec);
  if (st != PC_OK) return st;
  PC_CHECK(tokens && pi && A && E && ll, PC_ERR_NULL, "tokens, pi, A, E and ll are required");
  PC_CHECK(T == 1 || (FA && FB), PC_ERR_NULL, "the factors FA and FB are required when T > 1");
  PC_CHECK(ws, PC_ERR_NULL, "workspace is NULL");
  PC_CHECK(aligned16(ws), PC_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  HlWs w;
  const size_t need = carve_hl(nullptr, prec, H, T, V, B, K, &w) + 256;
  PC_CHECK(ws_bytes >= need, PC_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, need);
  return hl_run(H, T, V, B, K, tokens, pi, A, E, FA, FB, ll, dpi, dA, Wstat, dE, dFA, dFB, accumulate, prec, ws,
                static_cast<cudaStream_t>(stream));
}

}  // extern "C"
