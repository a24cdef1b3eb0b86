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
// Values. Every node keeps u_v[b][z] = n_v(z) / max_z n_v(z) (so max_z u_v = 1) and a
// per-sample log-offset O_v[b] = log max_z n_v in double. Each edge's sum layer
//   D_c[b][z] = sum_{z'} W_c[z,z'] u_c[b][z']
// is kept linear, and the product layer multiplies in float32 with an exact power-of-two
// exponent carried beside every running product, so a node with many children cannot
// underflow and no rounding but the multiplies' own round-to-nearest enters:
//   n'_v[b][z] = E_v[z, x_v] * prod_c D_c[b][z] = m_z 2^{e_z}   (m_z in [1/2, 1)),
//   u_v = n'_v / max_z n'_v,   O_v = log max_z n'_v + sum_c O_c,
//   LL_b = O_0[b] + log sum_z pi[z] u_0[b][z].
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
// Et[v][k][z] = E[v][z][k]: per-variable transpose, so that the emissions of one category
// are a contiguous row over the latents.
__global__ void k_hclt_et(const float* __restrict__ E, int H, int C, float* __restrict__ Et) {
  __shared__ float tile[32][33];
  const long long v = blockIdx.z;
  const int k0 = blockIdx.x * 32, z0 = blockIdx.y * 32;
  const float* src = E + v * H * C;
  float* dst = Et + v * H * C;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int z = z0 + i, k = k0 + threadIdx.x;
    tile[i][threadIdx.x] = (z < H && k < C) ? src[static_cast<long long>(z) * C + k] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int k = k0 + i, z = z0 + threadIdx.x;
    if (z < H && k < C) dst[static_cast<long long>(k) * H + z] = tile[threadIdx.x][i];
  }
}

// Product layer of the nodes in slots [s0, s0 + gridDim.x), one block per (node, sample):
// n' = E_v[., x_v] * prod_children D as float32 mantissas in [1/2, 1) with int exponents,
// u = n' / max n' (float32 and operand copies), O = log max n' + sum_children O. For the
// root it also forms LL and 1 / sum pi u.
template <int P>
__global__ void k_hclt_product(int s0, int root_slot, int nvars, int H, int B, const int* __restrict__ data,
                               const int* __restrict__ var_of_slot, const int* __restrict__ child_ptr,
                               const int* __restrict__ child_slots, const float* __restrict__ Et,
                               const float* __restrict__ D, int C, float* __restrict__ U32, void* uop,
                               long long uop_ld, size_t uop_lo, double* __restrict__ O, const float* __restrict__ pi,
                               double* __restrict__ ll, float* __restrict__ rroot) {
  extern __shared__ float mant[];  // H mantissas, then H exponents
  int* expo = reinterpret_cast<int*>(mant + H);
  __shared__ long long red[32];
  __shared__ double redd[32];
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
  for (int z = threadIdx.x; z < H; z += blockDim.x) {
    int e, k;
    float m = frexpf(xin ? er[z] : 0.f, &e);
    for (int c = c0; c < c1; ++c) {
      m = frexpf(m * D[(static_cast<long long>(child_slots[c]) * B + b) * H + z], &k);
      e += k;
    }
    mant[z] = m;
    expo[z] = e;
    if (m > 0.f) best = max(best, static_cast<long long>(e) * 4294967296LL + __float_as_uint(m));
  }
  for (int o = 16; o; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x < 32) {
    long long m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : kNone;
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) red[0] = m;
  }
  __syncthreads();
  best = red[0];
  const bool live = best != kNone;
  const unsigned mbits = static_cast<unsigned>(best & 0xffffffffLL);
  const int emax = live ? static_cast<int>((best - static_cast<long long>(mbits)) / 4294967296LL) : 0;
  const float mmax = live ? __uint_as_float(mbits) : 1.f;
  const long long row = static_cast<long long>(s) * B + b;
  double dot = 0.0;
  for (int z = threadIdx.x; z < H; z += blockDim.x) {
    const float m = mant[z];
    const float u = (live && m > 0.f) ? ldexpf(m / mmax, expo[z] - emax) : 0.f;
    U32[row * H + z] = u;
    if (uop) store_operand<P>(uop, static_cast<size_t>(row * uop_ld + z), uop_lo, u);
    if (s == root_slot) dot += static_cast<double>(pi[z]) * u;
  }
  if (threadIdx.x == 0) {
    double off = live ? static_cast<double>(emax) * 0.69314718055994530942 + log(static_cast<double>(mmax))
                      : -static_cast<double>(INFINITY);
    for (int c = c0; c < c1; ++c) off += O[static_cast<long long>(child_slots[c]) * B + b];
    O[row] = off;
  }
  if (s != root_slot) return;
  for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  if ((threadIdx.x & 31) == 0) redd[threadIdx.x >> 5] = dot;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += redd[w];
    const double off = O[row];
    const bool zero = !(t > 0.0) || !(off > -static_cast<double>(INFINITY));
    ll[b] = zero ? -static_cast<double>(INFINITY) : off + log(t);
    rroot[b] = zero ? 0.f : static_cast<float>(1.0 / t);
  }
}

// Root flows f_0[b][z] = pi[z] u_0[b][z] / sum_z pi u_0 (batch-major) and dpi += sum_b f_0.
__global__ void k_hclt_root_flows(int root_slot, int H, int B, const float* __restrict__ pi,
                                  const float* __restrict__ U32, const float* __restrict__ rroot,
                                  float* __restrict__ F32, float* dpi) {
  const int z = blockIdx.x * blockDim.x + threadIdx.x;
  if (z >= H) return;
  const float pz = pi[z];
  float acc = 0.f;
  const int b0 = blockIdx.y * 32;
  for (int b = b0; b < b0 + 32 && b < B; ++b) {
    const long long idx = (static_cast<long long>(root_slot) * B + b) * H + z;
    const float f = pz * U32[idx] * rroot[b];
    F32[idx] = f;
    acc += f;
  }
  if (dpi) atomicAdd(&dpi[z], acc);
}

// The layer's scaled flows of the edges in slots [s0, s0 + G): g[b][z] = f_parent[b][z] /
// D[b][z] (0 where D = 0), written batch-major (element contraction operand) and
// node-major (parameter contraction operand) through a 32 x 32 shared-memory tile.
template <int P>
__global__ void k_hclt_scaled_flows(int s0, int H, int B, const int* __restrict__ parent_slot,
                                    const float* __restrict__ F32, const float* __restrict__ D, void* gbm,
                                    long long gbm_ld, size_t gbm_lo, void* gnm, long long gnm_ld, size_t gnm_lo) {
  __shared__ float tile[32][33];
  const int g = blockIdx.z;
  const int s = s0 + g;
  const int ps = parent_slot[s];
  const int z0 = blockIdx.x * 32, b0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int b = b0 + i, z = z0 + threadIdx.x;
    float w = 0.f;
    if (b < B && z < H) {
      const float d = D[(static_cast<long long>(s) * B + b) * H + z];
      w = d > 0.f ? F32[(static_cast<long long>(ps) * B + b) * H + z] / d : 0.f;
      store_operand<P>(gbm, static_cast<size_t>((static_cast<long long>(g) * B + b) * gbm_ld + z), gbm_lo, w);
    }
    tile[i][threadIdx.x] = w;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int z = z0 + i, b = b0 + threadIdx.x;
    if (b < B && z < H)
      store_operand<P>(gnm, static_cast<size_t>((static_cast<long long>(g) * H + z) * gnm_ld + b), gnm_lo,
                       tile[threadIdx.x][i]);
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

// dEt[v][k][z] = sum over the samples of node s with category k of f[s][b][z].
__global__ void k_hclt_dE_gather(int H, int B, int C, const int* __restrict__ var_of_slot,
                                 const int* __restrict__ order, const int* __restrict__ off,
                                 const float* __restrict__ F32, float* __restrict__ dEt) {
  const int s = blockIdx.x, k = blockIdx.y;
  const int v = var_of_slot[s];
  const long long ob = static_cast<long long>(s) * (C + 1);
  const int e0 = off[ob + k], e1 = off[ob + k + 1];
  float* dst = dEt + (static_cast<long long>(v) * C + k) * H;
  for (int z = threadIdx.x; z < H; z += blockDim.x) {
    float acc = 0.f;
    for (int e = e0; e < e1; ++e)
      acc += F32[(static_cast<long long>(s) * B + order[static_cast<long long>(s) * B + e]) * H + z];
    dst[z] = acc;
  }
}

// dst[g][c][r] (+)= src[g][r][c] for G matrices of R x C.
__global__ void k_transpose_add_groups(const float* __restrict__ src, int R, int C, float* __restrict__ dst,
                                       int accumulate) {
  __shared__ float tile[32][33];
  const long long g = blockIdx.z;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const float* sg = src + g * R * C;
  float* dg = dst + g * R * C;
  for (int k = threadIdx.y; k < 32; k += 8) {
    const int r = r0 + k, c = c0 + threadIdx.x;
    tile[k][threadIdx.x] = (r < R && c < C) ? sg[static_cast<long long>(r) * C + c] : 0.f;
  }
  __syncthreads();
  for (int k = threadIdx.y; k < 32; k += 8) {
    const int c = c0 + k, r = r0 + threadIdx.x;
    if (r < R && c < C) {
      float* d = dg + static_cast<long long>(c) * R + r;
      *d = accumulate ? *d + tile[threadIdx.x][k] : tile[threadIdx.x][k];
    }
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

// Forward epilogue: D[g][b][z], the edge's sum layer kept linear; thread = parent latent z.
struct EpiHcltFwd : EpiNoHooks {
  // Every edge's D feeds the log-likelihood, and a tree chains hundreds of them: the bf16
  // mode accumulates K in slices of 16 k-steps so that the accumulator's truncation acts
  // on partial sums a fraction of D's size.
  static constexpr int kSliceBF16 = 16;
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
// The u block is staged in shared memory during the K loop (not in 3xTF32, whose ring
// needs the room).
template <int P>
struct EpiHcltElem : EpiNoHooks {
  struct Params {
    const float* U32;  // at the level's first slot, [G][B][H]
    float* F32;        // idem
    int H, B;
  };
  static constexpr bool kStage = P != kTF32x3;
  static constexpr int kSmemBytes = kStage ? kHcltBN * kBM * 4 : 0;

  __device__ static void prepare(const Params& p, int g, int m0, int n0, int et, uint8_t* smem) {
    if constexpr (kStage)
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
      if constexpr (kStage)
        u[c] = reinterpret_cast<const float*>(smem)[(col0 + c) * kBM + row];
      else
        u[c] = n0 + col0 + c < p.B ? p.U32[base + static_cast<long long>(c) * p.H] : 0.f;
    }
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if (n0 + col0 + c < p.B) p.F32[base + static_cast<long long>(c) * p.H] = u[c] * v[c];
  }
};

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
  float *Et, *U32, *D, *rroot, *F32, *dEt;
  double* O;
  int *cat_order, *cat_off;
};

size_t carve_hclt(void* base, pc_precision_t p, int n, int H, int C, int B, bool flows, bool want_dE, HcltWs* w) {
  Carver c(base);
  *w = HcltWs{};
  const long long E1 = n > 1 ? n - 1 : 1;
  w->plan = static_cast<int*>(c.take(size_t(4 * n + 2) * 4));
  w->Wop = c.operand(p, E1, H, H);
  w->Et = static_cast<float*>(c.take(size_t(n) * C * H * 4));
  w->U32 = static_cast<float*>(c.take(size_t(n) * B * H * 4));
  w->Uop = c.operand(p, E1, B, H);
  w->D = static_cast<float*>(c.take(size_t(E1) * B * H * 4));
  w->O = static_cast<double*>(c.take(size_t(n) * B * 8));
  w->rroot = static_cast<float*>(c.take(size_t(B) * 4));
  if (flows) {
    w->WopT = c.operand(p, E1, H, H);
    w->F32 = static_cast<float*>(c.take(size_t(n) * B * H * 4));
    w->Gbm = c.operand(p, E1, B, H);
    w->Gnm = c.operand(p, E1, H, B);
    w->Unm = c.operand(p, E1, H, B);
    if (want_dE) {
      w->dEt = static_cast<float*>(c.take(size_t(n) * C * H * 4));
      w->cat_order = static_cast<int*>(c.take(size_t(n) * B * 4));
      w->cat_off = static_cast<int*>(c.take(size_t(n) * (C + 1) * 4));
    }
  }
  return c.used;
}

size_t hclt_ws_bytes(pc_precision_t p, int n, int H, int C, int B) {
  HcltWs w;
  return carve_hclt(nullptr, p, n, H, C, B, true, true, &w) + 256;
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

template <int P>
pc_status_t hclt_run(int n, int H, int C, int B, const int32_t* parent, const int32_t* data, const float* pi,
                     const float* W, const float* Em, double* ll, float* dpi, float* dW, float* dE, int accumulate,
                     pc_precision_t prec, void* ws, cudaStream_t s) {
  constexpr int kParamBN = (P == kBF16) ? 256 : 128;
  HcltPlan pl;
  pc_status_t st;
  if ((st = make_plan(n, parent, &pl)) != PC_OK) return st;
  const bool flows = dpi || dW || dE;
  const bool down = flows && (dW || dE) && n >= 2;  // flows below the root are needed
  HcltWs w;
  void* base = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
  carve_hclt(base, prec, n, H, C, B, flows, dE != nullptr, &w);
  const int E = n - 1;
  const int root = n - 1;
  const int* d_var = w.plan + pl.off_var;
  const int* d_cptr = w.plan + pl.off_cptr;
  const int* d_cslots = w.plan + pl.off_cslots;
  const int* d_pslot = w.plan + pl.off_pslot;

  // the tree plan is a few KB of host data
  PC_CUDA(cudaMemcpyAsync(w.plan, pl.blob.data(), pl.blob.size() * sizeof(int), cudaMemcpyHostToDevice, s));
  if (dpi && !accumulate) PC_CUDA(cudaMemsetAsync(dpi, 0, size_t(H) * 4, s));
  if (dW && !accumulate) PC_CUDA(cudaMemsetAsync(dW, 0, size_t(H) * H * 4, s));  // W[0] has no edge

  k_hclt_et<<<dim3(cdiv(C, 32), cdiv(H, 32), n), dim3(32, 8), 0, s>>>(Em, H, C, w.Et);
  PC_LAUNCH_CHECK();
  if (E > 0 && (st = rows_to_operand<P>(W, H, static_cast<long long>(H) * H, E, H, H, w.Wop, s, d_var)) != PC_OK)
    return st;

  // -------------------------------------------------------------- forward
  const size_t prod_smem = size_t(H) * 8;  // mantissas and exponents, up to 64 KB
  if (prod_smem > 48 * 1024)
    PC_CUDA(cudaFuncSetAttribute(k_hclt_product<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(prod_smem)));
  OperandMaps ma, mb;
  for (int L = 0; L <= pl.maxh; ++L) {
    const int sA = pl.level_start[L], sB = pl.level_start[L + 1];
    const int G = sB - sA;
    if (G <= 0) continue;
    const bool edges = L < pl.maxh;
    k_hclt_product<P><<<dim3(G, B), 256, prod_smem, s>>>(
        sA, root, n, H, B, data, d_var, d_cptr, d_cslots, w.Et, w.D, C, w.U32, edges ? w.Uop.ptr : nullptr,
        w.Uop.ld, w.Uop.lo_elems, w.O, pi, ll, w.rroot);
    PC_LAUNCH_CHECK();
    if (!edges) continue;
    if ((st = encode_maps(&ma, operand_view(w.Wop, prec, sA, G), prec, kBM)) != PC_OK) return st;
    if ((st = encode_maps(&mb, operand_view(w.Uop, prec, sA, G), prec, kHcltBN)) != PC_OK) return st;
    EpiHcltFwd::Params ep{w.D + static_cast<long long>(sA) * B * H, H, B};
    if ((st = launch_gemm<P, kHcltBN, EpiHcltFwd>(dim3(cdiv(H, kBM), cdiv(B, kHcltBN), G), ma.hi, ma.lo, mb.hi,
                                                  mb.lo, num_k_blocks(H, prec), ep, s, PC_KIND_HCLT_FWD,
                                                  2ll * G * H * H * B)) != PC_OK)
      return st;
  }
  if (!flows) return PC_OK;

  // ------------------------------------------------------------- backward
  k_hclt_root_flows<<<dim3(cdiv(H, 256), cdiv(B, 32)), 256, 0, s>>>(root, H, B, pi, w.U32, w.rroot, w.F32, dpi);
  PC_LAUNCH_CHECK();
  if (down) {
    if ((st = transpose_to_operand<P>(W, H, static_cast<long long>(H) * H, E, H, H, w.WopT, s, d_var)) != PC_OK)
      return st;
    for (int L = pl.maxh - 1; L >= 0; --L) {
      const int sA = pl.level_start[L], sB = pl.level_start[L + 1];
      const int G = sB - sA;
      if (G <= 0) continue;
      k_hclt_scaled_flows<P><<<dim3(cdiv(H, 32), cdiv(B, 32), G), dim3(32, 8), 0, s>>>(
          sA, H, B, d_pslot, w.F32, w.D, w.Gbm.ptr, w.Gbm.ld, w.Gbm.lo_elems, w.Gnm.ptr, w.Gnm.ld,
          w.Gnm.lo_elems);
      PC_LAUNCH_CHECK();
      // element flows of the level's children
      if ((st = encode_maps(&ma, operand_view(w.WopT, prec, sA, G), prec, kBM)) != PC_OK) return st;
      if ((st = encode_maps(&mb, operand_view(w.Gbm, prec, 0, G), prec, kHcltBN)) != PC_OK) return st;
      typename EpiHcltElem<P>::Params ee{w.U32 + static_cast<long long>(sA) * B * H,
                                         w.F32 + static_cast<long long>(sA) * B * H, H, B};
      if ((st = launch_gemm<P, kHcltBN, EpiHcltElem<P>>(dim3(cdiv(H, kBM), cdiv(B, kHcltBN), G), ma.hi, ma.lo,
                                                        mb.hi, mb.lo, num_k_blocks(H, prec), ee, s,
                                                        PC_KIND_HCLT_ELEM, 2ll * G * H * H * B)) != PC_OK)
        return st;
      if (!dW) continue;
      // parameter flows of the level's edges
      if ((st = transpose_to_operand<P>(w.U32 + static_cast<long long>(sA) * B * H, H,
                                        static_cast<long long>(B) * H, G, B, H, w.Unm, s)) != PC_OK)
        return st;
      if ((st = encode_maps(&ma, operand_view(w.Gnm, prec, 0, G), prec, kBM)) != PC_OK) return st;
      if ((st = encode_maps(&mb, operand_view(w.Unm, prec, 0, G), prec, kParamBN)) != PC_OK) return st;
      EpiThetaScale::Params ep{dW, W, H, H, accumulate, d_var + sA};
      if ((st = launch_gemm<P, kParamBN, EpiThetaScale>(dim3(cdiv(H, kBM), cdiv(H, kParamBN), G), ma.hi, ma.lo,
                                                        mb.hi, mb.lo, num_k_blocks(B, prec), ep, s,
                                                        PC_KIND_HCLT_PARAM, 2ll * G * H * H * B)) != PC_OK)
        return st;
    }
  }
  if (dE) {
    k_hclt_cat_bucket<<<n, 32, size_t(C + 1) * 4, s>>>(n, B, C, data, d_var, w.cat_order, w.cat_off);
    PC_LAUNCH_CHECK();
    k_hclt_dE_gather<<<dim3(n, C), 256, 0, s>>>(H, B, C, d_var, w.cat_order, w.cat_off, w.F32, w.dEt);
    PC_LAUNCH_CHECK();
    k_transpose_add_groups<<<dim3(cdiv(H, 32), cdiv(C, 32), n), dim3(32, 8), 0, s>>>(w.dEt, C, H, dE, accumulate);
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

}  // extern "C"
