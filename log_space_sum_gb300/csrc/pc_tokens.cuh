// Token buckets of an HMM's (position, sample) pairs and the per-token gather-sum of the
// emission flows: dE is then deterministic (every output summed by one thread in a fixed
// order). Shared by the HMM circuits.
#pragma once

#include "pc_device.cuh"

namespace pc {
namespace {

// count[v] = number of (position, sample) pairs with token v (tokens outside [0, V)
// are ignored).
__global__ void k_token_hist(const int* __restrict__ tokens, int n, int V, int* __restrict__ count) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const int v = tokens[i];
    if (v >= 0 && v < V) atomicAdd(&count[v], 1);
  }
}

// offset[v] = sum_{u < v} count[u] for v = 0..V, one block of 1024 threads.
__global__ void k_exclusive_scan(const int* __restrict__ count, int V, int* __restrict__ offset) {
  __shared__ int part[1024];
  const int per = (V + 1023) / 1024;
  const int lo = threadIdx.x * per;
  int local = 0;
  for (int i = lo; i < lo + per && i < V; ++i) local += count[i];
  part[threadIdx.x] = local;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {
    const int add = threadIdx.x >= d ? part[threadIdx.x - d] : 0;
    __syncthreads();
    part[threadIdx.x] += add;
    __syncthreads();
  }
  int run = part[threadIdx.x] - local;  // exclusive prefix of this thread's range
  for (int i = lo; i < lo + per && i < V; ++i) {
    offset[i] = run;
    run += count[i];
  }
  if (threadIdx.x == 1023) offset[V] = part[1023];
}

// order[offset[v] ..] = the batch-major flow rows t*B + b of every pair with token v,
// in increasing token-array index b*T + t: a stable, deterministic bucketing. Each
// block owns kBucketSpan consecutive token values and scans the whole token array once.
constexpr int kBucketSpan = 16;
__global__ void k_token_bucket(const int* __restrict__ tokens, int T, int B, int V,
                               const int* __restrict__ offset, int* __restrict__ order) {
  __shared__ int warp_n[kBucketSpan][8];
  __shared__ int base[kBucketSpan];
  const int v0 = blockIdx.x * kBucketSpan;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < kBucketSpan) base[threadIdx.x] = v0 + threadIdx.x < V ? offset[v0 + threadIdx.x] : 0;
  __syncthreads();
  const int n = T * B;
  for (int i0 = 0; i0 < n; i0 += 256) {
    const int i = i0 + threadIdx.x;
    const int tok = i < n ? tokens[i] : -1;
    const int slot = tok - v0;                       // in [0, kBucketSpan) when this block owns it
    const bool mine = slot >= 0 && slot < kBucketSpan;
    unsigned my_bal = 0;
#pragma unroll
    for (int j = 0; j < kBucketSpan; ++j) {
      const unsigned bal = __ballot_sync(0xffffffffu, mine && slot == j);
      if (lane == 0) warp_n[j][warp] = __popc(bal);
      if (mine && slot == j) my_bal = bal;
    }
    __syncthreads();
    if (mine) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += warp_n[slot][w];
      const int b = i / T, t = i - b * T;
      order[base[slot] + before + __popc(my_bal & ((1u << lane) - 1u))] = t * B + b;
    }
    __syncthreads();
    if (threadIdx.x < kBucketSpan) {
      int total = 0;
      for (int w = 0; w < 8; ++w) total += warp_n[threadIdx.x][w];
      base[threadIdx.x] += total;
    }
    __syncthreads();
  }
}

// dEt[v][k] = sum over the pairs of bucket v (in bucket order) of the flows f[row][k].
__global__ void k_dE_gather(const float* __restrict__ fbm, int H, const int* __restrict__ offset,
                            const int* __restrict__ order, float* __restrict__ dEt) {
  const int v = blockIdx.x;
  const int k = blockIdx.y * blockDim.x + threadIdx.x;
  if (k >= H) return;
  float acc = 0.f;
  const int e1 = offset[v + 1];
  for (int e = offset[v]; e < e1; ++e) acc += fbm[static_cast<long long>(order[e]) * H + k];
  dEt[static_cast<long long>(v) * H + k] = acc;
}

}  // namespace
}  // namespace pc
