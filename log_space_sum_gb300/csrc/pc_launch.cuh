// Launch helpers: the tensor-core contraction and the small elementwise kernels that
// build its operands.
#pragma once

#include "pc_gemm.cuh"
#include "pc_host.h"

namespace pc {

template <int P, int BN, class Epi>
pc_status_t launch_gemm(dim3 grid, const CUtensorMap& a, const CUtensorMap& a_lo,
                        const CUtensorMap& b, const CUtensorMap& b_lo, int num_kb,
                        const typename Epi::Params& ep, cudaStream_t stream, int kind,
                        long long flops) {
  constexpr size_t smem = gemm_smem_bytes<P, BN, Epi>();
  static_assert(smem <= 232448, "shared memory per CTA");
  static bool attr_set[64] = {};
  int dev = 0;
  PC_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return set_error(PC_ERR_CUDA, "device index %d out of range", dev);
  if (!attr_set[dev]) {
    PC_CUDA(cudaFuncSetAttribute(k_umma_gemm<P, BN, Epi>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
    attr_set[dev] = true;
  }
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return PC_OK;
  const int slot = profile_begin(stream);
  k_umma_gemm<P, BN, Epi><<<grid, kGemmThreads, smem, stream>>>(a, a_lo, b, b_lo, num_kb,
                                                                device_status_word(), ep);
  PC_LAUNCH_CHECK();
  profile_end(slot, stream, kind, flops);
  return PC_OK;
}

// Tensor maps of an operand's hi and (3xTF32) lo parts.
struct OperandMaps {
  CUtensorMap hi, lo;
};

inline pc_status_t encode_maps(OperandMaps* m, const Operand& op, pc_precision_t p, int box_rows) {
  pc_status_t st = encode_operand_map(&m->hi, op, p, box_rows, 0);
  if (st != PC_OK) return st;
  if (p == PC_PREC_FP32) return encode_operand_map(&m->lo, op, p, box_rows, 1);
  m->lo = m->hi;
  return PC_OK;
}

inline int num_k_blocks(long long K, pc_precision_t p) {
  const int bk = 128 / operand_elem_bytes(p);
  return static_cast<int>((K + bk - 1) / bk);
}

inline unsigned cdiv(long long a, long long b) { return static_cast<unsigned>((a + b - 1) / b); }

// ---------------------------------------------------------------------------------
// Operand builders.

// dst[g][r][c] = op(src[g][r][c]); src row stride src_ld, group stride src_gs.
template <int P>
__global__ void k_rows_to_operand(const float* __restrict__ src, long long src_ld,
                                  long long src_gs, int G, int R, int C, void* dst,
                                  long long dst_ld, size_t lo, const int* gmap) {
  const long long total = static_cast<long long>(G) * R * C;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long c = idx % C;
    const long long gr = idx / C;
    const long long r = gr % R;
    const long long g = gr / R;
    const float v = src[(gmap ? gmap[g] : g) * src_gs + r * src_ld + c];
    store_operand<P>(dst, static_cast<size_t>((g * R + r) * dst_ld + c), lo, v);
  }
}

// dst[g][c][r] = op(src[g][r][c]) through 32x32 shared-memory tiles.
template <int P>
__global__ void k_transpose_to_operand(const float* __restrict__ src, long long src_ld,
                                       long long src_gs, int R, int C, void* dst,
                                       long long dst_ld, size_t lo, const int* gmap) {
  __shared__ float tile[32][33];
  const int g = blockIdx.z;
  const long long gs = gmap ? gmap[g] : g;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int k = ty; k < 32; k += 8) {
    const int r = r0 + k, c = c0 + tx;
    tile[k][tx] = (r < R && c < C) ? src[gs * src_gs + static_cast<long long>(r) * src_ld + c] : 0.f;
  }
  __syncthreads();
  for (int k = ty; k < 32; k += 8) {
    const int c = c0 + k, r = r0 + tx;
    if (r < R && c < C)
      store_operand<P>(dst, static_cast<size_t>((static_cast<long long>(g) * C + c) * dst_ld + r),
                       lo, tile[tx][k]);
  }
}

// Four consecutive columns per thread, blockIdx.x = matrix row (16-byte loads).
template <int P>
__global__ void k_rows_to_operand4(const float* __restrict__ src, long long src_ld, long long src_gs, int R,
                                   int C, void* dst, long long dst_ld, size_t lo, const int* gmap) {
  const long long gr = blockIdx.x;
  const long long g = gr / R, r = gr % R;
  const int c = 4 * (blockIdx.y * blockDim.x + threadIdx.x);
  if (c >= C) return;
  const float4 v = *reinterpret_cast<const float4*>(src + (gmap ? gmap[g] : g) * src_gs + r * src_ld + c);
  const size_t idx = static_cast<size_t>(gr * dst_ld + c);
  if constexpr (P == kBF16) {
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(dst) + idx) =
        make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  } else {
    const float4 h = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(dst) + idx) = h;
    if constexpr (P == kTF32x3)
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(dst) + idx + lo) =
          make_float4(tf32_rna(v.x - h.x), tf32_rna(v.y - h.y), tf32_rna(v.z - h.z), tf32_rna(v.w - h.w));
  }
}

template <int P>
pc_status_t rows_to_operand(const float* src, long long src_ld, long long src_gs, int G, int R,
                            int C, const Operand& dst, cudaStream_t s, const int* gmap = nullptr) {
  const long long total = static_cast<long long>(G) * R * C;
  if (total == 0) return PC_OK;
  const bool vec = (C % 4 == 0) && (src_ld % 4 == 0) && (src_gs % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(src) & 15) == 0 && static_cast<long long>(G) * R < (1ll << 31) &&
                   (C / 4 + 255) / 256 < 65536;
  if (vec) {
    const dim3 grid(static_cast<unsigned>(static_cast<long long>(G) * R), cdiv(C / 4, 256));
    k_rows_to_operand4<P><<<grid, 256, 0, s>>>(src, src_ld, src_gs, R, C, dst.ptr, dst.ld, dst.lo_elems, gmap);
  } else {
    const unsigned blocks = static_cast<unsigned>((total + 255) / 256 < 152 * 16 ? (total + 255) / 256 : 152 * 16);
    k_rows_to_operand<P><<<blocks, 256, 0, s>>>(src, src_ld, src_gs, G, R, C, dst.ptr, dst.ld, dst.lo_elems, gmap);
  }
  PC_LAUNCH_CHECK();
  return PC_OK;
}

template <int P>
pc_status_t transpose_to_operand(const float* src, long long src_ld, long long src_gs, int G,
                                 int R, int C, const Operand& dst, cudaStream_t s, const int* gmap = nullptr) {
  if (G == 0 || R == 0 || C == 0) return PC_OK;
  dim3 grid(cdiv(C, 32), cdiv(R, 32), G);
  k_transpose_to_operand<P><<<grid, dim3(32, 8), 0, s>>>(src, src_ld, src_gs, R, C, dst.ptr, dst.ld,
                                                         dst.lo_elems, gmap);
  PC_LAUNCH_CHECK();
  return PC_OK;
}

// Shared with the circuits: F[g][i][j] (+)= theta[g][i][j] * D[i,j].
struct EpiThetaScale : EpiNoHooks {
  static constexpr bool kTranspose = true;
  struct Params {
    float* F;
    const float* theta;
    int M, N, accumulate;
    const int* gmap;  // group g reads theta / writes F at matrix gmap[g] (NULL: g)
  };
  // Transposed so that lane l owns column col0 + l of the warp's 32 rows: every theta
  // load and F store of the warp covers one contiguous row segment. All loads of the
  // chunk are issued before the first store.
  __device__ static void apply(const Params& p, int g, int m0, int n0, int row, int col0,
                               float (&v)[32], uint8_t*, float* tbuf) {
    float w[32];
    warp_transpose32(v, w, tbuf);
    const int lane = threadIdx.x & 31;
    const int i0 = m0 + row - lane;
    const int j = n0 + col0 + lane;
    if (j >= p.N) return;
    const long long ld = p.N;
    const long long gm = p.gmap ? p.gmap[g] : g;
    const float* tp = p.theta + (gm * p.M + i0) * ld + j;
    float* Fp = p.F + (gm * p.M + i0) * ld + j;
    // two halves of 16 rows keep the loads-before-stores batch within the register budget
#pragma unroll
    for (int h = 0; h < 32; h += 16) {
      float t[16], f[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const bool in = i0 + h + r < p.M;
        t[r] = in ? tp[(h + r) * ld] : 0.f;
        f[r] = (in && p.accumulate) ? Fp[(h + r) * ld] : 0.f;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (i0 + h + r < p.M) Fp[(h + r) * ld] = f[r] + t[r] * w[h + r];
    }
  }
};

}  // namespace pc
