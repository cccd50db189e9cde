// fwd_f32.cu -- exact attention forward in fp32 on the CUDA cores.
//
// Serves fa_forward_fp32, where every product and sum stays in fp32: the
// tensor cores' reduced-precision (TF32) path could not hold the fp32 error
// bound, so this kernel uses FFMA only, with the accurate expf/logf.
//
// Algorithm: the FlashAttention-2 ordering described in "FlashAttention: GPU
// 메모리 계층을 활용한 어텐션 최적화 분석" (youngju.dev), sections 8.1-8.3:
// query rows are the outer, parallel dimension (one CTA per 32 query rows of
// one head, each warp owning whole rows, so warps never exchange partial
// results), key/value tiles are the inner loop, and the output stays
// unnormalised until the end.  Each tile updates the running max and running
// sum with eqs. (2)-(3) of "Flash Attention" (suniverse77.github.io, section
// "Online Softmax") and rescales the output accumulator as in eq. (4).
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>

#include "kernels.h"

namespace fattn {
namespace {

constexpr int kRowsPerCta = 32;
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = kRowsPerCta / kWarps;  // 4
constexpr int kKeysPerTile = 64;

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
    fwd_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                   const float *__restrict__ v, float *__restrict__ o, float *__restrict__ lse,
                   int N, float scale, int causal) {
  constexpr int kC = D / 32;  // output columns per lane
  extern __shared__ float smem[];
  float *sQ = smem;                               // [32][D]
  float *sK = sQ + kRowsPerCta * D;               // [64][D+1] (padded: no bank conflicts)
  float *sV = sK + kKeysPerTile * (D + 1);        // [64][D]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t head = blockIdx.x;
  const int row0 = blockIdx.y * kRowsPerCta;
  const float *qh = q + head * N * D, *kh = k + head * N * D, *vh = v + head * N * D;

  for (int idx = threadIdx.x; idx < kRowsPerCta * D; idx += blockDim.x) {
    const int r = idx / D;
    sQ[idx] = (row0 + r < N) ? qh[(int64_t)(row0 + r) * D + idx % D] : 0.f;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kC];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < kC; ++c) acc[r][c] = 0.f;
  }

  const int last_row = min(N, row0 + kRowsPerCta) - 1;
  const int n_keys = causal ? last_row + 1 : N;
  for (int j0 = 0; j0 < n_keys; j0 += kKeysPerTile) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kKeysPerTile * D; idx += blockDim.x) {
      const int j = idx / D, c = idx % D;
      const bool in = j0 + j < N;
      sK[j * (D + 1) + c] = in ? kh[(int64_t)(j0 + j) * D + c] : 0.f;
      sV[idx] = in ? vh[(int64_t)(j0 + j) * D + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int lr = warp * kRowsPerWarp + r;
      const int i = row0 + lr;
      if (i >= N) continue;
      const int limit = causal ? i + 1 : N;  // keys j < limit are visible
      // Scores of keys j0+lane and j0+lane+32.
      float s[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = lane + 32 * h;
        float dot = 0.f;
#pragma unroll 16
        for (int c = 0; c < D; ++c) dot = fmaf(sQ[lr * D + c], sK[j * (D + 1) + c], dot);
        s[h] = (j0 + j < limit) ? dot * scale : -INFINITY;
      }
      float tmax = fmaxf(s[0], s[1]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(~0u, tmax, off));
      if (tmax == -INFINITY) continue;  // no visible key in this tile
      const float m_new = fmaxf(m[r], tmax);                    // eq. (2)
      const float alpha = expf(m[r] - m_new);                   // 0 when m = -inf
      const float p0 = expf(s[0] - m_new), p1 = expf(s[1] - m_new);
      float psum = p0 + p1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(~0u, psum, off);
      l[r] = l[r] * alpha + psum;                               // eq. (3)
      m[r] = m_new;
#pragma unroll
      for (int c = 0; c < kC; ++c) acc[r][c] *= alpha;          // eq. (4), unnormalised
      for (int j = 0; j < kKeysPerTile; ++j) {
        const float pj = __shfl_sync(~0u, j < 32 ? p0 : p1, j & 31);
#pragma unroll
        for (int c = 0; c < kC; ++c) acc[r][c] = fmaf(pj, sV[j * D + lane + 32 * c], acc[r][c]);
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = row0 + warp * kRowsPerWarp + r;
    if (i >= N) continue;
    const float inv = 1.f / l[r];
#pragma unroll
    for (int c = 0; c < kC; ++c) o[(head * N + i) * D + lane + 32 * c] = acc[r][c] * inv;
    if (lse && lane == 0) lse[head * N + i] = m[r] + logf(l[r]);
  }
}

template <int D>
cudaError_t launch_fwd_f32_d(const float *q, const float *k, const float *v, float *o, float *lse,
                             int BH, int N, float scale, int causal, cudaStream_t stream) {
  const size_t smem = sizeof(float) * (kRowsPerCta * D + kKeysPerTile * (D + 1) + kKeysPerTile * D);
  cudaError_t e = cudaFuncSetAttribute(fwd_f32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(BH, (N + kRowsPerCta - 1) / kRowsPerCta);
  fwd_f32_kernel<D><<<grid, kWarps * 32, smem, stream>>>(q, k, v, o, lse, N, scale, causal);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
                           int BH, int N, int d, float scale, int causal, cudaStream_t stream) {
  if (d == 64) return launch_fwd_f32_d<64>(q, k, v, o, lse, BH, N, scale, causal, stream);
  return launch_fwd_f32_d<128>(q, k, v, o, lse, BH, N, scale, causal, stream);
}

}  // namespace fattn
