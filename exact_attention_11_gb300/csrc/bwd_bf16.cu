// bwd_bf16.cu -- backward pass of exact attention, bf16 in/out, on the
// sm_103a tensor cores.
//
// What is computed: given dO, the gradients of O = softmax(scale * Q K^T
// [+ causal mask]) V with respect to Q, K and V.  Following the
// recomputation strategy of "FlashAttention: GPU 메모리 계층을 활용한 어텐션
// 최적화 분석" (youngju.dev, section 7), nothing of size N x N is stored by the
// forward: S and P are rebuilt tile by tile from Q, K and the saved
// log-sum-exp, P = exp(S - LSE).  With D_i = sum_j P_ij dP_ij = dO_i . O_i:
//     dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//     dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Kernels:
//   bwd_prep_kernel   D = rowsum(dO * O) and the LSE in log2 units, written
//                     negated per 128-query block as [-LSE2 x 128 | -D x 128]
//                     (rows past N padded with -LSE2 = -inf, -D = 0) so one
//                     bulk copy brings a block's vectors and the packed fp32
//                     FMA/ADD use them as they are; zeroes the fp32 dQ
//                     accumulator
//   main kernel       one CTA per (128-key block j, head); K_j and V_j stay
//                     in shared memory and dK_j, dV_j in TMEM while the CTA
//                     visits every query block i that sees block j (the KV-
//                     outer order of FlashAttention-2's backward), in 64-query
//                     sub-tiles that two groups of warps take in turns.  dQ is
//                     summed across CTAs into an fp32 accumulator [BH][N][d].
//                     Head dimension 128: bwd_bf16_d128.cu; 64: bwd_bf16_d64.cu.
//   bwd_dq_kernel     dQ = scale * accumulator, rounded to bf16
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int BQ = 128;   // queries per block of the [-LSE2 | -D] vectors
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kVecFloats = 2 * BQ;   // [LSE2 | D] of one query block

// One 16-thread group per padded row (bh, i), i < n_qb * 128:
//   i < N:  vec[-LSE2] = -LSE * log2(e), vec[-D] = -rowsum(dO * O), and the
//           row of the dQ accumulator is zeroed
//   i >= N: vec[-LSE2] = -inf, vec[-D] = 0 (padding: P = 0 there).
template <int D>
__global__ void __launch_bounds__(256)
    bwd_prep_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                    const float *__restrict__ lse, float *__restrict__ vec,
                    float *__restrict__ dq_acc, int N, int n_qb, int64_t padded_rows) {
  // The main kernel may be scheduled once every block of this one has begun.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t prow = static_cast<int64_t>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  const int part = threadIdx.x & 15;
  const bool live = prow < padded_rows;
  const int64_t npad = static_cast<int64_t>(n_qb) * BQ;
  const int64_t bh = live ? prow / npad : 0;
  const int i = live ? static_cast<int>(prow - bh * npad) : 0;
  const bool real = live && i < N;
  const int64_t row = bh * N + i;
  float acc = 0.f;
  if (real) {
    for (int c = part * 8; c < D; c += 128) {
      const uint4 a = *reinterpret_cast<const uint4 *>(o + row * D + c);
      const uint4 b = *reinterpret_cast<const uint4 *>(dout + row * D + c);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(aw[e] << 16), __uint_as_float(bw[e] << 16), acc);
        acc = fmaf(__uint_as_float(aw[e] & 0xffff0000u), __uint_as_float(bw[e] & 0xffff0000u), acc);
      }
    }
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = part * 4; c < D; c += 64) *reinterpret_cast<float4 *>(dq_acc + row * D + c) = z;
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(~0u, acc, off);
  if (live && part == 0) {
    float *v = vec + (bh * n_qb + i / BQ) * kVecFloats;
    v[i % BQ] = real ? -lse[row] * kLog2e : -INFINITY;
    v[BQ + i % BQ] = real ? -acc : 0.f;
  }
}

// dQ = scale * accumulator as bf16, eight elements per thread (row-major
// accumulator [BH][N][D]).
__global__ void __launch_bounds__(256)
    bwd_dq_kernel(const float *__restrict__ acc, __nv_bfloat16 *__restrict__ dq, int64_t n8,
                  float scale) {
  // A programmatic dependent of the main kernel: wait for its last additions.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4 *>(acc)[2 * i];
  const float4 b = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
  uint4 w;
  w.x = pack_bf16x2(a.x * scale, a.y * scale);
  w.y = pack_bf16x2(a.z * scale, a.w * scale);
  w.z = pack_bf16x2(b.x * scale, b.y * scale);
  w.w = pack_bf16x2(b.z * scale, b.w * scale);
  reinterpret_cast<uint4 *>(dq)[i] = w;
}

template <int D>
cudaError_t launch_bwd_d(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const CUtensorMap &tdo, const CUtensorMap &tdq, const void *o,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv, int BH,
                         int N, float scale, int causal, float *ws, int *sched, int fault_cta,
                         int *dev_status, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(BH) * N;
  const int n_qb = (N + BQ - 1) / BQ;
  const int64_t padded = static_cast<int64_t>(BH) * n_qb * BQ;
  // Workspace: fp32 dQ accumulator (row-major [BH][N][D] in the first
  // BH * N * D of BH * Npad * D floats), then [-LSE2 | -D] per query block.
  float *dq_acc = ws, *vecs = ws + padded * D;
  bwd_prep_kernel<D><<<static_cast<unsigned>((padded + 15) / 16), 256, 0, stream>>>(
      reinterpret_cast<const __nv_bfloat16 *>(o), reinterpret_cast<const __nv_bfloat16 *>(dout),
      lse, vecs, dq_acc, N, n_qb, padded);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // Q and dO maps have 64-row boxes (the main kernels' 64-query sub-tiles).
  if constexpr (D == 128)
    e = launch_bwd_main_d128(tq, tk, tv, tdo, tdq, vecs, dk, dv, BH, N, scale, causal, sched,
                             fault_cta, dev_status, stream);
  else
    e = launch_bwd_main_d64(tq, tk, tv, tdo, tdq, vecs, dk, dv, BH, N, scale, causal, sched,
                            fault_cta, dev_status, stream);
  if (e != cudaSuccess) return e;
  const int64_t n8 = rows * D / 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n8 + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bwd_dq_kernel, static_cast<const float *>(dq_acc),
                            reinterpret_cast<__nv_bfloat16 *>(dq), n8, scale);
}

}  // namespace

size_t bwd_workspace_bytes(int BH, int N, int d) {
  const size_t n_qb = (static_cast<size_t>(N) + BQ - 1) / BQ;
  return sizeof(float) * static_cast<size_t>(BH) * n_qb * BQ * (static_cast<size_t>(d) + 2);
}

cudaError_t launch_bwd_bf16(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &tdo, const CUtensorMap &tdq, const void *o,
                            const void *dout, const float *lse, void *dq, void *dk, void *dv,
                            int BH, int N, int d, float scale, int causal, float *ws,
                            int *sched, int fault_cta, int *dev_status, cudaStream_t stream) {
  if (d == 64)
    return launch_bwd_d<64>(tq, tk, tv, tdo, tdq, o, dout, lse, dq, dk, dv, BH, N, scale, causal,
                            ws, sched, fault_cta, dev_status, stream);
  return launch_bwd_d<128>(tq, tk, tv, tdo, tdq, o, dout, lse, dq, dk, dv, BH, N, scale, causal,
                           ws, sched, fault_cta, dev_status, stream);
}

}  // namespace fattn
