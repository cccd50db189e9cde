// fp8_quant.cu -- block quantization of bf16 Q, K, V to E4M3 for the FP8
// forward, with the optional random orthogonal transform of Q and K
// ("FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화 분석", youngju.dev,
// section 9.2, item 3: block quantization and incoherent processing).
//
// What is computed, per head (d = 128):
//   Q, K: for every block of 128 rows, s = amax / 448 (fp32 division; 1 for
//         an all-zero block), codes E4M3_rn,sat(x * (1 / s)) with the
//         reciprocal and the product in fp32, and the dequantization scale s
//         (times fp32(1/sqrt(d)) when the transform is applied);
//   V:    one s for the whole head, codes written transposed, V^T [d][Npad]
//         with Npad = N rounded up to 16 and zero codes in the padding.
// The transform (signs given): each row x becomes (x * sigma) H, H the
// Sylvester-Hadamard matrix, evaluated as the fp32 butterfly with stages
// h = 1, 2, ..., 64, a pair (a, b) becoming (a + b, a - b).  One warp holds a
// row as four consecutive values per lane, so stages 1 and 2 stay inside a
// lane and stages 4 .. 64 pair lanes l and l ^ (h / 4).
//
// The work is HBM-bound: each kernel reads its 128 x 128 bf16 block once
// (V twice: once for the head's amax, once to code it) and writes 16 KB of
// codes.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx_f8.cuh"

namespace fattn {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;          // rows per quantization block
constexpr int kThreads = 256;       // 8 warps x 16 rows
constexpr int kRowsPerWarp = kRows / (kThreads / 32);

__device__ __forceinline__ float4 load_bf16x4(const uint16_t *p) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// One butterfly stage across lanes: the lane whose `mask` bit is clear keeps
// a + b, its partner a - b (a the lower-index value, b the higher).
__device__ __forceinline__ float bfly(float x, int mask, bool high) {
  const float y = __shfl_xor_sync(0xffffffffu, x, mask);
  return high ? __fsub_rn(y, x) : __fadd_rn(x, y);
}

__device__ __forceinline__ void hadamard_row(float4 &v, int lane) {
  // h = 1: (0,1), (2,3); h = 2: (0,2), (1,3) -- inside the lane.
  float a0 = __fadd_rn(v.x, v.y), a1 = __fsub_rn(v.x, v.y);
  float a2 = __fadd_rn(v.z, v.w), a3 = __fsub_rn(v.z, v.w);
  v = make_float4(__fadd_rn(a0, a2), __fadd_rn(a1, a3), __fsub_rn(a0, a2), __fsub_rn(a1, a3));
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool high = (lane & m) != 0;
    v.x = bfly(v.x, m, high);
    v.y = bfly(v.y, m, high);
    v.z = bfly(v.z, m, high);
    v.w = bfly(v.w, m, high);
  }
}

__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}

__device__ __forceinline__ float scale_of(float amax) {
  return amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
}

__device__ __forceinline__ uint32_t code4(float4 v, float inv) {
  return pack_e4m3x4(__fmul_rn(v.x, inv), __fmul_rn(v.y, inv), __fmul_rn(v.z, inv),
                     __fmul_rn(v.w, inv));
}

// grid (n_blk, BH, 3): z = 0 codes Q, z = 1 codes K, z = 2 records the
// block's |V| maximum in v_amax[bh * n_blk + blk].
template <bool ROT>
__global__ void __launch_bounds__(kThreads)
    fp8_quant_rows_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
                          const uint16_t *__restrict__ v, const float *__restrict__ signs,
                          uint8_t *__restrict__ q8, uint8_t *__restrict__ k8,
                          float *__restrict__ q_scale, float *__restrict__ k_scale,
                          float *__restrict__ v_amax, int N, int n_blk, float rot_factor) {
  __shared__ float red[kThreads / 32];
  const int blk = blockIdx.x, bh = blockIdx.y, which = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint16_t *src = which == 0 ? q : which == 1 ? k : v;
  const int64_t head = static_cast<int64_t>(bh) * N;
  const int r0 = blk * kRows + warp * kRowsPerWarp;
  float4 sg = make_float4(1.f, 1.f, 1.f, 1.f);
  if (ROT && which < 2) sg = *reinterpret_cast<const float4 *>(signs + 4 * lane);
  float4 x[kRowsPerWarp];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int r = r0 + i;
    x[i] = r < N ? load_bf16x4(src + (head + r) * kD + 4 * lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (ROT && which < 2) {
      x[i] = make_float4(x[i].x * sg.x, x[i].y * sg.y, x[i].z * sg.z, x[i].w * sg.w);
      hadamard_row(x[i], lane);
    }
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x[i].x), fabsf(x[i].y)),
                             fmaxf(fabsf(x[i].z), fabsf(x[i].w))));
  }
  amax = block_max(amax, red);
  if (which == 2) {
    if (threadIdx.x == 0) v_amax[static_cast<int64_t>(bh) * n_blk + blk] = amax;
    return;
  }
  const float s = scale_of(amax);
  const float inv = __fdiv_rn(1.f, s);
  uint8_t *dst = which == 0 ? q8 : k8;
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int r = r0 + i;
    if (r < N) *reinterpret_cast<uint32_t *>(dst + (head + r) * kD + 4 * lane) = code4(x[i], inv);
  }
  if (threadIdx.x == 0)
    (which == 0 ? q_scale : k_scale)[static_cast<int64_t>(bh) * n_blk + blk] =
        ROT ? __fmul_rn(s, rot_factor) : s;
}

// grid (n_blk, BH): codes one 128-row block of V with its head's scale and
// writes it transposed into V^T [BH][128][Npad].
__global__ void __launch_bounds__(kThreads)
    fp8_quant_v_kernel(const uint16_t *__restrict__ v, const float *__restrict__ v_amax,
                       uint8_t *__restrict__ vt8, float *__restrict__ v_scale, int N, int n_blk,
                       int n_pad) {
  constexpr int kPitch = kRows + 1;   // bytes per transposed row in shared memory
  __shared__ uint8_t tile[kD * kPitch];
  __shared__ float red[kThreads / 32];
  const int blk = blockIdx.x, bh = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float amax = 0.f;
  for (int i = threadIdx.x; i < n_blk; i += kThreads)
    amax = fmaxf(amax, v_amax[static_cast<int64_t>(bh) * n_blk + i]);
  amax = block_max(amax, red);
  const float s = scale_of(amax);
  const float inv = __fdiv_rn(1.f, s);
  const int64_t head = static_cast<int64_t>(bh) * N;
#pragma unroll 4
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int rl = warp * kRowsPerWarp + i;        // key within the block
    const int r = blk * kRows + rl;
    const float4 x =
        r < N ? load_bf16x4(v + (head + r) * kD + 4 * lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t c = code4(x, inv);
#pragma unroll
    for (int e = 0; e < 4; ++e) tile[(4 * lane + e) * kPitch + rl] = (c >> (8 * e)) & 0xffu;
  }
  __syncthreads();
  // Row c of V^T: keys blk*128 .. +127, as 32 words; words past Npad are
  // not written (Npad is a multiple of 16, so a word never straddles it).
  uint8_t *out = vt8 + static_cast<int64_t>(bh) * kD * n_pad;
  for (int w = threadIdx.x; w < kD * 32; w += kThreads) {
    const int c = w >> 5, kw = w & 31;
    const int key = blk * kRows + 4 * kw;
    if (key >= n_pad) continue;
    const uint8_t *t = tile + c * kPitch + 4 * kw;
    const uint32_t word = static_cast<uint32_t>(t[0]) | (static_cast<uint32_t>(t[1]) << 8) |
                          (static_cast<uint32_t>(t[2]) << 16) |
                          (static_cast<uint32_t>(t[3]) << 24);
    *reinterpret_cast<uint32_t *>(out + static_cast<int64_t>(c) * n_pad + key) = word;
  }
  if (blk == 0 && threadIdx.x == 0) v_scale[bh] = s;
}

}  // namespace

size_t fp8_quant_workspace_bytes(int BH, int N) {
  return sizeof(float) * static_cast<size_t>(BH) * static_cast<size_t>((N + kRows - 1) / kRows);
}

cudaError_t launch_fp8_quantize(const void *q, const void *k, const void *v, const float *signs,
                                void *q8, void *k8, void *vt8, float *q_scale, float *k_scale,
                                float *v_scale, float *v_amax, int BH, int N, int n_pad,
                                float rot_factor, cudaStream_t stream) {
  const int n_blk = (N + kRows - 1) / kRows;
  const dim3 g1(n_blk, BH, 3);
  const auto *qq = static_cast<const uint16_t *>(q);
  const auto *kk = static_cast<const uint16_t *>(k);
  const auto *vv = static_cast<const uint16_t *>(v);
  if (signs != nullptr)
    fp8_quant_rows_kernel<true><<<g1, kThreads, 0, stream>>>(
        qq, kk, vv, signs, static_cast<uint8_t *>(q8), static_cast<uint8_t *>(k8), q_scale,
        k_scale, v_amax, N, n_blk, rot_factor);
  else
    fp8_quant_rows_kernel<false><<<g1, kThreads, 0, stream>>>(
        qq, kk, vv, nullptr, static_cast<uint8_t *>(q8), static_cast<uint8_t *>(k8), q_scale,
        k_scale, v_amax, N, n_blk, rot_factor);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fp8_quant_v_kernel<<<dim3(n_blk, BH), kThreads, 0, stream>>>(
      vv, v_amax, static_cast<uint8_t *>(vt8), v_scale, N, n_blk, n_pad);
  return cudaGetLastError();
}

}  // namespace fattn
