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
// codes.  A CTA stages its block in shared memory with one 32 KB bulk copy,
// so the bytes in flight per SM are bounded by shared memory (up to seven
// blocks) rather than by registers.
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
static_assert(kThreads == 256 && kD == 128 && kRows == 128,
              "the V^T store pattern covers 128 rows with 8 warps x 4 passes");

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

// Stages rows r0 .. r0 + n_rows - 1 of one head (contiguous, 256 bytes each)
// in shared memory with one bulk copy; false if the copy did not arrive
// within the wait limit (then *dev_status is set).
__device__ __forceinline__ bool stage_rows(const uint16_t *src, uint32_t dst, int n_rows,
                                           uint32_t bar, volatile int *abort_flag,
                                           int *dev_status) {
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n_rows) * kD * 2);
    bulk_load(dst, src, static_cast<uint32_t>(n_rows) * kD * 2, bar);
  }
  if (!mbar_wait(bar, 0, abort_flag)) {
    if (threadIdx.x == 0) atomicExch(dev_status, kDevTimeout);
    return false;
  }
  return true;
}

// Four values of staged row r (lane's columns 4 lane .. 4 lane + 3); rows past
// the block's end read as zero.
__device__ __forceinline__ float4 staged4(const uint8_t *stage, int r, int n_rows, int lane) {
  if (r >= n_rows) return make_float4(0.f, 0.f, 0.f, 0.f);
  const uint2 u = *reinterpret_cast<const uint2 *>(stage + r * (kD * 2) + lane * 8);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// grid (n_blk, BH, 3): z = 0 codes Q, z = 1 codes K, z = 2 records the
// block's |V| maximum in v_amax[bh * n_blk + blk].  The block is staged in
// shared memory by one bulk copy, then read twice (maximum, then codes), so
// without the transform the registers hold no block data and seven CTAs fit
// per SM.
template <bool ROT>
__global__ void __launch_bounds__(kThreads)
    fp8_quant_rows_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
                          const uint16_t *__restrict__ v, const float *__restrict__ signs,
                          uint8_t *__restrict__ q8, uint8_t *__restrict__ k8,
                          float *__restrict__ q_scale, float *__restrict__ k_scale,
                          float *__restrict__ v_amax, int N, int n_blk, float rot_factor,
                          int *__restrict__ dev_status) {
  extern __shared__ __align__(128) uint8_t stage[];   // 128 rows x 256 bytes
  __shared__ float red[kThreads / 32];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int blk = blockIdx.x, bh = blockIdx.y, which = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint16_t *src = which == 0 ? q : which == 1 ? k : v;
  const int64_t head = static_cast<int64_t>(bh) * N;
  const int r0 = blk * kRows, n_rows = min(kRows, N - r0);
  // The V kernel may be scheduled once every block of this one has begun.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (!stage_rows(src + (head + r0) * kD, smem_u32(stage), n_rows, smem_u32(&bar), &abort_flag,
                  dev_status))
    return;
  const bool rot = ROT && which < 2;
  float4 sg = make_float4(1.f, 1.f, 1.f, 1.f);
  if (rot) sg = *reinterpret_cast<const float4 *>(signs + 4 * lane);
  auto row_values = [&](int r) {
    float4 x = staged4(stage, r, n_rows, lane);
    if (rot) {
      x = make_float4(x.x * sg.x, x.y * sg.y, x.z * sg.z, x.w * sg.w);
      hadamard_row(x, lane);
    }
    return x;
  };
  // With the transform the rotated rows are kept in registers between the
  // two passes (the butterfly is the costly part); without it they are
  // re-read from shared memory, which keeps the kernel at 32 registers.
  float4 xr[ROT ? kRowsPerWarp : 1];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const float4 x = row_values(warp * kRowsPerWarp + i);
    if (ROT) xr[ROT ? i : 0] = x;
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
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
    const int r = warp * kRowsPerWarp + i;
    const float4 x = ROT ? xr[ROT ? i : 0] : row_values(r);
    if (r < n_rows)
      *reinterpret_cast<uint32_t *>(dst + (head + r0 + r) * kD + 4 * lane) = code4(x, inv);
  }
  if (threadIdx.x == 0)
    (which == 0 ? q_scale : k_scale)[static_cast<int64_t>(bh) * n_blk + blk] =
        ROT ? __fmul_rn(s, rot_factor) : s;
}

// grid (n_blk, BH): codes one 128-row block of V with its head's scale and
// writes it transposed into V^T [BH][128][Npad].  The block's bulk copy is
// issued first, so it lands while the head's block maxima are reduced.
//
// Transposition: warp w codes keys 16 w .. 16 w + 15 of the block and lane l
// the four dimensions 4 l .. 4 l + 3, four keys at a time.  The four code
// words of four keys (one byte per dimension) are transposed in registers
// with byte permutes into four words of one dimension (one byte per key), so
// after four rounds the lane holds, for each of its dimensions, the 16 keys
// of the warp as one 16-byte chunk.  The chunks pass through shared memory
// (a 16 KB tile in the staging buffer, chunk index XOR-swizzled by the
// dimension, so that neither the writes nor the reads have bank conflicts)
// and leave as whole 128-byte rows of V^T: eight lanes per row, four rows per
// store instruction.
__global__ void __launch_bounds__(kThreads)
    fp8_quant_v_kernel(const uint16_t *__restrict__ v, const float *__restrict__ v_amax,
                       uint8_t *__restrict__ vt8, float *__restrict__ v_scale, int N, int n_blk,
                       int n_pad, int *__restrict__ dev_status) {
  extern __shared__ __align__(128) uint8_t stage[];   // 128 rows x 256 bytes
  // The V^T block (128 dims x 128 keys, 16 KB) reuses the staging buffer once
  // every row has been read, so a CTA needs 32 KB and seven fit per SM.
  uint8_t *tile = stage;
  __shared__ float red[kThreads / 32];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int blk = blockIdx.x, bh = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t head = static_cast<int64_t>(bh) * N;
  const int r0 = blk * kRows, n_rows = min(kRows, N - r0);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(smem_u32(&bar), static_cast<uint32_t>(n_rows) * kD * 2);
    bulk_load(smem_u32(stage), v + (head + r0) * kD, static_cast<uint32_t>(n_rows) * kD * 2,
              smem_u32(&bar));
  }
  // A programmatic dependent of the rows kernel: its V block is already on
  // the way; the per-block maxima it reads next come from that kernel.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float amax = 0.f;
  for (int i = threadIdx.x; i < n_blk; i += kThreads)
    amax = fmaxf(amax, v_amax[static_cast<int64_t>(bh) * n_blk + i]);
  amax = block_max(amax, red);
  const float s = scale_of(amax);
  const float inv = __fdiv_rn(1.f, s);
  if (!mbar_wait(smem_u32(&bar), 0, &abort_flag)) {
    if (threadIdx.x == 0) atomicExch(dev_status, kDevTimeout);
    return;
  }
  uint32_t t4[4][4];   // [dimension 4 lane + e][round]: keys 4 round .. +3 of the warp
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    uint32_t cw[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      cw[kk] = code4(staged4(stage, 16 * warp + 4 * r + kk, n_rows, lane), inv);
    const uint32_t lo01 = __byte_perm(cw[0], cw[1], 0x5140);   // [a0 b0 a1 b1]
    const uint32_t lo23 = __byte_perm(cw[2], cw[3], 0x5140);   // [c0 d0 c1 d1]
    const uint32_t hi01 = __byte_perm(cw[0], cw[1], 0x7362);   // [a2 b2 a3 b3]
    const uint32_t hi23 = __byte_perm(cw[2], cw[3], 0x7362);   // [c2 d2 c3 d3]
    t4[0][r] = __byte_perm(lo01, lo23, 0x5410);
    t4[1][r] = __byte_perm(lo01, lo23, 0x7632);
    t4[2][r] = __byte_perm(hi01, hi23, 0x5410);
    t4[3][r] = __byte_perm(hi01, hi23, 0x7632);
  }
  __syncthreads();   // every staged row has been read: the tile may overwrite it
  // Chunk w of dimension row dd sits at 16-byte slot w ^ ((dd >> 2) & 7).
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int dd = 4 * lane + e;
    *reinterpret_cast<uint4 *>(tile + dd * kRows + ((warp ^ ((dd >> 2) & 7)) << 4)) =
        make_uint4(t4[e][0], t4[e][1], t4[e][2], t4[e][3]);
  }
  __syncthreads();
  // Row dd of V^T, keys blk*128 .. +127: lane l of warp w stores chunk l & 7
  // of row 16 w + 4 i + (l >> 3) in pass i.  Chunks at or past Npad are not
  // written (Npad is a multiple of 16, so a chunk never straddles it).
  uint8_t *out = vt8 + static_cast<int64_t>(bh) * kD * n_pad;
  const int chunk = lane & 7;
  const int key = blk * kRows + 16 * chunk;
  if (key < n_pad) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int dd = 16 * warp + 4 * i + (lane >> 3);
      const uint4 o = *reinterpret_cast<const uint4 *>(
          tile + dd * kRows + ((chunk ^ ((dd >> 2) & 7)) << 4));
      *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(dd) * n_pad + key) = o;
    }
  }
  if (blk == 0 && threadIdx.x == 0) v_scale[bh] = s;
}

constexpr int kStageBytes = kRows * kD * 2;   // 32 KB of staged bf16 rows

}  // namespace

size_t fp8_quant_workspace_bytes(int BH, int N) {
  return sizeof(float) * static_cast<size_t>(BH) * static_cast<size_t>((N + kRows - 1) / kRows);
}

cudaError_t launch_fp8_quantize(const void *q, const void *k, const void *v, const float *signs,
                                void *q8, void *k8, void *vt8, float *q_scale, float *k_scale,
                                float *v_scale, float *v_amax, int BH, int N, int n_pad,
                                float rot_factor, int *dev_status, cudaStream_t stream) {
  const int n_blk = (N + kRows - 1) / kRows;
  const dim3 g1(n_blk, BH, 3);
  const auto *qq = static_cast<const uint16_t *>(q);
  const auto *kk = static_cast<const uint16_t *>(k);
  const auto *vv = static_cast<const uint16_t *>(v);
  cudaError_t e;
  if (signs != nullptr) {
    e = cudaFuncSetAttribute(fp8_quant_rows_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes);
    if (e != cudaSuccess) return e;
    fp8_quant_rows_kernel<true><<<g1, kThreads, kStageBytes, stream>>>(
        qq, kk, vv, signs, static_cast<uint8_t *>(q8), static_cast<uint8_t *>(k8), q_scale,
        k_scale, v_amax, N, n_blk, rot_factor, dev_status);
  } else {
    e = cudaFuncSetAttribute(fp8_quant_rows_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes);
    if (e != cudaSuccess) return e;
    fp8_quant_rows_kernel<false><<<g1, kThreads, kStageBytes, stream>>>(
        qq, kk, vv, nullptr, static_cast<uint8_t *>(q8), static_cast<uint8_t *>(k8), q_scale,
        k_scale, v_amax, N, n_blk, rot_factor, dev_status);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fp8_quant_v_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kStageBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_blk, BH);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kStageBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fp8_quant_v_kernel, vv, static_cast<const float *>(v_amax),
                            static_cast<uint8_t *>(vt8), v_scale, N, n_blk, n_pad, dev_status);
}

}  // namespace fattn
