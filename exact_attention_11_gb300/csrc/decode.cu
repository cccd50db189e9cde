// decode.cu -- single-query attention over a paged KV cache (bf16).
//
// Operation and cache layouts: "PagedAttention" (data-sketchers.com), the
// walkthrough of vLLM's single-query kernel: q [num_seqs, num_heads,
// head_size]; k_cache [num_blocks, num_heads, head_size/x, block_size, x]
// with x = 8 bf16 (one 16-byte vector); v_cache [num_blocks, num_heads,
// head_size, block_size]; a block table maps a sequence's logical blocks to
// physical ones (sections "Inputs", "Concepts", "Key", "Value").
//
// Work split: one CTA per (partition, head, sequence), a partition being 512
// consecutive context tokens (32 cache blocks), the split that the page's
// grid (num_heads, num_seqs, max_num_partitions) implies.  Inside a CTA each
// of the 4 warps streams whole cache blocks -- one (block, head) slice of K
// or V is 4 KB of contiguous memory -- with 16-byte loads arranged so every
// load instruction of the warp covers 512 contiguous bytes.  Rather than the
// page's two passes (all logits into shared memory, then a second sweep), a
// warp keeps the online-softmax state of "Flash Attention"
// (suniverse77.github.io, eqs. (2)-(4)) over the blocks it has seen, so each
// block's keys and values are read once, back to back.  The four warps'
// states, and later the partitions' states, are merged with eq. (4).  The
// last CTA of a (sequence, head) to finish -- found with a counter in the
// workspace -- performs the partition merge, so no second kernel is needed.
//
// Scores are kept in the log2 domain: q is pre-multiplied by scale*log2(e)
// so that exp(s - m) becomes exp2(t - m2).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "decode_util.cuh"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int kHead = kDecodeHeadSize;    // 128
constexpr int kBlk = kDecodeBlockSize;    // 16 tokens per cache block
constexpr int kX = 8;                     // bf16 per 16-byte vector
constexpr int kPartBlocks = kDecodePartitionTokens / kBlk;  // 32
constexpr int kWarps = 4;

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float dot8(const float *q8, uint4 kv) {
  float a = q8[0] * bf_lo(kv.x);
  a = fmaf(q8[1], bf_hi(kv.x), a);
  a = fmaf(q8[2], bf_lo(kv.y), a);
  a = fmaf(q8[3], bf_hi(kv.y), a);
  a = fmaf(q8[4], bf_lo(kv.z), a);
  a = fmaf(q8[5], bf_hi(kv.z), a);
  a = fmaf(q8[6], bf_lo(kv.w), a);
  a = fmaf(q8[7], bf_hi(kv.w), a);
  return a;
}

__device__ __forceinline__ float fma8(const float *p8, uint4 vv, float acc) {
  acc = fmaf(p8[0], bf_lo(vv.x), acc);
  acc = fmaf(p8[1], bf_hi(vv.x), acc);
  acc = fmaf(p8[2], bf_lo(vv.y), acc);
  acc = fmaf(p8[3], bf_hi(vv.y), acc);
  acc = fmaf(p8[4], bf_lo(vv.z), acc);
  acc = fmaf(p8[5], bf_hi(vv.z), acc);
  acc = fmaf(p8[6], bf_lo(vv.w), acc);
  acc = fmaf(p8[7], bf_hi(vv.w), acc);
  return acc;
}

__global__ void __launch_bounds__(kWarps * 32)
    paged_decode_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k_cache,
                        const __nv_bfloat16 *__restrict__ v_cache, const int *__restrict__ block_tables,
                        const int *__restrict__ context_lens, __nv_bfloat16 *__restrict__ out,
                        float *__restrict__ ws_o, float *__restrict__ ws_ml, int *__restrict__ counters,
                        int num_heads, int max_blocks, int max_parts, float qscale) {
  const int part = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int ctx = context_lens[s];
  const int n_blocks = (ctx + kBlk - 1) / kBlk;
  const int n_parts = (n_blocks + kPartBlocks - 1) / kPartBlocks;
  const int64_t sh = (int64_t)s * num_heads + h;
  __nv_bfloat16 *out_row = out + sh * kHead;

  if (ctx <= 0) {  // no visible token: zero output (only partition 0 writes)
    if (part == 0) out_row[threadIdx.x] = __float2bfloat16_rn(0.f);
    return;
  }
  if (part >= n_parts) return;

  __shared__ float sq[kHead];
  __shared__ float s_m[kWarps], s_l[kWarps];
  __shared__ float s_acc[kWarps][kHead];
  __shared__ int s_last;

  sq[threadIdx.x] = __bfloat162float(q[sh * kHead + threadIdx.x]) * qscale;
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Key mapping: lane -> token (lane & 15), chunk parity (lane >> 4); the
  // lane reads chunks c = 2i + parity, i = 0..7, of its token.
  const int ktok = lane & 15, kpar = lane >> 4;
  float qreg[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) qreg[i][e] = sq[(2 * i + kpar) * kX + e];
  // Value mapping: lane -> rows d = (lane >> 1) + 16 j, tokens 8 (lane & 1) .. +7.
  const int vrow = lane >> 1, vhalf = lane & 1;

  float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;

  const int b_begin = part * kPartBlocks;
  const int b_end = min(n_blocks, b_begin + kPartBlocks);
  const int *bt = block_tables + (int64_t)s * max_blocks;
  const int64_t head_stride = (int64_t)kHead * kBlk;           // elements of one (block, head)
  const int64_t block_stride = head_stride * num_heads;

  for (int b = b_begin + warp; b < b_end; b += kWarps) {
    const int64_t pb = bt[b];
    const __nv_bfloat16 *kb = k_cache + pb * block_stride + h * head_stride;
    const __nv_bfloat16 *vb = v_cache + pb * block_stride + h * head_stride;
    uint4 kv[8], vv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) kv[i] = ld_stream(kb + ((2 * i + kpar) * kBlk + ktok) * kX);
#pragma unroll
    for (int j = 0; j < 8; ++j) vv[j] = ld_stream(vb + (vrow + 16 * j) * kBlk + 8 * vhalf);
    const int nv = ctx - b * kBlk - 8 * vhalf;   // this lane's value tokens inside the context
    if (nv < 8) {
#pragma unroll
      for (int j = 0; j < 8; ++j) vv[j] = keep_first_16b(vv[j], nv);
    }

    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += dot8(qreg[i], kv[i]);
    t += __shfl_xor_sync(~0u, t, 16);
    if (b * kBlk + ktok >= ctx) t = -INFINITY;  // past the context: masked
    float bmax = t;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(~0u, bmax, off));
    const float m_new = fmaxf(m, bmax);           // eq. (2); finite: token b*16 < ctx
    const float alpha = ex2_approx(m - m_new);    // 0 on the first block
    const float p = ex2_approx(t - m_new);
    float psum = p;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) psum += __shfl_xor_sync(~0u, psum, off);
    l = l * alpha + psum;                          // eq. (3)
    m = m_new;
    float p8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) p8[e] = __shfl_sync(~0u, p, 8 * vhalf + e);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = fma8(p8, vv[j], acc[j] * alpha);  // eq. (4)
  }
  // The two lanes of a row hold tokens 0-7 and 8-15: add them.
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] += __shfl_xor_sync(~0u, acc[j], 1);
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
  if (vhalf == 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j) s_acc[warp][vrow + 16 * j] = acc[j];
  }
  __syncthreads();

  // Merge the warps (eq. (4)); warps that saw no block have m = -inf.
  float M = s_m[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_m[w]);
  float L = 0.f, O = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float f = (s_m[w] == -INFINITY) ? 0.f : ex2_approx(s_m[w] - M);
    L += s_l[w] * f;
    O += s_acc[w][threadIdx.x] * f;
  }

  if (n_parts == 1) {
    out_row[threadIdx.x] = __float2bfloat16_rn(O / L);
    return;
  }

  // Publish this partition's (m, l, unnormalised o) and count arrivals.
  const int64_t slot = sh * max_parts + part;
  ws_o[slot * kHead + threadIdx.x] = O;
  if (threadIdx.x == 0) {
    ws_ml[slot * 2 + 0] = M;
    ws_ml[slot * 2 + 1] = L;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&counters[sh], 1);
    s_last = (prev == n_parts - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // Last CTA: merge all partitions of this (sequence, head) with eq. (4).
  float Mp = -INFINITY;
  for (int p2 = 0; p2 < n_parts; ++p2) Mp = fmaxf(Mp, __ldcg(&ws_ml[(sh * max_parts + p2) * 2]));
  float Lt = 0.f, Ot = 0.f;
  for (int p2 = 0; p2 < n_parts; ++p2) {
    const int64_t sl = sh * max_parts + p2;
    const float f = ex2_approx(__ldcg(&ws_ml[sl * 2]) - Mp);
    Lt += __ldcg(&ws_ml[sl * 2 + 1]) * f;
    Ot += __ldcg(&ws_o[sl * kHead + threadIdx.x]) * f;
  }
  out_row[threadIdx.x] = __float2bfloat16_rn(Ot / Lt);
  if (threadIdx.x == 0) counters[sh] = 0;  // ready for the next call
}

}  // namespace

size_t decode_workspace_bytes(int num_seqs, int num_heads, int max_parts) {
  const size_t slots = (size_t)num_seqs * num_heads * max_parts;
  return slots * (kHead + 2) * sizeof(float);
}

int decode_max_parts(int max_num_blocks_per_seq) {
  return (max_num_blocks_per_seq + kPartBlocks - 1) / kPartBlocks;
}

cudaError_t launch_paged_decode(const void *q, const void *k_cache, const void *v_cache,
                                const int *block_tables, const int *context_lens, void *out,
                                int num_seqs, int num_heads, int max_blocks, float scale,
                                float *workspace, int *counters, cudaStream_t stream) {
  const int max_parts = decode_max_parts(max_blocks);
  const size_t slots = (size_t)num_seqs * num_heads * max_parts;
  float *ws_o = workspace;
  float *ws_ml = ws_o + slots * kHead;
  dim3 grid(max_parts, num_heads, num_seqs);
  const float qscale = scale * 1.4426950408889634f;  // scale * log2(e)
  paged_decode_kernel<<<grid, kWarps * 32, 0, stream>>>(
      reinterpret_cast<const __nv_bfloat16 *>(q), reinterpret_cast<const __nv_bfloat16 *>(k_cache),
      reinterpret_cast<const __nv_bfloat16 *>(v_cache), block_tables, context_lens,
      reinterpret_cast<__nv_bfloat16 *>(out), ws_o, ws_ml, counters, num_heads, max_blocks,
      max_parts, qscale);
  return cudaGetLastError();
}


}  // namespace fattn
