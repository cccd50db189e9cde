// decode_gqa.cu -- single-query paged decode with grouped key/value heads
// (bf16): num_heads query heads share num_kv_heads < num_heads cached
// key/value heads, G = num_heads / num_kv_heads query heads per cached head.
//
// Layouts: "PagedAttention" (data-sketchers.com), sections "Inputs" and
// "Key": k_cache [num_blocks, num_kv_heads, head_size/x, block_size, x],
// v_cache [num_blocks, num_kv_heads, head_size, block_size], the key pointer
// offset by kv_head_idx.  Query head h reads key/value head h / G
// (consecutive query heads share one cached head).
//
// The decode is bound by reading the cache, so the point of the grouping is
// to read each (block, key/value head) slice once for several query heads: one
// CTA per (partition, key/value head, sub-group, sequence) handles GC = min(G,
// 4) query heads (more would need more registers than a thread has: each lane
// keeps 8 accumulators per head), so a slice is read G / GC times instead of
// G times.  Four warps stream whole
// cache blocks exactly as the one-head kernel in decode.cu does (16-byte
// loads, 512 contiguous bytes per warp load), and for every block each warp
// updates GC online-softmax states ("Flash Attention", suniverse77.github.io,
// eqs. (2)-(4)) from the same key and value registers.  Warp states, then
// partition states, merge with eq. (4); the last CTA of a (sequence,
// key/value head, sub-group) merges the partitions of its query heads.
// With GC heads the arithmetic per block is GC times the one-head kernel's,
// so a warp cannot hide the load latency behind a single block's math: each
// warp keeps a ring of kStages blocks in shared memory (three CTAs per SM), filled by 4 KB bulk
// copies (TMA engine) that complete on an mbarrier, so the next blocks'
// loads overlap this block's math.
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
constexpr int kStages = 2;                          // blocks in flight per warp
constexpr int kSlice = kHead * kBlk * 2;            // bytes of one (block, head) slice: 4 KB
constexpr int kStageBytes = 2 * kSlice;             // K and V
constexpr int kRingBytes = kWarps * kStages * kStageBytes;   // 64 KB dynamic shared memory

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int G>
__global__ void __launch_bounds__(kWarps * 32, 3)
    paged_decode_gqa_kernel(const __nv_bfloat16 *__restrict__ q,
                            const __nv_bfloat16 *__restrict__ k_cache,
                            const __nv_bfloat16 *__restrict__ v_cache,
                            const int *__restrict__ block_tables,
                            const int *__restrict__ context_lens, __nv_bfloat16 *__restrict__ out,
                            float *__restrict__ ws_o, float *__restrict__ ws_ml,
                            int *__restrict__ counters, int num_heads, int num_kv_heads,
                            int max_blocks, int max_parts, float qscale,
                            int *__restrict__ dev_status) {
  // blockIdx.y = key/value head * n_sub + sub-group; this CTA's query heads
  // are kvh * (num_heads / num_kv_heads) + sub * G + 0 .. G-1.
  const int n_sub = num_heads / num_kv_heads / G;
  const int part = blockIdx.x, kvh = blockIdx.y / n_sub;
  const int s = blockIdx.z;
  const int ctx = context_lens[s];
  const int n_blocks = (ctx + kBlk - 1) / kBlk;
  const int n_parts = (n_blocks + kPartBlocks - 1) / kPartBlocks;
  const int64_t sh0 = (int64_t)s * num_heads + (int64_t)blockIdx.y * G;  // first (sequence, head) row
  __nv_bfloat16 *out_rows = out + sh0 * kHead;                      // G consecutive rows

  if (ctx <= 0) {  // no visible token: zero outputs (only partition 0 writes)
    if (part == 0)
      for (int i = threadIdx.x; i < G * kHead; i += kWarps * 32)
        out_rows[i] = __float2bfloat16_rn(0.f);
    return;
  }
  if (part >= n_parts) return;

  extern __shared__ __align__(128) uint8_t ring[];   // [warp][stage][K 4 KB | V 4 KB]
  __shared__ __align__(16) float sq[G][kHead];
  __shared__ float s_m[kWarps][G], s_l[kWarps][G];
  __shared__ float s_acc[kWarps][G][kHead];
  __shared__ __align__(8) uint64_t s_full[kWarps][kStages];
  __shared__ int s_last, s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The G query rows, pre-scaled by scale*log2(e) (scores in log2 units).
  for (int i = threadIdx.x; i < G * kHead; i += kWarps * 32)
    sq[i / kHead][i % kHead] = __bfloat162float(q[sh0 * kHead + i]) * qscale;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w)
      for (int st = 0; st < kStages; ++st) mbar_init(smem_u32(&s_full[w][st]), 1);
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Key mapping: lane -> token (lane & 15), chunk parity (lane >> 4); the lane
  // reads chunks c = 2i + parity, i = 0..7, of its token.
  const int ktok = lane & 15, kpar = lane >> 4;
  // Value mapping: lane -> rows d = (lane >> 1) + 16 j, tokens 8 (lane & 1) .. +7.
  const int vrow = lane >> 1, vhalf = lane & 1;

  // acc2[g][j]: two partial sums (even and odd tokens of the lane's eight)
  // of output row vrow + 16 j of head g, as one packed fp32 pair.
  float m[G], l[G];
  uint64_t acc2[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc2[g][j] = f2(0.f, 0.f);
  }

  const int b_begin = part * kPartBlocks;
  const int b_end = min(n_blocks, b_begin + kPartBlocks);
  const int *bt = block_tables + (int64_t)s * max_blocks;
  const int64_t head_stride = (int64_t)kHead * kBlk;             // elements of one (block, head)
  const int64_t block_stride = head_stride * num_kv_heads;

  // This warp's blocks: b_begin + warp + kWarps * k, k = 0 .. n_mine-1.
  const int n_mine = b_end > b_begin + warp ? (b_end - b_begin - warp + kWarps - 1) / kWarps : 0;
  uint8_t *my_ring = ring + warp * kStages * kStageBytes;
  const uint32_t my_ring_u32 = smem_u32(my_ring);
  int n_issued = 0;           // lane 0: copies issued so far (blocks 0 .. n_issued-1)
  auto issue = [&](int k) {   // lane 0: copy block k's K and V slices into stage k % kStages
    const int b = b_begin + warp + kWarps * k;
    const int64_t pb = bt[b];
    const int st = k % kStages;
    const uint32_t full = smem_u32(&s_full[warp][st]);
    mbar_arrive_expect_tx(full, kStageBytes);
    bulk_load(my_ring_u32 + st * kStageBytes, k_cache + pb * block_stride + kvh * head_stride,
              kSlice, full);
    bulk_load(my_ring_u32 + st * kStageBytes + kSlice,
              v_cache + pb * block_stride + kvh * head_stride, kSlice, full);
    n_issued = k + 1;
  };
  if (lane == 0)
    for (int k = 0; k < kStages && k < n_mine; ++k) issue(k);
  bool ok = true;

  for (int k = 0; k < n_mine; ++k) {
    const int b = b_begin + warp + kWarps * k;
    const int st = k % kStages;
    if (!(ok = __all_sync(~0u, mbar_wait(smem_u32(&s_full[warp][st]), (k / kStages) & 1,
                                         &s_abort)))) break;
    const uint8_t *kb = my_ring + st * kStageBytes;
    const uint8_t *vb = kb + kSlice;
    const bool tail = b * kBlk + ktok >= ctx;   // this lane's token is past the context

    // Scores: this lane's token against its 8 key chunks (dimensions 8c ..
    // 8c + 7, c = 2i + parity); each chunk is read and widened once and used
    // by every head, two dimensions per packed fp32 FMA.
    uint64_t t2[G];
#pragma unroll
    for (int g = 0; g < G; ++g) t2[g] = f2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = 2 * i + kpar;
      const uint4 kv = *reinterpret_cast<const uint4 *>(kb + ((c * kBlk + ktok) * kX) * 2);
      const uint64_t k01 = f2(bf_lo(kv.x), bf_hi(kv.x)), k23 = f2(bf_lo(kv.y), bf_hi(kv.y));
      const uint64_t k45 = f2(bf_lo(kv.z), bf_hi(kv.z)), k67 = f2(bf_lo(kv.w), bf_hi(kv.w));
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float4 *q4 = reinterpret_cast<const float4 *>(&sq[g][c * kX]);
        const float4 a = q4[0], b4 = q4[1];
        t2[g] = ffma2(f2(a.x, a.y), k01, t2[g]);
        t2[g] = ffma2(f2(a.z, a.w), k23, t2[g]);
        t2[g] = ffma2(f2(b4.x, b4.y), k45, t2[g]);
        t2[g] = ffma2(f2(b4.z, b4.w), k67, t2[g]);
      }
    }
    float alpha[G], p8[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float2 tt = f2_split(t2[g]);
      float t = tt.x + tt.y;
      t += __shfl_xor_sync(~0u, t, 16);
      if (tail) t = -INFINITY;
      float bmax = t;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(~0u, bmax, off));
      const float m_new = fmaxf(m[g], bmax);       // eq. (2); finite: token b*16 < ctx
      alpha[g] = ex2_approx(m[g] - m_new);         // 0 on the first block
      const float p = ex2_approx(t - m_new);
      float psum = p;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) psum += __shfl_xor_sync(~0u, psum, off);
      l[g] = l[g] * alpha[g] + psum;               // eq. (3)
      m[g] = m_new;
#pragma unroll
      for (int e = 0; e < 8; ++e) p8[g][e] = __shfl_sync(~0u, p, 8 * vhalf + e);
    }
    // Values: each 16-byte chunk read and widened once, used by all heads
    // (eq. (4)), two tokens per packed FMA.
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint64_t a2 = f2(alpha[g], alpha[g]);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc2[g][j] = fmul2(acc2[g][j], a2);
    }
    const int nv = ctx - b * kBlk - 8 * vhalf;   // this lane's value tokens inside the context
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint4 vv = *reinterpret_cast<const uint4 *>(vb + ((vrow + 16 * j) * kBlk + 8 * vhalf) * 2);
      if (nv < 8) vv = keep_first_16b(vv, nv);
      const uint64_t v01 = f2(bf_lo(vv.x), bf_hi(vv.x)), v23 = f2(bf_lo(vv.y), bf_hi(vv.y));
      const uint64_t v45 = f2(bf_lo(vv.z), bf_hi(vv.z)), v67 = f2(bf_lo(vv.w), bf_hi(vv.w));
#pragma unroll
      for (int g = 0; g < G; ++g) {
        uint64_t a = acc2[g][j];
        a = ffma2(f2(p8[g][0], p8[g][1]), v01, a);
        a = ffma2(f2(p8[g][2], p8[g][3]), v23, a);
        a = ffma2(f2(p8[g][4], p8[g][5]), v45, a);
        a = ffma2(f2(p8[g][6], p8[g][7]), v67, a);
        acc2[g][j] = a;
      }
    }
    // The stage has been read: refill it with block k + kStages.
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && k + kStages < n_mine) issue(k + kStages);
  }
  if (!ok) {
    // A copy did not arrive in time: wait (bounded) for the ones in flight,
    // report, and leave this partition's output unwritten.
    if (lane == 0) {
      for (int k = n_issued > kStages ? n_issued - kStages : 0; k < n_issued; ++k) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&s_full[warp][k % kStages]), (k / kStages) & 1) &&
               globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
      atomicExch(dev_status, kDevTimeout);
    }
  }
  // Every warp takes part in the merge; s_abort tells them to stop there.
  __syncthreads();
  if (s_abort) return;
  // The two lanes of a row hold tokens 0-7 and 8-15: add them (after the
  // even and odd halves of each lane's packed sums).
  float acc[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 a = f2_split(acc2[g][j]);
      acc[g][j] = a.x + a.y;
      acc[g][j] += __shfl_xor_sync(~0u, acc[g][j], 1);
    }
    if (lane == 0) {
      s_m[warp][g] = m[g];
      s_l[warp][g] = l[g];
    }
    if (vhalf == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) s_acc[warp][g][vrow + 16 * j] = acc[g][j];
    }
  }
  __syncthreads();

  // Merge the warps (eq. (4)) for each (query head g, column d); warps that
  // saw no block have m = -inf.
  const int64_t slot0 = sh0 * max_parts + part;   // workspace slot of head g: slot0 + g*max_parts
  for (int i = threadIdx.x; i < G * kHead; i += kWarps * 32) {
    const int g = i / kHead, d = i % kHead;
    float M = s_m[0][g];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_m[w][g]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = (s_m[w][g] == -INFINITY) ? 0.f : ex2_approx(s_m[w][g] - M);
      L += s_l[w][g] * f;
      O += s_acc[w][g][d] * f;
    }
    if (n_parts == 1) {
      out_rows[i] = __float2bfloat16_rn(O / L);
    } else {
      const int64_t slot = slot0 + (int64_t)g * max_parts;
      ws_o[slot * kHead + d] = O;
      if (d == 0) {
        ws_ml[slot * 2 + 0] = M;
        ws_ml[slot * 2 + 1] = L;
      }
    }
  }
  if (n_parts == 1) return;

  // Count arrivals per (sequence, key/value head, sub-group); the last CTA
  // merges.
  __threadfence();
  __syncthreads();
  const int64_t ci = (int64_t)s * num_kv_heads * n_sub + blockIdx.y;
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&counters[ci], 1);
    s_last = (prev == n_parts - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  for (int i = threadIdx.x; i < G * kHead; i += kWarps * 32) {
    const int g = i / kHead, d = i % kHead;
    const int64_t base = (sh0 + g) * max_parts;
    float Mp = -INFINITY;
    for (int p2 = 0; p2 < n_parts; ++p2) Mp = fmaxf(Mp, __ldcg(&ws_ml[(base + p2) * 2]));
    float Lt = 0.f, Ot = 0.f;
    for (int p2 = 0; p2 < n_parts; ++p2) {
      const int64_t sl = base + p2;
      const float f = ex2_approx(__ldcg(&ws_ml[sl * 2]) - Mp);
      Lt += __ldcg(&ws_ml[sl * 2 + 1]) * f;
      Ot += __ldcg(&ws_o[sl * kHead + d]) * f;
    }
    out_rows[i] = __float2bfloat16_rn(Ot / Lt);
  }
  if (threadIdx.x == 0) counters[ci] = 0;  // ready for the next call
}

template <int G>
cudaError_t launch_g(const void *q, const void *k_cache, const void *v_cache,
                     const int *block_tables, const int *context_lens, void *out, int num_seqs,
                     int num_heads, int num_kv_heads, int max_blocks, float qscale, float *ws_o,
                     float *ws_ml, int *counters, int max_parts, int *dev_status,
                     cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(paged_decode_gqa_kernel<G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(max_parts, num_heads / G, num_seqs);
  paged_decode_gqa_kernel<G><<<grid, kWarps * 32, kRingBytes, stream>>>(
      reinterpret_cast<const __nv_bfloat16 *>(q), reinterpret_cast<const __nv_bfloat16 *>(k_cache),
      reinterpret_cast<const __nv_bfloat16 *>(v_cache), block_tables, context_lens,
      reinterpret_cast<__nv_bfloat16 *>(out), ws_o, ws_ml, counters, num_heads, num_kv_heads,
      max_blocks, max_parts, qscale, dev_status);
  return cudaGetLastError();
}

}  // namespace

bool decode_gqa_group_supported(int group) {
  return group == 2 || (group >= 4 && group % 4 == 0);
}

cudaError_t launch_paged_decode_gqa(const void *q, const void *k_cache, const void *v_cache,
                                    const int *block_tables, const int *context_lens, void *out,
                                    int num_seqs, int num_heads, int num_kv_heads, int max_blocks,
                                    float scale, float *workspace, int *counters,
                                    int *dev_status, cudaStream_t stream) {
  const int max_parts = decode_max_parts(max_blocks);
  const size_t slots = (size_t)num_seqs * num_heads * max_parts;
  float *ws_o = workspace;
  float *ws_ml = ws_o + slots * kHead;
  const float qscale = scale * 1.4426950408889634f;  // scale * log2(e)
  const int group = num_heads / num_kv_heads;
  if (!decode_gqa_group_supported(group) || group * num_kv_heads != num_heads)
    return cudaErrorInvalidValue;
  if (group == 2)
    return launch_g<2>(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, num_heads,
                       num_kv_heads, max_blocks, qscale, ws_o, ws_ml, counters, max_parts, dev_status,
                       stream);
  return launch_g<4>(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, num_heads,
                     num_kv_heads, max_blocks, qscale, ws_o, ws_ml, counters, max_parts, dev_status,
                       stream);
}

}  // namespace fattn
