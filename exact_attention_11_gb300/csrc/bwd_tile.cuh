// bwd_tile.cuh -- the element-wise step shared by the backward kernels
// (bwd_bf16_d128.cu, bwd_bf16_d64.cu): from the recomputed scores S^T and
// dP^T of one 128-key x 64-query sub-tile in TMEM, the probabilities
// P^T = exp(S^T - LSE) and dS^T = P^T (dP^T - D) of the recomputation
// scheme of "FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화 분석"
// (youngju.dev, section 7), packed to bf16 for the MMAs that use them.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace fattn {
namespace bwd_tile {

constexpr int kSubQ = 64;   // queries per sub-tile

// P^T and dS^T of one 32-query chunk (columns ch*32 .. +31 of the sub-tile)
// for this lane's key row r.  vec holds [-LSE2 x 64 | -D x 64]; c2 =
// scale*log2e in both halves.  Returns both as packed bf16 pairs and stores
// dS^T row r to shared memory (128-byte swizzle).  With MASKED, P = 0 for
// keys >= N and, when diag (the causal diagonal block), for keys later than
// the query.
template <bool MASKED>
__device__ __forceinline__ void chunk(uint32_t R, int ch, const float *vec, uint8_t *ds_buf, int r,
                                      int key, int q0, int N, bool diag, uint64_t c2,
                                      uint32_t (&pk)[16], uint32_t (&dsk)[16]) {
  uint32_t sv[32], dp[32];
  tmem_ld32(R + ch * 32, sv);
  tmem_ld32(R + 64 + ch * 32, dp);
  tmem_wait_ld(sv);
  tmem_wait_ld(dp);
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    // -LSE2 and -D of queries ch*32+e .. +3 as packed pairs (broadcast).
    const ulonglong2 nl = *reinterpret_cast<const ulonglong2 *>(vec + ch * 32 + e);
    const ulonglong2 nd = *reinterpret_cast<const ulonglong2 *>(vec + kSubQ + ch * 32 + e);
    const float2 x01 = f2_split(ffma2(f2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                      c2, nl.x));
    const float2 x23 = f2_split(ffma2(f2(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])),
                                      c2, nl.y));
    float p[4] = {ex2_approx(x01.x), ex2_approx(x01.y), ex2_approx(x23.x), ex2_approx(x23.y)};
    if (MASKED) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (key >= N || (diag && key > q0 + ch * 32 + e + u)) p[u] = 0.f;
    }
    const uint64_t p01 = f2(p[0], p[1]), p23 = f2(p[2], p[3]);
    const float2 g01 = f2_split(fmul2(
        p01, fadd2(f2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd.x)));
    const float2 g23 = f2_split(fmul2(
        p23, fadd2(f2(__uint_as_float(dp[e + 2]), __uint_as_float(dp[e + 3])), nd.y)));
    pk[e >> 1] = pack_bf16x2(p[0], p[1]);
    pk[(e >> 1) + 1] = pack_bf16x2(p[2], p[3]);
    dsk[e >> 1] = pack_bf16x2(g01.x, g01.y);
    dsk[(e >> 1) + 1] = pack_bf16x2(g23.x, g23.y);
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint4 w;
    w.x = dsk[u * 4 + 0];
    w.y = dsk[u * 4 + 1];
    w.z = dsk[u * 4 + 2];
    w.w = dsk[u * 4 + 3];
    *reinterpret_cast<uint4 *>(ds_buf + r * 128 + (((4 * ch + u) ^ (r & 7)) << 4)) = w;
  }
}

// Both chunks of the sub-tile.  P^T ends at R[0,32) and dS^T at R[32,64) as
// packed bf16 pairs (queries 2c, 2c+1 in column c): chunk 1 (S columns 32-63)
// goes first so that dS^T of chunk 1 may overwrite S columns 48-63 at once;
// P^T of chunk 1 waits in registers until chunk 0 has read columns 0-31.
template <bool MASKED>
__device__ __forceinline__ void chunks(uint32_t R, const float *vec, uint8_t *ds_buf, int r,
                                       int key, int q0, int N, bool diag, uint64_t c2) {
  uint32_t pk1[16], dsk1[16], pk0[16], dsk0[16];
  chunk<MASKED>(R, 1, vec, ds_buf, r, key, q0, N, diag, c2, pk1, dsk1);
  tmem_st16(R + 48, dsk1);
  chunk<MASKED>(R, 0, vec, ds_buf, r, key, q0, N, diag, c2, pk0, dsk0);
  tmem_st16(R + 0, pk0);
  tmem_st16(R + 16, pk1);
  tmem_st16(R + 32, dsk0);
}

}  // namespace bwd_tile
}  // namespace fattn
