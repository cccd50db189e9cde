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
//   bwd_prep_kernel   D = rowsum(dO * O) and the LSE in log2 units (fp32)
//   bwd_main_kernel   one CTA per (128-key block j, head); K_j and V_j stay
//                     in shared memory and dK_j, dV_j in TMEM while the CTA
//                     visits every query block i that sees block j (the KV-
//                     outer order of FlashAttention-2's backward).  dQ is
//                     accumulated across CTAs with vector atomic adds into an
//                     fp32 buffer.
//   bwd_dq_kernel     dQ = scale * accumulator, rounded to bf16
//
// bwd_main_kernel, per query block i (warp 0 loads with TMA, warp 1 issues
// the MMAs, warps 4-7 own one key row each of the TMEM tiles):
//   S^T  = K_j Q_i^T   and   dP^T = V_j dO_i^T        (TMEM, lanes = keys)
//   P^T  = exp2(S^T * scale*log2e - LSE2_i),  dS^T = P^T (dP^T - D_i)
//          -> bf16 over the first half of each tile in TMEM; dS also into
//          shared memory in the layout an M-major MMA operand expects
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i                (A operand from TMEM)
//   dQ_i' = dS K_j                                     (two N = 64 halves, into
//          the TMEM columns the bf16 packing freed; lanes = queries)
//   the same warps read dQ_i' and add it into the fp32 accumulator.
// TMEM columns: [0,128) S^T / P^T, [128,256) dP^T / dS^T, [256,256+D) dV,
// [256+D, 256+2D) dK, and dQ' in [64,128) and [192,256).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int BM = 128;   // keys per CTA (MMA M of S^T, dP^T, dV, dK)
constexpr int BQ = 128;   // queries per step
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = 128 * D * 2;   // a 128 x D bf16 tile
  static constexpr int kBoxBytes = 128 * 128;      // 128 rows x 128 bytes
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;       // one stage
  static constexpr int kDO = kQ + kTileBytes;      // two stages
  static constexpr int kDS = kDO + 2 * kTileBytes; // dS^T, 128 keys x 128 queries bf16
  static constexpr int kVec = kDS + 128 * 128 * 2; // [2 bufs][LSE2 | D][128] f32
  static constexpr int kBar = kVec + 2 * 2 * BQ * 4;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
};

enum : int {
  kBarKV = 0,
  kBarQFull = 1,
  kBarQEmpty = 2,
  kBarDOFull = 3,    // +stage
  kBarDOEmpty = 5,   // +stage
  kBarSFull = 7,
  kBarPReady = 8,
  kBarDQFull = 9,
  kBarTmemFree = 10,
  kBarKVDone = 11,
  kBarDrain = 12,
  kBarVec = 13,      // +buffer: the 128 P/dS threads have written LSE2 and D
  kNumBars = 15
};

struct BMisc {
  uint32_t tmem_base;
  int abort;
};

// Bounded wait whose outcome is the same for every lane of the warp, so that
// the warp-collective TMEM loads that follow run on all lanes or on none.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t ph, volatile int *abort_flag) {
  return __all_sync(~0u, mbar_wait(bar, ph, abort_flag));
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t ph) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, ph) && globaltimer_ns() - t0 < kWaitLimitNs) {
  }
}

// D = rowsum(dO * O) and LSE2 = LSE * log2(e), one 16-thread group per row.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_prep_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                    const float *__restrict__ lse, float *__restrict__ dvec,
                    float *__restrict__ lse2, int64_t rows) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  const int part = threadIdx.x & 15;
  float acc = 0.f;
  if (row < rows) {
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
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(~0u, acc, off);
  if (row < rows && part == 0) {
    dvec[row] = acc;
    lse2[row] = lse[row] * kLog2e;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const float *__restrict__ lse2, const float *__restrict__ dvec,
                    float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dk,
                    __nv_bfloat16 *__restrict__ dv, int N, int BH, int n_kblocks,
                    float scale, int causal, int *__restrict__ dev_status) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t bars = s_base + C::kBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  BMisc *misc = reinterpret_cast<BMisc *>(smem + C::kBar + 8 * kNumBars);
  volatile int *abort_flag = &misc->abort;

  // Heaviest key blocks first: under the causal mask the first key block is
  // seen by every query block.
  const int jb = static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int k0 = jb * BM;
  const int n_qblocks = (N + BQ - 1) / BQ;
  const int i_first = causal ? jb : 0;   // key block jb is seen by query blocks >= jb
  const int n_steps = n_qblocks - i_first;

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarKV), 1);
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarDOFull + s), 1);
      mbar_init(bar(kBarDOEmpty + s), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarPReady), 4);
    mbar_init(bar(kBarDQFull), 1);
    mbar_init(bar(kBarTmemFree), 4);
    mbar_init(bar(kBarKVDone), 1);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarVec), 128);
    mbar_init(bar(kBarVec + 1), 128);
    misc->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar(kBarKV), 2 * C::kTileBytes);
      for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_3d(s_base + C::kK + b * C::kBoxBytes, &tm_k, b * 64, k0, bh, bar(kBarKV));
        tma_load_3d(s_base + C::kV + b * C::kBoxBytes, &tm_v, b * 64, k0, bh, bar(kBarKV));
      }
      int nq = 0, ndo = 0;
      bool ok = true;
      for (int s = 0; s < n_steps && ok; ++s) {
        const int q0 = (i_first + s) * BQ;
        const int st = s & 1;
        if (!(ok = mbar_wait(bar(kBarDOEmpty + st), ((s >> 1) & 1) ^ 1, abort_flag))) break;
        mbar_arrive_expect_tx(bar(kBarDOFull + st), C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(s_base + C::kDO + st * C::kTileBytes + b * C::kBoxBytes, &tm_do, b * 64,
                      q0, bh, bar(kBarDOFull + st));
        ndo = s + 1;
        if (!(ok = mbar_wait(bar(kBarQEmpty), (s & 1) ^ 1, abort_flag))) break;
        mbar_arrive_expect_tx(bar(kBarQFull), C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(s_base + C::kQ + b * C::kBoxBytes, &tm_q, b * 64, q0, bh, bar(kBarQFull));
        nq = s + 1;
      }
      if (!ok) {
        drain_wait(bar(kBarKV), 0);
        if (nq > 0) drain_wait(bar(kBarQFull), (nq - 1) & 1);
        for (int i = (ndo > 2 ? ndo - 2 : 0); i < ndo; ++i)
          drain_wait(bar(kBarDOFull + (i & 1)), (i >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BQ, false);        // S^T, dP^T
      constexpr uint32_t idesc_g = idesc_bf16_f32(BM, D, true);          // dV, dK
      constexpr uint32_t idesc_q = idesc_bf16_f32(BQ, 64, true, true);   // dQ' halves
      const uint64_t dk_desc = smem_desc_sw128(s_base + C::kK, 16, 1024);          // K-major
      const uint64_t dv_desc = smem_desc_sw128(s_base + C::kV, 16, 1024);
      const uint64_t dq_kmaj = smem_desc_sw128(s_base + C::kQ, 16, 1024);
      const uint64_t dq_mn = smem_desc_sw128(s_base + C::kQ, C::kBoxBytes, 1024);  // N-major
      const uint64_t ddo_kmaj = smem_desc_sw128(s_base + C::kDO, 16, 1024);
      const uint64_t ddo_mn = smem_desc_sw128(s_base + C::kDO, C::kBoxBytes, 1024);
      const uint64_t dk_mn = smem_desc_sw128(s_base + C::kK, C::kBoxBytes, 1024);
      const uint64_t dds = smem_desc_sw128(s_base + C::kDS, C::kBoxBytes, 1024);    // M-major
      bool ok = mbar_wait(bar(kBarKV), 0, abort_flag);
      for (int s = 0; s < n_steps && ok; ++s) {
        const int st = s & 1;
        const uint64_t do_off = (st * C::kTileBytes) >> 4;
        if (!(ok = mbar_wait(bar(kBarQFull), s & 1, abort_flag))) break;
        if (!(ok = mbar_wait(bar(kBarDOFull + st), (s >> 1) & 1, abort_flag))) break;
        // The previous step's dQ' has been read out of TMEM columns 64-255.
        if (s > 0 && !(ok = mbar_wait(bar(kBarTmemFree), (s - 1) & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::kColS, dk_desc + off, dq_kmaj + off, idesc_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::kColDP, dv_desc + off, ddo_kmaj + do_off + off, idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(kBarSFull));
        if (!(ok = mbar_wait(bar(kBarPReady), s & 1, abort_flag))) break;
        tc_fence_after();
        // dV += P^T dO, dK += dS^T Q  (A from TMEM, 16 queries per step).
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t off = (kk * 2048) >> 4;
          mma_ts(tmem + C::kColDV, tmem + C::kColS + kk * 8, ddo_mn + do_off + off, idesc_g,
                 (s > 0 || kk > 0) ? 1u : 0u);
          mma_ts(tmem + C::kColDK, tmem + C::kColDP + kk * 8, dq_mn + off, idesc_g,
                 (s > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(kBarQEmpty));
        mma_commit(bar(kBarDOEmpty + st));
        // dQ' = dS K: M = queries (dS^T in shared memory, M-major), N = 64
        // columns of d per half, K = keys.
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk) {
            const uint32_t off = (kk * 2048) >> 4;
            mma_ss(tmem + (h ? 192u : 64u), dds + off, dk_mn + ((h * C::kBoxBytes) >> 4) + off,
                   idesc_q, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(kBarDQFull));
      }
      if (ok) mma_commit(bar(kBarKVDone));
      mma_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0);
    }
  } else if (warp >= 4) {
    // -------------------------------------------- P, dS, dQ read-out, epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + (threadIdx.x & 31);   // key row of S^T; query row of dQ'
    const int tid = threadIdx.x - 128;                 // 0..127 among these warps
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int key = k0 + r;
    const float c = scale * kLog2e;
    float *vec = reinterpret_cast<float *>(smem + C::kVec);
    uint8_t *ds_smem = smem + C::kDS;
    bool ok = true;
    for (int s = 0; s < n_steps && ok; ++s) {
      const int q0 = (i_first + s) * BQ;
      // LSE2 and D of this step's 128 queries, shared by all key rows.
      float *lse_s = vec + (s & 1) * 2 * BQ, *d_s = lse_s + BQ;
      {
        const int qrow = q0 + tid;
        const bool in = qrow < N;
        lse_s[tid] = in ? lse2[static_cast<int64_t>(bh) * N + qrow] : INFINITY;
        d_s[tid] = in ? dvec[static_cast<int64_t>(bh) * N + qrow] : 0.f;
      }
      mbar_arrive(bar(kBarVec + (s & 1)));
      if (!(ok = wait_warp(bar(kBarVec + (s & 1)), (s >> 1) & 1, abort_flag))) break;
      if (!(ok = wait_warp(bar(kBarSFull), s & 1, abort_flag))) break;
      tc_fence_after();
      const bool diag = causal && (q0 < k0 + BM) && (q0 + BQ > k0);
#pragma unroll
      for (int ch = 0; ch < BQ / 32; ++ch) {
        uint32_t sv[32], dp[32];
        tmem_ld32(tmem + lane_off + C::kColS + ch * 32, sv);
        tmem_ld32(tmem + lane_off + C::kColDP + ch * 32, dp);
        tmem_wait_ld(sv);
        tmem_wait_ld(dp);
        uint32_t pk[16], dsk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p2[2], g2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int qi = ch * 32 + e + u;
            const int qrow = q0 + qi;
            float p = ex2_approx(fmaf(__uint_as_float(sv[e + u]), c, -lse_s[qi]));
            if (key >= N || (diag && key > qrow)) p = 0.f;
            p2[u] = p;
            g2[u] = p * (__uint_as_float(dp[e + u]) - d_s[qi]);
          }
          pk[e >> 1] = pack_bf16x2(p2[0], p2[1]);
          dsk[e >> 1] = pack_bf16x2(g2[0], g2[1]);
        }
        tmem_st16(tmem + lane_off + C::kColS + ch * 16, pk);
        tmem_st16(tmem + lane_off + C::kColDP + ch * 16, dsk);
        // dS^T row r into shared memory: queries 64b..64b+63 form box b, a
        // 128-byte row per key with the 128-byte swizzle (16-byte chunk index
        // XOR key % 8), the layout of an M-major MMA operand.
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int qc = ch * 32 + u * 8;        // first query of this 16-byte chunk
          const int box = qc >> 6, chunk = (qc & 63) >> 3;
          uint4 w;
          w.x = dsk[u * 4 + 0];
          w.y = dsk[u * 4 + 1];
          w.z = dsk[u * 4 + 2];
          w.w = dsk[u * 4 + 3];
          *reinterpret_cast<uint4 *>(ds_smem + box * C::kBoxBytes + r * 128 +
                                     ((chunk ^ (r & 7)) << 4)) = w;
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(bar(kBarPReady));
      // dQ' rows (lanes = queries) into the fp32 accumulator.
      if (!(ok = wait_warp(bar(kBarDQFull), s & 1, abort_flag))) break;
      tc_fence_after();
      const int qrow = q0 + r;
      float *dst = dq_acc + (static_cast<int64_t>(bh) * N + qrow) * D;
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t g[32];
          tmem_ld32(tmem + lane_off + (h ? 192u : 64u) + half * 32, g);
          tmem_wait_ld(g);
          if (qrow < N) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              red_add_v4(dst + h * 64 + half * 32 + e, __uint_as_float(g[e]),
                         __uint_as_float(g[e + 1]), __uint_as_float(g[e + 2]),
                         __uint_as_float(g[e + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(bar(kBarTmemFree));
    }
    // Epilogue: dK_j = scale * (dS^T Q), dV_j as bf16 rows.  Every lane runs
    // the TMEM loads (they are warp-collective); only rows < N are stored.
    if (ok && n_steps > 0) ok = wait_warp(bar(kBarKVDone), 0, abort_flag);
    if (ok) {
      tc_fence_after();
      const int64_t off = (static_cast<int64_t>(bh) * N + key) * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16 *dst = (which ? dk : dv) + off;
        const float mul = which ? scale : 1.f;
        const uint32_t col = which ? C::kColDK : C::kColDV;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t g[32];
          if (n_steps > 0) {
            tmem_ld32(tmem + lane_off + col + ch * 32, g);
            tmem_wait_ld(g);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) g[e] = 0u;  // no query sees this key block
          }
          if (key < N) {
            uint4 *w = reinterpret_cast<uint4 *>(dst + ch * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 x;
              x.x = pack_bf16x2(__uint_as_float(g[8 * e + 0]) * mul, __uint_as_float(g[8 * e + 1]) * mul);
              x.y = pack_bf16x2(__uint_as_float(g[8 * e + 2]) * mul, __uint_as_float(g[8 * e + 3]) * mul);
              x.z = pack_bf16x2(__uint_as_float(g[8 * e + 4]) * mul, __uint_as_float(g[8 * e + 5]) * mul);
              x.w = pack_bf16x2(__uint_as_float(g[8 * e + 6]) * mul, __uint_as_float(g[8 * e + 7]) * mul);
              w[e] = x;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && misc->abort) atomicExch(dev_status, kDevTimeout);
}

// dQ = scale * accumulator as bf16, eight elements per thread.
__global__ void __launch_bounds__(256)
    bwd_dq_kernel(const float *__restrict__ acc, __nv_bfloat16 *__restrict__ dq, int64_t n8,
                  float scale) {
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
                         const CUtensorMap &tdo, const void *o, const void *dout,
                         const float *lse, void *dq, void *dk, void *dv, int BH, int N,
                         float scale, int causal, float *ws, int *dev_status,
                         cudaStream_t stream) {
  using C = BCfg<D>;
  const int64_t rows = static_cast<int64_t>(BH) * N;
  // dQ accumulator first (16-byte aligned rows for the vector atomics), then D
  // and LSE2.
  float *dq_acc = ws, *dvec = ws + rows * D, *lse2 = dvec + rows;
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, sizeof(float) * rows * D, stream);
  if (e != cudaSuccess) return e;
  bwd_prep_kernel<D><<<static_cast<unsigned>((rows + 15) / 16), 256, 0, stream>>>(
      reinterpret_cast<const __nv_bfloat16 *>(o), reinterpret_cast<const __nv_bfloat16 *>(dout),
      lse, dvec, lse2, rows);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // At least 120 KB so that one CTA (which takes all 512 TMEM columns) runs
  // per SM.
  constexpr int kLaunchSmem = C::kAlloc > 120 * 1024 ? C::kAlloc : 120 * 1024;
  e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kLaunchSmem);
  if (e != cudaSuccess) return e;
  const int n_kblocks = (N + BM - 1) / BM;
  bwd_main_kernel<D><<<n_kblocks * BH, kThreads, kLaunchSmem, stream>>>(
      tq, tk, tv, tdo, lse2, dvec, dq_acc, reinterpret_cast<__nv_bfloat16 *>(dk),
      reinterpret_cast<__nv_bfloat16 *>(dv), N, BH, n_kblocks, scale, causal, dev_status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t n8 = rows * D / 8;
  bwd_dq_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream>>>(
      dq_acc, reinterpret_cast<__nv_bfloat16 *>(dq), n8, scale);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(int BH, int N, int d) {
  const size_t rows = static_cast<size_t>(BH) * N;
  return sizeof(float) * rows * (2 + static_cast<size_t>(d));
}

cudaError_t launch_bwd_bf16(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &tdo, const void *o, const void *dout,
                            const float *lse, void *dq, void *dk, void *dv, int BH, int N, int d,
                            float scale, int causal, float *ws, int *dev_status,
                            cudaStream_t stream) {
  if (d == 64)
    return launch_bwd_d<64>(tq, tk, tv, tdo, o, dout, lse, dq, dk, dv, BH, N, scale, causal, ws,
                            dev_status, stream);
  return launch_bwd_d<128>(tq, tk, tv, tdo, o, dout, lse, dq, dk, dv, BH, N, scale, causal, ws,
                           dev_status, stream);
}

}  // namespace fattn
