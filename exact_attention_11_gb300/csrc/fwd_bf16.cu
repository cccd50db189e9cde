// fwd_bf16.cu -- exact attention forward, bf16 in/out, on the sm_103a tensor
// cores (tcgen05 MMAs with TMEM accumulators, TMA-staged tiles).
//
// What is computed: O = softmax(scale * Q K^T [+ causal mask]) V and the
// row log-sum-exp, one 128-row query tile at a time, with key/value tiles as
// the inner loop ("FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화 분석",
// youngju.dev, sections 5 and 8.2: query blocks are the outer, parallel
// loop).  Each key tile updates the running row max and running row sum with
// eqs. (2)-(3) of "Flash Attention" (suniverse77.github.io, section "Online
// Softmax"); the output accumulator is rescaled as in eq. (4) and normalised
// once at the end (youngju.dev, section 8.1), so the score matrix never
// leaves the SM.
//
// GB300 mapping (the roles of the warp-specialised design of section 9.2,
// "FlashAttention-3", rebuilt on tcgen05):
//   warp 0      TMA producer: Q once, then K and V tiles into a 2-stage ring
//   warp 1      MMA issuer:   S = Q K^T into TMEM; O += P V with P from TMEM
//   warps 2-5   softmax:      one query row per thread, read from TMEM
// S is double-buffered in TMEM so the tensor core computes the next tile's
// scores while the softmax warps work on the current one (section 9.2,
// "matmul and softmax interleaving").  P is written back as bf16 over the
// first half of its S buffer and consumed from TMEM by the PV MMA.
//
// Rescaling the TMEM-resident output is skipped while the row max has grown
// by at most 8 (log2 units) since the value last used: the exponentials are
// then taken against that stale max, which bounds them by 2^8, and the final
// division by the running sum -- accumulated against the same stale max --
// cancels it exactly (the rescaling identity of youngju.dev, section 6.3).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int BM = 128;            // query rows per tile (MMA M)
constexpr int BN = 128;            // keys per tile (MMA N of QK^T, K of PV)
constexpr int kThreads = 192;      // 6 warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Smem {
  static constexpr int kBoxes = D / 64;             // 64-column (128-byte) boxes per row
  static constexpr int kTileBytes = BM * D * 2;     // one 128 x D bf16 tile
  static constexpr int kBoxBytes = BM * 128;        // 16 KB
  static constexpr int kQ = 0;
  static constexpr int kK0 = kQ + kTileBytes;
  static constexpr int kV0 = kK0 + 2 * kTileBytes;
  static constexpr int kBar = kV0 + 2 * kTileBytes;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;      // slack for 1 KB alignment
};

// Barrier slots (8 bytes each) inside the barrier block.
enum : int {
  kBarQFull = 0,
  kBarKFull = 1,    // +stage
  kBarKEmpty = 3,   // +stage
  kBarVFull = 5,    // +stage
  kBarVEmpty = 7,   // +stage
  kBarSFull = 9,    // +S buffer
  kBarPReady = 11,  // +S buffer
  kBarPV = 13,      // one phase per completed PV
  kBarDrain = 14,
  kNumBars = 15
};

struct SmemMisc {
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16 *__restrict__ o,
                       float *__restrict__ lse, int N, int BH, int n_qtiles, float scale_log2,
                       int causal, int *__restrict__ dev_status) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t bars = s_base + L::kBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  SmemMisc *misc = reinterpret_cast<SmemMisc *>(smem + L::kBar + 8 * kNumBars);
  volatile int *abort_flag = &misc->abort;

  // Heaviest tiles first: under the causal mask, high query tiles see more keys.
  const int qt = n_qtiles - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int q0 = qt * BM;
  const int n_kv_total = (N + BN - 1) / BN;
  const int n_kv = causal ? min(qt + 1, n_kv_total) : n_kv_total;

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarPReady + s), 128);
    }
    mbar_init(bar(kBarPV), 1);
    mbar_init(bar(kBarDrain), 1);
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
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(kBarQFull), L::kTileBytes);
      for (int b = 0; b < L::kBoxes; ++b)
        tma_load_3d(s_base + L::kQ + b * L::kBoxBytes, &tm_q, b * 64, q0, bh, bar(kBarQFull));
      int issued_k[2] = {0, 0}, issued_v[2] = {0, 0};
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        ok = mbar_wait(bar(kBarKEmpty + st), ph ^ 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(kBarKFull + st), L::kTileBytes);
        for (int b = 0; b < L::kBoxes; ++b)
          tma_load_3d(s_base + L::kK0 + st * L::kTileBytes + b * L::kBoxBytes, &tm_k, b * 64,
                      j * BN, bh, bar(kBarKFull + st));
        ++issued_k[st];
        ok = mbar_wait(bar(kBarVEmpty + st), ph ^ 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(kBarVFull + st), L::kTileBytes);
        for (int b = 0; b < L::kBoxes; ++b)
          tma_load_3d(s_base + L::kV0 + st * L::kTileBytes + b * L::kBoxBytes, &tm_v, b * 64,
                      j * BN, bh, bar(kBarVFull + st));
        ++issued_v[st];
      }
      if (!ok) {
        // Let copies already in flight land before the CTA exits.
        for (int st = 0; st < 2; ++st) {
          const uint64_t t0 = globaltimer_ns();
          while (issued_k[st] > 0 && !mbar_try_wait(bar(kBarKFull + st), (issued_k[st] - 1) & 1) &&
                 globaltimer_ns() - t0 < kWaitLimitNs) {
          }
          while (issued_v[st] > 0 && !mbar_try_wait(bar(kBarVFull + st), (issued_v[st] - 1) & 1) &&
                 globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, true);
      bool ok = mbar_wait(bar(kBarQFull), 0, abort_flag);
      auto issue_pv = [&](int jj) -> bool {
        const int st = jj & 1;
        const uint32_t ph = (jj >> 1) & 1;
        if (!mbar_wait(bar(kBarPReady + st), ph, abort_flag)) return false;
        if (!mbar_wait(bar(kBarVFull + st), ph, abort_flag)) return false;
        tc_fence_after();
        const uint32_t p_tmem = tmem + (st ? kColS1 : kColS0);
        const uint32_t v_addr = s_base + L::kV0 + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(v_addr + kk * 2048, L::kBoxBytes, 1024);
          mma_ts(tmem + kColO, p_tmem + kk * 8, bdesc, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(kBarVEmpty + st));
        mma_commit(bar(kBarPV));
        return true;
      };
      for (int j = 0; j < n_kv && ok; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        ok = mbar_wait(bar(kBarKFull + st), ph, abort_flag);
        // S buffer st is free once PV(j-2), which read P from it, is done.
        if (ok && j >= 2) ok = mbar_wait(bar(kBarPV), (j - 2) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_tmem = tmem + (st ? kColS1 : kColS0);
        const uint32_t k_addr = s_base + L::kK0 + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kBoxBytes + (kk & 3) * 32;
          const uint64_t adesc = smem_desc_sw128(s_base + L::kQ + off, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(k_addr + off, 16, 1024);
          mma_ss(s_tmem, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(kBarSFull + st));
        mma_commit(bar(kBarKEmpty + st));
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(n_kv - 1);
      // Drain: every MMA issued above has completed once this phase does.
      mma_commit(bar(kBarDrain));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar(kBarDrain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + (threadIdx.x & 31);
    const int row = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      ok = mbar_wait(bar(kBarSFull + st), ph, abort_flag);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_tmem = tmem + lane_off + (st ? kColS1 : kColS0);
      uint32_t sv[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + c * 32, sv[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_wait_ld(sv[c]);
#define S_(c) sv[(c) >> 5][(c) & 31]
      if (j == n_kv - 1) {
        // Keys past the sequence end, and (causal) keys after the query row.
        const int lim = (causal ? min(N, row + 1) : N) - j * BN;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= lim) S_(c) = __float_as_uint(-INFINITY);
      }
      float smax = __uint_as_float(S_(0));
#pragma unroll
      for (int c = 1; c < BN; ++c) smax = fmaxf(smax, __uint_as_float(S_(c)));
      const float tmax = smax * scale_log2;
      float alpha = 1.f;
      if (tmax > m + kRescaleThreshold) {  // also true while m = -inf
        alpha = ex2_approx(m - tmax);
        m = tmax;
      }
      const float neg_m = -m;
      float psum = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(S_(c)), scale_log2, neg_m));
        const float p1 = ex2_approx(fmaf(__uint_as_float(S_(c + 1)), scale_log2, neg_m));
        psum += p0 + p1;
        pk[c >> 1] = pack_bf16x2(p0, p1);
      }
#undef S_
      l = l * alpha + psum;
      tmem_st32(s_tmem, pk);
      tmem_st32(s_tmem + 32, pk + 32);
      // Rescale O by alpha (eq. (4)) once PV(j-1) has finished with it.
      if (j > 0 && __any_sync(~0u, alpha != 1.f)) {
        ok = mbar_wait(bar(kBarPV), (j - 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t o_tmem = tmem + lane_off + kColO;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(o_tmem + c * 32, ov);
          tmem_wait_ld(ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(o_tmem + c * 32, ov);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarPReady + st));
    }
    if (ok) ok = mbar_wait(bar(kBarPV), (n_kv - 1) & 1, abort_flag);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const uint32_t o_tmem = tmem + lane_off + kColO;
      __nv_bfloat16 *orow = o + (static_cast<int64_t>(bh) * N + row) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(o_tmem + c * 32, ov);
        tmem_wait_ld(ov);
        if (row < N) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(ov[8 * e + 0]) * inv_l, __uint_as_float(ov[8 * e + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(ov[8 * e + 2]) * inv_l, __uint_as_float(ov[8 * e + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(ov[8 * e + 4]) * inv_l, __uint_as_float(ov[8 * e + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(ov[8 * e + 6]) * inv_l, __uint_as_float(ov[8 * e + 7]) * inv_l);
            dst[e] = w;
          }
        }
      }
      if (lse != nullptr && row < N)
        lse[static_cast<int64_t>(bh) * N + row] = (m + __log2f(l)) * 0.6931471805599453f;
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

template <int D>
cudaError_t launch_d(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, void *o,
                     float *lse, int BH, int N, float scale, int causal, int *dev_status,
                     cudaStream_t stream) {
  using L = Smem<D>;
  cudaError_t e = cudaFuncSetAttribute(fwd_bf16_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int n_qtiles = (N + BM - 1) / BM;
  const float scale_log2 = scale * 1.4426950408889634f;
  dim3 grid(n_qtiles * BH);
  fwd_bf16_tc_kernel<D><<<grid, kThreads, L::kAlloc, stream>>>(
      tq, tk, tv, reinterpret_cast<__nv_bfloat16 *>(o), lse, N, BH, n_qtiles, scale_log2, causal,
      dev_status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            void *o, float *lse, int BH, int N, int d, float scale, int causal,
                            int *dev_status, cudaStream_t stream) {
  if (d == 64) return launch_d<64>(tq, tk, tv, o, lse, BH, N, scale, causal, dev_status, stream);
  return launch_d<128>(tq, tk, tv, o, lse, BH, N, scale, causal, dev_status, stream);
}

}  // namespace fattn
