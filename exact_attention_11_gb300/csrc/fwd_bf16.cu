// fwd_bf16.cu -- exact attention forward, bf16 in/out, on the sm_103a tensor
// cores (tcgen05 MMAs with TMEM accumulators, TMA-staged tiles).
//
// What is computed: O = softmax(scale * Q K^T [+ causal mask]) V and the row
// log-sum-exp, with query blocks as the outer, parallel loop and key/value
// tiles as the inner loop ("FlashAttention: GPU 메모리 계층을 활용한 어텐션
// 최적화 분석", youngju.dev, sections 5 and 8.2).  Each key tile updates the
// running row max and running row sum with eqs. (2)-(3) of "Flash Attention"
// (suniverse77.github.io, section "Online Softmax"); the output accumulator
// is rescaled as in eq. (4) and normalised once at the end (youngju.dev,
// section 8.1), so the score matrix never leaves the SM.
//
// GB300 mapping.  One CTA owns two 128-row query tiles, A and B, of one head
// (256 rows); both use every K/V tile the CTA loads.  Warp roles (the
// warp-specialised design of youngju.dev section 9.2, "FlashAttention-3",
// rebuilt on tcgen05 and TMEM):
//   warp 0      TMA producer: Q_A and Q_B once, then K and V tiles into
//               separate multi-stage rings
//   warp 1      MMA issuer:   S_T = Q_T K^T into TMEM; O_T += P_T V with P_T
//               read from TMEM (T = A, B)
//   warps 2-3   idle (they complete the producer warpgroup)
//   warps 4-7   softmax of tile A, one query row per thread
//   warps 8-11  softmax of tile B
// TMEM (512 columns): S_A | S_B | O_A | O_B.  P_T is written as bf16 over the
// first half of S_T.  The MMA warp issues, per key tile j,
//     PV_A(j)  QK_A(j+1)  PV_B(j)  QK_B(j+1)
// so while the softmax of A works on S_A(j+1) the tensor core runs PV_B(j)
// and QK_B(j+1), and vice versa: the two softmax warpgroups take turns on the
// exponential unit while the tensor core stays busy (the matmul/softmax
// interleaving of section 9.2).  tcgen05 MMAs of one thread execute in issue
// order, so QK_T(j+1) overwriting S_T (and the P_T inside it) never overtakes
// PV_T(j), and the commit that signals S_T(j+1) also certifies that PV_T(j)
// finished, which lets the softmax warps rescale O_T without another wait.
//
// Rescaling the TMEM-resident output is skipped while the row max has grown
// by at most 8 (log2 units) since the value in use: exponentials are taken
// against that stale max (so they stay below 2^8) and the final division by
// the running sum, accumulated against the same max, cancels it exactly (the
// rescaling identity of youngju.dev, section 6.3).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int BM = 128;             // query rows per tile (MMA M)
constexpr int BN = 128;             // keys per tile (MMA N of QK^T, K of PV)
constexpr int kThreads = 384;       // 12 warps = 3 warpgroups
// Register split (setmaxnreg): the launch gives every thread 168 registers
// (65536 / 384, rounded to 8); the producer warpgroup drops to 72 and the two
// softmax warpgroups rise to 216, so each SM sub-partition, which hosts one
// warp of every warpgroup, needs 72 + 216 + 216 = 3 * 168 registers per lane.
// The build checks that ptxas gives this kernel exactly 168 at launch.
constexpr uint32_t kRegsProducer = 72, kRegsSoftmax = 216;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Cfg {
  static constexpr int kStages = D == 64 ? 4 : 2;   // K and V ring depth
  static constexpr int kBoxes = D / 64;             // 64-column (128-byte) boxes per row
  static constexpr int kTileBytes = BM * D * 2;     // one 128 x D bf16 tile
  static constexpr int kBoxBytes = BM * 128;        // 16 KB
  static constexpr int kQ = 0;                      // Q_A, Q_B
  static constexpr int kK0 = kQ + 2 * kTileBytes;
  static constexpr int kV0 = kK0 + kStages * kTileBytes;
  static constexpr int kBar = kV0 + kStages * kTileBytes;
  static constexpr int kBytes = kBar + 512;
  static constexpr int kAlloc = kBytes + 1024;      // slack for 1 KB alignment
  static constexpr uint32_t kColS0 = 0, kColS1 = 128;
  static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
};

// Barrier slots (8 bytes each).
enum : int {
  kBarQFull = 0,
  kBarSFull = 1,    // +tile (A, B)
  kBarPReady = 3,   // +tile
  kBarODone = 5,    // +tile
  kBarDrain = 7,
  kBarKFull = 8,    // +stage (up to 4)
  kBarKEmpty = 12,
  kBarVFull = 16,
  kBarVEmpty = 20,
  kNumBars = 24
};

struct SmemMisc {
  uint32_t tmem_base;
  int abort;
};

// Waits with a time limit for the phase of parity `ph` of an mbarrier; used
// on the unwind paths.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t ph) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, ph) && globaltimer_ns() - t0 < kWaitLimitNs) {
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16 *__restrict__ o,
                       float *__restrict__ lse, int N, int BH, int n_qblocks, float scale_log2,
                       int causal, int *__restrict__ dev_status) {
  using C = Cfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t bars = s_base + C::kBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  SmemMisc *misc = reinterpret_cast<SmemMisc *>(smem + C::kBar + 8 * kNumBars);
  volatile int *abort_flag = &misc->abort;

  // Heaviest query blocks first: under the causal mask they see more keys.
  const int qb = n_qblocks - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int q0 = qb * 2 * BM;
  const int n_kv_total = (N + BN - 1) / BN;
  // Key tiles each query tile needs (causal: up to and including its diagonal).
  const int n_a = causal ? min(2 * qb + 1, n_kv_total) : n_kv_total;
  const int n_b = causal ? min(2 * qb + 2, n_kv_total) : n_kv_total;
  const int n_kv = n_b;  // >= n_a

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPReady + t), 128);
      mbar_init(bar(kBarODone + t), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
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
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsProducer));
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(kBarQFull), 2 * C::kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(s_base + C::kQ + t * C::kTileBytes + b * C::kBoxBytes, &tm_q, b * 64,
                      q0 + t * BM, bh, bar(kBarQFull));
      int nk = 0, nv = 0;  // tiles issued
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int st = j % S;
        const uint32_t ph = (j / S) & 1;
        if (!(ok = mbar_wait(bar(kBarKEmpty + st), ph ^ 1, abort_flag))) break;
        mbar_arrive_expect_tx(bar(kBarKFull + st), C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(s_base + C::kK0 + st * C::kTileBytes + b * C::kBoxBytes, &tm_k, b * 64,
                      j * BN, bh, bar(kBarKFull + st));
        ++nk;
        if (!(ok = mbar_wait(bar(kBarVEmpty + st), ph ^ 1, abort_flag))) break;
        mbar_arrive_expect_tx(bar(kBarVFull + st), C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(s_base + C::kV0 + st * C::kTileBytes + b * C::kBoxBytes, &tm_v, b * 64,
                      j * BN, bh, bar(kBarVFull + st));
        ++nv;
      }
      if (!ok) {
        // Let the copies in flight land before the CTA exits.
        drain_wait(bar(kBarQFull), 0);
        for (int i = (nk > S ? nk - S : 0); i < nk; ++i)
          drain_wait(bar(kBarKFull + i % S), (i / S) & 1);
        for (int i = (nv > S ? nv - S : 0); i < nv; ++i)
          drain_wait(bar(kBarVFull + i % S), (i / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, true);
      auto qk = [&](int t, int j) {
        const uint32_t k_addr = s_base + C::kK0 + (j % S) * C::kTileBytes;
        const uint32_t q_addr = s_base + C::kQ + t * C::kTileBytes;
        const uint32_t s_col = t ? C::kColS1 : C::kColS0;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
          mma_ss(tmem + s_col, smem_desc_sw128(q_addr + off, 16, 1024),
                 smem_desc_sw128(k_addr + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(kBarSFull + t));
      };
      auto pv = [&](int t, int j) {
        const uint32_t v_addr = s_base + C::kV0 + (j % S) * C::kTileBytes;
        const uint32_t s_col = t ? C::kColS1 : C::kColS0;
        const uint32_t o_col = t ? C::kColO1 : C::kColO0;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tmem + o_col, tmem + s_col + kk * 8,
                 smem_desc_sw128(v_addr + kk * 2048, C::kBoxBytes, 1024), idesc_pv,
                 (j > 0 || kk > 0) ? 1u : 0u);
      };
      auto wait_k = [&](int j) {
        return mbar_wait(bar(kBarKFull + j % S), (j / S) & 1, abort_flag);
      };
      bool ok = mbar_wait(bar(kBarQFull), 0, abort_flag) && wait_k(0);
      if (ok) {
        tc_fence_after();
        qk(0, 0);
        qk(1, 0);
        mma_commit(bar(kBarKEmpty + 0));
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int st = j % S;
        if (!(ok = mbar_wait(bar(kBarVFull + st), (j / S) & 1, abort_flag))) break;
        bool k_next_ready = false;
        if (j < n_a) {
          if (!(ok = mbar_wait(bar(kBarPReady + 0), j & 1, abort_flag))) break;
          tc_fence_after();
          pv(0, j);
          if (j == n_a - 1) mma_commit(bar(kBarODone + 0));
          if (j + 1 < n_a) {
            if (!(ok = wait_k(j + 1))) break;
            k_next_ready = true;
            tc_fence_after();
            qk(0, j + 1);
          }
        }
        if (!(ok = mbar_wait(bar(kBarPReady + 1), j & 1, abort_flag))) break;
        tc_fence_after();
        pv(1, j);
        mma_commit(bar(kBarVEmpty + st));
        if (j == n_b - 1) mma_commit(bar(kBarODone + 1));
        if (j + 1 < n_b) {
          if (!k_next_ready && !(ok = wait_k(j + 1))) break;
          tc_fence_after();
          qk(1, j + 1);
          mma_commit(bar(kBarKEmpty + (j + 1) % S));
        }
      }
      // Drain: every MMA issued above has completed once this phase does.
      mma_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;                 // query tile: 0 = A, 1 = B
    const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + (threadIdx.x & 31);
    const int row = q0 + t * BM + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + (t ? C::kColS1 : C::kColS0);
    const uint32_t o_tmem = tmem + lane_off + (t ? C::kColO1 : C::kColO0);
    const int n_mine = t ? n_b : n_a;
    const uint64_t c2 = f2(scale_log2, scale_log2);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_mine; ++j) {
      if (!(ok = mbar_wait(bar(kBarSFull + t), j & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t sv[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + c * 32, sv[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_wait_ld(sv[c]);
#define S_(c) sv[(c) >> 5][(c) & 31]
      if (j == n_mine - 1) {
        // Keys past the sequence end, and (causal) keys after the query row.
        const int lim = (causal ? min(N, row + 1) : N) - j * BN;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= lim) S_(c) = __float_as_uint(-INFINITY);
      }
      float mx[4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
        mx[a] = fmaxf(__uint_as_float(S_(2 * a)), __uint_as_float(S_(2 * a + 1)));
#pragma unroll
      for (int c = 8; c < BN; c += 8)
#pragma unroll
        for (int a = 0; a < 4; ++a)
          mx[a] = fmax3(mx[a], __uint_as_float(S_(c + 2 * a)), __uint_as_float(S_(c + 2 * a + 1)));
      const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
      float alpha = 1.f;
      if (tmax > m + kRescaleThreshold) {  // also true while m = -inf
        alpha = ex2_approx(m - tmax);
        m = tmax;
      }
      const uint64_t nm2 = f2(-m, -m);
      uint64_t sum2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 x = f2_split(
              ffma2(f2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), c2, nm2));
          const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
          sum2[(e >> 1) & 1] = fadd2(sum2[(e >> 1) & 1], f2(p0, p1));
          pk[e >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st16(s_tmem + c * 16, pk);
      }
#undef S_
      const float2 sa = f2_split(fadd2(sum2[0], sum2[1]));
      l = l * alpha + (sa.x + sa.y);
      // PV_T(j-1) was issued before QK_T(j), so O_T is complete: rescale it.
      if (j > 0 && __any_sync(~0u, alpha != 1.f)) {
        const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(o_tmem + c * 32, ov);
          tmem_wait_ld(ov);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 x =
                f2_split(fmul2(f2(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1])), a2));
            ov[e] = __float_as_uint(x.x);
            ov[e + 1] = __float_as_uint(x.y);
          }
          tmem_st32(o_tmem + c * 32, ov);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarPReady + t));
    }
    if (ok) ok = mbar_wait(bar(kBarODone + t), 0, abort_flag);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
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
            w.x = pack_bf16x2(__uint_as_float(ov[8 * e + 0]) * inv_l,
                              __uint_as_float(ov[8 * e + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(ov[8 * e + 2]) * inv_l,
                              __uint_as_float(ov[8 * e + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(ov[8 * e + 4]) * inv_l,
                              __uint_as_float(ov[8 * e + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(ov[8 * e + 6]) * inv_l,
                              __uint_as_float(ov[8 * e + 7]) * inv_l);
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
  using C = Cfg<D>;
  cudaError_t e = cudaFuncSetAttribute(fwd_bf16_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc);
  if (e != cudaSuccess) return e;
  const int n_qblocks = (N + 2 * BM - 1) / (2 * BM);
  const float scale_log2 = scale * 1.4426950408889634f;
  dim3 grid(n_qblocks * BH);
  fwd_bf16_tc_kernel<D><<<grid, kThreads, C::kAlloc, stream>>>(
      tq, tk, tv, reinterpret_cast<__nv_bfloat16 *>(o), lse, N, BH, n_qblocks, scale_log2, causal,
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
