// fwd_d256.cu -- exact attention forward for head dimension 256 (bf16 or
// fp16 in and out) on the sm_103a tensor cores.
//
// What is computed is the forward of fwd_bf16.cu: O = softmax(scale * Q K^T
// [+ causal mask]) V and the row log-sum-exp, key/value tiles as the inner
// loop with the running max and sum of eqs. (2)-(3) of "Flash Attention"
// (suniverse77.github.io, section "Online Softmax") and one normalisation at
// the end ("FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화 분석",
// youngju.dev, sections 5, 8.1 and 11.4, where head dimensions up to 256 are
// served).
//
// Why a kernel of its own: with d = 256 one 128-row output accumulator fills
// half of TMEM (256 of 512 columns), so the two-tile ping-pong of the d <= 128
// kernel has no room for its scores.  Here each CTA works on one 128-row query
// tile and double-buffers the scores instead:
//   TMEM  O [0, 256) | S_0 [256, 384) | S_1 [384, 512)
// and the MMA warp issues, per key tile g,
//   P V(g)  then  Q K^T(g + 2) into the S buffer P(g) came from,
// so the tensor core computes the scores two tiles ahead while the softmax
// works, and Q K^T(g + 2) can never overwrite P(g) before P V(g) has read it
// (tcgen05 MMAs of one thread execute in issue order).  The look-ahead runs
// across work items: the next item's first score tiles are computed while the
// current item's softmax and epilogue finish.  The output is rescaled only
// when a row max grows by more than 8 (log2 units) over the reference in use
// (the rescaling identity of youngju.dev, section 6.3), after the previous
// P V has finished.
//
// Shared memory (one CTA per SM): Q 64 KB (four 64-column boxes); K in a ring
// of five 16 KB chunks (128 keys x 64 dimensions, the unit one group of four
// Q K^T MMAs reads, freed chunk by chunk); V in a ring of two 32 KB halves (64
// keys x 256 dimensions, the unit one half of P V reads).  Warp roles:
//   warp 0       TMA producer of Q and K; claims the work items
//   warp 1       MMA issuer
//   warp 2       TMA producer of V
//   warp 3       idle
//   warps 4-7    softmax, one query row per thread, and the epilogue
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int BM = 128;                 // query rows per tile (MMA M)
constexpr int BN = 128;                 // keys per tile
constexpr int D = 256;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256;    // S_b at kColS + 128 b
constexpr float kRescaleThreshold = 8.0f;     // log2 units

constexpr int kBox = 128 * 128;               // 128 rows x 128 bytes (64 columns)
constexpr int kKChunks = 5;                   // K ring depth, in 64-dimension chunks
constexpr int kVBox = 64 * 128;               // 64 keys x 64 dimensions
constexpr int kVHalfBytes = 4 * kVBox;        // 64 keys x 256 dimensions
constexpr int kVHalves = 2;                   // V ring depth, in halves
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + 4 * kBox;
constexpr int kOffV = kOffK + kKChunks * kBox;
constexpr int kOffBar = kOffV + kVHalves * kVHalfBytes;
// Epilogue staging: per softmax warp its 32 rows x 64 columns of output, 4 KB.
constexpr int kOffStage = kOffBar + 512;
constexpr int kSmemBytes = kOffStage + 4 * 4096;
constexpr int kAlloc = kSmemBytes + 1024;     // slack for 1 KB alignment
static_assert(kAlloc <= 227 * 1024, "shared memory budget");

constexpr int kItemSlots = 4;
enum : int {
  kBarQFull = 0,
  kBarQEmpty = 1,
  kBarSFull = 2,       // + S buffer (2)
  kBarPReady = 4,      // + 2 * buffer + half (4), one arrival per softmax warp
  kBarPVDone = 8,      // + S buffer (2): P V of a tile from that buffer finished
  kBarDrain = 10,
  kBarKFull = 11,      // + chunk slot (5)
  kBarKEmpty = 16,     // + chunk slot (5)
  kBarVFull = 21,      // + half slot (2)
  kBarVEmpty = 23,     // + half slot (2)
  kBarItemFull = 25,   // + item slot (4)
  kBarItemEmpty = 29,  // + item slot (4)
  kNumBars = 33
};
// Arrivals that free an item slot: the V producer, the MMA thread (after the
// item's last P V) and the four softmax warps.
constexpr int kItemConsumers = 1 + 1 + 4;

struct SmemMisc {
  uint32_t tmem_base;
  int abort;
  int item[kItemSlots];
};
static_assert(8 * kNumBars + sizeof(SmemMisc) <= 512, "barrier area");

template <bool F16>
__device__ __forceinline__ constexpr uint32_t idesc16(uint32_t bf16_desc) {
  return F16 ? (bf16_desc & ~((1u << 7) | (1u << 10))) : bf16_desc;
}
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if (F16) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
  return pack_bf16x2(lo, hi);
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t ph) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, ph) && globaltimer_ns() - t0 < kWaitLimitNs) {
  }
}

// Work item w: one 128-row query block of one head, heaviest first.
struct Items {
  int BH, n_qb, causal;
  __device__ void decode(int w, int &q0, int &bh, int &n) const {
    const int qb = n_qb - 1 - w / BH;
    bh = w % BH;
    q0 = qb * BM;
    n = causal ? qb + 1 : n_qb;
  }
};

template <bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_d256_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, uint16_t *__restrict__ o,
                    float *__restrict__ lse, int N, int BH, float scale_log2, int causal,
                    int *__restrict__ sched, int *__restrict__ dev_status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  auto bar = [&](int i) { return s_base + kOffBar + 8u * i; };
  SmemMisc *misc = reinterpret_cast<SmemMisc *>(smem + kOffBar + 8 * kNumBars);
  volatile int *abort_flag = &misc->abort;

  Items items;
  items.BH = BH;
  items.n_qb = (N + BM - 1) / BM;
  items.causal = causal;
  const int n_items = items.n_qb * BH;

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarSFull + b), 1);
      mbar_init(bar(kBarPReady + 2 * b), 4);
      mbar_init(bar(kBarPReady + 2 * b + 1), 4);
      mbar_init(bar(kBarPVDone + b), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    for (int s = 0; s < kKChunks; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
    }
    for (int s = 0; s < kVHalves; ++s) {
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(bar(kBarItemFull + s), 1);
      mbar_init(bar(kBarItemEmpty + s), kItemConsumers);
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
  // Launched as a programmatic dependent of the kernel before it: the set-up
  // above overlaps that kernel's tail; global memory is touched only after it.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Reads item slot k once it is published (every consumer but the MMA
  // thread frees its share right away; the MMA thread frees it after the
  // item's last P V, because it reads the slot again then).
  auto read_item = [&](int k, int &w) -> bool {
    const int slot = k % kItemSlots;
    if (!mbar_wait(bar(kBarItemFull + slot), (k / kItemSlots) & 1, abort_flag)) return false;
    w = *reinterpret_cast<volatile int *>(&misc->item[slot]);
    return true;
  };

  if (warp == 0) {
    if (elect_one()) {
      // ------------------------------------------------ Q and K producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      int nq = 0, nk = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int slot = k % kItemSlots;
        if (!(ok = mbar_wait(bar(kBarItemEmpty + slot), ((k / kItemSlots) & 1) ^ 1, abort_flag)))
          break;
        const int w = atomicAdd(sched, 1);
        misc->item[slot] = w;
        mbar_arrive(bar(kBarItemFull + slot));
        if (w >= n_items) break;
        int q0, bh, n;
        items.decode(w, q0, bh, n);
        if (!(ok = mbar_wait(bar(kBarQEmpty), (nq & 1) ^ 1, abort_flag))) break;
        mbar_arrive_expect_tx(bar(kBarQFull), 4 * kBox);
        for (int b = 0; b < 4; ++b)
          tma_load_3d(s_base + kOffQ + b * kBox, &tm_q, b * 64, q0, bh, bar(kBarQFull));
        ++nq;
        for (int j = 0; j < n && ok; ++j) {
          for (int c = 0; c < 4; ++c, ++nk) {
            const int st = nk % kKChunks;
            if (!(ok = mbar_wait(bar(kBarKEmpty + st), ((nk / kKChunks) & 1) ^ 1, abort_flag)))
              break;
            mbar_arrive_expect_tx(bar(kBarKFull + st), kBox);
            tma_load_3d(s_base + kOffK + st * kBox, &tm_k, c * 64, j * BN, bh, bar(kBarKFull + st));
          }
        }
      }
      if (!ok) {
        if (nq > 0) drain_wait(bar(kBarQFull), (nq - 1) & 1);
        for (int i = (nk > kKChunks ? nk - kKChunks : 0); i < nk; ++i)
          drain_wait(bar(kBarKFull + i % kKChunks), (i / kKChunks) & 1);
      }
    }
  } else if (warp == 2) {
    if (elect_one()) {
      // ------------------------------------------------------ V producer
      tma_prefetch_desc(&tm_v);
      int nv = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int w;
        if (!(ok = read_item(k, w))) break;
        mbar_arrive(bar(kBarItemEmpty + k % kItemSlots));
        if (w >= n_items) break;
        int q0, bh, n;
        items.decode(w, q0, bh, n);
        for (int j = 0; j < n && ok; ++j) {
          for (int h = 0; h < 2; ++h, ++nv) {
            const int st = nv % kVHalves;
            if (!(ok = mbar_wait(bar(kBarVEmpty + st), ((nv / kVHalves) & 1) ^ 1, abort_flag)))
              break;
            mbar_arrive_expect_tx(bar(kBarVFull + st), kVHalfBytes);
            for (int b = 0; b < 4; ++b)
              tma_load_3d(s_base + kOffV + st * kVHalfBytes + b * kVBox, &tm_v, b * 64,
                          j * BN + h * 64, bh, bar(kBarVFull + st));
          }
        }
      }
      if (!ok)
        for (int i = (nv > kVHalves ? nv - kVHalves : 0); i < nv; ++i)
          drain_wait(bar(kBarVFull + i % kVHalves), (i / kVHalves) & 1);
    }
  } else if (warp == 1) {
    if (elect_one()) {
      // -------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_qk = idesc16<F16>(idesc_bf16_f32(BM, BN, false));
      constexpr uint32_t idesc_pv = idesc16<F16>(idesc_bf16_f32(BM, D, true));
      const uint32_t dq = sdesc_lo(s_base + kOffQ, 16);
      const uint32_t dk = sdesc_lo(s_base + kOffK, 16);
      const uint32_t dv = sdesc_lo(s_base + kOffV, kVBox);   // V is read N-major
      // Q K^T cursor: item kq, tile jq of nq_tiles; P V cursor: item kp, tile jp.
      int kq = 0, jq = 0, nq_tiles = 0, kp = 0, jp = 0;
      int n_qitems = 0;          // items whose Q was consumed (Q barrier parity)
      int nk = 0, nv = 0;        // K chunks and V halves consumed
      int gq = 0, gp = 0;        // tiles whose Q K^T / P V were issued
      bool more = true, ok = true;
      // Issues Q K^T for the next tile in order; false once there is none.
      auto issue_qk = [&]() -> bool {
        if (jq == nq_tiles) {
          int w;
          if (!(ok = read_item(kq, w))) return false;
          if (w >= n_items) {
            mbar_arrive(bar(kBarItemEmpty + kq % kItemSlots));
            more = false;
            return false;
          }
          int q0, bh;
          items.decode(w, q0, bh, nq_tiles);
          jq = 0;
          if (!(ok = mbar_wait(bar(kBarQFull), n_qitems & 1, abort_flag))) return false;
        }
        const int b = gq & 1;
        const uint32_t s_col = tmem + kColS + 128 * b;
#pragma unroll 1
        for (int c = 0; c < 4; ++c, ++nk) {
          const int st = nk % kKChunks;
          if (!(ok = mbar_wait(bar(kBarKFull + st), (nk / kKChunks) & 1, abort_flag))) return false;
          tc_fence_after();
          const uint32_t a = dq + ((c * kBox) >> 4);
          const uint32_t bb = dk + ((st * kBox) >> 4);
          mma_ss_lo(s_col, a, bb, idesc_qk, c > 0 ? 1u : 0u);
          mma_ss_lo(s_col, a + 2, bb + 2, idesc_qk, 1u);
          mma_ss_lo(s_col, a + 4, bb + 4, idesc_qk, 1u);
          mma_ss_lo(s_col, a + 6, bb + 6, idesc_qk, 1u);
          mma_commit(bar(kBarKEmpty + st));
        }
        mma_commit(bar(kBarSFull + b));
        if (++jq == nq_tiles) {
          mma_commit(bar(kBarQEmpty));   // the item's last Q K^T has been issued
          ++n_qitems;
          ++kq;
        }
        ++gq;
        return true;
      };
      if (issue_qk()) issue_qk();
      while (ok && gp < gq) {
        // P V for tile gp, in two halves of 64 keys.
        const int b = gp & 1;
        const int item_slot = kp % kItemSlots;
        const bool first = jp == 0;
#pragma unroll 1
        for (int h = 0; h < 2 && ok; ++h, ++nv) {
          if (!(ok = mbar_wait(bar(kBarPReady + 2 * b + h), (gp >> 1) & 1, abort_flag))) break;
          const int st = nv % kVHalves;
          if (!(ok = mbar_wait(bar(kBarVFull + st), (nv / kVHalves) & 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t p_col = tmem + kColS + 128 * b + 32 * h;
          const uint32_t bv = dv + ((st * kVHalfBytes) >> 4);
          mma_ts_lo(tmem + kColO, p_col, bv, idesc_pv, (first && h == 0) ? 0u : 1u);
          mma_ts_lo(tmem + kColO, p_col + 8, bv + (2048 >> 4), idesc_pv, 1u);
          mma_ts_lo(tmem + kColO, p_col + 16, bv + (4096 >> 4), idesc_pv, 1u);
          mma_ts_lo(tmem + kColO, p_col + 24, bv + (6144 >> 4), idesc_pv, 1u);
          mma_commit(bar(kBarVEmpty + st));
        }
        if (!ok) break;
        mma_commit(bar(kBarPVDone + b));
        ++gp;
        // The P V tile's item: free its slot after its last tile.
        {
          int w = *reinterpret_cast<volatile int *>(&misc->item[item_slot]);
          int q0, bh, n;
          items.decode(w, q0, bh, n);
          if (++jp == n) {
            mbar_arrive(bar(kBarItemEmpty + item_slot));
            ++kp;
            jp = 0;
          }
        }
        if (more) issue_qk();
      }
      mma_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int r_local = quarter * 32 + (threadIdx.x & 31);
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t o_tmem = tmem + lane_off + kColO;
    const uint64_t c2 = f2(scale_log2, scale_log2);
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int w;
      if (!(ok = read_item(k, w))) break;
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(bar(kBarItemEmpty + k % kItemSlots));
      if (w >= n_items) break;
      int q0, bh, n;
      items.decode(w, q0, bh, n);
      const int row = q0 + r_local;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j, ++g) {
        const int b = g & 1;
        const uint32_t s_tmem = tmem + lane_off + kColS + 128 * b;
        if (!(ok = mbar_wait(bar(kBarSFull + b), (g >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        uint32_t sv[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + c * 32, sv[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_wait_ld(sv[c]);
#define S_(c) sv[(c) >> 5][(c) & 31]
        if (j == n - 1) {
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
        // Rescale O once the previous tile's P V (from the other buffer) is
        // done; this tile's P V cannot start before its P exists.
        if (j > 0 && __any_sync(~0u, alpha != 1.f)) {
          if (!(ok = mbar_wait(bar(kBarPVDone + (b ^ 1)), ((g - 1) >> 1) & 1, abort_flag)))
            break;
          tc_fence_after();
          const uint64_t a2 = f2(alpha, alpha);
#pragma unroll 1
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
        const uint64_t nm2 = f2(-m, -m);
        uint64_t sum2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const uint64_t x2 =
                ffma2(f2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), c2, nm2);
            const float2 x = f2_split(x2);
            const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            sum2[(e >> 1) & 1] = fadd2(sum2[(e >> 1) & 1], f2(p.x, p.y));
            pk[e >> 1] = pack2<F16>(p.x, p.y);
          }
          tmem_st16(s_tmem + c * 16, pk);
          if (c & 1) {
            // Keys 0-63 (then 64-127) of P are in TMEM: let P V use them.
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(bar(kBarPReady + 2 * b + (c >> 1)));
          }
        }
#undef S_
        const float2 sa = f2_split(fadd2(sum2[0], sum2[1]));
        l = l * alpha + (sa.x + sa.y);
      }
      if (!ok) break;
      // Epilogue: O / l and the LSE once the item's last P V is done.
      const int bl = (g - 1) & 1;
      if (!(ok = mbar_wait(bar(kBarPVDone + bl), ((g - 1) >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const float inv_l = 1.f / l;
      // O rows leave through shared memory, 64 columns at a time: each warp
      // packs its 32 rows into a 4 KB buffer (16-byte chunks swizzled by the
      // row) and reads it back so that eight lanes store one row's 128
      // contiguous bytes, four whole lines per store instruction.
      const int lane = threadIdx.x & 31;
      uint8_t *stg = smem + kOffStage + quarter * 4096;
      const int row_w = row - lane;   // this warp's first row
#pragma unroll 1
      for (int h = 0; h < D / 64; ++h) {
        uint32_t ov[2][32];
        tmem_ld32(o_tmem + 64 * h, ov[0]);
        tmem_ld32(o_tmem + 64 * h + 32, ov[1]);
        tmem_wait_ld(ov[0]);
        tmem_wait_ld(ov[1]);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t *c8 = &ov[k >> 2][(k & 3) * 8];
          uint4 v;
          v.x = pack2<F16>(__uint_as_float(c8[0]) * inv_l, __uint_as_float(c8[1]) * inv_l);
          v.y = pack2<F16>(__uint_as_float(c8[2]) * inv_l, __uint_as_float(c8[3]) * inv_l);
          v.z = pack2<F16>(__uint_as_float(c8[4]) * inv_l, __uint_as_float(c8[5]) * inv_l);
          v.w = pack2<F16>(__uint_as_float(c8[6]) * inv_l, __uint_as_float(c8[7]) * inv_l);
          *reinterpret_cast<uint4 *>(stg + lane * 128 + ((k ^ (lane & 7)) * 16)) = v;
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int rr = (lane >> 3) + 4 * k, ch = lane & 7;
          const uint4 v = *reinterpret_cast<const uint4 *>(stg + rr * 128 + ((ch ^ (rr & 7)) * 16));
          if (row_w + rr < N)
            *reinterpret_cast<uint4 *>(o + (static_cast<int64_t>(bh) * N + row_w + rr) * D +
                                       64 * h + ch * 8) = v;
        }
        __syncwarp();
      }
      // O has been read: the next item's first P V may overwrite it (it
      // waits for this warpgroup's first P of that item).
      tc_fence_before();
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
  if (threadIdx.x == 0) {
    if (misc->abort) atomicExch(dev_status, kDevTimeout);
    __threadfence();
    if (atomicAdd(sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      sched[0] = 0;
      sched[1] = 0;
      __threadfence();
    }
  }
}

int g_num_sms[64] = {};

template <bool F16>
cudaError_t launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, void *o,
                   float *lse, int BH, int N, float scale, int causal, int *sched,
                   int *dev_status, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (g_num_sms[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_num_sms[dev] = n;
  }
  e = cudaFuncSetAttribute(fwd_d256_kernel<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kAlloc);
  if (e != cudaSuccess) return e;
  const long long n_items = static_cast<long long>((N + BM - 1) / BM) * BH;
  const int grid = static_cast<int>(n_items < g_num_sms[dev] ? n_items : g_num_sms[dev]);
  // A programmatic dependent launch: the kernel waits with
  // griddepcontrol.wait after its set-up for the work before it.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_d256_kernel<F16>, tq, tk, tv, static_cast<uint16_t *>(o),
                            lse, N, BH, scale * 1.4426950408889634f, causal, sched, dev_status);
}

}  // namespace

cudaError_t launch_fwd_d256(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            void *o, float *lse, int BH, int N, float scale, int causal,
                            int *sched, int *dev_status, cudaStream_t stream, bool f16) {
  return f16 ? launch<true>(tq, tk, tv, o, lse, BH, N, scale, causal, sched, dev_status, stream)
             : launch<false>(tq, tk, tv, o, lse, BH, N, scale, causal, sched, dev_status, stream);
}

}  // namespace fattn
