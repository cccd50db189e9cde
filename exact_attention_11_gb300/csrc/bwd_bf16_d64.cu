// bwd_bf16_d64.cu -- the main backward kernel for head dimension 64: the
// recomputation scheme of "FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화
// 분석" (youngju.dev, section 7: P = exp(S - LSE), dV = P^T dO, dP = dO V^T,
// dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q), scheduled like the
// head-dimension-128 kernel (bwd_bf16_d128.cu) so that the tensor cores and
// the CUDA cores work at the same time.
//
// One CTA per (128-key block j, head) keeps K_j, V_j in shared memory and
// dV_j, dK_j (fp32) in TMEM.  Each 128-query step is split into two 64-query
// sub-tiles t = 0, 1, each owned by one group of four warps.  While group t
// turns S_t, dP_t into P_t, dS_t, the MMA warp works on the other sub-tile
// (the two groups take turns, as the forward kernel's two query tiles do).
// Per sub-tile (TMEM region R_t = [128t, 128t+128)):
//   S_t^T  = K_j Q_t^T  -> R_t[0,64)      dP_t^T = V_j dO_t^T -> R_t[64,128)
//   group t: P_t^T = exp2(S^T scale log2e - LSE2) and dS_t^T = P^T (dP^T - D)
//            as packed bf16 at R_t[0,32) and R_t[32,64); dS^T also to shared
//            memory (128-byte swizzle, keys as rows), one buffer per step
//            parity so that a step's dS stays readable while the next one is
//            written
//   dV_j += P_t^T dO_t,  dK_j += dS_t^T Q_t            (A operands from TMEM)
// and once both sub-tiles of step i are done, for the whole step:
//   dQ_i' = dS_i K_j   (M = 128 queries, N = 64, K = 128 keys; A = dS^T of
//                       both sub-tiles from shared memory)  -> DQ[i % 2]
// With a head dimension of 64 the M = d product of the d = 128 kernel would
// be an M = 64 MMA; taking dQ' per 128-query step keeps every MMA at M = 128
// and fits TMEM: R_0 | R_1 | dV | dK | DQ[0] | DQ[1] = 512 columns.
// During step i each group reads its 32 columns of dQ_{i-1}' out of TMEM
// (lanes = queries), stages them in shared memory and adds them to the fp32
// dQ accumulator with a TMA reduce.
// MMA order: per sub-tile dV_t, dK_t, then S_t, dP_t of the next step (R_t
// is free once dV_t and dK_t have read it: MMAs of one thread execute in
// issue order); after sub-tile 1, dQ_i'.  Q and dO arrive as 64-row halves
// through 4-slot rings, two steps ahead.
//
// The CTAs are persistent (one per SM) and take (key block, head) items from
// a device-wide counter, heaviest first, as the head-dimension-128 kernel
// does: every barrier keeps counting across items, the next item's Q, dO and
// K, V loads and first S, dP overlap the current item's dV, dK epilogue, and
// its first dV, dK products wait only for that epilogue's TMEM read-out.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "bwd_tile.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int D = 64;
constexpr int BM = 128;      // keys per CTA
constexpr int BQ = 128;      // queries per step
constexpr int BH_ = 64;      // queries per sub-tile
constexpr int kSlots = 4;    // Q / dO half-tile ring depth
constexpr int kThreads = 384;
constexpr uint32_t kRegsLoad = 104, kRegsGroup = 200;
static_assert(kRegsLoad + 2 * kRegsGroup == 3 * 168,
              "the warpgroup register split must use exactly the launch budget");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDV = 256, kColDK = 320, kColDQ = 384;
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory (offsets from a 1024-byte aligned base; the kernel checks
// that the dynamic shared memory it is given starts on such a boundary).
constexpr int kTile = BM * D * 2;          // 16 KB: K or V, 128 rows x 128 bytes
constexpr int kHalf = BH_ * D * 2;         // 8 KB: 64 rows of Q or dO
constexpr int kDSBytes = BM * BH_ * 2;     // 16 KB: dS^T of a sub-tile (128 keys x 64 queries)
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTile;
constexpr int kOffQ = kOffV + kTile;                 // kSlots halves
constexpr int kOffDO = kOffQ + kSlots * kHalf;       // kSlots halves
constexpr int kOffDS = kOffDO + kSlots * kHalf;      // [step parity][sub-tile] x 16 KB
constexpr int kOffStage = kOffDS + 4 * kDSBytes;     // 8 group warps x 4 KB of dQ' staging
constexpr int kOffVec = kOffStage + 8 * 4096;        // kSlots x [LSE2 64 | D 64] f32
constexpr int kVecBytes = 2 * BH_ * 4;
constexpr int kOffBar = kOffVec + kSlots * kVecBytes;
constexpr int kSmemBytes = kOffBar + 512;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

enum : int {
  kBarKV = 0,
  kBarQFull = 1,        // + slot
  kBarQEmpty = 5,       // + slot
  kBarDOFull = 9,       // + slot
  kBarDOEmpty = 13,     // + slot
  kBarSFull = 17,       // + t
  kBarPReady = 19,      // + t, 4 warps
  kBarDQFull = 21,      // + step parity
  kBarDQFree = 23,      // + step parity, 8 warps: dQ' read out of TMEM
  kBarKVDone = 25,      // every MMA of the item is complete (K, V free; dV, dK final)
  kBarDrain = 26,
  kBarEpiDone = 27,     // 8 warps: the item's dV, dK have been read out of TMEM
  kBarItemFull = 28,    // + ring slot (2)
  kBarItemEmpty = 30,   // + ring slot (2)
  kNumBars = 32
};
// Arrivals that free an item-ring slot: the MMA thread and the 8 group warps.
constexpr int kItemConsumers = 1 + 8;

struct Misc {
  uint32_t tmem_base;
  int abort;
  int item[2];
};
static_assert(kNumBars * 8 + sizeof(Misc) <= 512, "barrier area");

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t ph, volatile int *abort_flag) {
  return __all_sync(~0u, mbar_wait(bar, ph, abort_flag));
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t ph) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, ph) && globaltimer_ns() - t0 < kWaitLimitNs) {
  }
}

// Status latched when the dynamic shared memory does not start on a 1024-byte
// boundary (the layout above assumes it; the kernel then does nothing).
constexpr int kDevBadSmemBase = -2;

// An item: key block jb of head bh (items heaviest first: under the causal
// mask key block 0 is visited by every query block).
struct BwdItem {
  int jb, bh, k0, i_first, n_steps, n_halves;
  __device__ void decode(int w, int BH, int n_qb, int causal) {
    jb = w / BH;
    bh = w - jb * BH;
    k0 = jb * BM;
    i_first = causal ? jb : 0;
    n_steps = n_qb - i_first;
    n_halves = 2 * n_steps;
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    bwd_pipe64_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_dq, const float *__restrict__ vecs,
                      __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv, int N,
                      int BH, float scale, int causal, int *__restrict__ sched, int fault_cta,
                      int *__restrict__ dev_status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s_base = smem_u32(smem);
  if ((s_base & 1023u) != 0) {
    if (threadIdx.x == 0) atomicExch(dev_status, kDevBadSmemBase);
    return;
  }
  const uint32_t bars = s_base + kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  Misc *misc = reinterpret_cast<Misc *>(smem + kOffBar + 8 * kNumBars);
  volatile int *abort_flag = &misc->abort;
  const int n_qb = (N + BQ - 1) / BQ;
  const int n_items = n_qb * BH;

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarKV), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 1);
      mbar_init(bar(kBarDOFull + s), 1);
      mbar_init(bar(kBarDOEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPReady + t), 4);
      mbar_init(bar(kBarDQFull + t), 1);
      mbar_init(bar(kBarDQFree + t), 8);
      mbar_init(bar(kBarItemFull + t), 1);
      mbar_init(bar(kBarItemEmpty + t), kItemConsumers);
    }
    mbar_init(bar(kBarKVDone), 1);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarEpiDone), 8);
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
  // A programmatic dependent of the preparation kernel: its set-up above
  // overlaps that kernel's tail; no global memory is touched before this wait.
  // The dQ kernel may be scheduled once every block of this one is past it.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Consumer side of the item ring: waits for entry k and frees it (one
  // arrival per warp, or the lone MMA thread).
  auto fetch_item = [&](int k, int &w, bool whole_warp) -> bool {
    const int slot = k & 1;
    if (!mbar_wait(bar(kBarItemFull + slot), (k >> 1) & 1, abort_flag)) return false;
    w = *reinterpret_cast<volatile int *>(&misc->item[slot]);
    if (whole_warp) __syncwarp();
    if (!whole_warp || (threadIdx.x & 31) == 0) mbar_arrive(bar(kBarItemEmpty + slot));
    return true;
  };

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLoad));
    if (warp == 0 && elect_one()) {
      // ---------------------------------------------------------- TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      int nq = 0, ndo = 0, nkv = 0;   // halves (and K/V pairs) issued so far
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int islot = k & 1;
        if (!(ok = mbar_wait(bar(kBarItemEmpty + islot), ((k >> 1) & 1) ^ 1, abort_flag))) break;
        const int w = atomicAdd(sched, 1);
        misc->item[islot] = w;
        mbar_arrive(bar(kBarItemFull + islot));
        if (w >= n_items) break;
        BwdItem it;
        it.decode(w, BH, n_qb, causal);
        const int h_base = nq;
        // Q / dO half h of the item (with its [LSE2 | D] vectors on QFull).
        auto load_half = [&](int h) -> bool {
          const int g = h_base + h, slot = g % kSlots, use = g / kSlots;
          const int qb = it.i_first + (h >> 1);
          const int qrow = qb * BQ + (h & 1) * BH_;
          if (!mbar_wait(bar(kBarQEmpty + slot), (use & 1) ^ 1, abort_flag)) return false;
          mbar_arrive_expect_tx(bar(kBarQFull + slot), kHalf + kVecBytes);
          tma_load_3d(s_base + kOffQ + slot * kHalf, &tm_q, 0, qrow, it.bh, bar(kBarQFull + slot));
          const float *vsrc =
              vecs + (static_cast<int64_t>(it.bh) * n_qb + qb) * (2 * BQ) + (h & 1) * BH_;
          bulk_load(s_base + kOffVec + slot * kVecBytes, vsrc, BH_ * 4, bar(kBarQFull + slot));
          bulk_load(s_base + kOffVec + slot * kVecBytes + BH_ * 4, vsrc + BQ, BH_ * 4,
                    bar(kBarQFull + slot));
          nq = g + 1;
          if (!mbar_wait(bar(kBarDOEmpty + slot), (use & 1) ^ 1, abort_flag)) return false;
          mbar_arrive_expect_tx(bar(kBarDOFull + slot), kHalf);
          tma_load_3d(s_base + kOffDO + slot * kHalf, &tm_do, 0, qrow, it.bh,
                      bar(kBarDOFull + slot));
          ndo = g + 1;
          return true;
        };
        // The first two halves as soon as ring slots free up; K and V once
        // the previous item's last MMA has read them.
        for (int h = 0; h < 2 && h < it.n_halves && ok; ++h) ok = load_half(h);
        if (!ok) break;
        if (static_cast<int>(blockIdx.x) == fault_cta) {
          // Failure-path test: stop here, as if the K and V copies were lost;
          // the MMA warp's bounded wait for them runs out.
          ok = false;
          break;
        }
        if (k > 0 && !(ok = mbar_wait(bar(kBarKVDone), (k - 1) & 1, abort_flag))) break;
        mbar_arrive_expect_tx(bar(kBarKV), 2 * kTile);
        tma_load_3d(s_base + kOffK, &tm_k, 0, it.k0, it.bh, bar(kBarKV));
        tma_load_3d(s_base + kOffV, &tm_v, 0, it.k0, it.bh, bar(kBarKV));
        nkv = k + 1;
        for (int h = 2; h < it.n_halves && ok; ++h) ok = load_half(h);
      }
      if (!ok) {
        if (nkv > 0) drain_wait(bar(kBarKV), (nkv - 1) & 1);
        for (int g = (nq > kSlots ? nq - kSlots : 0); g < nq; ++g)
          drain_wait(bar(kBarQFull + g % kSlots), (g / kSlots) & 1);
        for (int g = (ndo > kSlots ? ndo - kSlots : 0); g < ndo; ++g)
          drain_wait(bar(kBarDOFull + g % kSlots), (g / kSlots) & 1);
      }
    } else if (warp == 1 && elect_one()) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BH_, false);       // S^T, dP^T
      constexpr uint32_t idesc_g = idesc_bf16_f32(BM, D, true);          // dV, dK
      constexpr uint32_t idesc_q = idesc_bf16_f32(BQ, D, true, true);    // dQ'
      const uint32_t k_kmaj = sdesc_lo(s_base + kOffK, 16);
      const uint32_t v_kmaj = sdesc_lo(s_base + kOffV, 16);
      const uint32_t k_mn = sdesc_lo(s_base + kOffK, kTile);    // K as the N = d operand
      const uint32_t q_kmaj = sdesc_lo(s_base + kOffQ, 16);
      const uint32_t q_mn = sdesc_lo(s_base + kOffQ, kHalf);
      const uint32_t do_kmaj = sdesc_lo(s_base + kOffDO, 16);
      const uint32_t do_mn = sdesc_lo(s_base + kOffDO, kHalf);
      // dS of a step as the M = 128 queries operand: the two sub-tiles' 64
      // query columns are 16 KB apart.
      const uint32_t ds_mn = sdesc_lo(s_base + kOffDS, kDSBytes);
      // S_t^T = K Q_t^T and dP_t^T = V dO_t^T of ring half g into R_{h & 1}.
      auto issue_sdp = [&](int h, int g) {
        const uint32_t R = tmem + 128u * (h & 1);
        const uint32_t so = static_cast<uint32_t>((g % kSlots) * kHalf) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o32 = static_cast<uint32_t>(kk * 32) >> 4;
          mma_ss_lo(R, k_kmaj + o32, q_kmaj + so + o32, idesc_s, kk > 0 ? 1u : 0u);
          mma_ss_lo(R + 64, v_kmaj + o32, do_kmaj + so + o32, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(kBarSFull + (h & 1)));
      };
      bool ok = true;
      int g0 = 0;       // ring halves of the earlier items
      int steps = 0;    // steps of the earlier items
      for (int k = 0; ok; ++k) {
        int w;
        if (!(ok = fetch_item(k, w, false)) || w >= n_items) break;
        BwdItem it;
        it.decode(w, BH, n_qb, causal);
        if (!(ok = mbar_wait(bar(kBarKV), k & 1, abort_flag))) break;
        // The item's first S_t, dP_t (R_t was released by the previous item's
        // last dV_t, dK_t, which execute before them).
        for (int h = 0; h < 2 && h < it.n_halves && ok; ++h) {
          const int g = g0 + h;
          if (!(ok = mbar_wait(bar(kBarQFull + g % kSlots), (g / kSlots) & 1, abort_flag))) break;
          if (!(ok = mbar_wait(bar(kBarDOFull + g % kSlots), (g / kSlots) & 1, abort_flag))) break;
          tc_fence_after();
          issue_sdp(h, g);
        }
        for (int h = 0; h < it.n_halves && ok; ++h) {
          const int t = h & 1, st = steps + (h >> 1), g = g0 + h, slot = g % kSlots;
          const uint32_t R = tmem + 128u * t;
          if (!(ok = mbar_wait(bar(kBarPReady + t), st & 1, abort_flag))) break;
          tc_fence_after();
          // The previous item's dV, dK must have left TMEM before the first
          // product of this one overwrites them.
          if (h == 0 && k > 0) {
            if (!(ok = mbar_wait(bar(kBarEpiDone), (k - 1) & 1, abort_flag))) break;
            tc_fence_after();
          }
          // dV += P_t^T dO_t, dK += dS_t^T Q_t (A operands from TMEM); K = 64
          // queries.
          const uint32_t so = static_cast<uint32_t>(slot * kHalf) >> 4;
#pragma unroll
          for (int kk = 0; kk < BH_ / 16; ++kk) {
            const uint32_t ob = so + (static_cast<uint32_t>(kk * 2048) >> 4);
            const uint32_t acc = (h > 0 || kk > 0) ? 1u : 0u;
            mma_ts_lo(tmem + kColDV, R + kk * 8, do_mn + ob, idesc_g, acc);
            mma_ts_lo(tmem + kColDK, R + 32 + kk * 8, q_mn + ob, idesc_g, acc);
          }
          mma_commit(bar(kBarQEmpty + slot));
          mma_commit(bar(kBarDOEmpty + slot));
          // R_t is free once dV_t and dK_t have read it (in-order execution):
          // the next step's S_t and dP_t go next.
          const int h2 = h + 2;
          if (h2 < it.n_halves) {
            const int g2 = g0 + h2;
            if (!(ok = mbar_wait(bar(kBarQFull + g2 % kSlots), (g2 / kSlots) & 1, abort_flag))) break;
            if (!(ok = mbar_wait(bar(kBarDOFull + g2 % kSlots), (g2 / kSlots) & 1, abort_flag))) break;
            tc_fence_after();
            issue_sdp(h2, g2);
          }
          if (t == 1) {
            // Both sub-tiles of step st are done: dQ_st' = dS_st K, M = 128
            // queries, N = 64, K = 128 keys, into DQ[st % 2] once step
            // st - 2's dQ' has been read out of it.
            const int p = st & 1;
            if (st >= 2 && !(ok = mbar_wait(bar(kBarDQFree + p), ((st >> 1) - 1) & 1, abort_flag)))
              break;
            tc_fence_after();
            const uint32_t dso = static_cast<uint32_t>(p * 2 * kDSBytes) >> 4;
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk) {
              const uint32_t off = static_cast<uint32_t>(kk * 2048) >> 4;
              mma_ss_lo(tmem + kColDQ + 64u * p, ds_mn + dso + off, k_mn + off, idesc_q,
                        kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(kBarDQFull + p));
          }
        }
        if (ok) mma_commit(bar(kBarKVDone));
        g0 += it.n_halves;
        steps += it.n_steps;
      }
      mma_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsGroup));
    // ----------------- groups: P, dS, dQ' read-out and reduce, epilogue
    const int t = (warp - 4) >> 2;            // sub-tile of this group
    const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
    const int lane = threadIdx.x & 31;
    const int gw = warp - 4;                  // 0..7
    const int r = quarter * 32 + lane;        // key row of S^T, dP^T; query row of dQ'
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t R = tmem + lane_off + 128u * t;
    const uint64_t c2 = f2(scale * kLog2e, scale * kLog2e);
    // This warp's 4 KB staging tile: its dQ' boxes (32 queries x 32 fp32,
    // 128-byte rows with the 128-byte swizzle, the box of the accumulator's
    // tensor map), and at the end of an item its dV / dK rows.
    uint8_t *stage = smem + kOffStage + gw * 4096;
    const uint32_t stage_u32 = s_base + kOffStage + gw * 4096;
    bool ok = true;
    int steps = 0, g0 = 0;
    for (int k = 0; ok; ++k) {
      int w;
      if (!(ok = fetch_item(k, w, true)) || w >= n_items) break;
      BwdItem it;
      it.decode(w, BH, n_qb, causal);
      const int key = it.k0 + r;
      // Step i of the item (global step steps + i): its dQ' rows (lanes =
      // queries), columns 32 t .. 32 t + 31 of d: TMEM -> registers ->
      // staging tile -> TMA reduce-add.
      auto readout = [&](int i) -> bool {
        const int s = steps + i, p = s & 1;
        if (!wait_warp(bar(kBarDQFull + p), (s >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        uint32_t gq[32];
        tmem_ld32(tmem + lane_off + kColDQ + 64u * p + 32u * t, gq);
        tmem_wait_ld(gq);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarDQFree + p));
        // The previous reduce from this tile has finished reading it.
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4 v4;
          v4.x = gq[4 * j + 0];
          v4.y = gq[4 * j + 1];
          v4.z = gq[4 * j + 2];
          v4.w = gq[4 * j + 3];
          *reinterpret_cast<uint4 *>(stage + lane * 128 + ((j ^ (lane & 7)) << 4)) = v4;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dq, stage_u32, 32 * t, (it.i_first + i) * BQ + quarter * 32,
                            it.bh);
          bulk_commit();
        }
        return true;
      };
      for (int i = 0; i < it.n_steps && ok; ++i) {
        const int h = 2 * i + t, st = steps + i, g = g0 + h, slot = g % kSlots;
        const int q0 = (it.i_first + i) * BQ + t * BH_;   // first query of the sub-tile
        if (!(ok = wait_warp(bar(kBarSFull + t), st & 1, abort_flag))) break;
        // [LSE2 | D] of the sub-tile came with Q_t on QFull, which S_t needed.
        if (!(ok = wait_warp(bar(kBarQFull + slot), (g / kSlots) & 1, abort_flag))) break;
        tc_fence_after();
        const float *vec = reinterpret_cast<const float *>(smem + kOffVec + slot * kVecBytes);
        // Step st's dS buffer was last read by dQ_{st-2}', which the read-out
        // of step st - 1 (or the previous item's last read-out) waited for.
        uint8_t *ds_buf = smem + kOffDS + ((st & 1) * 2 + t) * kDSBytes;
        // Masking is needed only where a key of this warp is past N or, on the
        // diagonal block, later than a query (warp-uniform).
        const bool diag = causal && (q0 < it.k0 + BM) && (q0 + BH_ > it.k0);
        const bool masked = diag || (it.k0 + quarter * 32 + 31 >= N);
        if (masked)
          bwd_tile::chunks<true>(R, vec, ds_buf, r, key, q0, N, diag, c2);
        else
          bwd_tile::chunks<false>(R, vec, ds_buf, r, key, q0, N, diag, c2);
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPReady + t));
        if (i >= 1) ok = readout(i - 1);
      }
      if (ok) ok = readout(it.n_steps - 1);
      if (lane == 0) bulk_wait_all();
      __syncwarp();
      if (!ok) break;

      // Epilogue: group 0 writes dV_j, group 1 dK_j = scale * (dS^T Q), as
      // bf16 rows (rows >= N are not stored), through this warp's staging
      // tile (its reduces have all completed): the warp packs its 32 rows
      // into 4 KB (16-byte chunks swizzled by the row) and reads them back so
      // that eight lanes store one row's 128 contiguous bytes.
      if (!(ok = wait_warp(bar(kBarKVDone), k & 1, abort_flag))) break;
      tc_fence_after();
      __nv_bfloat16 *base = (t ? dk : dv) + static_cast<int64_t>(it.bh) * N * D;
      const float mul = t ? scale : 1.f;
      const uint32_t col = t ? kColDK : kColDV;
      const int key_w = key - lane;   // this warp's first key row
      uint32_t v[2][32];
      tmem_ld32(tmem + lane_off + col, v[0]);
      tmem_ld32(tmem + lane_off + col + 32, v[1]);
      tmem_wait_ld(v[0]);
      tmem_wait_ld(v[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarEpiDone));
#pragma unroll
      for (int kq = 0; kq < 8; ++kq) {
        const uint32_t *c8 = &v[kq >> 2][(kq & 3) * 8];
        uint4 x;
        x.x = pack_bf16x2(__uint_as_float(c8[0]) * mul, __uint_as_float(c8[1]) * mul);
        x.y = pack_bf16x2(__uint_as_float(c8[2]) * mul, __uint_as_float(c8[3]) * mul);
        x.z = pack_bf16x2(__uint_as_float(c8[4]) * mul, __uint_as_float(c8[5]) * mul);
        x.w = pack_bf16x2(__uint_as_float(c8[6]) * mul, __uint_as_float(c8[7]) * mul);
        *reinterpret_cast<uint4 *>(stage + lane * 128 + ((kq ^ (lane & 7)) * 16)) = x;
      }
      __syncwarp();
#pragma unroll
      for (int kq = 0; kq < 8; ++kq) {
        const int rr = (lane >> 3) + 4 * kq, ch = lane & 7;
        const uint4 x = *reinterpret_cast<const uint4 *>(stage + rr * 128 + ((ch ^ (rr & 7)) * 16));
        if (key_w + rr < N)
          *reinterpret_cast<uint4 *>(base + static_cast<int64_t>(key_w + rr) * D + ch * 8) = x;
      }
      // The next read-out writes dQ' boxes over the staging tile.
      __syncwarp();
      g0 += it.n_halves;
      steps += it.n_steps;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) {
    if (misc->abort) atomicExch(dev_status, kDevTimeout);
    // The last CTA to finish puts the launch's work counters back to zero.
    __threadfence();
    if (atomicAdd(sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      sched[0] = 0;
      sched[1] = 0;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t launch_bwd_main_d64(const CUtensorMap &tq64, const CUtensorMap &tk,
                                const CUtensorMap &tv, const CUtensorMap &tdo64,
                                const CUtensorMap &tdq, const float *vecs, void *dk, void *dv,
                                int BH, int N, float scale, int causal, int *sched,
                                int fault_cta, int *dev_status, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(bwd_pipe64_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, n_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int n_qb = (N + BQ - 1) / BQ;
  const long long n_items = static_cast<long long>(n_qb) * BH;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_items < n_sm ? n_items : n_sm));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bwd_pipe64_kernel, tq64, tk, tv, tdo64, tdq, vecs,
                            reinterpret_cast<__nv_bfloat16 *>(dk),
                            reinterpret_cast<__nv_bfloat16 *>(dv), N, BH, scale, causal, sched,
                            fault_cta, dev_status);
}

}  // namespace fattn
