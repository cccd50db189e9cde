// bwd_bf16_d128.cu -- the main backward kernel for head dimension 128: the
// same arithmetic as bwd_main_kernel in bwd_bf16.cu (recomputation scheme of
// "FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화 분석", youngju.dev,
// section 7: P = exp(S - LSE), dV = P^T dO, dP = dO V^T, dS = P (dP - D),
// dQ = scale dS K, dK = scale dS^T Q), scheduled so that the tensor cores and
// the CUDA cores work at the same time.
//
// One CTA per (128-key block j, head) keeps K_j, V_j in shared memory and
// dV_j, dK_j (fp32) in TMEM.  Each 128-query step is split into two 64-query
// sub-tiles t = 0, 1, each owned by one group of four warps.  While group t
// turns S_t, dP_t into P_t, dS_t, the MMA warp works on the other sub-tile,
// so the two groups take turns ("ping-pong"), as the forward kernel's two
// query tiles do.  Per sub-tile (TMEM region R_t = [128t, 128t+128)):
//   S_t^T  = K_j Q_t^T  -> R_t[0,64)      dP_t^T = V_j dO_t^T -> R_t[64,128)
//   group t: P_t^T = exp2(S^T scale log2e - LSE2) and dS_t^T = P^T (dP^T - D)
//            as packed bf16 at R_t[0,32) and R_t[32,64); dS^T also to shared
//            memory (128-byte swizzle, keys as rows)
//   dQ_t'^T = K_j^T dS_t^T -> R_t[64,128) (lanes = d, columns = queries)
//   dV_j += P_t^T dO_t,  dK_j += dS_t^T Q_t            (A operands from TMEM)
//   group t reads dQ_t'^T out of TMEM and adds it to the fp32 dQ accumulator
//   with TMA reduces: each warp stages its 32 d x 64 queries as two
//   [query][d] boxes in its own quarter of the dS^T buffer, which dQ_t'^T has
//   finished reading and the group only writes again in its next element
//   step.
// The kernel is bound by shared-memory bandwidth (MMA operands, TMA writes,
// dS stores), so operands come from TMEM wherever the TMEM budget allows.
// MMA order per sub-tile: dQ'_t, dV_t, dK_t, then S_t, dP_t of the next step
// (after group t has released R_t), then the other sub-tile.  Q and dO
// arrive as 64-row halves through 4-slot rings, two steps ahead.
//
// The CTAs are persistent (one per SM): the producer claims (key block,
// head) items from a device-wide counter, heaviest first, and hands them to
// the other roles through a two-entry ring in shared memory.  Every barrier
// keeps counting across items.  At an item boundary the producer loads the
// next item's first Q and dO halves as soon as ring slots free up and its K
// and V once the last MMA of the current item has read theirs; the MMA warp
// starts the next item's first S and dP while the groups write the current
// item's dV and dK, and its first dV, dK products wait only for the groups
// to have read those accumulators out of TMEM.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "bwd_tile.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int D = 128;
constexpr int BM = 128;      // keys per CTA
constexpr int BQ = 128;      // queries per step
constexpr int BH_ = 64;      // queries per sub-tile
constexpr int kSlots = 4;    // Q / dO half-tile ring depth
constexpr int kThreads = 384;
constexpr uint32_t kRegsLoad = 104, kRegsGroup = 200;
static_assert(kRegsLoad + 2 * kRegsGroup == 3 * 168,
              "the warpgroup register split must use exactly the launch budget");
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory (offsets from a 1024-byte aligned base; the kernel checks
// that the dynamic shared memory it is given starts on such a boundary).
constexpr int kTile = BM * D * 2;          // 32 KB: K or V
constexpr int kHalf = BH_ * D * 2;         // 16 KB: a 64-row half of Q or dO
constexpr int kHalfBox = BH_ * 128;        // 8 KB: 64 rows x 128 bytes (64 of d)
constexpr int kKeyBox = BM * 128;          // 16 KB: 128 rows x 128 bytes
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTile;
constexpr int kOffQ = kOffV + kTile;                 // kSlots halves
constexpr int kOffDO = kOffQ + kSlots * kHalf;       // kSlots halves
constexpr int kOffDS = kOffDO + kSlots * kHalf;      // 2 x 16 KB (per sub-tile)
constexpr int kDSBytes = BM * BH_ * 2;               // 16 KB
constexpr int kOffVec = kOffDS + 2 * kDSBytes;       // kSlots x [LSE2 64 | D 64] f32
constexpr int kVecBytes = 2 * BH_ * 4;               // 512 B
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
  kBarDQFull = 21,      // + t
  kBarTmemFree = 23,    // + t, 4 warps: dQ'_t read out of TMEM
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
    bwd_pipe_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq,
                    const float *__restrict__ vecs,
                    __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv, int N, int BH,
                    float scale, int causal, int *__restrict__ sched, int fault_cta,
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
      mbar_init(bar(kBarTmemFree + t), 4);
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
          for (int b = 0; b < 2; ++b)
            tma_load_3d(s_base + kOffQ + slot * kHalf + b * kHalfBox, &tm_q, b * 64, qrow, it.bh,
                        bar(kBarQFull + slot));
          const float *vsrc =
              vecs + (static_cast<int64_t>(it.bh) * n_qb + qb) * (2 * BQ) + (h & 1) * BH_;
          bulk_load(s_base + kOffVec + slot * kVecBytes, vsrc, BH_ * 4, bar(kBarQFull + slot));
          bulk_load(s_base + kOffVec + slot * kVecBytes + BH_ * 4, vsrc + BQ, BH_ * 4,
                    bar(kBarQFull + slot));
          nq = g + 1;
          if (!mbar_wait(bar(kBarDOEmpty + slot), (use & 1) ^ 1, abort_flag)) return false;
          mbar_arrive_expect_tx(bar(kBarDOFull + slot), kHalf);
          for (int b = 0; b < 2; ++b)
            tma_load_3d(s_base + kOffDO + slot * kHalf + b * kHalfBox, &tm_do, b * 64, qrow, it.bh,
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
        for (int b = 0; b < 2; ++b) {
          tma_load_3d(s_base + kOffK + b * kKeyBox, &tm_k, b * 64, it.k0, it.bh, bar(kBarKV));
          tma_load_3d(s_base + kOffV + b * kKeyBox, &tm_v, b * 64, it.k0, it.bh, bar(kBarKV));
        }
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
      // Fully unrolled issue with 32-bit descriptor words: a rolled loop
      // costs the issuing thread about 60 cycles per MMA, more than an
      // M = 128, N = 64 MMA takes on the tensor core.
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BH_, false);        // S^T, dP^T
      constexpr uint32_t idesc_q = idesc_bf16_f32(D, BH_, true, true);    // dQ'^T
      constexpr uint32_t idesc_g = idesc_bf16_f32(BM, D, true);           // dV, dK
      const uint32_t k_kmaj = sdesc_lo(s_base + kOffK, 16);
      const uint32_t v_kmaj = sdesc_lo(s_base + kOffV, 16);
      const uint32_t k_mn = sdesc_lo(s_base + kOffK, kKeyBox);   // K^T, M = d
      const uint32_t q_kmaj = sdesc_lo(s_base + kOffQ, 16);
      const uint32_t q_mn = sdesc_lo(s_base + kOffQ, kHalfBox);  // N = d
      const uint32_t do_kmaj = sdesc_lo(s_base + kOffDO, 16);
      const uint32_t do_mn = sdesc_lo(s_base + kOffDO, kHalfBox);
      const uint32_t ds_mn = sdesc_lo(s_base + kOffDS, kDSBytes); // dS^T as B
      // S_t^T = K Q_t^T and dP_t^T = V dO_t^T of ring half g into R_{h & 1}.
      auto issue_sdp = [&](int h, int g) {
        const uint32_t R = tmem + 128u * (h & 1);
        const uint32_t so = static_cast<uint32_t>((g % kSlots) * kHalf) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ok_ = static_cast<uint32_t>((kk >> 2) * kKeyBox + (kk & 3) * 32) >> 4;
          const uint32_t oh = static_cast<uint32_t>((kk >> 2) * kHalfBox + (kk & 3) * 32) >> 4;
          mma_ss_lo(R, k_kmaj + ok_, q_kmaj + so + oh, idesc_s, kk > 0 ? 1u : 0u);
          mma_ss_lo(R + 64, v_kmaj + ok_, do_kmaj + so + oh, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(kBarSFull + (h & 1)));
      };
      bool ok = true;
      int g0 = 0;       // ring halves of the earlier items
      int steps = 0;    // steps (per sub-tile) of the earlier items
      for (int k = 0; ok; ++k) {
        int w;
        if (!(ok = fetch_item(k, w, false)) || w >= n_items) break;
        BwdItem it;
        it.decode(w, BH, n_qb, causal);
        if (!(ok = mbar_wait(bar(kBarKV), k & 1, abort_flag))) break;
        // The item's first S_t, dP_t: R_t must have been read out (the dQ'_t
        // of the previous item's last step).
        for (int h = 0; h < 2 && h < it.n_halves && ok; ++h) {
          const int g = g0 + h;
          if (steps > 0 && !(ok = mbar_wait(bar(kBarTmemFree + h), (steps - 1) & 1, abort_flag)))
            break;
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
          // dQ_t'^T = K^T dS_t^T: M = d, N = 64 queries, K = 128 keys.
          const uint32_t dso = static_cast<uint32_t>(t * kDSBytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk) {
            const uint32_t off = static_cast<uint32_t>(kk * 2048) >> 4;
            mma_ss_lo(R + 64, k_mn + off, ds_mn + dso + off, idesc_q, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(kBarDQFull + t));
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
            mma_ts_lo(tmem + 256, R + kk * 8, do_mn + ob, idesc_g, acc);
            mma_ts_lo(tmem + 256 + D, R + 32 + kk * 8, q_mn + ob, idesc_g, acc);
          }
          mma_commit(bar(kBarQEmpty + slot));
          mma_commit(bar(kBarDOEmpty + slot));
          const int h2 = h + 2;
          if (h2 < it.n_halves) {
            const int g2 = g0 + h2;
            if (!(ok = mbar_wait(bar(kBarTmemFree + t), st & 1, abort_flag))) break;
            if (!(ok = mbar_wait(bar(kBarQFull + g2 % kSlots), (g2 / kSlots) & 1, abort_flag))) break;
            if (!(ok = mbar_wait(bar(kBarDOFull + g2 % kSlots), (g2 / kSlots) & 1, abort_flag))) break;
            tc_fence_after();
            issue_sdp(h2, g2);
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
    // ------------------------- groups: P, dS, dQ' read-out and reduce, epilogue
    const int t = (warp - 4) >> 2;            // sub-tile of this group
    const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
    const int lane = threadIdx.x & 31;
    const int r = quarter * 32 + lane;        // key row of S^T, dP^T; d row of dQ'^T
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t R = tmem + lane_off + 128u * t;
    const uint64_t c2 = f2(scale * kLog2e, scale * kLog2e);
    uint8_t *ds_buf = smem + kOffDS + t * kDSBytes;
    // This warp's quarter of the dS^T buffer: staging of its dQ' boxes and
    // of its dV / dK rows.
    uint8_t *stg = ds_buf + quarter * 4096;
    const uint32_t stg_u32 = s_base + kOffDS + t * kDSBytes + quarter * 4096;
    bool ok = true;
    int g0 = 0, steps = 0;
    for (int k = 0; ok; ++k) {
      int w;
      if (!(ok = fetch_item(k, w, true)) || w >= n_items) break;
      BwdItem it;
      it.decode(w, BH, n_qb, causal);
      const int key = it.k0 + r;
      for (int i = 0; i < it.n_steps && ok; ++i) {
        const int h = 2 * i + t, st = steps + i, g = g0 + h, slot = g % kSlots;
        const int q0 = (it.i_first + i) * BQ + t * BH_;   // first query of the sub-tile
        if (!(ok = wait_warp(bar(kBarSFull + t), st & 1, abort_flag))) break;
        // [LSE2 | D] of the sub-tile came with Q_t on QFull, which S_t needed.
        if (!(ok = wait_warp(bar(kBarQFull + slot), (g / kSlots) & 1, abort_flag))) break;
        tc_fence_after();
        const float *vec = reinterpret_cast<const float *>(smem + kOffVec + slot * kVecBytes);
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

        // dQ_t'^T row d = r: 64 query columns, read out, then R_t is released.
        if (!(ok = wait_warp(bar(kBarDQFull + t), st & 1, abort_flag))) break;
        tc_fence_after();
        uint32_t g0v[32], g1v[32];
        tmem_ld32(R + 64, g0v);
        tmem_ld32(R + 96, g1v);
        tmem_wait_ld(g0v);
        tmem_wait_ld(g1v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarTmemFree + t));
        // Add into the row-major accumulator with TMA reduces: this warp's
        // quarter of the dS^T buffer (its own key rows, free now that dQ'^T,
        // which read it, is complete) stages one 32-query x 32-d box at a time
        // as [query][d] fp32 rows with the 128-byte swizzle.
#pragma unroll
        for (int bx = 0; bx < 2; ++bx) {
          if (bx == 1) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
#pragma unroll
          for (int qq = 0; qq < 32; ++qq)
            *reinterpret_cast<uint32_t *>(stg + qq * 128 + ((((lane >> 2) ^ (qq & 7))) << 4) +
                                          (lane & 3) * 4) = bx ? g1v[qq] : g0v[qq];
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&tm_dq, stg_u32, 32 * quarter, q0 + 32 * bx, it.bh);
            bulk_commit();
          }
        }
        // The next element phase writes dS^T rows over the staging area.
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
      }
      if (!ok) break;

      // Epilogue: group 0 writes dV_j, group 1 dK_j = scale * (dS^T Q), as
      // bf16 rows (rows >= N are not stored).  Both 64-column halves are
      // read out of TMEM first, so the MMA warp may start the next item's
      // products into them while the rows are stored.
      if (!(ok = wait_warp(bar(kBarKVDone), k & 1, abort_flag))) break;
      tc_fence_after();
      __nv_bfloat16 *base = (t ? dk : dv) + static_cast<int64_t>(it.bh) * N * D;
      const float mul = t ? scale : 1.f;
      const uint32_t col = t ? 256u + D : 256u;
      uint32_t v[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + col + 32 * c, v[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_wait_ld(v[c]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarEpiDone));
      // The rows leave through this warp's staging quarter, 64 columns at a
      // time: the warp packs its 32 rows into 4 KB (16-byte chunks swizzled by
      // the row) and reads them back so that eight lanes store one row's 128
      // contiguous bytes.
      const int key_w = key - lane;   // this warp's first key row
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh) {
#pragma unroll
        for (int kq = 0; kq < 8; ++kq) {
          const uint32_t *c8 = &v[2 * hh + (kq >> 2)][(kq & 3) * 8];
          uint4 x;
          x.x = pack_bf16x2(__uint_as_float(c8[0]) * mul, __uint_as_float(c8[1]) * mul);
          x.y = pack_bf16x2(__uint_as_float(c8[2]) * mul, __uint_as_float(c8[3]) * mul);
          x.z = pack_bf16x2(__uint_as_float(c8[4]) * mul, __uint_as_float(c8[5]) * mul);
          x.w = pack_bf16x2(__uint_as_float(c8[6]) * mul, __uint_as_float(c8[7]) * mul);
          *reinterpret_cast<uint4 *>(stg + lane * 128 + ((kq ^ (lane & 7)) * 16)) = x;
        }
        __syncwarp();
#pragma unroll
        for (int kq = 0; kq < 8; ++kq) {
          const int rr = (lane >> 3) + 4 * kq, ch = lane & 7;
          const uint4 x = *reinterpret_cast<const uint4 *>(stg + rr * 128 + ((ch ^ (rr & 7)) * 16));
          if (key_w + rr < N)
            *reinterpret_cast<uint4 *>(base + static_cast<int64_t>(key_w + rr) * D + 64 * hh +
                                       ch * 8) = x;
        }
        __syncwarp();
      }
      g0 += it.n_halves;
      steps += it.n_steps;
    }
  }

  if (warp >= 4 && (threadIdx.x & 31) == 0) bulk_wait_all();
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

cudaError_t launch_bwd_main_d128(const CUtensorMap &tq64, const CUtensorMap &tk,
                                 const CUtensorMap &tv, const CUtensorMap &tdo64,
                                 const CUtensorMap &tdq,
                                 const float *vecs, void *dk, void *dv, int BH,
                                 int N, float scale, int causal, int *sched, int fault_cta,
                                 int *dev_status, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(bwd_pipe_kernel,
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
  return cudaLaunchKernelEx(&cfg, bwd_pipe_kernel, tq64, tk, tv, tdo64, tdq, vecs,
                            reinterpret_cast<__nv_bfloat16 *>(dk),
                            reinterpret_cast<__nv_bfloat16 *>(dv), N, BH, scale, causal, sched,
                            fault_cta, dev_status);
}

}  // namespace fattn
