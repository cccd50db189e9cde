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
// GB300 mapping.  The kernel is persistent: one CTA per SM takes work items
// from a device-wide counter until none are left, an item being two 128-row
// query tiles (A and B, 256 rows) of one head.  Items are numbered heaviest
// first (under the causal mask later query blocks see more keys), so the
// greedy claim order balances the CTAs' totals (longest-first list
// scheduling).  The producer warp claims each item and hands its number to
// the other roles through a two-entry ring in shared memory.  Both tiles of
// an item use every K/V tile the CTA loads.  Warp roles (the
// warp-specialised design of youngju.dev section 9.2, "FlashAttention-3",
// rebuilt on tcgen05 and TMEM):
//   warp 0       TMA producer: Q_A and Q_B per item, K and V tiles into
//                separate multi-stage rings that run on across items
//   warp 1       MMA issuer: S_T = Q_T K^T into TMEM; O_T += P_T V with P_T
//                read from TMEM (T = A, B)
//   warps 2-3    idle (they complete the producer warpgroup)
//   warps 4-7    softmax of tile A, one query row per thread, and its epilogue
//                (O_A / l from TMEM to bf16 rows, and the LSE)
//   warps 8-11   the same for tile B
// TMEM (512 columns): S_A | S_B | O_A | O_B.  P_T is written as bf16 over the
// first half of S_T.  Per key tile j the MMA warp issues
//     PV_A(j)  QK_A(j+1)  PV_B(j)  QK_B(j+1)
// so while the softmax of A works on S_A(j+1) the tensor core runs PV_B(j)
// and QK_B(j+1), and vice versa: the two softmax warpgroups take turns on the
// exponential unit while the tensor core stays busy (the matmul/softmax
// interleaving of section 9.2).  tcgen05 MMAs of one thread execute in issue
// order, so QK_T(j+1) overwriting S_T (and the P_T inside it) never overtakes
// PV_T(j), and the commit that signals S_T(j+1) also certifies that PV_T(j)
// finished, which lets the softmax warps rescale O_T without another wait.
// While a softmax warpgroup writes one item's output, the tensor core already
// computes the next item's first S tiles; the next PV_T cannot start before
// those warps have read O_T, because it waits for their first P_T.
// The E4M3 instantiation instead keeps P_T in shared memory (two buffers per
// tile) and issues QK_T(j+1) as soon as the softmax has loaded S_T(j), ahead
// of PV_T(j): there the softmax waits for PV_T(j) only before a rescale.
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
#include "ptx_f8.cuh"

namespace fattn {
namespace {

constexpr int BM = 128;             // query rows per tile (MMA M)
constexpr int BN = 128;             // keys per tile (MMA N of QK^T, K of PV)
constexpr int kThreads = 384;       // 12 warps = 3 warpgroups
// Register split (setmaxnreg): the launch gives every thread 168 registers
// (65536 / 384, rounded to 8); the producer warpgroup drops to 88 and the two
// softmax warpgroups rise to 208, so each SM sub-partition, which hosts one
// warp of every warpgroup, needs 88 + 208 + 208 = 3 * 168 registers per lane.
// The build checks that ptxas gives this kernel exactly 168 at launch.
constexpr uint32_t kRegsProducer = 88, kRegsSoftmax = 208;
constexpr uint32_t kTmemCols = 512;

// FP8 (E4M3) variant: Q and K arrive as E4M3 codes with one scale per 128-row
// block, V as E4M3 codes transposed to [d][keys] with one scale per head.  The
// softmax weights are carried as E4M3 of 2^4 * exp2(x - m_ref): with the
// output rescale skipped while the row max has grown by at most 4 (instead of
// 8), every weight stays at or below 2^8 < 448, and weights down to 2^-10 of
// the row max keep E4M3's full 3-bit mantissa.
template <bool FP8>
struct SoftmaxCfg {
  static constexpr float kRescaleThreshold = FP8 ? 4.0f : 8.0f;  // log2 units
  static constexpr float kPOffset = FP8 ? 4.0f : 0.0f;           // log2 of the weight scale
};

template <int D, bool FP8 = false>
struct Cfg {
  static constexpr int kElemBytes = FP8 ? 1 : 2;
  static constexpr int kStages = (D == 64 || FP8) ? 4 : 2;   // K and V ring depth
  static constexpr int kBoxes = D * kElemBytes / 128;        // 128-byte boxes per row
  static constexpr int kTileBytes = BM * D * kElemBytes;     // one 128 x D tile
  static constexpr int kBoxBytes = BM * 128;        // 16 KB
  static constexpr int kQ = 0;                      // Q_A, Q_B
  static constexpr int kK0 = kQ + 2 * kTileBytes;
  static constexpr int kV0 = kK0 + kStages * kTileBytes;
  static constexpr int kBar = kV0 + kStages * kTileBytes;
  // Epilogue staging: per softmax warp (2 tiles x 4) its 32 rows x 64 columns
  // of bf16 output, 4 KB.
  // FP8: P leaves the scores' TMEM columns for shared memory, two buffers
  // per query tile of 128 rows x 128 codes in the 128-byte-swizzle K-major
  // layout (the layout of Q), so that Q K^T(j+1) may overwrite the scores as
  // soon as the softmax has loaded S(j), without waiting for P V(j).  A
  // tile's output staging is its first P buffer (free during its epilogue).
  static constexpr int kStage = kBar + (FP8 ? 1024 : 512);
  static constexpr int kP = kStage;                  // FP8: 4 x 16 KB
  static constexpr int kPBuf = BM * BN;              // 16 KB
  static constexpr int kBytes = kStage + (FP8 ? 4 * kPBuf : 8 * 4096);
  static constexpr int kAlloc = kBytes + 1024;      // slack for 1 KB alignment
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
  static constexpr uint32_t kColS0 = 0, kColS1 = 128;
  static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
};

// 16-bit element type of Q, K, V, P and O: bf16 (F16 = false) or fp16.  The
// instruction descriptor's A and B type fields (bits 7-9, 10-12) are 1 for
// bf16 and 0 for fp16; both operands of every MMA share the type.
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

// Barrier slots (8 bytes each).
enum : int {
  kBarQFullA = 0,      // query tile A of the current item
  kBarQEmptyA = 1,
  kBarSFull = 2,       // +tile (A, B)
  kBarPReady = 4,      // +2 * tile + half: the first / second 64 columns of P
  kBarODone = 8,       // +tile
  kBarQFullB = 10,     // query tile B
  kBarQEmptyB = 11,
  kBarDrain = 12,
  kBarItemFull = 13,   // +ring slot (2)
  kBarItemEmpty = 32,  // +ring slot (2)
  kBarKFull = 16,      // +stage (up to 4)
  kBarKEmpty = 20,
  kBarVFull = 24,
  kBarVEmpty = 28,
  kBarSFree = 34,      // FP8, +tile: the softmax has loaded S(j) (4 warps)
  kBarPVDone = 36,     // FP8, +2 * tile + P buffer: P V(j) has completed
  kBarPReady1 = 40,    // FP8: kBarPReady's halves for P buffer 1
  kNumBars = 44
};
// The PReady barrier of half h of P(n) of tile t.  FP8: one set per P
// buffer, since there the softmax may finish P(n + 1) (its scores were
// computed ahead) before the MMA warp has waited for P(n); a set sees the
// tiles n, n + 2, ... and the softmax cannot reach n + 2 before P V(n) has
// been issued.  The phase parity of the wait follows.
template <bool FP8>
__device__ __forceinline__ int pready_slot(int t, int h, int n) {
  return ((FP8 && (n & 1)) ? kBarPReady1 : kBarPReady) + 2 * t + h;
}
template <bool FP8>
__device__ __forceinline__ uint32_t pready_parity(int n) {
  return static_cast<uint32_t>((FP8 ? n >> 1 : n) & 1);
}
// Arrivals that free an item-ring slot: the MMA thread plus every warp of the
// two softmax warpgroups.
constexpr int kItemConsumers = 1 + 4 + 4;

struct SmemMisc {
  uint32_t tmem_base;
  int abort;
  int item[2];
};
static_assert(8 * kNumBars + sizeof(SmemMisc) <= 512, "barrier area");

// Waits with a time limit for the phase of parity `ph` of an mbarrier; used
// on the unwind paths.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t ph) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, ph) && globaltimer_ns() - t0 < kWaitLimitNs) {
  }
}

// Work item w -> query block, head and the key tiles each query tile needs.
// With a mask, `ranges` holds per (mask head, item) the first key tile kv0
// that any of the item's rows can see and the tile counts n_a <= n_b of its
// query tiles (mask_tiles.cu); key tile j of the item is tile kv0 + j of the
// sequence.
struct ItemDecoder {
  int BH, n_qblocks, n_kv_total, causal;
  const int2 *ranges;
  int mask_shared;
  __device__ void decode(int w, int &q0, int &bh, int &n_a, int &n_b, int &kv0) const {
    const int qb = n_qblocks - 1 - w / BH;
    bh = w % BH;
    q0 = qb * 2 * BM;
    kv0 = 0;
    if (ranges != nullptr) {
      const int2 r = ranges[static_cast<int64_t>(mask_shared ? 0 : bh) * n_qblocks + qb];
      // Clamped into the sequence's key tiles, so that no summary can make
      // the item address tiles, flags or bits outside their buffers.
      kv0 = min(r.x & 0xffff, n_kv_total - 1);
      n_b = max(1, min(r.y, n_kv_total - kv0));
      n_a = max(1, min(r.x >> 16, n_b));
      return;
    }
    n_a = causal ? min(2 * qb + 1, n_kv_total) : n_kv_total;
    n_b = causal ? min(2 * qb + 2, n_kv_total) : n_kv_total;
  }
};

// MASK: a boolean mask decides visibility -- key j is visible to query row i
// of head bh iff mask[bh * mask_bh_stride + i * N + j] != 0 (N a multiple of 16;
// causal is then 0).  A row that sees no key gets O = 0 and LSE = -inf.
// mask_ranges / mask_flags: the per-tile summary of mask_tiles.cu: per item
// the key tiles its rows can see (the others are skipped), per 128 x 128
// block a flag (0: nothing visible, 1: partly, 2: everything; a fully
// visible tile reads no mask bytes), and mask_bits per row of each block its
// 128 visibility bits, which a partly visible tile reads in place of the
// row's 128 mask bytes.
// FP8: E4M3 inputs (tm_v then maps V^T, [BH][d][Npad]); q_scale and k_scale
// hold one dequantization scale per 128-row block of each head (n_sblk per
// head), v_scale one per head.  The output is bf16.
template <int D, bool F16, bool MASK, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, uint16_t *__restrict__ o,
                       float *__restrict__ lse, int N, int BH, int n_qblocks, float scale_log2,
                       int causal, int *__restrict__ sched, int *__restrict__ dev_status,
                       int fault_cta, const uint8_t *__restrict__ mask,
                       int64_t mask_bh_stride, const float *__restrict__ q_scale,
                       const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                       int n_sblk, const int2 *__restrict__ mask_ranges,
                       const uint8_t *__restrict__ mask_flags,
                       const uint4 *__restrict__ mask_bits) {
  using C = Cfg<D, FP8>;
  using SC = SoftmaxCfg<FP8>;
  static_assert(!FP8 || (D == 128 && !F16 && !MASK), "the FP8 variant is d = 128, unmasked");
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t bars = s_base + C::kBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  SmemMisc *misc = reinterpret_cast<SmemMisc *>(smem + C::kBar + 8 * kNumBars);
  volatile int *abort_flag = &misc->abort;

  ItemDecoder sch;
  sch.BH = BH;
  sch.n_qblocks = n_qblocks;
  sch.n_kv_total = (N + BN - 1) / BN;
  sch.causal = causal;
  sch.ranges = MASK ? mask_ranges : nullptr;
  sch.mask_shared = mask_bh_stride == 0;
  const int n_items = n_qblocks * BH;
  // Consumer side of the item ring: every lane of the calling warp waits for
  // ring entry k, reads it, and one arrival per warp (or the lone MMA thread)
  // frees the slot.
  auto fetch_item = [&](int k, int &w, bool whole_warp) -> bool {
    const int slot = k & 1;
    if (!mbar_wait(bar(kBarItemFull + slot), (k >> 1) & 1, abort_flag)) return false;
    w = *reinterpret_cast<volatile int *>(&misc->item[slot]);
    if (whole_warp) __syncwarp();
    if (!whole_warp || (threadIdx.x & 31) == 0) mbar_arrive(bar(kBarItemEmpty + slot));
    return true;
  };

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFullA), 1);
    mbar_init(bar(kBarQEmptyA), 1);
    mbar_init(bar(kBarQFullB), 1);
    mbar_init(bar(kBarQEmptyB), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPReady + 2 * t), 4);      // one arrival per softmax warp
      mbar_init(bar(kBarPReady + 2 * t + 1), 4);
      mbar_init(bar(kBarODone + t), 1);
      mbar_init(bar(kBarSFree + t), 4);
      mbar_init(bar(kBarPVDone + 2 * t), 1);
      mbar_init(bar(kBarPVDone + 2 * t + 1), 1);
      mbar_init(bar(kBarPReady1 + 2 * t), 4);
      mbar_init(bar(kBarPReady1 + 2 * t + 1), 4);
    }
    mbar_init(bar(kBarDrain), 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(kBarItemFull + k), 1);
      mbar_init(bar(kBarItemEmpty + k), kItemConsumers);
    }
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
  // The bf16 / fp16 forwards are launched as programmatic dependents of the
  // kernel before them on the stream (the mask summary kernels, or whatever
  // wrote Q, K and V): their set-up above overlaps that kernel's tail, and
  // nothing they read or write in global memory is touched before it has
  // finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsProducer));
    static_assert(kRegsProducer + 2 * kRegsSoftmax == 3 * 168,
                  "the warpgroup register split must use exactly the launch budget");
    if (warp == 0 && elect_one()) {
      // ---------------------------------------------------------- TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int it = 0, kv = 0, nk = 0, nv = 0, nqa = 0, nqb = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        // Claim the next item and publish it to the other roles.
        const int slot = k & 1;
        if (!(ok = mbar_wait(bar(kBarItemEmpty + slot), ((k >> 1) & 1) ^ 1, abort_flag))) break;
        const int w = atomicAdd(sched, 1);
        misc->item[slot] = w;
        mbar_arrive(bar(kBarItemFull + slot));
        if (w >= n_items) break;
        int q0, bh, n_a, n_b, kv0;
        sch.decode(w, q0, bh, n_a, n_b, kv0);
        // Query tile t of this item, once the previous item's last QK_t has
        // read the buffer.  Tile A goes first: the MMA warp starts it during
        // the previous item's last step.  Tile B follows the first key tile.
        auto load_q = [&](int t) -> bool {
          if (!mbar_wait(bar(t ? kBarQEmptyB : kBarQEmptyA), (it & 1) ^ 1, abort_flag))
            return false;
          const uint32_t full = bar(t ? kBarQFullB : kBarQFullA);
          mbar_arrive_expect_tx(full, C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(s_base + C::kQ + t * C::kTileBytes + b * C::kBoxBytes, &tm_q, b * 64,
                        q0 + t * BM, bh, full);
          return true;
        };
        if (!(ok = load_q(0))) break;
        ++nqa;
        if (static_cast<int>(blockIdx.x) == fault_cta) {
          if ((ok = load_q(1))) ++nqb;
          // Failure-path test: stop here, as if the key-tile copies were lost;
          // the MMA warp's bounded wait for them runs out.
          ok = false;
          break;
        }
        for (int j = 0; j < n_b; ++j, ++kv) {
          const int st = kv % S;
          const uint32_t ph = (kv / S) & 1;
          if (!(ok = mbar_wait(bar(kBarKEmpty + st), ph ^ 1, abort_flag))) break;
          mbar_arrive_expect_tx(bar(kBarKFull + st), C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(s_base + C::kK0 + st * C::kTileBytes + b * C::kBoxBytes, &tm_k, b * 64,
                        (kv0 + j) * BN, bh, bar(kBarKFull + st));
          nk = kv + 1;
          if (j == 0) {
            if (!(ok = load_q(1))) break;
            ++nqb;
          }
          if (!(ok = mbar_wait(bar(kBarVEmpty + st), ph ^ 1, abort_flag))) break;
          mbar_arrive_expect_tx(bar(kBarVFull + st), C::kTileBytes);
          if (FP8)   // V^T: rows are the d coordinates, keys run along x
            tma_load_3d(s_base + C::kV0 + st * C::kTileBytes, &tm_v, (kv0 + j) * BN, 0, bh,
                        bar(kBarVFull + st));
          else
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_3d(s_base + C::kV0 + st * C::kTileBytes + b * C::kBoxBytes, &tm_v, b * 64,
                          (kv0 + j) * BN, bh, bar(kBarVFull + st));
          nv = kv + 1;
        }
        ++it;
      }
      if (!ok) {
        // Let the copies in flight land before the CTA exits.
        if (nqa > 0) drain_wait(bar(kBarQFullA), (nqa - 1) & 1);
        if (nqb > 0) drain_wait(bar(kBarQFullB), (nqb - 1) & 1);
        for (int i = (nk > S ? nk - S : 0); i < nk; ++i)
          drain_wait(bar(kBarKFull + i % S), (i / S) & 1);
        for (int i = (nv > S ? nv - S : 0); i < nv; ++i)
          drain_wait(bar(kBarVFull + i % S), (i / S) & 1);
      }
    } else if (warp == 1 && elect_one()) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_qk =
          FP8 ? idesc_e4m3_f32(BM, BN) : idesc16<F16>(idesc_bf16_f32(BM, BN, false));
      constexpr uint32_t idesc_pv =
          FP8 ? idesc_e4m3_f32(BM, D) : idesc16<F16>(idesc_bf16_f32(BM, D, true));
      // Shared-memory descriptors are built once; moving an operand by `off`
      // bytes adds off >> 4 to the start-address field, which cannot carry
      // out of its 14 bits for addresses inside the 228 KB shared window.
      // Descriptors as their low 32-bit words (start address, leading offset);
      // the high word is the same for all three operands.
      const uint32_t dq = sdesc_lo(s_base + C::kQ, 16);
      const uint32_t dk = sdesc_lo(s_base + C::kK0, 16);
      // V (16-bit) is read N-major: its leading offset is the box stride.
      // V^T (FP8) is K-major like Q and K.
      const uint32_t dv = sdesc_lo(s_base + C::kV0, FP8 ? 16 : C::kBoxBytes);
      auto qk = [&](int t, int kvi) {
        const uint32_t a = dq + ((t * C::kTileBytes) >> 4);
        const uint32_t b = dk + (((kvi % S) * C::kTileBytes) >> 4);
        const uint32_t s_col = tmem + (t ? C::kColS1 : C::kColS0);
        if (FP8) {
          // K = 32 codes (32 bytes) per MMA.
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_f8_ss_lo(s_col, a + kk * 2, b + kk * 2, idesc_qk, kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
            mma_ss_lo(s_col, a + off, b + off, idesc_qk, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(kBarSFull + t));
      };
      // Half h of O_T += P_T V with P_T in TMEM over S_T (16-bit kernels):
      // keys 64h .. 64h+63 of the tile.
      auto pv = [&](int t, int kvi, bool first, int h) {
        const uint32_t b = dv + (((kvi % S) * C::kTileBytes) >> 4);
        const uint32_t s_col = tmem + (t ? C::kColS1 : C::kColS0);
        const uint32_t o_col = tmem + (t ? C::kColO1 : C::kColO0);
#pragma unroll
        for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
          mma_ts_lo(o_col, s_col + kk * 8, b + ((kk * 2048) >> 4), idesc_pv,
                    (!first || kk > 0) ? 1u : 0u);
      };
      auto wait_p = [&](int t, int h, int cnt) {
        return mbar_wait(bar(pready_slot<FP8>(t, h, cnt)), pready_parity<FP8>(cnt), abort_flag);
      };
      auto wait_k = [&](int kvi) {
        return mbar_wait(bar(kBarKFull + kvi % S), (kvi / S) & 1, abort_flag);
      };
      int it = 0, kv = 0;
      bool ok = true;
      if constexpr (FP8) {
        // P in shared memory: Q K^T(j+1) of a tile is issued as soon as its
        // softmax has loaded S(j) (SFree) and K(j+1) has landed, ahead of
        // P V(j), so the next scores are ready when the softmax finishes P(j).
        // Each commit covers every earlier MMA of this thread, so SFull(j+1)
        // still certifies P V(j-1) (the P buffer the softmax fills next);
        // P V(j) signals PVDone for the one thing that needs it, a rescale of O.
        const uint32_t dp = sdesc_lo(s_base + C::kP, 16);
        int qk_n[2] = {0, 0}, pv_n[2] = {0, 0};   // Q K^T and P V issued, per tile
        auto qk_free = [&](int t, int kvi) -> bool {
          if (qk_n[t] > 0 && !mbar_wait(bar(kBarSFree + t), (qk_n[t] - 1) & 1, abort_flag))
            return false;
          tc_fence_after();
          qk(t, kvi);
          ++qk_n[t];
          return true;
        };
        auto pv_smem = [&](int t, int kvi, bool first) -> bool {
          const int n = pv_n[t];
          const uint32_t a = dp + (((t * 2 + (n & 1)) * C::kPBuf) >> 4);
          const uint32_t b = dv + (((kvi % S) * C::kTileBytes) >> 4);
          const uint32_t o_col = tmem + (t ? C::kColO1 : C::kColO0);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (!wait_p(t, h, n)) return false;
            tc_fence_after();
#pragma unroll
            for (int kk = 2 * h; kk < 2 * h + 2; ++kk)
              mma_f8_ss_lo(o_col, a + kk * 2, b + kk * 2, idesc_pv, (!first || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(kBarPVDone + 2 * t + (n & 1)));
          ++pv_n[t];
          return true;
        };
        int w = 0;
        bool a0_issued = false;
        ok = fetch_item(0, w, false);
        for (int k = 0; ok && w < n_items; ++k) {
          int q0, bh, n_a, n_b, kv0;
          sch.decode(w, q0, bh, n_a, n_b, kv0);
          if (!a0_issued) {
            if (!(ok = mbar_wait(bar(kBarQFullA), it & 1, abort_flag) && wait_k(kv) &&
                       qk_free(0, kv)))
              break;
            if (n_a == 1) mma_commit(bar(kBarQEmptyA));
          }
          a0_issued = false;
          if (!(ok = mbar_wait(bar(kBarQFullB), it & 1, abort_flag) && wait_k(kv) &&
                     qk_free(1, kv)))
            break;
          mma_commit(bar(kBarKEmpty + kv % S));
          if (n_b == 1) mma_commit(bar(kBarQEmptyB));
          int w_next = n_items;
          bool fetched = false;
          for (int j = 0; j < n_b; ++j) {
            const int kvj = kv + j;
            const int st = kvj % S;
            if (j + 1 < n_a) {
              if (!(ok = wait_k(kvj + 1) && qk_free(0, kvj + 1))) break;
              if (j + 2 == n_a) mma_commit(bar(kBarQEmptyA));  // last QK_A of the item
            }
            if (!(ok = mbar_wait(bar(kBarVFull + st), (kvj / S) & 1, abort_flag))) break;
            if (j < n_a) {
              if (!(ok = pv_smem(0, kvj, j == 0))) break;
              if (j == n_a - 1) mma_commit(bar(kBarODone + 0));
            }
            if (j == n_b - 1) {
              // The next item's tile A, once S_A has been read.
              if (!(ok = fetch_item(k + 1, w_next, false))) break;
              fetched = true;
              if (w_next < n_items) {
                int nq0, nbh, nn_a, nn_b, nkv0;
                sch.decode(w_next, nq0, nbh, nn_a, nn_b, nkv0);
                if (!(ok = mbar_wait(bar(kBarQFullA), (it + 1) & 1, abort_flag) &&
                           wait_k(kv + n_b) && qk_free(0, kv + n_b)))
                  break;
                if (nn_a == 1) mma_commit(bar(kBarQEmptyA));
                a0_issued = true;
              }
            }
            if (j + 1 < n_b) {
              if (!(ok = wait_k(kvj + 1) && qk_free(1, kvj + 1))) break;
              mma_commit(bar(kBarKEmpty + (kvj + 1) % S));
              if (j + 2 == n_b) mma_commit(bar(kBarQEmptyB));  // last QK_B of the item
            }
            if (!(ok = pv_smem(1, kvj, j == 0))) break;
            mma_commit(bar(kBarVEmpty + st));
            if (j == n_b - 1) mma_commit(bar(kBarODone + 1));
          }
          if (!ok) break;
          kv += n_b;
          ++it;
          if (!fetched && !(ok = fetch_item(k + 1, w_next, false))) break;
          w = w_next;
        }
      } else {
        int cnt_a = 0, cnt_b = 0;
        // The next item's QK_A(0) is issued during this item's last step, before
        // the wait for tile B's last P, so that tile A's softmax of the next item
        // overlaps tile B's tail instead of following it.
        int w = 0;
        bool a0_issued = false;
        ok = fetch_item(0, w, false);
        for (int k = 0; ok && w < n_items; ++k) {
          int q0, bh, n_a, n_b, kv0;
          sch.decode(w, q0, bh, n_a, n_b, kv0);
          if (!a0_issued) {
            if (!(ok = mbar_wait(bar(kBarQFullA), it & 1, abort_flag) && wait_k(kv))) break;
            tc_fence_after();
            qk(0, kv);
            if (n_a == 1) mma_commit(bar(kBarQEmptyA));
          }
          a0_issued = false;
          if (!(ok = mbar_wait(bar(kBarQFullB), it & 1, abort_flag) && wait_k(kv))) break;
          tc_fence_after();
          qk(1, kv);
          mma_commit(bar(kBarKEmpty + kv % S));
          if (n_b == 1) mma_commit(bar(kBarQEmptyB));
          int w_next = n_items;
          bool fetched = false;
          for (int j = 0; j < n_b; ++j) {
            const int kvj = kv + j;
            const int st = kvj % S;
            if (!(ok = mbar_wait(bar(kBarVFull + st), (kvj / S) & 1, abort_flag))) break;
            bool k_next_ready = false;
            if (j < n_a) {
              if (!(ok = wait_p(0, 0, cnt_a))) break;
              tc_fence_after();
              pv(0, kvj, j == 0, 0);
              if (!(ok = wait_p(0, 1, cnt_a))) break;
              tc_fence_after();
              pv(0, kvj, j == 0, 1);
              ++cnt_a;
              if (j == n_a - 1) mma_commit(bar(kBarODone + 0));
              if (j + 1 < n_a) {
                if (!(ok = wait_k(kvj + 1))) break;
                k_next_ready = true;
                tc_fence_after();
                qk(0, kvj + 1);
                if (j + 2 == n_a) mma_commit(bar(kBarQEmptyA));  // last QK_A of the item
              }
            }
            if (j == n_b - 1) {
              // S_A is free (its last PV was issued above or at an earlier step):
              // start the next item's tile A now.
              if (!(ok = fetch_item(k + 1, w_next, false))) break;
              fetched = true;
              if (w_next < n_items) {
                int nq0, nbh, nn_a, nn_b, nkv0;
                sch.decode(w_next, nq0, nbh, nn_a, nn_b, nkv0);
                if (!(ok = mbar_wait(bar(kBarQFullA), (it + 1) & 1, abort_flag) &&
                           wait_k(kv + n_b)))
                  break;
                tc_fence_after();
                qk(0, kv + n_b);
                if (nn_a == 1) mma_commit(bar(kBarQEmptyA));
                a0_issued = true;
              }
            }
            if (!(ok = wait_p(1, 0, cnt_b))) break;
            tc_fence_after();
            pv(1, kvj, j == 0, 0);
            if (!(ok = wait_p(1, 1, cnt_b))) break;
            tc_fence_after();
            pv(1, kvj, j == 0, 1);
            ++cnt_b;
            mma_commit(bar(kBarVEmpty + st));
            if (j == n_b - 1) mma_commit(bar(kBarODone + 1));
            if (j + 1 < n_b) {
              if (!k_next_ready && !(ok = wait_k(kvj + 1))) break;
              tc_fence_after();
              qk(1, kvj + 1);
              mma_commit(bar(kBarKEmpty + (kvj + 1) % S));
              if (j + 2 == n_b) mma_commit(bar(kBarQEmptyB));  // last QK_B of the item
            }
          }
          if (!ok) break;
          kv += n_b;
          ++it;
          if (!fetched && !(ok = fetch_item(k + 1, w_next, false))) break;
          w = w_next;
        }
      }
      // Drain: every MMA issued above has completed once this phase does.
      mma_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;                 // query tile: 0 = A, 1 = B
    const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
    const int r_local = quarter * 32 + (threadIdx.x & 31);
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + (t ? C::kColS1 : C::kColS0);
    const uint32_t o_tmem = tmem + lane_off + (t ? C::kColO1 : C::kColO0);
    const uint64_t c2 = f2(scale_log2, scale_log2);
    int it = 0, sc = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int w;
      if (!(ok = fetch_item(k, w, true)) || w >= n_items) break;
      int q0, bh, n_a, n_b, kv0;
      sch.decode(w, q0, bh, n_a, n_b, kv0);
      const int row = q0 + t * BM + r_local;
      const int n_mine = t ? n_b : n_a;
      // MASK: this query tile's row of the tile summary (a tile past the
      // sequence end has no rows to keep: treat it as seeing nothing).
      const int n_t = (N + BM - 1) / BM;
      const int qt = q0 / BM + t;
      const int64_t blk_row = (static_cast<int64_t>(mask_bh_stride ? bh : 0) * n_t + qt) * n_t;
      const uint8_t *flag_row = MASK ? mask_flags + blk_row : nullptr;
      const uint4 *bits_row = MASK ? mask_bits + blk_row * BM + r_local : nullptr;
      // FP8: the scores are raw code products; this tile's Q block scale (a
      // tile past the last block has no rows to keep) times each key tile's
      // scale turns them into scale * q.k.
      float q_fac = scale_log2;
      if (FP8) {
        const int qblk = q0 / BM + t;
        if (qblk < n_sblk) q_fac *= q_scale[static_cast<int64_t>(bh) * n_sblk + qblk];
      }
      float m = -INFINITY, l = 0.f;
      // MASK: the block flag of key tile j + 1 is fetched one tile ahead (a
      // tile past the sequence end sees nothing), so that at tile j only the
      // row's 128 visibility bits, for a partly visible block, wait on a load;
      // they are fetched before the wait for the scores.  Holding the bits
      // themselves a tile ahead costs the softmax warps registers they spill.
      int flag_nx = (MASK && n_mine > 0 && qt < n_t) ? flag_row[kv0] : 0;
      for (int j = 0; j < n_mine; ++j, ++sc) {
        const float c_tile =
            FP8 ? q_fac * k_scale[static_cast<int64_t>(bh) * n_sblk + j] : scale_log2;
        uint4 mk = make_uint4(0u, 0u, 0u, 0u);   // keys past N are not visible
        int flag = 1;
        if (MASK) {
          flag = flag_nx;
          if (flag == 1) mk = bits_row[static_cast<int64_t>(kv0 + j) * BM];
          if (j + 1 < n_mine && qt < n_t) flag_nx = flag_row[kv0 + j + 1];
        }
        if (!(ok = mbar_wait(bar(kBarSFull + t), sc & 1, abort_flag))) break;
        tc_fence_after();
        uint32_t sv[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + c * 32, sv[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_wait_ld(sv[c]);
        if (FP8) {
          // The scores are in registers: the MMA warp may overwrite S_T with
          // the next tile's (P goes to shared memory).
          tc_fence_before();
          __syncwarp();
          if ((threadIdx.x & 31) == 0) mbar_arrive(bar(kBarSFree + t));
        }
#define S_(c) sv[(c) >> 5][(c) & 31]
        if (MASK) {
          if (flag != 2) {   // a fully visible tile needs no mask
#pragma unroll
            for (int c = 0; c < BN; ++c) {
              const uint32_t w = (&mk.x)[c >> 5];
              if (((w >> (c & 31)) & 1u) == 0u) S_(c) = __float_as_uint(-INFINITY);
            }
          }
        } else if (j == n_mine - 1) {
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
        const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c_tile;
        float alpha = 1.f;
        if (tmax > m + SC::kRescaleThreshold) {  // also true while m = -inf
          alpha = ex2_approx(m - tmax);
          m = tmax;
        }
        // PV_T(j-1) was issued before QK_T(j), so O_T is complete: rescale it
        // before the first half of P lets PV_T(j) accumulate into it.  (FP8:
        // QK_T(j) goes first, so wait for PV_T(j-1) itself.)
        if (j > 0 && __any_sync(~0u, alpha != 1.f)) {
          if (FP8) {
            const int pv = sc - 1;
            if (!(ok = mbar_wait(bar(kBarPVDone + 2 * t + (pv & 1)), (pv >> 1) & 1, abort_flag)))
              break;
            tc_fence_after();
          }
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
        // While a masked row has seen no visible key, m is -inf: use 0 so that
        // the (all masked) scores give p = 0 rather than NaN.
        const float mref = (MASK && m == -INFINITY) ? 0.f : m;
        const float nmv = FP8 ? SC::kPOffset - mref : -mref;
        const uint64_t nm2 = f2(nmv, nmv);
        uint64_t sum2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
        if (FP8) {
          const uint64_t c2t = f2(c_tile, c_tile);
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const uint64_t xa =
                  ffma2(f2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), c2t, nm2);
              const uint64_t xb = ffma2(
                  f2(__uint_as_float(sv[c][e + 2]), __uint_as_float(sv[c][e + 3])), c2t, nm2);
              const float2 x = f2_split(xa), y = f2_split(xb);
              const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              const float2 r = make_float2(ex2_approx(y.x), ex2_approx(y.y));
              sum2[0] = fadd2(sum2[0], f2(p.x, p.y));
              sum2[1] = fadd2(sum2[1], f2(r.x, r.y));
              // Four codes per column; columns 8(c & 1) .. 8(c & 1) + 7 of
              // this 64-key half.
              pk[(c & 1) * 8 + (e >> 2)] = pack_e4m3x4(p.x, p.y, r.x, r.y);
            }
            if (c & 1) {
              // Keys 0-63 (then 64-127) of P, 16-byte chunks 4(c >> 1) .. +3
              // of this row of P buffer sc & 1 (128-byte swizzle: chunk ^ row
              // % 8), are in shared memory: let PV_T use them.  (The buffer
              // was last read by PV_T(sc - 2), complete before S_T(sc).)
              uint8_t *prow = smem + C::kP + (t * 2 + (sc & 1)) * C::kPBuf +
                              (r_local >> 3) * 1024 + (r_local & 7) * 128;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int ch = 4 * (c >> 1) + q;
                *reinterpret_cast<uint4 *>(prow + ((ch ^ (r_local & 7)) << 4)) =
                    make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
              }
              fence_proxy_async_smem();
              tmem_wait_st();   // a rescale of O_T above has landed
              tc_fence_before();
              __syncwarp();
              if ((threadIdx.x & 31) == 0) mbar_arrive(bar(pready_slot<FP8>(t, c >> 1, sc)));
            }
          }
        } else {
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
              // Columns 0-63 (then 64-127) of P are in TMEM: let PV_T use them.
              tmem_wait_st();
              tc_fence_before();
              __syncwarp();
              if ((threadIdx.x & 31) == 0) mbar_arrive(bar(kBarPReady + 2 * t + (c >> 1)));
            }
          }
        }
#undef S_
        const float2 sa = f2_split(fadd2(sum2[0], sum2[1]));
        l = l * alpha + (sa.x + sa.y);
      }
      if (!ok) break;
      // Epilogue: O_T / l as bf16 rows and the LSE, once the last PV_T is done.
      if (!(ok = mbar_wait(bar(kBarODone + t), it & 1, abort_flag))) break;
      tc_fence_after();
      float inv_l = (MASK && l == 0.f) ? 0.f : 1.f / l;
      if (FP8) inv_l *= v_scale[bh];
      // O rows leave through shared memory: each warp packs its 32 rows, 64
      // columns at a time, into a 4 KB buffer (16-byte chunks swizzled by the
      // row so that neither side has bank conflicts) and reads it back so that
      // eight lanes store one row's 128 contiguous bytes: 4 lines per store
      // instruction instead of 32.
      uint8_t *stg = smem +
                     (FP8 ? C::kP + t * 2 * C::kPBuf + quarter * 4096
                          : C::kStage + (t * 4 + quarter) * 4096);
      const int lane = threadIdx.x & 31;
      const int row_w = row - lane;   // this warp's first row
#pragma unroll
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
      if (lse != nullptr && row < N)
        lse[static_cast<int64_t>(bh) * N + row] =
            (MASK && l == 0.f) ? -INFINITY
            : FP8              ? (m - SC::kPOffset + __log2f(l)) * 0.6931471805599453f
                               : (m + __log2f(l)) * 0.6931471805599453f;
      ++it;
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
    // The last CTA to finish returns the item counter to zero for the next
    // launch that uses this slot: every CTA has stopped claiming by now.
    __threadfence();
    if (atomicAdd(sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      sched[0] = 0;
      sched[1] = 0;
      __threadfence();
    }
  }
}

int g_num_sms[64] = {};

template <int D, bool F16, bool MASK, bool FP8 = false>
cudaError_t launch_d(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, void *o,
                     float *lse, int BH, int N, float scale, int causal, int *sched,
                     int *dev_status, int fault_cta, cudaStream_t stream, const uint8_t *mask,
                     int64_t mask_bh_stride, const float *q_scale = nullptr,
                     const float *k_scale = nullptr, const float *v_scale = nullptr,
                     const int2 *mask_ranges = nullptr, const uint8_t *mask_flags = nullptr,
                     const uint4 *mask_bits = nullptr) {
  using C = Cfg<D, FP8>;
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
  e = cudaFuncSetAttribute(fwd_bf16_tc_kernel<D, F16, MASK, FP8>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc);
  if (e != cudaSuccess) return e;
  const int n_qblocks = (N + 2 * BM - 1) / (2 * BM);
  const long long n_items = static_cast<long long>(n_qblocks) * BH;
  const int grid = static_cast<int>(n_items < g_num_sms[dev] ? n_items : g_num_sms[dev]);
  const float scale_log2 = scale * 1.4426950408889634f;
  const int n_sblk = (N + BM - 1) / BM;
  // A programmatic dependent launch: the kernel waits with
  // griddepcontrol.wait after its set-up for the work before it (the wait is
  // a no-op in an ordinary launch).  The FP8 forward is launched the ordinary
  // way: after the quantization kernels the dependent launch measured slower.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = FP8 ? 0 : 1;
  return cudaLaunchKernelEx(&cfg, fwd_bf16_tc_kernel<D, F16, MASK, FP8>, tq, tk, tv,
                            reinterpret_cast<uint16_t *>(o), lse, N, BH, n_qblocks, scale_log2,
                            causal, sched, dev_status, fault_cta, mask, mask_bh_stride, q_scale,
                            k_scale, v_scale, n_sblk, mask_ranges, mask_flags, mask_bits);
}

}  // namespace

cudaError_t launch_fwd_bf16(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            void *o, float *lse, int BH, int N, int d, float scale, int causal,
                            int *sched, int *dev_status, int fault_cta, cudaStream_t stream,
                            bool f16, const uint8_t *mask, int64_t mask_bh_stride,
                            const int2 *mask_ranges, const uint8_t *mask_flags,
                            const uint4 *mask_bits) {
#define FATTN_FWD_ARGS \
  tq, tk, tv, o, lse, BH, N, scale, causal, sched, dev_status, fault_cta, stream, mask, \
      mask_bh_stride, nullptr, nullptr, nullptr, mask_ranges, mask_flags, mask_bits
  if (mask != nullptr) {
    if (f16) return cudaErrorInvalidValue;   // masks are served for bf16 only
    return d == 64 ? launch_d<64, false, true>(FATTN_FWD_ARGS)
                   : launch_d<128, false, true>(FATTN_FWD_ARGS);
  }
  if (d == 64)
    return f16 ? launch_d<64, true, false>(FATTN_FWD_ARGS)
               : launch_d<64, false, false>(FATTN_FWD_ARGS);
  return f16 ? launch_d<128, true, false>(FATTN_FWD_ARGS)
             : launch_d<128, false, false>(FATTN_FWD_ARGS);
#undef FATTN_FWD_ARGS
}

cudaError_t launch_fwd_fp8(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tvt,
                           const float *q_scale, const float *k_scale, const float *v_scale,
                           void *o, float *lse, int BH, int N, float scale, int causal,
                           int *sched, int *dev_status, int fault_cta, cudaStream_t stream) {
  return launch_d<128, false, false, true>(tq, tk, tvt, o, lse, BH, N, scale, causal, sched,
                                           dev_status, fault_cta, stream, nullptr, 0, q_scale,
                                           k_scale, v_scale);
}

}  // namespace fattn
