// decode_gqa_tc.cu -- single-query paged decode with grouped key/value heads
// on the sm_103a tensor cores: the query heads that share one cached head are
// the N columns of tcgen05 MMAs whose M rows are 128 context tokens.
//
// What is computed: for every sequence s and query head h, the attention of
// q[s,h,:] over the context_lens[s] cached tokens of key/value head
// h / G ("PagedAttention", data-sketchers.com, sections "Inputs", "Key",
// "Value"), with the online softmax of eqs. (2)-(4) of "Flash Attention"
// (suniverse77.github.io, section "Online Softmax") and 1024-token partitions
// merged with eq. (4) by a second kernel.
//
// Per 128-token step (8 cache blocks), for a slice of gs <= 16 query heads:
//   S^T [128 tokens][16 heads] = K [128 tokens][128 d] . Q^T     (8 MMAs, K = 16 each)
//   P   = exp2(S^T scale log2e - m), written to shared memory   (one token per thread)
//   O^T [128 d][16 heads]     += V^T [128 d][128 tokens] . P^T  (8 MMAs, one per block)
// The caches' own layouts are MMA operands once TMA views reorder them: a K
// box is one token half of a block (16 dimension groups x 8 tokens x 8
// values, 2 KB), exactly the no-swizzle K-major core matrices (8 rows x 16
// bytes) of A = K, and 16 boxes 2 KB apart make one 128-row operand; a V box
// is a block's V^T (128 dimensions x 16 tokens, 4 KB) in the 32-byte-swizzle
// K-major layout of A = V^T, one MMA (K = 16 tokens) per block.  The softmax
// is cheap: each thread holds one token's scores, and a step needs one
// cross-warp maximum per head; row sums stay per thread until the end.
//
// Persistent CTAs (one per SM) take work units (sequence, partition, cached
// head, head slice) from a device-wide counter.  Warp roles:
//   warps 0-3   softmax (thread = token row of S^T)
//   warp 4      producer: claims units (prefetching the next unit's block ids
//               and queries), writes Q, issues the TMA copies
//   warp 5      MMA issuer (one lane), polling for whichever MMA group is ready
//   warps 6-9   epilogue (thread = dimension row of O^T, double-buffered)
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int kHead = kDecodeHeadSize;                       // 128
constexpr int kBlk = kDecodeBlockSize;                       // 16 tokens per cache block
// Blocks per partition (a work unit's context span; partitions are merged by
// a second kernel).  Up to 64: the producer warp holds two block ids a lane.
constexpr int kPartBlocks = 64;
static_assert(kPartBlocks % 8 == 0 && kPartBlocks <= 64, "partition size");
constexpr int kPartTokens = kPartBlocks * kBlk;
constexpr int kStepBlocks = 8;                               // 128 tokens per step
constexpr int kStepsPerPart = kPartBlocks / kStepBlocks;     // 8
constexpr int kNCols = 16;                                   // query heads per MMA (N)
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 64;     // S^T 2 x 16 | O^T 2 x 16
constexpr uint32_t kColS = 0, kColO = 32;

constexpr int kBox = 2048;                          // one K box (a V box is two)
constexpr int kStepK = 2 * kStepBlocks * kBox;      // 32 KB of K boxes
constexpr int kStepBytes = 2 * kStepK;              // K and V of a step
constexpr int kSlots = 3;                           // steps in flight
constexpr int kQBytes = kHead * kNCols * 2;         // 4 KB: Q as [16 d-groups][16 heads][8]
constexpr int kPBytes = 128 * kNCols * 2;           // 4 KB: P as [16 token groups][16 heads][8]
// Up to this many sequences, units are numbered densely from a prefix sum of
// the sequences' partition counts kept in shared memory; beyond it, units are
// (partition, sequence, ...) triples of which those past a context are empty.
constexpr int kDenseSeqs = 1024;
constexpr int kOffRing = 0;
constexpr int kOffQ = kOffRing + kSlots * kStepBytes;     // 2 buffers
constexpr int kOffP = kOffQ + 2 * kQBytes;                // 2 buffers
constexpr int kOffRed = kOffP + 2 * kPBytes;              // [2][4 warps][16] floats
constexpr int kOffStats = kOffRed + 2 * 4 * kNCols * 4;   // UnitStats [2]
constexpr int kOffSeq = kOffStats + 1024;                 // int2 [kDenseSeqs + 1]
constexpr int kOffPart = kOffSeq + (kDenseSeqs + 32) * 8;  // int16 [kDenseSeqs]: ragged tails
constexpr int kOffBins = kOffPart + kDenseSeqs * 2;       // int [16]: tails per step count
constexpr int kOffBar = kOffBins + 64;
constexpr int kSmemBytes = kOffBar + 512;
constexpr int kAlloc = kSmemBytes + 1024;
static_assert(kAlloc <= 227 * 1024, "shared memory budget");

constexpr int kItemSlots = 4;
enum : int {
  kBarKFull = 0,       // + slot (3): the step's K boxes have landed
  kBarSlotFree = 3,    // + slot (3)
  kBarQFull = 6,       // + buffer (2)
  kBarQEmpty = 8,      // + buffer (2)
  kBarSFull = 10,      // + S buffer (2)
  kBarPReady = 12,     // + P buffer (2), 4 softmax warps
  kBarPVDone = 14,     // + P buffer (2)
  kBarRed = 16,        // + 0/1: the 4 softmax warps' per-step values (count 4)
  kBarDrain = 18,
  kBarItemFull = 19,   // + slot (4)
  kBarItemEmpty = 23,  // + slot (4)
  kBarOFull = 27,      // + O buffer (2): the unit's last P V is done
  kBarOFree = 29,      // + O buffer (2): the epilogue has read O and the stats (count 4)
  kBarStats = 31,      // + O buffer (2): the softmax has written the stats (count 4)
  kBarVFull = 33,      // + slot (3): the step's V boxes have landed
  kNumBars = 36
};
// Arrivals that free an item slot: the MMA thread and the 4 softmax warps.
constexpr int kItemConsumers = 1 + 4;

// What the softmax hands the epilogue at the end of a unit: the unit (s < 0:
// no more units), each head's running maximum m (log2 units) and each softmax
// warp's partial row sums.
struct UnitStats {
  int s, hb, part, ctx;
  float m[kNCols];
  float l[4][kNCols];
};
static_assert(2 * sizeof(UnitStats) <= 1024, "stats area");

struct Misc {
  uint32_t tmem_base;
  int abort;
  int4 item[kItemSlots];   // (sequence or -1 at the end, first head, partition, context)
};
// Misc follows the barriers at the next 16-byte boundary (its int4 items).
constexpr int kOffMisc = kOffBar + (8 * kNumBars + 15) / 16 * 16;
static_assert(kOffMisc % 16 == 0 && alignof(Misc) == 16, "item alignment");
static_assert(kOffMisc + sizeof(Misc) <= kSmemBytes, "barrier area");

// No-swizzle K-major shared-memory descriptor: lbo = byte step between core
// matrices along K, sbo = along M or N.
__device__ __forceinline__ uint64_t desc_k_major(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// 32-byte-swizzle K-major descriptor (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_32B): rows of 32 bytes, sbo = byte step between
// 8-row groups; the leading offset is unused.
__device__ __forceinline__ uint64_t desc_k_major_sw32(uint32_t addr, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (1ull << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (6ull << 61);
}
// Instruction descriptor: bf16 A and B, both K-major, fp32 D, M = 128, N = 16.
constexpr uint32_t kIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | ((kNCols >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *m, int c0, int c1,
                                            int c2, int c3, int c4, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *m, int c0, int c1,
                                            int c2, int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// N consecutive 32-bit TMEM columns of this thread's lane (N = 4, 8, 16),
// waited for.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 16) {
    tmem_ld16(taddr, r);
  } else if constexpr (N == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  } else {
    static_assert(N == 4, "4, 8 or 16 columns");
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  }
}
// Stores N columns and waits for the store.
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[N]) {
  if constexpr (N == 16) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
        "%10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
  } else if constexpr (N == 8) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
        : "memory");
  } else {
    static_assert(N == 4, "4, 8 or 16 columns");
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t ph) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, ph) && globaltimer_ns() - t0 < kWaitLimitNs) {
  }
}

__device__ __forceinline__ int partitions_of(int ctx) {
  const int n_blocks = (max(ctx, 0) + kBlk - 1) / kBlk;
  return (n_blocks + kPartBlocks - 1) / kPartBlocks;
}
// Steps (of 8 blocks) of partition `part` of a context of ctx tokens.
__device__ __forceinline__ int steps_of(int part, int ctx) {
  const int n_blocks = (max(ctx, 0) + kBlk - 1) / kBlk;
  const int pb = min(n_blocks - part * kPartBlocks, kPartBlocks);
  return pb > 0 ? (pb + kStepBlocks - 1) / kStepBlocks : 0;
}

// A claimed unit: sequence s (-1: none left), cached head kvh, first query
// head hb of its slice, partition part, context length ctx.
struct Unit {
  int s, kvh, hb, part, ctx;
};

// Unit numbering.  Units of one (sequence, partition) pair are its cached
// heads' slices, next to each other so that a cached head's second slice is
// read from L2.
// Dense (longest first, so that the units claimed last are the shortest and
// the CTAs run out of work together): first every full partition
// (kPartTokens tokens), numbered sequence-major from the prefix sum seq[s].x
// of the sequences' full-partition counts (seq[s].y = context length); then
// each sequence's ragged last partition, if it has one, in the order of
// tail[] -- by step count, longest first.  seq[num_seqs] = (number of full
// partitions, number of ragged ones).  No unit is empty.
// Sparse: pairs are (partition, sequence) with partitions outermost, and
// those past a sequence's context are empty.
struct Numbering {
  int num_seqs, num_kv_heads, n_sub, group, gs, max_parts;
  bool dense;
  const int2 *seq;
  const int16_t *tail;
  const int *context_lens;
  __device__ int per_pair() const { return num_kv_heads * n_sub; }
  __device__ int n_units() const {
    return (dense ? seq[num_seqs].x + seq[num_seqs].y : max_parts * num_seqs) * per_pair();
  }
  // Unit w (< n_units) -> u; returns false if it is an empty unit.
  __device__ bool decode(int w, Unit &u) const {
    const int p = w / per_pair(), rem = w - p * per_pair();
    u.kvh = rem / n_sub;
    u.hb = u.kvh * group + (rem - u.kvh * n_sub) * gs;
    if (dense) {
      const int n_full = seq[num_seqs].x;
      if (p < n_full) {
        int lo = 0, hi = num_seqs - 1;   // the last s with seq[s].x <= p
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (seq[mid].x <= p) lo = mid; else hi = mid - 1;
        }
        u.s = lo;
        u.part = p - seq[lo].x;
      } else {
        u.s = tail[p - n_full];
        u.part = seq[u.s].y / kPartTokens;
      }
      u.ctx = seq[u.s].y;
      return true;
    }
    u.part = p / num_seqs;
    u.s = p - u.part * num_seqs;
    u.ctx = context_lens[u.s];
    return u.part < partitions_of(u.ctx);
  }
};

// Steps (128 tokens) in the ragged last partition of a context of c tokens;
// 0 if it has none.
__device__ __forceinline__ int tail_steps(int c) {
  if (c <= 0) return 0;
  const int r = c % kPartTokens;
  return (r + kStepBlocks * kBlk - 1) / (kStepBlocks * kBlk);
}

// NC = the query heads of a slice the softmax and epilogue handle (4, 8 or
// 16 >= gs); MMA columns past NC hold zero P and are never read back.
template <int NC>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_gqa_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_v,
                               const uint16_t *__restrict__ q,
                               const int *__restrict__ block_tables,
                               const int *__restrict__ context_lens, uint16_t *__restrict__ out,
                               float *__restrict__ ws_o, float *__restrict__ ws_ml,
                               int *__restrict__ sched, int num_seqs,
                               int num_heads, int num_kv_heads, int group, int gs, int max_blocks,
                               int max_parts, float qscale, int *__restrict__ dev_status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  auto bar = [&](int i) { return s_base + kOffBar + 8u * i; };
  Misc *misc = reinterpret_cast<Misc *>(smem + kOffMisc);
  volatile int *abort_flag = &misc->abort;
  int2 *seq = reinterpret_cast<int2 *>(smem + kOffSeq);
  UnitStats *stats = reinterpret_cast<UnitStats *>(smem + kOffStats);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Numbering nb;
  nb.num_seqs = num_seqs;
  nb.num_kv_heads = num_kv_heads;
  nb.n_sub = group / gs;
  nb.group = group;
  nb.gs = gs;
  nb.max_parts = max_parts;
  nb.dense = num_seqs <= kDenseSeqs;
  nb.seq = seq;
  int16_t *tail = reinterpret_cast<int16_t *>(smem + kOffPart);
  int *bins = reinterpret_cast<int *>(smem + kOffBins);
  nb.tail = tail;
  nb.context_lens = context_lens;

  // P columns past NC are never written: zero both P buffers once.
  for (int i = threadIdx.x; i < 2 * kPBytes / 16; i += kThreads)
    reinterpret_cast<uint4 *>(smem + kOffP)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(bar(kBarKFull + i), 1);
      mbar_init(bar(kBarVFull + i), 1);
      mbar_init(bar(kBarSlotFree + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarQFull + i), 1);
      mbar_init(bar(kBarQEmpty + i), 1);
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarPReady + i), 4);
      mbar_init(bar(kBarPVDone + i), 1);
      mbar_init(bar(kBarRed + i), 4);
      mbar_init(bar(kBarOFull + i), 1);
      mbar_init(bar(kBarOFree + i), 4);
      mbar_init(bar(kBarStats + i), 4);
    }
    mbar_init(bar(kBarDrain), 1);
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(bar(kBarItemFull + i), 1);
      mbar_init(bar(kBarItemEmpty + i), kItemConsumers);
    }
    misc->abort = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&misc->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  // Launched as a programmatic dependent of the kernel before it on the
  // stream (the previous call's merge kernel, say): the set-up above overlaps
  // that kernel's tail; no global memory is read or written before this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (nb.dense) {
    // Full-partition counts per sequence, then their exclusive prefix sum
    // (warp 0); warp 9 - t counts the ragged tails of t steps (t = 1 .. 8),
    // then lists them after the longer ones, in sequence order.  Sequences
    // with no context get zero outputs here, from CTA 0.
    for (int i = threadIdx.x; i < num_seqs; i += kThreads) {
      const int c = context_lens[i];
      seq[i] = make_int2(c > 0 ? c / kPartTokens : 0, c);
      if (c <= 0 && blockIdx.x == 0) {
        uint4 *o = reinterpret_cast<uint4 *>(out + static_cast<int64_t>(i) * num_heads * kHead);
        for (int j = 0; j < num_heads * kHead / 8; ++j) o[j] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    __syncthreads();
    const int t_steps = 9 - warp;   // warps 1 .. 8: tails of 8 .. 1 steps
    if (warp == 0) {
      int carry = 0;
      for (int base = 0; base < num_seqs; base += 32) {
        const int i = base + lane;
        const int v = i < num_seqs ? seq[i].x : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int t = __shfl_up_sync(~0u, incl, off);
          if (lane >= off) incl += t;
        }
        if (i < num_seqs) seq[i].x = carry + incl - v;
        carry += __shfl_sync(~0u, incl, 31);
      }
      if (lane == 0) seq[num_seqs].x = carry;
    } else if (warp <= 8) {
      int n = 0;
      for (int base = 0; base < num_seqs; base += 32) {
        const int i = base + lane;
        n += __popc(__ballot_sync(~0u, i < num_seqs && tail_steps(seq[i].y) == t_steps));
      }
      if (lane == 0) bins[t_steps] = n;
    }
    __syncthreads();
    if (warp >= 1 && warp <= 8) {
      int at = 0;   // tails with more steps come first
      for (int t = t_steps + 1; t <= kStepsPerPart; ++t) at += bins[t];
      for (int base = 0; base < num_seqs; base += 32) {
        const int i = base + lane;
        const bool mine = i < num_seqs && tail_steps(seq[i].y) == t_steps;
        const uint32_t m = __ballot_sync(~0u, mine);
        if (mine) tail[at + __popc(m & ((1u << lane) - 1u))] = static_cast<int16_t>(i);
        at += __popc(m);
      }
      if (warp == 1 && lane == 0) {
        int n_tails = 0;
        for (int t = 1; t <= kStepsPerPart; ++t) n_tails += bins[t];
        seq[num_seqs].y = n_tails;
      }
    }
  }
  __syncthreads();
  const int n_units = nb.n_units();
  // The merge kernel may be scheduled now: its threads wait (griddepcontrol)
  // until this grid has finished and its writes are visible.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  auto read_item = [&](int k, int4 &it) -> bool {
    if (!mbar_wait(bar(kBarItemFull + k % kItemSlots), (k / kItemSlots) & 1, abort_flag))
      return false;
    const volatile int *p = reinterpret_cast<const volatile int *>(&misc->item[k % kItemSlots]);
    it = make_int4(p[0], p[1], p[2], p[3]);
    return true;
  };

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // Hands each unit on through the item slots (then a final s = -1), writes
    // its Q, and streams its steps' K and V.  While a unit streams, the next
    // one is already claimed with its block ids and queries in registers, and
    // the claim of the one after is in flight.
    int n_active = 0, n_steps_loaded = 0;
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    Unit nxt;
    int lane_pb = 0;      // block id of the unit's block `lane` (the last one past the context)
    int lane_pb2 = 0;     // and of its block 32 + lane
    uint4 qv[8];          // 16-byte chunk lane + 32 i of the unit's [16 heads][128] queries
    int w_pending = 0;    // lane 0: the claim in flight
    bool pending = false;
    auto request = [&]() {
      if (lane == 0) w_pending = atomicAdd(sched, 1);
      pending = true;
    };
    // Takes the claim in flight into nxt (claiming on past empty units).
    auto finish = [&]() {
      for (;;) {
        const int w = __shfl_sync(~0u, w_pending, 0);
        pending = false;
        if (w >= n_units) {
          nxt.s = -1;
          return;
        }
        if (nb.decode(w, nxt)) return;
        if (nxt.part == 0 && nxt.ctx <= 0) {   // no context: zero outputs
          uint16_t *o = out + (static_cast<int64_t>(nxt.s) * num_heads + nxt.hb) * kHead;
          for (int i = lane; i < gs * kHead; i += 32) o[i] = 0;
        }
        request();
      }
    };
    auto prefetch = [&]() {
      if (nxt.s < 0) return;
      const int n_blocks = (nxt.ctx + kBlk - 1) / kBlk;
      const int *bt = block_tables + static_cast<int64_t>(nxt.s) * max_blocks;
      lane_pb = bt[min(nxt.part * kPartBlocks + lane, n_blocks - 1)];
      if (kPartBlocks > 32) lane_pb2 = bt[min(nxt.part * kPartBlocks + 32 + lane, n_blocks - 1)];
      const uint4 *qr = reinterpret_cast<const uint4 *>(
          q + (static_cast<int64_t>(nxt.s) * num_heads + nxt.hb) * kHead);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = lane + 32 * i;   // head c / 16, d-group c % 16
        qv[i] = (c >> 4) < gs ? __ldg(qr + c) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    request();
    finish();
    prefetch();
    if (nxt.s >= 0) request();
    for (int k = 0; ok; ++k) {
      const Unit cur = nxt;
      const int cur_pb = lane_pb, cur_pb2 = lane_pb2;
      if (lane == 0) {
        const int slot = k % kItemSlots;
        ok = mbar_wait(bar(kBarItemEmpty + slot), ((k / kItemSlots) & 1) ^ 1, abort_flag);
        if (ok) {
          misc->item[slot] = make_int4(cur.s, cur.hb, cur.part, cur.ctx);
          mbar_arrive(bar(kBarItemFull + slot));
        }
      }
      ok = __shfl_sync(~0u, ok, 0);
      if (!ok || cur.s < 0) break;
      const int n_steps = steps_of(cur.part, cur.ctx);
      for (int st = 0; st < n_steps; ++st) {
        const int slot = n_steps_loaded % kSlots;
        if (lane == 0)
          ok = mbar_wait(bar(kBarSlotFree + slot), ((n_steps_loaded / kSlots) & 1) ^ 1, abort_flag);
        if (!(ok = __shfl_sync(~0u, ok, 0))) break;
        const uint32_t kfull = bar(kBarKFull + slot), vfull = bar(kBarVFull + slot);
        if (lane == 0) {
          mbar_arrive_expect_tx(kfull, kStepK);
          mbar_arrive_expect_tx(vfull, kStepBytes - kStepK);
        }
        __syncwarp();
        // Lane b < 8 copies block b of the step: its two K boxes, then (after
        // every lane's K) its V box, on separate barriers so that Q K^T can
        // start while V is still arriving.  Blocks past the context repeat the
        // last block: finite or not, their tokens get zero weight and zero
        // values.
        const uint32_t base = s_base + kOffRing + slot * kStepBytes + (2 * (lane & 7)) * kBox;
        const int bi = st * kStepBlocks + (lane & 7);   // block of the partition
        const int pb0 = __shfl_sync(~0u, cur_pb, bi & 31);
        const int pb = (kPartBlocks > 32 && bi >= 32) ? __shfl_sync(~0u, cur_pb2, bi & 31) : pb0;
        if (lane < kStepBlocks) {
          tma_load_5d(base, &tm_k, 0, 0, 0, cur.kvh, pb, kfull);
          tma_load_5d(base + kBox, &tm_k, 0, 1, 0, cur.kvh, pb, kfull);
        }
        __syncwarp();
        if (lane < kStepBlocks) tma_load_4d(base + kStepK, &tm_v, 0, 0, cur.kvh, pb, vfull);
        ++n_steps_loaded;
        if (st == 0) {
          // With the first step's copies under way: Q into buffer n_active & 1
          // once the MMA thread's last Q K^T of the unit two before has read
          // it ([d-group][head][8], heads past the slice 0), then the next
          // unit's claim and loads.
          const int qb = n_active & 1;
          if (lane == 0)
            ok = mbar_wait(bar(kBarQEmpty + qb), ((n_active >> 1) & 1) ^ 1, abort_flag);
          if (!(ok = __shfl_sync(~0u, ok, 0))) break;
          uint8_t *qs = smem + kOffQ + qb * kQBytes;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = lane + 32 * i;
            *reinterpret_cast<uint4 *>(qs + ((c & 15) * kNCols + (c >> 4)) * 16) = qv[i];
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarQFull + qb));
          ++n_active;
          finish();
          prefetch();
          if (nxt.s >= 0) request();
        }
      }
    }
    // A claim still in flight (after an abort) completes before the CTA's exit
    // is counted, so that the counter reset cannot be overtaken.
    if (pending && __shfl_sync(~0u, w_pending, 0) == -1) misc->abort = 1;
    if (!ok && lane == 0)
      for (int i = (n_steps_loaded > kSlots ? n_steps_loaded - kSlots : 0); i < n_steps_loaded;
           ++i) {
        drain_wait(bar(kBarKFull + i % kSlots), (i / kSlots) & 1);
        drain_wait(bar(kBarVFull + i % kSlots), (i / kSlots) & 1);
      }
  } else if (warp == 5) {
    if (elect_one()) {
      // ------------------------------------------------------------ MMA issuer
      // Issues whichever MMA group is ready, never waiting on one while the
      // other could go: P V of step gp once its P is in shared memory (and,
      // for a unit's first step, once the epilogue has freed the unit's O
      // buffer), and Q K^T of step gq (at most two ahead of P V: S is
      // double-buffered) once its keys have landed.  Items are released as
      // soon as they are read; a unit's step count stays in a ring (at most
      // three units lie between the two cursors).
      int kq = 0, jq = 0, nq = 0, n_qunits = 0, gq = 0;     // Q K^T cursor
      int jp = 0, gp = 0, u_head = 0, u_tail = 0;           // P V cursor (u_head: its unit)
      int unit_steps[4];
      bool more = true, q_ready = false;
      uint64_t t_idle = 0;
      uint32_t idle = 0;
      for (;;) {
        bool progress = false;
        const int ob = u_head & 1;
        if (gp < gq && mbar_try_wait(bar(kBarPReady + (gp & 1)), (gp >> 1) & 1) &&
            mbar_try_wait(bar(kBarVFull + gp % kSlots), (gp / kSlots) & 1) &&
            (jp > 0 || mbar_try_wait(bar(kBarOFree + ob), ((u_head >> 1) & 1) ^ 1))) {
          tc_fence_after();
          const uint32_t vbase = s_base + kOffRing + (gp % kSlots) * kStepBytes + kStepK;
          const uint32_t pbase = s_base + kOffP + (gp & 1) * kPBytes;
#pragma unroll
          for (int blk = 0; blk < kStepBlocks; ++blk)
            mma_ss(tmem + kColO + kNCols * ob, desc_k_major_sw32(vbase + blk * 2 * kBox, 256),
                   desc_k_major(pbase + blk * 512, 256, 128), kIdesc,
                   (jp == 0 && blk == 0) ? 0u : 1u);
          mma_commit(bar(kBarPVDone + (gp & 1)));
          mma_commit(bar(kBarSlotFree + gp % kSlots));
          ++gp;
          if (++jp == unit_steps[u_head & 3]) {
            mma_commit(bar(kBarOFull + ob));   // the unit's O is complete
            ++u_head;
            jp = 0;
          }
          progress = true;
        }
        if (more && gq < gp + 2) {
          if (jq == nq) {
            if (mbar_try_wait(bar(kBarItemFull + kq % kItemSlots), (kq / kItemSlots) & 1)) {
              const volatile int *it =
                  reinterpret_cast<const volatile int *>(&misc->item[kq % kItemSlots]);
              const int s_it = it[0], part_it = it[2], ctx_it = it[3];
              mbar_arrive(bar(kBarItemEmpty + kq % kItemSlots));
              ++kq;
              if (s_it < 0) {
                more = false;
              } else {
                nq = steps_of(part_it, ctx_it);
                unit_steps[u_tail++ & 3] = nq;
                jq = 0;
                q_ready = false;
              }
              progress = true;
            }
          } else {
            if (!q_ready)
              q_ready = mbar_try_wait(bar(kBarQFull + (n_qunits & 1)), (n_qunits >> 1) & 1);
            if (q_ready && mbar_try_wait(bar(kBarKFull + gq % kSlots), (gq / kSlots) & 1)) {
              tc_fence_after();
              const uint32_t kbase = s_base + kOffRing + (gq % kSlots) * kStepBytes;
              const uint32_t qbase = s_base + kOffQ + (n_qunits & 1) * kQBytes;
#pragma unroll
              for (int kk = 0; kk < kHead / 16; ++kk)
                mma_ss(tmem + kColS + kNCols * (gq & 1), desc_k_major(kbase + kk * 256, 128, 2048),
                       desc_k_major(qbase + kk * 512, 256, 128), kIdesc, kk > 0 ? 1u : 0u);
              mma_commit(bar(kBarSFull + (gq & 1)));
              if (++jq == nq) {
                mma_commit(bar(kBarQEmpty + (n_qunits & 1)));   // the unit's Q has been read
                ++n_qunits;
              }
              ++gq;
              progress = true;
            }
          }
        }
        if (!more && gp == gq) break;
        // Bounded idling: give up (and tell the other roles) after the wait limit.
        if (progress) {
          idle = 0;
        } else if ((++idle & 15u) == 0) {
          if (*abort_flag) break;
          const uint64_t now = globaltimer_ns();
          if (idle == 16) {
            t_idle = now;
          } else if (now - t_idle > kWaitLimitNs) {
            *abort_flag = 1;
            break;
          }
        }
      }
      mma_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- softmax
    // Thread r = token row r of S^T.  At the end of a unit the running maxima
    // and the warps' partial row sums go to the epilogue warps; the next unit
    // starts at once (O is double-buffered in TMEM).
    const int r = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float *red = reinterpret_cast<float *>(smem + kOffRed);   // [2][4][16]
    int g = 0, n_red = 0;
    bool ok = true;
    // Cross-warp exchange: every warp's lane 0 has stored its values in
    // red[buf][warp][*]; returns buf once all four have (-1 on abort).
    auto red_sync = [&]() -> int {
      const int buf = n_red & 1;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarRed + buf));
      if (!mbar_wait(bar(kBarRed + buf), (n_red >> 1) & 1, abort_flag)) return -1;
      ++n_red;
      return buf;
    };
    for (int k = 0; ok; ++k) {
      const int ui = k, ob = ui & 1;   // units with steps, in order; their O buffer
      int4 it;
      if (!(ok = read_item(k, it))) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarItemEmpty + k % kItemSlots));
      if (it.x < 0) {
        // No more units: say so to the epilogue through the stats slot.
        if (!(ok = mbar_wait(bar(kBarOFree + ob), ((ui >> 1) & 1) ^ 1, abort_flag))) break;
        if (threadIdx.x == 0) stats[ob].s = -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarStats + ob));
        break;
      }
      const int part = it.z, ctx = it.w;
      const int n_steps = steps_of(part, ctx);
      const uint32_t o_tmem = tmem + lane_off + kColO + kNCols * ob;
      float m[NC], lp[NC];          // running max (log2 units); this token's partial sums
#pragma unroll
      for (int hh = 0; hh < NC; ++hh) {
        m[hh] = -INFINITY;
        lp[hh] = 0.f;
      }
      for (int j = 0; j < n_steps; ++j, ++g) {
        const int b = g & 1;
        if (!(ok = mbar_wait(bar(kBarSFull + b), (g >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        uint32_t sv[NC];
        tmem_ld_cols<NC>(tmem + lane_off + kColS + kNCols * b, sv);
        const bool valid = part * kPartTokens + j * 128 + r < ctx;
        if (j == n_steps - 1 && __any_sync(~0u, !valid)) {
          // Cache slots past the context hold whatever was there before; a
          // zero weight does not cancel a NaN or an infinity, so the value rows
          // of those tokens are cleared once the step's V boxes have landed.
          if (!(ok = mbar_wait(bar(kBarVFull + g % kSlots), (g / kSlots) & 1, abort_flag))) break;
          if (!valid) {
            // Token r's value of dimension d: block r / 16's box, row d, 16-byte
            // chunk (token half) swizzled by bit 2 of d.
            uint8_t *vt = smem + kOffRing + (g % kSlots) * kStepBytes + kStepK +
                          (r >> 4) * (2 * kBox) + (r & 7) * 2;
            const int half = (r >> 3) & 1;
#pragma unroll 16
            for (int d = 0; d < kHead; ++d)
              *reinterpret_cast<uint16_t *>(vt + d * 32 + ((half ^ (d >> 2)) & 1) * 16) = 0;
          }
        }
        float x[NC];
#pragma unroll
        for (int hh = 0; hh < NC; ++hh) {
          x[hh] = valid ? __uint_as_float(sv[hh]) * qscale : -INFINITY;
          float v = x[hh];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(~0u, v, off));
          if (lane == 0) red[(n_red & 1) * 64 + warp * kNCols + hh] = v;
        }
        const int buf = red_sync();
        ok = buf >= 0;
        if (!ok) break;
        float alpha[NC];
        bool rescale = false;
#pragma unroll
        for (int hh = 0; hh < NC; ++hh) {
          const float *rw = red + buf * 64 + hh;
          const float smax = fmaxf(fmaxf(rw[0], rw[kNCols]), fmaxf(rw[2 * kNCols], rw[3 * kNCols]));
          const float m_new = fmaxf(m[hh], smax);   // finite: every step has a visible token
          alpha[hh] = ex2_approx(m[hh] - m_new);    // 0 on the first step
          rescale |= j > 0 && alpha[hh] != 1.f;
          const float p = ex2_approx(x[hh] - m_new);
          lp[hh] = lp[hh] * alpha[hh] + p;
          m[hh] = m_new;
          x[hh] = p;
        }
        // P [token group][head][8 tokens]: this token's value for each head.
        {
          uint8_t *pr = smem + kOffP + b * kPBytes + (r >> 3) * (kNCols * 16) + (r & 7) * 2;
#pragma unroll
          for (int e = 0; e < NC / 2; ++e) {
            const uint32_t pk = pack_bf16x2(x[2 * e], x[2 * e + 1]);
            *reinterpret_cast<uint16_t *>(pr + (2 * e) * 16) = static_cast<uint16_t>(pk);
            *reinterpret_cast<uint16_t *>(pr + (2 * e + 1) * 16) = static_cast<uint16_t>(pk >> 16);
          }
        }
        // O^T (this thread's dimension row) picks up the new maxima once the
        // previous step's P V, from the other buffer, has finished.
        if (rescale) {
          if (!(ok = mbar_wait(bar(kBarPVDone + (b ^ 1)), ((g - 1) >> 1) & 1, abort_flag))) break;
          tc_fence_after();
          uint32_t ov[NC];
          tmem_ld_cols<NC>(o_tmem, ov);
#pragma unroll
          for (int hh = 0; hh < NC; ++hh) ov[hh] = __float_as_uint(__uint_as_float(ov[hh]) * alpha[hh]);
          tmem_st_cols<NC>(o_tmem, ov);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPReady + b));
      }
      if (!ok) break;
      // Hand the unit over: this warp's row sums, and (warp 0) the maxima.
#pragma unroll
      for (int hh = 0; hh < NC; ++hh) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lp[hh] += __shfl_xor_sync(~0u, lp[hh], off);
      }
      if (!(ok = mbar_wait(bar(kBarOFree + ob), ((ui >> 1) & 1) ^ 1, abort_flag))) break;
      if (lane == 0) {
        UnitStats &st = stats[ob];
#pragma unroll
        for (int hh = 0; hh < NC; ++hh) st.l[warp][hh] = lp[hh];
        if (warp == 0) {
          st.s = it.x;
          st.hb = it.y;
          st.part = part;
          st.ctx = ctx;
#pragma unroll
          for (int hh = 0; hh < NC; ++hh) st.m[hh] = m[hh];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarStats + ob));
    }
  } else {
    // --------------------------------------------------------------- epilogue
    // Warps 6-9: thread r = dimension row r of O^T (TMEM lane quarter warp % 4).
    // One-partition units are written out; the others leave their unscaled
    // row, maximum and sum in the workspace for the merge kernel.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    for (int ui = 0; ok; ++ui) {
      const int ob = ui & 1;
      if (!(ok = mbar_wait(bar(kBarStats + ob), (ui >> 1) & 1, abort_flag))) break;
      const UnitStats &st = stats[ob];
      const int s = st.s;
      if (s < 0) break;
      const int hb = st.hb, part = st.part, ctx = st.ctx;
      float mm[NC], L[NC];
#pragma unroll
      for (int hh = 0; hh < NC; ++hh) {
        mm[hh] = st.m[hh];
        L[hh] = st.l[0][hh] + st.l[1][hh] + st.l[2][hh] + st.l[3][hh];
      }
      if (!(ok = mbar_wait(bar(kBarOFull + ob), (ui >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t ov[NC];
      tmem_ld_cols<NC>(tmem + lane_off + kColO + kNCols * ob, ov);   // row r = dimension r
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarOFree + ob));   // O and the stats are read
      const int n_parts = partitions_of(ctx);
      const int64_t h0 = static_cast<int64_t>(s) * num_heads + hb;   // first (s, h) row
      if (n_parts == 1) {
#pragma unroll
        for (int hh = 0; hh < NC; ++hh)
          if (hh < gs)
            out[(h0 + hh) * kHead + r] =
                static_cast<uint16_t>(pack_bf16x2(__uint_as_float(ov[hh]) / L[hh], 0.f) & 0xffffu);
        continue;
      }
#pragma unroll
      for (int hh = 0; hh < NC; ++hh) {
        if (hh < gs) {
          const int64_t slot = (h0 + hh) * max_parts + part;
          ws_o[slot * kHead + r] = __uint_as_float(ov[hh]);
          if (r == 0) *reinterpret_cast<float2 *>(ws_ml + slot * 2) = make_float2(mm[hh], L[hh]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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

// Merges the partitions of every (sequence, query head) with more than one
// (eq. (4) of "Flash Attention", section "Online Softmax", across
// partitions): one warp per row, lane l holding dimensions 4l .. 4l + 3.
__global__ void __launch_bounds__(256)
    paged_decode_merge_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_ml,
                              const int *__restrict__ context_lens, uint16_t *__restrict__ out,
                              int num_seqs, int num_heads, int max_parts) {
  // Launched as a programmatic dependent of the decode kernel: wait for it to
  // finish (its workspace writes are then visible).  The next decode call may
  // be scheduled once every block of this kernel has begun.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(num_seqs) * num_heads) return;
  const float *ml = ws_ml + row * max_parts * 2;
  const float *o = ws_o + row * max_parts * kHead + 4 * lane;
  // The first kSpec partitions' (max, sum) pairs and output slices are loaded
  // together with the context length (one round trip to memory instead of
  // three); those past the row's partition count are loaded but not used.
  constexpr int kSpec = 4;
  float2 ml_s[kSpec];
  float4 o_s[kSpec];
  const int ctx = context_lens[row / num_heads];
#pragma unroll
  for (int p = 0; p < kSpec; ++p) {
    if (p < max_parts) {
      ml_s[p] = __ldcg(reinterpret_cast<const float2 *>(ml) + p);
      o_s[p] = __ldcg(reinterpret_cast<const float4 *>(o + static_cast<int64_t>(p) * kHead));
    }
  }
  const int n_parts = partitions_of(ctx);
  if (n_parts <= 1) return;   // written by the decode kernel
  if (n_parts <= kSpec) {
    float M = ml_s[0].x;
#pragma unroll
    for (int p = 1; p < kSpec; ++p)
      if (p < n_parts) M = fmaxf(M, ml_s[p].x);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int p = 0; p < kSpec; ++p) {
      if (p < n_parts) {
        const float f = ex2_approx(ml_s[p].x - M);
        L += ml_s[p].y * f;
        acc.x += f * o_s[p].x;
        acc.y += f * o_s[p].y;
        acc.z += f * o_s[p].z;
        acc.w += f * o_s[p].w;
      }
    }
    const float inv = 1.f / L;
    uint2 packed;
    packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(out + row * kHead + 4 * lane) = packed;
    return;
  }
  float M = -INFINITY;
  for (int p = lane; p < n_parts; p += 32) M = fmaxf(M, __ldcg(ml + 2 * p));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(~0u, M, off));
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int p0 = 0; p0 < n_parts; p0 += 32) {
    float f = 0.f;
    if (p0 + lane < n_parts) {
      const float2 v = __ldcg(reinterpret_cast<const float2 *>(ml) + p0 + lane);
      f = ex2_approx(v.x - M);
      L += v.y * f;
    }
    const int cnt = min(32, n_parts - p0);
#pragma unroll 4
    for (int j = 0; j < cnt; ++j) {
      const float fj = __shfl_sync(~0u, f, j);
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(o + static_cast<int64_t>(p0 + j) * kHead));
      acc.x += fj * v.x;
      acc.y += fj * v.y;
      acc.z += fj * v.z;
      acc.w += fj * v.w;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(~0u, L, off);
  const float inv = 1.f / L;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2 *>(out + row * kHead + 4 * lane) = packed;
}

int g_num_sms[64] = {};

template <int NC>
cudaError_t launch_nc(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const void *q,
                      const int *block_tables, const int *context_lens, void *out, int num_seqs,
                      int num_heads, int num_kv_heads, int group, int gs, int max_blocks,
                      int max_parts, float qscale, float *ws_o, float *ws_ml, int *sched,
                      int *dev_status, int grid, cudaStream_t stream) {
  const cudaError_t e = cudaFuncSetAttribute(paged_decode_gqa_tc_kernel<NC>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (e != cudaSuccess) return e;
  {
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
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, paged_decode_gqa_tc_kernel<NC>, tm_k, tm_v, static_cast<const uint16_t *>(q),
        block_tables, context_lens, static_cast<uint16_t *>(out), ws_o, ws_ml, sched, num_seqs,
        num_heads, num_kv_heads, group, gs, max_blocks, max_parts, qscale, dev_status);
    if (e != cudaSuccess) return e;
  }
  if (max_parts > 1) {
    // Programmatic dependent launch: the merge grid is scheduled while the
    // decode grid runs and starts its work when that grid completes, which
    // hides its launch latency.
    const long long rows = static_cast<long long>(num_seqs) * num_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, paged_decode_merge_kernel,
                                             static_cast<const float *>(ws_o),
                                             static_cast<const float *>(ws_ml), context_lens,
                                             static_cast<uint16_t *>(out), num_seqs, num_heads,
                                             max_parts);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace

bool decode_gqa_tc_supported(int group) { return group >= 2 && (group <= 16 || group % 16 == 0); }

cudaError_t launch_paged_decode_gqa_tc(const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                       const void *q, const int *block_tables,
                                       const int *context_lens, void *out, int num_seqs,
                                       int num_heads, int num_kv_heads, int max_blocks,
                                       float scale, float *workspace, int *sched,
                                       int *dev_status, cudaStream_t stream) {
  const int group = num_heads / num_kv_heads;
  if (!decode_gqa_tc_supported(group) || group * num_kv_heads != num_heads)
    return cudaErrorInvalidValue;
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
  const int gs = group <= kNCols ? group : kNCols;
  // Partitions of this kernel (no more than the split-K workspace holds).
  const int max_parts = (max_blocks + kPartBlocks - 1) / kPartBlocks;
  // The most units there can be; the kernel counts the actual ones.
  const long long n_units =
      static_cast<long long>(max_parts) * num_seqs * num_kv_heads * (group / gs);
  if (n_units > 0x7fffffffLL) return cudaErrorInvalidValue;
  const size_t slots = static_cast<size_t>(num_seqs) * num_heads * max_parts;
  float *ws_o = workspace;
  float *ws_ml = ws_o + slots * kHead;
  const float qscale = scale * 1.4426950408889634f;   // scale * log2(e)
  const int grid = static_cast<int>(n_units < g_num_sms[dev] ? n_units : g_num_sms[dev]);
#define FATTN_GQA_TC_ARGS                                                                       \
  tm_k, tm_v, q, block_tables, context_lens, out, num_seqs, num_heads, num_kv_heads, group, gs, \
      max_blocks, max_parts, qscale, ws_o, ws_ml, sched, dev_status, grid, stream
  if (gs <= 4) return launch_nc<4>(FATTN_GQA_TC_ARGS);
  if (gs <= 8) return launch_nc<8>(FATTN_GQA_TC_ARGS);
  return launch_nc<16>(FATTN_GQA_TC_ARGS);
#undef FATTN_GQA_TC_ARGS
}

}  // namespace fattn
