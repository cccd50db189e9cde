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
//   bwd_prep_kernel   D = rowsum(dO * O) and the LSE in log2 units, written
//                     negated per 128-query block as [-LSE2 x 128 | -D x 128]
//                     (rows past N padded with -LSE2 = -inf, -D = 0) so one
//                     bulk copy brings a block's vectors and the packed fp32
//                     FMA/ADD use them as they are; zeroes the fp32 dQ
//                     accumulator
//   bwd_main_kernel   (head dimension 64; 128 runs the pipelined kernel of
//                     bwd_bf16_d128.cu, same arithmetic and workspace)
//                     one CTA per (128-key block j, head); K_j and V_j stay
//                     in shared memory and dK_j, dV_j in TMEM while the CTA
//                     visits every query block i that sees block j (the KV-
//                     outer order of FlashAttention-2's backward).  dQ is
//                     summed across CTAs into an fp32 accumulator [BH][N][d]
//                     (TMA reduce-add of shared-memory tiles here; the d = 128
//                     kernel adds from registers).
//   bwd_dq_kernel     dQ = scale * accumulator, rounded to bf16
//
// bwd_main_kernel roles (384 threads): warp 0 loads with TMA, warp 1 issues
// the MMAs (warps 2-3 only take part in the register split), warps 4-11 are
// two groups of four ("G0" = warps 4-7, "G1" = warps 8-11); warp w owns TMEM
// lanes 32*(w%4) .. +31, G0 the first 64 queries of a step and G1 the last 64.  Per query block i:
//   S^T  = K_j Q_i^T   and   dP^T = V_j dO_i^T        (TMEM, lanes = keys)
//   P^T  = exp2(S^T * scale*log2e - LSE2_i),  dS^T = P^T (dP^T - D_i), packed
//          to bf16 in TMEM inside each group's own fp32 columns; dS also into
//          shared memory in the layout an M-major MMA operand expects
//   dQ_i' = dS K_j                                     (lanes = queries, into
//          TMEM columns the bf16 packing freed)
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i                (A operand from TMEM)
//   each group warp reads its rows of dQ_i' while dV/dK run, stages them in
//   its own shared-memory tile and adds them to the accumulator with a TMA
//   reduce.
// TMEM columns (D = 128): S^T [0,128) -> P^T at [0,32) (G0) and [96,128)
// (G1); dP^T [128,256) -> dS^T at [128,160) and [224,256); dQ' halves at
// [32,96) and [160,224) (D = 64: one N = 64 tile at [32,96)); dV [256,256+D),
// dK [256+D,256+2D).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fattn {
namespace {

constexpr int BM = 128;   // keys per CTA (MMA M of S^T, dP^T, dV, dK)
constexpr int BQ = 128;   // queries per step
constexpr int kGroupWarps = 8;
constexpr int kThreads = 384;        // 12 warps = 3 warpgroups
// Register split (setmaxnreg): the launch gives every thread 168 registers
// (65536 / 384, rounded to 8); the loader/MMA warpgroup drops to 104 and the
// two compute warpgroups rise to 200, so each SM sub-partition, which hosts
// one warp of every warpgroup, needs 104 + 200 + 200 = 3 * 168 registers per
// lane.  The build checks that ptxas gives this kernel exactly 168 at launch.
constexpr uint32_t kRegsLoad = 104, kRegsGroup = 200;
static_assert(kRegsLoad + 2 * kRegsGroup == 3 * 168,
              "the warpgroup register split must use exactly the launch budget");
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kVecFloats = 2 * BQ;   // [LSE2 | D] of one query block

template <int D>
struct BCfg {
  static constexpr int kTileBytes = 128 * D * 2;   // a 128 x D bf16 tile
  static constexpr int kBoxBytes = 128 * 128;      // 128 rows x 128 bytes
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;       // one stage
  static constexpr int kDO = kQ + kTileBytes;      // two stages
  static constexpr int kDS = kDO + 2 * kTileBytes; // dS^T (128 keys x 128 queries bf16)
  static constexpr int kStage = kDS + 128 * 128 * 2;  // 8 x 4 KB dQ' staging tiles
  static constexpr int kVec = kStage + kGroupWarps * 4096;  // [LSE2 | D] f32 of the step
  static constexpr int kBar = kVec + kVecFloats * 4;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  // dQ' = dS K: D/64 tiles of N = 64 columns.
  static constexpr int kDqTiles = D / 64;
  // Columns of dQ' each group warp reads, stages and reduces (32 per round).
  static constexpr int kDqColsPerGroup = D / 2;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

enum : int {
  kBarKV = 0,
  kBarQFull = 1,      // Q tile and the [LSE2 | D] vectors
  kBarQEmpty = 2,
  kBarDOFull = 3,     // +stage
  kBarDOEmpty = 5,    // +stage
  kBarSFull = 7,
  kBarPReady = 8,     // 8 group warps
  kBarDQFull = 9,
  kBarTmemFree = 10,  // 8 group warps: dQ' read out of TMEM
  kBarKVDone = 11,
  kBarDrain = 12,
  kNumBars = 13
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

// One 16-thread group per padded row (bh, i), i < n_qb * 128:
//   i < N:  vec[-LSE2] = -LSE * log2(e), vec[-D] = -rowsum(dO * O), and the
//           row of the dQ accumulator is zeroed
//   i >= N: vec[-LSE2] = -inf, vec[-D] = 0 (padding: P = 0 there).
template <int D>
__global__ void __launch_bounds__(256)
    bwd_prep_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                    const float *__restrict__ lse, float *__restrict__ vec,
                    float *__restrict__ dq_acc, int N, int n_qb, int64_t padded_rows) {
  // The main kernel may be scheduled once every block of this one has begun.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t prow = static_cast<int64_t>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  const int part = threadIdx.x & 15;
  const bool live = prow < padded_rows;
  const int64_t npad = static_cast<int64_t>(n_qb) * BQ;
  const int64_t bh = live ? prow / npad : 0;
  const int i = live ? static_cast<int>(prow - bh * npad) : 0;
  const bool real = live && i < N;
  const int64_t row = bh * N + i;
  float acc = 0.f;
  if (real) {
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
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = part * 4; c < D; c += 64) *reinterpret_cast<float4 *>(dq_acc + row * D + c) = z;
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(~0u, acc, off);
  if (live && part == 0) {
    float *v = vec + (bh * n_qb + i / BQ) * kVecFloats;
    v[i % BQ] = real ? -lse[row] * kLog2e : -INFINITY;
    v[BQ + i % BQ] = real ? -acc : 0.f;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const float *__restrict__ vecs,
                    __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv, int N, int BH,
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
    mbar_init(bar(kBarPReady), kGroupWarps);
    mbar_init(bar(kBarDQFull), 1);
    mbar_init(bar(kBarTmemFree), kGroupWarps);
    mbar_init(bar(kBarKVDone), 1);
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

  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLoad));
  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar(kBarKV), 2 * C::kTileBytes);
      for (int b = 0; b < D / 64; ++b) {
        tma_load_3d(s_base + C::kK + b * C::kBoxBytes, &tm_k, b * 64, k0, bh, bar(kBarKV));
        tma_load_3d(s_base + C::kV + b * C::kBoxBytes, &tm_v, b * 64, k0, bh, bar(kBarKV));
      }
      int nq = 0, ndo = 0;
      bool ok = true;
      for (int s = 0; s < n_steps && ok; ++s) {
        const int qb = i_first + s;
        const int st = s & 1;
        if (!(ok = mbar_wait(bar(kBarDOEmpty + st), ((s >> 1) & 1) ^ 1, abort_flag))) break;
        mbar_arrive_expect_tx(bar(kBarDOFull + st), C::kTileBytes);
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(s_base + C::kDO + st * C::kTileBytes + b * C::kBoxBytes, &tm_do, b * 64,
                      qb * BQ, bh, bar(kBarDOFull + st));
        ndo = s + 1;
        if (!(ok = mbar_wait(bar(kBarQEmpty), (s & 1) ^ 1, abort_flag))) break;
        mbar_arrive_expect_tx(bar(kBarQFull), C::kTileBytes + kVecFloats * 4);
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(s_base + C::kQ + b * C::kBoxBytes, &tm_q, b * 64, qb * BQ, bh,
                      bar(kBarQFull));
        bulk_load(s_base + C::kVec,
                  vecs + (static_cast<int64_t>(bh) * n_qblocks + qb) * kVecFloats,
                  kVecFloats * 4, bar(kBarQFull));
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
      constexpr uint32_t idesc_q = idesc_bf16_f32(BQ, 64, true, true);   // dQ' tiles
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
        // The previous step's dQ' has been read out of TMEM.
        if (s > 0 && !(ok = mbar_wait(bar(kBarTmemFree), (s - 1) & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::kColS, dk_desc + off, dq_kmaj + off, idesc_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::kColDP, dv_desc + off, ddo_kmaj + do_off + off, idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(kBarSFull));
        if (!(ok = mbar_wait(bar(kBarPReady), s & 1, abort_flag))) break;
        tc_fence_after();
        // dQ' = dS K: M = queries (dS^T in shared memory, M-major), N = 64
        // columns of d per tile, K = keys.  Issued first so that its read-out
        // overlaps the dV and dK MMAs.
#pragma unroll 1
        for (int h = 0; h < C::kDqTiles; ++h) {
#pragma unroll 1
          for (int kk = 0; kk < BM / 16; ++kk) {
            const uint32_t off = (kk * 2048) >> 4;
            mma_ss(tmem + (h ? 160u : 32u), dds + off, dk_mn + ((h * C::kBoxBytes) >> 4) + off,
                   idesc_q, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(kBarDQFull));
        // dV += P^T dO, dK += dS^T Q (A from TMEM, 16 queries per MMA; the
        // first 64 queries packed by G0 at +0, the last 64 by G1 at +96).
#pragma unroll 1
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t off = (kk * 2048) >> 4;
          const uint32_t acol = kk < 4 ? kk * 8 : 96 + (kk - 4) * 8;
          mma_ts(tmem + C::kColDV, tmem + C::kColS + acol, ddo_mn + do_off + off, idesc_g,
                 (s > 0 || kk > 0) ? 1u : 0u);
          mma_ts(tmem + C::kColDK, tmem + C::kColDP + acol, dq_mn + off, idesc_g,
                 (s > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(kBarQEmpty));
        mma_commit(bar(kBarDOEmpty + st));
      }
      if (ok) mma_commit(bar(kBarKVDone));
      mma_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsGroup));
    // ------------------------- group warps: P, dS, dQ' read-out, epilogue
    const int gw = warp - 4;                 // 0..7
    const int g = gw >> 2;                   // 0: queries [0,64) of a step, 1: [64,128)
    const int quarter = warp & 3;            // TMEM lane quarter of this warp
    const int lane = threadIdx.x & 31;
    const int r = quarter * 32 + lane;       // key row of S^T; query row of dQ'
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int key = k0 + r;
    const float c = scale * kLog2e;
    const float *vec = reinterpret_cast<const float *>(smem + C::kVec);
    uint8_t *ds_smem = smem + C::kDS;
    // This warp's 4 KB dQ' staging tile: 32 queries x 32 fp32, 128-byte rows
    // with the 128-byte swizzle, the box of the accumulator's tensor map.
    uint8_t *stage = smem + C::kStage + gw * 4096;
    const uint32_t stage_u32 = s_base + C::kStage + gw * 4096;
    const uint32_t dq_col = D == 128 ? (g ? 160u : 32u) : 32u + 32u * g;  // TMEM column
    const int dq_d0 = D == 128 ? 64 * g : 32 * g;                         // first d column
    constexpr int kRounds = C::kDqColsPerGroup / 32;
    bool ok = true;
    for (int s = 0; s < n_steps && ok; ++s) {
      const int q0 = (i_first + s) * BQ;
      if (!(ok = wait_warp(bar(kBarSFull), s & 1, abort_flag))) break;
      // The [LSE2 | D] vectors came with Q on QFull, whose phase S required.
      if (!(ok = wait_warp(bar(kBarQFull), s & 1, abort_flag))) break;
      tc_fence_after();
      const bool diag = causal && (q0 < k0 + BM) && (q0 + BQ > k0);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        // G1 walks its two chunks backwards so that its packed bf16 columns
        // [96,128) only overwrite fp32 columns it has already read.
        const int ch = g ? 1 - cc : cc;
        const int qbase = g * 64 + ch * 32;   // first query (of 128) in this chunk
        uint32_t sv[32], dp[32];
        tmem_ld32(tmem + lane_off + C::kColS + qbase, sv);
        tmem_ld32(tmem + lane_off + C::kColDP + qbase, dp);
        tmem_wait_ld(sv);
        tmem_wait_ld(dp);
        uint32_t pk[16], dsk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          // -LSE2 and -D of queries qbase+e .. +3 (same for every lane: broadcast).
          const float4 l4 = *reinterpret_cast<const float4 *>(vec + qbase + e);
          const float4 d4 = *reinterpret_cast<const float4 *>(vec + BQ + qbase + e);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv4[4] = {d4.x, d4.y, d4.z, d4.w};
          float p4[4], g4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float p = ex2_approx(fmaf(__uint_as_float(sv[e + u]), c, lv[u]));
            if (key >= N || (diag && key > q0 + qbase + e + u)) p = 0.f;
            p4[u] = p;
            g4[u] = p * (__uint_as_float(dp[e + u]) + dv4[u]);
          }
          pk[e >> 1] = pack_bf16x2(p4[0], p4[1]);
          pk[(e >> 1) + 1] = pack_bf16x2(p4[2], p4[3]);
          dsk[e >> 1] = pack_bf16x2(g4[0], g4[1]);
          dsk[(e >> 1) + 1] = pack_bf16x2(g4[2], g4[3]);
        }
        const uint32_t pcol = (g ? 96u : 0u) + ch * 16;
        tmem_st16(tmem + lane_off + C::kColS + pcol, pk);
        tmem_st16(tmem + lane_off + C::kColDP + pcol, dsk);
        // dS^T row r into shared memory: queries 64b..64b+63 form box b, a
        // 128-byte row per key with the 128-byte swizzle (16-byte chunk index
        // XOR key % 8), the layout of an M-major MMA operand.
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = (ch * 32 + u * 8) >> 3;   // 16-byte chunk within box g
          uint4 w;
          w.x = dsk[u * 4 + 0];
          w.y = dsk[u * 4 + 1];
          w.z = dsk[u * 4 + 2];
          w.w = dsk[u * 4 + 3];
          *reinterpret_cast<uint4 *>(ds_smem + g * C::kBoxBytes + r * 128 +
                                     ((chunk ^ (r & 7)) << 4)) = w;
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPReady));

      // dQ' rows q0 + r of this warp (lanes = queries), 32 columns per round:
      // TMEM -> registers -> staging tile -> TMA reduce-add into the
      // accumulator.  TMEM is released once the last round is in registers.
      if (!(ok = wait_warp(bar(kBarDQFull), s & 1, abort_flag))) break;
      tc_fence_after();
#pragma unroll
      for (int rd = 0; rd < kRounds; ++rd) {
        uint32_t gq[32];
        tmem_ld32(tmem + lane_off + dq_col + rd * 32, gq);
        tmem_wait_ld(gq);
        if (rd == kRounds - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarTmemFree));
        }
        // The previous reduce from this tile has finished reading it.
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4 w;
          w.x = gq[4 * j + 0];
          w.y = gq[4 * j + 1];
          w.z = gq[4 * j + 2];
          w.w = gq[4 * j + 3];
          *reinterpret_cast<uint4 *>(stage + lane * 128 + ((j ^ (lane & 7)) << 4)) = w;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dq, stage_u32, dq_d0 + rd * 32, q0 + quarter * 32, bh);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();

    // Epilogue: G0 writes dV_j, G1 writes dK_j = scale * (dS^T Q), bf16 rows.
    // Every lane runs the TMEM loads (warp-collective); rows >= N are not stored.
    if (ok && n_steps > 0) ok = wait_warp(bar(kBarKVDone), 0, abort_flag);
    if (ok) {
      tc_fence_after();
      const int64_t off = (static_cast<int64_t>(bh) * N + key) * D;
      __nv_bfloat16 *dst = (g ? dk : dv) + off;
      const float mul = g ? scale : 1.f;
      const uint32_t col = g ? C::kColDK : C::kColDV;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        if (n_steps > 0) {
          tmem_ld32(tmem + lane_off + col + ch * 32, v);
          tmem_wait_ld(v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;  // no query sees this key block
        }
        if (key < N) {
          uint4 *w = reinterpret_cast<uint4 *>(dst + ch * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 x;
            x.x = pack_bf16x2(__uint_as_float(v[8 * e + 0]) * mul, __uint_as_float(v[8 * e + 1]) * mul);
            x.y = pack_bf16x2(__uint_as_float(v[8 * e + 2]) * mul, __uint_as_float(v[8 * e + 3]) * mul);
            x.z = pack_bf16x2(__uint_as_float(v[8 * e + 4]) * mul, __uint_as_float(v[8 * e + 5]) * mul);
            x.w = pack_bf16x2(__uint_as_float(v[8 * e + 6]) * mul, __uint_as_float(v[8 * e + 7]) * mul);
            w[e] = x;
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

// dQ = scale * accumulator as bf16, eight elements per thread (row-major
// accumulator [BH][N][D]).
__global__ void __launch_bounds__(256)
    bwd_dq_kernel(const float *__restrict__ acc, __nv_bfloat16 *__restrict__ dq, int64_t n8,
                  float scale) {
  // A programmatic dependent of the main kernel: wait for its last additions.
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
                         const CUtensorMap &tdo, const CUtensorMap &tdq, const void *o,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv, int BH,
                         int N, float scale, int causal, float *ws, int *dev_status,
                         cudaStream_t stream) {
  using C = BCfg<D>;
  const int64_t rows = static_cast<int64_t>(BH) * N;
  const int n_qb = (N + BQ - 1) / BQ;
  const int64_t padded = static_cast<int64_t>(BH) * n_qb * BQ;
  // Workspace: fp32 dQ accumulator (row-major [BH][N][D] in the first
  // BH * N * D of BH * Npad * D floats), then [-LSE2 | -D] per query block.
  float *dq_acc = ws, *vecs = ws + padded * D;
  bwd_prep_kernel<D><<<static_cast<unsigned>((padded + 15) / 16), 256, 0, stream>>>(
      reinterpret_cast<const __nv_bfloat16 *>(o), reinterpret_cast<const __nv_bfloat16 *>(dout),
      lse, vecs, dq_acc, N, n_qb, padded);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if constexpr (D == 128) {
    // Q and dO maps have 64-row boxes here (the pipelined kernel's sub-tiles).
    e = launch_bwd_main_d128(tq, tk, tv, tdo, vecs, dq_acc, dk, dv, BH, N, scale, causal,
                             dev_status, stream);
  } else {
    // At least 120 KB so that one CTA (which takes all 512 TMEM columns) runs
    // per SM.
    constexpr int kLaunchSmem = C::kAlloc > 120 * 1024 ? C::kAlloc : 120 * 1024;
    e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kLaunchSmem);
    if (e != cudaSuccess) return e;
    bwd_main_kernel<D><<<n_qb * BH, kThreads, kLaunchSmem, stream>>>(
        tq, tk, tv, tdo, tdq, vecs, reinterpret_cast<__nv_bfloat16 *>(dk),
        reinterpret_cast<__nv_bfloat16 *>(dv), N, BH, scale, causal, dev_status);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  const int64_t n8 = rows * D / 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n8 + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bwd_dq_kernel, static_cast<const float *>(dq_acc),
                            reinterpret_cast<__nv_bfloat16 *>(dq), n8, scale);
}

}  // namespace

size_t bwd_workspace_bytes(int BH, int N, int d) {
  const size_t n_qb = (static_cast<size_t>(N) + BQ - 1) / BQ;
  return sizeof(float) * static_cast<size_t>(BH) * n_qb * BQ * (static_cast<size_t>(d) + 2);
}

cudaError_t launch_bwd_bf16(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &tdo, const CUtensorMap &tdq, const void *o,
                            const void *dout, const float *lse, void *dq, void *dk, void *dv,
                            int BH, int N, int d, float scale, int causal, float *ws,
                            int *dev_status, cudaStream_t stream) {
  if (d == 64)
    return launch_bwd_d<64>(tq, tk, tv, tdo, tdq, o, dout, lse, dq, dk, dv, BH, N, scale, causal,
                            ws, dev_status, stream);
  return launch_bwd_d<128>(tq, tk, tv, tdo, tdq, o, dout, lse, dq, dk, dv, BH, N, scale, causal,
                           ws, dev_status, stream);
}

}  // namespace fattn
