// mask_tiles.cu -- a per-tile summary of a boolean attention mask, so that
// the masked forward skips key tiles no query row of a work item can see and
// reads visibility only for tiles that are partly visible, as 16 bytes of
// bits per row instead of the row's 128 mask bytes.
//
// flags[mh][qt][kt] (uint8) for each 128 x 128 block of mask head mh (one head
// when the mask is shared): 0 = no visible key, 2 = every key visible (and
// the block lies inside the sequence), 1 = anything else.
// ranges[mh][qp] (int2 {kv0 | n_a << 16, n_b}) for each pair of query tiles A =
// 2qp, B = 2qp + 1, the work item of the forward: the item processes key tiles
// kv0 .. kv0 + n_b - 1, from the first tile either query tile sees to the last
// one; tile A stops after its own last visible tile (n_a <= n_b) when B's
// range reaches at least as far, else both run to the end.  An item that sees
// nothing gets one fully masked tile (n_a = n_b = 1), so that its rows are
// still written (O = 0, LSE = -inf).
// bits[mh][qt][kt][r] (16 bytes) for row r of each 128 x 128 block: bit c of
// the 128 (word c / 32, bit c % 32) set iff key kt * 128 + c is visible to
// query row qt * 128 + r (zero past N), so that the forward reads 16 bytes
// per row of a partly visible tile instead of its 128 mask bytes.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace fattn {
namespace {

constexpr int kT = 128;

__device__ __forceinline__ bool all_bytes_nonzero(uint32_t x) {
  // A byte of x is zero iff its high bit survives (x - 0x01..) & ~x.
  return ((x - 0x01010101u) & ~x & 0x80808080u) == 0u;
}

// Bit b (0..3) set iff byte b of x is nonzero: the high bit of each byte of
// (x & 0x7f..) + 0x7f.. | x marks a nonzero byte; the multiply gathers the
// four marks (bits 0, 8, 16, 24 after the shift) into bits 21 .. 24.
__device__ __forceinline__ uint32_t nonzero_nibble(uint32_t x) {
  const uint32_t hb = (((x & 0x7f7f7f7fu) + 0x7f7f7f7fu) | x) & 0x80808080u;
  return ((hb >> 7) * 0x00204081u >> 21) & 0xfu;
}

constexpr int kFlagThreads = 256;

// grid (n_t, n_t, mask heads), kFlagThreads threads: one 128 x 128 block each.
__global__ void __launch_bounds__(kFlagThreads)
    mask_tile_flags_kernel(const uint8_t *__restrict__ mask, int64_t bh_stride, int N, int n_t,
                           uint8_t *__restrict__ flags, uint4 *__restrict__ bits) {
  // The ranges kernel may be scheduled once every block of this one has begun.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int kt = blockIdx.x, qt = blockIdx.y, mh = blockIdx.z;
  const uint8_t *base = mask + static_cast<int64_t>(mh) * bh_stride;
  int any = 0, all = 1;
  // 128 rows x 8 chunks of 16 bytes, four chunks a thread, all four loads
  // issued before the first is used; N is a multiple of 16, so a chunk lies
  // wholly inside or wholly outside the sequence.
  constexpr int kPer = kT * 8 / kFlagThreads;
  uint4 v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = threadIdx.x + u * kFlagThreads;
    const int r = qt * kT + (i >> 3), c0 = kt * kT + (i & 7) * 16;
    v[u] = (r < N && c0 < N)
               ? __ldg(reinterpret_cast<const uint4 *>(base + static_cast<int64_t>(r) * N + c0))
               : make_uint4(0u, 0u, 0u, 0u);
  }
  const int lane = threadIdx.x & 31, l0 = lane & ~7, c = lane & 7;
  uint4 *brow = bits + ((static_cast<int64_t>(mh) * n_t + qt) * n_t + kt) * kT;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = threadIdx.x + u * kFlagThreads;
    const int r = qt * kT + (i >> 3), c0 = kt * kT + (i & 7) * 16;
    uint32_t m16 = 0u;   // bit b: byte b of this 16-byte chunk is nonzero
    if (r < N && c0 < N) {
      any |= (v[u].x | v[u].y | v[u].z | v[u].w) != 0u;
      all &= all_bytes_nonzero(v[u].x) && all_bytes_nonzero(v[u].y) &&
             all_bytes_nonzero(v[u].z) && all_bytes_nonzero(v[u].w);
      m16 = nonzero_nibble(v[u].x) | (nonzero_nibble(v[u].y) << 4) |
            (nonzero_nibble(v[u].z) << 8) | (nonzero_nibble(v[u].w) << 12);
    }
    // The row's eight chunks are on lanes l0 .. l0 + 7: chunk c fills
    // bits 16 (c % 2) .. + 15 of word c / 2.
    const uint32_t part = m16 << (16 * (c & 1));
    uint32_t wd[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      wd[q] = __shfl_sync(~0u, part, l0 + 2 * q) | __shfl_sync(~0u, part, l0 + 2 * q + 1);
    if (c == 0) brow[i >> 3] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  }
  any = __syncthreads_or(any);
  all = __syncthreads_and(all);
  if (threadIdx.x == 0)
    flags[(static_cast<int64_t>(mh) * n_t + qt) * n_t + kt] =
        !any ? 0 : (all && (kt + 1) * kT <= N) ? 2 : 1;
}

// grid (n_pairs, mask heads), one warp each.
__global__ void __launch_bounds__(32)
    mask_item_ranges_kernel(const uint8_t *__restrict__ flags, int n_t, int n_pairs,
                            int2 *__restrict__ ranges) {
  // A programmatic dependent of the flags kernel: wait for its flags; the
  // forward that follows may be scheduled meanwhile.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int qp = blockIdx.x, mh = blockIdx.y, lane = threadIdx.x;
  const uint8_t *fa = flags + (static_cast<int64_t>(mh) * n_t + 2 * qp) * n_t;
  const bool has_b = 2 * qp + 1 < n_t;
  int lo = -1, hi_a = -1, hi_b = -1;   // first visible tile; one past the last (A, B)
  for (int k0 = 0; k0 < n_t; k0 += 32) {
    const int kt = k0 + lane;
    const bool va = kt < n_t && fa[kt] != 0;
    const bool vb = kt < n_t && has_b && fa[n_t + kt] != 0;
    const unsigned ba = __ballot_sync(0xffffffffu, va);
    const unsigned bb = __ballot_sync(0xffffffffu, vb);
    if ((ba | bb) != 0u && lo < 0) lo = k0 + __ffs(ba | bb) - 1;
    if (ba != 0u) hi_a = k0 + 32 - __clz(ba);
    if (bb != 0u) hi_b = k0 + 32 - __clz(bb);
  }
  if (lane == 0) {
    int2 r = make_int2(1 << 16, 1);
    if (lo >= 0) {
      const int n_b = max(hi_a, hi_b) - lo;
      const int n_a = hi_a <= hi_b ? max(hi_a - lo, 1) : n_b;
      r = make_int2(lo | (n_a << 16), n_b);
    }
    ranges[static_cast<int64_t>(mh) * n_pairs + qp] = r;
  }
}

}  // namespace

size_t mask_summary_bytes(int mask_heads, int N) {
  const size_t n_t = static_cast<size_t>((N + kT - 1) / kT);
  const size_t n_pairs = (n_t + 1) / 2;
  const size_t flag_bytes = (static_cast<size_t>(mask_heads) * n_t * n_t + 15) / 16 * 16;
  const size_t range_bytes = (static_cast<size_t>(mask_heads) * n_pairs * sizeof(int2) + 15) / 16 * 16;
  return flag_bytes + range_bytes + static_cast<size_t>(mask_heads) * n_t * n_t * kT * 16;
}

cudaError_t launch_mask_summary(const uint8_t *mask, int64_t bh_stride, int N, int mask_heads,
                                void *ws, uint8_t **flags, const int2 **ranges,
                                const uint4 **bits, cudaStream_t stream) {
  const int n_t = (N + kT - 1) / kT;
  const int n_pairs = (n_t + 1) / 2;
  const size_t flag_bytes = (static_cast<size_t>(mask_heads) * n_t * n_t + 15) / 16 * 16;
  const size_t range_bytes = (static_cast<size_t>(mask_heads) * n_pairs * sizeof(int2) + 15) / 16 * 16;
  uint8_t *f = static_cast<uint8_t *>(ws);
  int2 *r = reinterpret_cast<int2 *>(f + flag_bytes);
  uint4 *b = reinterpret_cast<uint4 *>(f + flag_bytes + range_bytes);
  mask_tile_flags_kernel<<<dim3(n_t, n_t, mask_heads), kFlagThreads, 0, stream>>>(
      mask, bh_stride, N, n_t, f, b);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_pairs, mask_heads);
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mask_item_ranges_kernel, static_cast<const uint8_t *>(f), n_t,
                         n_pairs, r);
  if (e != cudaSuccess) return e;
  *flags = f;
  *ranges = r;
  *bits = b;
  return cudaGetLastError();
}

}  // namespace fattn
