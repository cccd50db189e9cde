// decode_noalloc.cu -- fa_paged_decode_noalloc: the paged decode with its
// split-K scratch taken from a fixed device array that is part of the library
// image, so a call never allocates device memory.
//
// Who needs this: some callers cannot allocate device memory when they call
// in.  A serving process may hand every byte of HBM to its own pool at start
// up and forbid later cudaMalloc calls; a real-time loop may not accept the
// device-wide synchronisation that cudaMalloc/cudaFree can cause; a plug-in
// may run under a host framework that owns all allocation.  fa_paged_decode
// grows a library-owned workspace on first use, which those callers cannot
// allow.  This entry point runs the same decode kernel, but its partial
// results and arrival counters live in g_decode_scratch below, which the CUDA
// runtime places in device memory when the library's module is loaded on a
// device and which stays there until the process exits.
//
// Limits and sharing:
//  * kScratchBytes (12 MiB per device) bounds the problem: it must hold
//    num_seqs*num_heads counters (4 bytes each, rounded up to 256 bytes) plus
//    num_seqs*num_heads*ceil(max_num_blocks_per_seq/32)*130 floats of partial
//    results.  Larger problems are rejected with FA_ERR_UNSUPPORTED before
//    anything is enqueued.
//  * Every call on a device uses the same array and leaves its contents
//    behind.  The counters, which must start at zero, are cleared by a
//    cudaMemsetAsync on the caller's stream at the start of each call.  Two
//    calls whose work overlaps on the GPU (different streams, no ordering
//    between them) race on the array and may return wrong results; order
//    them on one stream or with events.
//  * Every call looks up the array's device address on the current device
//    with cudaGetSymbolAddress.  The first lookup on a device may load the
//    library's module there, so make the first call on each device before
//    any stream capture begins.  Looking the address up on every call (it is
//    cheap once the module is loaded) keeps it right after a context
//    teardown such as cudaDeviceReset, which may reload the module at
//    another address.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fattn.h"
#include "kernels.h"

namespace {
constexpr size_t kScratchBytes = size_t(12) << 20;
constexpr int kMaxDevices = 64;
}  // namespace

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

namespace {

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

// Device address of g_decode_scratch on the current device.  Host code only
// holds a host-side stand-in under the array's name; the device address
// must come from the runtime.
int scratch_address(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
    return FA_ERR_CUDA;
  *out = p;
  return FA_OK;
}

}  // namespace

extern "C" int fa_paged_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                       const int *block_tables, const int *context_lens,
                                       void *out, int num_seqs, int num_heads, int head_size,
                                       int block_size, int max_num_blocks_per_seq, float scale,
                                       fa_stream_t stream) {
  auto aligned16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return FA_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_heads <= 0 || max_num_blocks_per_seq <= 0) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (head_size != fattn::kDecodeHeadSize || block_size != fattn::kDecodeBlockSize)
    return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return FA_ERR_ALIGNMENT;
  if (num_heads > 65535 || num_seqs > 65535) return FA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return FA_OK;

  const int max_parts = fattn::decode_max_parts(max_num_blocks_per_seq);
  const size_t n_counters = (size_t)num_seqs * num_heads;
  const size_t counter_bytes = round256(n_counters * sizeof(int));
  const size_t ws_bytes = fattn::decode_workspace_bytes(num_seqs, num_heads, max_parts);
  if (counter_bytes + ws_bytes > kScratchBytes) return FA_ERR_UNSUPPORTED;

  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      major != 10 || minor != 3)
    return FA_ERR_NO_DEVICE;
  void *base = nullptr;
  const int rc = scratch_address(&base);
  if (rc != FA_OK) return rc;

  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int *counters = static_cast<int *>(base);
  float *ws = reinterpret_cast<float *>(static_cast<unsigned char *>(base) + counter_bytes);
  if (cudaMemsetAsync(counters, 0, n_counters * sizeof(int), s) != cudaSuccess) return FA_ERR_CUDA;
  const cudaError_t e = fattn::launch_paged_decode(q, k_cache, v_cache, block_tables, context_lens,
                                                   out, num_seqs, num_heads,
                                                   max_num_blocks_per_seq, scale, ws, counters, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
