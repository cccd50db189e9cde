// api.cu -- the C ABI of libfattn (declared in include/fattn.h): argument
// validation, TMA tensor-map encoding, the per-device state the library
// owns, and kernel launches.  Every public function returns a status code;
// nothing here aborts or asserts.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>

#include "fattn.h"
#include "kernels.h"

namespace {

using fattn::launch_fwd_bf16;

constexpr int kMaxDevices = 64;

struct DeviceState {
  int *status = nullptr;          // device-side latched status word
  float *decode_ws = nullptr;     // split-K partials
  size_t decode_ws_bytes = 0;
  int *decode_counters = nullptr; // one int per (sequence, head), kept at zero
  size_t decode_counter_bytes = 0;
  int *fwd_sched = nullptr;       // 2 * kFwdSchedSlots pairs of work counters, kept at zero
  unsigned fwd_sched_next = 0;    // slot for the next eager launch
  unsigned fwd_sched_next_captured = 0;  // slot for the next launch captured into a graph
  void *mask_ws = nullptr;        // tile summary of the last mask (fa_forward_masked)
  size_t mask_ws_bytes = 0;
  CUtensorMap kv_map_k, kv_map_v; // last TMA views of paged caches (grouped decode)
  const void *kv_maps_k = nullptr, *kv_maps_v = nullptr;
  int kv_maps_hk = 0;
  bool kv_maps_valid = false;
  int inject_fault = 0;           // fa_debug_inject_fault: 1 next forward, 2 next backward
  int checked = 0;                // 1: sm_103 verified, -1: unsupported
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<int> g_decode_gqa_impl{0};   // fa_decode_gqa_select: 0 auto, 1 CUDA cores, 2 tensor cores

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Resolves the current device and makes sure its state exists.
int current_device(int *dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_NO_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_NO_DEVICE;
  DeviceState &st = g_dev[dev];
  if (st.checked == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_NO_DEVICE;
    st.checked = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (st.checked < 0) return FA_ERR_NO_DEVICE;
  if (st.status == nullptr) {
    if (cudaMalloc(&st.status, sizeof(int)) != cudaSuccess) return FA_ERR_NO_MEMORY;
    if (cudaMemset(st.status, 0, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  }
  if (st.fwd_sched == nullptr) {
    const size_t bytes = sizeof(int) * 2 * 2 * fattn::kFwdSchedSlots;
    if (cudaMalloc(&st.fwd_sched, bytes) != cudaSuccess) return FA_ERR_NO_MEMORY;
    if (cudaMemset(st.fwd_sched, 0, bytes) != cudaSuccess) return FA_ERR_CUDA;
  }
  *dev_out = dev;
  return FA_OK;
}

int get_encoder() {
  if (g_encode) return FA_OK;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return FA_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return FA_OK;
}

// 3-D bf16 view {d, N, BH} of a [BH, N, d] tensor; boxes of 64 x box_rows x 1
// (one 128-byte row segment per box row) with the 128-byte swizzle.  Rows
// past N read as zero.
int encode_qkv_map(CUtensorMap *m, const void *base, int BH, int N, int d, int box_rows = 128,
                   CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, dtype, 3, const_cast<void *>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 3-D E4M3 view {inner, rows, BH} of a [BH, rows, inner] byte tensor (inner
// = 128 codes of a row of Q or K, or Npad keys of a row of V^T), boxes of
// 128 x 128 x 1 with the 128-byte swizzle.  Reads past the extents give zero.
int encode_e4m3_map(CUtensorMap *m, const void *base, int BH, int rows, int inner) {
  const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)inner, (cuuint64_t)rows * inner};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// TMA views of the paged caches for the tensor-core grouped decode.  K cache
// [blocks][Hk][16 d-groups][16 tokens][8]: 5-D dims (8 tokens x 8 values,
// token half, d-group, head, block), boxes of 64 x 1 x 16 (one token half's
// 16 d-groups: 2 KB of no-swizzle core matrices, in 128-byte rows).  V cache
// [blocks][Hk][128 d][16 tokens]: 4-D dims (token, d, head, block), boxes of
// 16 x 128 (a block's V^T, 4 KB) written with the 32-byte swizzle.  The block
// extent is the largest int block id: which blocks are read comes from the
// block tables, as in the plain decode.
int encode_paged_kv_maps(CUtensorMap *tk, CUtensorMap *tv, const void *k_cache,
                         const void *v_cache, int num_kv_heads) {
  const cuuint64_t nb = 0x7fffffffull, hk = (cuuint64_t)num_kv_heads;
  const cuuint64_t kd[5] = {64, 2, 16, hk, nb};
  const cuuint64_t ks[4] = {128, 256, 4096, 4096 * hk};
  const cuuint32_t kb[5] = {64, 1, 16, 1, 1};
  const cuuint64_t vd[4] = {16, 128, hk, nb};
  const cuuint64_t vs[3] = {32, 4096, 4096 * hk};
  const cuuint32_t vb[4] = {16, 128, 1, 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  if (g_encode(tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(k_cache), kd, ks, kb,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return FA_ERR_CUDA;
  if (g_encode(tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(v_cache), vd, vs, vb,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return FA_ERR_CUDA;
  return FA_OK;
}

// Keys per row of the transposed FP8 V: N rounded up to 16.
long long fp8_vt_stride(int N) { return ((long long)N + 15) / 16 * 16; }

// 3-D fp32 view {d, N, BH} of the backward's row-major dQ accumulator, boxes
// of 32 x 32 x 1 (128-byte rows, 128-byte swizzle) for the TMA reduce-add.
int encode_dq_acc_map(CUtensorMap *m, void *base, int BH, int N, int d) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int check_forward_args(const void *q, const void *k, const void *v, const void *o,
                       const void *lse, int B, int H, int N, int d, float scale,
                       bool allow_d256 = false) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && !(allow_d256 && d == 256)) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_ALIGNMENT;
  // Grid and tensor-map limits: B*H and the tile count index 32-bit grids.
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL / 2 || (long long)N > 0x7fffffffLL / 2) return FA_ERR_UNSUPPORTED;
  if (BH * ((N + 127) / 128) > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Grows a library-owned buffer to at least `bytes`, in stream order on `s`:
// the old buffer is released with cudaFreeAsync and the new one taken with
// cudaMallocAsync, so growing never synchronises the device.  Earlier calls
// that used the old buffer are ordered before this one (the header's rule for
// calls that share library state), so the release cannot overtake them.
// During stream capture nothing may be allocated: a buffer that is too small
// then gives FA_ERR_UNSUPPORTED.  With `zero`, the new buffer is cleared on
// `s`.
int grow_on_stream(void **buf, size_t *have, size_t bytes, cudaStream_t s, bool zero) {
  if (*have >= bytes) return FA_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();  // the legacy stream while another stream captures: consume the error
    return FA_ERR_UNSUPPORTED;
  }
  if (cs != cudaStreamCaptureStatusNone) return FA_ERR_UNSUPPORTED;
  if (*buf != nullptr && cudaFreeAsync(*buf, s) != cudaSuccess) return FA_ERR_CUDA;
  *buf = nullptr;
  *have = 0;
  void *p = nullptr;
  if (cudaMallocAsync(&p, bytes, s) != cudaSuccess) return FA_ERR_NO_MEMORY;
  if (zero && cudaMemsetAsync(p, 0, bytes, s) != cudaSuccess) {
    cudaFreeAsync(p, s);
    return FA_ERR_CUDA;
  }
  *buf = p;
  *have = bytes;
  return FA_OK;
}

// Checks shared by the decode entry points; grows the library-owned split-K
// workspace and counters for (num_seqs, num_heads, max_num_blocks_per_seq)
// on the call's stream.
int decode_prepare(const void *q, const void *k_cache, const void *v_cache,
                   const int *block_tables, const int *context_lens, const void *out,
                   int num_seqs, int num_heads, int head_size, int block_size,
                   int max_num_blocks_per_seq, float scale, cudaStream_t stream, float **ws,
                   int **counters, int **status) {
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
  const size_t ws_bytes = fattn::decode_workspace_bytes(num_seqs, num_heads, max_parts);
  const size_t n_counters = (size_t)num_seqs * num_heads;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0, rc;
  if ((rc = current_device(&dev)) != FA_OK) return rc;
  DeviceState &st = g_dev[dev];
  if ((rc = grow_on_stream(reinterpret_cast<void **>(&st.decode_ws), &st.decode_ws_bytes,
                           ws_bytes, stream, false)) != FA_OK)
    return rc;
  if ((rc = grow_on_stream(reinterpret_cast<void **>(&st.decode_counters),
                           &st.decode_counter_bytes, n_counters * sizeof(int), stream, true)) !=
      FA_OK)
    return rc;
  *ws = st.decode_ws;
  *counters = st.decode_counters;
  *status = st.status;
  return FA_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// The work-counter pair of a persistent-kernel launch.  Eager launches take
// the first kFwdSchedSlots pairs round robin, so concurrent calls share one
// only with the 64th call after them.  A launch captured into a CUDA graph
// keeps its pair for every replay: it takes one of the other kFwdSchedSlots
// pairs, never handed to an eager launch, shared only with the 64th captured
// launch after it.  (A graph must not run concurrently with itself.)
int *sched_slot(DeviceState &st, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  bool captured = false;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess)
    cudaGetLastError();  // the legacy stream while another stream captures: not captured
  else
    captured = cs != cudaStreamCaptureStatusNone;
  const unsigned slot = captured
                            ? fattn::kFwdSchedSlots + st.fwd_sched_next_captured++ % fattn::kFwdSchedSlots
                            : st.fwd_sched_next++ % fattn::kFwdSchedSlots;
  return st.fwd_sched + 2 * slot;
}

}  // namespace

extern "C" {

int fa_version(void) { return 10000; }

const char *fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported size";
    case FA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device-side wait timed out";
    case FA_ERR_NO_MEMORY: return "out of device memory";
    case FA_ERR_NO_DEVICE: return "no usable sm_103 device";
    default: return "unknown status";
  }
}

namespace {
// fa_forward, fa_forward_f16 and fa_forward_masked: the tensor-core forward
// for 16-bit inputs.
int forward16(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
              int N, int d, float scale, int causal, fa_stream_t stream, bool f16,
              const uint8_t *mask = nullptr, long long mask_bh_stride = 0) {
  int rc = check_forward_args(q, k, v, o, lse, B, H, N, d, scale, mask == nullptr);
  if (rc != FA_OK) return rc;
  const int BH = B * H;
  if (BH == 0 || N == 0) return FA_OK;
  int dev = 0, fault_cta = -1;
  int *sched = nullptr;
  void *mask_ws = nullptr;
  const int mask_heads = mask_bh_stride != 0 ? BH : 1;
  if (mask != nullptr && (mask_heads > 65535 || (N + 127) / 128 > 65535)) return FA_ERR_UNSUPPORTED;
  CUtensorMap tq, tk, tv;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if ((rc = current_device(&dev)) != FA_OK) return rc;
    if ((rc = get_encoder()) != FA_OK) return rc;
    DeviceState &st = g_dev[dev];
    sched = sched_slot(st, reinterpret_cast<cudaStream_t>(stream));
    fault_cta = st.inject_fault == 1 ? 0 : -1;
    if (st.inject_fault == 1) st.inject_fault = 0;
    if (mask != nullptr) {
      const size_t need = fattn::mask_summary_bytes(mask_heads, N);
      if ((rc = grow_on_stream(&st.mask_ws, &st.mask_ws_bytes, need,
                               reinterpret_cast<cudaStream_t>(stream), false)) != FA_OK)
        return rc;
      mask_ws = st.mask_ws;
    }
  }
  const CUtensorMapDataType dt =
      f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if ((rc = encode_qkv_map(&tq, q, BH, N, d, 128, dt)) != FA_OK) return rc;
  if ((rc = encode_qkv_map(&tk, k, BH, N, d, 128, dt)) != FA_OK) return rc;
  if (d == 256) {
    // One 128-row query tile per CTA; V arrives in 64-key halves.
    if ((rc = encode_qkv_map(&tv, v, BH, N, d, 64, dt)) != FA_OK) return rc;
    return cuda_status(fattn::launch_fwd_d256(tq, tk, tv, o, lse, BH, N, scale, causal ? 1 : 0,
                                              sched, g_dev[dev].status,
                                              reinterpret_cast<cudaStream_t>(stream), f16));
  }
  if ((rc = encode_qkv_map(&tv, v, BH, N, d, 128, dt)) != FA_OK) return rc;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *flags = nullptr;
  const int2 *ranges = nullptr;
  const uint4 *bits = nullptr;
  if (mask != nullptr &&
      (rc = cuda_status(fattn::launch_mask_summary(mask, static_cast<int64_t>(mask_bh_stride), N,
                                                   mask_heads, mask_ws, &flags, &ranges, &bits,
                                                   s))) != FA_OK)
    return rc;
  return cuda_status(launch_fwd_bf16(tq, tk, tv, o, lse, BH, N, d, scale, causal ? 1 : 0, sched,
                                     g_dev[dev].status, fault_cta, s, f16, mask,
                                     static_cast<int64_t>(mask_bh_stride), ranges, flags, bits));
}
}  // namespace

int fa_forward(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
               int N, int d, float scale, int causal, fa_stream_t stream) {
  return forward16(q, k, v, o, lse, B, H, N, d, scale, causal, stream, false);
}

int fa_forward_f16(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                   int H, int N, int d, float scale, int causal, fa_stream_t stream) {
  return forward16(q, k, v, o, lse, B, H, N, d, scale, causal, stream, true);
}

int fa_forward_masked(const void *q, const void *k, const void *v, void *o, float *lse,
                      const void *mask, long long mask_bh_stride, int B, int H, int N, int d,
                      float scale, fa_stream_t stream) {
  if (!mask || mask_bh_stride < 0) return FA_ERR_INVALID_ARG;
  if (!aligned16(mask) || mask_bh_stride % 16 != 0) return FA_ERR_ALIGNMENT;
  if (N % 16 != 0) return FA_ERR_UNSUPPORTED;
  return forward16(q, k, v, o, lse, B, H, N, d, scale, 0, stream, false,
                   static_cast<const uint8_t *>(mask), mask_bh_stride);
}

int fa_forward_fp32(const float *q, const float *k, const float *v, float *o, float *lse, int B,
                    int H, int N, int d, float scale, int causal, fa_stream_t stream) {
  int rc = check_forward_args(q, k, v, o, lse, B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  const int BH = B * H;
  if (BH == 0 || N == 0) return FA_OK;
  if (BH > 0x7fffffff || (N + 31) / 32 > 65535) return FA_ERR_UNSUPPORTED;
  int dev = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if ((rc = current_device(&dev)) != FA_OK) return rc;
  }
  return cuda_status(fattn::launch_fwd_f32(q, k, v, o, lse, BH, N, d, scale, causal ? 1 : 0,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

unsigned long long fa_quantize_fp8_workspace_bytes(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0 || d < 0) return 0;
  return static_cast<unsigned long long>(
      fattn::fp8_quant_workspace_bytes(static_cast<int>((long long)B * H), N));
}

long long fa_fp8_vt_stride(int N) { return N < 0 ? 0 : fp8_vt_stride(N); }

int fa_quantize_fp8(const void *q, const void *k, const void *v, const float *signs, void *q8,
                    void *k8, void *vt8, float *q_scale, float *k_scale, float *v_scale, int B,
                    int H, int N, int d, void *workspace, unsigned long long workspace_bytes,
                    fa_stream_t stream) {
  if (!q || !k || !v || !q8 || !k8 || !vt8 || !q_scale || !k_scale || !v_scale)
    return FA_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q8) || !aligned16(k8) ||
      !aligned16(vt8) || (signs && !aligned16(signs)))
    return FA_ERR_ALIGNMENT;
  const long long BH = (long long)B * H;
  if (BH > 65535 || N > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if (BH == 0 || N == 0) return FA_OK;
  if (!workspace) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 4 != 0) return FA_ERR_ALIGNMENT;
  if (workspace_bytes < fattn::fp8_quant_workspace_bytes((int)BH, N)) return FA_ERR_INVALID_ARG;
  int dev = 0, rc;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if ((rc = current_device(&dev)) != FA_OK) return rc;
  }
  // The transform's 1/sqrt(d), rounded once to fp32, multiplies the scales.
  const float rot_factor = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  return cuda_status(fattn::launch_fp8_quantize(
      q, k, v, signs, q8, k8, vt8, q_scale, k_scale, v_scale, static_cast<float *>(workspace),
      (int)BH, N, (int)fp8_vt_stride(N), rot_factor, g_dev[dev].status,
      reinterpret_cast<cudaStream_t>(stream)));
}

int fa_forward_fp8(const void *q8, const void *k8, const void *vt8, const float *q_scale,
                   const float *k_scale, const float *v_scale, void *o, float *lse, int B, int H,
                   int N, int d, float scale, int causal, fa_stream_t stream) {
  if (!q_scale || !k_scale || !v_scale) return FA_ERR_INVALID_ARG;
  int rc = check_forward_args(q8, k8, vt8, o, lse, B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  const int BH = B * H;
  if (BH == 0 || N == 0) return FA_OK;
  int dev = 0, fault_cta = -1;
  int *sched = nullptr;
  CUtensorMap tq, tk, tvt;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if ((rc = current_device(&dev)) != FA_OK) return rc;
    if ((rc = get_encoder()) != FA_OK) return rc;
    DeviceState &st = g_dev[dev];
    sched = sched_slot(st, reinterpret_cast<cudaStream_t>(stream));
    fault_cta = st.inject_fault == 1 ? 0 : -1;
    if (st.inject_fault == 1) st.inject_fault = 0;
  }
  if ((rc = encode_e4m3_map(&tq, q8, BH, N, d)) != FA_OK) return rc;
  if ((rc = encode_e4m3_map(&tk, k8, BH, N, d)) != FA_OK) return rc;
  if ((rc = encode_e4m3_map(&tvt, vt8, BH, d, (int)fp8_vt_stride(N))) != FA_OK) return rc;
  return cuda_status(fattn::launch_fwd_fp8(tq, tk, tvt, q_scale, k_scale, v_scale, o, lse, BH, N,
                                           scale, causal ? 1 : 0, sched, g_dev[dev].status,
                                           fault_cta, reinterpret_cast<cudaStream_t>(stream)));
}

unsigned long long fa_backward_workspace_bytes(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0 || d < 0) return 0;
  return static_cast<unsigned long long>(
      fattn::bwd_workspace_bytes(static_cast<int>((long long)B * H), N, d));
}

int fa_backward(const void *q, const void *k, const void *v, const void *o, const void *dout,
                const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                float scale, int causal, void *workspace, unsigned long long workspace_bytes,
                fa_stream_t stream) {
  if (!dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  int rc = check_forward_args(q, k, v, o, lse, B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_ALIGNMENT;
  const int BH = B * H;
  if (BH == 0 || N == 0) return FA_OK;
  if (!workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return FA_ERR_ALIGNMENT;
  if (workspace_bytes < fattn::bwd_workspace_bytes(BH, N, d)) return FA_ERR_INVALID_ARG;
  // The preparation kernel runs 16 padded rows per block of its 1-D grid.
  if ((long long)BH * ((N + 127) / 128) * 8 > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  int dev = 0, fault_cta = -1;
  int *sched = nullptr;
  CUtensorMap tq, tk, tv, tdo, tdq;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if ((rc = current_device(&dev)) != FA_OK) return rc;
    if ((rc = get_encoder()) != FA_OK) return rc;
    sched = sched_slot(g_dev[dev], reinterpret_cast<cudaStream_t>(stream));
    if (g_dev[dev].inject_fault == 2) {
      fault_cta = 0;
      g_dev[dev].inject_fault = 0;
    }
  }
  const int qdo_rows = fattn::bwd_qdo_box_rows(d);
  if ((rc = encode_qkv_map(&tq, q, BH, N, d, qdo_rows)) != FA_OK) return rc;
  if ((rc = encode_qkv_map(&tk, k, BH, N, d)) != FA_OK) return rc;
  if ((rc = encode_qkv_map(&tv, v, BH, N, d)) != FA_OK) return rc;
  if ((rc = encode_qkv_map(&tdo, dout, BH, N, d, qdo_rows)) != FA_OK) return rc;
  if ((rc = encode_dq_acc_map(&tdq, workspace, BH, N, d)) != FA_OK) return rc;
  return cuda_status(fattn::launch_bwd_bf16(tq, tk, tv, tdo, tdq, o, dout, lse, dq, dk, dv, BH,
                                            N, d,
                                            scale, causal ? 1 : 0,
                                            reinterpret_cast<float *>(workspace), sched,
                                            fault_cta, g_dev[dev].status,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

int fa_paged_decode(const void *q, const void *k_cache, const void *v_cache,
                    const int *block_tables, const int *context_lens, void *out, int num_seqs,
                    int num_heads, int head_size, int block_size, int max_num_blocks_per_seq,
                    float scale, fa_stream_t stream) {
  float *ws = nullptr;
  int *counters = nullptr, *status = nullptr;
  const int rc = decode_prepare(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs,
                                num_heads, head_size, block_size, max_num_blocks_per_seq, scale,
                                reinterpret_cast<cudaStream_t>(stream), &ws, &counters, &status);
  if (rc != FA_OK || num_seqs == 0) return rc;
  return cuda_status(fattn::launch_paged_decode(q, k_cache, v_cache, block_tables, context_lens,
                                                out, num_seqs, num_heads, max_num_blocks_per_seq,
                                                scale, ws, counters,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

int fa_paged_decode_gqa(const void *q, const void *k_cache, const void *v_cache,
                        const int *block_tables, const int *context_lens, void *out,
                        int num_seqs, int num_heads, int num_kv_heads, int head_size,
                        int block_size, int max_num_blocks_per_seq, float scale,
                        fa_stream_t stream) {
  if (num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads != 0)
    return FA_ERR_INVALID_ARG;
  const int group = num_heads / num_kv_heads;
  const int impl = g_decode_gqa_impl.load();
  const bool cc_ok = fattn::decode_gqa_group_supported(group);
  const bool tc_ok = fattn::decode_gqa_tc_supported(group);
  // Automatic: the tensor-core kernel from group 3 up once there is at least
  // a unit (sequence, partition, cached head) per SM; measured faster there,
  // and slower for group 2 and for a handful of units.
  const long long units_bound = (long long)num_seqs * num_kv_heads *
                                fattn::decode_max_parts(max_num_blocks_per_seq);
  const bool tc_auto = tc_ok && (!cc_ok || (group >= 3 && units_bound >= fattn::kDecodeTcMinUnits));
  const bool tc = group > 1 && (impl == 2 ? tc_ok : impl == 0 ? tc_auto : false);
  if (group > 1 && !tc && (impl == 2 || !cc_ok)) return FA_ERR_UNSUPPORTED;
  float *ws = nullptr;
  int *counters = nullptr, *status = nullptr;
  const int rc = decode_prepare(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs,
                                num_heads, head_size, block_size, max_num_blocks_per_seq, scale,
                                reinterpret_cast<cudaStream_t>(stream), &ws, &counters, &status);
  if (rc != FA_OK || num_seqs == 0) return rc;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (group == 1)
    return cuda_status(fattn::launch_paged_decode(q, k_cache, v_cache, block_tables,
                                                  context_lens, out, num_seqs, num_heads,
                                                  max_num_blocks_per_seq, scale, ws, counters, s));
  if (tc) {
    CUtensorMap tk, tv;
    int *sched = nullptr;
    {
      // The views depend only on the caches' addresses and head count: the
      // last pair encoded on the device is reused while those stay the same.
      std::lock_guard<std::mutex> lock(g_mu);
      int dev = 0, rc2;
      if ((rc2 = current_device(&dev)) != FA_OK) return rc2;
      if ((rc2 = get_encoder()) != FA_OK) return rc2;
      DeviceState &st = g_dev[dev];
      sched = sched_slot(st, reinterpret_cast<cudaStream_t>(stream));
      if (!(st.kv_maps_valid && st.kv_maps_k == k_cache && st.kv_maps_v == v_cache &&
            st.kv_maps_hk == num_kv_heads)) {
        st.kv_maps_valid = false;
        if ((rc2 = encode_paged_kv_maps(&st.kv_map_k, &st.kv_map_v, k_cache, v_cache,
                                        num_kv_heads)) != FA_OK)
          return rc2;
        st.kv_maps_k = k_cache;
        st.kv_maps_v = v_cache;
        st.kv_maps_hk = num_kv_heads;
        st.kv_maps_valid = true;
      }
      tk = st.kv_map_k;
      tv = st.kv_map_v;
    }
    return cuda_status(fattn::launch_paged_decode_gqa_tc(
        tk, tv, q, block_tables, context_lens, out, num_seqs, num_heads, num_kv_heads,
        max_num_blocks_per_seq, scale, ws, sched, status, s));
  }
  return cuda_status(fattn::launch_paged_decode_gqa(q, k_cache, v_cache, block_tables,
                                                    context_lens, out, num_seqs, num_heads,
                                                    num_kv_heads, max_num_blocks_per_seq, scale,
                                                    ws, counters, status, s));
}

int fa_device_status(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0, rc;
  if ((rc = current_device(&dev)) != FA_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, g_dev[dev].status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  if (h != 0 && cudaMemset(g_dev[dev].status, 0, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  return h;
}

int fa_decode_gqa_select(int impl) {
  if (impl < 0 || impl > 2) return FA_ERR_INVALID_ARG;
  g_decode_gqa_impl.store(impl);
  return FA_OK;
}

int fa_debug_inject_fault(int mode) {
  if (mode != 0 && mode != 1 && mode != 2) return FA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0, rc;
  if ((rc = current_device(&dev)) != FA_OK) return rc;
  g_dev[dev].inject_fault = mode;
  return FA_OK;
}

void fa_release(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
  DeviceState &st = g_dev[dev];
  // The buffers grown in stream order may still be in use by work the caller
  // has not waited for; cudaFree does not order itself after it.
  cudaDeviceSynchronize();
  if (st.decode_ws) cudaFree(st.decode_ws);
  if (st.decode_counters) cudaFree(st.decode_counters);
  if (st.status) cudaFree(st.status);
  if (st.fwd_sched) cudaFree(st.fwd_sched);
  if (st.mask_ws) cudaFree(st.mask_ws);
  st = DeviceState{};
}

}  // extern "C"
