// kernels.h -- launchers shared between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace fattn {

constexpr int kDecodeHeadSize = 128;
constexpr int kDecodeBlockSize = 16;
constexpr int kDecodePartitionTokens = 512;

cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
                           int BH, int N, int d, float scale, int causal, cudaStream_t stream);

// q, k, v tensor maps: 3-D views {d, N, B*H} of the bf16 inputs, 64 x 128 x 1
// boxes with the 128-byte swizzle.  `sched` points to two ints (the item
// counter and the finished-CTA counter) that are zero before the launch; the
// kernel leaves them zero.  Launches that may run at the same time need
// different `sched` slots.
constexpr int kFwdSchedSlots = 64;
// fault_cta >= 0 makes that CTA's producer stop after its first Q loads (the
// failure-path test); -1 in normal use.
// f16 selects fp16 Q, K, V, O (tensor maps of CU_TENSOR_MAP_DATA_TYPE_FLOAT16).
// mask (bf16 only, causal 0, N a multiple of 16): uint8, key j visible to row i
// of head bh iff mask[bh * mask_bh_stride + i * N + j] != 0; mask_ranges,
// mask_flags and mask_bits: its tile summary from launch_mask_summary.
cudaError_t launch_fwd_bf16(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            void *o, float *lse, int BH, int N, int d, float scale, int causal,
                            int *sched, int *dev_status, int fault_cta, cudaStream_t stream,
                            bool f16 = false, const uint8_t *mask = nullptr,
                            int64_t mask_bh_stride = 0, const int2 *mask_ranges = nullptr,
                            const uint8_t *mask_flags = nullptr, const uint4 *mask_bits = nullptr);

// Tile summary of a boolean mask (mask_tiles.cu) for mask_heads heads (1 when
// the mask is shared): per 128 x 128 block a flag (0 nothing visible, 1
// partly, 2 everything), per pair of query tiles the key tiles to process
// (int2 {kv0 | n_a << 16, n_b}, see mask_tiles.cu), per row of each block its
// 128 visibility bits (16 bytes).  ws: mask_summary_bytes(mask_heads, N)
// bytes of 16-byte aligned device memory; *flags, *ranges and *bits point
// into it.
size_t mask_summary_bytes(int mask_heads, int N);
cudaError_t launch_mask_summary(const uint8_t *mask, int64_t bh_stride, int N, int mask_heads,
                                void *ws, uint8_t **flags, const int2 **ranges,
                                const uint4 **bits, cudaStream_t stream);

// Head dimension 256 (fwd_d256.cu), bf16 or (f16) fp16: tq and tk as for
// launch_fwd_bf16 (64 x 128 x 1 boxes), tv with 64 x 64 x 1 boxes.
cudaError_t launch_fwd_d256(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            void *o, float *lse, int BH, int N, float scale, int causal,
                            int *sched, int *dev_status, cudaStream_t stream, bool f16);

// FP8 forward (fwd_bf16.cu, d = 128): tq, tk are E4M3 maps {128, N, B*H}
// with 128 x 128 x 1 boxes, tvt the E4M3 map {Npad, 128, B*H} of V^T, same
// boxes; all with the 128-byte swizzle.  q_scale, k_scale: one fp32 per
// 128-row block of each head; v_scale: one per head.  o is bf16.  fault_cta
// as for launch_fwd_bf16.
cudaError_t launch_fwd_fp8(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tvt,
                           const float *q_scale, const float *k_scale, const float *v_scale,
                           void *o, float *lse, int BH, int N, float scale, int causal,
                           int *sched, int *dev_status, int fault_cta, cudaStream_t stream);

// FP8 block quantization (fp8_quant.cu, d = 128); v_amax: the workspace of
// fp8_quant_workspace_bytes(BH, N) bytes; signs: 128 fp32 +-1 values or null.
size_t fp8_quant_workspace_bytes(int BH, int N);
cudaError_t launch_fp8_quantize(const void *q, const void *k, const void *v, const float *signs,
                                void *q8, void *k8, void *vt8, float *q_scale, float *k_scale,
                                float *v_scale, float *v_amax, int BH, int N, int n_pad,
                                float rot_factor, int *dev_status, cudaStream_t stream);

// Backward: workspace = fp32 dQ accumulator (row-major [BH][N][d] inside
// B*H*Npad*d floats, Npad = N rounded up to 128), then [-LSE2 | -D] (2 x 128
// fp32) per 128-query block: 4 * B*H*Npad*(d + 2) bytes.  tq and tdo (the map
// of dO) are bf16 maps like the forward's but with boxes of
// bwd_qdo_box_rows(d) rows; tk, tv as in the forward; tdq is the fp32 map of
// the accumulator (boxes of 32 x 32 x 1, 128-byte swizzle).
inline int bwd_qdo_box_rows(int) { return 64; }
size_t bwd_workspace_bytes(int BH, int N, int d);
cudaError_t launch_bwd_bf16(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &tdo, const CUtensorMap &tdq, const void *o,
                            const void *dout, const float *lse, void *dq, void *dk, void *dv,
                            int BH, int N, int d, float scale, int causal, float *ws,
                            int *sched, int fault_cta, int *dev_status, cudaStream_t stream);

// The d = 128 main kernel (bwd_bf16_d128.cu); vecs = the [-LSE2 | -D]
// blocks, tdq = the fp32 map of the row-major dQ accumulator (TMA reduces);
// sched = a pair of work counters kept at zero (persistent CTAs).
cudaError_t launch_bwd_main_d128(const CUtensorMap &tq64, const CUtensorMap &tk,
                                 const CUtensorMap &tv, const CUtensorMap &tdo64,
                                 const CUtensorMap &tdq, const float *vecs, void *dk, void *dv,
                                 int BH,
                                 int N, float scale, int causal, int *sched, int fault_cta,
                                 int *dev_status, cudaStream_t stream);

// The d = 64 main kernel (bwd_bf16_d64.cu); tdq = the accumulator's fp32 map
// (its dQ' tiles are added with TMA reduces); sched as for d = 128.
cudaError_t launch_bwd_main_d64(const CUtensorMap &tq64, const CUtensorMap &tk,
                                const CUtensorMap &tv, const CUtensorMap &tdo64,
                                const CUtensorMap &tdq, const float *vecs, void *dk, void *dv,
                                int BH, int N, float scale, int causal, int *sched,
                                int fault_cta, int *dev_status, cudaStream_t stream);

int decode_max_parts(int max_num_blocks_per_seq);
// Grouped key/value heads (decode_gqa.cu): group = num_heads / num_kv_heads
// must be 2 or a multiple of 4.  Same workspace and counters as the one-head
// decode (counters indexed per (sequence, query-head group of the CTA)).
bool decode_gqa_group_supported(int group);
cudaError_t launch_paged_decode_gqa(const void *q, const void *k_cache, const void *v_cache,
                                    const int *block_tables, const int *context_lens, void *out,
                                    int num_seqs, int num_heads, int num_kv_heads, int max_blocks,
                                    float scale, float *workspace, int *counters,
                                    int *dev_status, cudaStream_t stream);
// Grouped key/value heads on the tensor cores (decode_gqa_tc.cu): group =
// num_heads / num_kv_heads from 2 to 16, or a multiple of 16.  tm_k / tm_v are
// the TMA views of the caches (encode_paged_kv_maps in api.cu); sched is a
// pair of work counters kept at zero; the workspace is the split-K one below
// (a second kernel merges the partitions; no counters).
bool decode_gqa_tc_supported(int group);
// Below this many (sequence, partition, cached head) units the automatic
// choice keeps the CUDA-core kernel (fewer launches, less set-up).
constexpr long long kDecodeTcMinUnits = 152;
cudaError_t launch_paged_decode_gqa_tc(const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                       const void *q, const int *block_tables,
                                       const int *context_lens, void *out, int num_seqs,
                                       int num_heads, int num_kv_heads, int max_blocks,
                                       float scale, float *workspace, int *sched,
                                       int *dev_status, cudaStream_t stream);
// Split-K workspace: per (sequence, head, partition) an unnormalised output
// row and its (max, sum) pair, in fp32.  `counters` holds one int per
// (sequence, head); it must be all zero before the first launch and every
// launch leaves it all zero again.
size_t decode_workspace_bytes(int num_seqs, int num_heads, int max_parts);
cudaError_t launch_paged_decode(const void *q, const void *k_cache, const void *v_cache,
                                const int *block_tables, const int *context_lens, void *out,
                                int num_seqs, int num_heads, int max_blocks, float scale,
                                float *workspace, int *counters, cudaStream_t stream);

}  // namespace fattn
