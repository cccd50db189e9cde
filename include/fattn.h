/*
 * fattn.h -- C ABI of libfattn: exact scaled-dot-product attention on one
 * NVIDIA GB300 (sm_103a).
 *
 * Every call takes plain device pointers and sizes, enqueues its kernels on
 * `stream` and returns without synchronising.  Nothing here depends on any
 * framework's tensor types.  Unless a call says otherwise:
 *
 *  - All tensor arguments are DEVICE pointers owned by the caller, dense and
 *    C-contiguous (row-major) in the layout stated for them, and must stay
 *    valid until the enqueued work has finished.
 *  - bf16 means IEEE-style bfloat16 (1 sign, 8 exponent, 7 mantissa bits),
 *    passed as `void *`.
 *  - The return value is an fa_status_t.  Argument errors are detected on the
 *    host before anything is enqueued and return a negative code; no call
 *    ever aborts the process or asserts.  A kernel launch failure returns
 *    FA_ERR_CUDA.  Errors that only the device can see (a pipeline wait that
 *    exceeded its time limit) are latched in a per-device status word that
 *    fa_device_status() reads.
 *  - NaN or Inf inputs are not checked for; they propagate per IEEE rules.
 *
 * The library owns only small per-device state: the split-K workspace of the
 * paged decodes and its counters, the block summary of the last boolean mask,
 * the work counters of the persistent kernels and the last TMA views of a
 * paged cache; fa_release() frees it.  Calls on one device from several host
 * threads are safe.  The decode workspace and the mask summary are one
 * buffer per device: calls that use the same one (fa_paged_decode and
 * fa_paged_decode_gqa with each other; fa_forward_masked with itself) must
 * not overlap on the GPU -- issue them on one stream, or make the later
 * call's stream wait for an event recorded after the earlier call.  These
 * buffers grow in stream order on the calling stream (cudaMallocAsync and
 * cudaFreeAsync), so a larger problem never synchronises the device; a call
 * being captured into a CUDA graph cannot grow them and returns
 * FA_ERR_UNSUPPORTED instead, so run one call of the largest size before
 * capturing.  The forward kernels, the backward's main kernel and the
 * tensor-core grouped decode take a pair of work counters per launch: eager launches rotate through 64 pairs,
 * launches captured into a graph through 64 others that a graph keeps for
 * every replay; so at most 64 eager calls may be in flight on a device at
 * once, and a graph must not run concurrently with itself.
 */
#ifndef FATTN_H_
#define FATTN_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = -1,  /* null pointer, negative size, inconsistent sizes */
    FA_ERR_UNSUPPORTED = -2,  /* a size the kernels are not built for (e.g. d) */
    FA_ERR_ALIGNMENT = -3,    /* a pointer not 16-byte aligned */
    FA_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed */
    FA_ERR_TIMEOUT = -5,      /* a device-side wait exceeded its limit */
    FA_ERR_NO_MEMORY = -6,    /* the library could not allocate its workspace */
    FA_ERR_NO_DEVICE = -7     /* no usable sm_103 device is current */
} fa_status_t;

/*
 * fa_forward -- exact attention forward, bf16 in / bf16 out, fp32 LSE.
 *
 * Computes, for every batch b < B, head h < H and query row i < N,
 *     O[b,h,i,:] = sum_j softmax_j(scale * Q[b,h,i,:] . K[b,h,j,:]) V[b,h,j,:]
 *     lse[b,h,i] = ln sum_j exp(scale * Q[b,h,i,:] . K[b,h,j,:])
 * over the visible keys j: all j < N, or j <= i when causal != 0 (the
 * causal mask fused in the kernel, as in section 11.3 of "FlashAttention:
 * GPU 메모리 계층을 활용한 어텐션 최적화 분석", youngju.dev).  The row is
 * evaluated tile by tile with the online-softmax running max and running sum
 * of "Flash Attention" (suniverse77.github.io, section "Online Softmax",
 * eqs. (2)-(4)), so the N x N score matrix never reaches device memory.
 *
 *   q, k, v  bf16 [B, H, N, d], read only.
 *   o        bf16 [B, H, N, d], written (rounded to nearest even).
 *   lse      fp32 [B, H, N] natural-log log-sum-exp of the scaled scores,
 *            written; may be NULL when the caller does not need it.
 *   d        head dimension: 64, 128 or 256 (else FA_ERR_UNSUPPORTED; section
 *            11.4 of the same page serves head dimensions up to 256).
 *   scale    multiplier applied to every score before the softmax (usually
 *            1/sqrt(d)); must be finite and > 0.
 *   causal   0 or non-zero.
 * Products are accumulated in fp32 on the tensor cores; the softmax weights
 * are rounded to bf16 before they multiply V.  B*H or N equal to 0 is a
 * no-op that returns FA_OK.  q, k, v, o, lse must be 16-byte aligned.
 */
int fa_forward(const void *q, const void *k, const void *v, void *o, float *lse,
               int B, int H, int N, int d, float scale, int causal,
               fa_stream_t stream);

/*
 * fa_forward_f16 -- fa_forward with IEEE fp16 q, k, v and o (1 sign, 5
 * exponent, 10 mantissa bits): the same operation, layouts, lse and errors.
 * The softmax weights are rounded to fp16 before they multiply V, and o is
 * rounded to nearest even fp16; inputs must be finite and |o| below 65504.
 */
int fa_forward_f16(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int H, int N, int d, float scale, int causal,
                   fa_stream_t stream);

/*
 * fa_forward_masked -- fa_forward with a boolean attention mask in place of
 * the causal flag ("FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화 분석",
 * youngju.dev, section 11.3: a custom boolean attn_mask, True = the key takes
 * part).  Key j is visible to query row i of head bh = b * H + h iff
 *     mask[bh * mask_bh_stride + i * N + j] != 0;
 * mask_bh_stride = 0 shares one [N, N] mask across batch and heads, N * N
 * gives every head its own.  mask is uint8, 16-byte aligned, N must be a
 * multiple of 16 (else FA_ERR_UNSUPPORTED) and mask_bh_stride a multiple of
 * 16 (else FA_ERR_ALIGNMENT).  A row with no visible key gets o = 0 and
 * lse = -inf.  Each call first summarises the mask per 128 x 128 block (one
 * read of the mask): key tiles that none of a query block's rows can see are
 * skipped, fully visible blocks are not read again, and a partly visible
 * block is read back as 16 bytes of visibility bits per row (N * N / 8 bytes
 * per mask head in all) instead of its 128 mask bytes.  The summary lives
 * in a library-owned buffer grown on demand in stream order; two masked
 * calls must not overlap on the GPU (order them on one stream or with an
 * event).  d is 64 or 128.  Other arguments, layouts and errors as for
 * fa_forward (bf16).
 */
int fa_forward_masked(const void *q, const void *k, const void *v, void *o, float *lse,
                      const void *mask, long long mask_bh_stride, int B, int H, int N, int d,
                      float scale, fa_stream_t stream);

/*
 * FP8 forward ("FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화 분석",
 * youngju.dev, section 9.2, item 3: FP8 low-precision support with block
 * quantization and incoherent processing).  Two calls: fa_quantize_fp8 codes
 * bf16 Q, K, V as E4M3 with per-block scales, fa_forward_fp8 runs the forward
 * on the codes.  d must be 128 (else FA_ERR_UNSUPPORTED).  E4M3: 1 sign, 4
 * exponent (bias 7) and 3 mantissa bits, largest finite value 448, byte
 * 0x7F/0xFF is NaN and is never written.
 *
 * fa_quantize_fp8_workspace_bytes -- bytes of device workspace that
 * fa_quantize_fp8 needs: 4 * B*H*ceil(N/128).  0 for negative sizes.
 *
 * fa_fp8_vt_stride -- Npad, the number of keys per row of the transposed V
 * codes: N rounded up to a multiple of 16.  0 for negative N.
 *
 * fa_quantize_fp8 -- in: q, k, v bf16 [B, H, N, 128] (contiguous, 16-byte
 * aligned); signs: null, or 128 fp32 values each +1 or -1 (device, 16-byte
 * aligned), the diagonal of the random orthogonal transform
 * M = diag(signs) H / sqrt(128) (H the Sylvester-Hadamard matrix) applied to
 * the rows of q and k (not v) before quantization; q M (k M)^T = q k^T.
 * out (device, caller-allocated):
 *   q8, k8    E4M3 [B, H, N, 128] (16-byte aligned);
 *   vt8       E4M3 [B, H, 128, Npad], V transposed (16-byte aligned), codes
 *             past N are zero;
 *   q_scale, k_scale  fp32 [B, H, ceil(N/128)]: one dequantization scale per
 *             block of 128 rows;  v_scale  fp32 [B, H]: one per head.
 * Per block, s = amax / 448 in fp32 (1 for an all-zero block) and a value x
 * (a row of q M or k M when signs are given, the fp32 butterfly
 * (x * signs) H without the 1/sqrt(128)) is coded as E4M3 of x * (1/s),
 * rounded to nearest even and saturated to +-448; the stored scale is s, or
 * s * fp32(1/sqrt(128)) with signs, so that code * scale stands for the
 * value.  workspace: at least fa_quantize_fp8_workspace_bytes bytes of device
 * memory (4-byte aligned), used during the call only; calls that may run at
 * the same time need separate workspaces.  Errors: FA_ERR_INVALID_ARG (null
 * pointer, negative size, workspace too small), FA_ERR_ALIGNMENT,
 * FA_ERR_UNSUPPORTED (d != 128, B*H > 65535 or N > 2^30), FA_ERR_CUDA.
 * Asynchronous on `stream`; B*H = 0 or N = 0 does nothing.
 *
 * fa_forward_fp8 -- o = softmax(scale * Qd Kd^T [+ causal mask]) Vd and lse
 * as in fa_forward, where Qd, Kd, Vd are the dequantized inputs (codes times
 * scales, with the buffers and layouts fa_quantize_fp8 writes).  Q Kd^T is
 * formed by E4M3 tensor-core products accumulated in fp32; the softmax
 * weights are rounded to E4M3 (relative error <= 2^-4, absolute <= 2^-14 of
 * the row maximum) before the product with V; lse is computed from the
 * unrounded weights.  o is bf16 [B, H, N, 128], lse fp32 [B, H, N] (may be
 * null).  Errors and the async contract as for fa_forward.
 */
unsigned long long fa_quantize_fp8_workspace_bytes(int B, int H, int N, int d);
long long fa_fp8_vt_stride(int N);
int fa_quantize_fp8(const void *q, const void *k, const void *v, const float *signs, void *q8,
                    void *k8, void *vt8, float *q_scale, float *k_scale, float *v_scale, int B,
                    int H, int N, int d, void *workspace, unsigned long long workspace_bytes,
                    fa_stream_t stream);
int fa_forward_fp8(const void *q8, const void *k8, const void *vt8, const float *q_scale,
                   const float *k_scale, const float *v_scale, void *o, float *lse, int B, int H,
                   int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * fa_forward_fp32 -- the same operation and contract as fa_forward with fp32
 * q, k, v and o (every product and sum in fp32 on the CUDA cores, no reduced
 * precision anywhere).  d is 64 or 128.
 */
int fa_forward_fp32(const float *q, const float *k, const float *v, float *o, float *lse,
                    int B, int H, int N, int d, float scale, int causal,
                    fa_stream_t stream);

/*
 * fa_backward_workspace_bytes -- size in bytes of the fp32 workspace that
 * fa_backward needs for these sizes: 4 * B*H*Npad*(d + 2) with Npad = N
 * rounded up to a multiple of 128 (an fp32 dQ accumulator, then two fp32
 * vectors per 128-query block).
 * Returns 0 for negative sizes.
 */
unsigned long long fa_backward_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_backward -- gradients of the bf16 exact-attention forward.
 *
 * For the forward O = softmax(scale * Q K^T [+ causal mask]) V of
 * fa_forward and an upstream gradient dO, computes dQ, dK and dV by the
 * recomputation scheme of section 7 of "FlashAttention: GPU 메모리 계층을
 * 활용한 어텐션 최적화 분석" (youngju.dev): the probabilities are rebuilt
 * tile by tile from Q, K and the forward's saved lse, P = exp(S - lse), and
 * with D_i = sum_c dO[i,c] O[i,c]:
 *     dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
 *     dQ = scale * dS K,  dK = scale * dS^T Q.
 * No N x N matrix reaches device memory.
 *
 *   q, k, v, o, dout  bf16 [B, H, N, d], read only; o and lse are what
 *                     fa_forward returned for these q, k, v, scale, causal.
 *   lse               fp32 [B, H, N] natural-log LSE from fa_forward.
 *   dq, dk, dv        bf16 [B, H, N, d], written.
 *   workspace         device memory owned by the caller, at least
 *                     fa_backward_workspace_bytes(B, H, N, d) bytes, 16-byte
 *                     aligned; its contents on entry do not matter and are
 *                     scratch afterwards.  Two calls whose work overlaps on
 *                     the GPU need separate workspaces.
 *   d, scale, causal  as for fa_forward.
 * Products accumulate in fp32 on the tensor cores; P and dS are rounded to
 * bf16 before they multiply dO, Q and K; dQ is summed over key blocks in
 * fp32 with atomic adds, so its last bits may vary from run to run.
 * FA_ERR_INVALID_ARG when workspace is NULL or smaller than needed; the
 * other errors as for fa_forward.  B*H or N equal to 0 is a no-op.
 */
int fa_backward(const void *q, const void *k, const void *v, const void *o,
                const void *dout, const float *lse, void *dq, void *dk, void *dv,
                int B, int H, int N, int d, float scale, int causal,
                void *workspace, unsigned long long workspace_bytes,
                fa_stream_t stream);

/*
 * fa_paged_decode -- single-query attention over a paged KV cache.
 *
 * One query token per sequence attends to all context_lens[s] tokens of its
 * sequence, whose keys and values live in fixed-size cache blocks found
 * through the block table ("PagedAttention", data-sketchers.com, sections
 * "Inputs", "Concepts", "Key" and "Value").  Token t of sequence s is stored
 * in physical block pb = block_tables[s * max_num_blocks_per_seq +
 * t / block_size] at offset t % block_size; with x = 8 (bf16 elements in 16
 * bytes), element c of its key is k_cache[pb][h][c / x][t % block_size][c % x]
 * and element c of its value is v_cache[pb][h][c][t % block_size].
 *
 *   q             bf16 [num_seqs, num_heads, head_size], read only.
 *   k_cache       bf16 [num_blocks, num_heads, head_size/8, block_size, 8].
 *   v_cache       bf16 [num_blocks, num_heads, head_size, block_size].
 *   block_tables  int32 [num_seqs, max_num_blocks_per_seq]; entries past the
 *                 sequence's last used block are never read.  Entries that
 *                 are read must be valid block numbers (not checked: the
 *                 caller owns the cache and knows num_blocks).
 *   context_lens  int32 [num_seqs], each in [0, max_num_blocks_per_seq *
 *                 block_size] (not checked on the device).  A sequence with
 *                 context 0 gets an all-zero output row.
 *   out           bf16 [num_seqs, num_heads, head_size], written.
 *   head_size     128;  block_size 16 (else FA_ERR_UNSUPPORTED).
 *   scale         score multiplier, finite and > 0.
 * num_kv_heads equals num_heads.  Long contexts are split into partitions
 * of 512 tokens whose partial (max, sum, output) triples are merged with the
 * output update of eq. (4) of the "Flash Attention" page; the partials live
 * in a workspace the library owns and grows, in stream order on `stream`,
 * the first time a problem needs more (cudaFreeAsync of the smaller buffer,
 * then cudaMallocAsync; the device is not synchronised).  That workspace is
 * one per device and is shared with fa_paged_decode_gqa: two decode calls
 * whose work could overlap on the GPU return wrong results; order them on
 * one stream, or make the second call's stream wait on an event recorded
 * after the first.  num_seqs == 0 is a no-op.
 */
int fa_paged_decode(const void *q, const void *k_cache, const void *v_cache,
                    const int *block_tables, const int *context_lens, void *out,
                    int num_seqs, int num_heads, int head_size, int block_size,
                    int max_num_blocks_per_seq, float scale, fa_stream_t stream);

/*
 * fa_paged_decode_gqa -- fa_paged_decode with grouped key/value heads:
 * num_heads query heads share num_kv_heads cached key/value heads.
 *
 * The caches carry a key/value head axis of num_kv_heads ("PagedAttention",
 * data-sketchers.com, section "Inputs": k_cache [num_blocks, num_kv_heads,
 * head_size/x, block_size, x], v_cache [num_blocks, num_kv_heads, head_size,
 * block_size]; section "Key" offsets the key pointer by kv_head_idx).  Query
 * head h attends with key/value head h / (num_heads / num_kv_heads), i.e.
 * consecutive query heads share one cached head (num_kv_heads = 1 is
 * multi-query attention).  q and out are [num_seqs, num_heads, head_size].
 * Each cached block is read once for up to 16 query heads of its group
 * (tensor-core kernel) or four (CUDA-core kernel).  Cache slots past a
 * sequence's context may hold any bits, NaN included: they never reach the
 * output.
 *
 * Arguments and errors as for fa_paged_decode, plus: FA_ERR_INVALID_ARG when
 * num_kv_heads <= 0 or does not divide num_heads; FA_ERR_UNSUPPORTED when the
 * selected kernel does not take the group size num_heads / num_kv_heads.  By
 * default sizes 1 to 16 and every multiple of 4 are taken; see
 * fa_decode_gqa_select.
 * Group size 1 is exactly fa_paged_decode.  Shares fa_paged_decode's
 * library-owned workspace, with the same ordering rule: decode calls must
 * not overlap on the GPU.
 */
int fa_paged_decode_gqa(const void *q, const void *k_cache, const void *v_cache,
                        const int *block_tables, const int *context_lens, void *out,
                        int num_seqs, int num_heads, int num_kv_heads, int head_size,
                        int block_size, int max_num_blocks_per_seq, float scale,
                        fa_stream_t stream);

/*
 * fa_decode_gqa_select -- chooses which kernel fa_paged_decode_gqa runs for
 * group sizes 2 and up (process-wide, every device; takes effect at the next
 * call).
 *
 *  impl 0 (the default): automatic -- the tensor-core kernel for group sizes
 *         3 and up when num_seqs x num_kv_heads x ceil(max_num_blocks_per_seq
 *         / 32) is at least 152, and for the sizes only it takes; otherwise
 *         the CUDA-core kernel (group 2, and small problems, where it is
 *         faster).
 *  impl 1: the CUDA-core kernel only (group 2 or a multiple of 4): up to four
 *         query heads per pass over a cached block, fp32 FMAs.
 *  impl 2: the tensor-core kernel only (group 2 to 16, or a multiple of 16):
 *         128 context tokens are the M rows and up to 16 query heads the N
 *         columns of tcgen05 MMAs; P is rounded to bf16 for the P V product.
 *
 * Both compute the same attention; results differ in rounding only.  Returns
 * FA_OK, or FA_ERR_INVALID_ARG for another impl.
 */
int fa_decode_gqa_select(int impl);

/*
 * fa_paged_decode_noalloc -- fa_paged_decode for callers that cannot allocate
 * device memory during a call.  The attention pages have no counterpart to
 * this entry point; it exists for deployment reasons only.
 *
 * Some callers are not allowed to allocate at call time: a serving process
 * that hands all device memory to its own pool at start-up, a latency-bound
 * loop that cannot accept the synchronisation cudaMalloc/cudaFree may cause,
 * a plug-in whose host framework owns every allocation.  fa_paged_decode grows
 * a library-owned workspace on first use; this call instead keeps the split-K
 * partials and counters in a fixed 12 MiB device array that is part of the
 * library image (each device that loads the library holds it until the
 * process exits), and it calls no allocating CUDA or library routine.
 *
 * Arguments, layouts, result and errors are those of fa_paged_decode, plus:
 *  - FA_ERR_UNSUPPORTED when the problem needs more than the 12 MiB:
 *    round_up_256(4 * num_seqs * num_heads) +
 *    520 * num_seqs * num_heads * ceil(max_num_blocks_per_seq / 32) bytes
 *    (64 sequences x 32 heads x 256 blocks needs about 8.5 MB).
 *  - Every call on a device shares the one array and leaves its contents in
 *    place; the counters that must start at zero are cleared on `stream` at
 *    the start of each call.  Calls whose work overlaps on the GPU race on
 *    the array: order them on one stream or with events.
 *  - Each call looks up the array's device address with
 *    cudaGetSymbolAddress on the current device.  The first lookup on a
 *    device may load the library's module there, so make the first call on
 *    each device before any stream capture begins.
 */
int fa_paged_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                            const int *block_tables, const int *context_lens, void *out,
                            int num_seqs, int num_heads, int head_size, int block_size,
                            int max_num_blocks_per_seq, float scale, fa_stream_t stream);

/*
 * fa_debug_inject_fault -- test hook for the device-side failure path.
 *
 * mode 1 arms the current device: the next tensor-core forward launched on
 * it (fa_forward, fa_forward_f16, fa_forward_masked or fa_forward_fp8, for
 * head dimension 64 or 128) makes its first CTA's TMA producer stop after
 * loading that CTA's first query tiles, as if a copy had been lost.  The MMA warp's bounded wait for the
 * missing key tile then runs out (after about 2 s), the CTA unwinds (in-flight
 * copies and MMAs drained, tensor memory freed) and fa_device_status()
 * returns FA_ERR_TIMEOUT.  That launch's output is incomplete; the CUDA
 * context and the library stay usable.  mode 2 does the same to the next
 * fa_backward: its main kernel's first CTA loses the K and V copies of its
 * first work item.  mode 0 disarms.  Returns FA_OK, or FA_ERR_INVALID_ARG
 * for another mode, or FA_ERR_NO_DEVICE.
 */
int fa_debug_inject_fault(int mode);

/* Human-readable name of a status code (static string, never NULL). */
const char *fa_status_string(int status);

/*
 * Reads and clears the current device's latched device-side status
 * (FA_OK or FA_ERR_TIMEOUT).  Synchronises the device first.
 */
int fa_device_status(void);

/* Frees the library-owned per-device state on the current device, after
 * synchronising the device.  No libfattn call may be enqueued or captured
 * concurrently with it. */
void fa_release(void);

/* Library version as major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H_ */
