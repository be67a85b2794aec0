/*
 * kvq.h -- C ABI of libkvq: decode attention over a sub-byte quantized paged KV cache
 * on NVIDIA GB300 (sm_103a).
 *
 * Operations (the method follows the pages int4_per_token_head.py,
 * triton_turboquant_decode.py and kpool_compress.py of tduncan/Nvidia-Optimization-Stack-VLLM):
 *   kvq_write_int4    reshape_and_cache_int4 / _reshape_cache_int4_kernel
 *   kvq_decode_int4   unified_attention_int4 / _attn_packed (split-KV) + log-sum-exp merge
 *   kvq_decode_tq     triton_turboquant_decode_attention / _tq_decode_stage1 (KEY_FP8) + merge
 *   kvq_fwht128       fwht128_quant_fp8 / _fwht_quant_kernel
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer owned by the caller (kvq_copy_async also takes
 *     pinned host memory); the library allocates no memory on any call path and keeps no
 *     pointer after the call returns.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default stream). KVQ_OK means
 *     the kernels were enqueued; data-dependent errors detected on the device (a block id
 *     outside [0, num_blocks), a slot outside the pool, a sequence longer than its block-table
 *     row) skip the offending access and raise a sticky device flag that kvq_device_error()
 *     reports.
 *   - Arguments are validated before anything is launched; a rejected call launches nothing
 *     and returns KVQ_ERR_INVALID_ARG or KVQ_ERR_UNSUPPORTED. Empty work (T == 0, rows == 0,
 *     B == 0) is a successful no-op.
 *   - Layouts are C-contiguous unless strides are given. Sizes are element counts.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

struct CUstream_st;
/* The same type as cudaStream_t. */
typedef struct CUstream_st *kvq_stream_t;

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, inconsistent sizes or strides    */
  KVQ_ERR_UNSUPPORTED = 2,  /* a shape outside the compiled set (D, block size, group)   */
  KVQ_ERR_WORKSPACE = 3,    /* workspace smaller than kvq_decode_workspace_bytes()        */
  KVQ_ERR_OUT_OF_RANGE = 4, /* device-side index check failed (see kvq_device_error)     */
  KVQ_ERR_CUDA = 5          /* a CUDA runtime call or kernel launch failed                */
} kvq_status;

typedef enum { KVQ_BF16 = 0, KVQ_F16 = 1, KVQ_F32 = 2 } kvq_dtype;

/* Static, human-readable name of a status. Never NULL. */
KVQ_API const char *kvq_status_string(kvq_status status);

/* ABI revision of this header (bumped on any signature or struct change). */
KVQ_API int32_t kvq_abi_version(void);

/*
 * kvq_write_int4 -- rotate, quantize to INT4 and scatter K and V rows into the paged cache.
 * Defined by int4_per_token_head.py, reshape_and_cache_int4 and _reshape_cache_int4_kernel.
 *
 * For every token t with slot_mapping[t] >= 0 and every kv head h, separately for K and V:
 *   r = bf16(H_D (x * rht_signs))    unnormalised Walsh-Hadamard butterfly in fp32, cast to bf16
 *                                     (identity when rht_signs == NULL)
 *   scale = max((max r - min r) / 15, 1e-6); zp = clamp(round_half_away(-min r / scale), 0, 15)
 *   q_i = clamp(round_half_away(r_i * (1/scale) + zp), 0, 15)     (IEEE fp32, no fused mul-add)
 *   cache[slot / block_size][slot % block_size][h][j] = q_{2j} | q_{2j+1} << 4
 *   scale_cache[...][h] = fp32 word (bits(scale) & ~0xF) | zp
 * The result is bit-exact: the same bytes for the same inputs, whatever the launch.
 *
 *   key, value        bf16 [T, Hk, D]; element (t, h, d) at ptr + t*stride_t + h*stride_h + d.
 *                     Base 16-byte aligned; strides multiples of 8 elements.
 *   k_cache, v_cache  uint8 [num_blocks, block_size, Hk, D/2], 16-byte aligned.
 *   k_scale, v_scale  fp32 words [num_blocks, block_size, Hk], 4-byte aligned.
 *   slot_mapping      int64 [T]; entries < 0 are skipped; entries >= num_blocks*block_size are
 *                     skipped and flagged. Two tokens with the same slot race (caller error).
 *   rht_signs         fp32 [D] of +1/-1, or NULL for no rotation; 16-byte aligned. Only each
 *                     entry's sign bit is read (the flip x * (+-1) is exact).
 *   D                 64 or 128.
 */
KVQ_API kvq_status kvq_write_int4(const void *key, const void *value, int64_t k_stride_t,
                          int64_t k_stride_h, int64_t v_stride_t, int64_t v_stride_h,
                          uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale,
                          const int64_t *slot_mapping, const float *rht_signs, int32_t T,
                          int32_t Hk, int32_t D, int32_t block_size, int64_t num_blocks,
                          kvq_stream_t stream);

/*
 * kvq_decode_workspace_bytes -- scratch size for kvq_decode_int4 / kvq_decode_tq.
 * num_splits > 0: every sequence is cut into num_splits ranges of ceil(L / num_splits) positions
 * (triton_turboquant_decode.py, _tq_decode_stage1). num_splits == 0: the library balances the
 * pages of the whole batch over a fixed number of CTAs derived from the CURRENT device's SM
 * count, so query with the device that will run the call current. Returns 0 for invalid sizes.
 */
KVQ_API size_t kvq_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                  int32_t num_splits);

/*
 * kvq_decode_int4 -- paged decode attention over the INT4 cache written by kvq_write_int4.
 * Defined by int4_per_token_head.py, unified_attention_int4 and _attn_packed (decode, 3D mode),
 * with the split results combined by a log-sum-exp merge (the reduce_segments step).
 *
 *   q_rot = bf16(H_D (q * rht_signs));  sm = softmax_scale / D          (rht_signs != NULL)
 *   for b, query head hq (kv head hq / (Hq/Hk)), positions n < seq_lens[b]:
 *     k_n, v_n = (nibble - zp) * scale' read from page block_table[b][n / 16], row n % 16
 *     o = sum_n softmax_n(sm * q_rot . k_n) v_n
 *   out[b][hq] = H_D(o) * rht_signs / D   (o itself when rht_signs == NULL, with sm = softmax_scale)
 * Rows with seq_lens[b] == 0 are written as zeros.
 *
 *   q            bf16 [B, Hq, D] contiguous, 16-byte aligned.
 *   k_cache...   as kvq_write_int4; block_size must be 16. The decode reads pages with TMA
 *                tensor copies, so k_scale and v_scale must be 16-byte aligned here.
 *   block_table  int32 [B, max_blocks]; entries at or past page ceil(seq_lens[b]/16) are not read.
 *   seq_lens     int32 [B]; values are clamped to [0, 16*max_blocks] (a clamp raises the flag).
 *   workspace    >= kvq_decode_workspace_bytes(B, Hq, Hk, D, num_splits) bytes, 16-byte aligned;
 *                holds the rotated query's MMA fragments (written by a pre-kernel) and the
 *                per-split partial results between the split kernel and the merge kernel (all
 *                three enqueued by this call). Contents need no initialisation and are
 *                clobbered. Calls that share a workspace must be ordered on one stream.
 *   out          [B, Hq, D] of out_dtype (KVQ_BF16 / KVQ_F16 / KVQ_F32), contiguous, written in full.
 *   Supported: D in {64, 128}; Hq % Hk == 0 with Hq / Hk <= 8; Hk in {1, 2, 4, 8} or a multiple of 8.
 * Numerics: fp32 accumulation (tensor-core products of exact nibbles with fp16 operands);
 * agrees with the float64 definition on the same cache to well within 2e-3 abs / 1e-2 rel.
 */
KVQ_API kvq_status kvq_decode_int4(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                           const float *k_scale, const float *v_scale,
                           const int32_t *block_table, int32_t max_blocks,
                           const int32_t *seq_lens, const float *rht_signs, float softmax_scale,
                           int32_t num_splits, void *workspace, size_t workspace_bytes,
                           void *out, kvq_dtype out_dtype, int32_t B, int32_t Hq, int32_t Hk,
                           int32_t D, int32_t block_size, int64_t num_blocks,
                           kvq_stream_t stream);

/*
 * kvq_score_mods / kvq_decode_int4_mods -- kvq_decode_int4 with the score modifiers of
 * unified_attention_int4 (int4_per_token_head.py): SLIDING_WINDOW, USE_SOFTCAP, USE_ALIBI_SLOPES
 * and USE_SINKS, in the tile loop's order. With L = seq_lens[b] and the query at position L - 1:
 *   S_n = sm * q_rot . k_n                                  (as kvq_decode_int4)
 *   S_n = softcap * tanh(S_n / softcap)                     softcap > 0
 *   key n is read only if (L - 1) - n < sliding_window      sliding_window > 0 (0: every key)
 *   S_n += alibi_slopes[hq] * (n - (L - 1))                 alibi_slopes != NULL
 *   o = sum_n e^{S_n} v_n / (e^{sinks[hq]} + sum_n e^{S_n}) sinks != NULL (else without the sink)
 * The window also limits what is read: pages that hold no key of the window are skipped.
 *
 *   mods                NULL: exactly kvq_decode_int4. Otherwise host memory read during the call.
 *   mods->sliding_window  >= 0 keys (the query's own position counts).
 *   mods->softcap         >= 0, finite (natural-log units of S, like softmax_scale).
 *   mods->sinks           fp32 [Hq] device array (4-byte aligned) or NULL.
 *   mods->alibi_slopes    fp32 [Hq] device array (4-byte aligned) or NULL.
 *   mods->q_len           query tokens per sequence (0 or 1: one). Multi-token decode (the
 *                         speculative-verify case): q and out are [B * q_len, Hq, D], row
 *                         b * q_len + i the query at position L - q_len + i, attending causally
 *                         to keys n <= L - q_len + i (a query with no key gets a zero row).
 *   mods->query_start_loc int32 [B + 1] device array (4-byte aligned) or NULL: ragged multi-token
 *                         decode (unified_attention_int4's cu_seqlens_q). Sequence b has
 *                         q_b = query_start_loc[b + 1] - query_start_loc[b] query tokens (0 allowed),
 *                         rows query_start_loc[b] .. of q and out ([total_q, Hq, D]); token i sits at
 *                         position L - q_b + i and attends causally to keys n <= L - q_b + i. A row
 *                         range outside [0, total_q) is skipped and raises flag 2. Overrides q_len.
 *   mods->total_q         rows of q and out with query_start_loc (>= 0); ignored otherwise.
 *                         In multi-token decode every modifier applies per query token, relative to
 *                         its own position (window, ALiBi); the tokens of a sequence are served in
 *                         blocks of 8 / (Hq / Hk) that read the sequence's keys once per block, and
 *                         the workspace is kvq_decode_int4_mods_workspace_bytes(...).
 *   mods->lse_out         fp32 [rows, Hq] device array (4-byte aligned; rows as out) or NULL. When
 *                         set, each row's log-sum-exp ln(e^{sinks[hq]} + sum_n e^{S_n}) (without
 *                         the sink term when sinks == NULL; -inf for a row with no key and no
 *                         sink) is written next to out, so that the caller can merge this result
 *                         with attention over other keys (the lse_buf of
 *                         triton_turboquant_decode.py, triton_turboquant_decode_attention).
 * Invalid fields return KVQ_ERR_INVALID_ARG. Other arguments, numerics and errors: as
 * kvq_decode_int4.
 */
typedef struct kvq_score_mods {
  int32_t sliding_window;
  float softcap;
  const float *sinks;
  const float *alibi_slopes;
  int32_t q_len;
  float *lse_out;
  const int32_t *query_start_loc;
  int32_t total_q;
} kvq_score_mods;

/* Workspace bytes of kvq_decode_int4_mods with these mods (any multi-token layout); equal to
   kvq_decode_workspace_bytes when mods is NULL or single-token. 0 for invalid sizes. */
KVQ_API size_t kvq_decode_int4_mods_workspace_bytes(int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                                    int32_t num_splits, const kvq_score_mods *mods);

KVQ_API kvq_status kvq_decode_int4_mods(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                const float *k_scale, const float *v_scale,
                                const int32_t *block_table, int32_t max_blocks,
                                const int32_t *seq_lens, const float *rht_signs, float softmax_scale,
                                int32_t num_splits, void *workspace, size_t workspace_bytes,
                                void *out, kvq_dtype out_dtype, int32_t B, int32_t Hq, int32_t Hk,
                                int32_t D, int32_t block_size, int64_t num_blocks,
                                const kvq_score_mods *mods, kvq_stream_t stream);

/*
 * kvq_decode_int4_noalloc -- kvq_decode_int4 for callers that must not allocate device memory.
 * The pages have no counterpart of this call; it exists for users of this library, not for the
 * method.
 *
 * Some callers cannot call cudaMalloc or own a device buffer of their own: a plug-in inside a
 * serving process whose allocator has already reserved all of HBM for its paged KV pool, a C
 * caller with no access to the host framework's caching allocator, or a latency-critical path
 * where an allocation's implicit device synchronization is not acceptable. This entry point
 * takes the same arguments as kvq_decode_int4 except the workspace, which it replaces with a
 * file-scope device array of KVQ_NOALLOC_SCRATCH_BYTES bytes inside the library (every GPU that
 * loads the library holds that array until the process exits). It calls no allocating routine.
 *
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current); make that first call before any stream capture. The address
 *     is kept for the life of the process: after a cudaDeviceReset (or any teardown of the
 *     device's primary context) this entry point must not be called again in that process.
 *   - A call whose scratch need, kvq_decode_workspace_bytes(B, Hq, Hk, D, num_splits), exceeds
 *     KVQ_NOALLOC_SCRATCH_BYTES is rejected with KVQ_ERR_WORKSPACE before anything is launched.
 *   - Every call on a device shares the one array and overwrites what the previous call left
 *     there (nothing in it needs to start at zero). Calls that may overlap on the GPU -- on
 *     different streams without ordering, or from several threads -- race on it and corrupt
 *     each other's results: order them on one stream.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)
KVQ_API kvq_status kvq_decode_int4_noalloc(const void *q, const uint8_t *k_cache,
                                           const uint8_t *v_cache, const float *k_scale,
                                           const float *v_scale, const int32_t *block_table,
                                           int32_t max_blocks, const int32_t *seq_lens,
                                           const float *rht_signs, float softmax_scale,
                                           int32_t num_splits, void *out, kvq_dtype out_dtype,
                                           int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                           int32_t block_size, int64_t num_blocks,
                                           kvq_stream_t stream);

/*
 * kvq_decode_tq -- paged decode attention over the TurboQuant combined slot with FP8 keys.
 * Defined by triton_turboquant_decode.py, triton_turboquant_decode_attention and
 * _tq_decode_stage1 with KEY_FP8 = 1, followed by the split merge (_fwd_kernel_stage2).
 *
 * Slot of (page, row, kv head), slot_bytes long, slot_bytes % 16 == 0:
 *   [0, D)            E4M3FN key codes
 *   [D, D + VDB)      value indices, VDB = ceil(D * value_bits / 8): 4-bit two per byte (even d
 *                     low nibble), 3-bit an LSB-first bit stream
 *   [D + VDB, +2)     value scale, fp16 little-endian;  [D + VDB + 2, +4) value zero, fp16
 *   score = attn_scale * sum_d q_d * k_d;   v_d = idx_d * scale + zero
 *
 *   q         fp32 [B, Hq, D] contiguous (already in the cache's rotated space), 16-byte aligned.
 *   kv_cache  uint8 [num_blocks, block_size(=16), Hk, slot_bytes], 16-byte aligned.
 *   out       fp32 [B, Hq, D] contiguous; rows with seq_lens[b] == 0 are zeros.
 *   workspace as kvq_decode_int4.
 *   value_bits 3 or 4; D 64 or 128; other arguments as kvq_decode_int4.
 */
KVQ_API kvq_status kvq_decode_tq(const float *q, const uint8_t *kv_cache, int32_t slot_bytes,
                         int32_t value_bits, const int32_t *block_table, int32_t max_blocks,
                         const int32_t *seq_lens, float attn_scale, int32_t num_splits,
                         void *workspace, size_t workspace_bytes, float *out, int32_t B,
                         int32_t Hq, int32_t Hk, int32_t D, int32_t block_size,
                         int64_t num_blocks, kvq_stream_t stream);

/*
 * kvq_decode_tq_lse -- kvq_decode_tq that also returns each row's log-sum-exp, as
 * triton_turboquant_decode_attention returns lse_buf next to the output:
 *   lse_out[b][hq] = ln(sum_n e^{score_n})     (-inf for seq_lens[b] == 0)
 *   lse_out   fp32 [B, Hq] device array, 4-byte aligned, or NULL (then exactly kvq_decode_tq).
 * Everything else as kvq_decode_tq.
 */
KVQ_API kvq_status kvq_decode_tq_lse(const float *q, const uint8_t *kv_cache, int32_t slot_bytes,
                             int32_t value_bits, const int32_t *block_table, int32_t max_blocks,
                             const int32_t *seq_lens, float attn_scale, int32_t num_splits,
                             void *workspace, size_t workspace_bytes, float *out, float *lse_out,
                             int32_t B, int32_t Hq, int32_t Hk, int32_t D, int32_t block_size,
                             int64_t num_blocks, kvq_stream_t stream);

/*
 * kvq_decode_tq_mse -- TurboQuant decode with MSE keys. Defined by triton_turboquant_decode.py,
 * _tq_decode_stage1 with KEY_FP8 = 0 (NORM_CORRECTION optional) and
 * triton_turboquant_decode_attention with key_fp8 = False.
 *
 *   q_rot = q @ rotation^T                                    (fp32, computed by the call)
 *   per key n (slot of kv head hq / (Hq/Hk)): idx_d = key_bits-bit field d of the LSB-first
 *     stream at byte 0 (bits key_bits*d ..), c_d = centroids[idx_d];
 *     with norm_correction: c = c / sqrt(sum_d c_d^2 + 1e-16);
 *     norm = fp16 at byte MSE_BYTES = ceil(D * key_bits / 8);
 *     S_n = attn_scale * norm * (q_rot . c)
 *   values from byte key_packed_size: value_bits-bit indices (as kvq_decode_tq), fp16 scale and
 *   zero right after the ceil(D * value_bits / 8) value bytes; v = idx * scale + zero
 *   out[b][hq] = sum_n softmax_n(S_n) v_n  (fp32; zero rows for seq_lens[b] == 0)
 *
 *   q             fp32 [B, Hq, D] (the original query), 16-byte aligned.
 *   rotation      fp32 [D, D] (Pi), 16-byte aligned.   centroids  fp32 [2^key_bits].
 *   kv_cache      uint8 [num_blocks, 16, Hk, slot_bytes]; slot_bytes a multiple of 16, at most 512,
 *                 >= key_packed_size + ceil(D * value_bits / 8) + 4; that used part of a slot at
 *                 most 236 bytes (KVQ_ERR_UNSUPPORTED otherwise).
 *   key_bits, value_bits  3 or 4.   key_packed_size  even, >= MSE_BYTES + 2.
 *   workspace     >= kvq_decode_tq_mse_workspace_bytes(...) bytes, 256-byte aligned (holds q_rot
 *                 and the split partials); contents need no initialisation.
 *   Supported: D in {64, 128}; Hq / Hk <= 8; block_size 16. Errors as kvq_decode_tq.
 * Numerics: centroids and q_rot enter the tensor cores as fp16 hi + lo pairs (three products per
 * step, ~22 bits), fp32 accumulation; within 2e-3 abs / 1e-2 rel of the float64 definition.
 */
KVQ_API size_t kvq_decode_tq_mse_workspace_bytes(int32_t B, int32_t Hq, int32_t Hk, int32_t D,
                                         int32_t num_splits);

KVQ_API kvq_status kvq_decode_tq_mse(const float *q, const float *rotation, const float *centroids,
                             const uint8_t *kv_cache, int32_t slot_bytes, int32_t key_bits,
                             int32_t key_packed_size, int32_t value_bits, int32_t norm_correction,
                             const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                             float attn_scale, int32_t num_splits, void *workspace,
                             size_t workspace_bytes, float *out, int32_t B, int32_t Hq, int32_t Hk,
                             int32_t D, int32_t block_size, int64_t num_blocks, kvq_stream_t stream);

/*
 * kvq_kpool_write -- kpool compress-and-write: one FP8 cache entry per pool of pool_size tokens.
 * Defined by kpool_compress.py, _kpool_softmax_rotate_write_cache_kernel and
 * kpool_compress_and_write_cache (write_cache = True, return_compressed = False).
 *
 * For pool p with write_mask[p] (every pool when write_mask == NULL), per dimension d (fp32, each
 * operation rounded to nearest):
 *   z_s = slot_score[p][s][d] + ape[s][d];  M = max_s z_s;  w_s = exp(z_s - M)
 *   x_d = bf16(sum_s slot_k[p][s][d] * w_s / sum_s w_s)            (sums in slot order)
 *   y = bf16(H_128(x) * fp32(1/sqrt(128)));  a = max(max |y|, 1e-4)
 *   scale = smallest power of two >= a * fp32(1/448) (round_scale), else a * fp32(1/448)
 *   codes = E4M3FN(clamp(y / scale, -448, 448))
 *   page = loc[p] / page_size, row = loc[p] % page_size of kv_cache:
 *     bytes [row * 128, +128) of the page = codes; fp32 at byte page_size * 128 + 4 * row = scale.
 * exp is the library's fp32 exponential (within 1 ulp; results below 2^-125 are 0), so the codes
 * are reproducible bit for bit. Bytes of other pages and rows are not touched.
 *
 *   kv_cache    uint8 [num_blocks, page_size, 132], 16-byte aligned; page_size a multiple of 4.
 *   slot_k      bf16 [n_pools, pool_size, 128], contiguous, 16-byte aligned.
 *   slot_score  fp32 [n_pools, pool_size, 128], contiguous, 16-byte aligned.
 *   ape         fp32 [pool_size, 128], contiguous, 16-byte aligned.
 *   loc         int64 [n_pools]; a location outside [0, num_blocks * page_size) is skipped and flagged.
 *   write_mask  bool (one byte) [n_pools] or NULL.
 *   head_dim    must be 128 (KVQ_ERR_UNSUPPORTED otherwise). n_pools == 0 is a no-op.
 */
KVQ_API kvq_status kvq_kpool_write(uint8_t *kv_cache, const void *slot_k, const float *slot_score,
                           const float *ape, const int64_t *loc, const uint8_t *write_mask,
                           int64_t n_pools, int32_t pool_size, int32_t head_dim, int32_t page_size,
                           int64_t num_blocks, int32_t round_scale, kvq_stream_t stream);

/*
 * kvq_kpool_seed_tail / kvq_kpool_decode_update -- the kpool tail ring. Defined by kpool_compress.py,
 * _kpool_tail_seed_kernel / kpool_seed_tail_cache and _kpool_decode_update_batched_kernel /
 * kpool_decode_update_and_maybe_write_cache_batched.
 *
 * The tail cache is bf16 [tail_blocks][2][ring][128] addressed through tail_block_stride and
 * tail_half_stride (elements; the tail may alias a padded cache): half 0 keys, half 1 gate scores.
 *
 * Seed (prefill): token i (key / gate_score rows i, bf16 [n_tokens, 128]) with tslot[i] >= 0 is one
 *   of its request's last kpool tokens iff tslot[i + kpool] is past the batch, negative, or in
 *   another block (tslot / ring); such a token is copied to ring position tslot[i] % ring of block
 *   tslot[i] / ring.
 * Decode update: one request at a time is independent; within a request its next_n tokens run in
 *   order. For token (r, t) with pos = positions[r][t] >= 0:
 *     if slot_mapping[r][t] >= 0 and pos % pool_size == pool_size - 1: the pool ending at pos is
 *       compressed exactly as kvq_kpool_write does (its earlier slots from ring positions
 *       (pos - pool_size + 1 + j) % ring of block tail_slot[r][t] / ring, its last slot the current
 *       key and score, both bf16 here) and written at slot_mapping[r][t] of kv_cache;
 *     then, if tail_slot[r][t] >= 0, the current key and score are stored at ring position pos % ring.
 *   key, slot_score  bf16 [R, next_n, 128] with element strides (b, t) multiples of 4, last dim
 *                    contiguous; ape fp32 [pool_size, 128]; tail_slot_mapping, slot_mapping,
 *                    positions int32 [R, next_n] contiguous. ring >= pool_size, ring % pool_size == 0.
 *   kv_cache, page_size, num_blocks, round_scale: as kvq_kpool_write.
 * Block ids >= tail_blocks and locations outside the cache are skipped and flagged.
 */
KVQ_API kvq_status kvq_kpool_seed_tail(void *tail, int64_t tail_block_stride, int64_t tail_half_stride,
                               int32_t ring, int64_t tail_blocks, const void *key, const void *gate_score,
                               const int32_t *tslot, int64_t n_tokens, int32_t kpool, int32_t head_dim,
                               kvq_stream_t stream);

KVQ_API kvq_status kvq_kpool_decode_update(uint8_t *kv_cache, int32_t page_size, int64_t num_blocks, void *tail,
                                   int64_t tail_block_stride, int64_t tail_half_stride, int32_t ring,
                                   int64_t tail_blocks, const int32_t *tail_slot_mapping, const void *key,
                                   int64_t key_stride_b, int64_t key_stride_t, const void *slot_score,
                                   int64_t score_stride_b, int64_t score_stride_t, const float *ape,
                                   const int32_t *slot_mapping, const int32_t *positions,
                                   int32_t num_requests, int32_t next_n, int32_t pool_size, int32_t head_dim,
                                   int32_t round_scale, kvq_stream_t stream);

/*
 * kvq_fwht128 -- fused normalised Walsh-Hadamard-128 rotation + per-row power-of-two FP8 quant.
 * Defined by kpool_compress.py, fwht128_quant_fp8 and _fwht_quant_kernel.
 *   x = bf16(FWHT128(row) * fp32(0.08838834764831845));  a = max(max |x|, 1e-4)
 *   s = smallest power of two >= a * fp32(1/448);   y = e4m3_rne(clamp(x / s, -448, 448))
 *   x         bf16 [rows, 128] contiguous, 16-byte aligned.
 *   y_e4m3    uint8 [rows, 128] (E4M3FN codes), 16-byte aligned.    row_scale  fp32 [rows] (s).
 * Bit-exact.
 */
KVQ_API kvq_status kvq_fwht128(const void *x, uint8_t *y_e4m3, float *row_scale, int64_t rows,
                       kvq_stream_t stream);

/*
 * kvq_copy_async -- copy `bytes` bytes from src to dst with a kernel: the SMs' 16-byte loads and
 * stores (plumbing for a serving step; no counterpart on the pages). Either pointer may be device
 * memory or pinned host memory mapped into the device's address space (cudaHostAlloc /
 * cudaMallocHost, pinned torch tensors), which the SMs of a Grace-Blackwell node reach over the
 * coherent chip-to-chip link. A step's inputs can thus come in and its result go out as kernel
 * nodes of the step's CUDA graph, with no hand-off to a copy engine between kernels.
 *   dst, src   16-byte aligned, not overlapping; bytes a multiple of 16 (0: a no-op).
 * Returns KVQ_ERR_INVALID_ARG for a null or misaligned pointer, a size that is not a multiple of
 * 16, overlapping ranges, or a host pointer that is not pinned and mapped (checked with
 * cudaPointerGetAttributes before anything is launched).
 */
KVQ_API kvq_status kvq_copy_async(void *dst, const void *src, size_t bytes, kvq_stream_t stream);

/*
 * kvq_debug_set_wait -- for tests of the error path only (no counterpart on the pages).
 * Every wait of the decode kernels (INT4 and TurboQuant) on a page copy is bounded; when one runs
 * out the kernel raises flag 8, lets the copies it has issued land, and returns, so the context
 * stays usable. This call makes that path reachable on purpose, without any fault:
 *   wait_limit_ns   the limit of every such wait from now on in this process (0: the default, 2 s).
 *   withhold_stage  >= 0: the NEXT decode call (kvq_decode_int4, _int4_mods, _tq, _tq_lse or
 *                   _tq_mse; that one call only) does not issue the copies of that ring stage in
 *                   its first CTA (TurboQuant: of that ring tile of the CTA's first warp), so the
 *                   wait on it runs out after wait_limit_ns (plus ~0.1 s for the bounded drain) and
 *                   flag 8 is raised; that call's results are not valid. -1: none.
 * Returns KVQ_ERR_INVALID_ARG for withhold_stage < -1.
 */
KVQ_API kvq_status kvq_debug_set_wait(uint64_t wait_limit_ns, int32_t withhold_stage);

/*
 * kvq_device_error -- synchronize `stream`, then read and clear the sticky device-side flags
 * of every libkvq kernel on the current device. *flags (may be NULL) receives their bitwise OR:
 *   1 block-table entry outside [0, num_blocks)   2 seq_len above 16 * max_blocks (clamped)
 *   4 slot_mapping entry beyond the pool             8 a bounded wait on a page copy ran out
 *   16 a decode input outside the supported range: a query element beyond ~2^100 in magnitude
 *      (q, or q_rot for MSE keys, or a centroid), or a softmax weight beyond fp32 (value scales
 *      near fp32's maximum); the rows concerned may hold inf/NaN
 * Returns KVQ_OK when no flag was set, KVQ_ERR_OUT_OF_RANGE otherwise, KVQ_ERR_CUDA if the
 * synchronization or the read failed.
 */
KVQ_API kvq_status kvq_device_error(kvq_stream_t stream, uint32_t *flags);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
