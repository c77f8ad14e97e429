/*
 * pkv.h -- C ABI of libpkv: split-KV paged decode attention on GB300 (sm_103a).
 *
 * Two attention operations and the cache write that precedes them, each one
 * or two kernel launches on the caller's stream:
 *
 *  - pkv_paged_decode_attn: GQA decode.  Every request has one query token per
 *    query head; it attends to the keys of its KV cache, gathered page by page
 *    through a per-request block table, optionally restricted to a sliding
 *    window and with a per-head attention sink in the softmax denominator.
 *    Defined by "vllm.models.flint.ops.decode_attention" (flint_decode_attention:
 *    parameters and the module's numerics paragraph) and, for the block table,
 *    by the transformers page "Atencion paginada" (decode path).
 *
 *  - pkv_mla_verify_attn: MLA causal verify.  qlen consecutive verify tokens of
 *    a request, 128 query heads each, attend to one shared 576-wide latent head;
 *    V is the first 512 dims of the latent K; verify token t sees
 *    max(min(L - qlen + 1 + t, L_real), 0) keys.  The latent cache is bf16 or
 *    FP8 e4m3 with a scalar dequantisation factor.  Defined by
 *    "vllm.v1.attention.ops.triton_decode_attention"
 *    (decode_attention_fwd_verify: parameters).
 *
 *  - pkv_mla_quantize_q + pkv_mla_verify_attn_fp8_native: the same MLA verify
 *    over an FP8 cache with the query quantised to e4m3 per (row, head), so
 *    that the score MMAs run on 8-bit operands (an opt-in numerics change).
 *
 *  - pkv_gqa_kv_append / pkv_mla_kv_append: the step before either call,
 *    writing the current token (or the verify tokens' latent rows) into the
 *    paged cache in place through the same block table (transformers page,
 *    decode path).
 *
 * Both attention calls compute the fp32 online softmax of the pages (exp2 with the softmax
 * scale folded into log2(e), P rounded to bf16 for P.V, fp32 accumulation),
 * split each request's keys over several CTAs, and merge the fp32
 * (unnormalised O, running max m, sum l) partials of the splits into a bf16
 * output and a natural-log LSE that is -inf for rows with no key.
 *
 * Conventions shared by every entry point
 *  - Return value: PKV_OK (0) or a negative PKV_ERR_* code.  No call aborts
 *    the process.  The message of the last failure on the calling thread is
 *    returned by pkv_last_error().
 *  - Tensors are caller-owned device memory described by pkv_tensor (shape and
 *    strides in elements).  The library never frees caller memory.  It owns
 *    only its per-device workspace (split partials, arrival counters,
 *    scheduler words, error word), allocated once by pkv_init() or by the
 *    first call on a device, and never moved afterwards, so launches captured
 *    in a CUDA graph keep valid pointers.
 *  - Calls that share a device's workspace must be ordered on one stream (as
 *    within one model forward).  When a call arrives on a different stream
 *    than the previous call on that device (and neither is being captured),
 *    the new stream first waits for the previous one: the library records an
 *    event on the previous call's stream at that moment, so that stream must
 *    still exist (destroy a stream only after another call on the device has
 *    been made from a live stream, or after pkv_shutdown()).  No event is
 *    recorded between calls on one stream, which keeps consecutive launches
 *    overlapping (programmatic dependent launch).
 *  - Programmatic dependent launch: the attention kernels launch as dependents
 *    of the kernel before them on the stream and may start while it runs.
 *    Before waiting for it, pkv_paged_decode_attn (and its no-alloc variant)
 *    reads seq_lens, block_table and up to 8 tiles of the leading KV pages of
 *    each CTA's first work item -- never the page holding position
 *    seq_len - 1; the MLA verify calls' planning kernel reads seq_lens.  So
 *    seq_lens, block_table and the cache pages before the current token's
 *    must not be written by a kernel that may still be running when the
 *    call's kernel starts (the kernel immediately before it on the
 *    stream, or one an earlier dependent launch let run early).  Writing the
 *    current token's slot right before the call (pkv_gqa_kv_append) is fine,
 *    as is anything written by copies or by kernels that completed.  q, sinks,
 *    the workspace and all outputs are touched only after the wait.
 *  - The launch shape depends only on the device and the batch size, never on
 *    the sequence lengths or the block table, which the kernels read on the
 *    device: a captured graph stays valid when seq_lens and block_table change.
 *  - The call's device is the device holding its first tensor argument (q, or
 *    the cache for the append calls): it must be the current device and the
 *    stream's device, else PKV_ERR_INVALID_ARG.  (While the stream is being
 *    captured these pointer queries are skipped and the current device is
 *    used: a capture follows an eager call that has checked them.)  Outputs may not share memory
 *    with any input or with each other (PKV_ERR_INVALID_ARG): the kernels read
 *    the inputs of one request after writing the outputs of another.  A block
 *    table of width W over pages of P tokens needs W x P < 2^31.
 *  - Data-dependent input errors that the host cannot see (a block-table entry
 *    outside the cache, a seq_len longer than the block table) never fault:
 *    the kernel clamps or zero-fills, raises a bit in the device error word and
 *    finishes; pkv_check_errors() reads and clears that word.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_API __attribute__((visibility("default")))

/* Status codes. */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG -1     /* NULL pointer, bad shape, dtype or value */
#define PKV_ERR_UNSUPPORTED -2     /* valid but not built: head dim, page size, group size, batch */
#define PKV_ERR_ALIGNMENT -3       /* pointer or stride breaks a 16-byte rule */
#define PKV_ERR_WORKSPACE -4       /* the workspace cannot hold this call's split partials */
#define PKV_ERR_CAPTURE -5         /* workspace first needed while the stream is being captured */
#define PKV_ERR_CUDA -6            /* a CUDA runtime or driver call failed (see pkv_last_error) */
#define PKV_ERR_BAD_BLOCK_TABLE -7 /* reported by pkv_check_errors for bad block-table data */

/* Element types of pkv_tensor. */
#define PKV_DTYPE_BF16 1
#define PKV_DTYPE_F32 2
#define PKV_DTYPE_I32 3
#define PKV_DTYPE_FP8_E4M3 4 /* OCP float8 e4m3 ("fn": no infinities) */

/* A strided view of caller-owned device memory. */
typedef struct pkv_tensor {
  void* data;        /* device pointer */
  int32_t dtype;     /* PKV_DTYPE_* */
  int32_t ndim;      /* 0..5 (0 = scalar) */
  int64_t shape[5];  /* sizes of the first ndim dimensions */
  int64_t stride[5]; /* strides in elements */
} pkv_tensor;

/*
 * pkv_init -- allocate the workspace of `device` once (idempotent).
 *   workspace_bytes: bytes for split partials; 0 selects the default
 *   (1 GiB).  The first call on a device fixes the size; later calls are
 *   no-ops that return PKV_OK.  Also zeroes the arrival counters and the
 *   scheduler words, which the kernels keep at zero between calls.
 *   Errors: PKV_ERR_CAPTURE when called while the current stream of the
 *   device is capturing, PKV_ERR_CUDA when allocation fails.
 *   Source: "vllm.models.flint.ops.decode_attention", _workspace (persistent
 *   partials and counters allocated once per device at a fixed maximum,
 *   never replaced; counters zeroed only at allocation).
 */
PKV_API int pkv_init(int device, size_t workspace_bytes);

/*
 * pkv_paged_decode_attn -- GQA paged decode attention with sinks, one query
 * token per request.
 * Source: "vllm.models.flint.ops.decode_attention", flint_decode_attention
 * (parameters; numerics paragraph of the module; _launch_config /
 * _supports_kv_cache for the layout rules).
 *
 *   q            bf16 [B, Hq, 128]; last dim contiguous; strides multiples of 8;
 *                16-byte aligned.
 *   kv_cache     bf16 [num_blocks, Hkv, P, 256] HND pages: K in [..., :128],
 *                V in [..., 128:]; stride(3) == 1, stride(2) == 256,
 *                stride(0) and stride(1) multiples of 8; 16-byte aligned.
 *                Hq == 8 * Hkv: query head h reads kv head h / 8.
 *   block_table  int32 [B, max_blocks]; row b lists the physical block of
 *                each logical page of request b; entries past the request's
 *                last page (and before its window) are never read and may be
 *                -1.  stride(1) == 1.
 *   seq_lens     int32 [B]: attended positions of request b including the
 *                current token (keys [0, L)); 0 writes zeros and lse = -inf.
 *   sinks        fp32 [Hq] natural-log sink logits (not multiplied by scale),
 *                or NULL for none.  They enter only the output's denominator;
 *                lse is over the keys alone.
 *   window       > 0: attend to keys [max(L - window, 0), L); <= 0: all keys.
 *   scale        softmax scale applied to q.k.
 *   page_size    P, tokens per page: 16 or 32 (must equal kv_cache.shape[2]).
 *   num_kv_splits static cap on the number of KV splits of one (request, kv
 *                head); 0 selects the library's cap; values above 256 act as
 *                256.  Each request uses as many splits as its own length
 *                warrants (at least 256 keys per split), at most this many.
 *   out          bf16 [B, Hq, 128]; last dim contiguous; shares no memory with
 *                any input or with lse.
 *   lse          fp32 [B, Hq] or NULL.
 *   stream       cudaStream_t (NULL = legacy default stream).
 * B == 0 returns PKV_OK without launching.
 * Errors: PKV_ERR_INVALID_ARG (shapes, dtypes, overlapping outputs, q not on
 * the current device or the stream's), PKV_ERR_UNSUPPORTED (head dim != 128,
 * Hq != 8*Hkv, P not in {16, 32}, B > 2048), PKV_ERR_ALIGNMENT,
 * PKV_ERR_WORKSPACE (B * Hkv * cap partials do not fit; a cap of 1 needs
 * none), PKV_ERR_CAPTURE, PKV_ERR_CUDA.
 */
PKV_API int pkv_paged_decode_attn(const pkv_tensor* q, const pkv_tensor* kv_cache,
                                  const pkv_tensor* block_table, const pkv_tensor* seq_lens,
                                  const pkv_tensor* sinks, int window, float scale,
                                  int page_size, int num_kv_splits, const pkv_tensor* out,
                                  const pkv_tensor* lse, void* stream);

/*
 * pkv_paged_decode_attn_noalloc -- pkv_paged_decode_attn on scratch memory the
 * library never allocates.  The pages have no counterpart: this entry point
 * exists for callers that cannot let a library call cudaMalloc, e.g. a serving
 * engine that reserves all of HBM for its own KV-cache pool and treats any
 * other device allocation as an out-of-memory risk, or a framework whose
 * memory manager must own every device buffer.
 *
 * Arguments, layouts, results and error codes are those of
 * pkv_paged_decode_attn, and so is the launch shape (split cap, grid, items
 * per CTA), computed on this array's limits.  The split partials, arrival
 * counters, work-queue words and device error word live in one file-scope
 * __device__ array of about 8.2 MiB that every GPU loading the library holds
 * until the process exits.  Limits: batch x kv heads <= 4096, and batch x kv
 * heads x splits <= 2048 whenever a request may split (cap > 1; the cap is
 * chosen to fit when num_kv_splits is 0, falling to 1 above 1024 pairs);
 * larger calls return PKV_ERR_WORKSPACE and launch nothing.  The call
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine,
 * and it never touches the workspace of pkv_init.  Each call clears the
 * array's counters, queue words and error word with cudaMemsetAsync on
 * `stream` before its launch.
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress); make that first call before any stream
 *     capture.
 *   - Every call shares the one array: calls whose kernels may overlap on the
 *     GPU (different streams without ordering, different threads) race and
 *     give wrong results.  Order them on one stream.
 *   - Device-side errors of the last call are kept in the array's error word
 *     until the next call clears it; pkv_check_errors(device) reads (and
 *     clears) it together with the workspace's word: bit 1 a block-table
 *     entry outside the cache (the tile reads as zeros), bit 2 a seq_len
 *     longer than the block table (clamped), bit 4 a pipeline wait that gave
 *     up (that CTA drained; its outputs are wrong), bit 8 more work items
 *     than the array holds (the excess was dropped), bit 16 a CTA that drew
 *     more items than the launch has (it stopped).  Any bit other than 1 and
 *     2 means the outputs of that call are not to be trusted.
 */
PKV_API int pkv_paged_decode_attn_noalloc(const pkv_tensor* q, const pkv_tensor* kv_cache,
                                          const pkv_tensor* block_table,
                                          const pkv_tensor* seq_lens, const pkv_tensor* sinks,
                                          int window, float scale, int page_size,
                                          int num_kv_splits, const pkv_tensor* out,
                                          const pkv_tensor* lse, void* stream);

/*
 * pkv_mla_verify_attn -- causal MLA verify over a per-request block table.
 * Source: "vllm.v1.attention.ops.triton_decode_attention",
 * decode_attention_fwd_verify (parameters).
 *
 *   q             bf16 [B*qlen, H, 576], a request's verify tokens contiguous;
 *                 last dim contiguous; 16-byte aligned rows.
 *   latent_cache  bf16 or FP8 e4m3 [num_pages, P, 1, 576] (or
 *                 [num_pages*P, 1, 576]); one latent head; last dim contiguous;
 *                 pages 16-byte aligned.  V is latent[..., :512].
 *   block_table   int32 [B, max_pages].
 *   seq_lens      int32 [B], kernel KV lengths L.
 *   real_seq_lens int32 [B] or NULL (= seq_lens).  Verify token t of request b
 *                 attends to keys [0, max(min(L - qlen + 1 + t, L_real), 0)).
 *   qlen          verify tokens per request (>= 1).
 *   scale         softmax scale.
 *   page_size     P, tokens per page (16 or 32).
 *   k_scale       fp32 device scalar (ndim 0 or 1 element) dequantising an FP8
 *                 cache, or NULL (= 1); ignored for a bf16 cache.
 *   out           bf16 [B*qlen, H, 512].
 *   lse           fp32 [B*qlen, H]; -inf for rows with no key (their out is 0).
 *   num_kv_splits static cap on KV splits per request, 0 = the library's choice
 *                 (an addition to the page's list: the workspace the page passes
 *                 as attn_logits is owned by the library here).
 *   stream        cudaStream_t.
 * Errors: as pkv_paged_decode_attn; PKV_ERR_UNSUPPORTED unless Lk == 576,
 * Lv == 512 and H == 128.
 */
PKV_API int pkv_mla_verify_attn(const pkv_tensor* q, const pkv_tensor* latent_cache,
                                const pkv_tensor* block_table, const pkv_tensor* seq_lens,
                                const pkv_tensor* real_seq_lens, int qlen, float scale,
                                int page_size, const pkv_tensor* k_scale, const pkv_tensor* out,
                                const pkv_tensor* lse, int num_kv_splits, void* stream);

/*
 * pkv_mla_quantize_q -- per-(row, head) e4m3 quantisation of an MLA query, the
 * input of pkv_mla_verify_attn_fp8_native.  The pages give no recipe (the
 * verify page's FP8 path dequantises the cache by a scalar k_scale); this is
 * the library's reading: with a = max |q[r, h, :]| over the 576 bf16 values,
 * q_scale[r, h] = a / 448 in fp32 (round to nearest even; 1 when a = 0) and
 * q8[r, h, d] = e4m3(q[r, h, d] / q_scale[r, h]), the quotient rounded to fp32
 * (nearest even) and then to the nearest e4m3 value, ties to even, saturating
 * at +-448; NaN stays NaN.  One launch.
 *   q        bf16 [R, 128, 576], last dim contiguous, 16-byte aligned rows.
 *   q8       FP8 e4m3 [R, 128, 576] (caller-owned output): heads contiguous
 *            rows of 576 bytes, row stride a multiple of 16, 16-byte aligned.
 *   q_scale  fp32 [R, 128] (caller-owned output), last dim contiguous.
 *   stream   cudaStream_t.
 * Errors: PKV_ERR_INVALID_ARG (shapes, dtypes), PKV_ERR_ALIGNMENT,
 * PKV_ERR_UNSUPPORTED unless H == 128 and the last dim is 576; R == 0 is a
 * no-op.
 */
PKV_API int pkv_mla_quantize_q(const pkv_tensor* q, const pkv_tensor* q8,
                               const pkv_tensor* q_scale, void* stream);

/*
 * pkv_mla_verify_attn_fp8_native -- pkv_mla_verify_attn over an FP8 e4m3 cache
 * with the query given as e4m3 codes q8 and per-(row, head) scales q_scale
 * (pkv_mla_quantize_q): the query of (row r, head h) is code value x
 * q_scale[r, h], and S = Q K^T runs as kind::f8f6f4 tensor-core MMAs on the
 * raw e4m3 operands (scores scaled by q_scale x k_scale x scale afterwards).
 * Everything else (row limits, softmax, P.V in bf16, split merge, out, lse) is
 * pkv_mla_verify_attn's.  Source: "vllm.v1.attention.ops.
 * triton_decode_attention", decode_attention_fwd_verify (parameters); the
 * query quantisation is the library's, see pkv_mla_quantize_q.
 *   q8, q_scale   as written by pkv_mla_quantize_q ([B*qlen, 128, 576] e4m3
 *                 with 16-byte aligned rows; [B*qlen, 128] fp32).
 *   latent_cache  FP8 e4m3 only (PKV_ERR_UNSUPPORTED for bf16).
 *   other arguments as pkv_mla_verify_attn.
 * Two launches (the unit plan, then the kernel).
 */
PKV_API int pkv_mla_verify_attn_fp8_native(const pkv_tensor* q8, const pkv_tensor* q_scale,
                                           const pkv_tensor* latent_cache,
                                           const pkv_tensor* block_table,
                                           const pkv_tensor* seq_lens,
                                           const pkv_tensor* real_seq_lens, int qlen, float scale,
                                           int page_size, const pkv_tensor* k_scale,
                                           const pkv_tensor* out, const pkv_tensor* lse,
                                           int num_kv_splits, void* stream);

/*
 * pkv_num_kv_splits -- static upper bound on KV splits, safe to bake into a
 * CUDA graph (host only, no GPU needed).
 * Source: "vllm.v1.attention.ops.triton_decode_attention", verify_num_kv_splits
 * (its contract: programs per split = batch x row blocks; if one split of
 * every request fits in one dispatch round of occupancy x sm_count slots, use
 * as many splits as fit; else the n <= max_splits minimising rounds(n)/n,
 * preferring the fewest splits within 5 % of the best; never more than
 * cdiv(max_seq_len, min_work_per_split) nor 2 x sm_count, never fewer than 1).
 *   row blocks = cdiv(qlen * num_heads, block_h).
 * Returns the cap (>= 1), or PKV_ERR_INVALID_ARG for non-positive sm_count,
 * block_h, qlen or num_heads, or a negative occupancy.
 * Advisory: the attention calls do not call it.  A caller may pass its result
 * as num_kv_splits; with num_kv_splits == 0 the library picks its own cap, and
 * in either case each request's actual split count is chosen on the device
 * from the lengths (GQA: about four work items per CTA, at least 256 keys per
 * split; MLA: at least 4096 keys per split, 6144 when two verify tokens share
 * a CTA pair and the batch still gives every CTA pair a unit at that size).
 */
PKV_API int pkv_num_kv_splits(int max_seq_len, int batch, int qlen, int num_heads, int sm_count,
                              int block_h, double occupancy, int min_work_per_split,
                              int max_splits);

/*
 * pkv_gqa_kv_append -- write each request's current token into the paged GQA
 * cache, in place, before the decode call reads it.
 * Source: "Atencion paginada" (transformers), decode path, "Comportamiento de
 * la cache" and "Ejemplo" (the cache is updated in place through block_table:
 * a sequence with n cached tokens puts its new token at logical position n);
 * position convention of "vllm.models.flint.ops.decode_attention",
 * flint_decode_attention parameters (seq_lens counts the current token).
 *
 *   k, v          bf16 [B, Hkv, 128], last dim contiguous, 16-byte aligned rows
 *                 (strides % 8 == 0): the current token's key and value.
 *   kv_cache      bf16 [num_blocks, Hkv, P, 256] as for pkv_paged_decode_attn;
 *                 K goes to [..., :128], V to [..., 128:].  Written in place.
 *   block_table   int32 [B, max_blocks].
 *   seq_lens      int32 [B], lengths including the current token: the token is
 *                 written at position seq_lens[b] - 1, i.e. page
 *                 block_table[b][pos / P], slot pos % P.  seq_lens[b] <= 0
 *                 writes nothing.
 *   page_size     P (16 or 32).
 *   stream        cudaStream_t.
 * A position whose page entry lies beyond max_blocks or outside
 * [0, num_blocks) is not written; it raises bit 2 or bit 1 of the device error
 * word (pkv_check_errors).  Nothing else of the cache changes.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_ALIGNMENT, PKV_ERR_UNSUPPORTED (shapes,
 * strides, dtypes, page size) before any CUDA call; PKV_ERR_CUDA on a failed
 * launch.  B == 0 is a no-op.  Only the device error word of the workspace
 * is used (the workspace is allocated on first use, as for the attention
 * calls).
 */
PKV_API int pkv_gqa_kv_append(const pkv_tensor* k, const pkv_tensor* v, const pkv_tensor* kv_cache,
                              const pkv_tensor* block_table, const pkv_tensor* seq_lens,
                              int page_size, void* stream);

/*
 * pkv_mla_kv_append -- write the latent rows of each request's verify tokens
 * into the paged latent cache, in place.
 * Source: as pkv_gqa_kv_append, with the verify layout of
 * "vllm.v1.attention.ops.triton_decode_attention", decode_attention_fwd_verify
 * (parameters): a request's qlen verify tokens are its last qlen positions.
 *
 *   latent        bf16 [B*qlen, 576] (row r = b*qlen + t), last dim contiguous,
 *                 16-byte aligned rows.
 *   latent_cache  bf16 or FP8 e4m3 [num_pages, P, 1, 576] (or
 *                 [num_pages*P, 1, 576]), as for pkv_mla_verify_attn.
 *   block_table   int32 [B, max_pages].
 *   seq_lens      int32 [B]: row t of request b goes to position
 *                 seq_lens[b] - qlen + t (nothing when negative).
 *   qlen          verify tokens per request (>= 1).
 *   page_size     P (16 or 32).
 *   k_scale       fp32 device scalar, or NULL (= 1).  An e4m3 cache stores
 *                 e4m3(x / k_scale): the quotient in fp32 (IEEE division),
 *                 then the nearest e4m3 value, ties to even, saturating at
 *                 +-448.  Ignored for a bf16 cache (rows are copied).
 *   stream        cudaStream_t.
 * Bad table entries and error codes as for pkv_gqa_kv_append.
 */
PKV_API int pkv_mla_kv_append(const pkv_tensor* latent, const pkv_tensor* latent_cache,
                              const pkv_tensor* block_table, const pkv_tensor* seq_lens, int qlen,
                              int page_size, const pkv_tensor* k_scale, void* stream);

/*
 * pkv_check_errors -- read and clear the device error words of `device` (the
 * workspace's, and that of pkv_paged_decode_attn_noalloc's static array once
 * a call has set it up; synchronises the device).  *flags receives the OR of
 * the bits raised since the last check: 1 bad block-table entry, 2 seq_len longer than the block
 * table, 4 a pipeline wait gave up, 8 work items beyond the workspace, 16 a
 * CTA drew more work items than the launch has (the CTA stopped).
 * Returns PKV_OK when no bit was set, PKV_ERR_BAD_BLOCK_TABLE for bits 1|2,
 * PKV_ERR_CUDA otherwise (or on a failed CUDA call).
 */
PKV_API int pkv_check_errors(int device, int32_t* flags);

/*
 * pkv_selftest_wait_timeout -- failure-detection self-test.  Launches, on
 * `stream` of `device` (which must have a workspace: pkv_init), one CTA that
 * waits on an mbarrier nothing ever arrives on, through the same bounded wait
 * the attention kernels use.  The wait gives up after about 2^31 SM cycles
 * (about a second), raises bit 4 of the device error word and the kernel
 * returns: no fault, no hang, and the context stays usable.
 * pkv_check_errors(device) then reports the bit.  Returns PKV_OK, or
 * PKV_ERR_INVALID_ARG / PKV_ERR_CUDA.
 */
PKV_API int pkv_selftest_wait_timeout(int device, void* stream);

/*
 * pkv_check_counters -- count the non-zero arrival counters and scheduler
 * words of `device` (synchronises the device).  The kernels reset every
 * counter they use before returning, so a non-zero count after a completed
 * call means a broken invariant.  *nonzero receives the count.
 */
PKV_API int pkv_check_counters(int device, int64_t* nonzero);

/* Message of the last failed call on this thread ("" if none). */
PKV_API const char* pkv_last_error(void);

/* Free every device's workspace.  Later calls allocate afresh. */
PKV_API int pkv_shutdown(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
PKV_API int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
