/*
 * packedattn.h -- C ABI of libpackedattn, forward attention over flat-packed
 * variable-length sequences on NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor argument is a DEVICE pointer to caller-owned memory.  The
 *   library never allocates, frees or keeps a reference to caller memory;
 *   outputs are written asynchronously on `stream` and are valid once the
 *   stream has reached that point.
 * - Attention tensors are bf16, token-major and contiguous: element
 *   (token t, head h, dim d) sits at offset (t * H + h) * D + d.
 * - Sequence boundaries are int32 "cu_seqlens" arrays of batch + 1 entries:
 *   cu[0] = 0, non-decreasing, sequence b owns rows [cu[b], cu[b+1]).
 * - Every call returns a pa_status.  Arguments are checked on the host before
 *   anything is launched; a failed check launches nothing.  Nothing blocks
 *   the host, synchronizes the device or copies device -> host, except
 *   pa_get_device_status.  Nothing aborts, traps or throws.
 * - Checks that need the contents of device arrays (cu_seqlens monotone and
 *   consistent with the totals, lengths within max_q / max_k) run inside the
 *   kernels: a violation records an error code in a per-device status word
 *   (read with pa_get_device_status) and the offending work is skipped.
 * - Every kernel wait on the GPU is bounded; a wait that runs out records
 *   PA_DEVICE_ERR_TIMEOUT in the status word and the kernel returns.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).
 */
#ifndef PACKEDATTN_H
#define PACKEDATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pa_stream_t; /* identical to cudaStream_t */

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* null pointer, negative or zero size, non-finite scale */
  PA_ERR_UNSUPPORTED = 2,  /* valid but not implemented: D not 64/128, too many sequences */
  PA_ERR_MISALIGNED = 3,   /* a pointer or row pitch breaks the 16-byte rule */
  PA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (launch, tensor map) */
  PA_ERR_DEVICE = 5        /* pa_get_device_status found a recorded device error */
} pa_status;

/* Device-side error codes recorded in the status word (first error wins). */
#define PA_DEVICE_OK 0
#define PA_DEVICE_ERR_CU_SEQLENS 1   /* cu[0] != 0, decreasing, or cu[batch] != total */
#define PA_DEVICE_ERR_MAX_LEN 2      /* a sequence longer than max_q / max_k / s_max */
#define PA_DEVICE_ERR_TIMEOUT 3      /* a bounded pipeline wait ran out */
#define PA_DEVICE_ERR_LENGTH 4       /* a negative length, or a sum above INT32_MAX, in
                                        pa_cu_seqlens_from_lengths */
#define PA_DEVICE_ERR_CAPACITY 5     /* pa_varlen_work_order: more items than capacity */
#define PA_DEVICE_ERR_SMEM_ALIGN 6   /* dynamic shared memory not 1024-byte aligned (kernel skipped) */
#define PA_DEVICE_ERR_SEGMENT 7      /* pa_cfg_combine: bad sequence index, image offset or
                                        mismatched positive/negative image spans */

/* Largest batch (number of packed sequences) the attention kernels accept. */
#define PA_MAX_BATCH 1024

/* Query rows per work item of pa_varlen_attn_fwd (two 128-row tensor-core tiles). */
#define PA_VARLEN_TILE_M 256

/*
 * pa_varlen_attn_fwd -- non-causal softmax attention over a flat packed batch.
 *
 * Defined by the flat varlen attention path of "[Perf][Diffusion][Qwen-Image]
 * Replace per-bucket varlen loop with flat varlen attention for mixfusion"
 * (Key changes: AttentionMetadata with q_cu_seqlens / kv_cu_seqlens /
 * max_q_len / max_kv_len, packed [total_tokens, heads, head_dim] Q/K/V, no
 * attention mask, no padded tokens) and "feat: Support dynamic batching for
 * heterogeneous diffusion requests" (AttentionMetadata: tokens of one request
 * never attend to another's).  For sequence b, head h and query row i of b:
 *   out[i,h,:] = sum_j softmax_j(scale * <q[i,h,:], k[j,h,:]>) * v[j,h,:]
 * over the key rows j of the same sequence only.  A sequence with queries but
 * no keys gets all-zero output rows.
 *
 * q     [total_q, H, D] bf16      k, v [total_k, H, D] bf16
 * out   [total_q, H, D] bf16, written only at rows that belong to a sequence
 *       (rows >= cu_seqlens_q[batch] are left untouched)
 * cu_seqlens_q / cu_seqlens_k: device int32 [batch + 1]
 * batch in [1, PA_MAX_BATCH]; total_q/total_k >= cu[batch] (extra rows are
 * padding that belongs to no sequence and is never written); max_q / max_k
 * bound every sequence length; H >= 1; D in {64, 128}; scale finite
 * (1/sqrt(D) is usual).
 * Rows outside a sequence never change its result, whatever their bits
 * (NaN and Inf included): the last 128-row key tile of a sequence is loaded
 * whole, so up to 127 rows after the sequence end (the next sequence's rows
 * or trailing padding, within total_k) are read into shared memory, but
 * their scores are masked and their value rows are cleared before use.
 * q, k, v, out must be 16-byte aligned.
 * Deterministic: every output row is computed by one CTA in a fixed order, so
 * a sequence's result does not depend on which other sequences share the
 * batch (bit-identical to running it alone).
 */
pa_status pa_varlen_attn_fwd(const void *q, const void *k, const void *v, void *out,
                             const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                             int32_t batch, int32_t total_q, int32_t total_k,
                             int32_t max_q, int32_t max_k, int32_t H, int32_t D,
                             float scale, pa_stream_t stream);

/*
 * pa_block_window_attn_fwd -- block-local attention of the Token2Wav DiT.
 *
 * Defined by "[Perf][Model] Use block-sparse attention in Qwen2.5-Omni
 * Token2Wav DiT" (Purpose; Change: the same result as dense attention under
 * the block-difference mask).  Frames are grouped in blocks of `block`; query
 * i attends to key j iff j < n and
 *   -look_back <= floor(j / block) - floor(i / block) <= look_ahead
 * (look_back blocks before, look_ahead blocks after).  Whether any masking is
 * needed is decided from these integers on the host; nothing is read back
 * from the device.
 *
 * q, k, v, out [batch, n, H, D] bf16 contiguous (token-major per batch entry).
 * batch >= 1, n >= 1, block >= 1, look_back >= 0, look_ahead >= 0, H >= 1,
 * D in {64, 128}, scale finite; pointers 16-byte aligned.
 */
pa_status pa_block_window_attn_fwd(const void *q, const void *k, const void *v, void *out,
                                   int32_t batch, int32_t n, int32_t block,
                                   int32_t look_back, int32_t look_ahead,
                                   int32_t H, int32_t D, float scale, pa_stream_t stream);

/*
 * pa_block_window_attn_fwd_f32 -- the same block-local attention in fp32.
 *
 * The Token2Wav DiT runs in fp32 with classifier-free guidance as batch 2
 * ("[Perf][Model] Use block-sparse attention in Qwen2.5-Omni Token2Wav DiT",
 * Purpose), and its block-local result stayed within 6e-6 of the dense masked
 * SDPA (Test Result).  The window rule and the argument rules are those of
 * pa_block_window_attn_fwd; q, k, v, out are fp32 [batch, n, H, D]
 * contiguous, 16-byte aligned, caller-owned; out must not overlap q, k or v.
 * Every product and sum is IEEE fp32 (no tensor-core tf32); the softmax runs
 * in base 2 on the hardware exp2 with scale * log2(e) folded into q, so the
 * result is within a few fp32 roundings of the exact one.  Rows are staged
 * with TMA tensor copies (strides H * D * 4 and n * H * D * 4 bytes, so the
 * 16-byte alignment above is what they need); a wait that runs out records
 * PA_DEVICE_ERR_TIMEOUT in the device status word.
 */
pa_status pa_block_window_attn_fwd_f32(const float *q, const float *k, const float *v,
                                       float *out, int32_t batch, int32_t n, int32_t block,
                                       int32_t look_back, int32_t look_ahead, int32_t H,
                                       int32_t D, float scale, pa_stream_t stream);

/*
 * pa_cu_seqlens_from_lengths -- cu[0] = 0, cu[b+1] = cu[b] + lengths[b].
 *
 * The flat path's boundaries come from each request's real token count
 * ("[Perf][Diffusion][Qwen-Image] Replace per-bucket varlen loop with flat
 * varlen attention for mixfusion", Key changes: cu_seqlens built from real
 * text lengths via mask.sum).  lengths: device int32 [batch]; cu: device int32
 * [batch + 1].  batch >= 1.  A negative length records
 * PA_DEVICE_ERR_LENGTH and is treated as 0.
 */
pa_status pa_cu_seqlens_from_lengths(const int32_t *lengths, int32_t *cu, int32_t batch,
                                     pa_stream_t stream);

/*
 * pa_pack -- copy the real rows of a padded batch into the flat layout.
 *
 * Only real tokens enter the packed tensor ("feat: Support dynamic batching
 * for heterogeneous diffusion requests", How batching works).  padded is
 * [batch, s_max, row_bytes] bytes, flat is [total, row_bytes]; row r of
 * sequence b (r < cu[b+1] - cu[b]) goes from padded[b, r] to flat[cu[b] + r].
 * Flat rows >= cu[batch] are not touched.  cu: device int32 [batch + 1].
 * batch >= 1, s_max >= 0, total >= 0, row_bytes > 0 and a multiple of 16;
 * pointers 16-byte aligned.  A sequence longer than s_max records
 * PA_DEVICE_ERR_MAX_LEN, boundaries outside [0, total] or decreasing record
 * PA_DEVICE_ERR_CU_SEQLENS; such a sequence is skipped.
 */
pa_status pa_pack(const void *padded, void *flat, const int32_t *cu, int32_t batch,
                  int32_t s_max, int32_t total, int64_t row_bytes, pa_stream_t stream);

/*
 * pa_unpack -- the inverse scatter: flat[cu[b] + r] -> padded[b, r] for
 * r < cu[b+1] - cu[b]; padding rows of `padded` are left untouched (output
 * unpacked by cu_seqlens, same page as pa_cu_seqlens_from_lengths).
 * Same argument rules as pa_pack.
 */
pa_status pa_unpack(const void *flat, void *padded, const int32_t *cu, int32_t batch,
                    int32_t s_max, int32_t total, int64_t row_bytes, pa_stream_t stream);

/*
 * pa_rope_packed -- rotary position embedding on packed q and k, in place,
 * with request-local positions.
 *
 * The dynamic path rebuilds RoPE per request from request-local state and
 * never infers positions from packed global offsets, so a request gets the
 * same RoPE alone or inside a mixed batch ("feat: Support dynamic batching
 * for heterogeneous diffusion requests", Correctness model).  The pages give
 * no formula; this is the rotary embedding of Su et al. (RoFormer) on
 * interleaved pairs: token j of sequence b sits at position
 * p = pos_offset[b] + j and every head's pair (x_2i, x_2i+1) is rotated by the
 * angle p * base^(-2i/D).  Angles are reduced exactly (double-precision
 * fraction of a turn), sin/cos and the rotation in fp32, output bf16.
 *
 * q [total_q, H, D] and k [total_k, H, D] bf16 are updated in place at the
 * rows of their sequences (rows past cu[batch] are left untouched).
 * cu_seqlens_q / cu_seqlens_k: device int32 [batch + 1]; pos_offset: device
 * int32 [batch] or NULL (all zero).  batch in [1, 65535], H >= 1, D even,
 * a multiple of 8 and at most 512, base finite and > 0; q, k 16-byte
 * aligned.  Bad boundaries record PA_DEVICE_ERR_CU_SEQLENS; the sequence is
 * skipped.
 */
pa_status pa_rope_packed(void *q, void *k, const int32_t *cu_seqlens_q,
                         const int32_t *cu_seqlens_k, const int32_t *pos_offset,
                         int32_t batch, int32_t total_q, int32_t total_k, int32_t H,
                         int32_t D, float base, pa_stream_t stream);

/*
 * pa_linear_bf16 -- batch-invariant packed-M linear layer.
 *
 *   y[m, n] = sum_k x[m, k] * w[n, k] + bias[n]
 *
 * The packed path runs its projections on the flat [total_tokens, C]
 * activations of all requests at once, and batched and serial outputs are
 * bit-identical because these GEMMs give each row the same result whatever
 * the packed M is ("feat: Support dynamic batching for heterogeneous
 * diffusion requests", packed varlen step batching: Setup, Determinism;
 * Notes, item 1).  Here every M runs one tile shape with a fixed K order and
 * no split-K, so row m of y depends only on row m of x, w and bias: rows
 * computed packed, alone or at any row offset are equal bit for bit.
 *
 * x [M, K], w [N, K] (out_features x in_features), y [M, N]: bf16 row-major
 * contiguous, device, caller-owned; bias: bf16 [N] or NULL.  Accumulation
 * in fp32, bias added in fp32, one round to bf16 (nearest even).  M >= 0
 * (M = 0 does nothing and x, y may then be NULL), N >= 1, K >= 1; K and N
 * multiples of 8 and every pointer 16-byte aligned, else PA_ERR_MISALIGNED.
 * y must not overlap x, w or bias.
 */
pa_status pa_linear_bf16(const void *x, const void *w, const void *bias, void *y, int32_t M,
                         int32_t N, int32_t K, pa_stream_t stream);

/*
 * pa_cfg_combine -- segment-aware unpack of each request's image span with
 * the per-request classifier-free-guidance combine.
 *
 * Defined by "feat: Support dynamic batching for heterogeneous diffusion
 * requests" (AttentionSegment: text / image / negative-text spans used to
 * scatter outputs back to request-local state; CFG behavior: after the
 * per-request split, out = negative + true_cfg_scale * (positive - negative),
 * with true_cfg_scale and cfg_normalize per request).  Request r's positive
 * pass is packed sequence pos_seq[r], its negative pass sequence neg_seq[r]
 * (< 0: no CFG, the positive image rows are copied).  The image span of
 * sequence b is rows [cu[b] + img_off[b], cu[b+1]) of `flat`.  With
 * cfg_normalize[r] != 0 each combined row is rescaled to the L2 norm of its
 * positive row (rows whose combined norm is 0 are written as 0).
 *
 * flat [total, row_elems] bf16; out [requests, img_max, row_elems] bf16:
 * rows [0, n_img(r)) of slot r are written, the others left untouched.
 * cu device int32 [batch + 1]; img_off device int32 [batch]; pos_seq,
 * neg_seq, cfg_normalize device int32 [requests]; cfg_scale device float
 * [requests].  Arithmetic in fp32, output rounded to bf16.
 * batch in [1, 65535], requests in [1, 65535], total >= 0, img_max >= 0,
 * row_elems a positive multiple of 8; flat and out 16-byte aligned.
 * A request with an out-of-range sequence or image offset, positive and
 * negative image spans of different lengths, or more than img_max image
 * rows records PA_DEVICE_ERR_SEGMENT and is skipped.
 */
pa_status pa_cfg_combine(const void *flat, void *out, const int32_t *cu,
                         const int32_t *img_off, const int32_t *pos_seq,
                         const int32_t *neg_seq, const float *cfg_scale,
                         const int32_t *cfg_normalize, int32_t batch, int32_t requests,
                         int32_t total, int32_t img_max, int32_t row_elems,
                         pa_stream_t stream);

/*
 * pa_varlen_num_work_items -- host-side count of attention work items,
 * sum_b H * ceil(Lq[b] / tile_m), from HOST copies of cu_seqlens_q.
 * Returns -1 on invalid arguments.
 */
int64_t pa_varlen_num_work_items(const int32_t *cu_seqlens_q_host, int32_t batch,
                                 int32_t H, int32_t tile_m);

/*
 * pa_varlen_work_order -- the order in which the attention kernel visits its
 * work items, written by the same device code the kernel schedules with.
 *
 * Sequences are taken longest key length first (equal lengths: lower index
 * first); within a sequence heads in order, within a head query tiles of
 * tile_m rows in order.  The largest request dominates a mixed batch and the
 * old per-bucket loop left bubbles ("[Perf][Diffusion][Qwen-Image] Replace
 * per-bucket varlen loop ...", Purpose), so the longest work starts first.
 * items: device int32 [capacity, 3] receiving (sequence, head, q_tile) for
 * item 0, 1, ...; when there are more items than capacity, the first
 * `capacity` are written and PA_DEVICE_ERR_CAPACITY is recorded.  Boundaries
 * are checked as in pa_varlen_attn_fwd (without totals or maxima); a bad
 * sequence gets no items.  batch in [1, PA_MAX_BATCH], H >= 1, tile_m >= 1.
 * PA_VARLEN_TILE_M is the tile the attention kernel uses.
 */
pa_status pa_varlen_work_order(const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                               int32_t batch, int32_t H, int32_t tile_m,
                               int32_t *items, int64_t capacity, pa_stream_t stream);

/*
 * pa_get_device_status -- synchronize the current device, then read and
 * clear its status word.  *code receives PA_DEVICE_OK or the first
 * PA_DEVICE_ERR_* recorded since the last call.  Returns PA_ERR_DEVICE when
 * an error was recorded, PA_ERR_CUDA when the synchronize fails.  For tests
 * and debugging: it blocks the host.
 */
pa_status pa_get_device_status(int32_t *code);

/*
 * pa_selftest_wait_timeout -- exercises the bounded-wait path the pipelined
 * kernels use: one CTA waits on an mbarrier that nothing ever arrives at,
 * gives up after about `timeout_us` microseconds (1 .. 10,000,000), records
 * PA_DEVICE_ERR_TIMEOUT in the status word and returns, leaving the context
 * usable.  No counterpart on the pages; it tests this library's own failure
 * handling without faulting the GPU.
 */
pa_status pa_selftest_wait_timeout(int32_t timeout_us, pa_stream_t stream);

/* Name of the last CUDA error this thread met inside the library, the cause
 * behind a PA_ERR_CUDA (static string, never NULL; "cudaSuccess" if none). */
const char *pa_last_cuda_error(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif

#endif /* PACKEDATTN_H */
