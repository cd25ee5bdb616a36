/*
 * dap.h -- C ABI of the paged decode-attention library for NVIDIA GB300 (sm_103a).
 *
 * Single-token GQA decode attention over a paged KV cache (bf16 or fp8 e4m3), its
 * contiguous-cache form, multi-token causal decode, masked decode (bool masks, with the
 * causal rule), the fp8 sliding-window latent (K = V) variant, and the cache appends that
 * feed them.  Plain pointers and sizes only.
 *
 * Conventions shared by every entry point:
 *   - The caller owns every buffer.  The library allocates no device memory and never
 *     synchronises the stream; all work is enqueued on `stream` (a cudaStream_t passed
 *     as void*, NULL = the legacy default stream).
 *   - "device" marks a device pointer; "host" a host value.  bf16 buffers are raw
 *     IEEE bfloat16 bit patterns (passed as void*).
 *   - Kernels are launched as programmatic dependents (CUDA programmatic dependent
 *     launch; all but the balanced schedule's persistent kernel and the self-test): each
 *     waits for the work before it on the stream to complete before it reads or writes
 *     global memory, so stream order holds as for ordinary launches, but its launch and
 *     prologue may overlap the end of the previous kernel.  Events recorded between two
 *     calls still mark the boundary.
 *   - Errors that the host can see (null pointers, bad sizes, unsupported shapes,
 *     misaligned pointers, a workspace that is too small) are returned as a dap_status
 *     before anything is launched.  A failed launch returns DAP_ERR_CUDA.
 *   - Errors that only the device can see (a page index outside the pool, a sequence
 *     length outside [0, max_kv_len], an fp8 slot outside the cache, a pipeline wait
 *     that timed out) never trap: the kernel records a bit in a library-wide device
 *     error word (read it with dap_get_device_errors) and keeps every access in bounds.
 *
 * Sources of the operation (web pages the library follows):
 *   [A] AstrAI "CUDA Kernels" developer doc: section "Python Wrappers" (q/k/v are
 *       [batch, seq_len, n_heads, head_dim], scale 1/sqrt(head_dim)) and section
 *       "Q Scheduling and KV Addressing" (a KV policy translates a logical position to
 *       a physical address; ContigKV / PagedKV).
 *   [B] AstrAI csrc commit log: the split-KV commit (partition KV across blocks that
 *       emit unnormalised (O, m, l) partials, merged by a combine kernel; split count
 *       chosen to fill the device, single pass when batch*kv_head already fills it),
 *       the split-planner commit (bandwidth saturates near 256-512 blocks), the
 *       per-element page lookup commit (any page_size), the numerics commit (fmaf for
 *       V accumulation, divide guard 1e-20, atol = rtol = 0.01).
 *   [C] nvfp4-megamoe-kernel cutedsl/native_swa_decode.py: native_swa_decode_attention
 *       and _fallback_batched_sdp (fp8 K = V sliding-window decode semantics).
 */
#ifndef DAP_H_
#define DAP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DAP_OK = 0,
    DAP_ERR_NULL = 1,        /* a required pointer is NULL */
    DAP_ERR_SHAPE = 2,       /* a size or stride is out of range or inconsistent */
    DAP_ERR_UNSUPPORTED = 3, /* a valid shape this build has no kernel for */
    DAP_ERR_WORKSPACE = 4,   /* workspace missing or smaller than dap_workspace_bytes */
    DAP_ERR_ALIGN = 5,       /* a pointer or stride breaks the 16-byte rule */
    DAP_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed */
    DAP_ERR_SCRATCH_LIMIT = 7 /* needs more split scratch than DAP_NOALLOC_SCRATCH_BYTES */
} dap_status;

/* Bits of the device error word. */
#define DAP_DEVERR_TIMEOUT 0x1u  /* a pipeline wait gave up; the launch's output is invalid */
#define DAP_DEVERR_SEQLEN 0x2u   /* seq_lens[b] < 0 or > max_kv_len; clamped */
#define DAP_DEVERR_PAGE 0x4u     /* block_table entry outside [0, num_pages); page 0 read instead */
#define DAP_DEVERR_SLOT 0x8u     /* fp8 slot index >= num_blocks*block_size; row skipped */
#define DAP_DEVERR_QMAP 0x10u    /* multi-token work map names no token of a sequence; tile skipped */

/* Human-readable name of a status code.  Never NULL. */
const char *dap_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int dap_version(void);

/* Number of SMs of the current CUDA device (cudaDevAttrMultiProcessorCount), or -1 when
 * no device is usable. */
int dap_device_sm_count(void);

/*
 * Split planner [B: split-KV and split-planner commits].
 * Returns a recommended num_splits S >= 1 for the per-sequence schedule: every sequence is
 * cut into chunks of dap_chunk_tokens(max_kv_len, S) tokens, so sequence b runs
 * ceil(seq_lens[b] / chunk) splits (at least 1).  When B * Hkv (sequence, kv head) units
 * are fewer than the GPU's resident CTAs (2 per SM), S is the number of chunks that fills
 * one wave (8 instead of more while 8 chunks fill at least four fifths of it: up to 8 chunks
 * merge inside a thread-block cluster); otherwise S keeps the largest chunk near a tenth of
 * one SM's share of the KV rows.  S never exceeds the number of 64-token chunks of the longest sequence.  Every decode
 * entry point runs this plan when given num_splits = 0 (see dap_resolve_splits).
 *   sm_count   SMs available (dap_device_sm_count()).
 *   total_kv   sum of seq_lens (host); 0 means "unknown", taken as B * max_kv_len.
 * Pure host function; no CUDA call.
 */
int dap_plan_splits(int sm_count, int B, int Hq, int Hkv, int D, int page_size,
                    int max_kv_len, long long total_kv);

/* Tokens per split chunk for a plan: ceil(max_kv_len / num_splits) rounded up to a
 * multiple of 64 tokens (at least 64).  Pure host function. */
int dap_chunk_tokens(int max_kv_len, int num_splits);

/* num_splits value selecting the balanced persistent schedule of decode_attn_paged /
 * decode_attn_contig / decode_attn_paged_noalloc (see decode_attn_paged). */
#define DAP_SPLITS_BALANCED (-1)

/*
 * The split count a decode call runs for the num_splits it is given (every decode entry
 * point resolves its argument this way, with sm_count = dap_device_sm_count() and
 * total_kv = 0):
 *   num_splits == 0: dap_plan_splits(sm_count, B, Hq, Hkv, D, page_size, max_kv_len, total_kv);
 *   num_splits >= 1: num_splits;
 *   then lowered to the number of dap_chunk_tokens-long chunks that can hold a token
 *   (ceil(max_kv_len / chunk), at least 1), so no split is empty for every sequence.
 *   num_splits == DAP_SPLITS_BALANCED returns DAP_SPLITS_BALANCED (1 when B > 4096: so many
 *   sequences fill the device with one CTA per sequence and kv head).
 * Returns 0 for invalid arguments (num_splits < -1, B < 0, ...).  Size the workspace with
 * dap_workspace_bytes(B, Hq, Hkv, D, <the value returned>).  Pure host function.
 */
int dap_resolve_splits(int num_splits, int sm_count, int B, int Hq, int Hkv, int D, int page_size,
                       int max_kv_len, long long total_kv);

/* Workspace bytes a decode call needs for a resolved split count (dap_resolve_splits):
 *   num_splits == 1: 0;
 *   num_splits >= 2: room for B*num_splits*Hq partial rows of (D + 2) floats (unnormalised
 *                    acc, running max m, running sum l);
 *   num_splits == DAP_SPLITS_BALANCED: the balanced schedule's partial slots (two per
 *                    persistent CTA, for at most 1024 CTAs) plus 8 bytes per (sequence,
 *                    kv head); 0 when B > 4096;
 *   num_splits == 0: 0 (0 is not a split count: resolve it first).
 * Pure host function. */
size_t dap_workspace_bytes(int B, int Hq, int Hkv, int D, int num_splits);

/*
 * Paged GQA decode attention [A][B].
 *   out[b,h,:] = sum_t softmax_t(scale * q[b,h,:] . K[b,t,h/G,:]) V[b,t,h/G,:],
 *   t < seq_lens[b], G = Hq / Hkv (consecutive query heads share a kv head).
 *
 *   q            device bf16 [B, Hq, D], element strides (q_stride_b, q_stride_h, 1).
 *   k_cache,     device bf16 [num_pages, page_size, Hkv, D], contiguous: logical position
 *   v_cache      t of sequence b lives in page block_table[b, t / page_size], slot
 *                t % page_size.
 *   block_table  device int32 [B, max_pages], row-major.  Entries past a sequence's
 *                last page are never used (they may be read, within the table).
 *   seq_lens     device int32 [B].  Each entry must lie in [0, max_kv_len].
 *   max_kv_len   host: an upper bound of seq_lens (<= max_pages * page_size); it sets
 *                the chunk length of the split plan.
 *   scale        softmax scale applied in fp32 to q . k (normally 1/sqrt(D)).
 *   num_splits   S > 0 = per-sequence schedule: every sequence is cut into chunks of
 *                dap_chunk_tokens(max_kv_len, S) tokens, one CTA each, and the splits of a
 *                sequence are merged by a combine kernel (or, when 2 <= S <= 8 and the grid
 *                fits one wave, inside the thread-block cluster its CTAs form: the same
 *                arithmetic, no second kernel).  0 = the same schedule with the
 *                planner's S (dap_plan_splits with total_kv = 0; a caller that knows the
 *                summed lengths can pass its own plan instead).  DAP_SPLITS_BALANCED =
 *                balanced schedule: a persistent grid of SMs x resident CTAs cuts the
 *                flattened (sequence, kv head, 64-token tile) space into equal contiguous
 *                ranges, whatever the length mix, and a combine kernel merges the pieces
 *                of a sequence (B > 4096 runs one CTA per sequence and kv head instead).
 *                The planner's schedule measures faster on every batch measured (a single
 *                long sequence included).
 *   workspace    device scratch of at least dap_workspace_bytes(B, Hq, Hkv, D,
 *                dap_resolve_splits(num_splits, ...)) bytes, 16-byte aligned (may be NULL
 *                when that is 0).  Needs no initialisation; its contents are undefined
 *                afterwards.
 *   out          device bf16 [B, Hq, D], element strides (out_stride_b, out_stride_h, 1).
 *                Written in full (an empty sequence gives a zero row).
 *   Supported: D in {32, 64, 128, 256}; G in {1, 2, 4, 8}; any page_size >= 1 (page sizes
 *   that are multiples of 8 move K/V in TMA boxes, others row by row with 16-byte copies
 *   into the same tiles).  q, out, k_cache and v_cache 16-byte aligned; q/out strides
 *   multiples of 8 elements, nonzero where the extent they step over is above 1.
 *   The result is bit-identical under any permutation of the physical pages for a fixed
 *   num_splits (the summation order depends only on logical positions).
 */
dap_status decode_attn_paged(const void *q, long long q_stride_b, long long q_stride_h,
                             const void *k_cache, const void *v_cache, int num_pages,
                             int page_size, const int32_t *block_table, int max_pages,
                             const int32_t *seq_lens, int max_kv_len, int B, int Hq, int Hkv,
                             int D, float scale, int num_splits, void *workspace,
                             size_t workspace_bytes, void *out, long long out_stride_b,
                             long long out_stride_h, void *stream);

/*
 * Contiguous-cache GQA decode attention [A: ContigKV]: the same operation with
 * k, v device bf16 [B, max_len, Hkv, D] contiguous; position t of sequence b is row
 * (b, t).  seq_lens[b] must lie in [0, max_kv_len] and max_kv_len <= max_len.
 * Everything else as decode_attn_paged.
 */
dap_status decode_attn_contig(const void *q, long long q_stride_b, long long q_stride_h,
                              const void *k, const void *v, int max_len,
                              const int32_t *seq_lens, int max_kv_len, int B, int Hq, int Hkv,
                              int D, float scale, int num_splits, void *workspace,
                              size_t workspace_bytes, void *out, long long out_stride_b,
                              long long out_stride_h, void *stream);

/*
 * Paged GQA decode over an fp8 (OCP e4m3) K/V cache.  The fp8 cache convention of [C]
 * (codes plus a bf16 dequantisation factor: value = e4m3(code) * factor), applied to the
 * GQA cache with one factor per (slot, kv head) for K and one for V:
 *   K[b, t, h, :] = e4m3(k_codes[page, slot, h, :]) * k_scale[page, h, slot],
 *   page = block_table[b, t / page_size], slot = t % page_size; V likewise;
 *   out[b, hq, :] = sum_t softmax_t(scale * q[b, hq, :] . K[b, t, hq/G, :]) V[b, t, hq/G, :].
 *
 *   k_codes, v_codes  device uint8 [num_pages, page_size, Hkv, D] contiguous (e4m3 codes).
 *   k_scale, v_scale  device bf16 [num_pages, Hkv, page_size] contiguous (one factor per
 *                     slot and kv head; kv-head-major inside a page so that a page's
 *                     factors of one head are contiguous).
 *   num_splits        >= 1: per-sequence splits as decode_attn_paged; 0 = the planner's S
 *                     (dap_resolve_splits(0, SMs, B, Hq, Hkv, D, page_size, max_kv_len, 0)).
 *                     DAP_SPLITS_BALANCED is not supported here.
 *   workspace         >= dap_workspace_bytes(B, Hq, Hkv, D, S) for the S used.
 *   q, out, block_table, seq_lens, max_kv_len, scale, strides: as decode_attn_paged.
 *   Supported: D in {64, 128, 256}; G in {1, 2, 4, 8}; any page_size >= 1 (page sizes
 *   that are multiples of 8 move codes and factors in TMA boxes, others row by row); codes
 *   and factor arrays 16-byte aligned.  q is used in f16 after an exact power-of-two shift (so any
 *   finite bf16 q is representable); the result is within the bf16 path's tolerance of
 *   the exact dequantised attention.
 */
dap_status decode_attn_paged_fp8kv(const void *q, long long q_stride_b, long long q_stride_h,
                                   const uint8_t *k_codes, const uint8_t *v_codes,
                                   const void *k_scale, const void *v_scale, int num_pages,
                                   int page_size, const int32_t *block_table, int max_pages,
                                   const int32_t *seq_lens, int max_kv_len, int B, int Hq, int Hkv,
                                   int D, float scale, int num_splits, void *workspace,
                                   size_t workspace_bytes, void *out, long long out_stride_b,
                                   long long out_stride_h, void *stream);

/*
 * Append the new token's K and V to the fp8 GQA cache that decode_attn_paged_fp8kv reads.
 * Every (sequence b, kv head h) row of k_new / v_new is quantised as kv_append_fp8 does
 * (amax / 448 stored as bf16, codes e4m3(x / factor) RNE, saturating) and written at
 * logical position positions[b] through the block table: codes to [page, slot, h, :],
 * factors to [page, h, slot].
 *   k_new, v_new  device bf16 [B, Hkv, D] contiguous.  positions  device int32 [B].
 *   Supported: D in {64, 128, 256}.  A position outside [0, max_pages * page_size) or a page
 *   outside the pool skips that sequence and sets DAP_DEVERR_SEQLEN / DAP_DEVERR_PAGE.
 */
dap_status kv_append_paged_fp8(const void *k_new, const void *v_new, uint8_t *k_codes,
                               uint8_t *v_codes, void *k_scale, void *v_scale, int num_pages,
                               int page_size, const int32_t *block_table, int max_pages,
                               const int32_t *positions, int B, int Hkv, int D, void *stream);

/*
 * Multi-token decode: several new tokens per sequence (speculative-decoding verification,
 * chunked short prefill) attending the paged cache causally [A: "Q Scheduling and KV
 * Addressing", the packed-q work map].
 *
 * The new tokens of all sequences are packed back to back: qo_indptr[0] = 0 and
 * qo_indptr[b+1] = qo_indptr[b] + q_len[b]; total_q = qo_indptr[B].  The caches already hold
 * the new tokens' K and V (append them first), so sequence b has seq_lens[b] >= q_len[b]
 * keys and its token i (0 <= i < q_len[b]) sits at position p = seq_lens[b] - q_len[b] + i:
 *   out[qo_indptr[b] + i, h, :] = sum_{t <= p} softmax_t(scale * q[.., h, :] . K[b,t,h/G,:])
 *                                 V[b,t,h/G,:].
 * (With q_len[b] = 1 this is decode_attn_paged.)  A token with p < 0 (q_len[b] > seq_lens[b],
 * flagged DAP_DEVERR_SEQLEN) gives a zero row.
 *
 * Work map: every sequence's tokens are cut into tiles of tokens_per_tile tokens; tile w
 * covers tokens [tile_index[w] * tokens_per_tile, ...) of sequence tile_batch[w].  A tile's
 * tokens x the G heads of a kv head are its query columns, and every tile streams its
 * sequence's keys once, so the fewer tiles a sequence has, the fewer times its K/V are
 * read.  Three tile sizes: 16 / G tokens (16 columns), 32 / G tokens (32 columns; not with a
 * mask) and, for D 64, 128 and 256, 128 / G tokens (128 query rows of tensor-memory
 * products: up to 16 tokens at G = 8 against one K/V stream).
 * dap_multi_tokens_per_tile(Hq, Hkv, D, max_q_len) picks 16 / G when the longest new-token
 * count fits it, else 128 / G where D allows (D = 0: head dim not known, no 128-row tiles),
 * else 32 / G (G = 8, D = 128: 2 tokens up to q_len 2, then 16).
 * dap_q_tile_map builds the map on the host:
 *   q_lens      host int32 [B], each >= 0.
 *   qo_indptr   host int32 [B + 1] (written).
 *   tile_batch, tile_index   host int32 [max_tiles] (written).
 * Returns the number of tiles, or -1 when max_tiles is too small or an input is invalid.
 * Pure host functions; no CUDA call.
 */
int dap_multi_tokens_per_tile(int Hq, int Hkv, int D, int max_q_len);
int dap_q_tile_map(const int32_t *q_lens, int B, int tokens_per_tile, int32_t *qo_indptr,
                   int32_t *tile_batch, int32_t *tile_index, int max_tiles);

/* Workspace bytes of decode_attn_paged_multi: 0 for num_splits <= 1, else room for
 * total_q * num_splits * Hq partial rows of (D + 2) floats.  Pure host function. */
size_t dap_workspace_bytes_multi(int total_q, int Hq, int D, int num_splits);

/*
 *   q            device bf16 [total_q, Hq, D], element strides (q_stride_t, q_stride_h, 1).
 *   k_cache, v_cache, block_table, num_pages, page_size, max_pages: as decode_attn_paged.
 *   seq_lens     device int32 [B], in [q_len[b], max_kv_len].
 *   qo_indptr    device int32 [B + 1]; tile_batch, tile_index device int32 [num_tiles]: the
 *                work map above (copies of dap_q_tile_map's output), built with
 *   tokens_per_tile  16 / G, 32 / G or, at D 64, 128 and 256, 128 / G (else DAP_ERR_SHAPE;
 *                32 / G with a mask, 128 / G at D = 32: DAP_ERR_UNSUPPORTED).
 *   num_splits   >= 1: the per-sequence schedule of decode_attn_paged, per tile: the tile's
 *                keys (up to its last token's position) are cut into chunks of
 *                dap_chunk_tokens(max_kv_len, num_splits) keys, one CTA per (tile, kv head,
 *                chunk), merged by a combine kernel.  0 = the planner's S over the tiles
 *                (dap_resolve_splits(0, SMs, num_tiles, Hq, Hkv, D, page_size, max_kv_len,
 *                0)).  DAP_SPLITS_BALANCED is not supported here.
 *   mask         device uint8 [total_q, mask_stride] or NULL: the 3-D bool mask [batch,
 *                q_len, kv_len] of [A: "Python Wrappers"] with its q rows packed like q
 *                (row qo_indptr[b] + i; nonzero = keep).  Token i keeps key t only if t is
 *                at or before its position and its mask byte is set (causal and mask
 *                together).  mask_stride >= max_kv_len, a multiple of 16; mask 16-byte
 *                aligned.  A token with no key left gives a zero row.
 *   workspace    device, >= dap_workspace_bytes_multi(total_q, Hq, D, S) bytes for the
 *                split count S used, 16-byte aligned.
 *   out          device bf16 [total_q, Hq, D], strides (out_stride_t, out_stride_h, 1).
 *   Supported: D in {32, 64, 128, 256}; G in {1, 2, 4, 8}; any page_size >= 1;
 *   alignment and strides as decode_attn_paged.  A work-map entry that names no token of its
 *   sequence is skipped and flagged (DAP_DEVERR_QMAP).
 */
dap_status decode_attn_paged_multi(const void *q, long long q_stride_t, long long q_stride_h,
                                   const void *k_cache, const void *v_cache, int num_pages,
                                   int page_size, const int32_t *block_table, int max_pages,
                                   const int32_t *seq_lens, const int32_t *qo_indptr,
                                   const int32_t *tile_batch, const int32_t *tile_index,
                                   int num_tiles, int tokens_per_tile, int total_q, const uint8_t *mask,
                                   long long mask_stride, int max_kv_len, int B, int Hq, int Hkv,
                                   int D, float scale, int num_splits, void *workspace,
                                   size_t workspace_bytes, void *out, long long out_stride_t,
                                   long long out_stride_h, void *stream);

/*
 * Masked paged GQA decode [A: "Python Wrappers", the 2-D bool mask [batch, kv_len], True =
 * keep]: decode_attn_paged where key t of sequence b takes part only if
 * mask[b * mask_stride + t] is nonzero.  A sequence with no key left gives a zero row.
 *   mask         device uint8 [B, mask_stride]; mask_stride >= max_kv_len, a multiple of 16;
 *                mask 16-byte aligned (bytes past seq_lens[b] are not used).
 *   num_splits   >= 1: per-sequence splits as decode_attn_paged; 0 = the planner's S
 *                (dap_resolve_splits(0, SMs, B, Hq, Hkv, D, page_size, max_kv_len, 0)).
 *                DAP_SPLITS_BALANCED is not supported here.
 *   workspace    >= dap_workspace_bytes(B, Hq, Hkv, D, S) for the S used.
 *   Everything else as decode_attn_paged.  Supported: D in {32, 64, 128, 256}; G in
 *   {1, 2, 4, 8}; any page_size >= 1.
 */
dap_status decode_attn_paged_masked(const void *q, long long q_stride_b, long long q_stride_h,
                                    const void *k_cache, const void *v_cache, int num_pages,
                                    int page_size, const int32_t *block_table, int max_pages,
                                    const int32_t *seq_lens, const uint8_t *mask,
                                    long long mask_stride, int max_kv_len, int B, int Hq, int Hkv,
                                    int D, float scale, int num_splits, void *workspace,
                                    size_t workspace_bytes, void *out, long long out_stride_b,
                                    long long out_stride_h, void *stream);

/*
 * fp8 sliding-window latent decode, K = V [C].
 *   For token t and window position j < W, slot = slot_idx[t, j]; the row takes part iff
 *   j < lens[t] and slot >= 0.  Its value is bf16(e4m3(kv_cache[slot / block_size,
 *   slot % block_size, :]) * inv_scale[slot]) (the fp8 code times the bf16 inverse scale,
 *   rounded to bf16).  out[t, h, :] = sum_j softmax_j(scale * q[t,h,:] . kv_j) kv_j;
 *   a token with no row gives a zero row.
 *
 *   q          device bf16 [T, NH, HD] contiguous.
 *   kv_cache   device uint8 [num_blocks, block_size, HD] contiguous, OCP e4m3 (E4M3FN) codes.
 *   inv_scale  device bf16 [num_blocks * block_size] (one per slot).
 *   slot_idx   device int64 [T, W] row-major, -1 = padding.
 *   lens       device int64 [T].
 *   out        device bf16 [T, NH, HD] contiguous.
 *   Supported: HD = 512, NH a multiple of 128 (NH <= 1024), 1 <= W <= 128, T <= 65535.
 *   Slots >= num_blocks*block_size are skipped and flagged (DAP_DEVERR_SLOT).
 */
dap_status decode_attn_paged_fp8(const void *q, const uint8_t *kv_cache, const void *inv_scale,
                                 const int64_t *slot_idx, const int64_t *lens, int T, int NH,
                                 int HD, int W, int num_blocks, int block_size, float scale,
                                 void *out, void *stream);

/*
 * Append the new decode token's K and V to a paged cache (the step before decode).
 *   For every sequence b and kv head h: k_new[b, h, :] and v_new[b, h, :] are written to
 *   logical position positions[b] of sequence b, i.e. page block_table[b, positions[b] /
 *   page_size], slot positions[b] % page_size of the [num_pages, page_size, Hkv, D] caches
 *   (the translation decode_attn_paged reads through; [A: ContigKV / PagedKV]).
 *   k_new, v_new  device bf16 [B, Hkv, D] contiguous.
 *   positions     device int32 [B] (normally the sequence length before the append).
 *   Supported: D a multiple of 8; pointers 16-byte aligned.  A position outside
 *   [0, max_pages * page_size) or a page outside the pool skips that sequence and sets
 *   DAP_DEVERR_SEQLEN / DAP_DEVERR_PAGE.
 */
dap_status kv_append_paged(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                           int num_pages, int page_size, const int32_t *block_table,
                           int max_pages, const int32_t *positions, int B, int Hkv, int D,
                           void *stream);

/*
 * Quantise latent rows (K = V) into the fp8 cache that decode_attn_paged_fp8 reads [C].
 *   Row t (HD bf16 values) goes to slot slots[t] of kv_cache [num_blocks, block_size, HD]
 *   with its dequantisation factor in inv_scale[slot], so that the decode side's
 *   e4m3(code) * inv_scale restores it.  In binary32: amax = max |x|; s = amax / 448 (1 for
 *   an all-zero row), stored as bf16; code = e4m3(x / s_stored), round to nearest even,
 *   saturating at +-448 (the quantiser multiplies by the multiplier 1/s and keeps amax in
 *   the input domain, as the AstrAI doc's FP8 section describes).
 *   rows       device bf16 [T, HD] contiguous.   slots  device int64 [T].
 *   Supported: HD in {256, 512}.  A slot outside the cache is skipped (DAP_DEVERR_SLOT).
 */
dap_status kv_append_fp8(const void *rows, uint8_t *kv_cache, void *inv_scale,
                         const int64_t *slots, int T, int HD, int num_blocks, int block_size,
                         void *stream);

/*
 * Paged GQA decode that allocates nothing and takes no workspace.  The web pages this
 * library follows have no counterpart to it; it exists for callers that cannot hand the
 * library scratch memory: hosts that reserve their whole device-memory budget up front and
 * forbid later cudaMalloc calls (a cudaMalloc can synchronise the device and can fail in
 * the middle of serving), and plugin-style interfaces that pass a kernel only its input and
 * output buffers.
 *
 * Same operation, arguments and results as decode_attn_paged, without `workspace` and
 * `workspace_bytes`.  The split partials live in one file-scope device array of
 * DAP_NOALLOC_SCRATCH_BYTES bytes that every GPU loading the library holds until the
 * process exits.  Sizes:
 *   - num_splits == 0 runs the planner's S (as decode_attn_paged does), lowered until its
 *     partials, dap_workspace_bytes(B, Hq, Hkv, D, S), fit the array;
 *   - a num_splits >= 1, or DAP_SPLITS_BALANCED, whose partials exceed the array is
 *     rejected with DAP_ERR_SCRATCH_LIMIT (nothing launched).
 * Start-up: under CUDA's lazy module loading (the runtime's default) the array is reserved
 * on a device only when the first call on that device loads the library's module and looks
 * up the array's address (cudaGetSymbolAddress, with that device current), so that first
 * call can still take 16 MiB of device memory and fail with DAP_ERR_CUDA if there is none.
 * Make one call per device at start-up, before serving and before any stream capture (or
 * run with CUDA_MODULE_LOADING=EAGER); later calls reserve nothing.
 * The array keeps what the last call left in it; nothing in it has to start at zero,
 * because every partial a call reads was written earlier in that same call.  All calls
 * share the one array, so calls that overlap on the GPU (on different streams, or from
 * different host threads) race and corrupt each other's results: serialise them.
 * Calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define DAP_NOALLOC_SCRATCH_BYTES (16u << 20)
dap_status decode_attn_paged_noalloc(const void *q, long long q_stride_b, long long q_stride_h,
                                     const void *k_cache, const void *v_cache, int num_pages,
                                     int page_size, const int32_t *block_table, int max_pages,
                                     const int32_t *seq_lens, int max_kv_len, int B, int Hq,
                                     int Hkv, int D, float scale, int num_splits, void *out,
                                     long long out_stride_b, long long out_stride_h, void *stream);

/* Tracing hook.  When set (non-NULL cudaEvent_t handles passed as void*), every following
 * decode_attn_paged / decode_attn_contig call records `split_begin` just before its split
 * kernel, `split_end` just after it and `combine_end` after the combine kernel (or right
 * after split_end when there is none), all on the call's stream.  Pass NULLs to turn it
 * off.  Process-wide, not thread-safe; meant for benchmarks and profilers. */
void dap_set_trace_events(void *split_begin, void *split_end, void *combine_end);

/* Read (and, when `clear` is nonzero, reset) the device error word of the current
 * device.  Synchronises the device.  Returns DAP_ERR_CUDA if the read fails. */
dap_status dap_get_device_errors(unsigned int *flags, int clear);

/* Diagnostic for the failure path of every pipeline wait: launches one thread on `stream`
 * (a cudaStream_t, NULL = the default stream) that waits, through the same bounded wait
 * the decode kernels use, on a shared-memory barrier nothing ever arrives on.  After its
 * limit (about 2e9 SM cycles, near one second) the wait gives up, sets DAP_DEVERR_TIMEOUT
 * in the device error word and the kernel returns normally, so the context stays usable.
 * Asynchronous; returns DAP_ERR_CUDA if the launch fails.  For tests only. */
dap_status dap_selftest_wait_timeout(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DAP_H_ */
