// dap_internal.h -- host-side interface between the C ABI (dap_api.cu) and the kernel
// launchers (dap_decode.cu, dap_fp8.cu).  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dap.h"

namespace dap {

// The per-sequence split chunk is a multiple of this many tokens (a multiple of every
// kernel configuration's tile, so a TMA box never straddles a page).
constexpr int kTileTokens = 64;
// Balanced schedule: at most this many persistent CTAs (workspace is sized for it), and
// batches above kMaxBalancedBatch sequences use the per-sequence schedule instead (their
// units already fill the device, and every persistent CTA scans seq_lens once).
constexpr int kMaxPersistentCtas = 1024;
constexpr int kMaxBalancedBatch = 4096;

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of the balanced schedule: per-CTA partial slots (two each), the first tile and
// tile count of every unit, and the total tile count.
struct BalancedLayout {
    size_t acc, ml, info, total, bytes;
};
inline BalancedLayout balanced_layout(int B, int units_per_seq, int heads_per_unit, int D) {
    BalancedLayout l;
    const size_t slots = 2 * (size_t)kMaxPersistentCtas * heads_per_unit;
    l.acc = 0;
    l.ml = l.acc + align256(slots * D * sizeof(float));
    l.info = l.ml + align256(slots * 2 * sizeof(float));
    l.total = l.info + align256((size_t)B * units_per_seq * 2 * sizeof(int));
    l.bytes = l.total + 256;
    return l;
}
// Query heads and kv heads that one unit of the balanced schedule covers.
int balanced_heads_per_unit(int D, int G);
int balanced_kv_heads_per_unit(int D, int G);

// Everything a decode launch needs, already validated.
struct DecodeArgs {
    bool paged;
    const void *q;
    long long q_sb, q_sh;        // element strides
    const void *k, *v;           // paged: [num_pages, ps, Hkv, D]; contig: [B, max_len, Hkv, D]
    int num_pages, page_size;    // paged only
    int max_len;                 // contig only
    const int32_t *block_table;  // paged only
    int max_pages;
    const int32_t *seq_lens;
    int max_kv_len;
    int B, Hq, Hkv, D;
    float scale;
    int num_splits;              // 0 = balanced schedule, else per-sequence splits (>= 1)
    int chunk;                   // per-sequence: tokens per split chunk
    void *workspace;
    void *out;
    long long o_sb, o_sh;
    // e4m3 cache only: bf16 dequantisation factors [num_pages, Hkv, page_size] of k and v
    const void *k_scale, *v_scale;
    // multi-token decode only: packed-q work map (q_sb / o_sb are then token strides); none
    // (all NULL) for masked single-token decode
    const int32_t *qo_indptr, *tile_batch, *tile_index;
    int num_tiles, total_q, tokens_per_tile;
    // optional bool mask [total_q, mask_stride] bytes (nonzero = keep)
    const uint8_t *mask;
    long long mask_stride;
};

dap_status launch_decode(const DecodeArgs &a, cudaStream_t stream);
// paged cache with a page size that is not a multiple of 8 (row-gather producer)
dap_status launch_decode_gather(const DecodeArgs &a, cudaStream_t stream);
dap_status launch_decode_multi_gather(const DecodeArgs &a, cudaStream_t stream);
dap_status launch_decode_multi_tc(const DecodeArgs &a, cudaStream_t stream);
dap_status launch_decode_masked_gather(const DecodeArgs &a, cudaStream_t stream);
dap_status launch_decode_multi(const DecodeArgs &a, cudaStream_t stream);
dap_status launch_decode_masked(const DecodeArgs &a, cudaStream_t stream);
dap_status launch_decode_fp8kv(const DecodeArgs &a, cudaStream_t stream);
int multi_tokens_per_tile(int G, int D, int max_q_len);

// Events of dap_set_trace_events (nullptr when tracing is off).
struct TraceEvents {
    cudaEvent_t split_begin, split_end, combine_end;
};
extern TraceEvents g_trace;

struct Fp8Args {
    const void *q;
    const uint8_t *kv_cache;
    const void *inv_scale;
    const int64_t *slot_idx;
    const int64_t *lens;
    int T, NH, HD, W, num_blocks, block_size;
    float scale;
    void *out;
};

dap_status launch_fp8(const Fp8Args &a, cudaStream_t stream);

dap_status launch_append_paged(const void *k_new, const void *v_new, void *k_cache, void *v_cache, int num_pages,
                               int page_size, const int32_t *block_table, int max_pages, const int32_t *pos, int B,
                               int Hkv, int D, cudaStream_t stream);
dap_status launch_append_fp8(const void *rows, uint8_t *kv_cache, void *inv_scale, const int64_t *slots, int T,
                             int HD, int num_blocks, int block_size, cudaStream_t stream);
dap_status launch_append_paged_fp8(const void *k_new, const void *v_new, uint8_t *k_codes, uint8_t *v_codes,
                                   void *k_scale, void *v_scale, int num_pages, int page_size,
                                   const int32_t *block_table, int max_pages, const int32_t *pos, int B, int Hkv,
                                   int D, cudaStream_t stream);
bool read_errors_multi(unsigned int *flags, bool clear);
bool read_errors_multi_gather(unsigned int *flags, bool clear);
bool read_errors_multi_tc(unsigned int *flags, bool clear);
bool read_errors_fp8kv(unsigned int *flags, bool clear);
bool read_errors_append(unsigned int *flags, bool clear);

// Host readers of each translation unit's device error word (cudaMemcpyFromSymbol on the
// current device); `clear` resets it.  Return false when the copy fails.
bool read_errors_decode(unsigned int *flags, bool clear);
bool read_errors_decode_gather(unsigned int *flags, bool clear);
dap_status launch_selftest_wait(cudaStream_t stream);
bool read_errors_fp8(unsigned int *flags, bool clear);

// Driver entry point for cuTensorMapEncodeTiled, fetched through the runtime so the
// library does not link libcuda directly.  Returns nullptr if unavailable.
void *tensor_map_encoder();

// Offsets of the split partials inside the workspace.
inline size_t partial_acc_bytes(int B, int Hq, int D, int S) {
    return ((size_t)B * S * Hq * D * sizeof(float) + 255) & ~(size_t)255;
}
inline size_t partial_ml_bytes(int B, int Hq, int S) {
    return ((size_t)B * S * Hq * 2 * sizeof(float) + 255) & ~(size_t)255;
}

}  // namespace dap
