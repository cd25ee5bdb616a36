// dap_api.cu -- the C ABI: argument validation, split planning, workspace sizing, the
// device error word and the tensor-map encoder lookup.  Every host-detectable error is
// returned before any CUDA call is made, so these checks also run on machines without
// a GPU.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "dap.h"
#include "dap_internal.h"

namespace dap {

TraceEvents g_trace = {nullptr, nullptr, nullptr};

void *tensor_map_encoder() {
    static void *fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = p;
    });
    return fn;
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

bool supported_group(int G) { return G == 1 || G == 2 || G == 4 || G == 8; }

// Shared checks of the decode entry points.  `balanced_ok`: the entry point has the
// balanced schedule, so num_splits may be DAP_SPLITS_BALANCED.
dap_status check_common(const void *q, long long q_sb, long long q_sh, const int32_t *seq_lens,
                        int max_kv_len, int B, int Hq, int Hkv, int D, float scale, int num_splits,
                        const void *out, long long o_sb, long long o_sh, bool balanced_ok = false) {
    if (B < 0 || Hq < 1 || Hkv < 1 || D < 1 || max_kv_len < 0 || num_splits < DAP_SPLITS_BALANCED ||
        num_splits > 65536 || Hq % Hkv != 0 || !isfinite(scale) || q_sb < 0 || q_sh < 0 ||
        o_sb < 0 || o_sh < 0)
        return DAP_ERR_SHAPE;
    if (num_splits == DAP_SPLITS_BALANCED && !balanced_ok) return DAP_ERR_UNSUPPORTED;
    if (B == 0) return DAP_OK;
    if ((Hq > 1 && (q_sh == 0 || o_sh == 0)) || (B > 1 && (q_sb == 0 || o_sb == 0))) return DAP_ERR_SHAPE;
    if (!q || !seq_lens || !out) return DAP_ERR_NULL;
    if (!(D == 32 || D == 64 || D == 128 || D == 256) || !supported_group(Hq / Hkv)) return DAP_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(out) || !aligned4(seq_lens) || (q_sb & 7) || (q_sh & 7) ||
        (o_sb & 7) || (o_sh & 7))
        return DAP_ERR_ALIGN;
    return DAP_OK;
}

// The split count of a call (dap_resolve_splits on the current device) and its chunk, after
// checking the workspace against it.  `units` is the number of rows the planner schedules
// (sequences, or the work map's tiles).  On return *S_out is 0 for the balanced schedule,
// else the per-sequence S >= 1.
dap_status resolve_splits(int units, int rows, int Hq, int Hkv, int D, int page_size, int max_kv_len, int num_splits,
                          void *workspace, size_t workspace_bytes, bool multi, int *S_out, int *chunk_out) {
    int sms = 0;
    if (num_splits == 0) {
        sms = dap_device_sm_count();
        if (sms <= 0) return DAP_ERR_CUDA;
    }
    const int S = dap_resolve_splits(num_splits, sms, units, Hq, Hkv, D, page_size, max_kv_len, 0);
    if (S == 0) return DAP_ERR_SHAPE;
    if (S == DAP_SPLITS_BALANCED) {
        const size_t need = dap_workspace_bytes(rows, Hq, Hkv, D, DAP_SPLITS_BALANCED);
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DAP_ERR_WORKSPACE;
        *S_out = 0;
        *chunk_out = 0;
        return DAP_OK;
    }
    if (S > 1) {
        const size_t need = multi ? dap_workspace_bytes_multi(rows, Hq, D, S) : dap_workspace_bytes(rows, Hq, Hkv, D, S);
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DAP_ERR_WORKSPACE;
    }
    *S_out = S;
    *chunk_out = dap_chunk_tokens(max_kv_len, S);
    return DAP_OK;
}

// A bool mask (NULL = none): rows of mask_stride bytes, each covering at least max_kv_len
// keys, 16-byte aligned rows (it is read by TMA).
dap_status check_mask(const uint8_t *mask, long long mask_stride, int max_kv_len) {
    if (!mask) return DAP_OK;
    if (mask_stride < max_kv_len || mask_stride < 1 || mask_stride > (1LL << 32)) return DAP_ERR_SHAPE;
    if (!aligned16(mask) || (mask_stride & 15)) return DAP_ERR_ALIGN;
    return DAP_OK;
}

}  // namespace
}  // namespace dap

using namespace dap;

extern "C" {

const char *dap_status_string(int status) {
    switch (status) {
        case DAP_OK: return "ok";
        case DAP_ERR_NULL: return "a required pointer is NULL";
        case DAP_ERR_SHAPE: return "a size or stride is out of range or inconsistent";
        case DAP_ERR_UNSUPPORTED: return "shape not supported by this build";
        case DAP_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case DAP_ERR_ALIGN: return "pointer or stride breaks the 16-byte alignment rule";
        case DAP_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case DAP_ERR_SCRATCH_LIMIT:
            return "split partials exceed the no-allocation entry point's fixed scratch (DAP_NOALLOC_SCRATCH_BYTES)";
        default: return "unknown status";
    }
}

int dap_version(void) { return 100; }

int dap_device_sm_count(void) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

int dap_chunk_tokens(int max_kv_len, int num_splits) {
    const int S = std::max(1, num_splits);
    const long long per = ceil_div_ll(std::max(1, max_kv_len), S);
    const long long tiles = ceil_div_ll(per, kTileTokens);
    return (int)std::max<long long>(kTileTokens, tiles * kTileTokens);
}

int dap_plan_splits(int sm_count, int B, int Hq, int Hkv, int D, int page_size, int max_kv_len,
                    long long total_kv) {
    (void)Hq;
    (void)D;
    (void)page_size;
    if (sm_count <= 0 || B <= 0 || Hkv <= 0 || max_kv_len <= 0) return 1;
    if (total_kv <= 0) total_kv = (long long)B * max_kv_len;
    // Resident CTAs of the tensor-core configuration; one CTA per (sequence, kv head, chunk).
    const long long slots = (long long)sm_count * 2;
    const long long units = (long long)B * Hkv;
    long long S;
    if (units < slots) {
        // Too few units to fill the GPU: cut every sequence into as many chunks as fit one
        // wave, so equal-length batches finish together (AstrAI csrc log, split-KV commit:
        // choose the split count to fill the device).  Up to 8 chunks of a unit merge inside
        // one thread-block cluster, with no combine kernel: 8 is preferred to more while 8
        // chunks still fill four fifths of the wave.
        S = slots / units;
        if (S > 8 && 8 * units * 5 >= slots * 4) S = 8;
    } else {
        // Enough units: keep the largest unit a small fraction of one SM's share of the KV
        // rows so the last units to finish leave little of the GPU idle.
        const long long share = (total_kv * Hkv + sm_count - 1) / sm_count;
        const long long chunk_target = std::max<long long>(256, share / 10);
        S = ceil_div_ll(max_kv_len, chunk_target);
    }
    S = std::min(S, ceil_div_ll(max_kv_len, kTileTokens));
    S = std::min<long long>(S, 1024);
    return (int)std::max<long long>(1, S);
}

int dap_resolve_splits(int num_splits, int sm_count, int B, int Hq, int Hkv, int D, int page_size, int max_kv_len,
                       long long total_kv) {
    if (num_splits < DAP_SPLITS_BALANCED || B < 0 || Hq < 1 || Hkv < 1 || D < 1 || max_kv_len < 0) return 0;
    if (num_splits == DAP_SPLITS_BALANCED) return B <= kMaxBalancedBatch ? DAP_SPLITS_BALANCED : 1;
    const int S = num_splits == 0 ? dap_plan_splits(sm_count, B, Hq, Hkv, D, page_size, max_kv_len, total_kv)
                                  : num_splits;
    // splits that could never hold a token are dropped: S chunks must cover max_kv_len
    const int chunk = dap_chunk_tokens(max_kv_len, S);
    const int needed = max_kv_len > 0 ? (int)ceil_div_ll(max_kv_len, chunk) : 1;
    return std::max(1, std::min(S, needed));
}

size_t dap_workspace_bytes(int B, int Hq, int Hkv, int D, int num_splits) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || num_splits < DAP_SPLITS_BALANCED || num_splits == 0 ||
        num_splits == 1)
        return 0;
    if (num_splits == DAP_SPLITS_BALANCED) {
        if (B > kMaxBalancedBatch || Hq % Hkv != 0) return 0;
        const int G = Hq / Hkv;
        const int hg = balanced_kv_heads_per_unit(D, G);
        return balanced_layout(B, std::max(1, Hkv / hg), balanced_heads_per_unit(D, G), D).bytes;
    }
    return partial_acc_bytes(B, Hq, D, num_splits) + partial_ml_bytes(B, Hq, num_splits);
}

dap_status decode_attn_paged(const void *q, long long q_stride_b, long long q_stride_h,
                             const void *k_cache, const void *v_cache, int num_pages, int page_size,
                             const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                             int max_kv_len, int B, int Hq, int Hkv, int D, float scale,
                             int num_splits, void *workspace, size_t workspace_bytes, void *out,
                             long long out_stride_b, long long out_stride_h, void *stream) {
    dap_status st = check_common(q, q_stride_b, q_stride_h, seq_lens, max_kv_len, B, Hq, Hkv, D,
                                 scale, num_splits, out, out_stride_b, out_stride_h, true);
    if (st != DAP_OK || B == 0) return st;
    if (num_pages < 1 || page_size < 1 || max_pages < 1 ||
        (long long)max_kv_len > (long long)max_pages * page_size)
        return DAP_ERR_SHAPE;
    if (!k_cache || !v_cache || !block_table) return DAP_ERR_NULL;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned4(block_table)) return DAP_ERR_ALIGN;
    DecodeArgs a = {};
    a.paged = true;
    a.q = q;
    a.q_sb = q_stride_b;
    a.q_sh = q_stride_h;
    a.k = k_cache;
    a.v = v_cache;
    a.num_pages = num_pages;
    a.page_size = page_size;
    a.max_len = 0;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.seq_lens = seq_lens;
    a.max_kv_len = max_kv_len;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.scale = scale;
    a.workspace = workspace;
    a.out = out;
    a.o_sb = out_stride_b;
    a.o_sh = out_stride_h;
    st = resolve_splits(B, B, Hq, Hkv, D, page_size, max_kv_len, num_splits, workspace, workspace_bytes, false,
                        &a.num_splits, &a.chunk);
    if (st != DAP_OK) return st;
    return launch_decode(a, static_cast<cudaStream_t>(stream));
}

dap_status decode_attn_contig(const void *q, long long q_stride_b, long long q_stride_h, const void *k,
                              const void *v, int max_len, const int32_t *seq_lens, int max_kv_len,
                              int B, int Hq, int Hkv, int D, float scale, int num_splits,
                              void *workspace, size_t workspace_bytes, void *out,
                              long long out_stride_b, long long out_stride_h, void *stream) {
    dap_status st = check_common(q, q_stride_b, q_stride_h, seq_lens, max_kv_len, B, Hq, Hkv, D,
                                 scale, num_splits, out, out_stride_b, out_stride_h, true);
    if (st != DAP_OK || B == 0) return st;
    if (max_len < 1 || max_kv_len > max_len) return DAP_ERR_SHAPE;
    if (!k || !v) return DAP_ERR_NULL;
    if (!aligned16(k) || !aligned16(v)) return DAP_ERR_ALIGN;
    DecodeArgs a = {};
    a.paged = false;
    a.q = q;
    a.q_sb = q_stride_b;
    a.q_sh = q_stride_h;
    a.k = k;
    a.v = v;
    a.num_pages = 0;
    a.page_size = 0;
    a.max_len = max_len;
    a.block_table = nullptr;
    a.max_pages = 0;
    a.seq_lens = seq_lens;
    a.max_kv_len = max_kv_len;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.scale = scale;
    a.workspace = workspace;
    a.out = out;
    a.o_sb = out_stride_b;
    a.o_sh = out_stride_h;
    st = resolve_splits(B, B, Hq, Hkv, D, max_len, max_kv_len, num_splits, workspace, workspace_bytes, false,
                        &a.num_splits, &a.chunk);
    if (st != DAP_OK) return st;
    return launch_decode(a, static_cast<cudaStream_t>(stream));
}

int dap_multi_tokens_per_tile(int Hq, int Hkv, int D, int max_q_len) {
    if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 0) return 0;
    return multi_tokens_per_tile(Hq / Hkv, D, max_q_len);
}

int dap_q_tile_map(const int32_t *q_lens, int B, int tokens_per_tile, int32_t *qo_indptr, int32_t *tile_batch,
                   int32_t *tile_index, int max_tiles) {
    if (B < 0 || tokens_per_tile < 1 || max_tiles < 0 || (B > 0 && (!q_lens || !qo_indptr))) return -1;
    if (B == 0) {
        if (qo_indptr) qo_indptr[0] = 0;
        return 0;
    }
    long long total = 0;
    int n = 0;
    qo_indptr[0] = 0;
    for (int b = 0; b < B; ++b) {
        const int len = q_lens[b];
        if (len < 0) return -1;
        total += len;
        if (total > 0x7FFFFFFFLL) return -1;
        qo_indptr[b + 1] = (int32_t)total;
        const int tiles = (int)ceil_div_ll(len, tokens_per_tile);
        for (int j = 0; j < tiles; ++j) {
            if (n >= max_tiles || !tile_batch || !tile_index) return -1;
            tile_batch[n] = b;
            tile_index[n] = j;
            ++n;
        }
    }
    return n;
}

size_t dap_workspace_bytes_multi(int total_q, int Hq, int D, int num_splits) {
    if (total_q <= 0 || Hq <= 0 || D <= 0 || num_splits <= 1) return 0;
    return partial_acc_bytes(total_q, Hq, D, num_splits) + partial_ml_bytes(total_q, Hq, num_splits);
}

dap_status decode_attn_paged_multi(const void *q, long long q_stride_t, long long q_stride_h,
                                   const void *k_cache, const void *v_cache, int num_pages, int page_size,
                                   const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                                   const int32_t *qo_indptr, const int32_t *tile_batch,
                                   const int32_t *tile_index, int num_tiles, int tokens_per_tile, int total_q,
                                   const uint8_t *mask,
                                   long long mask_stride, int max_kv_len, int B, int Hq, int Hkv, int D,
                                   float scale, int num_splits, void *workspace, size_t workspace_bytes,
                                   void *out, long long out_stride_t, long long out_stride_h, void *stream) {
    if (total_q < 0 || num_tiles < 0 || B < 0) return DAP_ERR_SHAPE;
    if (total_q == 0 && num_tiles == 0) return DAP_OK;
    // tokens without tiles, tiles without tokens, or more tiles than tokens
    if (B == 0 || total_q == 0 || num_tiles == 0 || num_tiles > total_q) return DAP_ERR_SHAPE;
    dap_status st = check_common(q, q_stride_t, q_stride_h, seq_lens, max_kv_len, total_q, Hq, Hkv, D, scale,
                                 num_splits, out, out_stride_t, out_stride_h);
    if (st != DAP_OK) return st;
    if (num_pages < 1 || page_size < 1 || max_pages < 1 ||
        (long long)max_kv_len > (long long)max_pages * page_size)
        return DAP_ERR_SHAPE;
    if (!k_cache || !v_cache || !block_table || !qo_indptr || !tile_batch || !tile_index) return DAP_ERR_NULL;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned4(block_table) || !aligned4(qo_indptr) ||
        !aligned4(tile_batch) || !aligned4(tile_index))
        return DAP_ERR_ALIGN;
    {
        const int G = Hq / Hkv;
        const int cols = tokens_per_tile * G;
        if (cols != 16 && cols != 32 && cols != 128) return DAP_ERR_SHAPE;
        if (mask && cols == 32) return DAP_ERR_UNSUPPORTED;
        if (cols == 128 && D != 64 && D != 128 && D != 256) return DAP_ERR_UNSUPPORTED;
    }
    if ((st = check_mask(mask, mask_stride, max_kv_len)) != DAP_OK) return st;
    int S = 0, chunk = 0;
    if ((st = resolve_splits(num_tiles, total_q, Hq, Hkv, D, page_size, max_kv_len, num_splits, workspace,
                             workspace_bytes, true, &S, &chunk)) != DAP_OK)
        return st;
    DecodeArgs a = {};
    a.paged = true;
    a.q = q;
    a.q_sb = q_stride_t;
    a.q_sh = q_stride_h;
    a.k = k_cache;
    a.v = v_cache;
    a.num_pages = num_pages;
    a.page_size = page_size;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.seq_lens = seq_lens;
    a.max_kv_len = max_kv_len;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.scale = scale;
    a.num_splits = S;
    a.chunk = chunk;
    a.workspace = workspace;
    a.out = out;
    a.o_sb = out_stride_t;
    a.o_sh = out_stride_h;
    a.qo_indptr = qo_indptr;
    a.tile_batch = tile_batch;
    a.tile_index = tile_index;
    a.num_tiles = num_tiles;
    a.tokens_per_tile = tokens_per_tile;
    a.total_q = total_q;
    a.mask = mask;
    a.mask_stride = mask_stride;
    return launch_decode_multi(a, static_cast<cudaStream_t>(stream));
}

dap_status decode_attn_paged_masked(const void *q, long long q_stride_b, long long q_stride_h, const void *k_cache,
                                    const void *v_cache, int num_pages, int page_size, const int32_t *block_table,
                                    int max_pages, const int32_t *seq_lens, const uint8_t *mask,
                                    long long mask_stride, int max_kv_len, int B, int Hq, int Hkv, int D,
                                    float scale, int num_splits, void *workspace, size_t workspace_bytes,
                                    void *out, long long out_stride_b, long long out_stride_h, void *stream) {
    dap_status st = check_common(q, q_stride_b, q_stride_h, seq_lens, max_kv_len, B, Hq, Hkv, D, scale, num_splits,
                                 out, out_stride_b, out_stride_h);
    if (st != DAP_OK || B == 0) return st;
    if (num_pages < 1 || page_size < 1 || max_pages < 1 ||
        (long long)max_kv_len > (long long)max_pages * page_size)
        return DAP_ERR_SHAPE;
    if (!k_cache || !v_cache || !block_table) return DAP_ERR_NULL;
    if (!mask) return DAP_ERR_NULL;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned4(block_table)) return DAP_ERR_ALIGN;
    if ((st = check_mask(mask, mask_stride, max_kv_len)) != DAP_OK) return st;
    int S = 0, chunk = 0;
    if ((st = resolve_splits(B, B, Hq, Hkv, D, page_size, max_kv_len, num_splits, workspace, workspace_bytes, false,
                             &S, &chunk)) != DAP_OK)
        return st;
    DecodeArgs a = {};
    a.paged = true;
    a.q = q;
    a.q_sb = q_stride_b;
    a.q_sh = q_stride_h;
    a.k = k_cache;
    a.v = v_cache;
    a.num_pages = num_pages;
    a.page_size = page_size;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.seq_lens = seq_lens;
    a.max_kv_len = max_kv_len;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.scale = scale;
    a.num_splits = S;
    a.chunk = chunk;
    a.workspace = workspace;
    a.out = out;
    a.o_sb = out_stride_b;
    a.o_sh = out_stride_h;
    a.num_tiles = B;  // one token per sequence, no work map
    a.tokens_per_tile = 1;
    a.total_q = B;
    a.mask = mask;
    a.mask_stride = mask_stride;
    return launch_decode_masked(a, static_cast<cudaStream_t>(stream));
}

dap_status decode_attn_paged_fp8kv(const void *q, long long q_stride_b, long long q_stride_h,
                                   const uint8_t *k_codes, const uint8_t *v_codes, const void *k_scale,
                                   const void *v_scale, int num_pages, int page_size, const int32_t *block_table,
                                   int max_pages, const int32_t *seq_lens, int max_kv_len, int B, int Hq, int Hkv,
                                   int D, float scale, int num_splits, void *workspace, size_t workspace_bytes,
                                   void *out, long long out_stride_b, long long out_stride_h, void *stream) {
    dap_status st = check_common(q, q_stride_b, q_stride_h, seq_lens, max_kv_len, B, Hq, Hkv, D, scale, num_splits,
                                 out, out_stride_b, out_stride_h);
    if (st != DAP_OK || B == 0) return st;
    if (num_pages < 1 || page_size < 1 || max_pages < 1 ||
        (long long)max_kv_len > (long long)max_pages * page_size)
        return DAP_ERR_SHAPE;
    if (!k_codes || !v_codes || !k_scale || !v_scale || !block_table) return DAP_ERR_NULL;
    if (D != 64 && D != 128 && D != 256) return DAP_ERR_UNSUPPORTED;
    if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scale) || !aligned16(v_scale) ||
        !aligned4(block_table))
        return DAP_ERR_ALIGN;
    int S = 0, chunk = 0;
    if ((st = resolve_splits(B, B, Hq, Hkv, D, page_size, max_kv_len, num_splits, workspace, workspace_bytes, false,
                             &S, &chunk)) != DAP_OK)
        return st;
    DecodeArgs a = {};
    a.paged = true;
    a.q = q;
    a.q_sb = q_stride_b;
    a.q_sh = q_stride_h;
    a.k = k_codes;
    a.v = v_codes;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.num_pages = num_pages;
    a.page_size = page_size;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.seq_lens = seq_lens;
    a.max_kv_len = max_kv_len;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.scale = scale;
    a.num_splits = S;
    a.chunk = chunk;
    a.workspace = workspace;
    a.out = out;
    a.o_sb = out_stride_b;
    a.o_sh = out_stride_h;
    return launch_decode_fp8kv(a, static_cast<cudaStream_t>(stream));
}

dap_status kv_append_paged_fp8(const void *k_new, const void *v_new, uint8_t *k_codes, uint8_t *v_codes,
                               void *k_scale, void *v_scale, int num_pages, int page_size,
                               const int32_t *block_table, int max_pages, const int32_t *positions, int B, int Hkv,
                               int D, void *stream) {
    if (B < 0 || Hkv < 1 || D < 1 || num_pages < 1 || page_size < 1 || max_pages < 1) return DAP_ERR_SHAPE;
    if (B == 0) return DAP_OK;
    if (!(D == 64 || D == 128 || D == 256)) return DAP_ERR_UNSUPPORTED;
    if (!k_new || !v_new || !k_codes || !v_codes || !k_scale || !v_scale || !block_table || !positions)
        return DAP_ERR_NULL;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_codes) || !aligned16(v_codes) ||
        (reinterpret_cast<uintptr_t>(k_scale) & 1u) || (reinterpret_cast<uintptr_t>(v_scale) & 1u) ||
        !aligned4(block_table) || !aligned4(positions))
        return DAP_ERR_ALIGN;
    return launch_append_paged_fp8(k_new, v_new, k_codes, v_codes, k_scale, v_scale, num_pages, page_size,
                                   block_table, max_pages, positions, B, Hkv, D, static_cast<cudaStream_t>(stream));
}

dap_status decode_attn_paged_fp8(const void *q, const uint8_t *kv_cache, const void *inv_scale,
                                 const int64_t *slot_idx, const int64_t *lens, int T, int NH, int HD,
                                 int W, int num_blocks, int block_size, float scale, void *out,
                                 void *stream) {
    if (T < 0 || NH < 1 || HD < 1 || W < 1 || num_blocks < 1 || block_size < 1 || !isfinite(scale) ||
        (long long)num_blocks * block_size > 0x7FFFFFFFLL)
        return DAP_ERR_SHAPE;
    if (T == 0) return DAP_OK;
    if (!q || !kv_cache || !inv_scale || !slot_idx || !lens || !out) return DAP_ERR_NULL;
    if (HD != 512 || NH % 128 != 0 || NH > 1024 || W > 128 || T > 65535) return DAP_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(out) || !aligned16(kv_cache) ||
        (reinterpret_cast<uintptr_t>(inv_scale) & 1u) || (reinterpret_cast<uintptr_t>(slot_idx) & 7u) ||
        (reinterpret_cast<uintptr_t>(lens) & 7u))
        return DAP_ERR_ALIGN;
    Fp8Args a;
    a.q = q;
    a.kv_cache = kv_cache;
    a.inv_scale = inv_scale;
    a.slot_idx = slot_idx;
    a.lens = lens;
    a.T = T;
    a.NH = NH;
    a.HD = HD;
    a.W = W;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.scale = scale;
    a.out = out;
    return launch_fp8(a, static_cast<cudaStream_t>(stream));
}

dap_status kv_append_paged(const void *k_new, const void *v_new, void *k_cache, void *v_cache, int num_pages,
                           int page_size, const int32_t *block_table, int max_pages, const int32_t *positions, int B,
                           int Hkv, int D, void *stream) {
    if (B < 0 || Hkv < 1 || D < 1 || num_pages < 1 || page_size < 1 || max_pages < 1) return DAP_ERR_SHAPE;
    if (B == 0) return DAP_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !positions) return DAP_ERR_NULL;
    if (D % 8 != 0) return DAP_ERR_UNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned4(block_table) || !aligned4(positions))
        return DAP_ERR_ALIGN;
    return launch_append_paged(k_new, v_new, k_cache, v_cache, num_pages, page_size, block_table, max_pages,
                               positions, B, Hkv, D, static_cast<cudaStream_t>(stream));
}

dap_status kv_append_fp8(const void *rows, uint8_t *kv_cache, void *inv_scale, const int64_t *slots, int T, int HD,
                         int num_blocks, int block_size, void *stream) {
    if (T < 0 || HD < 1 || num_blocks < 1 || block_size < 1 || (long long)num_blocks * block_size > 0x7FFFFFFFLL)
        return DAP_ERR_SHAPE;
    if (T == 0) return DAP_OK;
    if (!rows || !kv_cache || !inv_scale || !slots) return DAP_ERR_NULL;
    if (HD != 256 && HD != 512) return DAP_ERR_UNSUPPORTED;
    if (!aligned16(rows) || !aligned16(kv_cache) || (reinterpret_cast<uintptr_t>(inv_scale) & 1u) ||
        (reinterpret_cast<uintptr_t>(slots) & 7u))
        return DAP_ERR_ALIGN;
    return launch_append_fp8(rows, kv_cache, inv_scale, slots, T, HD, num_blocks, block_size,
                             static_cast<cudaStream_t>(stream));
}

void dap_set_trace_events(void *split_begin, void *split_end, void *combine_end) {
    g_trace.split_begin = static_cast<cudaEvent_t>(split_begin);
    g_trace.split_end = static_cast<cudaEvent_t>(split_end);
    g_trace.combine_end = static_cast<cudaEvent_t>(combine_end);
}

dap_status dap_selftest_wait_timeout(void *stream) {
    return launch_selftest_wait(static_cast<cudaStream_t>(stream));
}

dap_status dap_get_device_errors(unsigned int *flags, int clear) {
    if (!flags) return DAP_ERR_NULL;
    *flags = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return DAP_ERR_CUDA;
    if (!read_errors_decode(flags, clear != 0)) return DAP_ERR_CUDA;
    if (!read_errors_decode_gather(flags, clear != 0)) return DAP_ERR_CUDA;
    if (!read_errors_fp8(flags, clear != 0)) return DAP_ERR_CUDA;
    if (!read_errors_append(flags, clear != 0)) return DAP_ERR_CUDA;
    if (!read_errors_multi(flags, clear != 0)) return DAP_ERR_CUDA;
    if (!read_errors_multi_gather(flags, clear != 0)) return DAP_ERR_CUDA;
    if (!read_errors_multi_tc(flags, clear != 0)) return DAP_ERR_CUDA;
    if (!read_errors_fp8kv(flags, clear != 0)) return DAP_ERR_CUDA;
    return DAP_OK;
}

}  // extern "C"
