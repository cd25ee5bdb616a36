// dap_tile.cuh -- pieces shared by the bf16 paged decode kernels: the single-token
// schedules (dap_decode.cu) and the multi-token one (dap_multi.cu).  Launch parameters,
// the shared-memory alignment rule of the swizzled tiles, the TMA issue of one K/V box,
// the consumer-warp barrier, the normalised bf16 store, the row merge of split partials
// and the host-side tensor-map encoding and launch helpers.
#pragma once

#include <math.h>

#include <mutex>
#include <type_traits>

#include "dap_device.cuh"
#include "dap_internal.h"

namespace dap {

struct SplitParams {
    const __nv_bfloat16 *q;
    long long q_sb, q_sh;
    const __nv_bfloat16 *k_cache, *v_cache;  // read directly by the row-gather producer
    const uint8_t *k_codes, *v_codes;        // e4m3 cache (row gather): codes and factors
    const void *k_scale, *v_scale;
    const int32_t *block_table;
    int max_pages;
    const int32_t *seq_lens;
    int max_kv_len;
    int B, Hq, Hkv;
    int page_size, num_pages, box_rows;
    int num_splits, chunk;  // per-sequence schedule
    int num_ctas;           // balanced schedule: P
    float qscale;           // scale * log2(e)
    float *o_part;
    float *ml_part;
    int *unit_info;         // balanced: [units][2] = first tile, tiles
    long long *total_tiles; // balanced: T
    __nv_bfloat16 *out;
    long long o_sb, o_sh;
    // multi-token decode: packed q / out rows are tokens; q_sb / o_sb are the token strides
    const int32_t *qo_indptr, *tile_batch, *tile_index;
    int num_tiles, total_q;
};

__device__ __forceinline__ void store_out_pair(__nv_bfloat16 *o, float a0, float a1, float l) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    *reinterpret_cast<__nv_bfloat162 *>(o) = __floats2bfloat162_rn(a0 * inv, a1 * inv);
}

// 1024-byte aligned view of the dynamic shared memory (the 128-byte swizzle is a function
// of address bits 4..9, so swizzled tiles must start on 1024-byte boundaries).
template <class C>
__device__ __forceinline__ uint8_t *aligned_smem(uint8_t *raw) {
    if constexpr (C::SWZ) return raw + ((1024u - (smem_addr(raw) & 1023u)) & 1023u);
    return raw;
}

// Barrier among the NWC consumer warps on an mbarrier (count NWC, one arrival per warp),
// so that a wait is bounded like every other wait in the pipeline.
struct ConsumerBarrier {
    uint64_t *bar;
    uint32_t phase;
    __device__ __forceinline__ bool sync(int lane) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
        const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar, phase & 1));
        ++phase;
        return ok;
    }
};

// K / V tile layout: boxes of R = 2^rb rows (R = gcd(page size, BT) for TMA-fed paged
// tiles, BT for the contiguous cache and the row gather), each box [NBLK column blocks][R
// rows][SWB bytes], SWB-byte swizzled (the layout one 5-D TMA box over [SWB/2 dims, rows,
// column block, kv head, page] produces).  Byte offset of 16-byte chunk `ch` (0 .. NBLK * CPB
// - 1) of tile row `key`; the 128-byte swizzle XORs the chunk index within its block with
// key & 7, the 64-byte one with (key >> 1) & 3 (every box segment starts on a swizzle atom).
template <class C>
__device__ __forceinline__ uint32_t tile_off(int key, int ch, int rb) {
    const int blk = ch / C::CPB, cib = ch % C::CPB;
    const int sw = C::SWB == 128 ? (key & 7) : ((key >> 1) & 3);
    return (uint32_t)((((key >> rb) * C::NBLK + blk) << rb) * C::SWB + (key & ((1 << rb) - 1)) * C::SWB +
                      ((cib ^ sw) << 4));
}

// The K and V boxes of one producer lane: box j of the stage covers tile rows [j*R,
// (j+1)*R), every column block of them (one TMA copy per tensor).
template <class C>
__device__ __forceinline__ void issue_kv_box(uint8_t *stage, int j, int R, const CUtensorMap *mk,
                                             const CUtensorMap *mv, int kvh0, int row, int page, uint64_t *bar) {
    static_assert(C::SWZ, "swizzled tiles");
    uint8_t *dst = stage + j * R * C::ROWB;
    tma_load_5d(dst, mk, 0, row, 0, kvh0, page, bar);
    tma_load_5d(dst + C::TILE_BYTES, mv, 0, row, 0, kvh0, page, bar);
}

// ---- row gather: page sizes that are not multiples of 8 ---------------------------------
// Such a page size cuts a tile into boxes of fewer than 8 rows, which could not start on
// the boundaries of the swizzle pattern (8 rows), so the producer warp copies the rows
// itself: 16-byte cp.async chunks written straight to the swizzled positions the consumers
// read.  (Measured on the ragged batch: as fast as the TMA boxes of a page size of 16,
// while 8-row TMA boxes for the groups of rows that lie in one page were slower.)

template <class C>
struct RowPages {
    static constexpr int N = (C::BT + 31) / 32;  // tile rows per lane: lane, lane + 32, ...
    int pg[N], slot[N];
};

// Raw page ids (block-table entries) and in-page slots of this lane's rows of a tile whose
// first token is `tok`; rows at or past `nvalid` get page 0.  The loads are only issued
// here: the values are first used by fill_tile_rows, one tile later.
template <class C>
__device__ __forceinline__ void lookup_rows(RowPages<C> &rp, const int32_t *table, int tok, int nvalid,
                                            int page_size, int lane) {
#pragma unroll
    for (int k = 0; k < RowPages<C>::N; ++k) {
        const int r = lane + 32 * k;
        rp.pg[k] = 0;
        rp.slot[k] = 0;
        if (r < nvalid) {
            const int t = tok + r;
            rp.pg[k] = __ldg(table + t / page_size);
            rp.slot[k] = t % page_size;
        }
    }
}

// Copy rows [0, nvalid) of kv head `kvh` into the stage's [NBLK][BT][SWB] K and V tiles
// (128-byte swizzle: 16-byte chunk index XOR row & 7; 64-byte: XOR (row >> 1) & 3), and
// arrive on `full`: lane 0 once, with the `extra_tx` bytes of the TMA copies that
// `extra()` (run by lane 0) issues (q, mask), and every lane once its cp.async copies have
// landed (the barrier counts 33 arrivals).  Lane = (row r0 of every RPI rows, chunk c):
// a warp-wide copy reads RPI whole rows, and the row step is a compile-time constant (the
// copy loop is issue-bound: a per-chunk index search made it three times slower).  Page
// ids outside the pool are read as page 0 and flagged, as in the TMA path.
template <class C, class Extra>
__device__ __forceinline__ void fill_tile_rows(uint8_t *stage, const RowPages<C> &rp, int nvalid, int kvh,
                                               const SplitParams &p, uint32_t extra_tx, Extra extra, uint64_t *full,
                                               int lane) {
    constexpr int CPR = C::ROWB / 16;  // 16-byte chunks per row
    constexpr int N = RowPages<C>::N, RPI = 32 / CPR;
    static_assert(CPR <= 32 && 32 % CPR == 0 && C::BT % RPI == 0, "whole rows per warp-wide copy");
    long long row[N];                  // element offset of this lane's rows in the cache
#pragma unroll
    for (int k = 0; k < N; ++k) {
        int pg = rp.pg[k];
        if (lane + 32 * k < nvalid && (pg < 0 || pg >= p.num_pages)) {
            flag_error(DAP_DEVERR_PAGE);
            pg = 0;
        }
        row[k] = (((long long)pg * p.page_size + rp.slot[k]) * p.Hkv + kvh) * C::D;
    }
    if (lane == 0) {
        if (extra_tx) mbar_arrive_expect_tx(full, extra_tx);
        else mbar_arrive(full);
        extra();
    }
    const int c = lane % CPR, r0 = lane / CPR;
    const int blk = c / C::CPB, cib = c % C::CPB;
    const uint32_t sk = smem_addr(stage) + blk * (C::BT * C::SWB), sv = sk + C::TILE_BYTES;
    const __nv_bfloat16 *kc = p.k_cache + c * 8, *vc = p.v_cache + c * 8;
#pragma unroll
    for (int it = 0; it < C::BT / RPI; ++it) {
        const int r = r0 + RPI * it;
        const long long off = __shfl_sync(0xFFFFFFFFu, row[(RPI * it) >> 5], r & 31);
        if (r < nvalid) {
            const int sw = C::SWB == 128 ? (r & 7) : ((r >> 1) & 3);
            const uint32_t dst = (uint32_t)(r * C::SWB + ((cib ^ sw) << 4));
            cp_async_16(sk + dst, kc + off);
            cp_async_16(sv + dst, vc + off);
        }
    }
    cp_async_mbar_arrive(full);
}

// Arrivals a stage's full barrier expects: one (the producer's arrive with the TMA byte
// count), or in row-gather mode one per producer lane plus lane 0's own arrive (which
// carries the bytes of the tile's TMA copies).
template <class C>
__host__ __device__ constexpr uint32_t full_arrivals() {
    return C::GATHER ? 33u : 1u;
}

// Merge of split partials for one output row, one warp, lanes over D: M = max_s m_s,
// out = sum_s 2^(m_s-M) acc_s / sum_s 2^(m_s-M) l_s (AstrAI csrc log, split-KV commit: the
// combine kernel; numerics commit: guarded division).
// DPV consecutive floats of a partial row (DPV = D / 32 in 1..8), vector loads where they fit.
template <int DPV>
__device__ __forceinline__ void load_row_part(const float *src, float (&x)[DPV]) {
    if constexpr (DPV % 4 == 0) {
#pragma unroll
        for (int j = 0; j < DPV; j += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(src + j);
            x[j] = v.x;
            x[j + 1] = v.y;
            x[j + 2] = v.z;
            x[j + 3] = v.w;
        }
    } else if constexpr (DPV == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(src);
        x[0] = v.x;
        x[1] = v.y;
    } else {
#pragma unroll
        for (int j = 0; j < DPV; ++j) x[j] = src[j];
    }
}

// Normalise and store one lane's DPV output values (bf16, round to nearest even).
template <int DPV>
__device__ __forceinline__ void store_row_part(__nv_bfloat16 *o, const float (&a)[DPV], float l) {
    if constexpr (DPV == 1) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        *o = __float2bfloat16_rn(a[0] * inv);
    } else {
#pragma unroll
        for (int j = 0; j < DPV; j += 2) store_out_pair(o + j, a[j], a[j + 1], l);
    }
}

template <int D>
struct RowMerge {
    static constexpr int DPV = D / 32;
    float acc[DPV];
    float lsum, Mu;
    __device__ __forceinline__ void begin(float m_max) {
        Mu = (m_max == -INFINITY) ? 0.f : m_max;
        lsum = 0.f;
#pragma unroll
        for (int j = 0; j < DPV; ++j) acc[j] = 0.f;
    }
    // add the partial rows o[0..n) (n <= 8), whose loads are all issued before any use
    __device__ __forceinline__ void add_batch(const float *const *o, const float2 *ml, int n, int lane) {
        float x[8][DPV];
        float f[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < n) {
                load_row_part<DPV>(o[k] + lane * DPV, x[k]);
                f[k] = ex2(ml[k].x - Mu);
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < n) {
                lsum = fmaf(f[k], ml[k].y, lsum);
#pragma unroll
                for (int j = 0; j < DPV; ++j) acc[j] = fmaf(f[k], x[k][j], acc[j]);
            }
        }
    }
    __device__ __forceinline__ void store(__nv_bfloat16 *o, int lane) { store_row_part<DPV>(o + lane * DPV, acc, lsum); }
};

// Per-sequence schedule: merge the splits of every (sequence, head) row that more than one
// CTA worked on, one warp per row; waits for the split grid (programmatic dependent launch).
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const SplitParams p) {
    // the next decode call may be launched now (it waits for this grid before its reads)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= p.B * p.Hq) return;
    const int b = gw / p.Hq, hq = gw - b * p.Hq;
    const int L = min(max(p.seq_lens[b], 0), p.max_kv_len);
    const int nsplit = max(1, (L + p.chunk - 1) / p.chunk);
    if (nsplit == 1) return;
    const long long row0 = (long long)b * p.num_splits * p.Hq + hq;
    float M = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, p.ml_part[(row0 + (long long)s * p.Hq) * 2]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    RowMerge<D> r;
    r.begin(M);
    for (int s0 = 0; s0 < nsplit; s0 += 8) {
        const float *o[8];
        float2 ml[8];
        const int n = min(8, nsplit - s0);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const long long row = row0 + (long long)min(s0 + k, nsplit - 1) * p.Hq;
            o[k] = p.o_part + row * D;
            ml[k] = *reinterpret_cast<const float2 *>(p.ml_part + row * 2);
        }
        r.add_batch(o, ml, n, lane);
    }
    r.store(p.out + (long long)b * p.o_sb + (long long)hq * p.o_sh, lane);
}

// Per-sequence schedule with many splits: one CTA per (sequence, head) row, warp w taking
// splits w, w + 8, ... (one batch of loads per warp for up to 64 splits), the eight warp
// partials summed in warp order through shared memory (a fixed order, so results do not
// depend on timing); waits for the split grid (programmatic dependent launch).
template <int D>
__global__ void __launch_bounds__(256) combine_wide_kernel(const SplitParams p) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int DPV = D / 32;
    __shared__ float red_acc[8][D];
    __shared__ float red_m[8], red_l[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x / p.Hq, hq = blockIdx.x - b * p.Hq;
    if (b >= p.B) return;
    const int L = min(max(p.seq_lens[b], 0), p.max_kv_len);
    const int nsplit = max(1, (L + p.chunk - 1) / p.chunk);
    if (nsplit == 1) return;
    const long long row0 = (long long)b * p.num_splits * p.Hq + hq;
    float M = -INFINITY;
    for (int s = threadIdx.x; s < nsplit; s += 256) M = fmaxf(M, p.ml_part[(row0 + (long long)s * p.Hq) * 2]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    if (lane == 0) red_m[warp] = M;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < 8; ++w) M = fmaxf(M, red_m[w]);
    RowMerge<D> r;
    r.begin(M);
    for (int s0 = warp; s0 < nsplit; s0 += 64) {
        const float *o[8];
        float2 ml[8];
        const int n = min(8, (nsplit - s0 + 7) / 8);  // splits s0, s0 + 8, ... below nsplit
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const long long row = row0 + (long long)(s0 + 8 * min(k, n - 1)) * p.Hq;
            o[k] = p.o_part + row * D;
            ml[k] = *reinterpret_cast<const float2 *>(p.ml_part + row * 2);
        }
        r.add_batch(o, ml, n, lane);
    }
#pragma unroll
    for (int j = 0; j < DPV; ++j) red_acc[warp][lane * DPV + j] = r.acc[j];
    if (lane == 0) red_l[warp] = r.lsum;
    __syncthreads();
    if (threadIdx.x < D / 2) {
        const int d = 2 * threadIdx.x;
        float a0 = 0.f, a1 = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            a0 += red_acc[w][d];
            a1 += red_acc[w][d + 1];
            l += red_l[w];
        }
        store_out_pair(p.out + (long long)b * p.o_sb + (long long)hq * p.o_sh + d, a0, a1, l);
    }
}

// ---- host side ----------------------------------------------------------------------------

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

bool encode_bf16(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims,
                 const cuuint64_t *strides_bytes, const cuuint32_t *box,
                 CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE) {
    EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) return false;
    const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), dims,
               strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, Hkv, D] cache (per page, or per sequence for the contiguous cache) viewed for the
// swizzled tile layout (see tile_off).
template <class C>
bool encode_cache_map(CUtensorMap *map, const void *base, int D, int Hkv, long long rows, long long outer,
                      int box_rows) {
    static_assert(C::SWZ, "swizzled tiles");
    // [SWB/2 dims, rows, column block, kv head, page]: one box = box_rows rows of every
    // column block of one kv head, landing block-major
    const cuuint64_t dims[5] = {(cuuint64_t)(C::SWB / 2), (cuuint64_t)rows, (cuuint64_t)(D * 2 / C::SWB),
                                (cuuint64_t)Hkv, (cuuint64_t)outer};
    const cuuint64_t strides[4] = {(cuuint64_t)Hkv * D * 2, (cuuint64_t)C::SWB, (cuuint64_t)D * 2,
                                   (cuuint64_t)rows * Hkv * D * 2};
    const cuuint32_t box[5] = {(cuuint32_t)(C::SWB / 2), (cuuint32_t)box_rows, (cuuint32_t)(D * 2 / C::SWB), 1u, 1u};
    return encode_bf16(map, base, 5, dims, strides, box,
                       C::SWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

// [D, Hq, B] view of q with its strides, box [D, hpu, 1].
bool encode_q_map(CUtensorMap *map, const DecodeArgs &a, int hpu) {
    const cuuint64_t dims[3] = {(cuuint64_t)a.D, (cuuint64_t)a.Hq, (cuuint64_t)a.B};
    // a stride over an extent of 1 is never used; give TMA a valid one
    const long long sh = a.Hq > 1 ? a.q_sh : a.D;
    const long long sb = a.B > 1 ? a.q_sb : (long long)a.Hq * sh;
    const cuuint64_t strides[2] = {(cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
    const cuuint32_t box[3] = {(cuuint32_t)a.D, (cuuint32_t)hpu, 1u};
    return encode_bf16(map, a.q, 3, dims, strides, box);
}

int gcd_int(int x, int y) {
    while (y) {
        const int t = x % y;
        x = y;
        y = t;
    }
    return x;
}

std::mutex g_attr_mu;

// Function attributes belong to a device's context, so a kernel is prepared once per device.
constexpr int kMaxDevices = 64;
struct PerDeviceOcc {
    int occ[kMaxDevices];
};

// Raise the dynamic shared-memory limit of `kern` once per device (the current one), and
// return its resident CTAs per SM there (0 on failure).
template <class K>
int prepare_kernel(K kern, int threads, int smem, PerDeviceOcc *cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(g_attr_mu);
    if (cache->occ[dev] > 0) return cache->occ[dev];
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem) != cudaSuccess) return 0;
    cache->occ[dev] = occ;
    return occ;
}

// A launch that may overlap the previous kernel on the stream (programmatic dependent
// launch); the kernel orders its own reads with griddepcontrol.wait.
template <class K, class... Args>
cudaError_t launch_dependent_smem(K kern, dim3 grid, dim3 block, int smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The same, as thread-block clusters of `cluster_x` CTAs along x.
template <class K, class... Args>
cudaError_t launch_cluster_dependent_smem(K kern, dim3 grid, dim3 block, int smem, int cluster_x,
                                          cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <class K, class... Args>
cudaError_t launch_dependent(K kern, dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The combine of the per-sequence schedule: a warp per row, or a CTA per row when rows have
// more than 16 splits (measured: the warp per row is faster at 9 splits, the CTA per row at
// 38).
template <int D>
cudaError_t launch_combine(const SplitParams &p, int B, int Hq, int S, cudaStream_t stream) {
    if (S > 16) return launch_dependent(combine_wide_kernel<D>, dim3((unsigned)((long long)B * Hq)), dim3(256), stream, p);
    return launch_dependent(combine_kernel<D>, dim3((unsigned)(((long long)B * Hq + 7) / 8)), dim3(256), stream, p);
}

SplitParams make_params(const DecodeArgs &a) {
    SplitParams p = {};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.q_sb = a.q_sb;
    p.q_sh = a.q_sh;
    p.k_cache = static_cast<const __nv_bfloat16 *>(a.k);
    p.v_cache = static_cast<const __nv_bfloat16 *>(a.v);
    p.k_codes = static_cast<const uint8_t *>(a.k);
    p.v_codes = static_cast<const uint8_t *>(a.v);
    p.k_scale = a.k_scale;
    p.v_scale = a.v_scale;
    p.block_table = a.block_table;
    p.max_pages = a.max_pages;
    p.seq_lens = a.seq_lens;
    p.max_kv_len = a.max_kv_len;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.page_size = a.paged ? a.page_size : a.max_len;
    p.num_pages = a.paged ? a.num_pages : a.B;
    p.num_splits = a.num_splits;
    p.chunk = a.chunk;
    p.qscale = a.scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.o_sb = a.o_sb;
    p.o_sh = a.o_sh;
    p.qo_indptr = a.qo_indptr;
    p.tile_batch = a.tile_batch;
    p.tile_index = a.tile_index;
    p.num_tiles = a.num_tiles;
    p.total_q = a.total_q;
    return p;
}

}  // namespace
}  // namespace dap
