// dap_decode.cuh -- bf16 GQA decode attention over a paged (or contiguous) KV cache: the
// kernels and their launch templates, instantiated by dap_decode.cu (TMA-fed tiles) and
// dap_decode_gather.cu (row-gather tiles for page sizes that are not multiples of 8).
//
// Operation (AstrAI "CUDA Kernels" doc, "Python Wrappers": blhd layout, scale
// 1/sqrt(head_dim); AstrAI csrc log, split-KV commit): for sequence b and query head h,
//   out[b,h] = sum_t softmax_t(scale * q[b,h] . K[b,t,h/G]) V[b,t,h/G],   t < seq_lens[b].
//
// Work.  A "unit" is (sequence b, kv head); its keys are cut into tiles of BT tokens (64,
// 32 at D = 256).  Two schedules share one per-tile pipeline:
//   * balanced (num_splits == 0 here; DAP_SPLITS_BALANCED at the interface): a persistent
//     grid of P CTAs (SMs x resident CTAs); the flattened (unit, tile) sequence of all T
//     tiles is cut into P contiguous ranges of T/P tiles, so every CTA streams the same
//     number of tiles whatever the length mix.  A range crosses unit boundaries without
//     draining the pipeline.  A unit covered by one CTA is finished in place; a unit shared
//     by several CTAs gets one partial (acc, m, l) from each (at most two per CTA: the unit
//     its range starts in and the one it ends in), and the combine kernel merges them in
//     CTA order;
//   * per-sequence (num_splits = S > 0): a grid of (unit, split) CTAs, split s owning tokens
//     [s*chunk, (s+1)*chunk) (AstrAI csrc log, split-KV commit: partition KV across
//     gridDim.z blocks that emit unnormalised (O, m, l) partials, reduced by a combine
//     kernel; single-pass direct write when one split suffices).  With 2..8 splits in one
//     wave the splits of a unit form a thread-block cluster and merge in shared memory.
// Either way the summation order depends only on logical positions and the schedule, so
// the output is bit-identical under any permutation of the physical pages.
//
// Data movement.  K and V tiles are staged in shared memory as 128-byte-swizzled column
// blocks (64-byte at D = 32), from the cache viewed as [pages, page_size, Hkv, D]
// (contiguous cache: [B, max_len, Hkv, D], one "page" per sequence).  Page sizes that are
// multiples of 8: 4-D TMA boxes of R = gcd(page_size, BT) tokens of one page; one producer
// warp resolves page ids one tile ahead, arms the stage's mbarrier with the byte count and
// issues the boxes.  Any other page size (csrc log, per-element page lookup commit: any
// page size works): the producer warp looks up every row's page and copies the rows in
// 16-byte cp.async chunks straight into the swizzled layout.  NS stages keep NS-1 tiles in
// flight (csrc log, multi-stage pipeline commit).  Out-of-range page ids are replaced by
// page 0 and flagged.
//
// Arithmetic.  Per 16-key slice a consumer warp computes S^T = K . Q^T with mma.m16n8k16
// (the G heads of the kv head in N), the base-2 online softmax on the fragments, and
// O^T += V^T . P^T with the bf16 probabilities as B operand.  The scale is applied in fp32
// after the dot product (csrc log, "apply scale in float32 after Q@K^T"), V is accumulated
// with fused multiply-adds (numerics commit), rows past the sequence end are masked to
// -inf before the max and kept out of PV, and the final division is guarded (an empty
// sequence gives zeros).
#pragma once

#include <math.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "dap_tile.cuh"

namespace dap {

// Tile header written by the producer into the stage (balanced schedule).
enum : int { H_B = 0, H_KVG = 1, H_TOK0 = 2, H_NVALID = 3, H_FLAGS = 4, H_SLOT = 5 };
enum : int { F_FIRST = 1, F_LAST = 2 };

// ---- tensor-core consumer ---------------------------------------------------------------
// For each 16-key slice a warp computes S^T = K . Q^T with mma.m16n8k16 (M = 16 keys,
// N = 8 query heads of the kv head, padded with zero rows of q when G < 8, K = 16 dims per
// step), runs the base-2 online softmax on the fragments (lane g/t holds keys g, g+8 for
// heads 2t, 2t+1), transposes the bf16 probabilities into the B operand with movmatrix,
// and accumulates O^T = V^T . P^T (M = 16 dims per step, N = 8 heads, K = 16 keys) in
// registers.  Tiles are TMA-loaded with the 128-byte swizzle as [D/64][BT][128 B] so that
// ldmatrix reads are conflict-free (GATHER: page sizes that are not multiples of 8, whose
// rows the producer warp copies into the same layout with cp.async).  The scale multiplies
// S in fp32 (the bf16 q is never rescaled: AstrAI csrc log, "apply scale in float32 after
// Q@K^T").

template <int D_, int G_, int NWC_, int BT_, int NS_, int MINB_, bool GATHER_ = false>
struct MmaCfg {
    static constexpr int D = D_, G = G_, HG = 1, NWC = NWC_, BT = BT_, NS = NS_, MINB = MINB_;
    static constexpr bool GATHER = GATHER_;        // row-gather producer instead of TMA boxes
    static constexpr bool MMA = true;
    static constexpr bool SWZ = true;              // swizzled column blocks, one box each
    static constexpr int WPH = NWC;                // every consumer warp serves the one kv head
    static constexpr int KPW = BT / NWC;           // keys per warp per tile
    static constexpr int ROWB = D * 2;
    static constexpr int HPU = G;
    static constexpr int SWB = D >= 64 ? 128 : 64;  // swizzled column block: 128 B (64 B at D = 32)
    static constexpr int NBLK = ROWB / SWB;         // column blocks per row
    static constexpr int CPB = SWB / 16;            // 16-byte chunks per block row
    static constexpr int TILE_BYTES = BT * ROWB;
    static constexpr int QBYTES = G * ROWB;
    static constexpr int STAGE_BYTES = (2 * TILE_BYTES + QBYTES + 1023) & ~1023;
    static constexpr int MRG_OFF = NS * STAGE_BYTES;
    static constexpr int MRG_BYTES = NWC * G * (D / 2 + 2) * 4;
    static constexpr int HDR_OFF = MRG_OFF + MRG_BYTES;
    static constexpr int HDR_INTS = 8;
    static constexpr int MISC_OFF = HDR_OFF + NS * HDR_INTS * 4;
    static constexpr int BAR_OFF = (MISC_OFF + 16 + 7) & ~7;
    static constexpr int SMEM = BAR_OFF + (2 * NS + 1) * 8 + 1024;  // + slack to align the base
    static constexpr int THREADS = (NWC + 1) * 32;
    static_assert(KPW == 16, "one m16 key slice per warp per tile");
    static_assert(G <= 8, "the query heads of a kv head fill at most N = 8");
    static_assert(D % 32 == 0 && ROWB % SWB == 0, "whole swizzled column blocks");
};

template <class C>
struct MmaConsumer {
    static constexpr int D = C::D, G = C::G, KS = D / 16;
    uint32_t qb[KS][2];  // Q^T B fragments: head g, dims 16k+2t.. and 16k+2t+8..
    float acc[KS][4];    // O^T fragments: dims 16m+g, 16m+g+8 x heads 2t, 2t+1
    float m_run[2], l_run[2];
    float qscale;
    int warp, lane, g, t, key0, rb;  // rb: log2 of the tile's box rows (tile_off)
    static constexpr int hh = 0;

    __device__ __forceinline__ void init(int w, int l, uint8_t *, int box_rows_log2) {
        warp = w;
        lane = l;
        g = l >> 2;
        t = l & 3;
        key0 = w * C::KPW;
        rb = box_rows_log2;
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            m_run[j] = -INFINITY;
            l_run[j] = 0.f;
        }
#pragma unroll
        for (int m = 0; m < KS; ++m)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[m][j] = 0.f;
    }

    __device__ __forceinline__ void load_q(const __nv_bfloat16 *base, long long hstride, float qs) {
        qscale = qs;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            if (g < G) {
                const __nv_bfloat16 *r = base + g * hstride + 16 * k + 2 * t;
                qb[k][0] = *reinterpret_cast<const uint32_t *>(r);
                qb[k][1] = *reinterpret_cast<const uint32_t *>(r + 8);
            } else {
                qb[k][0] = qb[k][1] = 0u;
            }
        }
    }

    // byte offset of (key, dim) in the swizzled tile (tile_off)
    __device__ __forceinline__ uint32_t off(int key, int dim) const { return tile_off<C>(key, dim >> 3, rb); }

    __device__ __forceinline__ void tile(uint8_t *stage, int nvalid) {
        const int nv = nvalid - key0;
        if (nv <= 0) return;  // no key of this slice is valid
        uint8_t *sV = stage + C::TILE_BYTES;
        if (nv < 16) {  // rows past the end may hold anything: zero their V so 0 * V stays 0
            for (int i = lane; i < (16 - nv) * C::NBLK * C::CPB; i += 32) {
                const int row = key0 + nv + i / (C::NBLK * C::CPB);
                *reinterpret_cast<uint4 *>(sV + tile_off<C>(row, i % (C::NBLK * C::CPB), rb)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        const uint32_t kbase = smem_addr(stage), vbase = smem_addr(sV);
        // S^T = K . Q^T
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int key = key0 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int dcol = ((lane >> 4) & 1) * 8;
#pragma unroll
            for (int k = 0; k < KS; ++k) {
                uint32_t a[4];
                ldmatrix_x4(a, kbase + off(key, 16 * k + dcol));
                mma_bf16_16816(c, a, qb[k][0], qb[k][1]);
            }
        }
        // online softmax, base 2; keys g (c0, c1) and g + 8 (c2, c3)
        const bool v0 = g < nv, v1 = g + 8 < nv;
        float s[4];
        s[0] = v0 ? __fmul_rn(c[0], qscale) : -INFINITY;  // (rounded once: the same value feeds max and exp)
        s[1] = v0 ? __fmul_rn(c[1], qscale) : -INFINITY;
        s[2] = v1 ? __fmul_rn(c[2], qscale) : -INFINITY;
        s[3] = v1 ? __fmul_rn(c[3], qscale) : -INFINITY;
        float mx[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xFFFFFFFFu, mx[0], o));
            mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xFFFFFFFFu, mx[1], o));
        }
        float alpha[2], mu[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float m_new = fmaxf(m_run[j], mx[j]);
            mu[j] = (m_new == -INFINITY) ? 0.f : m_new;
            alpha[j] = ex2(m_run[j] - mu[j]);
            m_run[j] = m_new;
        }
        const uint32_t w0 = pack_bf16x2(ex2(s[0] - mu[0]), ex2(s[1] - mu[1]));
        const uint32_t w1 = pack_bf16x2(ex2(s[2] - mu[0]), ex2(s[3] - mu[1]));
        {   // l sums the rounded probabilities PV actually uses
            const float2 p0 = bf16x2_to_float2(w0), p1 = bf16x2_to_float2(w1);
            l_run[0] = l_run[0] * alpha[0] + (p0.x + p1.x);
            l_run[1] = l_run[1] * alpha[1] + (p0.y + p1.y);
        }
#pragma unroll
        for (int m = 0; m < KS; ++m) {
            acc[m][0] *= alpha[0];
            acc[m][1] *= alpha[1];
            acc[m][2] *= alpha[0];
            acc[m][3] *= alpha[1];
        }
        const uint32_t b0 = movmatrix_trans(w0), b1 = movmatrix_trans(w1);
        // O^T += V^T . P^T
        {
            const int key = key0 + (lane & 7) + ((lane >> 4) & 1) * 8;
            const int dcol = ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int m = 0; m < KS; ++m) {
                uint32_t a[4];
                ldmatrix_x4_trans(a, vbase + off(key, 16 * m + dcol));
                mma_bf16_16816(acc[m], a, b0, b1);
            }
        }
    }

    template <class Sync, class Emit>
    __device__ __forceinline__ bool finish(float *mrg, Sync sync, Emit emit) {
        constexpr int NWC = C::NWC, DH = D / 2;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l_run[0] += __shfl_xor_sync(0xFFFFFFFFu, l_run[0], o);
            l_run[1] += __shfl_xor_sync(0xFFFFFFFFu, l_run[1], o);
        }
        float *macc = mrg;                 // [NWC][G][D/2]
        float *mml = mrg + NWC * G * DH;   // [NWC][G][2]
        if (g == 0) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
                if (2 * t + j < G) {
                    mml[(warp * G + 2 * t + j) * 2 + 0] = m_run[j];
                    mml[(warp * G + 2 * t + j) * 2 + 1] = l_run[j];
                }
        }
        const int tid = warp * 32 + lane;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int m = half * KS / 2; m < (half + 1) * KS / 2; ++m) {
                const int d = 16 * m + g - half * DH;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (2 * t + j < G) {
                        float *row = macc + (warp * G + 2 * t + j) * DH;
                        row[d] = acc[m][j];
                        row[d + 8] = acc[m][j + 2];
                    }
                }
            }
            if (!sync()) return false;
            for (int e = tid * 2; e < G * DH; e += NWC * 32 * 2) {
                const int hh2 = e / DH, dd = e % DH;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < NWC; ++w) M = fmaxf(M, mml[(w * G + hh2) * 2]);
                const float Mu = (M == -INFINITY) ? 0.f : M;
                float a0 = 0.f, a1 = 0.f, lv = 0.f;
#pragma unroll
                for (int w = 0; w < NWC; ++w) {
                    const float f = ex2(mml[(w * G + hh2) * 2] - Mu);
                    lv = fmaf(f, mml[(w * G + hh2) * 2 + 1], lv);
                    const float2 x = *reinterpret_cast<const float2 *>(macc + (w * G + hh2) * DH + dd);
                    a0 = fmaf(f, x.x, a0);
                    a1 = fmaf(f, x.y, a1);
                }
                emit(0, hh2, half * DH + dd, a0, a1, M, lv);
            }
            if (!sync()) return false;
        }
        return true;
    }
};

template <class C>
using ConsumerOf = MmaConsumer<C>;

// ---- per-sequence schedule: one CTA per (unit, split) ------------------------------------

// ---- thread-block cluster pieces (the in-cluster merge of a unit's splits) --------------

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of shared-memory location `saddr` of this CTA mapped into CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_u4(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// CLUSTER: the num_splits CTAs of a unit form one thread-block cluster (blockIdx.x = unit *
// num_splits + split = cluster rank); instead of writing partials for a combine kernel,
// every CTA stages its (acc, m, l) in shared memory, ranks 1.. copy theirs into rank 0's
// shared memory, and rank 0 merges them in split order (the combine kernel's arithmetic,
// so the result is the same bit for bit) and writes the output.
template <class C, bool PAGED, bool CLUSTER = false>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
    split_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                 const SplitParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = aligned_smem<C>(smem_raw);
    constexpr int G = C::G, HG = C::HG, NWC = C::NWC, BT = C::BT, NS = C::NS, D = C::D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int nkvg = p.Hkv / HG;
    const int units = p.B * nkvg;
    const int s = CLUSTER ? (int)(blockIdx.x % (unsigned)p.num_splits) : (int)(blockIdx.x / units);
    const int rem = CLUSTER ? (int)(blockIdx.x / (unsigned)p.num_splits) : (int)(blockIdx.x - s * units);
    const int b = rem / nkvg;
    const int kvg = rem - b * nkvg;
    // The pipeline barriers and the tensor maps touch nothing the previous kernel writes:
    // they are set up before the wait below, overlapping that kernel's end.
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + NS;
    int *misc = reinterpret_cast<int *>(smem + C::MISC_OFF);  // [0] tiles issued, [1] abort
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], full_arrivals<C>());
            mbar_init(&empty[i], NWC);
        }
        misc[0] = 0;
        misc[1] = 0;
        fence_barrier_init();
    }
    if (!C::GATHER && warp == NWC && lane == 0) {
        prefetch_tensormap(&mapK);
        prefetch_tensormap(&mapV);
    }
    // Launched as a programmatic dependent: the CTA may be resident before the previous
    // kernel on the stream has finished, so nothing that kernel may write is read before
    // this wait; the combine that follows may be launched as soon as every CTA is here.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the sequence length and the producer's page ids of the first tile are loaded together
    // (table entries from position s * chunk on; those past the sequence's end are read
    // within the table but not used)
    int L = p.seq_lens[b];
    const int R = PAGED ? p.box_rows : BT;
    int pg_first = 0;
    if (PAGED && !C::GATHER && warp == NWC && lane * R < BT) {
        const long long t = (long long)s * p.chunk + lane * R;
        if (t < (long long)p.max_pages * p.page_size)
            pg_first = __ldg(p.block_table + (long long)b * p.max_pages + t / p.page_size);
    }
    if (L < 0 || L > p.max_kv_len) {
        if (threadIdx.x == 0 && s == 0 && kvg == 0) flag_error(DAP_DEVERR_SEQLEN);
        L = min(max(L, 0), p.max_kv_len);
    }
    const int nsplit = max(1, (L + p.chunk - 1) / p.chunk);
    if (!CLUSTER && s >= nsplit) return;  // (in a cluster every CTA takes part in the merge)
    const int tok0 = s * p.chunk;
    const int tok1 = min(L, tok0 + p.chunk);
    const int ntiles = tok1 > tok0 ? (tok1 - tok0 + BT - 1) / BT : 0;
    __syncthreads();

    if (C::GATHER && warp == NWC) {  // ---- producer warp, row gather: page lookup + cp.async
        const int32_t *table = p.block_table + (long long)b * p.max_pages;
        RowPages<C> rp_next;
        if (ntiles > 0) lookup_rows<C>(rp_next, table, tok0, min(BT, tok1 - tok0), p.page_size, lane);
        int issued = 0;
        for (int i = 0; i < ntiles; ++i) {
            const int st = i % NS;
            const RowPages<C> rp = rp_next;
            const int t = tok0 + i * BT;
            if (i + 1 < ntiles) lookup_rows<C>(rp_next, table, t + BT, min(BT, tok1 - t - BT), p.page_size, lane);
            if (i >= NS && !__all_sync(0xFFFFFFFFu, mbar_wait(&empty[st], ((i / NS) - 1) & 1))) {
                misc[1] = 1;
                break;
            }
            fill_tile_rows<C>(smem + st * C::STAGE_BYTES, rp, min(BT, tok1 - t), kvg * HG, p, 0u, [] {}, &full[st],
                              lane);
            issued = i + 1;
        }
        if (lane == 0) misc[0] = issued;
        __syncthreads();  // pairs with the consumers' final __syncthreads
        return;
    }
    if (warp == NWC) {  // ---- producer warp: page lookup + TMA issue
        const int32_t *table = PAGED ? p.block_table + (long long)b * p.max_pages : nullptr;
        auto lookup = [&](int tile) -> int {  // page id of this lane's box of `tile`
            if (!PAGED) return b;
            const int t = tok0 + tile * BT + lane * R;
            if (lane * R >= BT || t >= tok1) return 0;
            int pg = tile == 0 ? pg_first : __ldg(table + t / p.page_size);
            if (pg < 0 || pg >= p.num_pages) {
                flag_error(DAP_DEVERR_PAGE);
                pg = 0;
            }
            return pg;
        };
        int pg_next = ntiles > 0 ? lookup(0) : 0;
        int issued = 0;
        for (int i = 0; i < ntiles; ++i) {
            const int st = i % NS;
            const int pg = pg_next;
            if (i + 1 < ntiles) pg_next = lookup(i + 1);
            if (i >= NS && !__all_sync(0xFFFFFFFFu, mbar_wait(&empty[st], ((i / NS) - 1) & 1))) {
                misc[1] = 1;
                break;
            }
            const int t = tok0 + i * BT;
            const int nvalid = min(BT, tok1 - t);
            const int nbox = PAGED ? (nvalid + R - 1) / R : 1;
            const uint32_t bytes = (uint32_t)(nbox * R * HG * C::ROWB * 2);
            if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes);
            __syncwarp();
            if (lane < nbox) {
                const int tt = t + lane * R;
                issue_kv_box<C>(smem + st * C::STAGE_BYTES, lane, R, &mapK, &mapV, kvg * HG,
                                PAGED ? tt % p.page_size : tt, pg, &full[st]);
            }
            issued = i + 1;
        }
        if (lane == 0) misc[0] = issued;
        __syncthreads();  // pairs with the consumers' final __syncthreads
        return;
    }

    // ---- consumer warps
    ConsumerOf<C> cs;
    cs.init(warp, lane, smem, 31 - __clz(PAGED && !C::GATHER ? R : BT));
    cs.reset();
    const int kvh = kvg * HG + cs.hh;
    cs.load_q(p.q + (long long)b * p.q_sb + (long long)kvh * G * p.q_sh, p.q_sh, p.qscale);
    int consumed = 0;
    for (int i = 0; i < ntiles; ++i) {
        const int st = i % NS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[st], (i / NS) & 1))) {
            misc[1] = 1;
            break;
        }
        cs.tile(smem + st * C::STAGE_BYTES, min(BT, tok1 - (tok0 + i * BT)));
        if (lane == 0) mbar_arrive(&empty[st]);
        consumed = i + 1;
    }
    __syncthreads();  // every consumer is done; the producer has finished issuing
    if (misc[1]) {    // a wait timed out: drain the copies still in flight (bounded), write nothing
        if (threadIdx.x == 0)
            for (int i = consumed; i < misc[0]; ++i) (void)mbar_wait(&full[i % NS], (i / NS) & 1);
        if constexpr (!CLUSTER) return;
        cs.reset();  // (in a cluster: take part in the merge with an empty partial)
    }
    if constexpr (CLUSTER) {
        // stage this CTA's (acc, m, l) at the start of its (now idle) stage ring: [G][D] acc,
        // then [G] (m, l); ranks 1.. copy theirs into rank 0's ring at slot `rank`
        constexpr int SLOT = (G * (D + 2) + 3) & ~3;  // floats, a whole number of 16-byte chunks
        static_assert(C::HG == 1 && (SLOT * 4) % 16 == 0, "one kv head per CTA; 16-byte slots");
        static_assert(8 * SLOT * 4 <= C::NS * C::STAGE_BYTES, "eight slots fit the stage ring");
        float *stg = reinterpret_cast<float *>(smem);
        cs.finish(reinterpret_cast<float *>(smem + C::MRG_OFF),
                  [] { named_sync(1, NWC * 32); return true; },
                  [&](int, int g, int d, float a0, float a1, float M, float lv) {
                      *reinterpret_cast<float2 *>(stg + g * D + d) = make_float2(a0, a1);
                      if (d == 0) *reinterpret_cast<float2 *>(stg + G * D + g * 2) = make_float2(M, lv);
                  });
        cluster_sync_all();  // every CTA of the cluster has staged its partial and is done with its ring
        const int tid = threadIdx.x;
        if (s != 0) {
            const uint32_t dst = cluster_map(smem_addr(stg + s * SLOT), 0);
            for (int i = tid; i < SLOT / 4; i += NWC * 32)
                st_cluster_u4(dst + i * 16, *reinterpret_cast<const uint4 *>(stg + 4 * i));
        }
        cluster_sync_all();  // rank 0 holds every partial
        if (s == 0) {
            for (int e = tid * 2; e < G * D; e += NWC * 32 * 2) {
                const int g = e / D, d = e - g * D;
                float M = -INFINITY;
                for (int k = 0; k < p.num_splits; ++k) M = fmaxf(M, stg[k * SLOT + G * D + g * 2]);
                const float Mu = (M == -INFINITY) ? 0.f : M;
                float a0 = 0.f, a1 = 0.f, lsum = 0.f;
                for (int k = 0; k < p.num_splits; ++k) {
                    const float *sl = stg + k * SLOT;
                    const float f = ex2(sl[G * D + g * 2] - Mu);
                    lsum = fmaf(f, sl[G * D + g * 2 + 1], lsum);
                    const float2 x = *reinterpret_cast<const float2 *>(sl + g * D + d);
                    a0 = fmaf(f, x.x, a0);
                    a1 = fmaf(f, x.y, a1);
                }
                const int hq = kvg * G + g;
                store_out_pair(p.out + (long long)b * p.o_sb + (long long)hq * p.o_sh + d, a0, a1, lsum);
            }
        }
        return;
    }
    const bool direct = (nsplit == 1);
    cs.finish(reinterpret_cast<float *>(smem + C::MRG_OFF),
              [] { named_sync(1, NWC * 32); return true; },
              [&](int hl, int g, int d, float a0, float a1, float M, float lv) {
                  const int hq = (kvg * HG + hl) * G + g;
                  if (direct) {
                      store_out_pair(p.out + (long long)b * p.o_sb + (long long)hq * p.o_sh + d, a0, a1, lv);
                  } else {
                      const long long row = ((long long)b * p.num_splits + s) * p.Hq + hq;
                      *reinterpret_cast<float2 *>(p.o_part + row * D + d) = make_float2(a0, a1);
                      if (d == 0) *reinterpret_cast<float2 *>(p.ml_part + row * 2) = make_float2(M, lv);
                  }
              });
}

// ---- balanced schedule: persistent CTAs over equal ranges of the flattened tile space ---

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

template <class C, bool PAGED>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
    balanced_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                    const __grid_constant__ CUtensorMap mapQ, const SplitParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = aligned_smem<C>(smem_raw);
    constexpr int G = C::G, HG = C::HG, NWC = C::NWC, BT = C::BT, NS = C::NS, D = C::D, HPU = C::HPU;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int P = p.num_ctas;
    const int nkvg = p.Hkv / HG;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + NS;
    uint64_t *cbar = empty + NS;
    volatile int *misc = reinterpret_cast<volatile int *>(smem + C::MISC_OFF);  // tiles, abort, issued
    int *hdr_all = reinterpret_cast<int *>(smem + C::HDR_OFF);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], full_arrivals<C>());
            mbar_init(&empty[i], NWC);
        }
        mbar_init(cbar, NWC);
        misc[0] = 0;
        misc[1] = 0;
        fence_barrier_init();
    }
    // the combine grid may start launching now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    // tiles of a sequence (an empty sequence still takes one tile, which writes its zeros)
    auto seq_len = [&](int b) -> int {
        int L = __ldg(p.seq_lens + b);
        if (L < 0 || L > p.max_kv_len) {
            flag_error(DAP_DEVERR_SEQLEN);
            L = min(max(L, 0), p.max_kv_len);
        }
        return L;
    };
    auto tiles_of = [](int L) { return max(1, (L + BT - 1) / BT); };

    long long s_c = 0;
    if (warp == NWC) {
        long long total = 0;
        for (int base = 0; base < p.B; base += 32) {
            const int b = base + lane;
            int tb = b < p.B ? tiles_of(seq_len(b)) : 0;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) tb += __shfl_xor_sync(0xFFFFFFFFu, tb, o);
            total += tb;
        }
        const long long T = total * nkvg;
        s_c = (long long)c * T / P;
        const long long e_c = (long long)(c + 1) * T / P;
        if (lane == 0) {
            misc[0] = (int)(e_c - s_c);
            if (c == 0) *p.total_tiles = T;
        }
    }
    __syncthreads();
    const int ntiles = misc[0];

    if (warp == NWC) {  // ---- producer warp
        if (lane == 0) {
            if (!C::GATHER) {
                prefetch_tensormap(&mapK);
                prefetch_tensormap(&mapV);
            }
            prefetch_tensormap(&mapQ);
        }
        int issued = 0;
        if (ntiles > 0) {
            // locate the unit holding tile s_c
            long long before = 0;
            int b = -1, tb = 1;
            for (int base = 0; base < p.B && b < 0; base += 32) {
                const int bb = base + lane;
                const int t1 = bb < p.B ? tiles_of(seq_len(bb)) : 0;
                const int w = t1 * nkvg;
                const int incl = warp_incl_scan(w, lane);
                const unsigned hit = __ballot_sync(0xFFFFFFFFu, bb < p.B && before + incl > s_c);
                if (hit) {
                    const int f = __ffs(hit) - 1;
                    b = base + f;
                    tb = __shfl_sync(0xFFFFFFFFu, t1, f);
                    before += __shfl_sync(0xFFFFFFFFu, incl - w, f);
                } else {
                    before += __shfl_sync(0xFFFFFFFFu, incl, 31);
                }
            }
            const long long rem = s_c - before;
            int kvg = (int)(rem / tb);
            int j = (int)(rem % tb);
            int L = seq_len(b);
            bool in_u0 = true;  // the cursor is still in the unit the range starts in
            int seg_j0 = j;
            const int R = PAGED ? p.box_rows : BT;

            auto lookup_box = [&](int bb, int tt, int LL) -> int {  // page of the box at token tt
                if (!PAGED) return bb;
                if (tt >= LL) return 0;
                int pg = __ldg(p.block_table + (long long)bb * p.max_pages + tt / p.page_size);
                if (pg < 0 || pg >= p.num_pages) {
                    flag_error(DAP_DEVERR_PAGE);
                    pg = 0;
                }
                return pg;
            };
            auto lookup = [&](int bb, int jj, int LL) -> int {  // page of this lane's box
                if (lane * R >= BT) return 0;
                return lookup_box(bb, jj * BT + lane * R, LL);
            };
            // row-gather mode: this lane's rows of the next tile
            auto lookup_tile = [&](RowPages<C> &rp, int bb, int jj, int LL) {
                lookup_rows<C>(rp, p.block_table + (long long)bb * p.max_pages, jj * BT,
                               max(0, min(BT, LL - jj * BT)), p.page_size, lane);
            };
            RowPages<C> rp_next;
            int pg_next = 0;
            if constexpr (C::GATHER) lookup_tile(rp_next, b, j, L);
            else pg_next = lookup(b, j, L);
            for (int i = 0; i < ntiles; ++i) {
                const int st = i % NS;
                const int pg = pg_next;
                const RowPages<C> rp = rp_next;
                // cursor of the next tile
                int nb = b, nk = kvg, nj = j + 1, nL = L, ntb = tb;
                bool n_in_u0 = in_u0;
                if (nj == tb) {
                    nj = 0;
                    n_in_u0 = false;
                    if (++nk == nkvg) {
                        nk = 0;
                        ++nb;
                        nL = (nb < p.B && i + 1 < ntiles) ? seq_len(nb) : 0;
                        ntb = tiles_of(nL);
                    }
                }
                if (i + 1 < ntiles) {
                    if constexpr (C::GATHER) lookup_tile(rp_next, nb, nj, nL);
                    else pg_next = lookup(nb, nj, nL);
                }
                if (i >= NS && !__all_sync(0xFFFFFFFFu, mbar_wait(&empty[st], ((i / NS) - 1) & 1))) {
                    misc[1] = 1;
                    break;
                }
                const bool first = (i == 0) || (j == 0);
                const bool last = (i == ntiles - 1) || (j == tb - 1);
                if (first) seg_j0 = j;
                const int nvalid = max(0, min(BT, L - j * BT));
                const int slot = (seg_j0 == 0 && j == tb - 1) ? -1 : 2 * c + (in_u0 ? 0 : 1);
                const bool need_q = first && nvalid > 0;
                const int nbox = PAGED ? (nvalid + R - 1) / R : (nvalid > 0 ? 1 : 0);
                const uint32_t bytes = (uint32_t)(nbox * R * HG * C::ROWB * 2 + (need_q ? C::QBYTES : 0));
                uint8_t *stage = smem + st * C::STAGE_BYTES;
                if (lane == 0) {
                    int *h = hdr_all + st * C::HDR_INTS;
                    h[H_B] = b;
                    h[H_KVG] = kvg;
                    h[H_TOK0] = j * BT;
                    h[H_NVALID] = nvalid;
                    h[H_FLAGS] = (first ? F_FIRST : 0) | (last ? F_LAST : 0);
                    h[H_SLOT] = slot;
                    if (j == 0) {  // this CTA holds the unit's first tile: record where it starts
                        p.unit_info[2 * (b * nkvg + kvg)] = (int)(s_c + i);
                        p.unit_info[2 * (b * nkvg + kvg) + 1] = tb;
                    }
                    if (!C::GATHER) mbar_arrive_expect_tx(&full[st], bytes);
                }
                if constexpr (C::GATHER) {
                    fill_tile_rows<C>(stage, rp, nvalid, kvg * HG, p, need_q ? (uint32_t)C::QBYTES : 0u,
                                      [&] {
                                          if (need_q)
                                              tma_load_3d(stage + 2 * C::TILE_BYTES, &mapQ, 0, kvg * HPU, b, &full[st]);
                                      },
                                      &full[st], lane);
                    b = nb;
                    kvg = nk;
                    j = nj;
                    L = nL;
                    tb = ntb;
                    in_u0 = n_in_u0;
                    issued = i + 1;
                    continue;
                }
                __syncwarp();
                for (int jb = lane; jb < nbox; jb += 32) {
                    const int tt = j * BT + jb * R;
                    const int pgb = jb == lane ? pg : lookup_box(b, tt, L);
                    issue_kv_box<C>(stage, jb, R, &mapK, &mapV, kvg * HG, PAGED ? tt % p.page_size : tt, pgb,
                                    &full[st]);
                }
                if (need_q && lane == 0)
                    tma_load_3d(stage + 2 * C::TILE_BYTES, &mapQ, 0, kvg * HPU, b, &full[st]);
                b = nb;
                kvg = nk;
                j = nj;
                L = nL;
                tb = ntb;
                in_u0 = n_in_u0;
                issued = i + 1;
            }
        }
        if (lane == 0) misc[2] = issued;
        __syncthreads();  // pairs with the consumers' final __syncthreads
        return;
    }

    // ---- consumer warps
    ConsumerOf<C> cs;
    cs.init(warp, lane, smem, 31 - __clz(PAGED && !C::GATHER ? p.box_rows : BT));
    cs.reset();
    float *mrg = reinterpret_cast<float *>(smem + C::MRG_OFF);
    ConsumerBarrier cb{cbar, 0u};
    int consumed = 0;
    for (int i = 0; i < ntiles; ++i) {
        const int st = i % NS;
        if (__any_sync(0xFFFFFFFFu, misc[1] != 0)) break;  // another warp gave up
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[st], (i / NS) & 1))) {
            misc[1] = 1;
            break;
        }
        const uint8_t *stage = smem + st * C::STAGE_BYTES;
        const int *h = hdr_all + st * C::HDR_INTS;
        const int b = h[H_B], kvg = h[H_KVG], nvalid = h[H_NVALID], flags = h[H_FLAGS], slot = h[H_SLOT];
        if (flags & F_FIRST) {
            cs.reset();
            if (nvalid > 0)
                cs.load_q(reinterpret_cast<const __nv_bfloat16 *>(stage + 2 * C::TILE_BYTES) + cs.hh * G * D, D,
                          p.qscale);
        }
        cs.tile(const_cast<uint8_t *>(stage), nvalid);
        if (lane == 0) mbar_arrive(&empty[st]);
        consumed = i + 1;
        if (flags & F_LAST) {
            const bool ok = cs.finish(mrg, [&] { return cb.sync(lane); },
                                      [&](int hl, int g, int d, float a0, float a1, float M, float lv) {
                                          const int hl2 = hl * G + g;
                                          if (slot < 0) {
                                              const int hq = kvg * HPU + hl2;
                                              store_out_pair(p.out + (long long)b * p.o_sb + (long long)hq * p.o_sh + d,
                                                             a0, a1, lv);
                                          } else {
                                              const long long row = (long long)slot * HPU + hl2;
                                              *reinterpret_cast<float2 *>(p.o_part + row * D + d) = make_float2(a0, a1);
                                              if (d == 0)
                                                  *reinterpret_cast<float2 *>(p.ml_part + row * 2) = make_float2(M, lv);
                                          }
                                      });
            if (!ok) {
                misc[1] = 1;
                break;
            }
        }
    }
    __syncthreads();
    if (misc[1] && threadIdx.x == 0) {  // a wait gave up: let the copies in flight land (bounded)
        const int issued = misc[2];
        for (int i = consumed; i < issued; ++i) (void)mbar_wait(&full[i % NS], (i / NS) & 1);
    }
}

// ---- combine kernels -------------------------------------------------------------------
// Merge the partials of every output row that more than one CTA worked on, in a fixed
// order: M = max_s m_s, out = sum_s 2^(m_s-M) acc_s / sum_s 2^(m_s-M) l_s (AstrAI csrc log,
// split-KV commit: the combine kernel; numerics commit: guarded division).  One warp per
// output row, lanes over D.  Both wait for the split grid (programmatic dependent launch).


// Balanced schedule: one CTA per output row.  Its threads resolve, in parallel, which
// partial slot every CTA of the unit's range wrote (none for CTAs with an empty range) and
// the row maximum; the four warps then split the partial-row loads, and the per-warp sums
// are added through shared memory.
template <int D>
__global__ void __launch_bounds__(128) combine_balanced_kernel(const SplitParams p, int hpu, int nkvg) {
    constexpr int DPV = D / 32;
    __shared__ int slots[kMaxPersistentCtas];
    __shared__ float wts[kMaxPersistentCtas];
    __shared__ float red[4][D + 2];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = blockIdx.x;
    const int u = row / hpu, hl2 = row - u * hpu;
    const long long start = p.unit_info[2 * u], tb = p.unit_info[2 * u + 1];
    const long long T = *p.total_tiles;
    const long long P = p.num_ctas;
    const int c_first = (int)(((start + 1) * P - 1) / T);
    const int c_last = (int)(((start + tb) * P - 1) / T);
    if (c_first == c_last) return;  // finished in place by one CTA
    const int n = c_last - c_first + 1;
    float M = -INFINITY;
    for (int i = tid; i < n; i += 128) {
        const int c = c_first + i;
        const long long s_c = (long long)c * T / P, e_c = (long long)(c + 1) * T / P;
        const int sl = (s_c == e_c) ? -1 : 2 * c + ((c == c_first && s_c < start) ? 1 : 0);
        slots[i] = sl;
        const float m = sl >= 0 ? p.ml_part[((long long)sl * hpu + hl2) * 2] : -INFINITY;
        wts[i] = m;
        M = fmaxf(M, m);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    if (lane == 0) red[warp][D] = M;
    __syncthreads();
    M = fmaxf(fmaxf(red[0][D], red[1][D]), fmaxf(red[2][D], red[3][D]));
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float lsum = 0.f;
    for (int i = tid; i < n; i += 128) {
        const int sl = slots[i];
        float f = 0.f;
        if (sl >= 0) {
            f = ex2(wts[i] - Mu);
            lsum = fmaf(f, p.ml_part[((long long)sl * hpu + hl2) * 2 + 1], lsum);
        }
        wts[i] = f;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, o);
    __syncthreads();  // wts complete; red[.][D] read by everyone
    if (lane == 0) red[warp][D + 1] = lsum;
    float acc[DPV];
#pragma unroll
    for (int j = 0; j < DPV; ++j) acc[j] = 0.f;
    for (int i0 = warp; i0 < n; i0 += 4 * 8) {
        float x[8][DPV];
        float f[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = i0 + 4 * k;
            const int sl = i < n ? slots[i] : -1;
            f[k] = sl >= 0 ? wts[i] : 0.f;
            if (sl >= 0) {
                const float *o = p.o_part + ((long long)sl * hpu + hl2) * D + lane * DPV;
#pragma unroll
                for (int j = 0; j < DPV; ++j) x[k][j] = o[j];
            } else {
#pragma unroll
                for (int j = 0; j < DPV; ++j) x[k][j] = 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
#pragma unroll
            for (int j = 0; j < DPV; ++j) acc[j] = fmaf(f[k], x[k][j], acc[j]);
    }
#pragma unroll
    for (int j = 0; j < DPV; ++j) red[warp][lane * DPV + j] = acc[j];
    __syncthreads();
    if (warp == 0) {
        const float L = red[0][D + 1] + red[1][D + 1] + red[2][D + 1] + red[3][D + 1];
        float a[DPV];
#pragma unroll
        for (int j = 0; j < DPV; ++j)
            a[j] = red[0][lane * DPV + j] + red[1][lane * DPV + j] + red[2][lane * DPV + j] + red[3][lane * DPV + j];
        const int b = u / nkvg, kvg = u - b * nkvg;
        __nv_bfloat16 *o = p.out + (long long)b * p.o_sb + (long long)(kvg * hpu + hl2) * p.o_sh + lane * DPV;
        store_row_part<DPV>(o, a, L);
    }
}

// ---- host side ----------------------------------------------------------------------------

namespace {

// K / V tensor maps with boxes of R rows (none in row-gather mode, which reads the cache
// directly).
template <class C>
bool encode_maps(const DecodeArgs &a, long long rows, long long outer, int R, CUtensorMap *mk, CUtensorMap *mv) {
    if (C::GATHER) return true;
    return encode_cache_map<C>(mk, a.k, a.D, a.Hkv, rows, outer, R) &&
           encode_cache_map<C>(mv, a.v, a.D, a.Hkv, rows, outer, R);
}

template <class C, bool PAGED>
dap_status launch_per_sequence(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    const int R = PAGED ? gcd_int(a.page_size, C::BT) : C::BT;
    p.box_rows = R;
    CUtensorMap mk = {}, mv = {};
    const long long rows = PAGED ? a.page_size : a.max_len;
    const long long outer = PAGED ? a.num_pages : a.B;
    if (!encode_maps<C>(a, rows, outer, R, &mk, &mv)) return DAP_ERR_CUDA;
    auto kern = split_kernel<C, PAGED, false>;
    auto kern_cl = split_kernel<C, PAGED, true>;
    static PerDeviceOcc occ = {}, occ_cl = {};
    const int per_sm = prepare_kernel(kern, C::THREADS, C::SMEM, &occ);
    if (per_sm <= 0 || prepare_kernel(kern_cl, C::THREADS, C::SMEM, &occ_cl) <= 0) return DAP_ERR_CUDA;
    const long long grid = (long long)a.B * (a.Hkv / C::HG) * a.num_splits;
    if (grid > 0x7FFFFFFFLL) return DAP_ERR_SHAPE;
    // A unit's splits merge inside a thread-block cluster (no combine kernel, no partials in
    // the workspace) when there are 2..8 of them and the grid is one wave: every cluster is
    // then resident from the start.
    const int sms = dap_device_sm_count();
    const bool cluster = a.num_splits >= 2 && a.num_splits <= 8 && sms > 0 && grid <= (long long)sms * per_sm;
    p.o_part = static_cast<float *>(a.workspace);
    p.ml_part = a.num_splits > 1 ? reinterpret_cast<float *>(static_cast<char *>(a.workspace) +
                                                             partial_acc_bytes(a.B, a.Hq, a.D, a.num_splits))
                                 : nullptr;
    if (g_trace.split_begin) cudaEventRecord(g_trace.split_begin, stream);
    const cudaError_t e =
        cluster ? launch_cluster_dependent_smem(kern_cl, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM,
                                                a.num_splits, stream, mk, mv, p)
                : launch_dependent_smem(kern, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM, stream, mk, mv, p);
    if (e != cudaSuccess) return DAP_ERR_CUDA;
    if (g_trace.split_end) cudaEventRecord(g_trace.split_end, stream);
    if (a.num_splits > 1 && !cluster) {
        if (launch_combine<C::D>(p, a.B, a.Hq, a.num_splits, stream) != cudaSuccess) return DAP_ERR_CUDA;
    }
    if (g_trace.combine_end) cudaEventRecord(g_trace.combine_end, stream);
    return DAP_OK;
}

template <class C, bool PAGED>
dap_status launch_balanced(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    const int R = PAGED ? gcd_int(a.page_size, C::BT) : C::BT;
    p.box_rows = R;
    CUtensorMap mk = {}, mv = {}, mq;
    const long long rows = PAGED ? a.page_size : a.max_len;
    const long long outer = PAGED ? a.num_pages : a.B;
    if (!encode_q_map(&mq, a, C::HPU) || !encode_maps<C>(a, rows, outer, R, &mk, &mv)) return DAP_ERR_CUDA;
    auto kern = balanced_kernel<C, PAGED>;
    static PerDeviceOcc occ = {};
    const int per_sm = prepare_kernel(kern, C::THREADS, C::SMEM, &occ);
    const int sms = dap_device_sm_count();
    if (per_sm <= 0 || sms <= 0) return DAP_ERR_CUDA;
    const int nkvg = a.Hkv / C::HG;
    // no more CTAs than the tiles there can be (each sequence takes at least one tile)
    const long long max_tiles =
        (long long)a.B * nkvg * std::max<long long>(1, (a.max_kv_len + C::BT - 1) / C::BT);
    const int P = (int)std::min<long long>(std::min(sms * per_sm, kMaxPersistentCtas), max_tiles);
    const BalancedLayout lay = balanced_layout(a.B, nkvg, C::HPU, a.D);
    char *ws = static_cast<char *>(a.workspace);
    p.o_part = reinterpret_cast<float *>(ws + lay.acc);
    p.ml_part = reinterpret_cast<float *>(ws + lay.ml);
    p.unit_info = reinterpret_cast<int *>(ws + lay.info);
    p.total_tiles = reinterpret_cast<long long *>(ws + lay.total);
    p.num_ctas = P;
    if (g_trace.split_begin) cudaEventRecord(g_trace.split_begin, stream);
    kern<<<P, C::THREADS, C::SMEM, stream>>>(mk, mv, mq, p);
    if (cudaGetLastError() != cudaSuccess) return DAP_ERR_CUDA;
    if (g_trace.split_end) cudaEventRecord(g_trace.split_end, stream);
    const dim3 cgrid((unsigned)(a.B * nkvg * C::HPU));
    const cudaError_t e =
        launch_dependent(combine_balanced_kernel<C::D>, cgrid, dim3(128), stream, p, (int)C::HPU, nkvg);
    if (e != cudaSuccess) return DAP_ERR_CUDA;
    if (g_trace.combine_end) cudaEventRecord(g_trace.combine_end, stream);
    return DAP_OK;
}

// Configurations: one kv head per CTA, four consumer warps of 16 keys each, 64-token tiles
// in 128-byte-swizzled column blocks, three stages, two CTAs per SM.  D = 256: 32-token
// tiles and two consumer warps keep a stage near 34 KB (two CTAs per SM); D = 32: six
// stages of 8 KB at three CTAs per SM.  The row-gather configurations (page sizes that are
// not multiples of 8, whose boxes of fewer than 8 rows could not start on the 1024-byte
// boundaries the swizzle needs) keep the same tiles.
template <int D, int G>
using MmaCfgFor = typename std::conditional<
    D == 256, MmaCfg<256, G, 2, 32, 3, 2>,
    typename std::conditional<D == 32, MmaCfg<32, G, 4, 64, 6, 3>, MmaCfg<D, G, 4, 64, 3, 2>>::type>::type;
// The same tensor-core tiles filled by the row-gather producer.
template <int D, int G>
using GatherCfgFor = typename std::conditional<
    D == 256, MmaCfg<256, G, 2, 32, 3, 2, true>,
    typename std::conditional<D == 32, MmaCfg<32, G, 4, 64, 6, 3, true>, MmaCfg<D, G, 4, 64, 3, 2, true>>::type>::type;

template <class C>
dap_status run(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    if constexpr (C::GATHER) {  // paged only
        return a.num_splits == 0 ? launch_balanced<C, true>(a, p, stream) : launch_per_sequence<C, true>(a, p, stream);
    } else {
        if (a.num_splits == 0)
            return a.paged ? launch_balanced<C, true>(a, p, stream) : launch_balanced<C, false>(a, p, stream);
        return a.paged ? launch_per_sequence<C, true>(a, p, stream) : launch_per_sequence<C, false>(a, p, stream);
    }
}

}  // namespace
}  // namespace dap
