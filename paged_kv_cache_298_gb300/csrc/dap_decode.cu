// dap_decode.cu -- bf16 GQA decode attention over a paged (or contiguous) KV cache.
//
// Operation (AstrAI "CUDA Kernels" doc, "Python Wrappers": blhd layout, scale
// 1/sqrt(head_dim); AstrAI csrc log, split-KV commit): for sequence b and query head h,
//   out[b,h] = sum_t softmax_t(scale * q[b,h] . K[b,t,h/G]) V[b,t,h/G],   t < seq_lens[b].
//
// Work decomposition.  A CTA owns one work unit (sequence b, group of HG kv heads,
// split s): the tokens [s*chunk, min(L_b, (s+1)*chunk)).  A sequence whose length fits one
// chunk is finished in place (normalised bf16 row); otherwise the CTA writes an
// unnormalised partial (acc, m, l) and the combine kernel merges the splits in split
// order (csrc log, split-KV commit: "(O, m, l) partials, reduced by a combine kernel";
// "single-pass direct-write" when one split suffices).  Units are numbered split-major,
// so every sequence's first chunk is scheduled before any second chunk.
//
// Data movement.  K and V tiles of kTileTokens tokens are staged in shared memory by
// 4-D TMA boxes over the cache viewed as [pages, page_size, Hkv, D] (contiguous cache:
// [B, max_len, Hkv, D], one "page" per sequence).  A box covers R = gcd(page_size, 32)
// tokens of one page, so any page size works and every page-table entry is read once
// per box (csrc log, per-element page lookup commit: "works for any page_size").  One
// producer warp resolves the page ids (prefetched one tile ahead), arms the stage's
// mbarrier with the byte count and issues the boxes; NS stages keep NS-1 tiles in flight
// (csrc log, multi-stage pipeline commit).  Out-of-range page ids are replaced by page 0
// and flagged, so no access leaves the pool.
//
// Arithmetic.  q is held in fp32 registers, pre-multiplied by scale*log2(e) in fp32 (the
// bf16 q is never rescaled: csrc log, "apply scale in float32 after Q@K^T").  QK^T uses
// packed fp32 FMAs (FFMA2) with LPR lanes per key row and a reduce-scatter across them;
// the online softmax runs in base 2; PV accumulates with FFMA2 (fused multiply-add, csrc
// log numerics commit: fmaf for V accumulation).  Rows past the sequence end are masked
// to -inf before the max and never read in PV, so stale or poisoned shared memory cannot
// leak into the result.  The summation order depends only on logical positions: the
// output is bit-identical under any permutation of the physical pages.
#include <math.h>

#include <algorithm>

#include "dap_device.cuh"
#include "dap_internal.h"

namespace dap {

struct SplitParams {
    const __nv_bfloat16 *q;
    long long q_sb, q_sh;
    const int32_t *block_table;
    int max_pages;
    const int32_t *seq_lens;
    int max_kv_len;
    int B, Hq, Hkv;
    int page_size, num_pages, box_rows;
    int num_splits, chunk;
    float qscale;  // scale * log2(e)
    float *o_part;
    float *ml_part;
    __nv_bfloat16 *out;
    long long o_sb, o_sh;
};

template <int D_, int G_, int HG_, int NWC_, int BT_, int NS_, int MINB_>
struct SplitCfg {
    static constexpr int D = D_, G = G_, HG = HG_, NWC = NWC_, BT = BT_, NS = NS_;
    static constexpr int MINB = MINB_;  // CTAs per SM the register budget must allow
    static constexpr int WPH = NWC / HG;        // warps per kv head
    static constexpr int RW = BT / WPH;         // tile rows per warp
    static constexpr int DPL = (G <= 4) ? 16 : 8;  // QK dims per lane
    static constexpr int CPL = DPL / 8;         // 16-byte chunks per lane
    static constexpr int LPR = D / DPL;         // lanes per key row in QK
    static constexpr int RPP = 32 / LPR;        // key rows per QK pass
    static constexpr int PASSES = RW / RPP;
    static constexpr int DPV = D / 32;          // PV dims per lane
    static constexpr int ROWB = D * 2;          // bytes of one (token, kv head) row
    static constexpr int TILE_BYTES = BT * HG * ROWB;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int PBUF_OFF = NS * STAGE_BYTES;
    static constexpr int PBUF_BYTES = NWC * RW * G * 4;
    static constexpr int ABUF_OFF = PBUF_OFF + PBUF_BYTES;
    static constexpr int ABUF_BYTES = NWC * G * 4;
    static constexpr int MISC_OFF = ABUF_OFF + ABUF_BYTES;  // issued-tile count, abort flag
    static constexpr int BAR_OFF = (MISC_OFF + 8 + 7) & ~7;
    static constexpr int SMEM = BAR_OFF + 2 * NS * 8;
    static constexpr int THREADS = (NWC + 1) * 32;
    static_assert(NWC % HG == 0, "warps must split evenly over the kv heads of a CTA");
    static_assert(BT % WPH == 0 && RW % RPP == 0 && PASSES >= 1, "tile rows per warp");
    static_assert(G <= LPR, "one (row, head) score per lane after the reduction");
    static_assert(BT <= 32, "one box per producer lane");
    static_assert(NWC * G * (D + 2) * 4 <= NS * STAGE_BYTES, "merge area fits the stages");
    static_assert(TILE_BYTES % 128 == 0, "TMA destinations stay 128-byte aligned");
};

// Reduce-scatter G partial dot products across the LPR lanes of a key row: after
// log2(LPR) exchange levels the lane holds the full sum for head head_of_lane(lane).
template <int G, int LPR>
__device__ __forceinline__ float row_reduce_scatter(float (&v)[G], int lane) {
    int n = G;
#pragma unroll
    for (int m = LPR / 2; m >= 1; m >>= 1) {
        if (n > 1) {
            const bool up = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < G / 2; ++i) {
                if (i < n / 2) {
                    const float send = up ? v[i] : v[i + n / 2];
                    const float keep = up ? v[i + n / 2] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, m);
                }
            }
            n >>= 1;
        } else {
            v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], m);
        }
    }
    return v[0];
}

template <int G, int LPR>
__device__ __forceinline__ int head_of_lane(int lane) {
    int h = 0, n = G;
#pragma unroll
    for (int m = LPR / 2; m >= 1 && n > 1; m >>= 1) {
        if (lane & m) h += n / 2;
        n >>= 1;
    }
    return h;
}

template <class C, bool PAGED>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
    split_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                 const SplitParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int D = C::D, G = C::G, HG = C::HG, NWC = C::NWC, BT = C::BT, NS = C::NS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- work unit -------------------------------------------------------------------
    const int nkvg = p.Hkv / HG;
    const int units = p.B * nkvg;
    const int s = blockIdx.x / units;
    const int rem = blockIdx.x - s * units;
    const int b = rem / nkvg;
    const int kvg = rem - b * nkvg;
    int L = p.seq_lens[b];
    if (L < 0 || L > p.max_kv_len) {
        if (threadIdx.x == 0 && s == 0 && kvg == 0) flag_error(DAP_DEVERR_SEQLEN);
        L = min(max(L, 0), p.max_kv_len);
    }
    const int nsplit = max(1, (L + p.chunk - 1) / p.chunk);
    if (s >= nsplit) return;
    const int tok0 = s * p.chunk;
    const int tok1 = min(L, tok0 + p.chunk);
    const int ntiles = tok1 > tok0 ? (tok1 - tok0 + BT - 1) / BT : 0;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + NS;
    int *misc = reinterpret_cast<int *>(smem + C::MISC_OFF);  // [0] tiles issued, [1] abort
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NWC);
        }
        misc[0] = 0;
        misc[1] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NWC) {
        // ---- producer warp: page lookup + TMA issue ------------------------------------
        if (lane == 0) {
            prefetch_tensormap(&mapK);
            prefetch_tensormap(&mapV);
        }
        const int R = PAGED ? p.box_rows : BT;
        const int kvh0 = kvg * HG;
        const int32_t *table = PAGED ? p.block_table + (long long)b * p.max_pages : nullptr;
        auto lookup = [&](int tile) -> int {  // page id of this lane's box of `tile`
            if (!PAGED) return b;
            const int t = tok0 + tile * BT + lane * R;
            if (lane * R >= BT || t >= tok1) return 0;
            int pg = __ldg(table + t / p.page_size);
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
                uint8_t *sK = smem + st * C::STAGE_BYTES + lane * R * HG * C::ROWB;
                uint8_t *sV = sK + C::TILE_BYTES;
                const int tt = t + lane * R;
                const int slot = PAGED ? tt % p.page_size : tt;
                tma_load_4d(sK, &mapK, 0, kvh0, slot, pg, &full[st]);
                tma_load_4d(sV, &mapV, 0, kvh0, slot, pg, &full[st]);
            }
            issued = i + 1;
        }
        if (lane == 0) misc[0] = issued;
        __syncthreads();  // pairs with the consumers' final __syncthreads
        return;
    }

    // ---- consumer warps --------------------------------------------------------------
    const int hh = warp % HG;           // kv head within the CTA's group
    const int ph = warp / HG;           // row phase of this warp
    const int kvh = kvg * HG + hh;
    const int row0 = ph * C::RW;
    const int qlane = lane % C::LPR;
    const int rgrp = lane / C::LPR;
    const int hsel = head_of_lane<G, C::LPR>(lane);

    float2 q2[G][C::CPL][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const __nv_bfloat16 *qrow = p.q + (long long)b * p.q_sb + (long long)(kvh * G + g) * p.q_sh;
#pragma unroll
        for (int i = 0; i < C::CPL; ++i) {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(qrow + 8 * (qlane + i * C::LPR)));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = bf16x2_to_float2(ws[j]);
                q2[g][i][j] = make_float2(f.x * p.qscale, f.y * p.qscale);
            }
        }
    }

    float m_run = -INFINITY, l_run = 0.f;
    float2 acc[G][C::DPV / 2 > 0 ? C::DPV / 2 : 1];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < C::DPV / 2; ++j) acc[g][j] = make_float2(0.f, 0.f);
    float *pbuf = reinterpret_cast<float *>(smem + C::PBUF_OFF) + warp * C::RW * G;
    float *abuf = reinterpret_cast<float *>(smem + C::ABUF_OFF) + warp * G;

    int consumed = 0;
    for (int i = 0; i < ntiles; ++i) {
        const int st = i % NS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[st], (i / NS) & 1))) {  // warp-uniform
            misc[1] = 1;
            break;
        }
        const uint8_t *sK = smem + st * C::STAGE_BYTES;
        const uint8_t *sV = sK + C::TILE_BYTES;
        const int nvalid = min(BT, tok1 - (tok0 + i * BT));
        const int nv_w = min(max(nvalid - row0, 0), C::RW);

        // scores: one (row, head) value per lane per pass
        float sc[C::PASSES];
#pragma unroll
        for (int ps = 0; ps < C::PASSES; ++ps) {
            const int r = ps * C::RPP + rgrp;
            const uint8_t *krow = sK + ((row0 + r) * HG + hh) * C::ROWB;
            float2 a2[G];
#pragma unroll
            for (int g = 0; g < G; ++g) a2[g] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < C::CPL; ++c) {
                const uint4 w = lds128(krow + (qlane + c * C::LPR) * 16);
                const float2 k0 = bf16x2_to_float2(w.x), k1 = bf16x2_to_float2(w.y);
                const float2 k2 = bf16x2_to_float2(w.z), k3 = bf16x2_to_float2(w.w);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    a2[g] = ffma2(q2[g][c][0], k0, a2[g]);
                    a2[g] = ffma2(q2[g][c][1], k1, a2[g]);
                    a2[g] = ffma2(q2[g][c][2], k2, a2[g]);
                    a2[g] = ffma2(q2[g][c][3], k3, a2[g]);
                }
            }
            float part[G];
#pragma unroll
            for (int g = 0; g < G; ++g) part[g] = a2[g].x + a2[g].y;
            const float v = row_reduce_scatter<G, C::LPR>(part, lane);
            sc[ps] = (r < nv_w) ? v : -INFINITY;
        }

        // online softmax (base 2) for head hsel
        float mx = sc[0];
#pragma unroll
        for (int ps = 1; ps < C::PASSES; ++ps) mx = fmaxf(mx, sc[ps]);
#pragma unroll
        for (int m = C::LPR; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, m));
        const float m_new = fmaxf(m_run, mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2(m_run - m_use);
        float psum = 0.f;
#pragma unroll
        for (int ps = 0; ps < C::PASSES; ++ps) {
            sc[ps] = ex2(sc[ps] - m_use);
            psum += sc[ps];
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
#pragma unroll
        for (int ps = 0; ps < C::PASSES; ++ps) pbuf[(ps * C::RPP + rgrp) * G + hsel] = sc[ps];
        if (rgrp == 0) abuf[hsel] = alpha;
        __syncwarp();

        // PV
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float a = abuf[g];
#pragma unroll
            for (int j = 0; j < C::DPV / 2; ++j) acc[g][j] = __fmul2_rn(acc[g][j], make_float2(a, a));
        }
        const uint8_t *vbase = sV + (row0 * HG + hh) * C::ROWB + lane * C::DPV * 2;
#pragma unroll 4
        for (int r = 0; r < nv_w; ++r) {
            const uint8_t *vrow = vbase + r * HG * C::ROWB;
            float2 vv[C::DPV / 2];
            if constexpr (C::DPV == 4) {
                const uint2 w = *reinterpret_cast<const uint2 *>(vrow);
                vv[0] = bf16x2_to_float2(w.x);
                vv[1] = bf16x2_to_float2(w.y);
            } else {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(vrow);
                vv[0] = bf16x2_to_float2(w);
            }
            const float *pr = pbuf + r * G;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pg = pr[g];
                const float2 pp = make_float2(pg, pg);
#pragma unroll
                for (int j = 0; j < C::DPV / 2; ++j) acc[g][j] = ffma2(pp, vv[j], acc[g][j]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        consumed = i + 1;
    }

    // ---- merge the warps of each kv head and write --------------------------------------
#pragma unroll
    for (int m = C::LPR; m < 32; m <<= 1) l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, m);
    __syncthreads();  // every consumer is done with the stages; producer has finished issuing
    if (misc[1]) {
        // A wait timed out.  Drain the copies still in flight (bounded), write nothing.
        if (threadIdx.x == 0) {
            for (int i = consumed; i < misc[0]; ++i) (void)mbar_wait(&full[i % NS], (i / NS) & 1);
        }
        return;
    }
    float *macc = reinterpret_cast<float *>(smem);                // [NWC][G][D]
    float *mml = macc + NWC * G * D;                               // [NWC][G][2]
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < C::DPV / 2; ++j)
            *reinterpret_cast<float2 *>(macc + (warp * G + g) * D + lane * C::DPV + 2 * j) = acc[g][j];
    if (rgrp == 0) {
        mml[(warp * G + hsel) * 2 + 0] = m_run;
        mml[(warp * G + hsel) * 2 + 1] = l_run;
    }
    named_sync(1, NWC * 32);

    const bool direct = (nsplit == 1);
    for (int e = threadIdx.x * 2; e < HG * G * D; e += NWC * 32 * 2) {
        const int hl = e / (G * D);
        const int g = (e / D) % G;
        const int d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::WPH; ++w) M = fmaxf(M, mml[((w * HG + hl) * G + g) * 2]);
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float a0 = 0.f, a1 = 0.f, lv = 0.f;
#pragma unroll
        for (int w = 0; w < C::WPH; ++w) {
            const int ww = w * HG + hl;
            const float f = ex2(mml[(ww * G + g) * 2] - Mu);
            lv = fmaf(f, mml[(ww * G + g) * 2 + 1], lv);
            const float2 x = *reinterpret_cast<const float2 *>(macc + (ww * G + g) * D + d);
            a0 = fmaf(f, x.x, a0);
            a1 = fmaf(f, x.y, a1);
        }
        const int hq = (kvg * HG + hl) * G + g;
        if (direct) {
            const float inv = lv > 0.f ? 1.f / lv : 0.f;
            *reinterpret_cast<__nv_bfloat162 *>(p.out + (long long)b * p.o_sb + (long long)hq * p.o_sh + d) =
                __floats2bfloat162_rn(a0 * inv, a1 * inv);
        } else {
            const long long row = ((long long)b * p.num_splits + s) * p.Hq + hq;
            *reinterpret_cast<float2 *>(p.o_part + row * D + d) = make_float2(a0, a1);
            if (d == 0) *reinterpret_cast<float2 *>(p.ml_part + row * 2) = make_float2(M, lv);
        }
    }
}

// Merge the split partials of every (sequence, query head) with more than one split, in
// split order: M = max_s m_s, out = sum_s 2^(m_s-M) acc_s / sum_s 2^(m_s-M) l_s.  One warp
// per output row (AstrAI csrc log, split-KV commit: the combine kernel).
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const SplitParams p) {
    constexpr int DPV = D / 32;
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= p.B * p.Hq) return;
    const int b = gw / p.Hq, hq = gw - b * p.Hq;
    const int L = min(max(p.seq_lens[b], 0), p.max_kv_len);
    const int nsplit = max(1, (L + p.chunk - 1) / p.chunk);
    if (nsplit == 1) return;
    const long long row0 = (long long)b * p.num_splits * p.Hq + hq;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, p.ml_part[(row0 + (long long)s * p.Hq) * 2]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float acc[DPV];
#pragma unroll
    for (int j = 0; j < DPV; ++j) acc[j] = 0.f;
    float lsum = 0.f;
    for (int s = 0; s < nsplit; ++s) {
        const long long row = row0 + (long long)s * p.Hq;
        const float2 ml = *reinterpret_cast<const float2 *>(p.ml_part + row * 2);
        const float f = ex2(ml.x - Mu);
        lsum = fmaf(f, ml.y, lsum);
        const float *o = p.o_part + row * D + lane * DPV;
        if constexpr (DPV == 4) {
            const float4 x = *reinterpret_cast<const float4 *>(o);
            acc[0] = fmaf(f, x.x, acc[0]);
            acc[1] = fmaf(f, x.y, acc[1]);
            acc[2] = fmaf(f, x.z, acc[2]);
            acc[3] = fmaf(f, x.w, acc[3]);
        } else {
            const float2 x = *reinterpret_cast<const float2 *>(o);
            acc[0] = fmaf(f, x.x, acc[0]);
            acc[1] = fmaf(f, x.y, acc[1]);
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    __nv_bfloat16 *o = p.out + (long long)b * p.o_sb + (long long)hq * p.o_sh + lane * DPV;
#pragma unroll
    for (int j = 0; j < DPV; j += 2)
        *reinterpret_cast<__nv_bfloat162 *>(o + j) = __floats2bfloat162_rn(acc[j] * inv, acc[j + 1] * inv);
}

// ---- host side -----------------------------------------------------------------------

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// [D, Hkv, rows, outer] bf16 view of a cache, box [D, HG, box_rows, 1].
bool encode_cache_map(CUtensorMap *map, const void *base, int D, int Hkv, long long rows,
                      long long outer, int HG, int box_rows) {
    EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)rows, (cuuint64_t)outer};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2,
                                   (cuuint64_t)rows * Hkv * D * 2};
    const cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)HG, (cuuint32_t)box_rows, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gcd_int(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

template <class C, bool PAGED>
dap_status launch_split(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    const int R = PAGED ? gcd_int(a.page_size, C::BT) : C::BT;
    p.box_rows = R;
    CUtensorMap mk, mv;
    const long long rows = PAGED ? a.page_size : a.max_len;
    const long long outer = PAGED ? a.num_pages : a.B;
    if (!encode_cache_map(&mk, a.k, a.D, a.Hkv, rows, outer, C::HG, R) ||
        !encode_cache_map(&mv, a.v, a.D, a.Hkv, rows, outer, C::HG, R))
        return DAP_ERR_CUDA;
    auto kern = split_kernel<C, PAGED>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return DAP_ERR_CUDA;
    const long long grid = (long long)a.B * (a.Hkv / C::HG) * a.num_splits;
    if (grid > 0x7FFFFFFFLL) return DAP_ERR_SHAPE;
    if (g_trace.split_begin) cudaEventRecord(g_trace.split_begin, stream);
    kern<<<(unsigned)grid, C::THREADS, C::SMEM, stream>>>(mk, mv, p);
    if (cudaGetLastError() != cudaSuccess) return DAP_ERR_CUDA;
    if (g_trace.split_end) cudaEventRecord(g_trace.split_end, stream);
    if (a.num_splits > 1) {
        const int rows_out = a.B * a.Hq;
        if (a.D == 128)
            combine_kernel<128><<<(rows_out + 7) / 8, 256, 0, stream>>>(p);
        else
            combine_kernel<64><<<(rows_out + 7) / 8, 256, 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess) return DAP_ERR_CUDA;
    }
    if (g_trace.combine_end) cudaEventRecord(g_trace.combine_end, stream);
    return DAP_OK;
}

template <int D, int G>
dap_status dispatch_layout(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    using C = SplitCfg<D, G, 1, 4, 32, 4, (G <= 4 ? 3 : 2)>;
    return a.paged ? launch_split<C, true>(a, p, stream) : launch_split<C, false>(a, p, stream);
}

}  // namespace

bool read_errors_decode(unsigned int *flags, bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_errors, sizeof v) != cudaSuccess) return false;
    if (clear) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_device_errors, &z, sizeof z) != cudaSuccess) return false;
    }
    *flags |= v;
    return true;
}

dap_status launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    SplitParams p;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.q_sb = a.q_sb;
    p.q_sh = a.q_sh;
    p.block_table = a.block_table;
    p.max_pages = a.max_pages;
    p.seq_lens = a.seq_lens;
    p.max_kv_len = a.max_kv_len;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.page_size = a.paged ? a.page_size : a.max_len;
    p.num_pages = a.paged ? a.num_pages : a.B;
    p.box_rows = 0;
    p.num_splits = a.num_splits;
    p.chunk = a.chunk;
    p.qscale = a.scale * 1.4426950408889634f;
    p.o_part = static_cast<float *>(a.workspace);
    p.ml_part = a.num_splits > 1
                    ? reinterpret_cast<float *>(static_cast<char *>(a.workspace) +
                                                partial_acc_bytes(a.B, a.Hq, a.D, a.num_splits))
                    : nullptr;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.o_sb = a.o_sb;
    p.o_sh = a.o_sh;
    const int G = a.Hq / a.Hkv;
    if (a.D == 128) {
        switch (G) {
            case 1: return dispatch_layout<128, 1>(a, p, stream);
            case 2: return dispatch_layout<128, 2>(a, p, stream);
            case 4: return dispatch_layout<128, 4>(a, p, stream);
            case 8: return dispatch_layout<128, 8>(a, p, stream);
        }
    } else if (a.D == 64) {
        switch (G) {
            case 1: return dispatch_layout<64, 1>(a, p, stream);
            case 2: return dispatch_layout<64, 2>(a, p, stream);
            case 4: return dispatch_layout<64, 4>(a, p, stream);
            case 8: return dispatch_layout<64, 8>(a, p, stream);
        }
    }
    return DAP_ERR_UNSUPPORTED;
}

}  // namespace dap
