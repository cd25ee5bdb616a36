// dap_multi.cuh -- multi-token causal decode over the paged KV cache: the kernel, its
// launch and dispatch templates, instantiated by dap_multi.cu (TMA-fed tiles) and
// dap_multi_gather.cu (row-gather tiles for page sizes that are not multiples of 8).
//
// Several new tokens per sequence (speculative-decoding verification, chunked short
// prefill) attend the cache causally.  The tokens of all sequences are packed back to back
// and cut into work tiles by the packed-q work map of the AstrAI "CUDA Kernels" doc
// ("Q Scheduling and KV Addressing": qo_indptr, q_tile_to_batch, q_tile_to_index).  A
// tile holds 16 / G tokens so that its tokens x the G heads of one kv head make 16 query
// columns: the tensor-core N dimension, against which every K/V tile staged by TMA is
// used once for all of the tile's tokens.  The producer warp and the stage ring are the
// single-token per-sequence schedule's; the consumer adds a causal mask per column.
#pragma once

#include "dap_tile.cuh"

namespace dap {

// ---- multi-token consumer ---------------------------------------------------------------
// The query columns are (token, head) pairs: 16 columns = QT = 16 / G new tokens x G heads
// of the kv head (two n8 tiles).  Per 16-key slice: S^T = K . Q^T for each n tile, a causal
// mask per column (key position <= the column's token position), the online softmax per
// column, movmatrix into the B operands and O^T += V^T . P^T.  q is read from global memory
// (the per-sequence schedule gives each CTA one unit), and the four warps merge their
// partial states in quarters of D.

// NT n8 tiles of query columns per warp (2 for multi-token decode; 1 for masked single-token
// decode, whose tiles hold one token); CG column groups (1, or 2 for 32-column tiles: warps
// w and w + 4 take the same 16 keys of every tile for columns 0..15 and 16..31, so all
// of a sequence's new tokens meet each K/V tile once); MASK: a bool mask tile rides with
// every K/V tile.
// Head dims: 64 and 128 in 64-key tiles of 128-byte-swizzled column blocks; 256 in 32-key
// tiles (two key slices, so a stage stays near 32 KB at two CTAs per SM); 32 in 64-key
// tiles of 64-byte rows with the 64-byte swizzle, six stages.
// GATHER: page sizes that are not multiples of 8; the producer warp copies the rows of each
// tile into the same swizzled layout with cp.async (dap_tile.cuh, row gather).
template <int D_, int G_, int NT_ = 2, bool MASK_ = false, int CG_ = 1, bool GATHER_ = false>
struct MultiCfg {
    static constexpr bool GATHER = GATHER_;
    static constexpr int CG = CG_, KW = D_ == 256 ? 2 : 4;  // column groups, key slices
    static constexpr int D = D_, G = G_, HG = 1, NWC = KW * CG, BT = 16 * KW;
    static constexpr int NS = D == 32 ? 6 : (CG == 2 ? 5 : 3);
    static constexpr int MINB = D == 32 ? (CG == 2 ? 2 : 3) : (CG == 2 ? 1 : 2);
    static constexpr bool MMA = true, SWZ = true, MASK = MASK_;
    static constexpr int NT = NT_;
    static constexpr int NCOL = 8 * NT * CG;        // query columns
    static constexpr int QT = NCOL / G;             // new tokens per work tile
    static constexpr int WPH = NWC, KPW = BT / KW;
    static constexpr int ROWB = D * 2, HPU = G, SWB = D >= 64 ? 128 : 64, NBLK = ROWB / SWB, CPB = SWB / 16;
    static constexpr int TILE_BYTES = BT * ROWB;
    static constexpr int QBYTES = 0;
    static constexpr int MASK_OFF = 2 * TILE_BYTES;  // [QT tokens][BT keys] bytes, 1024-aligned
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES + (MASK ? 1024 : 0);
    static constexpr int NPART = D == 32 ? 2 : 4;   // merge in parts of D (16 dims or more each)
    static constexpr int MRG_OFF = NS * STAGE_BYTES;
    static constexpr int MRG_BYTES = KW * NCOL * (D / NPART + 2) * 4;
    static constexpr int HDR_OFF = MRG_OFF + MRG_BYTES;
    static constexpr int HDR_INTS = 8;
    static constexpr int MISC_OFF = HDR_OFF + NS * HDR_INTS * 4;
    static constexpr int BAR_OFF = (MISC_OFF + 16 + 7) & ~7;
    static constexpr int SMEM = BAR_OFF + (2 * NS + 1) * 8 + 1024;
    static constexpr int THREADS = (NWC + 1) * 32;
    static_assert(KPW == 16 && NCOL % G == 0 && QT >= 1 && STAGE_BYTES % 1024 == 0 && (!MASK || QT * BT <= 1024),
                  "multi-token tiling");
    static_assert(!MASK || CG == 1, "masked tiles use one column group");
    static_assert((D / 16) % NPART == 0 && ROWB % SWB == 0, "whole 16-dim steps per merge part");
};

template <class C>
struct MultiConsumer {
    static constexpr int D = C::D, G = C::G, KS = D / 16, NT = C::NT;
    uint32_t qb[KS][NT][2];
    float acc[KS][NT][4];
    float m_run[NT][2], l_run[NT][2];
    float qscale;
    int warp, lane, g, t, kw, key0, col0, nq, p_base, rb;  // rb: log2 of the tile's box rows (tile_off)
    static constexpr int hh = 0;

    __device__ __forceinline__ void init(int w, int l, uint8_t *, int box_rows_log2) {
        warp = w;
        lane = l;
        rb = box_rows_log2;
        g = l >> 2;
        t = l & 3;
        kw = w % C::KW;
        key0 = kw * C::KPW;
        col0 = (w / C::KW) * (8 * NT);  // first query column of this warp's group
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                m_run[n][j] = -INFINITY;
                l_run[n][j] = 0.f;
            }
#pragma unroll
        for (int m = 0; m < KS; ++m)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[m][n][j] = 0.f;
    }

    // q of the tile's tokens: token i, head h at base + i * tstride + h * hstride
    __device__ __forceinline__ void load_q(const __nv_bfloat16 *base, long long tstride, long long hstride,
                                           int ntok, int pos0, float qs) {
        qscale = qs;
        nq = ntok;
        p_base = pos0;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int c = col0 + n * 8 + g;
            const int ti = c / G, hc = c % G;
#pragma unroll
            for (int k = 0; k < KS; ++k) {
                if (ti < ntok) {
                    const __nv_bfloat16 *r = base + ti * tstride + hc * hstride + 16 * k + 2 * t;
                    qb[k][n][0] = *reinterpret_cast<const uint32_t *>(r);
                    qb[k][n][1] = *reinterpret_cast<const uint32_t *>(r + 8);
                } else {
                    qb[k][n][0] = qb[k][n][1] = 0u;
                }
            }
        }
    }

    // byte offset of (key, dim) in the swizzled tile (tile_off)
    __device__ __forceinline__ uint32_t off(int key, int dim) const { return tile_off<C>(key, dim >> 3, rb); }

    // tile_pos: absolute position of the tile's first key
    __device__ __forceinline__ void tile(uint8_t *stage, int nvalid, int tile_pos) {
        const int nv = nvalid - key0;
        if (nv <= 0) return;
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
        float c[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j) c[n][j] = 0.f;
        {
            const int key = key0 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int dcol = ((lane >> 4) & 1) * 8;
#pragma unroll
            for (int k = 0; k < KS; ++k) {
                uint32_t a[4];
                ldmatrix_x4(a, kbase + off(key, 16 * k + dcol));
#pragma unroll
                for (int n = 0; n < NT; ++n) mma_bf16_16816(c[n], a, qb[k][n][0], qb[k][n][1]);
            }
        }
        const int kpos0 = tile_pos + key0 + g, kpos1 = kpos0 + 8;  // absolute key positions
        uint32_t b0[NT], b1[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            float s[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int col = col0 + n * 8 + 2 * t + j;
                const int ti = col / G;
                const int lim = p_base + ti;  // this column's token sees keys <= lim
                bool keep0 = ti < nq && g < nv && kpos0 <= lim;
                bool keep1 = ti < nq && g + 8 < nv && kpos1 <= lim;
                if constexpr (C::MASK) {  // the token's mask bytes of keys g, g+8 of this slice
                    const uint8_t *mk = stage + C::MASK_OFF + ti * C::BT + key0 + g;
                    keep0 = keep0 && mk[0] != 0;
                    keep1 = keep1 && mk[8] != 0;
                }
                s[j] = keep0 ? __fmul_rn(c[n][j], qscale) : -INFINITY;  // (rounded once: feeds max and exp)
                s[j + 2] = keep1 ? __fmul_rn(c[n][j + 2], qscale) : -INFINITY;
            }
            float mx[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xFFFFFFFFu, mx[0], o));
                mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xFFFFFFFFu, mx[1], o));
            }
            float alpha[2], mu[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float m_new = fmaxf(m_run[n][j], mx[j]);
                mu[j] = (m_new == -INFINITY) ? 0.f : m_new;
                alpha[j] = ex2(m_run[n][j] - mu[j]);
                m_run[n][j] = m_new;
            }
            const uint32_t w0 = pack_bf16x2(ex2(s[0] - mu[0]), ex2(s[1] - mu[1]));
            const uint32_t w1 = pack_bf16x2(ex2(s[2] - mu[0]), ex2(s[3] - mu[1]));
            const float2 p0 = bf16x2_to_float2(w0), p1 = bf16x2_to_float2(w1);
            l_run[n][0] = l_run[n][0] * alpha[0] + (p0.x + p1.x);
            l_run[n][1] = l_run[n][1] * alpha[1] + (p0.y + p1.y);
            // the running max rarely moves after the first tiles: rescale only when it did
            if (__any_sync(0xFFFFFFFFu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
                for (int m = 0; m < KS; ++m) {
                    acc[m][n][0] *= alpha[0];
                    acc[m][n][1] *= alpha[1];
                    acc[m][n][2] *= alpha[0];
                    acc[m][n][3] *= alpha[1];
                }
            }
            b0[n] = movmatrix_trans(w0);
            b1[n] = movmatrix_trans(w1);
        }
        {
            const int key = key0 + (lane & 7) + ((lane >> 4) & 1) * 8;
            const int dcol = ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int m = 0; m < KS; ++m) {
                uint32_t a[4];
                ldmatrix_x4_trans(a, vbase + off(key, 16 * m + dcol));
#pragma unroll
                for (int n = 0; n < NT; ++n) mma_bf16_16816(acc[m][n], a, b0[n], b1[n]);
            }
        }
    }

    // merge the four key slices per column in C::NPART parts of D; emit(col, d, a0, a1, M, l)
    template <class Sync, class Emit>
    __device__ __forceinline__ bool finish(float *mrg, Sync sync, Emit emit) {
        constexpr int NWC = C::NWC, KW = C::KW, NC = C::NCOL, DP = D / C::NPART, MP = KS / C::NPART;
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                l_run[n][0] += __shfl_xor_sync(0xFFFFFFFFu, l_run[n][0], o);
                l_run[n][1] += __shfl_xor_sync(0xFFFFFFFFu, l_run[n][1], o);
            }
        float *macc = mrg;               // [KW][NC][DP]
        float *mml = mrg + KW * NC * DP;   // [KW][NC][2]
        if (g == 0) {
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    mml[(kw * NC + col0 + n * 8 + 2 * t + j) * 2 + 0] = m_run[n][j];
                    mml[(kw * NC + col0 + n * 8 + 2 * t + j) * 2 + 1] = l_run[n][j];
                }
        }
        const int tid = warp * 32 + lane;
#pragma unroll
        for (int part = 0; part < C::NPART; ++part) {
#pragma unroll
            for (int m = part * MP; m < (part + 1) * MP; ++m) {
                const int d = 16 * m + g - part * DP;
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float *row = macc + (kw * NC + col0 + n * 8 + 2 * t + j) * DP;
                        row[d] = acc[m][n][j];
                        row[d + 8] = acc[m][n][j + 2];
                    }
            }
            if (!sync()) return false;
            for (int e = tid * 2; e < NC * DP; e += NWC * 32 * 2) {
                const int col = e / DP, dd = e % DP;
                if (col / G < nq) {
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < KW; ++w) M = fmaxf(M, mml[(w * NC + col) * 2]);
                    const float Mu = (M == -INFINITY) ? 0.f : M;
                    float a0 = 0.f, a1 = 0.f, lv = 0.f;
#pragma unroll
                    for (int w = 0; w < KW; ++w) {
                        const float f = ex2(mml[(w * NC + col) * 2] - Mu);
                        lv = fmaf(f, mml[(w * NC + col) * 2 + 1], lv);
                        const float2 x = *reinterpret_cast<const float2 *>(macc + (w * NC + col) * DP + dd);
                        a0 = fmaf(f, x.x, a0);
                        a1 = fmaf(f, x.y, a1);
                    }
                    emit(col, part * DP + dd, a0, a1, M, lv);
                }
            }
            if (!sync()) return false;
        }
        return true;
    }
};

// ---- multi-token decode: one CTA per (q tile, kv head, split) ----------------------------
// The packed-q work map (AstrAI "CUDA Kernels" doc, "Q Scheduling and KV Addressing"): q
// holds the new tokens of all sequences back to back, qo_indptr is the prefix sum of their
// counts, and work tile w covers tokens [tile_index[w] * QT, +QT) of sequence tile_batch[w].
// Token i of a sequence with q_len new tokens and L cached keys (the new ones included)
// sits at position L - q_len + i and attends keys 0 .. that position.  The tile's KV range
// ends after its last token's position and is cut into chunks of p.chunk keys.

struct MultiTile {
    int b, q0, qlen, i0, ntok, pos0, kv_end;
};

// The tile's tokens and KV range from its work-map entry (sequence b, tile index) and the
// values q0 = qo_indptr[b], q1 = qo_indptr[b + 1], L = seq_lens[b] (loaded by the caller,
// from sequence 0 when b is out of range); false for an entry that names no token
// (flagged).  Shared by the attention kernel and its combine so both agree on the splits.
__device__ __forceinline__ bool multi_tile(const SplitParams &p, int b, int tindex, int q0, int q1, int L,
                                           int qt, bool report, MultiTile *t) {
    if (b < 0 || b >= p.B) {
        if (report) flag_error(DAP_DEVERR_QMAP);
        return false;
    }
    t->b = b;
    t->q0 = q0;
    t->qlen = q1 - q0;
    t->i0 = tindex * qt;
    t->ntok = min(qt, t->qlen - t->i0);
    if (tindex < 0 || t->ntok <= 0 || q0 < 0 || q1 > p.total_q) {
        if (report) flag_error(DAP_DEVERR_QMAP);
        return false;
    }
    if (L < 0 || L > p.max_kv_len || t->qlen > L) {
        if (report) flag_error(DAP_DEVERR_SEQLEN);
        L = min(max(L, 0), p.max_kv_len);
    }
    t->pos0 = L - t->qlen + t->i0;  // negative for tokens that would sit before the cache start
    t->kv_end = max(0, t->pos0 + t->ntok);
    return true;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
    multi_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                 const __grid_constant__ CUtensorMap mapM, const SplitParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = aligned_smem<C>(smem_raw);
    constexpr int G = C::G, NWC = C::NWC, BT = C::BT, NS = C::NS, D = C::D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int units = p.num_tiles * p.Hkv;
    const int s = blockIdx.x / units;
    const int rem = blockIdx.x - s * units;
    const int w = rem / p.Hkv;
    const int kvh = rem - w * p.Hkv;
    // Launched as a programmatic dependent of the previous kernel on the stream: nothing
    // global is read before the wait (that kernel may still write the inputs); the combine
    // of this call may launch at once (it waits for this grid before its reads).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Every load the schedule needs before the first TMA is issued at once: the work-map
    // entry, then its sequence's q range and length together with the producer's page ids
    // of the first tile (read from position s * chunk on; entries past the sequence's end
    // are read within the table but not used).
    // (no work map: one token per sequence, tile w = sequence w)
    const int wb = p.tile_batch ? p.tile_batch[w] : w, wi = p.tile_index ? p.tile_index[w] : 0;
    const int bb = (wb >= 0 && wb < p.B) ? wb : 0;
    const int q0 = p.qo_indptr ? p.qo_indptr[bb] : bb, q1 = p.qo_indptr ? p.qo_indptr[bb + 1] : bb + 1;
    const int Lraw = p.seq_lens[bb];
    const int R = p.box_rows;
    int pg_first = 0;
    if (!C::GATHER && warp == NWC && lane * R < BT) {
        const long long t = (long long)s * p.chunk + lane * R;
        if (t < (long long)p.max_pages * p.page_size)
            pg_first = __ldg(p.block_table + (long long)bb * p.max_pages + t / p.page_size);
    }
    MultiTile tl;
    if (!multi_tile(p, wb, wi, q0, q1, Lraw, C::QT, threadIdx.x == 0 && s == 0 && kvh == 0, &tl)) return;
    const int nsplit = max(1, (tl.kv_end + p.chunk - 1) / p.chunk);
    if (s >= nsplit) return;
    const int tok0 = s * p.chunk;
    const int tok1 = min(tl.kv_end, tok0 + p.chunk);
    const int ntiles = tok1 > tok0 ? (tok1 - tok0 + BT - 1) / BT : 0;

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
    __syncthreads();

    if (C::GATHER && warp == NWC) {  // ---- producer warp, row gather (as in split_kernel)
        if (C::MASK && lane == 0) prefetch_tensormap(&mapM);
        const int32_t *table = p.block_table + (long long)tl.b * p.max_pages;
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
            // (with a mask: the tile's mask bytes by TMA, zeros past either end)
            fill_tile_rows<C>(smem + st * C::STAGE_BYTES, rp, min(BT, tok1 - t), kvh, p,
                              C::MASK ? (uint32_t)(C::QT * BT) : 0u,
                              [&] {
                                  if (C::MASK)
                                      tma_load_3d(smem + st * C::STAGE_BYTES + C::MASK_OFF, &mapM, t, tl.q0 + tl.i0, 0,
                                                  &full[st]);
                              },
                              &full[st], lane);
            issued = i + 1;
        }
        if (lane == 0) misc[0] = issued;
        __syncthreads();
        return;
    }
    if (warp == NWC) {  // ---- producer warp: page lookup + TMA issue (as in split_kernel)
        if (lane == 0) {
            prefetch_tensormap(&mapK);
            prefetch_tensormap(&mapV);
            if (C::MASK) prefetch_tensormap(&mapM);
        }
        const int32_t *table = p.block_table + (long long)tl.b * p.max_pages;
        auto lookup = [&](int tile) -> int {
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
            const int nbox = (nvalid + R - 1) / R;
            const uint32_t bytes = (uint32_t)(nbox * R * C::ROWB * 2 + (C::MASK ? C::QT * BT : 0));
            if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes);
            __syncwarp();
            if (lane < nbox) {
                const int tt = t + lane * R;
                issue_kv_box<C>(smem + st * C::STAGE_BYTES, lane, R, &mapK, &mapV, kvh, tt % p.page_size, pg,
                                &full[st]);
            }
            // the tile's mask bytes: keys [t, t + BT) of the tile's tokens (zeros past the ends)
            if (C::MASK && lane == 31)
                tma_load_3d(smem + st * C::STAGE_BYTES + C::MASK_OFF, &mapM, t, tl.q0 + tl.i0, 0, &full[st]);
            issued = i + 1;
        }
        if (lane == 0) misc[0] = issued;
        __syncthreads();
        return;
    }

    // ---- consumer warps
    MultiConsumer<C> cs;
    cs.init(warp, lane, smem, 31 - __clz(C::GATHER ? BT : R));
    cs.reset();
    cs.load_q(p.q + (long long)(tl.q0 + tl.i0) * p.q_sb + (long long)kvh * G * p.q_sh, p.q_sb, p.q_sh, tl.ntok,
              tl.pos0, p.qscale);
    int consumed = 0;
    for (int i = 0; i < ntiles; ++i) {
        const int st = i % NS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[st], (i / NS) & 1))) {
            misc[1] = 1;
            break;
        }
        const int t = tok0 + i * BT;
        cs.tile(smem + st * C::STAGE_BYTES, min(BT, tok1 - t), t);
        if (lane == 0) mbar_arrive(&empty[st]);
        consumed = i + 1;
    }
    __syncthreads();
    if (misc[1]) {
        if (threadIdx.x == 0)
            for (int i = consumed; i < misc[0]; ++i) (void)mbar_wait(&full[i % NS], (i / NS) & 1);
        return;
    }
    const bool direct = (nsplit == 1);
    const int r0 = tl.q0 + tl.i0;
    cs.finish(reinterpret_cast<float *>(smem + C::MRG_OFF), [] { named_sync(1, NWC * 32); return true; },
              [&](int col, int d, float a0, float a1, float M, float lv) {
                  const long long r = r0 + col / G;
                  const int hq = kvh * G + col % G;
                  if (direct) {
                      store_out_pair(p.out + r * p.o_sb + (long long)hq * p.o_sh + d, a0, a1, lv);
                  } else {
                      const long long row = (r * p.num_splits + s) * p.Hq + hq;
                      *reinterpret_cast<float2 *>(p.o_part + row * D + d) = make_float2(a0, a1);
                      if (d == 0) *reinterpret_cast<float2 *>(p.ml_part + row * 2) = make_float2(M, lv);
                  }
              });
}

// Merge of the split partials of every (token, head) row whose tile took more than one
// split: one warp per (token, HPW consecutive heads), which share the token's sequence and
// so its split count.  The sequence of token r is the last b with qo_indptr[b] <= r, found
// by a 32-way search (one load per lane and step: two dependent loads for up to 1024
// sequences, the last step also yielding qo_indptr[b] and qo_indptr[b + 1]).  The
// partials are merged online in split order, SB splits per batch of loads: M = the running
// max of the m_s, the sums rescaled by 2^(M_old - M_new) when it grows (AstrAI csrc log,
// split-KV commit: the combine kernel; numerics commit: guarded division).  Waits for the
// attention grid (programmatic dependent launch).
template <int D, int HPW, int SB>
__global__ void __launch_bounds__(256) combine_multi_kernel(const SplitParams p, int qt) {
    // the next kernel on the stream may be launched now (it waits for this grid before its
    // reads)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int DPV = D / 32;
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int ngroups = p.Hq / HPW;
    if (gw >= p.total_q * ngroups) return;
    const int r = gw / ngroups, hq0 = (gw - r * ngroups) * HPW;
    int b = r, q0 = r, q1 = r + 1;  // no work map: row r is sequence r's one token
    if (p.qo_indptr) {
        int lo = 0, hi = p.B;  // qo_indptr[lo] <= r < qo_indptr[hi] for a well-formed map
        while (hi - lo > 31) {
            const int step = (hi - lo + 31) >> 5;
            const int x = lo + lane * step;
            const bool le = x < hi && p.qo_indptr[x] <= r;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, le);
            const int j = bal ? 31 - __clz(bal) : 0;
            lo += j * step;
            hi = min(lo + step, hi);
        }
        const int x = lo + lane;  // entries lo .. hi (hi - lo <= 31, hi <= B)
        const int v = x <= hi ? p.qo_indptr[x] : 0x7FFFFFFF;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, x < hi && v <= r);
        const int j = bal ? 31 - __clz(bal) : 0;
        q0 = __shfl_sync(0xFFFFFFFFu, v, j);
        q1 = __shfl_sync(0xFFFFFFFFu, v, j + 1);
        b = lo + j;
    }
    MultiTile tl;
    if (!multi_tile(p, b, (r - q0) / qt, q0, q1, p.seq_lens[b], qt, false, &tl)) return;
    const int nsplit = max(1, (tl.kv_end + p.chunk - 1) / p.chunk);
    if (nsplit == 1) return;
    const long long rbase = (long long)r * p.num_splits * p.Hq + hq0;  // row (r, s, hq) = (r S + s) Hq + hq
    float acc[HPW][DPV], lsum[HPW], Mrun[HPW];
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
        lsum[h] = 0.f;
        Mrun[h] = -INFINITY;
#pragma unroll
        for (int j = 0; j < DPV; ++j) acc[h][j] = 0.f;
    }
    for (int s0 = 0; s0 < nsplit; s0 += SB) {
        const int n = min(SB, nsplit - s0);
        float x[HPW][SB][DPV];
        float2 ml[HPW][SB];
#pragma unroll
        for (int h = 0; h < HPW; ++h)
#pragma unroll
            for (int k = 0; k < SB; ++k)
                if (k < n) {
                    const long long row = rbase + (long long)(s0 + k) * p.Hq + h;
                    load_row_part<DPV>(p.o_part + row * D + lane * DPV, x[h][k]);
                    ml[h][k] = *reinterpret_cast<const float2 *>(p.ml_part + row * 2);
                }
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
            float Mn = Mrun[h];
#pragma unroll
            for (int k = 0; k < SB; ++k)
                if (k < n) Mn = fmaxf(Mn, ml[h][k].x);
            const float Mu = (Mn == -INFINITY) ? 0.f : Mn;
            const float sc = ex2(Mrun[h] - Mu);  // 0 while nothing was added
            lsum[h] *= sc;
#pragma unroll
            for (int j = 0; j < DPV; ++j) acc[h][j] *= sc;
#pragma unroll
            for (int k = 0; k < SB; ++k)
                if (k < n) {
                    const float f = ex2(ml[h][k].x - Mu);
                    lsum[h] = fmaf(f, ml[h][k].y, lsum[h]);
#pragma unroll
                    for (int j = 0; j < DPV; ++j) acc[h][j] = fmaf(f, x[h][k][j], acc[h][j]);
                }
            Mrun[h] = Mn;
        }
    }
#pragma unroll
    for (int h = 0; h < HPW; ++h)
        store_row_part<DPV>(p.out + (long long)r * p.o_sb + (long long)(hq0 + h) * p.o_sh + lane * DPV, acc[h], lsum[h]);
}

namespace {

// mask [rows, mask_stride] bytes viewed as [mask_stride, rows, 1]; box [BT, QT, 1]
bool encode_mask_map(CUtensorMap *map, const void *base, long long stride, long long rows, int qt, int bt) {
    EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)stride, (cuuint64_t)rows, 1u};
    const cuuint64_t strides[2] = {(cuuint64_t)stride, (cuuint64_t)(stride * rows)};
    const cuuint32_t box[3] = {(cuuint32_t)bt, (cuuint32_t)qt, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G, int NT, bool MASK, int CG, bool GATHER>
dap_status launch_multi(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    using C = MultiCfg<D, G, NT, MASK, CG, GATHER>;
    const int R = gcd_int(a.page_size, C::BT);
    p.box_rows = R;
    CUtensorMap mk = {}, mv = {}, mm = {};  // (the row-gather producer reads the cache directly)
    if (!GATHER && (!encode_cache_map<C>(&mk, a.k, a.D, a.Hkv, a.page_size, a.num_pages, R) ||
                    !encode_cache_map<C>(&mv, a.v, a.D, a.Hkv, a.page_size, a.num_pages, R)))
        return DAP_ERR_CUDA;
    if (MASK && !encode_mask_map(&mm, a.mask, a.mask_stride, a.total_q, C::QT, C::BT)) return DAP_ERR_CUDA;
    auto kern = multi_kernel<C>;
    static PerDeviceOcc occ = {};
    if (prepare_kernel(kern, C::THREADS, C::SMEM, &occ) <= 0) return DAP_ERR_CUDA;
    const long long grid = (long long)a.num_tiles * a.Hkv * a.num_splits;
    if (grid > 0x7FFFFFFFLL) return DAP_ERR_SHAPE;
    p.o_part = static_cast<float *>(a.workspace);
    p.ml_part = a.num_splits > 1 ? reinterpret_cast<float *>(static_cast<char *>(a.workspace) +
                                                             partial_acc_bytes(a.total_q, a.Hq, a.D, a.num_splits))
                                 : nullptr;
    if (g_trace.split_begin) cudaEventRecord(g_trace.split_begin, stream);
    if (launch_dependent_smem(kern, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM, stream, mk, mv, mm, p) !=
        cudaSuccess)
        return DAP_ERR_CUDA;
    if (g_trace.split_end) cudaEventRecord(g_trace.split_end, stream);
    if (a.num_splits > 1) {
        // one warp per (token, HPW heads), SB splits per batch of loads
        constexpr int HPW_MAX = 4, SB = 1;
        const int hpw = a.Hq % HPW_MAX == 0 ? HPW_MAX : a.Hq % 2 == 0 ? 2 : 1;
        const dim3 cgrid((unsigned)(((long long)a.total_q * (a.Hq / hpw) + 7) / 8));
        const cudaError_t e =
            hpw == HPW_MAX ? launch_dependent(combine_multi_kernel<D, HPW_MAX, SB>, cgrid, dim3(256), stream, p, (int)C::QT)
            : hpw == 2     ? launch_dependent(combine_multi_kernel<D, 2, SB>, cgrid, dim3(256), stream, p, (int)C::QT)
                           : launch_dependent(combine_multi_kernel<D, 1, SB>, cgrid, dim3(256), stream, p, (int)C::QT);
        if (e != cudaSuccess) return DAP_ERR_CUDA;
    }
    if (g_trace.combine_end) cudaEventRecord(g_trace.combine_end, stream);
    return DAP_OK;
}

}  // namespace

namespace {

template <int D, int NT, bool MASK, int CG, bool GATHER>
dap_status dispatch_g(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    switch (a.Hq / a.Hkv) {
        case 1: return launch_multi<D, 1, NT, MASK, CG, GATHER>(a, p, stream);
        case 2: return launch_multi<D, 2, NT, MASK, CG, GATHER>(a, p, stream);
        case 4: return launch_multi<D, 4, NT, MASK, CG, GATHER>(a, p, stream);
        case 8: return launch_multi<D, 8, NT, MASK, CG, GATHER>(a, p, stream);
    }
    return DAP_ERR_UNSUPPORTED;
}

template <int NT, bool MASK, int CG, bool GATHER>
dap_status dispatch_d(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    switch (a.D) {
        case 32: return dispatch_g<32, NT, MASK, CG, GATHER>(a, p, stream);
        case 64: return dispatch_g<64, NT, MASK, CG, GATHER>(a, p, stream);
        case 128: return dispatch_g<128, NT, MASK, CG, GATHER>(a, p, stream);
        case 256: return dispatch_g<256, NT, MASK, CG, GATHER>(a, p, stream);
    }
    return DAP_ERR_UNSUPPORTED;
}

// Multi-token decode: 16-column tiles (tokens_per_tile = 16 / G), or 32-column tiles
// (32 / G) in two column groups; with a mask, 16-column tiles only.
template <bool GATHER>
dap_status multi_entry(const DecodeArgs &a, cudaStream_t stream) {
    SplitParams p = make_params(a);
    const int G = a.Hq / a.Hkv;
    if (a.tokens_per_tile * G == 32) {
        if (a.mask) return DAP_ERR_UNSUPPORTED;
        return dispatch_d<2, false, 2, GATHER>(a, p, stream);
    }
    return a.mask ? dispatch_d<2, true, 1, GATHER>(a, p, stream) : dispatch_d<2, false, 1, GATHER>(a, p, stream);
}

// Masked single-token decode: one token per sequence with no work map (tile w = sequence w),
// one n8 tile of query columns (G heads of the one token).
template <bool GATHER>
dap_status masked_entry(const DecodeArgs &a, cudaStream_t stream) {
    SplitParams p = make_params(a);
    return dispatch_d<1, true, 1, GATHER>(a, p, stream);
}


}  // namespace

}  // namespace dap
