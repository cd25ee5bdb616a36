// dap_multi_tc.cu -- multi-token causal decode on the tcgen05 tensor cores: one work tile
// holds 128 / G new tokens, so its tokens x the G heads of one kv head fill the 128 rows of
// an M = 128 product and every K/V tile staged by TMA is read once for up to 16 tokens at
// G = 8 (the mma.sync consumer of dap_multi.cuh holds at most 32 query columns).
//
// The work map, the tile's KV range, the splits and their merge are those of dap_multi.cuh
// (AstrAI "CUDA Kernels" doc, "Q Scheduling and KV Addressing"); only the consumer differs.
// Per CTA (work tile, kv head, split), tensor memory holds, lane = query row r = (token
// r / G, head r % G):
//   q  columns [0, D/2)          two bf16 per column, stored once;
//   S  columns [64, 96), [96, 128)  fp32 scores of two 32-key half tiles (ping-pong); P
//                                 (bf16 pairs) overwrites the first 16 columns of its half
//                                 once they are read;
//   O  columns [128, 128 + D)    fp32 output accumulator.
// Warps: four consumers (rows), a producer (K/V tiles) and two MMA warps: one thread
// issues, per half tile, S = Q . K^T (A = q from tensor memory, B = the K tile K-major from
// shared memory), another, once the consumers have turned the row of scores into P,
// O += P . V (A = P from tensor memory, B = the V tile MN-major); the commit of a tile's
// last product frees its stage.  The scores of the next half tile are computed while the
// consumers work on the current one.  Consumer thread r masks its row causally (key
// position <= the token's position; with a bool mask, also by the token's mask byte, which
// rides with the stage) and takes the base-2 online softmax; the running max is moved
// lazily: O and l are rescaled only when a half tile's max exceeds the reference by more
// than 2^8 (the weights stay <= 256, far inside fp32), and the reference is stored with the
// partial, so the merge and the final division see the same softmax.
// The K/V tiles are laid out column block major, [D / 64 blocks][64 keys][128 bytes] with
// the 128-byte swizzle, whatever the page size: the layout the row gather (page sizes that
// are not multiples of 8, dap_tile.cuh) writes, and the one TMA writes here with one copy
// per (page segment, column block).  Every 8-key group then sits 1024 bytes after the last,
// so one product spans a whole 32-key half tile, where the other kernels' box-major layout
// would need one product per page segment (N = 16 at a page size of 16).
#include "dap_multi.cuh"
#include "dap_tc.cuh"

namespace dap {

namespace {

template <int D_, int G_, bool MASK_, bool GATHER_>
struct TcCfg {
    static constexpr bool GATHER = GATHER_, MASK = MASK_, SWZ = true;
    static constexpr int D = D_, G = G_, BT = 64, HT = 32;  // keys per K/V tile, per half tile
    static constexpr int ROWB = D * 2, SWB = 128, NBLK = ROWB / SWB, CPB = SWB / 16;
    static constexpr int ROWS = 128, QT = ROWS / G;  // query rows = TMEM lanes; tokens per tile
    static constexpr int TILE_BYTES = BT * ROWB;
    // a stage: the K and V tiles, then (with a mask) the tile's mask bytes [QT tokens][BT keys]
    static constexpr int MASK_OFF = 2 * TILE_BYTES, MASK_BYTES = MASK ? QT * BT : 0;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES + (MASK_BYTES + 1023) / 1024 * 1024;
    // 96 KB of stages (up to 108 KB with masks): two CTAs per SM; D = 256: three stages of
    // 64 KB (and the masks) at one CTA per SM
    static constexpr int MINB = D == 256 ? 1 : 2;
    static constexpr int NS = D == 256 ? 3 : (MASK ? 110592 : 98304) / STAGE_BYTES;
    // warps: 4 consumers, the producer, the S issuer, the PV issuer
    static constexpr int NWC = 4, PRODUCER = 4, S_ISSUER = 5, PV_ISSUER = 6, THREADS = 7 * 32;
    // tensor-memory columns: q, the two half-tile score buffers (P over their first 16
    // columns), O
    // (D = 256: q [0, 128), scores [128, 192), O [256, 512) of 512 columns)
    static constexpr int TQ = 0, TS0 = D == 256 ? 128 : 64, TS1 = TS0 + 32, TO = D == 256 ? 256 : 128;
    static constexpr int TMEM_COLS = D == 256 ? 512 : 256;
    // barriers: full[NS], empty[NS], s_done[2], p_ready[2], pv_done[2], q_ready, fin[2]
    static constexpr int BAR_OFF = NS * STAGE_BYTES;
    static constexpr int NBAR = 2 * NS + 9;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int SMEM = MISC_OFF + 32 + 1024;  // + slack to align the base to 1024
    static_assert((D == 64 || D == 128 || D == 256) && ROWS % G == 0 && NS >= 2 &&
                      SMEM <= (MINB == 2 ? 113 : 227) * 1024,
                  "tcgen05 multi-token tiling");
    static_assert(TQ + D / 2 <= TS0 && TS1 + HT <= TO && TO + D <= TMEM_COLS, "tensor-memory columns");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
    multi_tc_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                    const __grid_constant__ CUtensorMap mapM, const SplitParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = aligned_smem<C>(smem_raw);
    constexpr int G = C::G, NWC = C::NWC, BT = C::BT, HT = C::HT, NS = C::NS, D = C::D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + NS;
    uint64_t *s_done = empty + NS, *p_ready = s_done + 2;
    uint64_t *pv_done = p_ready + 2, *q_ready = pv_done + 2, *fin = q_ready + 1;
    int *misc = reinterpret_cast<int *>(smem + C::MISC_OFF);  // [0] tiles issued, [1] abort, [2] tiles landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc + 4);

    const int units = p.num_tiles * p.Hkv;
    const int s = blockIdx.x / units;
    const int rem = blockIdx.x - s * units;
    const int w = rem / p.Hkv;
    const int kvh = rem - w * p.Hkv;

    // Tensor memory touches nothing the previous kernel writes: it is allocated before the
    // wait below, overlapping that kernel's end.
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Programmatic dependent launch: nothing global is read before the wait.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int wb = p.tile_batch[w], wi = p.tile_index[w];
    const int bb = (wb >= 0 && wb < p.B) ? wb : 0;
    const int q0 = p.qo_indptr[bb], q1 = p.qo_indptr[bb + 1];
    const int Lraw = p.seq_lens[bb];
    const int R = p.box_rows;
    MultiTile tl;
    const bool live = multi_tile(p, wb, wi, q0, q1, Lraw, C::QT, threadIdx.x == 0 && s == 0 && kvh == 0, &tl);
    const int nsplit = live ? max(1, (tl.kv_end + p.chunk - 1) / p.chunk) : 0;
    const int tok0 = s * p.chunk;
    const int tok1 = live ? min(tl.kv_end, tok0 + p.chunk) : 0;
    const int ntiles = (live && s < nsplit && tok1 > tok0) ? (tok1 - tok0 + BT - 1) / BT : 0;
    const int J = 2 * ntiles;  // half tiles
    const bool work = live && s < nsplit;
    // Query row r = (token r / G, head r % G) sits in TMEM lane r; only the consumer warps
    // that hold rows of the tile's tokens run the softmax.  (M = 64 products for tiles of
    // at most 64 rows measured no faster: the products' cost is set by N.)
    const int nrows = work ? tl.ntok * G : 0;
    const int active = (nrows + 31) / 32;  // consumer warps holding rows
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], full_arrivals<C>());
            mbar_init(&empty[i], 1);  // one tcgen05.commit after the tile's last PV product
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_done[b], 1);
            mbar_init(&p_ready[b], (uint32_t)max(active, 1));  // one arrival per active warp
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&pv_done[b], 1);
            mbar_init(&fin[b], 1);
        }
        mbar_init(q_ready, NWC);
        misc[0] = misc[1] = misc[2] = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();  // barriers and the TMEM address are visible
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tQ = tmem + C::TQ, tO = tmem + C::TO;
    // Key k of column block cb of a stage's K or V tile sits at cb * CS + k * 128 (8-key
    // groups 1024 bytes apart).  S: K-major, 16 dims (32 bytes) per product step; PV: V
    // MN-major, 64 dims per swizzle atom (atoms CS apart), 16 keys per product step.
    constexpr uint32_t CS = BT * 128;
    constexpr uint32_t idS = idesc_bf16(128, HT, 0), idO = idesc_bf16(128, D, 1);

    if (work && warp == C::PRODUCER) {
        if (C::GATHER) {  // ---- producer warp, row gather
            if (C::MASK && lane == 0) prefetch_tensormap(&mapM);
            const int32_t *table = p.block_table + (long long)tl.b * p.max_pages;
            RowPages<C> rp_next;
            if (ntiles > 0) lookup_rows<C>(rp_next, table, tok0, min(BT, tok1 - tok0), p.page_size, lane);
            int issued = 0;
            for (int i = 0; i < ntiles; ++i) {
                const int st = i % NS;
                const RowPages<C> rp = rp_next;
                const int t = tok0 + i * BT;
                if (i + 1 < ntiles)
                    lookup_rows<C>(rp_next, table, t + BT, min(BT, tok1 - t - BT), p.page_size, lane);
                if (i >= NS && !__all_sync(0xFFFFFFFFu, mbar_wait(&empty[st], ((i / NS) - 1) & 1))) {
                    misc[1] = 1;
                    break;
                }
                // (with a mask: the tile's mask bytes by TMA, zeros past either end)
                fill_tile_rows<C>(smem + st * C::STAGE_BYTES, rp, min(BT, tok1 - t), kvh, p, (uint32_t)C::MASK_BYTES,
                                  [&] {
                                      if (C::MASK)
                                          tma_load_3d(smem + st * C::STAGE_BYTES + C::MASK_OFF, &mapM, t,
                                                      tl.q0 + tl.i0, 0, &full[st]);
                                  },
                                  &full[st], lane);
                issued = i + 1;
            }
            if (lane == 0) misc[0] = issued;
        } else {  // ---- producer warp: page lookup + TMA copies
            if (lane == 0) {
                prefetch_tensormap(&mapK);
                prefetch_tensormap(&mapV);
                if (C::MASK) prefetch_tensormap(&mapM);
            }
            const int32_t *table = p.block_table + (long long)tl.b * p.max_pages;
            auto lookup = [&](int tile) -> int {
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
                const int nbox = (min(BT, tok1 - t) + R - 1) / R;
                if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)(nbox * R * C::ROWB * 2 + C::MASK_BYTES));
                __syncwarp();
                // lane (box j, column block cb) copies rows [j R, (j + 1) R) of block cb;
                // the page id of box j is in lane j
                const int j = lane / C::NBLK, cb = lane % C::NBLK;
                const int pj = __shfl_sync(0xFFFFFFFFu, pg, j & 31);
                if (j < nbox) {
                    uint8_t *dst = smem + st * C::STAGE_BYTES + cb * CS + j * R * 128;
                    const int row = (t + j * R) % p.page_size;
                    tma_load_5d(dst, &mapK, 0, row, cb, kvh, pj, &full[st]);
                    tma_load_5d(dst + C::TILE_BYTES, &mapV, 0, row, cb, kvh, pj, &full[st]);
                }
                // the tile's mask bytes: keys [t, t + BT) of the tile's tokens (zeros past the ends)
                if (C::MASK && lane == 31)
                    tma_load_3d(smem + st * C::STAGE_BYTES + C::MASK_OFF, &mapM, t, tl.q0 + tl.i0, 0, &full[st]);
                issued = i + 1;
            }
            if (lane == 0) misc[0] = issued;
        }
    } else if (work && warp == C::S_ISSUER) {
        // ---- the S thread.  Half tile j (keys [32 (j & 1), +32) of tile j / 2) has its
        // scores in buffer j & 1; S(j) reuses the buffer PV(j - 2) reads P from, so it is
        // issued once that product has completed.  (One warp issues about one tcgen05.mma
        // per hundred cycles whatever N is, so the S and PV products have a warp each.)
        if (lane == 0) {
            bool ok = mbar_wait(q_ready, 0);
            int landed = 0;
            for (int j = 0; ok && j < J; ++j) {
                const int i = j >> 1, h = j & 1, st = i % NS;
                if (j >= 2 && !mbar_wait(&pv_done[h], ((j >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (h == 0) {
                    if (!mbar_wait(&full[st], (i / NS) & 1)) {
                        ok = false;
                        break;
                    }
                    landed = i + 1;
                }
                tc_fence_after();
                const uint32_t sK = smem_addr(smem + st * C::STAGE_BYTES) + h * HT * 128;
                const uint32_t tS = tmem + (h ? C::TS1 : C::TS0);
#pragma unroll
                for (int k16 = 0; k16 < D / 16; ++k16)
                    umma_bf16_tmem_a(tS, tQ + k16 * 8, sw128_desc(sK + (k16 >> 2) * CS + (k16 & 3) * 32, 16, 1024),
                                     idS, k16 > 0);
                umma_commit(&s_done[h]);
            }
            if (!ok) misc[1] = 1;
            misc[2] = landed;
            umma_commit(&fin[0]);  // this thread's products have completed when fin[0] completes
        }
        __syncwarp();
    } else if (work && warp == C::PV_ISSUER) {
        // ---- the PV thread: O += P(j) . V once the consumers have written P(j); the commit
        // after a tile's second half frees its stage (its S products completed before P)
        if (lane == 0) {
            bool ok = true;
            for (int j = 0; j < J; ++j) {
                const int i = j >> 1, h = j & 1, st = i % NS;
                if (!mbar_wait(&p_ready[h], (j >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int nv = min(HT, min(BT, tok1 - (tok0 + i * BT)) - h * HT);  // keys of this half
                const uint32_t sV = smem_addr(smem + st * C::STAGE_BYTES + C::TILE_BYTES) + h * HT * 128;
                const uint32_t tP = tmem + (h ? C::TS1 : C::TS0);
                for (int kk = 0; kk * 16 < nv; ++kk)
                    umma_bf16_tmem_a(tO, tP + kk * 8, sw128_desc(sV + kk * 2048, CS, 1024), idO, j > 0 || kk > 0);
                if (h == 1) umma_commit(&empty[st]);
                umma_commit(&pv_done[h]);
            }
            if (!ok) misc[1] = 1;
            umma_commit(&fin[1]);
        }
        __syncwarp();
    }

    // ---- consumer warps: thread r = query row r = TMEM lane r
    const int r = threadIdx.x;
    const int ti = r / G, hc = r - (r / G) * G;
    const bool rvalid = work && warp < NWC && r < nrows;
    const int lim = work ? tl.pos0 + ti : 0;  // the row's token sees keys at positions <= lim
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    float m_ref = -INFINITY, l = 0.f;
    if (work && warp < NWC) {
        {   // q row -> tensor memory (zeros for rows without a token)
            uint4 qv[D / 8];
            const __nv_bfloat16 *src =
                p.q + (long long)(tl.q0 + tl.i0 + ti) * p.q_sb + (long long)(kvh * G + hc) * p.q_sh;
#pragma unroll
            for (int c = 0; c < D / 8; ++c)
                qv[c] = rvalid ? __ldg(reinterpret_cast<const uint4 *>(src + 8 * c)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t x[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    x[4 * j] = qv[4 * c + j].x;
                    x[4 * j + 1] = qv[4 * c + j].y;
                    x[4 * j + 2] = qv[4 * c + j].z;
                    x[4 * j + 3] = qv[4 * c + j].w;
                }
                tmem_st16(tQ + lane_base + 16 * c, x);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        }
        // Rows are independent through both products, so a warp whose rows hold no token
        // skips the tiles: whatever its rows of P hold reaches only its own rows of O, which
        // are never stored.
        for (int j = 0; j < (warp < active ? J : 0); ++j) {
            const int i = j >> 1, h = j & 1, st = i % NS;
            const int t = tok0 + i * BT + h * HT;  // position of the half tile's first key
            const int nvalid = min(BT, tok1 - (tok0 + i * BT));
            const uint32_t tS = tmem + (h ? C::TS1 : C::TS0) + lane_base;
            // (the mask bytes are read by these threads: they see the stage land themselves)
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&s_done[h], (j >> 1) & 1) &&
                                             (!C::MASK || h == 1 || mbar_wait(&full[st], (i / NS) & 1)))) {
                misc[1] = 1;
                break;
            }
            tc_fence_after();
            {
                float sv[HT];
                {
                    uint32_t x[HT];
                    tmem_ld32_issue(tS, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < HT; ++k) sv[k] = __uint_as_float(x[k]);
                }
                // keys [0, klim) of the half tile are seen by this row; scores rounded once
                // (they feed the max and the exponent)
                const int klim = min(nvalid - h * HT, lim - t + 1);
                if (C::MASK) {  // the row's token's mask bytes of these 32 keys
                    uint4 mb[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
                    if (rvalid) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(smem + st * C::STAGE_BYTES + C::MASK_OFF +
                                                                           ti * BT + h * HT);
                        mb[0] = src[0];
                        mb[1] = src[1];
                    }
                    const uint32_t w[8] = {mb[0].x, mb[0].y, mb[0].z, mb[0].w, mb[1].x, mb[1].y, mb[1].z, mb[1].w};
#pragma unroll
                    for (int k = 0; k < HT; ++k) {
                        const bool keep = rvalid && k < klim && ((w[k >> 2] >> (8 * (k & 3))) & 0xFFu) != 0u;
                        sv[k] = keep ? __fmul_rn(sv[k], p.qscale) : -INFINITY;
                    }
                } else if (__all_sync(0xFFFFFFFFu, !rvalid || klim >= HT)) {
#pragma unroll
                    for (int k = 0; k < HT; ++k) sv[k] = __fmul_rn(sv[k], p.qscale);
                } else {
#pragma unroll
                    for (int k = 0; k < HT; ++k) sv[k] = (rvalid && k < klim) ? __fmul_rn(sv[k], p.qscale) : -INFINITY;
                }
                float m4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
                for (int k = 4; k < HT; ++k) m4[k & 3] = fmaxf(m4[k & 3], sv[k]);
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                // lazy reference move: the first finite max sets it; afterwards O and l are
                // rescaled only when the max passes the reference by more than 8 (base 2)
                float alpha = 1.f;
                if (rvalid && mx > m_ref) {
                    if (m_ref == -INFINITY) {
                        m_ref = mx;
                    } else if (mx - m_ref > 8.f) {
                        alpha = ex2(m_ref - mx);
                        m_ref = mx;
                        l *= alpha;
                    }
                }
                if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
                    // O holds PV(j - 1) once that product completes
                    const bool g =
                        __all_sync(0xFFFFFFFFu, mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1));
                    tc_fence_after();
                    if (!g) {
                        misc[1] = 1;
                        break;
                    }
#pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        float o[32];
                        tmem_ld32(tO + lane_base + c, o);
                        uint32_t y[16];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
#pragma unroll
                            for (int k = 0; k < 16; ++k) y[k] = __float_as_uint(o[16 * u + k] * alpha);
                            tmem_st16(tO + lane_base + c + 16 * u, y);
                        }
                    }
                }
                const float mu = m_ref == -INFINITY ? 0.f : m_ref;
                float l4[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t y[HT / 2];
#pragma unroll
                for (int k = 0; k < HT / 2; ++k) {
                    y[k] = pack_bf16x2(ex2(sv[2 * k] - mu), ex2(sv[2 * k + 1] - mu));
                    const float2 f = bf16x2_to_float2(y[k]);
                    l4[k & 3] += f.x + f.y;  // the weights the PV product uses
                }
                tmem_st16(tS, y);
                l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
            }
            const int end = nvalid - h * HT;  // the tile's end within this half, if it is here
            if (end > 0 && end < HT && end % 16 != 0) {
                // V rows end .. (rounded up to 16) enter the product with zero weights: zero
                // them so that 0 * V stays 0
                const int nz = 16 - end % 16;
                for (int e = threadIdx.x; e < nz * C::NBLK * C::CPB; e += active * 32) {
                    const int row = h * HT + end + e / (C::NBLK * C::CPB);
                    *reinterpret_cast<uint4 *>(smem + st * C::STAGE_BYTES + C::TILE_BYTES +
                                               tile_off<C>(row, e % (C::NBLK * C::CPB), 6)) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_async_smem();
            }
            __syncwarp();
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_ready[h]);
        }
    }
    __syncthreads();
    if (warp < NWC && work) {
        // every product has completed once both fin barriers have (each issuing thread
        // commits its own last)
        const bool g = __all_sync(0xFFFFFFFFu, mbar_wait(&fin[0], 0) && mbar_wait(&fin[1], 0));
        tc_fence_after();
        if (g && misc[1] == 0 && __any_sync(0xFFFFFFFFu, rvalid)) {  // (tcgen05.ld is warp-wide)
            const long long rq = tl.q0 + tl.i0 + ti;
            const int hq = kvh * G + hc;
            const bool direct = nsplit == 1;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const long long prow = (rq * p.num_splits + s) * p.Hq + hq;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                float o[32];
                if (J > 0) {
                    __syncwarp();
                    tmem_ld32(tO + lane_base + c, o);
                } else {  // no key in range: zero rows
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = 0.f;
                }
                if (rvalid && direct) {
                    __nv_bfloat16 *dst = p.out + rq * p.o_sb + (long long)hq * p.o_sh + c;
#pragma unroll
                    for (int k = 0; k < 32; k += 8)
                        *reinterpret_cast<uint4 *>(dst + k) =
                            make_uint4(pack_bf16x2(o[k] * inv, o[k + 1] * inv), pack_bf16x2(o[k + 2] * inv, o[k + 3] * inv),
                                       pack_bf16x2(o[k + 4] * inv, o[k + 5] * inv),
                                       pack_bf16x2(o[k + 6] * inv, o[k + 7] * inv));
                } else if (rvalid) {
                    float *dst = p.o_part + prow * D + c;
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        *reinterpret_cast<float4 *>(dst + k) = make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]);
                }
            }
            if (!direct && rvalid) *reinterpret_cast<float2 *>(p.ml_part + prow * 2) = make_float2(m_ref, l);
        }
        if (threadIdx.x == 0 && misc[1]) {
            // A wait gave up: let the copies still in flight land (bounded) before the shared
            // memory is released (the products have, with the fin barriers).
            for (int i = misc[2]; i < misc[0]; ++i) (void)mbar_wait(&full[i % NS], (i / NS) & 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
    }
}

// The paged cache [pages][page rows][Hkv][D] viewed as [64 dims, rows, column block, kv
// head, page] (as encode_cache_map), with a box of one column block: R rows x 128 bytes.
bool encode_block_map(CUtensorMap *map, const void *base, int D, int Hkv, int page_size, int num_pages, int R) {
    const cuuint64_t dims[5] = {64u, (cuuint64_t)page_size, (cuuint64_t)(D / 64), (cuuint64_t)Hkv,
                                (cuuint64_t)num_pages};
    const cuuint64_t strides[4] = {(cuuint64_t)Hkv * D * 2, 128u, (cuuint64_t)D * 2,
                                   (cuuint64_t)page_size * Hkv * D * 2};
    const cuuint32_t box[5] = {64u, (cuuint32_t)R, 1u, 1u, 1u};
    return encode_bf16(map, base, 5, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int D, int G, bool MASK, bool GATHER>
dap_status launch_multi_tc(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    using C = TcCfg<D, G, MASK, GATHER>;
    const int R = GATHER ? C::BT : gcd_int(a.page_size, C::BT);
    p.box_rows = R;
    CUtensorMap mk = {}, mv = {};  // (the row-gather producer reads the cache directly)
    if (!GATHER && (!encode_block_map(&mk, a.k, a.D, a.Hkv, a.page_size, a.num_pages, R) ||
                    !encode_block_map(&mv, a.v, a.D, a.Hkv, a.page_size, a.num_pages, R)))
        return DAP_ERR_CUDA;
    CUtensorMap mm = {};
    if (MASK && !encode_mask_map(&mm, a.mask, a.mask_stride, a.total_q, C::QT, C::BT)) return DAP_ERR_CUDA;
    auto kern = multi_tc_kernel<C>;
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

template <int D, bool MASK, bool GATHER>
dap_status dispatch_tc_g(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    switch (a.Hq / a.Hkv) {
        case 1: return launch_multi_tc<D, 1, MASK, GATHER>(a, p, stream);
        case 2: return launch_multi_tc<D, 2, MASK, GATHER>(a, p, stream);
        case 4: return launch_multi_tc<D, 4, MASK, GATHER>(a, p, stream);
        case 8: return launch_multi_tc<D, 8, MASK, GATHER>(a, p, stream);
    }
    return DAP_ERR_UNSUPPORTED;
}

template <bool MASK, bool GATHER>
dap_status dispatch_tc(const DecodeArgs &a, cudaStream_t stream) {
    SplitParams p = make_params(a);
    switch (a.D) {
        case 64: return dispatch_tc_g<64, MASK, GATHER>(a, p, stream);
        case 128: return dispatch_tc_g<128, MASK, GATHER>(a, p, stream);
        case 256: return dispatch_tc_g<256, MASK, GATHER>(a, p, stream);
    }
    return DAP_ERR_UNSUPPORTED;
}

}  // namespace

// Multi-token decode with 128 / G tokens per work tile (D 64 or 128; with or without a mask).
dap_status launch_decode_multi_tc(const DecodeArgs &a, cudaStream_t stream) {
    const bool gather = a.page_size % 8 != 0;
    if (a.mask) return gather ? dispatch_tc<true, true>(a, stream) : dispatch_tc<true, false>(a, stream);
    return gather ? dispatch_tc<false, true>(a, stream) : dispatch_tc<false, false>(a, stream);
}

bool read_errors_multi_tc(unsigned int *flags, bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_errors, sizeof v) != cudaSuccess) return false;
    if (clear) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_device_errors, &z, sizeof z) != cudaSuccess) return false;
    }
    *flags |= v;
    return true;
}

}  // namespace dap
