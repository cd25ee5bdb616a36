// dap_fp8.cu -- fp8 (e4m3) sliding-window latent decode attention, K = V, on the
// sm_100-family tensor cores (tcgen05, accumulators in tensor memory).
//
// Operation (nvfp4-megamoe-kernel native_swa_decode.py, native_swa_decode_attention and
// _fallback_batched_sdp): for decode token t the window slots are slot_idx[t, j], j < W; a
// slot takes part iff j < lens[t] and slot >= 0; its row is
//     kv_j = bf16( e4m3(kv_cache[slot / bs, slot % bs, :]) * inv_scale[slot] )
// and keys and values are the same rows.  Every query head h of the token attends to them:
//     out[t, h] = sum_j softmax_j(scale * q[t, h] . kv_j) kv_j.
// A token with no row gives a zero row (the page's kernel stub normalises only when the
// row sum is nonzero).
//
// Why tensor cores: 128 query heads share every row, so QK^T and PV are dense GEMMs with
// M = 128 heads (the page's stub groups heads per CTA for the same reason and imports the
// tcgen05 module, but leaves the tile loop empty).
//
// One CTA per (token, head group of 128, half of HD):
//   1. q[t, heads, :] streams in by TMA (128B swizzle, eight 64-wide blocks through a
//      4-stage ring started at entry) and moves on into tensor memory (head = TMEM lane, two
//      bf16 per column): blocks 0..3 while the rows travel, 4..7 (the ring refilled
//      meanwhile) after step 2;
//   2. every warp loads the slots of every eighth window position and, right after, the rows
//      of its kept positions (a half-warp per 256-byte half of a row) with their inverse
//      scales: two dependent round trips; the rows are dequantised (e4m3 -> f16 -> f32,
//      times the f32 inverse scale, rounded once to bf16: the same single rounding the
//      page's fallback does) into a 128-byte-swizzled [hd block][row][64] tile in shared
//      memory, rows in warp order;
//      rows n..n16-1 are zero (n16 = n rounded up to 16);
//   3. one thread issues S = Q . KV^T (M=128, N=n16, K=512) into TMEM, A (q) read from
//      tensor memory, B (the rows) from shared memory;
//   4. two threads own each head (one TMEM lane, alternate 32-column chunks of the scores):
//      base-2 softmax over its n scores, the probabilities rounded to bf16 into a swizzled
//      P tile, l = their sum;
//   5. O[:, half] = P . KV[:, half] (M=128, N=256, K=n16) reads the same KV tile as an
//      MN-major operand, into the tensor-memory columns q held;
//   6. out = O / l in bf16.
// Holding q in tensor memory (the ring only passes it through) leaves shared memory to a
// whole 128-row KV tile, so no window waits for q blocks to be refilled after its first
// products.  The two CTAs of a token recompute S (cheap on tensor
// cores) so that O's 256 fp32 columns and S's columns fit tensor memory together.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "dap_device.cuh"
#include "dap_internal.h"
#include "dap_tc.cuh"

namespace dap {

bool read_errors_fp8(unsigned int *flags, bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_errors, sizeof v) != cudaSuccess) return false;
    if (clear) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_device_errors, &z, sizeof z) != cudaSuccess) return false;
    }
    *flags |= v;
    return true;
}

namespace fp8 {

constexpr int kHD = 512;            // latent width
constexpr int kHeads = 128;         // heads per CTA = MMA M
constexpr int kMaxRows = 128;       // window rows a CTA holds
constexpr int kHalf = kHD / 2;      // output columns per CTA
constexpr int kThreads = 256;       // 8 warps: warps w and w+4 share TMEM lanes
constexpr int kQStages = 4;
// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int kQOff = 0;                                    // q ring: 4 stages of 128 heads x 64
constexpr int kQStage = kHeads * 128;                       // 16 KB per stage
constexpr int kPOff = kQOff;                                // P: 2 blocks of 128 heads x 64, after q
constexpr int kKvOff = kQOff + kQStages * kQStage;          // 65536: KV tile [8 blocks][n16 rows][128 B]
constexpr int kOOff = kKvOff;                               // bf16 output staging after PV (64 KB)
constexpr int kPBlock = kHeads * 128;                       // 16 KB per 64-wide row block
constexpr int kXchOff = kKvOff + 8 * kMaxRows * 128;        // softmax max/sum exchange (2 KB)
constexpr int kCntOff = kXchOff + 4 * kHeads * 4;           // per-warp row counts [0..7], abort [12]
constexpr int kBarOff = kCntOff + 64;                       // mbarriers
constexpr int kNumBars = kQStages + 2;                      // q_full[4], mma_done[2]
constexpr int kTmemOff = kBarOff + kNumBars * 8;
constexpr int kSmemUsed = kTmemOff + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;                // slack to align the base
constexpr int kTmemCols = 512;  // q: cols [0,256) (two bf16 per column) until S is complete,
                                // then O: [0,256); S: [256,384)
constexpr int kSCol = 256;
static_assert(kOOff + kHeads * kHalf * 2 <= kXchOff, "the output staging fits in the KV tile");
static_assert(kPOff + 2 * kPBlock <= kKvOff, "P fits in the q ring");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

// Byte offset of 16-byte chunk `k` (0..7) of row `r` in a 128-byte-swizzled tile whose
// rows are 128 bytes apart (chunk k of row r sits at chunk k ^ (r mod 8)).
__device__ __forceinline__ uint32_t sw128_off(int r, int k) {
    return (uint32_t)r * 128u + ((uint32_t)(k ^ (r & 7)) << 4);
}

struct Params {
    const uint8_t *kv_cache;
    const __nv_bfloat16 *inv_scale;
    const int64_t *slot_idx;
    const int64_t *lens;
    __nv_bfloat16 *out;
    int T, NH, W;
    long long max_slots;
    float qscale;  // scale * log2(e)
};


// Moves the four q blocks of ring round `round` (blocks 4 round .. 4 round + 3) into tensor
// memory: thread (head h, half c) waits for each stage, reads its 32 values (64 bytes, four
// 128B-swizzled chunks) of row h and stores them at columns 32 block + 16 c of lane h (two
// bf16 per column, the lower index in the low half).  A wait that gives up sets the abort
// word; the caller still reaches every barrier.
__device__ __forceinline__ void q_to_tmem(uint8_t *smem, uint64_t *q_full, uint32_t tmem_lane, int h, int c,
                                          int round, int *cnt) {
#pragma unroll
    for (int st = 0; st < kQStages; ++st) {
        if (!mbar_wait(&q_full[st], round & 1)) cnt[12] = 1;
        const uint8_t *blk = smem + kQOff + st * kQStage;
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = *reinterpret_cast<const uint4 *>(blk + sw128_off(h, 4 * c + i));
            r[4 * i] = v.x;
            r[4 * i + 1] = v.y;
            r[4 * i + 2] = v.z;
            r[4 * i + 3] = v.w;
        }
        tmem_st16(tmem_lane + (round * kQStages + st) * 32 + 16 * c, r);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    swa_kernel(const __grid_constant__ CUtensorMap qmap, const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte swizzle is a function of address bits 4..9: tiles start 1024-aligned
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col_half = blockIdx.x;    // which 256 output columns
    const int hg = blockIdx.y;          // head group of 128
    const int t = blockIdx.z;           // decode token
    int *cnt = reinterpret_cast<int *>(smem + kCntOff);     // [0..7] warp counts, [12] abort
    uint64_t *q_full = reinterpret_cast<uint64_t *>(smem + kBarOff);
    uint64_t *mma_done = q_full + kQStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kTmemOff);

    // thread = (head hrow = TMEM lane, half qhalf of q's 512 values / of the score columns):
    // warps w and w + 4 serve the same 32 lanes
    const int hrow = tid & (kHeads - 1);
    const int chalf = warp >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int qrow = t * p.NH + hg * kHeads;

    // Barriers and tensor memory touch nothing the previous kernel writes: they are set up
    // before the wait below, overlapping that kernel's end.
    if (tid == 0) {
        for (int i = 0; i < kQStages; ++i) mbar_init(&q_full[i], 1);
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        cnt[12] = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Launched as a programmatic dependent of the previous kernel on the stream: nothing
    // global is read before the wait (that kernel may still write q, the cache or the
    // slot table); the next launch may start at once (it waits the same way).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // ---- 1a. q's first four 64-wide blocks, right away: they travel during the compaction
    if (tid == 0) {
        for (int kb = 0; kb < kQStages; ++kb) {
            mbar_arrive_expect_tx(&q_full[kb], kQStage);
            tma_load_2d(smem + kQOff + kb * kQStage, &qmap, kb * 64, qrow, &q_full[kb]);
        }
    }

    // ---- 1b. the window's slots and length; 2. the kept rows and their inverse scales --------
    // Warp w holds window positions w, w + 8, ..., w + 120 (lanes l and l + 16 the same
    // one), so every warp holds about an eighth of any window's rows.  Each warp loads the
    // rows of its kept positions into registers right after the slots, a half-warp per
    // 256-byte half of a row (16 codes per lane), with their inverse scales: two dependent
    // round trips in all before the rows are in registers.
    const int jpos = warp + 8 * (lane & 15);
    long long slot = -1;
    if (jpos < p.W) slot = p.slot_idx[(long long)t * p.W + jpos];
    long long len = p.lens[t];
    len = len < 0 ? 0 : (len > p.W ? p.W : len);
    bool keep = false;
    if (jpos < len) {
        if (slot >= p.max_slots) {
            if (lane < 16) flag_error(DAP_DEVERR_SLOT);
            slot = -1;
        }
        keep = slot >= 0;
    }
    const uint32_t ball = __ballot_sync(0xFFFFFFFFu, keep) & 0xFFFFu;
    uint4 raw[16];
    float invf = 0.f;
    if (keep) invf = __bfloat162float(p.inv_scale[slot]);
    const uint8_t *piece = p.kv_cache + (lane & 15) * 16 + (lane >> 4) * 256;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const long long s = __shfl_sync(0xFFFFFFFFu, slot, i);
        raw[i] = make_uint4(0u, 0u, 0u, 0u);
        if ((ball >> i) & 1u) raw[i] = __ldg(reinterpret_cast<const uint4 *>(piece + s * kHD));
    }
    if (lane == 0) cnt[warp] = __popc(ball);
    tc_fence_before();
    __syncthreads();  // the counts and the TMEM address are visible
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int base = 0, n = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const int c = cnt[w];
        base += w < warp ? c : 0;
        n += c;
    }
    const int n16 = (n + 15) & ~15;
    const int kvb = n16 * 128;  // bytes per 64-wide hd block of the KV tile

    // While the rows travel, q blocks 0..3 move from the ring into tensor memory and thread
    // 0 refills the ring with blocks 4..7 once every thread has read its stage.
    q_to_tmem(smem, q_full, tmem + lane_base, hrow, chalf, 0, cnt);
    __syncthreads();  // the ring is read
    if (tid == 0) {
        for (int kb = 0; kb < kQStages; ++kb) {
            mbar_arrive_expect_tx(&q_full[kb], kQStage);
            tma_load_2d(smem + kQOff + kb * kQStage, &qmap, (kb + kQStages) * 64, qrow, &q_full[kb]);
        }
    }
    // dequantise the rows into the swizzled KV tile (e4m3 -> f16 exactly, to f32, times the
    // inverse scale: the product of a 4-bit and an 8-bit significand is exact in fp32, then
    // one bf16 rounding, the page's fallback's one rounding), rows in warp order (the result
    // does not depend on the rows' order beyond rounding)
    {
        const int blk = (lane & 15) / 4 + 4 * (lane >> 4);  // 64-wide hd block of this piece
        const int k0 = ((lane & 15) % 4) * 2;               // first 16-byte chunk in the 128-byte row
        uint8_t *tile = smem + kKvOff + blk * kvb;
        int r = base;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float inv = __shfl_sync(0xFFFFFFFFu, invf, i);
            if ((ball >> i) & 1u) {
                uint32_t o[8];
                const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)((w4[q] >> (16 * jj)) & 0xFFFFu);
                        const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
                        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * inv, f.y * inv);
                        o[2 * q + jj] = *reinterpret_cast<const uint32_t *>(&b);
                    }
                }
                *reinterpret_cast<uint4 *>(tile + sw128_off(r, k0)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4 *>(tile + sw128_off(r, k0 + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
                ++r;
            }
        }
        // rows n .. n16 - 1 take part in the products as zeros
        for (int idx = tid; idx < (n16 - n) * 64; idx += kThreads) {
            const int rr = n + idx / 64, c = idx % 64;
            *reinterpret_cast<uint4 *>(smem + kKvOff + (c >> 3) * kvb + sw128_off(rr, c & 7)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    }
    q_to_tmem(smem, q_full, tmem + lane_base, hrow, chalf, 1, cnt);  // blocks 4..7
    tmem_wait_st();  // this thread's q columns are in tensor memory
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tS = tmem + kSCol;
    // ---- 3. S = Q . KV^T, one thread issues; A = q from tensor memory ------------------------
    if (tid == 0 && n > 0) {
        const uint32_t idS = idesc_bf16(kHeads, n16, 0);
        for (int kb = 0; kb < 8; ++kb) {
            const uint32_t kva = smem_addr(smem + kKvOff + kb * kvb);
#pragma unroll
            for (int k16 = 0; k16 < 4; ++k16)  // 16 values = 8 columns of q per product
                umma_bf16_tmem_a(tS, tmem + kb * 32 + k16 * 8, sw128_desc(kva + 32 * k16, 16, 1024), idS,
                                 (kb | k16) != 0);
        }
        umma_commit(&mma_done[0]);
    }

    // ---- 4. softmax: thread = head = TMEM lane, 32-column chunks chalf, chalf + 2 ---------------
    bool waited = true;
    if (n > 0) waited = mbar_wait(&mma_done[0], 0);
    const int good = __syncthreads_and(waited && cnt[12] == 0);
    tc_fence_after();
    float *xch = reinterpret_cast<float *>(smem + kXchOff);  // [2][128] max, then [2][128] sum
    float l = 0.f;
    if (good && n > 0) {
        float v[2][32];
        float m = -INFINITY;
        {   // both chunks' loads in flight together (columns n .. n16 - 1 are read but masked)
            uint32_t r[2][32];
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (32 * (chalf + 2 * u) < n16) tmem_ld32_issue(tS + lane_base + 32 * (chalf + 2 * u), r[u]);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int i = 0; i < 32; ++i) v[u][i] = __uint_as_float(r[u][i]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int c0 = 32 * (chalf + 2 * u);
            if (c0 < n16) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (c0 + i < n) m = fmaxf(m, __fmul_rn(v[u][i], p.qscale));
            }
        }
        xch[chalf * kHeads + hrow] = m;
        __syncthreads();
        m = fmaxf(xch[hrow], xch[kHeads + hrow]);
        float lp = 0.f;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int c0 = 32 * (chalf + 2 * u);
            if (c0 < n16) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int j0 = c0 + 8 * g;
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float p0 = (j0 + e < n) ? ex2(__fmul_rn(v[u][8 * g + e], p.qscale) - m) : 0.f;
                        const float p1 = (j0 + e + 1 < n) ? ex2(__fmul_rn(v[u][8 * g + e + 1], p.qscale) - m) : 0.f;
                        const __nv_bfloat162 b = __floats2bfloat162_rn(p0, p1);
                        const float2 r2 = __bfloat1622float2(b);
                        lp += r2.x + r2.y;  // the sum of the weights PV actually uses
                        pk[e / 2] = *reinterpret_cast<const uint32_t *>(&b);
                    }
                    uint8_t *tile = smem + kPOff + (j0 >> 6) * kPBlock;
                    *reinterpret_cast<uint4 *>(tile + sw128_off(hrow, (j0 & 63) >> 3)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
        }
        xch[2 * kHeads + chalf * kHeads + hrow] = lp;
        __syncthreads();
        l = xch[2 * kHeads + hrow] + xch[3 * kHeads + hrow];
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- 5. O[:, half] = P . KV[:, half], into the columns q held (S is complete) --------------
    if (tid == 0 && good && n > 0) {
        const uint32_t idO = idesc_bf16(kHeads, kHalf, 1);
        const uint32_t pa = smem_addr(smem + kPOff);
        const uint32_t kvh = smem_addr(smem + kKvOff + col_half * 4 * kvb);
        for (int k16 = 0; k16 < n16 / 16; ++k16)
            umma_bf16(tmem, sw128_desc(pa + (k16 >> 2) * kPBlock + (k16 & 3) * 32, 16, 1024),
                      sw128_desc(kvh + k16 * 2048, (uint32_t)kvb, 1024), idO, k16 > 0);
        umma_commit(&mma_done[0]);
    }
    bool waited2 = true;
    if (good && n > 0) waited2 = mbar_wait(&mma_done[0], 1);
    const int good2 = __syncthreads_and(good && waited2);
    tc_fence_after();

    // ---- 6. out = O / l --------------------------------------------------------------------------
    // Each thread turns half of its head's 256 columns into bf16 in a staging area (the KV
    // tile, read by no one now; 16-byte chunk c of row h at chunk c ^ (h mod 32),
    // conflict-free both ways); then the CTA writes the 128 rows out with fully coalesced
    // 16-byte stores.
    if (good2) {
        uint8_t *ostage = smem + kOOff;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        for (int c0 = chalf * (kHalf / 2); c0 < (chalf + 1) * (kHalf / 2); c0 += 64) {
            float v[64];
            if (n > 0) {
                tmem_ld64(tmem + lane_base + c0, v);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) v[i] = 0.f;
            }
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                uint32_t pk[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) pk[i] = pack_bf16(v[8 * q8 + 2 * i] * inv, v[8 * q8 + 2 * i + 1] * inv);
                const int ch = c0 / 8 + q8;  // 0..31
                *reinterpret_cast<uint4 *>(ostage + hrow * (kHalf * 2) + ((ch ^ (hrow & 31)) << 4)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
        __syncthreads();
        __nv_bfloat16 *obase = p.out + ((long long)t * p.NH + hg * kHeads) * kHD + col_half * kHalf;
        for (int idx = tid; idx < kHeads * 32; idx += kThreads) {
            const int row = idx >> 5, ch = idx & 31;
            const uint4 val = *reinterpret_cast<const uint4 *>(ostage + row * (kHalf * 2) + ((ch ^ (row & 31)) << 4));
            *reinterpret_cast<uint4 *>(obase + (long long)row * kHD + ch * 8) = val;
        }
    } else if (tid == 0) {
        // A wait gave up.  Let the copies and products still in flight land (bounded) before
        // the tensor memory and the shared memory are released.
        for (int i = 0; i < kQStages; ++i) (void)mbar_wait(&q_full[i], 1);
        umma_commit(&mma_done[1]);
        (void)mbar_wait(&mma_done[1], 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace fp8

dap_status launch_fp8(const Fp8Args &a, cudaStream_t stream) {
    typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                      const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                      CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);
    EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) return DAP_ERR_CUDA;
    // q as a [T*NH, 512] bf16 matrix; a box is 128 heads x 64 values (128 bytes), swizzled
    CUtensorMap qmap;
    const cuuint64_t dims[2] = {(cuuint64_t)fp8::kHD, (cuuint64_t)a.T * a.NH};
    const cuuint64_t strides[1] = {(cuuint64_t)fp8::kHD * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)fp8::kHeads};
    const cuuint32_t estr[2] = {1u, 1u};
    if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DAP_ERR_CUDA;
    fp8::Params p;
    p.kv_cache = a.kv_cache;
    p.inv_scale = static_cast<const __nv_bfloat16 *>(a.inv_scale);
    p.slot_idx = a.slot_idx;
    p.lens = a.lens;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.T = a.T;
    p.NH = a.NH;
    p.W = a.W;
    p.max_slots = (long long)a.num_blocks * a.block_size;
    p.qscale = a.scale * 1.4426950408889634f;
    if (cudaFuncSetAttribute(fp8::swa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fp8::kSmemBytes) !=
        cudaSuccess)
        return DAP_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, a.NH / fp8::kHeads, a.T);
    cfg.blockDim = dim3(fp8::kThreads);
    cfg.dynamicSmemBytes = fp8::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fp8::swa_kernel, qmap, p) != cudaSuccess) return DAP_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DAP_OK : DAP_ERR_CUDA;
}

}  // namespace dap
