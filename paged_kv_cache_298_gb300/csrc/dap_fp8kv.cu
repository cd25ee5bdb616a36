// dap_fp8kv.cu -- GQA decode attention over a paged e4m3 (fp8) K/V cache.
//
// Operation: the paged GQA decode of dap_decode.cu with K and V stored as OCP e4m3 codes
// [num_pages, page_size, Hkv, D] (D in {64, 128, 256}) and one bf16 dequantisation factor
// per (slot, kv head)
// for each, laid out [num_pages, Hkv, page_size]: the key of logical position t is
// e4m3(code) * factor (the decode side of the fp8 cache convention of
// nvfp4-megamoe-kernel native_swa_decode.py, applied per kv head), likewise the value.
//
// Schedule and data movement: the per-sequence split schedule of dap_decode.cu (one CTA
// per (sequence, pair of kv heads, split), split partials merged by the shared combine
// kernel; one kv head per CTA at D = 256 or an odd Hkv).  Code rows are stored in lines of
// LB = min(D, 128) bytes (two column blocks at D = 256), 128-byte swizzled (64-byte at
// D = 64).  Page sizes that are multiples of 8: per 64-key tile the producer warp issues,
// per page run, TMA boxes of the K and V code rows of the CTA's kv heads and the factor
// runs of those heads, which the [pages, Hkv, page_size] layout keeps contiguous.  Other
// page sizes: the producer copies every code row in 16-byte cp.async chunks to its
// swizzled position and stores the factors it loaded one tile earlier (the row gather of
// the bf16 kernels).  At D = 128 a stage carries as many bytes as a bf16 stage of one kv
// head, so three stages at two CTAs per SM keep the same bytes in flight.
//
// Arithmetic (tensor cores, mma.m16n8k16 in f16): every e4m3 value is an f16 value, so the
// hardware conversion (two e4m3 codes -> one f16 pair) turns codes into operands exactly,
// straight from the swizzled tile.  QK: A = the codes of 16 keys (lane t holding D / 4
// consecutive dims of every line block), B = q in f16 in the same dim order; the factor
// of each key and the softmax scale are applied to the fp32 scores (scale after the dot
// product, as the AstrAI csrc log's numerics commit asks); q is converted to f16 after an
// exact power-of-two shift that keeps its largest element below 2^15 (the shift goes back
// into the scale).  PV: the A operand wants pairs of keys of one dim, so each lane reads
// DPL = D / 8 dims of four key rows and byte-interleaves two keys' codes before the
// conversion (dims DPL g + 2m, DPL g + 2m + 1 in rows g, g+8 of step m); the probabilities
// times each key's V factor
// form the f16 B operand, measured in a per-warp power-of-two unit (above the largest
// factor seen so far) so they stay within [0, 1); the accumulator is rescaled exactly when
// the unit grows and multiplied back at the end.
#include "dap_tile.cuh"

namespace dap {
namespace f8kv {

// Four e4m3 codes [c0 c1 c2 c3] (low byte first) -> the f16 pairs (c0, c1) and (c2, c3),
// exactly (the NaN codes 0x7F / 0xFF become f16 NaNs; the cache writers never produce them)
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// 2^(E - 127) for a biased exponent E in 1..254 (exact)
__device__ __forceinline__ float pow2_biased(int E) { return __int_as_float(E << 23); }

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// HG kv heads per CTA (2 when Hkv is even and D <= 128): one TMA box carries both heads'
// rows of a page run and the shared tile is [column block][box][head][row][LB bytes].
// Consumer warp w serves the 16-key slice w % 4 of every tile for HPW kv heads (the heads as
// independent streams), so a CTA runs 4 * HG / HPW consumer warps.  GATHER: page sizes that
// are not multiples of 8, the tile filled row by row as one box of BT rows.
template <int D_, int G_, int HG_, bool GATHER_ = false, int HPW_ = 1>
struct Cfg {
    static constexpr int D = D_, G = G_, HG = HG_, HPW = HPW_, KW = 4, NWC = KW * (HG / HPW), BT = 64;
    static constexpr bool GATHER = GATHER_;
    static constexpr bool SWZ = true;
    static constexpr int LB = D < 128 ? D : 128;          // bytes of a code line (one row block)
    static constexpr int NB = D / LB;                     // line blocks per code row
    static constexpr int CODE_BLK = BT * HG * LB;         // one line block of a code tile
    static constexpr int CODE_BYTES = NB * CODE_BLK;      // one tile of K (or V) codes
    static constexpr bool BIG = 2 * CODE_BYTES >= 32768;  // stage near 33 KB: 3 stages, 2 CTAs / SM
    static constexpr int NS = BIG ? 3 : 4, MINB = BIG ? 2 : 3;
    static constexpr int THREADS = (NWC + 1) * 32;
    static constexpr int KPW = BT / KW;                   // 16 keys per consumer warp
    // The tile's K factors, then its V factors: box j (HG x R factors, R <= 64) lands in its
    // own slot, a tensor copy's shared destination being 128-byte aligned.
    static constexpr int FSLOT = 128 * HG;
    static constexpr int KS_OFF = 2 * CODE_BYTES;
    static constexpr int VS_OFF = KS_OFF + (BT / 8) * FSLOT;   // at most BT / 8 boxes (R >= 8)
    static constexpr int STAGE_BYTES = (VS_OFF + (BT / 8) * FSLOT + 1023) & ~1023;
    static constexpr int MRG_BYTES = KW * HG * G * (D / 2 + 2) * 4;  // aliases stage 0 after the last tile
    static constexpr int MISC_OFF = NS * STAGE_BYTES;
    static constexpr int BAR_OFF = MISC_OFF + 16;
    static constexpr int SMEM = BAR_OFF + 2 * NS * 8 + 1024;
    static_assert(KPW == 16 && HG % HPW == 0 && MRG_BYTES <= STAGE_BYTES && FSLOT >= 2 * HG * BT, "fp8 tiling");
    static_assert((D == 64 || D == 128 || D == 256) && (D <= 128 || HG == 1), "fp8 head dims");
};

template <class C>
struct Consumer {
    static constexpr int D = C::D, G = C::G, HG = C::HG, HW = C::HPW, KS = D / 16;
    static constexpr int LB = C::LB, NB = C::NB, WPB = LB / 16;  // QK code words per lane per line block
    static constexpr int DPL = D / 8, VW = D / 32;               // PV: dims per lane, code words per key row
    // QK dim order: word m of a lane's codes = dims qdim(m) .. qdim(m) + 3
    static __device__ __forceinline__ int qdim(int m, int t) { return (m / WPB) * LB + t * (LB / 4) + 4 * (m % WPB); }
    uint32_t qb[HW][KS][2];  // q (f16) B fragments of head g of each kv head: dims qdim(m)+0, 1 | +2, 3
    float acc[HW][KS][4];    // O^T: dims DPL g + 2m, +1 x heads 2t, 2t+1, in units of 2^(vE-127)
    float m_run[HW][2], l_run[HW][2];
    float qscale[HW];        // scale * log2(e) * 2^qshift
    int vE[HW];              // biased exponent of the V-factor unit (0 = none yet)
    int warp, lane, g, t, kw, hw0, key0;  // key slice kw, first kv head hw0 (within the CTA's HG)
    int line0, line1;        // 128-byte line of keys g, g+8 of head hw0 inside a code tile
    int vline0, vline2;      // lines of keys 2t and 2t+8 of head hw0 (keys 2t+1, 2t+9: the next lines)
    int f0, f1;              // byte offsets of the factors of keys g, g+8 of head hw0 in a factor block
    int hline, hfac;         // per-head strides of the two (R lines, 2R bytes)

    // R: rows per TMA box (a power of two, 8..64)
    __device__ __forceinline__ void init(int w, int l, int R) {
        warp = w;
        lane = l;
        g = l >> 2;
        t = l & 3;
        kw = w % C::KW;
        hw0 = (w / C::KW) * HW;
        key0 = kw * C::KPW;
        const int rb = __ffs(R) - 1;
        const int r0 = key0 + g, r1 = r0 + 8;
        line0 = (r0 >> rb) * (HG * R) + (r0 & (R - 1));
        line1 = (r1 >> rb) * (HG * R) + (r1 & (R - 1));
        // an even row and the next one share a box (boxes are multiples of 8 rows)
        const int r2 = key0 + 2 * t, r3 = r2 + 8;
        vline0 = (r2 >> rb) * (HG * R) + (r2 & (R - 1));
        vline2 = (r3 >> rb) * (HG * R) + (r3 & (R - 1));
        f0 = (r0 >> rb) * C::FSLOT + (r0 & (R - 1)) * 2;
        f1 = (r1 >> rb) * C::FSLOT + (r1 & (R - 1)) * 2;
        hline = R;
        hfac = 2 * R;
        line0 += hw0 * hline;
        line1 += hw0 * hline;
        vline0 += hw0 * hline;
        vline2 += hw0 * hline;
        f0 += hw0 * hfac;
        f1 += hw0 * hfac;
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int h = 0; h < HW; ++h) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                m_run[h][j] = -INFINITY;
                l_run[h][j] = 0.f;
            }
#pragma unroll
            for (int m = 0; m < KS; ++m)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[h][m][j] = 0.f;
            vE[h] = 0;
        }
    }

    // q of the G query heads of the warp's kv head h (head g at base + g * hstride);
    // qs = scale * log2(e).
    __device__ __forceinline__ void load_q(int h, const __nv_bfloat16 *base, long long hstride, float qs) {
        constexpr int NQ = D / 8;  // bf16 pairs of a lane: LB / 4 dims of every line block
        uint32_t w[NQ];
#pragma unroll
        for (int i = 0; i < NQ / 4; ++i) {
            const int blk = i / (LB / 32), k = i % (LB / 32);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (g < G) v = reinterpret_cast<const uint4 *>(base + g * hstride + blk * LB + t * (LB / 4))[k];
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < NQ; ++k) {
            const float2 f = bf16x2_to_float2(w[k]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        // shift so that amax * 2^-e < 2^15: f16 then holds every bf16 element exactly
        const int eb = (__float_as_int(amax) >> 23) & 0xFF;  // amax < 2^(eb - 126)
        const int e = max(0, eb - 126 - 15);
        const float sh = pow2_biased(127 - e);
#pragma unroll
        for (int m = 0; m < KS; ++m) {
            const float2 lo = bf16x2_to_float2(w[2 * m]), hi = bf16x2_to_float2(w[2 * m + 1]);
            qb[h][m][0] = pack_f16x2(lo.x * sh, lo.y * sh);  // dims qdim(m) + 0, 1
            qb[h][m][1] = pack_f16x2(hi.x * sh, hi.y * sh);  // dims qdim(m) + 2, 3
        }
        qscale[h] = qs * pow2_biased(127 + e);
    }

    // Byte offset of 16-byte chunk `ch` of line `line` in a line block: 128-byte swizzle
    // (chunk XOR line & 7) for 128-byte lines, 64-byte (chunk XOR (line >> 1) & 3) for 64.
    static __device__ __forceinline__ int chunk_off(int line, int ch) {
        return line * LB + ((LB == 128 ? (ch ^ (line & 7)) : (ch ^ ((line >> 1) & 3))) << 4);
    }

    // This lane's QK code words of a key row: LB / 4 bytes of every line block (words in
    // qdim order)
    __device__ __forceinline__ void line_words(const uint8_t *tile, int line, uint32_t (&w)[KS]) const {
#pragma unroll
        for (int blk = 0; blk < NB; ++blk) {
#pragma unroll
            for (int k = 0; k < WPB / 4; ++k) {
                const uint4 a = lds128(tile + blk * C::CODE_BLK + chunk_off(line, (WPB / 4) * t + k));
                w[blk * WPB + 4 * k] = a.x;
                w[blk * WPB + 4 * k + 1] = a.y;
                w[blk * WPB + 4 * k + 2] = a.z;
                w[blk * WPB + 4 * k + 3] = a.w;
            }
        }
    }

    // This lane's PV code words of a key row: dims DPL g .. DPL g + DPL - 1
    __device__ __forceinline__ void v_words(const uint8_t *tile, int line, uint32_t (&w)[VW]) const {
        if constexpr (VW == 2) {  // 8 bytes: half g & 1 of chunk g >> 1 (64-byte lines)
            const uint2 a = *reinterpret_cast<const uint2 *>(tile + chunk_off(line, g >> 1) + (g & 1) * 8);
            w[0] = a.x;
            w[1] = a.y;
        } else {  // 16-byte chunks (DPL g) / 16 .. of line block (DPL g) / LB
#pragma unroll
            for (int k = 0; k < VW / 4; ++k) {
                const int byte = DPL * g + 16 * k;
                const uint4 a = lds128(tile + (byte / LB) * C::CODE_BLK + chunk_off(line, (byte % LB) >> 4));
                w[4 * k] = a.x;
                w[4 * k + 1] = a.y;
                w[4 * k + 2] = a.z;
                w[4 * k + 3] = a.w;
            }
        }
    }

    __device__ __forceinline__ void tile(const uint8_t *stage, int nvalid) {
        const int nv = nvalid - key0;
        if (nv <= 0) return;
        const bool v0 = g < nv, v1 = g + 8 < nv;
#pragma unroll
        for (int h = 0; h < HW; ++h) {
            const uint8_t *sK = stage, *sV = stage + C::CODE_BYTES;
            const int l0 = line0 + h * hline, l1 = line1 + h * hline;
            const int o0 = f0 + h * hfac, o1 = f1 + h * hfac;
            const float kfac0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(stage + C::KS_OFF + o0));
            const float kfac1 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(stage + C::KS_OFF + o1));
            const float vfac0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(stage + C::VS_OFF + o0));
            const float vfac1 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(stage + C::VS_OFF + o1));
            // V: dims DPL g .. of keys 2t, 2t+1, 2t+8, 2t+9 (the boxes being multiples of 8
            // rows, an even key and the next one are consecutive lines)
            uint32_t vw[4][VW];
#pragma unroll
            for (int j = 0; j < 4; ++j) v_words(sV, (j < 2 ? vline0 : vline2) + (j & 1) + h * hline, vw[j]);
            // S^T = K . Q^T (keys g, g+8 x heads 2t, 2t+1)
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            {
                uint32_t k0[KS], k1[KS];
                line_words(sK, l0, k0);
                line_words(sK, l1, k1);
#pragma unroll
                for (int m = 0; m < KS; ++m) {
                    uint32_t a[4];
                    e4m3x4_to_f16(k0[m], a[0], a[2]);
                    e4m3x4_to_f16(k1[m], a[1], a[3]);
                    mma_f16_16816(c, a, qb[h][m][0], qb[h][m][1]);
                }
            }
            const float ks0 = kfac0 * qscale[h], ks1 = kfac1 * qscale[h];
            float s[4];
            s[0] = v0 ? __fmul_rn(c[0], ks0) : -INFINITY;  // (rounded once: the same value feeds max and exp)
            s[1] = v0 ? __fmul_rn(c[1], ks0) : -INFINITY;
            s[2] = v1 ? __fmul_rn(c[2], ks1) : -INFINITY;
            s[3] = v1 ? __fmul_rn(c[3], ks1) : -INFINITY;
            float mx[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
            float vm = fmaxf(v0 ? vfac0 : 0.f, v1 ? vfac1 : 0.f);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xFFFFFFFFu, mx[0], o));
                mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xFFFFFFFFu, mx[1], o));
                vm = fmaxf(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, o));
            }
            // V-factor unit: a power of two above every factor seen (vm < 2^(E - 127))
            float rescale = 1.f;
            {
                const int E = min(254, ((__float_as_int(vm) >> 23) & 0xFF) + 1);
                if (vm > 0.f && E > vE[h]) {
                    rescale = vE[h] - E + 127 >= 1 ? pow2_biased(vE[h] - E + 127) : 0.f;
                    vE[h] = E;
                }
            }
            const float vu = vE[h] > 0 ? pow2_biased(254 - vE[h]) : 0.f;  // 2^(127 - vE): factor -> [0, 1)
            float alpha[2], mu[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float m_new = fmaxf(m_run[h][j], mx[j]);
                mu[j] = (m_new == -INFINITY) ? 0.f : m_new;
                alpha[j] = ex2(m_run[h][j] - mu[j]);
                m_run[h][j] = m_new;
            }
            const float p0 = ex2(s[0] - mu[0]), p1 = ex2(s[1] - mu[1]);
            const float p2 = ex2(s[2] - mu[0]), p3 = ex2(s[3] - mu[1]);
            l_run[h][0] = l_run[h][0] * alpha[0] + (p0 + p2);
            l_run[h][1] = l_run[h][1] * alpha[1] + (p1 + p3);
            const float vs0 = v0 ? vfac0 * vu : 0.f;
            const float vs1 = v1 ? vfac1 * vu : 0.f;
            const uint32_t b0 = movmatrix_trans(pack_f16x2(p0 * vs0, p1 * vs0));
            const uint32_t b1 = movmatrix_trans(pack_f16x2(p2 * vs1, p3 * vs1));
            const float fa = alpha[0] * rescale, fb = alpha[1] * rescale;
            if (__any_sync(0xFFFFFFFFu, fa != 1.f || fb != 1.f)) {
#pragma unroll
                for (int m = 0; m < KS; ++m) {
                    acc[h][m][0] *= fa;
                    acc[h][m][1] *= fb;
                    acc[h][m][2] *= fa;
                    acc[h][m][3] *= fb;
                }
            }
            // O^T += V^T . P'^T; rows past the end read as code 0 so 0 * V stays 0
            if (nv < 16) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (2 * t + (j & 1) + 8 * (j >> 1) >= nv)
#pragma unroll
                        for (int k = 0; k < VW; ++k) vw[j][k] = 0u;
            }
            // A rows g, g+8 = dims DPL g + 2m, + 1; k = keys: byte-interleave keys 2t, 2t+1
            // (and 2t+8, 2t+9) so that one conversion yields a key pair of one dim
#pragma unroll
            for (int m = 0; m < KS; ++m) {
                const int wi = m >> 1;
                const uint32_t sel = (m & 1) ? 0x7362u : 0x5140u;
                const uint32_t ab = __byte_perm(vw[0][wi], vw[1][wi], sel);
                const uint32_t cd = __byte_perm(vw[2][wi], vw[3][wi], sel);
                uint32_t a[4];
                e4m3x4_to_f16(ab, a[0], a[1]);
                e4m3x4_to_f16(cd, a[2], a[3]);
                mma_f16_16816(acc[h][m], a, b0, b1);
            }
        }
    }

    // Merge the four key slices per (kv head, query head) in two halves of D (the row merge
    // of the bf16 path); emit(kv head in unit, query head, d, a0, a1, M, l) gets dims d, d+1
    // in natural order.
    template <class Sync, class Emit>
    __device__ __forceinline__ bool finish(float *mrg, Sync sync, Emit emit) {
        constexpr int NWC = C::NWC, KW = C::KW, DH = D / 2, NR = HG * G;  // rows per key slice
        float *macc = mrg;                // [KW][HG * G][D/2]
        float *mml = mrg + KW * NR * DH;  // [KW][HG * G][2]
#pragma unroll
        for (int h = 0; h < HW; ++h) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                l_run[h][0] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h][0], o);
                l_run[h][1] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h][1], o);
            }
            if (g == 0) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (2 * t + j < G) {
                        mml[(kw * NR + (hw0 + h) * G + 2 * t + j) * 2 + 0] = m_run[h][j];
                        mml[(kw * NR + (hw0 + h) * G + 2 * t + j) * 2 + 1] = l_run[h][j];
                    }
            }
        }
        const int tid = warp * 32 + lane;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if ((g >> 2) == half) {  // this lane's dims DPL g .. DPL g + DPL - 1 lie in this half
#pragma unroll
                for (int h = 0; h < HW; ++h) {
                    // back from units of 2^(vE - 127) (V factors); dims DPL g + 2m, +1
                    const float unit = vE[h] > 0 ? pow2_biased(vE[h]) : 0.f;
#pragma unroll
                    for (int m = 0; m < KS; ++m) {
                        const int dlo = DPL * g + 2 * m - half * DH;
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            if (2 * t + j < G) {
                                float *row = macc + (kw * NR + (hw0 + h) * G + 2 * t + j) * DH;
                                row[dlo] = acc[h][m][j] * unit;
                                row[dlo + 1] = acc[h][m][j + 2] * unit;
                            }
                        }
                    }
                }
            }
            if (!sync()) return false;
            for (int e = tid * 2; e < NR * DH; e += NWC * 32 * 2) {
                const int rr = e / DH, dd = e % DH;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < KW; ++w) M = fmaxf(M, mml[(w * NR + rr) * 2]);
                const float Mu = (M == -INFINITY) ? 0.f : M;
                float a0 = 0.f, a1 = 0.f, lv = 0.f;
#pragma unroll
                for (int w = 0; w < KW; ++w) {
                    const float f = ex2(mml[(w * NR + rr) * 2] - Mu);
                    lv = fmaf(f, mml[(w * NR + rr) * 2 + 1], lv);
                    const float2 x = *reinterpret_cast<const float2 *>(macc + (w * NR + rr) * DH + dd);
                    a0 = fmaf(f, x.x, a0);
                    a1 = fmaf(f, x.y, a1);
                }
                emit(rr / G, rr % G, half * DH + dd, a0, a1, M, lv);
            }
            if (!sync()) return false;
        }
        return true;
    }
};

// ---- row gather (page sizes that are not multiples of 8) -------------------------------
// The tile is one box of BT rows: code line of (row r, head h) = h * BT + r, factors at
// byte (h * BT + r) * 2 of the tile's factor slots.  Page ids are looked up one tile ahead,
// factors loaded one tile ahead (after the page ids have landed), so that the copy of a
// tile never waits on a global load.

template <class C>
struct GatherPages {
    static constexpr int N = C::BT / 32;  // rows per lane: lane, lane + 32
    int pg[N], slot[N];
    __device__ __forceinline__ void lookup(const int32_t *table, int tok, int nvalid, int page_size, int lane) {
#pragma unroll
        for (int k = 0; k < N; ++k) {
            const int r = lane + 32 * k;
            pg[k] = 0;
            slot[k] = 0;
            if (r < nvalid) {
                pg[k] = __ldg(table + (tok + r) / page_size);
                slot[k] = (tok + r) % page_size;
            }
        }
    }
    // page ids outside the pool are read as page 0 and flagged
    __device__ __forceinline__ void check(int nvalid, int num_pages, int lane) {
#pragma unroll
        for (int k = 0; k < N; ++k)
            if (lane + 32 * k < nvalid && (pg[k] < 0 || pg[k] >= num_pages)) {
                flag_error(DAP_DEVERR_PAGE);
                pg[k] = 0;
            }
    }
    // the K and V factor bits of this lane's rows, heads kvh0 .. kvh0 + HG - 1
    __device__ __forceinline__ void load_factors(uint32_t (&f)[N][C::HG], const SplitParams &p, int kvh0,
                                                 int nvalid, int lane) const {
        const uint16_t *ks = reinterpret_cast<const uint16_t *>(p.k_scale);
        const uint16_t *vs = reinterpret_cast<const uint16_t *>(p.v_scale);
#pragma unroll
        for (int k = 0; k < N; ++k)
#pragma unroll
            for (int h = 0; h < C::HG; ++h) {
                f[k][h] = 0u;
                if (lane + 32 * k < nvalid) {
                    const long long i = ((long long)pg[k] * p.Hkv + kvh0 + h) * p.page_size + slot[k];
                    f[k][h] = (uint32_t)__ldg(ks + i) | ((uint32_t)__ldg(vs + i) << 16);
                }
            }
    }
};

// Copy rows [0, nvalid) of the CTA's kv heads into the stage (codes by cp.async, factors
// stored from registers) and arrive on `full` twice per lane: once when its copies have
// landed, once after its factor stores (64 arrivals).
template <class C>
__device__ __forceinline__ void gather_codes(uint8_t *stage, const GatherPages<C> &gp,
                                             const uint32_t (&fac)[GatherPages<C>::N][C::HG], int nvalid, int kvh0,
                                             const SplitParams &p, uint64_t *full, int lane) {
    constexpr int D = C::D, LB = C::LB, BT = C::BT, HG = C::HG, N = GatherPages<C>::N;
    constexpr int CPR = D / 16, IPI = 32 / CPR;  // chunks per code row; (row, head) items per copy
    long long row[N];                            // byte offset of this lane's rows (head kvh0)
#pragma unroll
    for (int k = 0; k < N; ++k) row[k] = (((long long)gp.pg[k] * p.page_size + gp.slot[k]) * p.Hkv + kvh0) * D;
    // lane = (item r0 of every IPI items, chunk c); item = h * BT + r
    const int c = lane % CPR, r0 = lane / CPR;
    const int blk = c / (LB / 16), cib = c % (LB / 16);
    const uint32_t sk = smem_addr(stage) + blk * C::CODE_BLK, sv = sk + C::CODE_BYTES;
    const uint8_t *kc = p.k_codes + c * 16, *vc = p.v_codes + c * 16;
#pragma unroll
    for (int it = 0; it < HG * BT / IPI; ++it) {
        const int h = (IPI * it) / BT, r = (IPI * it) % BT + r0;
        const long long off = __shfl_sync(0xFFFFFFFFu, row[((IPI * it) % BT) >> 5], r & 31) + h * D;
        if (r < nvalid) {
            const int line = h * BT + r;
            const int sw = LB == 128 ? (line & 7) : ((line >> 1) & 3);
            const uint32_t dst = (uint32_t)(line * LB + ((cib ^ sw) << 4));
            cp_async_16(sk + dst, kc + off);
            cp_async_16(sv + dst, vc + off);
        }
    }
    uint16_t *fk = reinterpret_cast<uint16_t *>(stage + C::KS_OFF);
    uint16_t *fv = reinterpret_cast<uint16_t *>(stage + C::VS_OFF);
#pragma unroll
    for (int k = 0; k < N; ++k)
#pragma unroll
        for (int h = 0; h < HG; ++h) {
            const int r = lane + 32 * k;
            fk[h * BT + r] = (uint16_t)(fac[k][h] & 0xFFFFu);
            fv[h * BT + r] = (uint16_t)(fac[k][h] >> 16);
        }
    cp_async_mbar_arrive(full);
    mbar_arrive(full);  // (release: this lane's factor stores)
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
    fp8kv_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                 const __grid_constant__ CUtensorMap mapKS, const __grid_constant__ CUtensorMap mapVS,
                 const SplitParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = aligned_smem<C>(smem_raw);
    constexpr int G = C::G, HG = C::HG, NWC = C::NWC, BT = C::BT, NS = C::NS, D = C::D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int nkvg = p.Hkv / HG;
    const int units = p.B * nkvg;
    const int s = blockIdx.x / units;
    const int rem = blockIdx.x - s * units;
    const int b = rem / nkvg;
    const int kvg = rem - b * nkvg;
    // Launched as a programmatic dependent of the previous kernel on the stream: nothing
    // global is read before the wait (that kernel may still write the inputs); the combine
    // of this call may launch at once (it waits for this grid before its reads).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int L = p.seq_lens[b];
    const int R = C::GATHER ? BT : p.box_rows;  // (row gather: the tile is one box of BT rows)
    int pg_first = 0;  // loaded with the length (entries past the end are read, not used)
    if (!C::GATHER && warp == NWC && lane * R < BT) {
        const long long t = (long long)s * p.chunk + lane * R;
        if (t < (long long)p.max_pages * p.page_size)
            pg_first = __ldg(p.block_table + (long long)b * p.max_pages + t / p.page_size);
    }
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
            mbar_init(&full[i], C::GATHER ? 64u : 1u);  // row gather: two arrivals per producer lane
            mbar_init(&empty[i], NWC);
        }
        misc[0] = 0;
        misc[1] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (C::GATHER && warp == NWC) {  // ---- producer warp, row gather
        // Software pipeline over three buffers, each one tile's page ids and factors: at the
        // start of step i, buffer A holds tile i (both landed), B tile i + 1 (factors in
        // flight), C tile i + 2 (page ids in flight).  Step i fills tile i from A, then loads
        // C's factors and issues A's page ids for tile i + 3; the next step takes (B, C, A).
        // The roles rotate by unrolling three steps, so no register that a load in flight
        // will write is ever copied (a copy waits for the load: rotating by copies left a
        // full memory latency in every step and held the copy to a third of the TMA path).
        struct Buf {
            GatherPages<C> g;
            uint32_t f[GatherPages<C>::N][HG];  // (K | V << 16) factor bits
        };
        const int32_t *table = p.block_table + (long long)b * p.max_pages;
        const int kvh0 = kvg * HG;
        auto nval = [&](int i) { return max(0, min(BT, tok1 - (tok0 + i * BT))); };
        Buf A, B2, C2;
        A.g.lookup(table, tok0, nval(0), p.page_size, lane);
        B2.g.lookup(table, tok0 + BT, nval(1), p.page_size, lane);
        C2.g.lookup(table, tok0 + 2 * BT, nval(2), p.page_size, lane);
        A.g.check(nval(0), p.num_pages, lane);
        A.g.load_factors(A.f, p, kvh0, nval(0), lane);
        B2.g.check(nval(1), p.num_pages, lane);
        B2.g.load_factors(B2.f, p, kvh0, nval(1), lane);
        int issued = 0;
        // one step: fill tile i from x, load z's factors (tile i + 2), issue x's page ids
        // for tile i + 3; false when a wait gave up
        auto step = [&](int i, Buf &x, Buf &z) -> bool {
            const int st = i % NS;
            if (i >= NS && !__all_sync(0xFFFFFFFFu, mbar_wait(&empty[st], ((i / NS) - 1) & 1))) {
                misc[1] = 1;
                return false;
            }
            gather_codes<C>(smem + st * C::STAGE_BYTES, x.g, x.f, nval(i), kvh0, p, &full[st], lane);
            issued = i + 1;
            z.g.check(nval(i + 2), p.num_pages, lane);
            z.g.load_factors(z.f, p, kvh0, nval(i + 2), lane);
            x.g.lookup(table, tok0 + (i + 3) * BT, nval(i + 3), p.page_size, lane);
            return true;
        };
        for (int i = 0; i < ntiles; i += 3) {
            if (!step(i, A, C2) || i + 1 >= ntiles) break;
            if (!step(i + 1, B2, A) || i + 2 >= ntiles) break;
            if (!step(i + 2, C2, B2)) break;
        }
        if (lane == 0) misc[0] = issued;
        __syncthreads();
        return;
    }
    if (warp == NWC) {  // ---- producer warp
        if (lane == 0) {
            prefetch_tensormap(&mapK);
            prefetch_tensormap(&mapV);
            prefetch_tensormap(&mapKS);
            prefetch_tensormap(&mapVS);
        }
        const int32_t *table = p.block_table + (long long)b * p.max_pages;
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
            const int nbox = (min(BT, tok1 - t) + R - 1) / R;
            if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)(nbox * R * HG * (2 * D + 4)));
            __syncwarp();
            if (lane < nbox) {
                uint8_t *stage = smem + st * C::STAGE_BYTES;
                const int row = (t + lane * R) % p.page_size;
#pragma unroll
                for (int blk = 0; blk < C::NB; ++blk) {
                    uint8_t *dst = stage + blk * C::CODE_BLK + lane * R * HG * C::LB;
                    tma_load_4d(dst, &mapK, blk * C::LB, row, kvg * HG, pg, &full[st]);
                    tma_load_4d(dst + C::CODE_BYTES, &mapV, blk * C::LB, row, kvg * HG, pg, &full[st]);
                }
                tma_load_3d(stage + C::KS_OFF + lane * C::FSLOT, &mapKS, row, kvg * HG, pg, &full[st]);
                tma_load_3d(stage + C::VS_OFF + lane * C::FSLOT, &mapVS, row, kvg * HG, pg, &full[st]);
            }
            issued = i + 1;
        }
        if (lane == 0) misc[0] = issued;
        __syncthreads();
        return;
    }

    // ---- consumer warps
    Consumer<C> cs;
    cs.init(warp, lane, R);
    cs.reset();
#pragma unroll
    for (int h = 0; h < C::HPW; ++h)
        cs.load_q(h, p.q + (long long)b * p.q_sb + (long long)(kvg * HG + cs.hw0 + h) * G * p.q_sh, p.q_sh,
                  p.qscale);
    int consumed = 0;
    for (int i = 0; i < ntiles; ++i) {
        const int st = i % NS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[st], (i / NS) & 1))) {
            misc[1] = 1;
            break;
        }
        cs.tile(smem + st * C::STAGE_BYTES, min(BT, tok1 - (tok0 + i * BT)));
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        consumed = i + 1;
    }
    __syncthreads();  // every tile consumed; stage 0 is free for the merge
    if (misc[1]) {
        if (threadIdx.x == 0)
            for (int i = consumed; i < misc[0]; ++i) (void)mbar_wait(&full[i % NS], (i / NS) & 1);
        return;
    }
    const bool direct = (nsplit == 1);
    cs.finish(reinterpret_cast<float *>(smem), [] { named_sync(1, NWC * 32); return true; },
              [&](int hl, int hh, int d, float a0, float a1, float M, float lv) {
                  const int hq = (kvg * HG + hl) * G + hh;
                  if (direct) {
                      store_out_pair(p.out + (long long)b * p.o_sb + (long long)hq * p.o_sh + d, a0, a1, lv);
                  } else {
                      const long long row = ((long long)b * p.num_splits + s) * p.Hq + hq;
                      *reinterpret_cast<float2 *>(p.o_part + row * D + d) = make_float2(a0, a1);
                      if (d == 0) *reinterpret_cast<float2 *>(p.ml_part + row * 2) = make_float2(M, lv);
                  }
              });
}

// ---- host side -------------------------------------------------------------------------

namespace {

bool encode_map(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, int rank, const cuuint64_t *dims,
                const cuuint64_t *strides_bytes, const cuuint32_t *box, CUtensorMapSwizzle swz) {
    EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) return false;
    const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    return enc(map, dtype, (cuuint32_t)rank, const_cast<void *>(base), dims, strides_bytes, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// codes [P, ps, Hkv, D] bytes viewed as [D, ps, Hkv, P] (the head dim outside the slot
// dim); box [LB, R, HG, 1] lands head-major, 128-byte swizzled (64-byte for 64-byte lines)
bool encode_codes(CUtensorMap *map, const void *base, int D, int LB, int Hkv, int ps, int P, int R, int HG) {
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)ps, (cuuint64_t)Hkv, (cuuint64_t)P};
    const cuuint64_t strides[3] = {(cuuint64_t)Hkv * D, (cuuint64_t)D, (cuuint64_t)ps * Hkv * D};
    const cuuint32_t box[4] = {(cuuint32_t)LB, (cuuint32_t)R, (cuuint32_t)HG, 1u};
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 4, dims, strides, box,
                      LB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

// factors [P, Hkv, ps] bf16 viewed as [ps, Hkv, P]; box [R, HG, 1]
bool encode_factors(CUtensorMap *map, const void *base, int Hkv, int ps, int P, int R, int HG) {
    const cuuint64_t dims[3] = {(cuuint64_t)ps, (cuuint64_t)Hkv, (cuuint64_t)P};
    const cuuint64_t strides[2] = {(cuuint64_t)ps * 2, (cuuint64_t)Hkv * ps * 2};
    const cuuint32_t box[3] = {(cuuint32_t)R, (cuuint32_t)HG, 1u};
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, 3, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int D, int G, int HG, bool GATHER>
dap_status launch_g(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    using C = Cfg<D, G, HG, GATHER>;
    const int R = gcd_int(a.page_size, C::BT);
    p.box_rows = R;
    CUtensorMap mk = {}, mv = {}, mks = {}, mvs = {};  // (the row-gather producer reads the cache directly)
    if (!GATHER && (!encode_codes(&mk, a.k, D, C::LB, a.Hkv, a.page_size, a.num_pages, R, HG) ||
                    !encode_codes(&mv, a.v, D, C::LB, a.Hkv, a.page_size, a.num_pages, R, HG) ||
                    !encode_factors(&mks, a.k_scale, a.Hkv, a.page_size, a.num_pages, R, HG) ||
                    !encode_factors(&mvs, a.v_scale, a.Hkv, a.page_size, a.num_pages, R, HG)))
        return DAP_ERR_CUDA;
    auto kern = fp8kv_kernel<C>;
    static PerDeviceOcc occ = {};
    if (prepare_kernel(kern, C::THREADS, C::SMEM, &occ) <= 0) return DAP_ERR_CUDA;
    const long long grid = (long long)a.B * (a.Hkv / HG) * a.num_splits;
    if (grid > 0x7FFFFFFFLL) return DAP_ERR_SHAPE;
    p.o_part = static_cast<float *>(a.workspace);
    p.ml_part = a.num_splits > 1 ? reinterpret_cast<float *>(static_cast<char *>(a.workspace) +
                                                             partial_acc_bytes(a.B, a.Hq, a.D, a.num_splits))
                                 : nullptr;
    if (g_trace.split_begin) cudaEventRecord(g_trace.split_begin, stream);
    if (launch_dependent_smem(kern, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM, stream, mk, mv, mks, mvs, p) !=
        cudaSuccess)
        return DAP_ERR_CUDA;
    if (g_trace.split_end) cudaEventRecord(g_trace.split_end, stream);
    if (a.num_splits > 1) {
        if (launch_combine<D>(p, a.B, a.Hq, a.num_splits, stream) != cudaSuccess) return DAP_ERR_CUDA;
    }
    if (g_trace.combine_end) cudaEventRecord(g_trace.combine_end, stream);
    return DAP_OK;
}

// two kv heads per CTA when they pair up, a row is at most 128 bytes and the tiles come by
// TMA (the row-gather producer's registers spilled at two heads per CTA)
template <int D, bool GATHER>
dap_status launch_d(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    constexpr bool WIDE = D > 128 || GATHER;
    const bool pair = !WIDE && a.Hkv % 2 == 0;
    switch (a.Hq / a.Hkv) {
        case 1: return pair ? launch_g<D, 1, WIDE ? 1 : 2, GATHER>(a, p, stream) : launch_g<D, 1, 1, GATHER>(a, p, stream);
        case 2: return pair ? launch_g<D, 2, WIDE ? 1 : 2, GATHER>(a, p, stream) : launch_g<D, 2, 1, GATHER>(a, p, stream);
        case 4: return pair ? launch_g<D, 4, WIDE ? 1 : 2, GATHER>(a, p, stream) : launch_g<D, 4, 1, GATHER>(a, p, stream);
        case 8: return pair ? launch_g<D, 8, WIDE ? 1 : 2, GATHER>(a, p, stream) : launch_g<D, 8, 1, GATHER>(a, p, stream);
    }
    return DAP_ERR_UNSUPPORTED;
}

template <bool GATHER>
dap_status launch_any(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    switch (a.D) {
        case 64: return launch_d<64, GATHER>(a, p, stream);
        case 128: return launch_d<128, GATHER>(a, p, stream);
        case 256: return launch_d<256, GATHER>(a, p, stream);
    }
    return DAP_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace f8kv

dap_status launch_decode_fp8kv(const DecodeArgs &a, cudaStream_t stream) {
    SplitParams p = make_params(a);
    return a.page_size % 8 == 0 ? f8kv::launch_any<false>(a, p, stream) : f8kv::launch_any<true>(a, p, stream);
}

bool read_errors_fp8kv(unsigned int *flags, bool clear) {
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
