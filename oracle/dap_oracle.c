/*
 * dap_oracle.c -- plain fp64 CPU oracle for paged GQA decode attention and for the
 * fp8 sliding-window latent (K = V) decode variant.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path may link, load or call this
 * file; only the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header, table or constant with the CUDA kernels: every
 * conversion (bf16 bits -> value, e4m3 bits -> value, round-to-bf16) is written out
 * here from its definition.
 *
 * What is computed, and where it is defined:
 *
 *   decode attention (AstrAI "CUDA Kernels" developer doc, section "Python Wrappers":
 *   q/k/v are [batch, seq_len, n_heads, head_dim] and the scale is 1/sqrt(head_dim);
 *   AstrAI csrc commit log, split-KV commit: the decode op reads every KV position of
 *   the sequence):
 *       for every sequence b and query head h, with G = Hq / Hkv and kv head h / G,
 *       s_t   = scale * sum_d q[b,h,d] * K[b,t,h/G,d]         for t < seq_lens[b]
 *       out   = sum_t softmax(s)_t * V[b,t,h/G,:]
 *   computed in double, softmax by its definition with the maximum subtracted first
 *   (two passes over t).  An empty sequence (seq_lens[b] == 0) gives a zero row: the
 *   pages guard the normalising division (csrc commit log, numerics-unification
 *   commit: divide-by-zero guard), so the empty sum stays 0.
 *
 *   paged addressing (csrc commit log, per-element page lookup commit; "CUDA Kernels",
 *   section "Q Scheduling and KV Addressing": a KV policy only translates a logical
 *   position into a physical address):
 *       logical position t of sequence b lives in physical page block_table[b][t / ps]
 *       at in-page slot t % ps; the cache is [num_pages, ps, Hkv, D].
 *   The walk below is a plain loop over t; nothing is blocked or reordered.
 *
 *   fp8 sliding-window latent decode (nvfp4-megamoe-kernel native_swa_decode.py,
 *   _fallback_batched_sdp):
 *       for token t and window position j < W the slot is idx = indices[t][j]; the row
 *       takes part iff j < lens[t] and idx >= 0; its block is idx / bs and offset
 *       idx % bs; its value is round_to_bf16(e4m3(byte) * inv_scale[idx]) (the
 *       fallback multiplies the bf16 cast of the fp8 value by the bf16 inverse scale
 *       and keeps a bf16 result); keys and values are the same rows (K = V);
 *       s_j = scale * q[t,h,:] . kv_j and out = sum_j softmax(s)_j * kv_j.
 *   Readings where the page is silent: a token with no participating row gives a zero
 *   row (the page's kernel stub normalises only when the row sum is nonzero); a slot
 *   at or past num_blocks * bs is treated like a padded slot (the page's fallback
 *   would raise an indexing error there).
 *
 *   GQA decode over an e4m3 cache (the fp8 cache convention of native_swa_decode.py, one
 *   dequantisation factor per (slot, kv head) for K and for V): the paged decode above with
 *   K = e4m3(code) * factor and V likewise, the product exact; the matching append
 *   quantises each (sequence, kv head) row by the fp8 append rule further down.
 *
 *   multi-token decode and the packed-q work map (AstrAI "CUDA Kernels", "Q Scheduling and
 *   KV Addressing"): token i of the q_len new tokens of sequence b sits at position
 *   seq_lens[b] - q_len + i and attends the keys up to it.
 *
 * Parity pins (tests/test_oracle_pins.py) tie each function to something other than
 * itself: closed forms (constant V, a single key, a key shift, q = 0), brute force
 * against torch's float64 scaled_dot_product_attention, page-permutation invariance,
 * the e4m3 table against torch's float8_e4m3fn conversion for all 256 codes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- scalar conversions, from their definitions ------------------------------------ */

/* bf16 is the upper half of an IEEE binary32: widen the bits and read the float. */
double oracle_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP E4M3FN: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, subnormals when
 * the exponent field is 0, no infinities, S.1111.111 is NaN. */
double oracle_e4m3_value(uint8_t byte) {
    int sign = (byte >> 7) & 1;
    int e = (byte >> 3) & 0xF;
    int m = byte & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round a double that is exactly representable as a binary32 to the nearest bf16,
 * ties to even (keep the upper 16 bits after adding half an ulp plus the tie bit). */
double oracle_round_to_bf16(double x) {
    float f = (float)x;
    uint32_t u;
    if (isnan(f)) return NAN;
    memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    u &= 0xFFFF0000u;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---- one query head against n logical rows ----------------------------------------- */

/* softmax(scale * q . k_t) weighted sum of v_t over t < n.  krows[t] / vrows[t] point at
 * the bf16 rows (D elements); q is D doubles.  s is caller scratch of n doubles. */
static void attend_one(const double *q, const uint16_t *const *krows,
                       const uint16_t *const *vrows, int n, int D, double scale,
                       double *s, double *out) {
    int t, d;
    double mx = -INFINITY, z = 0.0;
    for (d = 0; d < D; ++d) out[d] = 0.0;
    if (n <= 0) return;
    for (t = 0; t < n; ++t) {
        double dot = 0.0;
        for (d = 0; d < D; ++d) dot += q[d] * oracle_bf16_value(krows[t][d]);
        s[t] = scale * dot;
        if (s[t] > mx) mx = s[t];
    }
    for (t = 0; t < n; ++t) {
        double w = exp(s[t] - mx);
        z += w;
        for (d = 0; d < D; ++d) out[d] += w * oracle_bf16_value(vrows[t][d]);
    }
    for (d = 0; d < D; ++d) out[d] /= z;
}

/* ---- paged GQA decode --------------------------------------------------------------- */

/* One (b, h) output row of paged decode.  q is [B, Hq, D] with element strides
 * (q_stride_b, q_stride_h, 1); caches are [num_pages, ps, Hkv, D]; block_table is
 * [B, max_pages].  Returns 0, or -1 when the row would read outside the given buffers
 * (a page index outside [0, num_pages) or seq_len beyond max_pages * ps). */
static int paged_row_keep(const uint16_t *q, long long q_stride_b, long long q_stride_h,
                          const uint16_t *k_cache, const uint16_t *v_cache, int num_pages,
                          const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                          int Hq, int Hkv, int D, int page_size, double scale, int b, int h,
                          const uint8_t *keep, double *out);

static int paged_row(const uint16_t *q, long long q_stride_b, long long q_stride_h,
                     const uint16_t *k_cache, const uint16_t *v_cache, int num_pages,
                     const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                     int Hq, int Hkv, int D, int page_size, double scale, int b, int h,
                     double *out) {
    return paged_row_keep(q, q_stride_b, q_stride_h, k_cache, v_cache, num_pages, block_table, max_pages,
                          seq_lens, Hq, Hkv, D, page_size, scale, b, h, NULL, out);
}

/* The same row over the kept keys only: key t takes part iff keep == NULL or keep[t] != 0
 * (a bool mask with True = keep, [CK] "Python Wrappers" interface); no kept key gives a
 * zero row. */
static int paged_row_keep(const uint16_t *q, long long q_stride_b, long long q_stride_h,
                          const uint16_t *k_cache, const uint16_t *v_cache, int num_pages,
                          const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                          int Hq, int Hkv, int D, int page_size, double scale, int b, int h,
                          const uint8_t *keep, double *out) {
    int G = Hq / Hkv, kh = h / G, L = seq_lens[b], t, d, rc = 0, n = 0;
    double *qd, *s;
    const uint16_t **kr, **vr;
    if (L < 0 || (long long)L > (long long)max_pages * page_size) return -1;
    qd = (double *)malloc(sizeof(double) * (size_t)D);
    s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    kr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(L > 0 ? L : 1));
    vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(L > 0 ? L : 1));
    for (d = 0; d < D; ++d) qd[d] = oracle_bf16_value(q[b * q_stride_b + h * q_stride_h + d]);
    for (t = 0; t < L; ++t) {
        int32_t page = block_table[(long long)b * max_pages + t / page_size];
        int slot = t % page_size;
        long long row;
        if (page < 0 || page >= num_pages) { rc = -1; break; }
        if (keep && !keep[t]) continue;
        row = (((long long)page * page_size + slot) * Hkv + kh) * D;
        kr[n] = k_cache + row;
        vr[n] = v_cache + row;
        ++n;
    }
    if (rc == 0) attend_one(qd, kr, vr, n, D, scale, s, out);
    free(qd); free(s); free(kr); free(vr);
    return rc;
}

/* Full paged decode: out is [B, Hq, D] doubles.  Returns the number of rows that
 * failed the bounds check (their output is left as NaN). */
int oracle_decode_paged(const uint16_t *q, long long q_stride_b, long long q_stride_h,
                        const uint16_t *k_cache, const uint16_t *v_cache, int num_pages,
                        const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                        int B, int Hq, int Hkv, int D, int page_size, double scale,
                        double *out) {
    int bad = 0;
    long long i, n = (long long)B * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (i = 0; i < n; ++i) {
        int b = (int)(i / Hq), h = (int)(i % Hq), d;
        double *o = out + i * D;
        if (paged_row(q, q_stride_b, q_stride_h, k_cache, v_cache, num_pages, block_table,
                      max_pages, seq_lens, Hq, Hkv, D, page_size, scale, b, h, o) != 0) {
            for (d = 0; d < D; ++d) o[d] = NAN;
            ++bad;
        }
    }
    return bad;
}

/* Masked paged decode ([CK] "Python Wrappers": mask 2-D [batch, kv_len], bool, True =
 * keep): key t of sequence b takes part iff t < seq_lens[b] and mask[b * mask_stride + t]
 * != 0.  A sequence with no kept key gives a zero row.  Everything else as
 * oracle_decode_paged. */
int oracle_decode_paged_masked(const uint16_t *q, long long q_stride_b, long long q_stride_h,
                               const uint16_t *k_cache, const uint16_t *v_cache, int num_pages,
                               const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                               const uint8_t *mask, long long mask_stride, int B, int Hq, int Hkv, int D,
                               int page_size, double scale, double *out) {
    int bad = 0;
    long long i, n = (long long)B * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (i = 0; i < n; ++i) {
        int b = (int)(i / Hq), h = (int)(i % Hq), d;
        double *o = out + i * D;
        if (paged_row_keep(q, q_stride_b, q_stride_h, k_cache, v_cache, num_pages, block_table, max_pages,
                           seq_lens, Hq, Hkv, D, page_size, scale, b, h, mask + (long long)b * mask_stride,
                           o) != 0) {
            for (d = 0; d < D; ++d) o[d] = NAN;
            ++bad;
        }
    }
    return bad;
}

/* Selected rows only: rows[i] = b * Hq + h; out is [nrows, D]. */
int oracle_decode_paged_rows(const uint16_t *q, long long q_stride_b, long long q_stride_h,
                             const uint16_t *k_cache, const uint16_t *v_cache, int num_pages,
                             const int32_t *block_table, int max_pages,
                             const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                             int page_size, double scale, const int64_t *rows, int nrows,
                             double *out) {
    int bad = 0, i;
    (void)B;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (i = 0; i < nrows; ++i) {
        int b = (int)(rows[i] / Hq), h = (int)(rows[i] % Hq), d;
        double *o = out + (long long)i * D;
        if (paged_row(q, q_stride_b, q_stride_h, k_cache, v_cache, num_pages, block_table,
                      max_pages, seq_lens, Hq, Hkv, D, page_size, scale, b, h, o) != 0) {
            for (d = 0; d < D; ++d) o[d] = NAN;
            ++bad;
        }
    }
    return bad;
}

/* ---- contiguous GQA decode ---------------------------------------------------------- */

/* k, v are [B, max_len, Hkv, D]; the first seq_lens[b] positions of sequence b are
 * read.  out is [B, Hq, D]. */
int oracle_decode_contig(const uint16_t *q, long long q_stride_b, long long q_stride_h,
                         const uint16_t *k, const uint16_t *v, int max_len,
                         const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                         double scale, double *out) {
    int bad = 0;
    long long i, n = (long long)B * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (i = 0; i < n; ++i) {
        int b = (int)(i / Hq), h = (int)(i % Hq), G = Hq / Hkv, kh = h / G;
        int L = seq_lens[b], t, d;
        double *o = out + i * D;
        double *qd, *s;
        const uint16_t **kr, **vr;
        if (L < 0 || L > max_len) {
            for (d = 0; d < D; ++d) o[d] = NAN;
            ++bad;
            continue;
        }
        qd = (double *)malloc(sizeof(double) * (size_t)D);
        s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        kr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(L > 0 ? L : 1));
        vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(L > 0 ? L : 1));
        for (d = 0; d < D; ++d) qd[d] = oracle_bf16_value(q[b * q_stride_b + h * q_stride_h + d]);
        for (t = 0; t < L; ++t) {
            long long row = (((long long)b * max_len + t) * Hkv + kh) * D;
            kr[t] = k + row;
            vr[t] = v + row;
        }
        attend_one(qd, kr, vr, L, D, scale, s, o);
        free(qd); free(s); free(kr); free(vr);
    }
    return bad;
}

/* ---- fp8 sliding-window latent decode (K = V) --------------------------------------- */

/* q [T, NH, HD] bf16 bits; kv_cache [num_blocks, block_size, HD] e4m3 bytes;
 * inv_scale [num_blocks * block_size] bf16 bits; indices [T, W] int64 (-1 padded);
 * lens [T] int64.  out is [T, NH, HD] doubles.  Tokens in [t0, t1) only. */
void oracle_fp8_swa_range(const uint16_t *q, const uint8_t *kv_cache,
                          const uint16_t *inv_scale, const int64_t *indices,
                          const int64_t *lens, int T, int NH, int HD, int W,
                          int num_blocks, int block_size, double scale, int t0, int t1,
                          double *out) {
    int t;
    long long max_slots = (long long)num_blocks * block_size;
    (void)T;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = t0; t < t1; ++t) {
        /* rows taking part for this token, dequantised once (they serve every head) */
        double *kv = (double *)malloc(sizeof(double) * (size_t)W * HD);
        double *s = (double *)malloc(sizeof(double) * (size_t)(W > 0 ? W : 1));
        int n = 0, j, h, d;
        for (j = 0; j < W; ++j) {
            int64_t idx = indices[(long long)t * W + j];
            long long block, offset;
            double inv;
            if (!(j < lens[t]) || idx < 0 || idx >= max_slots) continue;
            block = idx / block_size;
            offset = idx % block_size;
            inv = oracle_bf16_value(inv_scale[idx]);
            for (d = 0; d < HD; ++d) {
                uint8_t byte = kv_cache[(block * block_size + offset) * HD + d];
                kv[(long long)n * HD + d] = oracle_round_to_bf16(oracle_e4m3_value(byte) * inv);
            }
            ++n;
        }
        for (h = 0; h < NH; ++h) {
            const uint16_t *qr = q + ((long long)t * NH + h) * HD;
            double *o = out + ((long long)t * NH + h) * HD;
            double mx = -INFINITY, z = 0.0;
            for (d = 0; d < HD; ++d) o[d] = 0.0;
            if (n == 0) continue;
            for (j = 0; j < n; ++j) {
                double dot = 0.0;
                for (d = 0; d < HD; ++d) dot += oracle_bf16_value(qr[d]) * kv[(long long)j * HD + d];
                s[j] = scale * dot;
                if (s[j] > mx) mx = s[j];
            }
            for (j = 0; j < n; ++j) {
                double w = exp(s[j] - mx);
                z += w;
                for (d = 0; d < HD; ++d) o[d] += w * kv[(long long)j * HD + d];
            }
            for (d = 0; d < HD; ++d) o[d] /= z;
        }
        free(kv);
        free(s);
    }
}

void oracle_fp8_swa(const uint16_t *q, const uint8_t *kv_cache, const uint16_t *inv_scale,
                    const int64_t *indices, const int64_t *lens, int T, int NH, int HD, int W,
                    int num_blocks, int block_size, double scale, double *out) {
    oracle_fp8_swa_range(q, kv_cache, inv_scale, indices, lens, T, NH, HD, W, num_blocks,
                         block_size, scale, 0, T, out);
}

/* ---- KV append (the step before decode) -------------------------------------------- */

/* Paged append: for each sequence b and kv head h, the new token's K and V rows go to
 * logical position pos[b] of sequence b, i.e. page block_table[b][pos / ps], slot pos % ps
 * (the same translation decode reads through).  Caches are [num_pages, ps, Hkv, D] bf16
 * bits; k_new / v_new are [B, Hkv, D].  Returns the number of rows that could not be
 * placed (position or page out of range); those are skipped. */
int oracle_kv_append_paged(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_cache,
                           uint16_t *v_cache, int num_pages, int page_size,
                           const int32_t *block_table, int max_pages, const int32_t *pos, int B,
                           int Hkv, int D) {
    int b, h, d, bad = 0;
    for (b = 0; b < B; ++b) {
        long long p = pos[b];
        int32_t page;
        if (p < 0 || p >= (long long)max_pages * page_size) { bad += Hkv; continue; }
        page = block_table[(long long)b * max_pages + p / page_size];
        if (page < 0 || page >= num_pages) { bad += Hkv; continue; }
        for (h = 0; h < Hkv; ++h) {
            long long dst = (((long long)page * page_size + p % page_size) * Hkv + h) * D;
            long long src = ((long long)b * Hkv + h) * D;
            for (d = 0; d < D; ++d) {
                k_cache[dst + d] = k_new[src + d];
                v_cache[dst + d] = v_new[src + d];
            }
        }
    }
    return bad;
}

/* Round a binary32 value to the nearest OCP E4M3FN code, ties to even, saturating to
 * +-448 (the largest finite code); NaN gives 0x7F.  Written from the format: a code is
 * (-1)^s * 2^(e-7) * (1 + m/8) for e in 1..15 (except e = 15, m = 7), and
 * (-1)^s * 2^-6 * (m/8) for e = 0. */
uint8_t oracle_e4m3_from_float(float x) {
    int code, best = 0, sign = 0;
    double ax, bestdiff = INFINITY;
    if (isnan(x)) return 0x7F;
    if (signbit(x)) { sign = 1; x = -x; }
    ax = (double)x;
    if (ax >= 448.0) return (uint8_t)((sign << 7) | 0x7E);
    /* the finite non-negative codes 0x00..0x7E are increasing in value: take the nearest,
     * an exact tie going to the code with an even mantissa (even code) */
    for (code = 0; code <= 0x7E; ++code) {
        double v = oracle_e4m3_value((uint8_t)code);
        double diff = fabs(v - ax);
        if (diff < bestdiff || (diff == bestdiff && (code & 1) == 0)) {
            bestdiff = diff;
            best = code;
        }
    }
    return (uint8_t)((sign << 7) | best);
}

/* fp8 append of latent rows (K = V): row t (HD bf16 values) goes to slot slots[t] of the
 * [num_blocks, block_size, HD] e4m3 cache with its dequantisation factor in inv_scale[slot]
 * (the decode side computes e4m3 * inv_scale).  In binary32, as the kernel does:
 *   amax = max |x|;  s = amax / 448 (1 when amax is 0);  s is stored as bf16 (RNE);
 *   code = e4m3_rne_satfinite(x / s_stored)  (an IEEE binary32 division).
 * Returns the number of rows skipped because their slot is outside the cache. */
int oracle_kv_append_fp8(const uint16_t *rows, uint8_t *kv_cache, uint16_t *inv_scale,
                         const int64_t *slots, int T, int HD, int num_blocks, int block_size) {
    int t, d, bad = 0;
    long long max_slots = (long long)num_blocks * block_size;
    for (t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        float amax = 0.0f, s, sb;
        uint32_t u;
        uint16_t sbits;
        if (slot < 0 || slot >= max_slots) { ++bad; continue; }
        for (d = 0; d < HD; ++d) {
            float x = (float)oracle_bf16_value(rows[(long long)t * HD + d]);
            if (fabsf(x) > amax) amax = fabsf(x);
        }
        s = amax > 0.0f ? amax / 448.0f : 1.0f;
        sb = (float)oracle_round_to_bf16((double)s);
        memcpy(&u, &sb, sizeof u);
        sbits = (uint16_t)(u >> 16);
        inv_scale[slot] = sbits;
        for (d = 0; d < HD; ++d) {
            float x = (float)oracle_bf16_value(rows[(long long)t * HD + d]);
            kv_cache[slot * HD + d] = oracle_e4m3_from_float(x / sb);
        }
    }
    return bad;
}

/* ---- multi-token decode ---------------------------------------------------------------- */

/* Several new tokens per sequence (already in the cache): sequence b has q_len_b =
 * qo_indptr[b+1] - qo_indptr[b] new tokens at positions seq_lens[b] - q_len_b + i, and
 * token i attends the keys t <= its own position (causal among the new tokens).  q and out
 * are packed [total_q, Hq, D] (token r = qo_indptr[b] + i).  Everything else as
 * oracle_decode_paged.  Returns the number of rows that failed the bounds checks. */
int oracle_decode_paged_multi(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                              int num_pages, const int32_t *block_table, int max_pages,
                              const int32_t *seq_lens, const int32_t *qo_indptr, const uint8_t *mask,
                              long long mask_stride, int B, int Hq, int Hkv, int D, int page_size,
                              double scale, double *out) {
    int bad = 0, b;
    for (b = 0; b < B; ++b) {
        int q0 = qo_indptr[b], qlen = qo_indptr[b + 1] - qo_indptr[b], L = seq_lens[b], i;
        for (i = 0; i < qlen; ++i) {
            int upto = L - qlen + i + 1; /* keys 0 .. position of token i */
            int32_t one = upto < 0 ? 0 : upto, h, d;
            /* an optional mask row of the packed token (3-D mask [batch, q_len, kv_len] with the
             * q rows packed; True = keep) applies together with the causal rule */
            const uint8_t *keep = mask ? mask + (long long)(q0 + i) * mask_stride : NULL;
            for (h = 0; h < Hq; ++h) {
                double *o = out + ((long long)(q0 + i) * Hq + h) * D;
                /* reuse the single-token row with the sequence cut at this token */
                if (paged_row_keep(q + (long long)(q0 + i) * Hq * D, 0, D, k_cache,
                                   v_cache, num_pages, block_table + (long long)b * max_pages, max_pages,
                                   &one, Hq, Hkv, D, page_size, scale, 0, h, keep, o) != 0) {
                    for (d = 0; d < D; ++d) o[d] = NAN;
                    ++bad;
                }
            }
        }
    }
    return bad;
}

/* The packed-Q work map (AstrAI "CUDA Kernels" doc, "Q Scheduling and KV Addressing"):
 * qo_indptr is the prefix sum of the q lengths; every sequence's tokens are cut into tiles
 * of `tokens_per_tile`, and tile w covers tile index tile_index[w] of sequence
 * tile_batch[w].  Returns the number of tiles, or -1 when max_tiles is too small. */
int oracle_q_tile_map(const int32_t *q_lens, int B, int tokens_per_tile, int32_t *qo_indptr,
                      int32_t *tile_batch, int32_t *tile_index, int max_tiles) {
    int b, n = 0, j;
    qo_indptr[0] = 0;
    for (b = 0; b < B; ++b) {
        int tiles = (q_lens[b] + tokens_per_tile - 1) / tokens_per_tile;
        qo_indptr[b + 1] = qo_indptr[b] + q_lens[b];
        for (j = 0; j < tiles; ++j) {
            if (n >= max_tiles) return -1;
            tile_batch[n] = b;
            tile_index[n] = j;
            ++n;
        }
    }
    return n;
}

/* ---- paged GQA decode over an fp8 cache ------------------------------------------------ */

/* The GQA decode above with K and V held as OCP e4m3 codes and one dequantisation factor
 * per (slot, kv head) for each (the fp8 cache convention of nvfp4-megamoe-kernel
 * native_swa_decode.py, applied to the GQA cache: the decoded value is the code's value
 * times the bf16 factor):
 *   K[b, t, kh, d] = e4m3(k_codes[page, slot, kh, d]) * bf16(k_scale[page, kh, slot]),
 *   page = block_table[b][t / ps], slot = t % ps, likewise V with v_codes and v_scale;
 * the product is taken exactly (in double).  Codes are [num_pages, ps, Hkv, D] bytes;
 * the factors [num_pages, Hkv, ps] bf16 bits.  Then s_t = scale * q . K_t and
 * out = sum_t softmax(s)_t V_t as in oracle_decode_paged (zero row for an empty sequence).
 * Returns the number of rows that failed the bounds checks (left NaN). */
static int paged_row_fp8kv(const uint16_t *q, long long q_stride_b, long long q_stride_h,
                           const uint8_t *k_codes, const uint8_t *v_codes, const uint16_t *k_scale,
                           const uint16_t *v_scale, int num_pages, const int32_t *block_table,
                           int max_pages, const int32_t *seq_lens, int Hq, int Hkv, int D,
                           int page_size, double scale, int b, int h, double *out) {
    int G = Hq / Hkv, kh = h / G, L = seq_lens[b], t, d;
    double *qd, *s, *vrow, mx = -INFINITY, z = 0.0;
    long long *rowoff, *scaleoff;
    if (L < 0 || (long long)L > (long long)max_pages * page_size) return -1;
    for (t = 0; t < L; ++t) {
        int32_t page = block_table[(long long)b * max_pages + t / page_size];
        if (page < 0 || page >= num_pages) return -1;
    }
    for (d = 0; d < D; ++d) out[d] = 0.0;
    if (L == 0) return 0;
    qd = (double *)malloc(sizeof(double) * (size_t)D);
    vrow = (double *)malloc(sizeof(double) * (size_t)D);
    s = (double *)malloc(sizeof(double) * (size_t)L);
    rowoff = (long long *)malloc(sizeof(long long) * (size_t)L);
    scaleoff = (long long *)malloc(sizeof(long long) * (size_t)L);
    for (d = 0; d < D; ++d) qd[d] = oracle_bf16_value(q[b * q_stride_b + h * q_stride_h + d]);
    for (t = 0; t < L; ++t) {
        long long page = block_table[(long long)b * max_pages + t / page_size];
        int slot = t % page_size;
        rowoff[t] = ((page * page_size + slot) * Hkv + kh) * D;
        scaleoff[t] = (page * Hkv + kh) * page_size + slot;
    }
    for (t = 0; t < L; ++t) {
        double ks = oracle_bf16_value(k_scale[scaleoff[t]]), dot = 0.0;
        for (d = 0; d < D; ++d) dot += qd[d] * (oracle_e4m3_value(k_codes[rowoff[t] + d]) * ks);
        s[t] = scale * dot;
        if (s[t] > mx) mx = s[t];
    }
    for (t = 0; t < L; ++t) {
        double w = exp(s[t] - mx), vs = oracle_bf16_value(v_scale[scaleoff[t]]);
        z += w;
        for (d = 0; d < D; ++d) vrow[d] = oracle_e4m3_value(v_codes[rowoff[t] + d]) * vs;
        for (d = 0; d < D; ++d) out[d] += w * vrow[d];
    }
    for (d = 0; d < D; ++d) out[d] /= z;
    free(qd); free(vrow); free(s); free(rowoff); free(scaleoff);
    return 0;
}

int oracle_decode_paged_fp8kv(const uint16_t *q, long long q_stride_b, long long q_stride_h,
                              const uint8_t *k_codes, const uint8_t *v_codes, const uint16_t *k_scale,
                              const uint16_t *v_scale, int num_pages, const int32_t *block_table,
                              int max_pages, const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                              int page_size, double scale, double *out) {
    int bad = 0;
    long long i, n = (long long)B * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (i = 0; i < n; ++i) {
        int b = (int)(i / Hq), h = (int)(i % Hq), d;
        double *o = out + i * D;
        if (paged_row_fp8kv(q, q_stride_b, q_stride_h, k_codes, v_codes, k_scale, v_scale, num_pages,
                            block_table, max_pages, seq_lens, Hq, Hkv, D, page_size, scale, b, h, o) != 0) {
            for (d = 0; d < D; ++d) o[d] = NAN;
            ++bad;
        }
    }
    return bad;
}

/* fp8 append for the GQA cache: every (sequence b, kv head h) row of k_new / v_new
 * [B, Hkv, D] bf16 is quantised by the per-row rule of oracle_kv_append_fp8 (amax / 448
 * stored as bf16, codes e4m3(x / factor) RNE saturating) and written at logical position
 * pos[b]: codes to [page, slot, h, :] of the [num_pages, ps, Hkv, D] caches, factors to
 * [page, h, slot] of the [num_pages, Hkv, ps] scale arrays.  Returns the number of rows
 * skipped (position or page out of range). */
static void quantise_row(const uint16_t *x, int n, uint8_t *codes, uint16_t *factor) {
    float amax = 0.0f, s, sb;
    uint32_t u;
    int d;
    for (d = 0; d < n; ++d) {
        float v = (float)oracle_bf16_value(x[d]);
        if (fabsf(v) > amax) amax = fabsf(v);
    }
    s = amax > 0.0f ? amax / 448.0f : 1.0f;
    sb = (float)oracle_round_to_bf16((double)s);
    memcpy(&u, &sb, sizeof u);
    *factor = (uint16_t)(u >> 16);
    for (d = 0; d < n; ++d) codes[d] = oracle_e4m3_from_float((float)oracle_bf16_value(x[d]) / sb);
}

int oracle_kv_append_paged_fp8(const uint16_t *k_new, const uint16_t *v_new, uint8_t *k_codes,
                               uint8_t *v_codes, uint16_t *k_scale, uint16_t *v_scale, int num_pages,
                               int page_size, const int32_t *block_table, int max_pages,
                               const int32_t *pos, int B, int Hkv, int D) {
    int b, h, bad = 0;
    for (b = 0; b < B; ++b) {
        long long p = pos[b], page;
        int slot;
        if (p < 0 || p >= (long long)max_pages * page_size) { bad += Hkv; continue; }
        page = block_table[(long long)b * max_pages + p / page_size];
        if (page < 0 || page >= num_pages) { bad += Hkv; continue; }
        slot = (int)(p % page_size);
        for (h = 0; h < Hkv; ++h) {
            long long src = ((long long)b * Hkv + h) * D;
            long long dst = ((page * page_size + slot) * Hkv + h) * D;
            long long f = (page * Hkv + h) * page_size + slot;
            quantise_row(k_new + src, D, k_codes + dst, k_scale + f);
            quantise_row(v_new + src, D, v_codes + dst, v_scale + f);
        }
    }
    return bad;
}
