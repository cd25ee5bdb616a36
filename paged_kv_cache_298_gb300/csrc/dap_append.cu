// dap_append.cu -- writing the new decode token into the caches (the step before decode).
//
// Paged append: each sequence's new K and V rows (one per kv head) go to its logical
// position through the block table, the same translation the decode kernels read through
// (AstrAI "CUDA Kernels" doc, "Q Scheduling and KV Addressing": a KV policy translates a
// logical position into a physical address).
//
// fp8 append: a latent row (K = V) is quantised to OCP e4m3 with one scale per slot; the
// decode side dequantises as code * inv_scale (nvfp4-megamoe-kernel native_swa_decode.py,
// _fallback_batched_sdp).  Per slot, in binary32: amax = max |x|, s = amax / 448 (1 for an
// all-zero row), stored as bf16; code = e4m3(x / s_stored), round to nearest even,
// saturating at +-448 (AstrAI doc, FP8 section: quantize multiplies by the quantisation
// multiplier, amax is kept in the input domain).
//
// GQA fp8 append: the same quantiser per (sequence, kv head) row of the K and the V cache,
// one factor per (slot, kv head) each.
//
// One warp per row; accesses are coalesced (16 bytes per lane; 2 to 8 for the GQA fp8
// codes).  Out-of-range positions, pages and slots are skipped and flagged in the device
// error word.
#include <cuda_fp8.h>

#include "dap_device.cuh"
#include "dap_internal.h"

namespace dap {

namespace {

__global__ void __launch_bounds__(256)
    append_paged_kernel(const __nv_bfloat16 *k_new, const __nv_bfloat16 *v_new, __nv_bfloat16 *k_cache,
                        __nv_bfloat16 *v_cache, int num_pages, int page_size, const int32_t *block_table,
                        int max_pages, const int32_t *pos, int B, int Hkv, int D) {
    // launched as a programmatic dependent: nothing global is read before the previous
    // kernel on the stream is done; the next launch (the decode that reads these rows
    // waits the same way) may start at once
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);  // (b, h)
    const int lane = threadIdx.x & 31;
    if (row >= B * Hkv) return;
    const int b = row / Hkv, h = row - b * Hkv;
    const long long p = pos[b];
    if (p < 0 || p >= (long long)max_pages * page_size) {
        if (lane == 0 && h == 0) flag_error(DAP_DEVERR_SEQLEN);
        return;
    }
    const int page = block_table[(long long)b * max_pages + p / page_size];
    if (page < 0 || page >= num_pages) {
        if (lane == 0 && h == 0) flag_error(DAP_DEVERR_PAGE);
        return;
    }
    const long long dst = (((long long)page * page_size + p % page_size) * Hkv + h) * D;
    const long long src = (long long)row * D;
    for (int c = lane; c < D / 8; c += 32) {
        reinterpret_cast<uint4 *>(k_cache + dst)[c] = reinterpret_cast<const uint4 *>(k_new + src)[c];
        reinterpret_cast<uint4 *>(v_cache + dst)[c] = reinterpret_cast<const uint4 *>(v_new + src)[c];
    }
}

// HD / 256 groups of 8 values per lane (HD a multiple of 256).
template <int HD>
__global__ void __launch_bounds__(256)
    append_fp8_kernel(const __nv_bfloat16 *rows, uint8_t *kv_cache, __nv_bfloat16 *inv_scale, const int64_t *slots,
                      int T, long long max_slots) {
    // launched as a programmatic dependent: nothing global is read before the previous
    // kernel on the stream is done; the next launch (the decode that reads these rows
    // waits the same way) may start at once
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int NG = HD / 256;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const int64_t slot = slots[t];
    if (slot < 0 || slot >= max_slots) {
        if (lane == 0) flag_error(DAP_DEVERR_SLOT);
        return;
    }
    float x[NG][8];
    float amax = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        const uint4 w = reinterpret_cast<const uint4 *>(rows + (long long)t * HD)[g * 32 + lane];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = bf16x2_to_float2(ws[j]);
            x[g][2 * j] = f.x;
            x[g][2 * j + 1] = f.y;
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const __nv_bfloat16 sb16 = __float2bfloat16_rn(s);
    const float sb = __bfloat162float(sb16);
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        uint32_t packed[2];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float2 y = make_float2(__fdiv_rn(x[g][4 * half + 2 * j], sb),
                                             __fdiv_rn(x[g][4 * half + 2 * j + 1], sb));
                const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
                word |= (uint32_t)c << (16 * j);
            }
            packed[half] = word;
        }
        reinterpret_cast<uint2 *>(kv_cache + slot * HD)[g * 32 + lane] = make_uint2(packed[0], packed[1]);
    }
    if (lane == 0) inv_scale[slot] = sb16;
}

// fp8 append for the GQA cache: one warp per (sequence, kv head) row of D values, VPL =
// D / 32 per lane; the K row and the V row are quantised one after the other by the rule
// above.  Codes go to [page, slot, h, :] of the [num_pages, ps, Hkv, D] caches, the
// factors to [page, h, slot] of the [num_pages, Hkv, ps] arrays.
template <int VPL>
__device__ __forceinline__ void quantise_row(const __nv_bfloat16 *src, uint8_t *codes, __nv_bfloat16 *factor,
                                             int lane) {
    float x[VPL];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; i += 2) {
        const float2 f = bf16x2_to_float2(reinterpret_cast<const uint32_t *>(src + lane * VPL)[i / 2]);
        x[i] = f.x;
        x[i + 1] = f.y;
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const __nv_bfloat16 sb16 = __float2bfloat16_rn(s);
    const float sb = __bfloat162float(sb16);
    uint8_t c[VPL];
#pragma unroll
    for (int i = 0; i < VPL; i += 2) {
        const __nv_fp8x2_storage_t two = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(x[i], sb), __fdiv_rn(x[i + 1], sb)), __NV_SATFINITE, __NV_E4M3);
        c[i] = (uint8_t)(two & 0xFF);
        c[i + 1] = (uint8_t)(two >> 8);
    }
    if constexpr (VPL == 2) {
        reinterpret_cast<uint16_t *>(codes)[lane] = (uint16_t)(c[0] | (c[1] << 8));
    } else {
#pragma unroll
        for (int i = 0; i < VPL; i += 4)
            reinterpret_cast<uint32_t *>(codes + lane * VPL)[i / 4] =
                (uint32_t)c[i] | ((uint32_t)c[i + 1] << 8) | ((uint32_t)c[i + 2] << 16) | ((uint32_t)c[i + 3] << 24);
    }
    if (lane == 0) *factor = sb16;
}

template <int D>
__global__ void __launch_bounds__(256)
    append_paged_fp8_kernel(const __nv_bfloat16 *k_new, const __nv_bfloat16 *v_new, uint8_t *k_codes,
                            uint8_t *v_codes, __nv_bfloat16 *k_scale, __nv_bfloat16 *v_scale, int num_pages,
                            int page_size, const int32_t *block_table, int max_pages, const int32_t *pos, int B,
                            int Hkv) {
    // launched as a programmatic dependent: nothing global is read before the previous
    // kernel on the stream is done; the next launch (the decode that reads these rows
    // waits the same way) may start at once
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);  // (b, h)
    const int lane = threadIdx.x & 31;
    if (row >= B * Hkv) return;
    const int b = row / Hkv, h = row - b * Hkv;
    const long long p = pos[b];
    if (p < 0 || p >= (long long)max_pages * page_size) {
        if (lane == 0 && h == 0) flag_error(DAP_DEVERR_SEQLEN);
        return;
    }
    const int page = block_table[(long long)b * max_pages + p / page_size];
    if (page < 0 || page >= num_pages) {
        if (lane == 0 && h == 0) flag_error(DAP_DEVERR_PAGE);
        return;
    }
    const long long slot = p % page_size;
    const long long dst = (((long long)page * page_size + slot) * Hkv + h) * D;
    const long long f = ((long long)page * Hkv + h) * page_size + slot;
    quantise_row<D / 32>(k_new + (long long)row * D, k_codes + dst, k_scale + f, lane);
    quantise_row<D / 32>(v_new + (long long)row * D, v_codes + dst, v_scale + f, lane);
}

// Launch with programmatic stream serialization (the kernels order their own reads).
template <class K, class... Args>
cudaError_t launch_pdl(K kern, dim3 grid, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

dap_status launch_append_paged_fp8(const void *k_new, const void *v_new, uint8_t *k_codes, uint8_t *v_codes,
                                   void *k_scale, void *v_scale, int num_pages, int page_size,
                                   const int32_t *block_table, int max_pages, const int32_t *pos, int B, int Hkv,
                                   int D, cudaStream_t stream) {
    const dim3 grid((unsigned)((B * Hkv + 7) / 8));
    const __nv_bfloat16 *kn = static_cast<const __nv_bfloat16 *>(k_new), *vn = static_cast<const __nv_bfloat16 *>(v_new);
    __nv_bfloat16 *ks = static_cast<__nv_bfloat16 *>(k_scale), *vs = static_cast<__nv_bfloat16 *>(v_scale);
    switch (D) {
        case 64:
            if (launch_pdl(append_paged_fp8_kernel<64>, grid, stream, kn, vn, k_codes, v_codes, ks, vs, num_pages,
                           page_size, block_table, max_pages, pos, B, Hkv) != cudaSuccess)
                return DAP_ERR_CUDA;
            break;
        case 128:
            if (launch_pdl(append_paged_fp8_kernel<128>, grid, stream, kn, vn, k_codes, v_codes, ks, vs, num_pages,
                           page_size, block_table, max_pages, pos, B, Hkv) != cudaSuccess)
                return DAP_ERR_CUDA;
            break;
        case 256:
            if (launch_pdl(append_paged_fp8_kernel<256>, grid, stream, kn, vn, k_codes, v_codes, ks, vs, num_pages,
                           page_size, block_table, max_pages, pos, B, Hkv) != cudaSuccess)
                return DAP_ERR_CUDA;
            break;
        default: return DAP_ERR_UNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? DAP_OK : DAP_ERR_CUDA;
}

dap_status launch_append_paged(const void *k_new, const void *v_new, void *k_cache, void *v_cache, int num_pages,
                               int page_size, const int32_t *block_table, int max_pages, const int32_t *pos, int B,
                               int Hkv, int D, cudaStream_t stream) {
    const int rows = B * Hkv;
    if (launch_pdl(append_paged_kernel, dim3((unsigned)((rows + 7) / 8)), stream,
                   static_cast<const __nv_bfloat16 *>(k_new), static_cast<const __nv_bfloat16 *>(v_new),
                   static_cast<__nv_bfloat16 *>(k_cache), static_cast<__nv_bfloat16 *>(v_cache), num_pages, page_size,
                   block_table, max_pages, pos, B, Hkv, D) != cudaSuccess)
        return DAP_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DAP_OK : DAP_ERR_CUDA;
}

dap_status launch_append_fp8(const void *rows, uint8_t *kv_cache, void *inv_scale, const int64_t *slots, int T,
                             int HD, int num_blocks, int block_size, cudaStream_t stream) {
    const long long max_slots = (long long)num_blocks * block_size;
    const dim3 grid((unsigned)((T + 7) / 8));
    const __nv_bfloat16 *r = static_cast<const __nv_bfloat16 *>(rows);
    __nv_bfloat16 *inv = static_cast<__nv_bfloat16 *>(inv_scale);
    switch (HD) {
        case 256:
            if (launch_pdl(append_fp8_kernel<256>, grid, stream, r, kv_cache, inv, slots, T, max_slots) != cudaSuccess)
                return DAP_ERR_CUDA;
            break;
        case 512:
            if (launch_pdl(append_fp8_kernel<512>, grid, stream, r, kv_cache, inv, slots, T, max_slots) != cudaSuccess)
                return DAP_ERR_CUDA;
            break;
        default: return DAP_ERR_UNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? DAP_OK : DAP_ERR_CUDA;
}

bool read_errors_append(unsigned int *flags, bool clear) {
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
