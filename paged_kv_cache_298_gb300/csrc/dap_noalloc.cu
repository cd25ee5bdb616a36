// dap_noalloc.cu -- decode_attn_paged_noalloc: paged decode with its split partials in a
// fixed file-scope device array instead of a caller workspace, for callers that cannot
// allocate device memory (see include/dap.h).  Runs the same kernels as decode_attn_paged.
#include <cuda_runtime.h>

#include <mutex>

#include "dap.h"
#include "dap_internal.h"

namespace {

// The scratch.  Host code must not pass `g_noalloc_scratch` itself to a kernel: in host
// code that name is a host-side stand-in, not a device address.  The device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DAP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.  Under
// lazy module loading this lookup is what loads this file's module on the device and
// reserves the array there.
dap_status scratch_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DAP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DAP_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return DAP_OK;
}

}  // namespace

extern "C" dap_status decode_attn_paged_noalloc(
    const void *q, long long q_stride_b, long long q_stride_h, const void *k_cache,
    const void *v_cache, int num_pages, int page_size, const int32_t *block_table, int max_pages,
    const int32_t *seq_lens, int max_kv_len, int B, int Hq, int Hkv, int D, float scale,
    int num_splits, void *out, long long out_stride_b, long long out_stride_h, void *stream) {
    if (B == 0 || num_splits < DAP_SPLITS_BALANCED)  // nothing to run, or a size error decode_attn_paged reports
        return decode_attn_paged(q, q_stride_b, q_stride_h, k_cache, v_cache, num_pages, page_size,
                                 block_table, max_pages, seq_lens, max_kv_len, B, Hq, Hkv, D, scale,
                                 num_splits, nullptr, 0, out, out_stride_b, out_stride_h, stream);
    const size_t cap = DAP_NOALLOC_SCRATCH_BYTES;
    int S = num_splits;
    if (S == 0) {
        // the planner's split count, lowered until its partials fit the scratch
        const int sms = dap_device_sm_count();
        if (sms <= 0) return DAP_ERR_CUDA;
        const int planned = dap_resolve_splits(0, sms, B, Hq, Hkv, D, page_size, max_kv_len, 0);
        if (planned >= 1) {
            S = planned;
            while (S > 1 && dap_workspace_bytes(B, Hq, Hkv, D, S) > cap) --S;
        }
    }
    void *scratch = nullptr;
    const dap_status st = scratch_address(&scratch);
    if (st != DAP_OK) return st;
    const dap_status r = decode_attn_paged(q, q_stride_b, q_stride_h, k_cache, v_cache, num_pages,
                                           page_size, block_table, max_pages, seq_lens, max_kv_len, B,
                                           Hq, Hkv, D, scale, S, scratch, cap, out, out_stride_b,
                                           out_stride_h, stream);
    // The scratch is never NULL and is 256-byte aligned, so a workspace refusal can only
    // mean the partials do not fit.
    return r == DAP_ERR_WORKSPACE ? DAP_ERR_SCRATCH_LIMIT : r;
}
