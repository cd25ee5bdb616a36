// dap_multi.cu -- multi-token causal decode and masked decode over the paged KV cache:
// the entry points, the TMA-fed configurations (page sizes that are multiples of 8) and
// the tile-size rule.  Kernels: dap_multi.cuh.
#include "dap_multi.cuh"

namespace dap {

int multi_tokens_per_tile(int G, int max_q_len) {
    if (G < 1 || G > 16) return 0;
    return max_q_len <= 16 / G ? 16 / G : 32 / G;
}

dap_status launch_decode_multi(const DecodeArgs &a, cudaStream_t stream) {
    if (a.page_size % 8 != 0) return launch_decode_multi_gather(a, stream);
    return multi_entry<false>(a, stream);
}

dap_status launch_decode_masked(const DecodeArgs &a, cudaStream_t stream) {
    if (a.page_size % 8 != 0) return launch_decode_masked_gather(a, stream);
    return masked_entry<false>(a, stream);
}

bool read_errors_multi(unsigned int *flags, bool clear) {
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
