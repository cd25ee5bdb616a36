// dap_multi.cu -- multi-token causal decode and masked decode over the paged KV cache:
// the entry points, the TMA-fed configurations (page sizes that are multiples of 8) and
// the tile-size rule.  Kernels: dap_multi.cuh.
#include "dap_multi.cuh"

namespace dap {

// 16 / G tokens (mma.sync consumer, 16 columns) while they hold the longest run of new
// tokens; beyond that the 128-row tensor-memory tiles where the head dim has them (64, 128
// and 256: one K/V stream for up to 128 / G tokens), else 32 / G (two column groups).
int multi_tokens_per_tile(int G, int D, int max_q_len) {
    if (G < 1 || G > 16) return 0;
    if (max_q_len <= 16 / G) return 16 / G;
    return (D == 64 || D == 128 || D == 256) ? 128 / G : 32 / G;
}

dap_status launch_decode_multi(const DecodeArgs &a, cudaStream_t stream) {
    if (a.tokens_per_tile * (a.Hq / a.Hkv) == 128) return launch_decode_multi_tc(a, stream);
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
