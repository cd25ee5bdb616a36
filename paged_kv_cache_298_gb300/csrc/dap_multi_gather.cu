// dap_multi_gather.cu -- multi-token and masked decode over a paged cache whose page size
// is not a multiple of 8: the configurations of dap_multi.cuh with the row-gather producer.
#include "dap_multi.cuh"

namespace dap {

dap_status launch_decode_multi_gather(const DecodeArgs &a, cudaStream_t stream) { return multi_entry<true>(a, stream); }

dap_status launch_decode_masked_gather(const DecodeArgs &a, cudaStream_t stream) {
    return masked_entry<true>(a, stream);
}

bool read_errors_multi_gather(unsigned int *flags, bool clear) {
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
