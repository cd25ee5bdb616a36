// dap_fp8.cu -- fp8 (e4m3) sliding-window latent decode attention, K = V.
#include "dap_device.cuh"
#include "dap_internal.h"

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

dap_status launch_fp8(const Fp8Args &a, cudaStream_t stream) {
    (void)a;
    (void)stream;
    return DAP_ERR_UNSUPPORTED;
}

}  // namespace dap
