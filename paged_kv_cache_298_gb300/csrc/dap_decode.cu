// dap_decode.cu -- bf16 GQA decode attention, TMA-fed configurations (page sizes that are
// multiples of 8, and the contiguous cache), the dispatch over head dims and group sizes,
// and the library's other decode entry points.  Kernels: dap_decode.cuh.
#include "dap_decode.cuh"

namespace dap {
namespace {

template <int D, int G>
dap_status dispatch(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    return run<MmaCfgFor<D, G>>(a, p, stream);
}

template <int D>
dap_status dispatch_groups(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    switch (a.Hq / a.Hkv) {
        case 1: return dispatch<D, 1>(a, p, stream);
        case 2: return dispatch<D, 2>(a, p, stream);
        case 4: return dispatch<D, 4>(a, p, stream);
        case 8: return dispatch<D, 8>(a, p, stream);
    }
    return DAP_ERR_UNSUPPORTED;
}

}  // namespace

int balanced_heads_per_unit(int D, int G) {
    (void)D;
    return G;  // CfgFor uses one kv head per unit
}

int balanced_kv_heads_per_unit(int D, int G) {
    (void)D;
    (void)G;
    return 1;
}

namespace {

// One thread waits on a barrier that nothing arrives on: the bounded wait gives up and
// flags DAP_DEVERR_TIMEOUT (the failure path of every pipeline wait, run on purpose).
__global__ void selftest_wait_kernel() {
    __shared__ uint64_t bar;
    mbar_init(&bar, 1);
    fence_barrier_init();
    (void)mbar_wait(&bar, 0);
}

}  // namespace

dap_status launch_selftest_wait(cudaStream_t stream) {
    selftest_wait_kernel<<<1, 1, 0, stream>>>();
    return cudaGetLastError() == cudaSuccess ? DAP_OK : DAP_ERR_CUDA;
}

bool read_errors_decode(unsigned int *flags, bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_errors, sizeof v) != cudaSuccess) return false;
    if (clear) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_device_errors, &z, sizeof z) != cudaSuccess) return false;
    }
    *flags |= v;
    return true;
}

dap_status launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    if (a.paged && a.page_size % 8 != 0) return launch_decode_gather(a, stream);
    SplitParams p = make_params(a);
    switch (a.D) {
        case 32: return dispatch_groups<32>(a, p, stream);
        case 64: return dispatch_groups<64>(a, p, stream);
        case 128: return dispatch_groups<128>(a, p, stream);
        case 256: return dispatch_groups<256>(a, p, stream);
    }
    return DAP_ERR_UNSUPPORTED;
}
}  // namespace dap
