// dap_decode_gather.cu -- bf16 GQA decode attention over a paged cache whose page size is
// not a multiple of 8: the tensor-core configurations of dap_decode.cuh with the row-gather
// producer (every row's page looked up, rows copied in 16-byte cp.async chunks into the
// swizzled tiles), for head dims 32, 64, 128 and 256 and both schedules.
#include "dap_decode.cuh"

namespace dap {
namespace {

template <int D>
dap_status dispatch_gather(const DecodeArgs &a, SplitParams &p, cudaStream_t stream) {
    switch (a.Hq / a.Hkv) {
        case 1: return run<GatherCfgFor<D, 1>>(a, p, stream);
        case 2: return run<GatherCfgFor<D, 2>>(a, p, stream);
        case 4: return run<GatherCfgFor<D, 4>>(a, p, stream);
        case 8: return run<GatherCfgFor<D, 8>>(a, p, stream);
    }
    return DAP_ERR_UNSUPPORTED;
}

}  // namespace

dap_status launch_decode_gather(const DecodeArgs &a, cudaStream_t stream) {
    if (!a.paged) return DAP_ERR_UNSUPPORTED;
    SplitParams p = make_params(a);
    switch (a.D) {
        case 32: return dispatch_gather<32>(a, p, stream);
        case 64: return dispatch_gather<64>(a, p, stream);
        case 128: return dispatch_gather<128>(a, p, stream);
        case 256: return dispatch_gather<256>(a, p, stream);
    }
    return DAP_ERR_UNSUPPORTED;
}

bool read_errors_decode_gather(unsigned int *flags, bool clear) {
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
