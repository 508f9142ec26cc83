// gdn_decode.cu -- entry of the decode step: dispatch on the activation type (one unit per
// type, gdn_decode_{f32,bf16,f16}.cu, instantiating gdn_decode.cuh for every Dk, Dv), the
// wait-timeout self-test kernel, and the decode watchdog words.
#include "gdn_internal.h"
#include "gdn_tma.cuh"

namespace gdn {

cudaError_t launch_decode(const gdn_params &p, cudaStream_t stream) {
    if (!tiled_dims(p)) return launch_general(p, true, stream);
    switch (p.act_dtype) {
        case GDN_F32: return launch_decode_f32(p, stream);
        case GDN_BF16: return launch_decode_bf16(p, stream);
        case GDN_F16: return launch_decode_f16(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

namespace {
// This unit's watchdog word (the wait-timeout self-test below), read and cleared.
cudaError_t read_own_watchdog(unsigned *flag, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_watchdog, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
    const unsigned zero = 0;
    if (*flag) e = cudaMemcpyToSymbolAsync(g_watchdog, &zero, sizeof(unsigned), 0,
                                           cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return e;
}

// A wait that cannot complete: the barrier's one arrival comes with 16 expected bytes and no
// copy ever sends them, so the bounded wait runs out, sets the watchdog word and returns.
__global__ void gdn_wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
        mbar_arrive_expect_tx(&bar, 16);
    }
    __syncthreads();
    mbar_wait_bounded(&bar, 0, limit_ns);
}
}  // namespace

cudaError_t launch_wait_timeout(cudaStream_t stream, uint64_t limit_ns) {
    gdn_wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t decode_watchdog(unsigned *flag, cudaStream_t stream) {
    cudaError_t (*const words[])(unsigned *, cudaStream_t) = {
        read_own_watchdog, decode_watchdog_f32, decode_watchdog_bf16, decode_watchdog_f16};
    unsigned any = 0;
    for (auto read : words) {
        unsigned f = 0;
        const cudaError_t e = read(&f, stream);
        if (e != cudaSuccess) return e;
        any |= f;
    }
    *flag = any;
    return cudaSuccess;
}

}  // namespace gdn
