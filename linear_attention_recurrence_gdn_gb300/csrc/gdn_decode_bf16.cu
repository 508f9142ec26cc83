// gdn_decode_bf16.cu -- the decode step for bf16 activations (every Dk, Dv).
#include "gdn_decode.cuh"

namespace gdn {

cudaError_t launch_decode_bf16(const gdn_params &p, cudaStream_t stream) {
    return launch_dim<__nv_bfloat16>(p, stream);
}

cudaError_t decode_watchdog_bf16(unsigned *flag, cudaStream_t stream) {
    return read_decode_watchdog(flag, stream);
}

}  // namespace gdn
