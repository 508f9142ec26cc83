// gdn_decode_f16.cu -- the decode step for f16 activations (every Dk, Dv).
#include "gdn_decode.cuh"

namespace gdn {

cudaError_t launch_decode_f16(const gdn_params &p, cudaStream_t stream) {
    return launch_dim<__half>(p, stream);
}

cudaError_t decode_watchdog_f16(unsigned *flag, cudaStream_t stream) {
    return read_decode_watchdog(flag, stream);
}

}  // namespace gdn
