// gdn_decode_f32.cu -- the decode step for f32 activations (every Dk, Dv).
#include "gdn_decode.cuh"

namespace gdn {

cudaError_t launch_decode_f32(const gdn_params &p, cudaStream_t stream) {
    return launch_dim<float>(p, stream);
}

cudaError_t decode_watchdog_f32(unsigned *flag, cudaStream_t stream) {
    return read_decode_watchdog(flag, stream);
}

}  // namespace gdn
