// gdn_scan_tc_dk256.cu -- the tensor-core scan for Dk = 256 (every activation type and Dv).
#include "gdn_scan_tc.cuh"

namespace gdn {

cudaError_t launch_scan_tc_dk256(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream) {
    return launch_tc_dk<256>(p, sp, stream);
}

cudaError_t scan_watchdog_dk256(unsigned *flag, cudaStream_t stream) {
    return read_watchdog(flag, stream);
}

}  // namespace gdn
