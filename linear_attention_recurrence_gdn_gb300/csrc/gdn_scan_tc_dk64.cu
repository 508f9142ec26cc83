// gdn_scan_tc_dk64.cu -- the tensor-core scan for Dk = 64 (every activation type and Dv).
#include "gdn_scan_tc.cuh"

namespace gdn {

cudaError_t launch_scan_tc_dk64(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream) {
    return launch_tc_dk<64>(p, sp, stream);
}

cudaError_t scan_watchdog_dk64(unsigned *flag, cudaStream_t stream) {
    return read_watchdog(flag, stream);
}

}  // namespace gdn
