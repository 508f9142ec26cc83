// gdn_scan_tc_dk16.cu -- the tensor-core scan for Dk = 16 (every activation type and Dv).
#include "gdn_scan_tc.cuh"

namespace gdn {

cudaError_t launch_scan_tc_dk16(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream) {
    return launch_tc_dk<16>(p, sp, stream);
}

cudaError_t scan_watchdog_dk16(unsigned *flag, cudaStream_t stream) {
    return read_watchdog(flag, stream);
}

}  // namespace gdn
