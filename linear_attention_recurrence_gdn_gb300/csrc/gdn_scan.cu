// gdn_scan.cu -- the scan entry behind gdn_scan().
//
// The recurrence and the gated RMSNorm run in the tensor-core kernel of gdn_scan_tc.cuh,
// instantiated per key head dim in gdn_scan_tc_dk*.cu: the norm, which couples all Dv rows of a
// head (logicaffeine_compile::codegen_cuda::gdn, GDN_KERNELS: "needs the whole head"), is
// applied by the CTA that owns the head, or by the cluster of CTAs a head's rows are split
// over.
#include "gdn_internal.h"

namespace gdn {

cudaError_t launch_scan(const gdn_params &p, cudaStream_t stream) {
    if ((p.flags & GDN_FLAG_SCAN_TMEM) && scan_umma_supported(p)) return launch_scan_umma(p, stream);
    switch (p.Dk) {
        case 16: return launch_scan_tc_dk16(p, stream);
        case 32: return launch_scan_tc_dk32(p, stream);
        case 64: return launch_scan_tc_dk64(p, stream);
        case 128: return launch_scan_tc_dk128(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t scan_watchdog(unsigned *flag, cudaStream_t stream) {
    unsigned f[5] = {0, 0, 0, 0, 0};
    cudaError_t e;
    if ((e = scan_watchdog_dk16(&f[0], stream)) != cudaSuccess) return e;
    if ((e = scan_watchdog_dk32(&f[1], stream)) != cudaSuccess) return e;
    if ((e = scan_watchdog_dk64(&f[2], stream)) != cudaSuccess) return e;
    if ((e = scan_watchdog_dk128(&f[3], stream)) != cudaSuccess) return e;
    if ((e = scan_umma_watchdog(&f[4], stream)) != cudaSuccess) return e;
    *flag = f[0] | f[1] | f[2] | f[3] | f[4];
    return cudaSuccess;
}

}  // namespace gdn
