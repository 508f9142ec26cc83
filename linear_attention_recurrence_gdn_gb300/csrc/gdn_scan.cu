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
        case 48: return launch_scan_tc_dk48(p, stream);
        case 64: return launch_scan_tc_dk64(p, stream);
        case 80: return launch_scan_tc_dk80(p, stream);
        case 96: return launch_scan_tc_dk96(p, stream);
        case 112: return launch_scan_tc_dk112(p, stream);
        case 128: return launch_scan_tc_dk128(p, stream);
        case 256: return launch_scan_tc_dk256(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t scan_watchdog(unsigned *flag, cudaStream_t stream) {
    cudaError_t (*const words[])(unsigned *, cudaStream_t) = {
        scan_watchdog_dk16,
        scan_watchdog_dk32,
        scan_watchdog_dk48,
        scan_watchdog_dk64,
        scan_watchdog_dk80,
        scan_watchdog_dk96,
        scan_watchdog_dk112,
        scan_watchdog_dk128,
        scan_watchdog_dk256,
        scan_umma_watchdog};
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
