// gdn_scan.cu -- the scan entry behind gdn_scan().
//
// The recurrence and the gated RMSNorm run in gdn_scan_tc.cu (tensor cores, memory in
// registers): the norm, which couples all Dv rows of a head (logicaffeine_compile::codegen_cuda::
// gdn, GDN_KERNELS: "needs the whole head"), is applied by the CTA that owns the head, or by the
// cluster of CTAs a head's rows are split over.
#include "gdn_internal.h"

namespace gdn {

cudaError_t launch_scan(const gdn_params &p, cudaStream_t stream) {
    return launch_scan_tc(p, stream);
}

}  // namespace gdn
