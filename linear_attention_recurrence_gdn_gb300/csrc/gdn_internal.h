// gdn_internal.h -- launchers behind the C ABI (arguments already validated by gdn_api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// One decode step: one CTA per (b, hv) head, gated norm fused in the CTA tail.
cudaError_t launch_decode(const gdn_params &p, cudaStream_t stream);

// Reads and clears the decode kernels' watchdog word (synchronises `stream`).
cudaError_t decode_watchdog(unsigned *flag, cudaStream_t stream);

// One CTA whose mbarrier wait runs out after limit_ns, setting the decode watchdog word.
cudaError_t launch_wait_timeout(cudaStream_t stream, uint64_t limit_ns);

// Multi-token scan (S >= 1): state resident on chip across the time axis.
cudaError_t launch_scan(const gdn_params &p, cudaStream_t stream);

// The scan on tensor cores (gdn_scan_tc.cu).
cudaError_t launch_scan_tc(const gdn_params &p, cudaStream_t stream);

// Reads and clears the scan kernels' watchdog word (synchronises `stream`).
cudaError_t scan_watchdog(unsigned *flag, cudaStream_t stream);

}  // namespace gdn
