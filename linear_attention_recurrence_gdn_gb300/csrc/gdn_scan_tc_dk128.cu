// gdn_scan_tc_dk128.cu -- the tensor-core scan for Dk = 128 (every activation type and Dv).
#include "gdn_scan_tc.cuh"

namespace gdn {

cudaError_t launch_scan_tc_dk128(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream) {
    return launch_tc_dk<128>(p, sp, stream);
}

// CTAs that the whole-sequence block-kernel launch of a 16-bit Dk = Dv = 128 scan would give
// the busiest SM, at once or in waves (the candidates of launch_tc_dv for that shape).
cudaError_t scan_tc_dk128_plan(const gdn_params &p, int64_t *per_sm, int *ctas_per_head) {
    const ScanSplit whole{1, p.S, 0, nullptr, nullptr, nullptr};
    constexpr int nws[3] = {8, 4, 2};                    // row warps per CTA, as launched below
    int best = -1;
    const cudaError_t e = p.act_dtype == GDN_BF16
                              ? choose_tc<__nv_bfloat16, 128, 128, 8, 4, 2>(p, whole, &best, per_sm)
                              : choose_tc<__half, 128, 128, 8, 4, 2>(p, whole, &best, per_sm);
    *ctas_per_head = e == cudaSuccess ? 128 / (16 * nws[best]) : 1;
    return e;
}

cudaError_t scan_watchdog_dk128(unsigned *flag, cudaStream_t stream) {
    return read_watchdog(flag, stream);
}

}  // namespace gdn
