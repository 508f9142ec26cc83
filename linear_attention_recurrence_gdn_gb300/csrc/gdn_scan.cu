// gdn_scan.cu -- the scan entry behind gdn_scan() and the stand-alone gated RMSNorm.
//
// The recurrence itself runs in gdn_scan_tc.cu (tensor cores, memory in registers).  When a
// head's rows are split over several CTAs the gated norm, which couples all Dv rows of a head
// (logicaffeine_compile::codegen_cuda::gdn, GDN_KERNELS: "needs the whole head"), runs here
// afterwards: y <- rmsnorm(o * silu(z)) * GN in place, gate first (module description).
#include <math.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

// Gated RMSNorm in place on y (raw o -> rmsnorm(o * silu(z)) * gn), one warp per (b, t, hv)
// output row.  z has y's layout, so rows are simply consecutive runs of Dv elements.
template <typename TA, int DV>
__global__ void __launch_bounds__(256) gdn_gated_norm_kernel(const gdn_params p, int64_t rows) {
    using A = Act<TA>;
    constexpr int EPL = (DV + 31) / 32;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float *y = p.y + row * DV;
    const TA *z = static_cast<const TA *>(p.z) + row * DV;
    float x[EPL];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        const int j = lane + 32 * i;
        x[i] = (j < DV) ? y[j] * silu(A::one(z + j)) : 0.f;
        ss = fmaf(x[i], x[i], ss);
    }
    ss = group_sum<32>(ss);
    const float rr = rsqrtf(ss / static_cast<float>(DV) + p.norm_eps);
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        const int j = lane + 32 * i;
        if (j < DV) y[j] = x[i] * rr * p.gn[j];
    }
}

template <typename TA>
cudaError_t launch_norm_typed(const gdn_params &p, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(p.B) * p.S * p.Hv;
    const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
    switch (p.Dv) {
        case 16: gdn_gated_norm_kernel<TA, 16><<<blocks, 256, 0, stream>>>(p, rows); break;
        case 32: gdn_gated_norm_kernel<TA, 32><<<blocks, 256, 0, stream>>>(p, rows); break;
        case 64: gdn_gated_norm_kernel<TA, 64><<<blocks, 256, 0, stream>>>(p, rows); break;
        case 128: gdn_gated_norm_kernel<TA, 128><<<blocks, 256, 0, stream>>>(p, rows); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gated_norm(const gdn_params &p, cudaStream_t stream) {
    switch (p.act_dtype) {
        case GDN_F32: return launch_norm_typed<float>(p, stream);
        case GDN_BF16: return launch_norm_typed<__nv_bfloat16>(p, stream);
        case GDN_F16: return launch_norm_typed<__half>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_scan(const gdn_params &p, cudaStream_t stream) {
    return launch_scan_tc(p, stream);
}

}  // namespace gdn
