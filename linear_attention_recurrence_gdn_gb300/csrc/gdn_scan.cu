// gdn_scan.cu -- the scan entries behind gdn_scan() and gdn_scan_split().
//
// The recurrence and the gated RMSNorm run in the tensor-core kernel of gdn_scan_tc.cuh,
// instantiated per key head dim in gdn_scan_tc_dk*.cu: the norm, which couples all Dv rows of a
// head (logicaffeine_compile::codegen_cuda::gdn, GDN_KERNELS: "needs the whole head"), is
// applied by the CTA that owns the head, or by the cluster of CTAs a head's rows are split
// over.
//
// Sequence split.  The page's update is affine in the memory (codegen_cuda::gdn, "The fusion"):
// S_t = S_{t-1} A_t + B_t with A_t = alpha_t (I - beta_t k^_t k^_t^T) and B_t = beta_t v_t k^_t^T.
// Over a segment of tokens, then, S_end = S_start M + N with M = A_1 ... A_T (the memory that
// the identity becomes with v = 0) and N = sum_t B_t A_{t+1} ... A_T (the memory reached from
// zeros).  Segments run in parallel twice: once for M and N, once for the outputs from each
// segment's start, which a short sequential composition provides in between.
#include <algorithm>

#include "gdn_internal.h"

namespace gdn {

namespace {

cudaError_t launch_scan_dk(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream) {
    switch (p.Dk) {
        case 16: return launch_scan_tc_dk16(p, sp, stream);
        case 32: return launch_scan_tc_dk32(p, sp, stream);
        case 48: return launch_scan_tc_dk48(p, sp, stream);
        case 64: return launch_scan_tc_dk64(p, sp, stream);
        case 80: return launch_scan_tc_dk80(p, sp, stream);
        case 96: return launch_scan_tc_dk96(p, sp, stream);
        case 112: return launch_scan_tc_dk112(p, sp, stream);
        case 128: return launch_scan_tc_dk128(p, sp, stream);
        case 256: return launch_scan_tc_dk256(p, sp, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Start memories of every segment: St[0] = s0 (zeros when NULL), St[g+1] = St[g] M_g + N_g.
// The rows of a memory are independent, so CTA (head, 16-row block) composes its own rows
// through all segments; its rows of St[g] stay in shared memory between steps.
__global__ void __launch_bounds__(256)
gdn_scan_compose_kernel(const float *s0, const float *M, const float *N, float *St, int64_t bh,
                        int dv, int dk, int nseg) {
    extern __shared__ float cur[];                         // [16][dk]
    const int64_t head = blockIdx.x;
    const int r0 = blockIdx.y * 16;
    const int tid = threadIdx.x;
    const int n = 16 * dk;                                 // outputs of this CTA per step
    const int64_t mem = static_cast<int64_t>(dv) * dk;
    for (int o = tid; o < n; o += blockDim.x) {
        const float v0 = s0 ? s0[head * mem + static_cast<int64_t>(r0) * dk + o] : 0.f;
        cur[o] = v0;
        St[head * mem + static_cast<int64_t>(r0) * dk + o] = v0;
    }
    for (int g = 0; g + 1 < nseg; g++) {
        const float *Mg = M + (static_cast<int64_t>(g) * bh + head) * dk * dk;
        const float *Ng = N + (static_cast<int64_t>(g) * bh + head) * mem + static_cast<int64_t>(r0) * dk;
        float *Sn = St + (static_cast<int64_t>(g + 1) * bh + head) * mem + static_cast<int64_t>(r0) * dk;
        __syncthreads();                                   // cur holds St[g]
        float acc[16];                                     // n / blockDim.x <= 16 (dk <= 256)
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const int o = tid + j * 256;
            if (o >= n) break;
            const int r = o / dk, c = o - r * dk;
            float a = Ng[o];
            for (int i = 0; i < dk; i++) a = fmaf(cur[r * dk + i], Mg[static_cast<int64_t>(i) * dk + c], a);
            acc[j] = a;
        }
        __syncthreads();                                   // every read of St[g] done
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const int o = tid + j * 256;
            if (o >= n) break;
            cur[o] = acc[j];
            Sn[o] = acc[j];
        }
    }
}

}  // namespace

cudaError_t launch_scan(const gdn_params &p, cudaStream_t stream) {
    if (!tiled_dims(p)) return launch_general(p, false, stream);
    if ((p.flags & GDN_FLAG_SCAN_TMEM) && scan_umma_supported(p)) return launch_scan_umma(p, stream);
    if (!(p.flags & (GDN_FLAG_SCAN_TMEM | GDN_FLAG_SCAN_BLOCK16)) && scan_wy_supported(p)) {
        if (p.flags & GDN_FLAG_SCAN_CHUNKED) return launch_scan_wy(p, stream);
        // The chunked kernel runs one CTA per head; the block kernel splits a head's rows over a
        // cluster of CTAs when heads are few.  Measured on GB300 (S 4096, 4 to 256 heads): for
        // f16 the chunked kernel is 1.35-4.8x faster at every head count (the block kernel
        // splits f16 rows into bf16 hi + lo, three MMA terms); for bf16 the block kernel is
        // 1.1-1.17x faster when it splits each head over 2 or 4 CTAs with at most one CTA per
        // SM (up to 64 heads), the chunked kernel 1.06x faster at one CTA per head (128 heads)
        // and 2-3x faster once the block kernel stacks CTAs on an SM.
        if (p.act_dtype != GDN_BF16) return launch_scan_wy(p, stream);
        int64_t per_sm = 0;
        int per_head = 1;
        const cudaError_t e = scan_tc_dk128_plan(p, &per_sm, &per_head);
        if (e != cudaSuccess) return e;
        if (per_sm > 1 || per_head == 1) return launch_scan_wy(p, stream);
    }
    const ScanSplit whole{1, p.S, 0, nullptr, nullptr, nullptr};
    return launch_scan_dk(p, whole, stream);
}

// Segments of ceil(S / nseg) tokens (no empty segment).
static int seg_len_of(int S, int nseg) { return (S + nseg - 1) / nseg; }
static int nseg_of(int S, int nseg) {
    const int len = seg_len_of(S, nseg);
    return (S + len - 1) / len;
}

size_t scan_split_workspace_floats(const gdn_params &p, int nseg) {
    if (p.S < 1 || nseg < 1 || !tiled_dims(p)) return 0;   // general dims: one launch, no split
    const int g = nseg_of(p.S, nseg);
    if (g < 2) return 0;
    const size_t bh = static_cast<size_t>(p.B) * p.Hv;
    const size_t m = bh * p.Dk * p.Dk, nn = bh * p.Dv * p.Dk;
    return (g - 1) * m + (g - 1) * nn + g * nn;            // M, N of all but the last; all starts
}

cudaError_t launch_scan_split(const gdn_params &p, int nseg, float *ws, cudaStream_t stream) {
    if (!tiled_dims(p)) return launch_general(p, false, stream);  // the whole sequence in one launch
    const int len = seg_len_of(p.S, nseg);
    const int g = nseg_of(p.S, nseg);
    if (g < 2) return launch_scan(p, stream);
    const int64_t bh = static_cast<int64_t>(p.B) * p.Hv;
    float *M = ws;                                         // [g-1][bh][Dk][Dk]
    float *N = M + (g - 1) * bh * p.Dk * p.Dk;             // [g-1][bh][Dv][Dk]
    float *St = N + (g - 1) * bh * p.Dv * p.Dk;            // [g][bh][Dv][Dk]
    cudaError_t e;
    // 1. transitions of segments 0 .. g-2 (the identity's Dk rows through the update, v = 0)
    //    and 2. their offsets (from zeros with the real v).  One grid for both when Dk == Dv and
    //    their (segment, head) pairs fit in half the SMs; else two launches (the transitions
    //    have Dk rows).  Measured on GB300 (8 heads, f16, S 16384; one grid / two launches):
    //    2 segments 2.26 / 3.26 ms, 4 segments 1.24 / 1.75 ms, 8 segments 1.33 / 1.08 ms --
    //    beyond half the SMs the one grid is cut into CTAs of 8 row warps, slower here.
    gdn_params pn = p;
    pn.z = nullptr;
    pn.gn = nullptr;
    pn.y = nullptr;
    pn.s0 = nullptr;
    pn.flags = 0;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (p.Dk == p.Dv && 2 * (g - 1) * bh <= sms / 2) {
        if ((e = launch_scan_dk(pn, ScanSplit{2 * (g - 1), len, 3, nullptr, M, N}, stream)) != cudaSuccess)
            return e;
    } else {
        gdn_params pm = pn;
        pm.Dv = p.Dk;
        if ((e = launch_scan_dk(pm, ScanSplit{g - 1, len, 1, nullptr, M, nullptr}, stream)) != cudaSuccess)
            return e;
        if ((e = launch_scan_dk(pn, ScanSplit{g - 1, len, 2, nullptr, N, nullptr}, stream)) != cudaSuccess)
            return e;
    }
    // 3. every segment's start memory
    const int smem = 16 * p.Dk * static_cast<int>(sizeof(float));
    gdn_scan_compose_kernel<<<dim3(static_cast<unsigned>(bh), p.Dv / 16), 256, smem, stream>>>(
        p.s0, M, N, St, bh, p.Dv, p.Dk, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 4. outputs of every segment; the last writes the final memory
    gdn_params po = p;
    po.flags = 0;
    return launch_scan_dk(po, ScanSplit{g, len, 0, St, nullptr, nullptr}, stream);
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
        scan_umma_watchdog,
        scan_wy_watchdog};
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
