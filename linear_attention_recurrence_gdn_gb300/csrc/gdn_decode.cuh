// gdn_decode.cuh -- single-token GDN step, one HBM read and one HBM write of every state row.
//
// Algorithm: logicaffeine_compile::codegen_cuda::gdn, "The fusion": because the update is
// affine in S, o[a] = alpha (S_old q^)[a] + coef[a] (k^ . q^) with coef[a] = beta (v[a] -
// alpha u[a]), so one pass over a state row gives u[a] = S_old[a,:] k^ and w[a] = S_old[a,:] q^,
// and the updated row alpha S_old[a,:] + coef[a] k^ is formed in the registers that already
// hold it.  The gated RMSNorm (GDN_KERNELS: "needs the whole head") runs in the same CTA
// because one CTA owns a whole head at a time, so there is no second kernel and o never
// round-trips through memory.
//
// GB300 mapping (differs from the page's one-block-per-(head, row) launch):
//   * persistent CTAs, one per SM for Dk = Dv = 128: a CTA processes a contiguous range of
//     heads (up to 32 heads per CTA; measured faster there) or heads c, c + grid, ...
//     A unit's state (64 KB), its q, k, v and z rows arrive in shared memory by bulk
//     asynchronous copies (TMA, cp.async.bulk) that complete on an mbarrier; NST stages keep
//     the next unit's copy in flight while the current one is computed.  Measured on GB300:
//     two stages beat three -- the state is updated in place, and HBM serves an in-place
//     stream best when a row's write follows its read closely;
//   * a unit of work is a head, or for heads of more than 64 KB of state (a head dim of 256)
//     a block of its rows; a head's units run back to back on one CTA, and the gated RMSNorm
//     then keeps the head's gated outputs in shared memory until its last unit;
//   * every warp owns 16 rows of the unit (8 for Dk = 256); a row is split over L lanes (L = 8
//     for Dk = 128 and 256), each lane holding NV float4 column groups (NV = 4; 8 for
//     Dk = 256), read from shared memory without bank conflicts (8 lanes read one 128-byte
//     run);
//   * row dot products reduce over the L lanes of the row with xor shuffles (log2 L stages);
//   * q^, k^ are normalised in registers (the same lane layout, so the norm sums also reduce
//     over L lanes); k^.q^ is one scalar per head, as the page notes;
//   * the updated rows go from the registers back into their stage in shared memory and out to
//     HBM as one bulk copy per unit (TMA), which leaves the load/store units to the
//     shared-memory traffic; the stage is refilled once that copy has read it.
#pragma once

#include <math.h>

#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tma.cuh"

namespace gdn {
namespace {

template <int DK> struct DecodeGeom;
// float4s per lane per row (NV) and rows per warp (RW): Dk = 128 uses 8 lanes per row and 16
// rows per warp; Dk = 256 8 lanes per row with 8 float4 each and 8 rows per warp (the same 64
// state floats per lane); every other Dk (a multiple of 16) 4 lanes per row with Dk / 16 float4.
template <int DK> struct DecodeGeom { static constexpr int NV = DK / 16, RW = 16; };
template <> struct DecodeGeom<128> { static constexpr int NV = 4, RW = 16; };
template <> struct DecodeGeom<256> { static constexpr int NV = 8, RW = 8; };

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Rows of one unit of work: the whole head when its state is at most 64 KB, else the largest
// divisor of Dv that is a multiple of 16 with at most 64 KB of state (a head's row blocks then
// run one after another on the same CTA).
constexpr int decode_rows(int dk, int dv) {
    if (dv * dk <= 16384) return dv;
    for (int r = dv; r >= 16; r -= 16)
        if (dv % r == 0 && r * dk <= 16384) return r;
    return 16;
}

// Tuning knobs (defaults are the measured best on GB300):
//   GDN_DECODE_STAGES_128  pipeline stages for Dk = Dv = 128 (64 KB of state each)
//   GDN_DECODE_SPLIT       bulk copies a head's state is cut into
//   GDN_DECODE_LDGSTS      1: per-thread cp.async (LSU path) instead of TMA bulk copies
#ifndef GDN_DECODE_STAGES_128
#define GDN_DECODE_STAGES_128 2
#endif
#ifndef GDN_DECODE_SPLIT
#define GDN_DECODE_SPLIT 1
#endif
#ifndef GDN_DECODE_LDGSTS
#define GDN_DECODE_LDGSTS 0
#endif
//   GDN_DECODE_LATE_ISSUE  1: issue the next copy into a freed stage after the row updates
//   GDN_DECODE_MINB        minimum resident CTAs per SM requested from the compiler
#ifndef GDN_DECODE_LATE_ISSUE
#define GDN_DECODE_LATE_ISSUE 1
#endif
#ifndef GDN_DECODE_MINB
#define GDN_DECODE_MINB 1
#endif
//   GDN_DECODE_BULK_STORE  1: updated rows go back into the stage and out by one bulk copy per
//                          unit, the stage refilled at the next unit's start; 0: float4 stores
//                          from the registers.  Measured on GB300 (B = 32 / 64 / 256): 5351 /
//                          5877 / 6591 GB/s against 5340 / 5860 / 6584
#ifndef GDN_DECODE_BULK_STORE
#define GDN_DECODE_BULK_STORE 1
#endif
#if GDN_DECODE_BULK_STORE && (GDN_DECODE_LDGSTS || !GDN_DECODE_LATE_ISSUE)
#error "GDN_DECODE_BULK_STORE needs the TMA copies and the late reissue"
#endif
//   GDN_DECODE_CONTIG_MAX  most heads per CTA for which a CTA takes a contiguous range of heads
#ifndef GDN_DECODE_CONTIG_MAX
#define GDN_DECODE_CONTIG_MAX 32
#endif

template <typename TA, int DK, int DV> struct DecodeCfg {
    static constexpr int NV = DecodeGeom<DK>::NV;   // float4 per lane per row
    static constexpr int RW = DecodeGeom<DK>::RW;   // rows per warp
    static constexpr int L = DK / (4 * NV);         // lanes per row
    static constexpr int RPS = 32 / L;              // rows covered by one warp-wide access
    static constexpr int R = RW / RPS;              // row slots per lane
    static constexpr int RBK = decode_rows(DK, DV); // rows per unit (a row block of a head)
    static constexpr int NRBK = DV / RBK;           // units per head
    static constexpr int NWARPS = RBK / RW;
    static constexpr int NT = NWARPS * 32;
    static constexpr int STATE = RBK * DK;          // state floats per unit
    // stages: 2 for 64 KB heads (measured best) and for 32 KB heads (then several CTAs share
    // an SM: Dk = 128, Dv = 64 ran at 5261 GB/s with 2 stages, 4136 GB/s with 4), else 4
    static constexpr int NST = (STATE >= 128 * 128) ? GDN_DECODE_STAGES_128 : (STATE >= 64 * 128 ? 2 : 4);
    // shared-memory layout (every copy destination 16-byte aligned)
    static constexpr size_t ST_OFF = 0;
    static constexpr size_t Q_OFF = ST_OFF + size_t(NST) * STATE * 4;
    static constexpr size_t K_OFF = Q_OFF + size_t(NST) * DK * sizeof(TA);
    static constexpr size_t V_OFF = K_OFF + size_t(NST) * DK * sizeof(TA);
    static constexpr size_t Z_OFF = V_OFF + size_t(NST) * RBK * sizeof(TA);
    static constexpr size_t BAR_OFF = align_up(Z_OFF + size_t(NST) * RBK * sizeof(TA), 16);
    static constexpr size_t RED_OFF = BAR_OFF + size_t(NST) * 8;
    static constexpr size_t XO_OFF = align_up(RED_OFF + size_t(NWARPS) * 4, 16);
    // a head of several units keeps its gated outputs here until its last unit
    static constexpr size_t BYTES = XO_OFF + (NRBK > 1 ? size_t(DV) * 4 : 0);
    static_assert(L * 4 * NV == DK && RPS * L == 32 && R * RPS == RW, "geometry");
    static_assert(DV % RBK == 0 && RBK % RW == 0 && NWARPS >= 1, "row blocks");
    static_assert(DK * sizeof(TA) % 16 == 0 && RBK * sizeof(TA) % 16 == 0, "bulk copy sizes");
};

template <typename TA, int DK, int DV>
__global__ void __launch_bounds__(DecodeCfg<TA, DK, DV>::NT, GDN_DECODE_MINB)
gdn_decode_kernel(const gdn_params p, int64_t nheads, int64_t per) {
    using C = DecodeCfg<TA, DK, DV>;
    using A = Act<TA>;
    constexpr int NV = C::NV, L = C::L, RPS = C::RPS, R = C::R, NST = C::NST;
    constexpr int STATE = C::STATE, RBK = C::RBK, NRBK = C::NRBK;

    extern __shared__ __align__(128) unsigned char smem[];
    float *st_s = reinterpret_cast<float *>(smem + C::ST_OFF);
    TA *q_s = reinterpret_cast<TA *>(smem + C::Q_OFF);
    TA *k_s = reinterpret_cast<TA *>(smem + C::K_OFF);
    TA *v_s = reinterpret_cast<TA *>(smem + C::V_OFF);
    TA *z_s = reinterpret_cast<TA *>(smem + C::Z_OFF);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    float *red = reinterpret_cast<float *>(smem + C::RED_OFF);
    float *xo = reinterpret_cast<float *>(smem + C::XO_OFF);

    const bool gated = p.z != nullptr;
    // host_io: q, k, v, z (and the gates, y) may be in mapped host memory; the threads stage
    // the inputs with plain loads (below) and the stage copies carry the state only
    const bool host_io = (p.flags & GDN_FLAG_HOST_IO) != 0;
    const unsigned tx =
        STATE * 4 + (host_io ? 0u : 2 * DK * sizeof(TA) + (gated ? 2 : 1) * RBK * sizeof(TA));
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane / L;                              // row within a warp-wide access
    const int part = lane % L;                           // column part of the row
    const int row0 = warp * C::RW + g;                   // unit rows row0 + r * RPS
    const int group = p.Hv / p.Hk;
    // this CTA's heads: the contiguous range [blockIdx.x * per, + per) when per > 0, else
    // blockIdx.x, blockIdx.x + grid, ...; unit u = (head i, row block rb)
    const bool contig = per > 0;
    const int64_t first = contig ? static_cast<int64_t>(blockIdx.x) * per : blockIdx.x;
    const int64_t stride = contig ? 1 : gridDim.x;
    const int64_t nmine =
        contig ? (first < nheads ? min(per, nheads - first) : 0)
               : ((blockIdx.x < nheads) ? (nheads - 1 - blockIdx.x) / gridDim.x + 1 : 0);
    const int64_t nunits = nmine * NRBK;

    if (tid == 0) {
        for (int s = 0; s < NST; s++) mbar_init(&bar[s], 1);
        mbar_init_fence();
    }
    __syncthreads();
    // Programmatic dependent launch: the next kernel on the stream may start its set-up now;
    // this one reads nothing from global memory before the previous kernel (the step that
    // wrote the state, or whatever produced the inputs) has completed.  Both are no-ops in a
    // plain launch.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    auto head_of = [&](int64_t i) -> int64_t { return first + i * stride; };
#if GDN_DECODE_LDGSTS
    // every thread copies the state float4s it will read itself; the threads copy the small
    // vectors in turn; one cp.async group per unit (empty groups keep the count uniform)
    auto issue = [&](int64_t u, int s) {
        if (u < nunits) {
            const int64_t h = head_of(u / NRBK);
            const int rb = static_cast<int>(u % NRBK);
            const int b = static_cast<int>(h / p.Hv);
            const int hk = static_cast<int>(h - static_cast<int64_t>(b) * p.Hv) / group;
            const int64_t qo = (static_cast<int64_t>(b) * p.Hk + hk) * DK;
            const int64_t vo = h * DV + rb * RBK;
            const float *src = p.state + h * (static_cast<int64_t>(DV) * DK) + rb * STATE;
            float *dst = st_s + s * STATE;
#pragma unroll
            for (int r = 0; r < R; r++)
#pragma unroll
                for (int c = 0; c < NV; c++) {
                    const int off = (row0 + r * RPS) * DK + 4 * (c * L + part);
                    cp_async16(dst + off, src + off);
                }
            constexpr int QP = DK * sizeof(TA) / 16, VP = RBK * sizeof(TA) / 16;
            for (int t = tid; t < (host_io ? 0 : QP); t += C::NT) {
                cp_async16(reinterpret_cast<char *>(q_s + s * DK) + 16 * t,
                           reinterpret_cast<const char *>(static_cast<const TA *>(p.q) + qo) + 16 * t);
                cp_async16(reinterpret_cast<char *>(k_s + s * DK) + 16 * t,
                           reinterpret_cast<const char *>(static_cast<const TA *>(p.k) + qo) + 16 * t);
            }
            for (int t = tid; t < (host_io ? 0 : VP); t += C::NT) {
                cp_async16(reinterpret_cast<char *>(v_s + s * RBK) + 16 * t,
                           reinterpret_cast<const char *>(static_cast<const TA *>(p.v) + vo) + 16 * t);
                if (gated)
                    cp_async16(reinterpret_cast<char *>(z_s + s * RBK) + 16 * t,
                               reinterpret_cast<const char *>(static_cast<const TA *>(p.z) + vo) + 16 * t);
            }
        }
        cp_async_commit();
    };
    for (int64_t u = 0; u < NST; u++) issue(u, static_cast<int>(u));
#else
    // thread 0: bulk copies of unit u's state rows and inputs into stage s
    auto issue = [&](int64_t u, int s) {
        const int64_t h = head_of(u / NRBK);
        const int rb = static_cast<int>(u % NRBK);
        const int b = static_cast<int>(h / p.Hv);
        const int hk = static_cast<int>(h - static_cast<int64_t>(b) * p.Hv) / group;
        const int64_t qo = (static_cast<int64_t>(b) * p.Hk + hk) * DK;   // S == 1
        const int64_t vo = h * DV + rb * RBK;
        const float *src = p.state + h * (static_cast<int64_t>(DV) * DK) + rb * STATE;
        constexpr int SPLIT = (STATE * 4 / GDN_DECODE_SPLIT) % 16 == 0 ? GDN_DECODE_SPLIT : 1;
        constexpr int PIECE = STATE / SPLIT;
        mbar_arrive_expect_tx(&bar[s], tx);
#pragma unroll
        for (int j = 0; j < SPLIT; j++)
            bulk_g2s(st_s + s * STATE + j * PIECE, src + j * PIECE, PIECE * 4, &bar[s]);
        if (host_io) return;
        bulk_g2s(q_s + s * DK, static_cast<const TA *>(p.q) + qo, DK * sizeof(TA), &bar[s]);
        bulk_g2s(k_s + s * DK, static_cast<const TA *>(p.k) + qo, DK * sizeof(TA), &bar[s]);
        bulk_g2s(v_s + s * RBK, static_cast<const TA *>(p.v) + vo, RBK * sizeof(TA), &bar[s]);
        if (gated)
            bulk_g2s(z_s + s * RBK, static_cast<const TA *>(p.z) + vo, RBK * sizeof(TA), &bar[s]);
    };
    if (tid == 0)
        for (int64_t u = 0; u < nunits && u < NST; u++) issue(u, static_cast<int>(u));
#endif

    // host_io: the q, k, v, z rows of a unit travel as 16-byte pieces, loaded by the threads in
    // turn two units ahead and stored into the unit's stage one unit ahead (its previous unit
    // has consumed that stage by then); the loop-top barrier orders the stores before the reads
    constexpr int QP = DK * sizeof(TA) / 16, VP = RBK * sizeof(TA) / 16;
    constexpr int PPT = (2 * QP + 2 * VP + C::NT - 1) / C::NT;   // pieces per thread, at most
    const int npieces = 2 * QP + (gated ? 2 : 1) * VP;
    uint4 held[PPT];
    auto piece = [&](int64_t u, int i, int s, const uint4 *&src, uint4 *&dst) {
        const int64_t h = head_of(u / NRBK);
        const int rb = static_cast<int>(u % NRBK);
        const int b = static_cast<int>(h / p.Hv);
        const int hk = static_cast<int>(h - static_cast<int64_t>(b) * p.Hv) / group;
        const int64_t qo = (static_cast<int64_t>(b) * p.Hk + hk) * DK;
        const int64_t vo = h * DV + rb * RBK;
        if (i < QP) {
            src = reinterpret_cast<const uint4 *>(static_cast<const TA *>(p.q) + qo) + i;
            dst = reinterpret_cast<uint4 *>(q_s + s * DK) + i;
        } else if (i < 2 * QP) {
            src = reinterpret_cast<const uint4 *>(static_cast<const TA *>(p.k) + qo) + (i - QP);
            dst = reinterpret_cast<uint4 *>(k_s + s * DK) + (i - QP);
        } else if (i < 2 * QP + VP) {
            src = reinterpret_cast<const uint4 *>(static_cast<const TA *>(p.v) + vo) + (i - 2 * QP);
            dst = reinterpret_cast<uint4 *>(v_s + s * RBK) + (i - 2 * QP);
        } else {
            src = reinterpret_cast<const uint4 *>(static_cast<const TA *>(p.z) + vo) + (i - 2 * QP - VP);
            dst = reinterpret_cast<uint4 *>(z_s + s * RBK) + (i - 2 * QP - VP);
        }
    };
    auto load_pieces = [&](int64_t u) {
#pragma unroll
        for (int j = 0; j < PPT; j++) {
            const int i = tid + j * C::NT;
            if (i < npieces) {
                const uint4 *src;
                uint4 *dst;
                piece(u, i, 0, src, dst);
                held[j] = *src;
            }
        }
    };
    auto store_pieces = [&](int64_t u) {
#pragma unroll
        for (int j = 0; j < PPT; j++) {
            const int i = tid + j * C::NT;
            if (i < npieces) {
                const uint4 *src;
                uint4 *dst;
                piece(u, i, static_cast<int>(u % NST), src, dst);
                *dst = held[j];
            }
        }
    };
    if (host_io && nunits > 0) {
        load_pieces(0);
        store_pieces(0);
        if (nunits > 1) load_pieces(1);
    }

    // gates of the next head are prefetched one head ahead into registers
    float gl = 0.f, gb = 0.f, alpha = 0.f, beta = 0.f;
    if (nmine > 0) {
        gl = load_gate(p.log_decay, p.gate_dtype, head_of(0));
        gb = load_gate(p.beta, p.gate_dtype, head_of(0));
    }
    const float inv_sqrt_dk = rsqrtf(static_cast<float>(DK));
    float head_ss = 0.f;                                 // sum of squares over a head's units

    for (int64_t u = 0; u < nunits; u++) {
        const int s = static_cast<int>(u % NST);
        const int64_t i = u / NRBK;
        const int rb = static_cast<int>(u % NRBK);
        const int64_t h = head_of(i);
#if GDN_DECODE_BULK_STORE
        if (tid == 0 && u >= 1) {          // the previous unit's store has read its stage
            bulk_wait_read_all();
            if (u - 1 + NST < nunits) issue(u - 1 + NST, static_cast<int>((u - 1) % NST));
        }
#endif
        if (rb == 0) {
            alpha = expf(gl);
            beta = gb;
            if (i + 1 < nmine) {
                gl = load_gate(p.log_decay, p.gate_dtype, head_of(i + 1));
                gb = load_gate(p.beta, p.gate_dtype, head_of(i + 1));
            }
        }

#if GDN_DECODE_LDGSTS
        cp_async_wait<NST - 1>();
        __syncthreads();
#else
        // wait for stage s; a timed-out wait (watchdog set) ends the whole CTA together
        const bool ok = mbar_wait_bounded(&bar[s], static_cast<unsigned>((u / NST) & 1));
        if (__syncthreads_or(!ok)) {
            if (tid == 0) { // let this CTA's copies still in flight land before leaving
                for (int64_t j = u; j < nunits && j < u + NST; j++)
                    mbar_wait_bounded(&bar[j % NST], static_cast<unsigned>((j / NST) & 1));
#if GDN_DECODE_BULK_STORE
                bulk_wait_all();
#endif
            }
            return;
        }
#endif

        // 1. this lane's state rows and the head's inputs, from shared memory
        const float *S = st_s + s * STATE;
        float4 sr[R][NV];
#pragma unroll
        for (int r = 0; r < R; r++)
#pragma unroll
            for (int c = 0; c < NV; c++)
                sr[r][c] = *reinterpret_cast<const float4 *>(
                    S + (row0 + r * RPS) * DK + 4 * (c * L + part));
        float4 kh[NV], qh[NV];
#pragma unroll
        for (int c = 0; c < NV; c++) {
            kh[c] = A::four(k_s + s * DK + 4 * (c * L + part));
            qh[c] = A::four(q_s + s * DK + 4 * (c * L + part));
        }
        float vr[R], zr[R];
#pragma unroll
        for (int r = 0; r < R; r++) {
            vr[r] = A::one(v_s + s * RBK + row0 + r * RPS);
            zr[r] = gated ? A::one(z_s + s * RBK + row0 + r * RPS) : 0.f;
        }
#if !GDN_DECODE_BULK_STORE
        __syncthreads();                                 // stage s consumed by every thread
#endif
        if (host_io) {                                   // next unit's inputs into its stage
            if (u + 1 < nunits) store_pieces(u + 1);
            if (u + 2 < nunits) load_pieces(u + 2);
        }
#if !GDN_DECODE_LATE_ISSUE
#if GDN_DECODE_LDGSTS
        issue(u + NST, s);
#else
        if (tid == 0 && u + NST < nunits) issue(u + NST, s);
#endif
#endif

        // 2. q^, k^ and k^.q^
        float ssk = 0.f, ssq = 0.f, skq = 0.f;
#pragma unroll
        for (int c = 0; c < NV; c++) {
            ssk = dot4(kh[c], kh[c], ssk);
            ssq = dot4(qh[c], qh[c], ssq);
            skq = dot4(kh[c], qh[c], skq);
        }
        ssk = group_sum<L>(ssk);
        ssq = group_sum<L>(ssq);
        skq = group_sum<L>(skq);
        const float rk = rsqrtf(ssk + p.qk_eps);
        const float rq = rsqrtf(ssq + p.qk_eps) * inv_sqrt_dk;
#pragma unroll
        for (int c = 0; c < NV; c++) {
            kh[c].x *= rk; kh[c].y *= rk; kh[c].z *= rk; kh[c].w *= rk;
            qh[c].x *= rq; qh[c].y *= rq; qh[c].z *= rq; qh[c].w *= rq;
        }
        const float kq = skq * rk * rq;                  // k^ . q^, one scalar per head

        // 3. fused pass per row: u, w from the registers, updated row straight to HBM (or back
        //    into the stage, for one bulk copy of the unit)
        float *Sg = p.state + h * (static_cast<int64_t>(DV) * DK) + rb * STATE;
#if GDN_DECODE_BULK_STORE
        float *Sw = st_s + s * STATE;
#else
        float *Sw = Sg;
#endif
        float o[R];
#pragma unroll
        for (int r = 0; r < R; r++) {
            float pu = 0.f, pw = 0.f;
#pragma unroll
            for (int c = 0; c < NV; c++) {
                pu = dot4(sr[r][c], kh[c], pu);
                pw = dot4(sr[r][c], qh[c], pw);
            }
            pu = group_sum<L>(pu);
            pw = group_sum<L>(pw);
            const float coef = beta * (vr[r] - alpha * pu);
            float *row = Sw + (row0 + r * RPS) * DK;
#pragma unroll
            for (int c = 0; c < NV; c++) {
                float4 n;
                n.x = fmaf(alpha, sr[r][c].x, coef * kh[c].x);
                n.y = fmaf(alpha, sr[r][c].y, coef * kh[c].y);
                n.z = fmaf(alpha, sr[r][c].z, coef * kh[c].z);
                n.w = fmaf(alpha, sr[r][c].w, coef * kh[c].w);
                *reinterpret_cast<float4 *>(row + 4 * (c * L + part)) = n;
            }
            o[r] = fmaf(alpha, pw, coef * kq);
        }

#if GDN_DECODE_BULK_STORE
        fence_async_smem_writes();
        __syncthreads();                                 // the unit's rows are in stage s
        if (tid == 0) {
            bulk_s2g(Sg, st_s + s * STATE, STATE * 4);
            bulk_commit();
        }
#elif GDN_DECODE_LATE_ISSUE
#if GDN_DECODE_LDGSTS
        issue(u + NST, s);
#else
        if (tid == 0 && u + NST < nunits) issue(u + NST, s);
#endif
#endif

        // 4. output: gated RMSNorm over the head's Dv rows, or the raw o
        float *yp = p.y + h * DV + rb * RBK;
        if (gated) {
            float x[R];
            float ss = 0.f;
#pragma unroll
            for (int r = 0; r < R; r++) {
                x[r] = o[r] * silu(zr[r]);
                ss = fmaf(x[r], x[r], ss);
            }
            if constexpr (NRBK > 1) {
                if (part == 0) {
#pragma unroll
                    for (int r = 0; r < R; r++) xo[rb * RBK + row0 + r * RPS] = x[r];
                }
            }
            // every row's x is replicated over its L lanes: count it once (part == 0)
            ss = (part == 0) ? ss : 0.f;
            ss = group_sum<32>(ss);
            if (lane == 0) red[warp] = ss;
            __syncthreads();                             // red (and this unit's xo) complete
            float total = 0.f;
#pragma unroll
            for (int w = 0; w < C::NWARPS; w++) total += red[w];
            if constexpr (NRBK == 1) {
                const float rr = rsqrtf(total / static_cast<float>(DV) + p.norm_eps);
                if (part == 0) {
#pragma unroll
                    for (int r = 0; r < R; r++) {
                        const int a = row0 + r * RPS;
                        yp[a] = x[r] * rr * p.gn[a];
                    }
                }
            } else {
                head_ss += total;
                if (rb == NRBK - 1) {                    // the head's last unit: all of y
                    const float rr = rsqrtf(head_ss / static_cast<float>(DV) + p.norm_eps);
                    for (int a = tid; a < DV; a += C::NT) p.y[h * DV + a] = xo[a] * rr * p.gn[a];
                    head_ss = 0.f;
                }
            }
        } else if (part == 0) {
#pragma unroll
            for (int r = 0; r < R; r++) yp[row0 + r * RPS] = o[r];
        }
    }
#if GDN_DECODE_BULK_STORE
    if (tid == 0) bulk_wait_all();                       // shared memory outlives the stores
#endif
}

constexpr int kMaxDevices = 64;

// Per-device launch configuration of one kernel instantiation, computed on first use (the
// attribute call and the occupancy query cost more than a small decode step's launch).
struct LaunchSlots {
    int slots[kMaxDevices] = {};   // resident CTAs on the whole device; 0 = not computed
};

template <typename TA, int DK, int DV>
cudaError_t launch_typed(const gdn_params &p, cudaStream_t stream) {
    using C = DecodeCfg<TA, DK, DV>;
    static LaunchSlots cache;
    auto kern = gdn_decode_kernel<TA, DK, DV>;
    const int bytes = static_cast<int>(C::BYTES);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int slots = (dev >= 0 && dev < kMaxDevices) ? cache.slots[dev] : 0;
    if (slots == 0) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) !=
            cudaSuccess)
            return e;
        int occ = 0, sms = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::NT, bytes)) !=
            cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        slots = std::max(1, sms) * std::max(1, occ);
        if (dev >= 0 && dev < kMaxDevices) cache.slots[dev] = slots;
    }
    const int64_t heads = static_cast<int64_t>(p.B) * p.Hv;
    int64_t grid = std::min<int64_t>(heads, slots);
    // Up to GDN_DECODE_CONTIG_MAX heads per CTA, a CTA takes a contiguous range of heads (the
    // fewest CTAs with the same most heads per CTA); beyond, every grid-th head.  Measured on
    // two GB300s (Dk = Dv = 128, bf16; contiguous vs every grid-th): 7 heads per CTA (B = 32)
    // 5386 vs 5288 and 5370 vs 5295 GB/s; 14 (B = 64) 5928 vs 5860 and 5863 vs 5861; 54
    // (B = 256, one GB300) 6599 vs 6625.
    int64_t per = (heads + grid - 1) / grid;
    if (per <= GDN_DECODE_CONTIG_MAX) grid = (heads + per - 1) / per;
    else per = 0;
    // launched as a programmatic dependent of the previous kernel on the stream: its CTAs
    // become resident as that kernel's CTAs retire and wait (griddepcontrol.wait) for its
    // completion, which hides the launch gap between consecutive decode steps
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::NT);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, heads, per);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename TA, int DK>
cudaError_t launch_dv(const gdn_params &p, cudaStream_t stream) {
    switch (p.Dv) {
        case 16: return launch_typed<TA, DK, 16>(p, stream);
        case 32: return launch_typed<TA, DK, 32>(p, stream);
        case 48: return launch_typed<TA, DK, 48>(p, stream);
        case 64: return launch_typed<TA, DK, 64>(p, stream);
        case 80: return launch_typed<TA, DK, 80>(p, stream);
        case 96: return launch_typed<TA, DK, 96>(p, stream);
        case 112: return launch_typed<TA, DK, 112>(p, stream);
        case 128: return launch_typed<TA, DK, 128>(p, stream);
        case 256: return launch_typed<TA, DK, 256>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <typename TA>
cudaError_t launch_dim(const gdn_params &p, cudaStream_t stream) {
    switch (p.Dk) {
        case 16: return launch_dv<TA, 16>(p, stream);
        case 32: return launch_dv<TA, 32>(p, stream);
        case 48: return launch_dv<TA, 48>(p, stream);
        case 64: return launch_dv<TA, 64>(p, stream);
        case 80: return launch_dv<TA, 80>(p, stream);
        case 96: return launch_dv<TA, 96>(p, stream);
        case 112: return launch_dv<TA, 112>(p, stream);
        case 128: return launch_dv<TA, 128>(p, stream);
        case 256: return launch_dv<TA, 256>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

// This unit's watchdog word, read and cleared (synchronises `stream`).
inline cudaError_t read_decode_watchdog(unsigned *flag, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_watchdog, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
    const unsigned zero = 0;
    if (*flag) e = cudaMemcpyToSymbolAsync(g_watchdog, &zero, sizeof(unsigned), 0,
                                           cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return e;
}

}  // namespace
}  // namespace gdn
