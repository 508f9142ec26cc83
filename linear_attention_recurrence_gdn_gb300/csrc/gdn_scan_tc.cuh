// gdn_scan_tc.cuh -- multi-token GDN recurrence on tensor cores, memory resident in registers.
// Kernel and launchers as templates over the activation type, Dk, Dv and the rows per CTA;
// gdn_scan_tc_dk{16,32,64,128}.cu instantiate one key head dim each (parallel compilation).
//
// What is computed is the page's per-token recurrence (logicaffeine_compile::codegen_cuda::gdn,
// module description; time loop of torch_to_nnef.op.gated_delta, gated_delta_reference), not
// an approximation of it: blocks of B = 16 tokens are written out exactly.  The l2 norms are
// per-token scalars, k^_t = rk_t k_t and q^_t = rq_t q_t (rq_t carries 1/sqrt(Dk)), so the
// products below run on the raw k and q.  With S' the registers at the block start (true
// memory lam S') and x_t = S' k_t, y_t = S' q_t:
//     u_t = lam D_t rk_t x_t + sum_{s<t} d_s KK[s][t]          (u: the page's S k)
//     d_t = beta_t (v_t - alpha_t u_t)                           (d: the page's coef)
//     o_t = alpha_t (lam D_t rq_t y_t + sum_{s<t} d_s QX[s][t]) + d_t (k^_t . q^_t)
//     S'  <- S' + sum_s (W_s rk_s d_s / lam') k_s,   lam' = lam Gam
// D_t = prod_{r<t} alpha_r, W_s = prod_{r>s} alpha_r, Gam = prod over the block,
// KK[s][t] = prod_{s<r<t} alpha_r (k^_s . k^_t), QX[s][t] = prod_{s<r<t} alpha_r (k^_s . q^_t);
// every decay product is exp of a non-positive sum of log_decay.  This is the page's update
// expanded the way its "The fusion" section expands o (the update is affine in S).
//
// GB300 mapping:
//   * a warp owns 16 rows of a head's memory; the rows live in registers as the f32
//     accumulator fragments of m16n8k16 tensor-core MMAs (16 x D per warp: D/8 n-tiles);
//   * X = S' K^T and Y = S' Q^T for the block's 16 tokens are MMAs whose A operand is the
//     accumulator itself (an m16n8 accumulator pair has the m16k16 A-fragment layout), and the
//     rank-16 update S' += C K is an MMA accumulating into the same registers;
//   * accuracy: f32 operands are split into bf16 hi + lo parts and a product is formed as
//     hi.hi + hi.lo + lo.hi (relative error about 2^-16 per product, f32 accumulation).  bf16
//     inputs are exact bf16 operands, so their products take two MMAs (hi.k + lo.k) and the
//     raw rows are copied straight into the operand arrays; f16 inputs split exactly;
//   * the block's coefficients solve a unit-triangular system that is the same for every row:
//     with r_t = beta_t (v_t - alpha_t lam D_t rk_t x_t) and N[s][t] = beta_t alpha_t KK[s][t]
//     (s < t), the recurrence d_t + sum_{s<t} N[s][t] d_s = r_t gives d = r (I + N)^-1, and
//     O = lam alpha D rq Y + d QX' with QX'[s][t] = alpha_t QX[s][t] (s < t), QX'[t][t] =
//     k^_t . q^_t.  Per chunk, one small MMA per block forms KK and QX and one warp per block
//     inverts I + N; every warp then gets d and O of its 16 rows as two more MMAs whose A
//     operands are accumulator fragments (no per-row serial loop, no transposes);
//   * warp specialisation: 4 producer warps stage chunk c+1 (cp.async copies of q, k, v, z two
//     chunks ahead; the norms; decay products; KK, QX; the triangular inverse) and write y for
//     finished chunks, while the row warps run chunk c.  Hand-off through rings of shared
//     memory slots and named barriers (full / empty per chunk parity);
//   * the producers apply the gated RMSNorm: over the CTA when it owns a whole head; when a
//     head's rows are split over NRB CTAs, those CTAs form a thread-block cluster and each
//     token's partial sum of squares goes to the other CTAs through distributed shared memory
//     (st.async completing on their mbarriers) before every CTA normalises its own rows;
//   * a launch may cover segments of the sequence (the sequence-split scan): each CTA takes
//     its segment from the grid and reads the segment's tokens with the whole sequence's
//     strides.  A transition launch carries the identity (Dk rows) through the update with
//     v = 0, an offset launch starts from zeros; neither writes y, both write their end memory
//     to the split scan's workspace.  The plain scan is one segment.
#pragma once

#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_mma.cuh"
#include "gdn_tma.cuh"

namespace gdn {
namespace {

constexpr int kT = 32;                     // tokens per staged chunk
constexpr int kB = 16;                     // tokens per MMA block
static_assert(kT == 32 && kT % kB == 0, "one lane per chunk token in the decay prefix scan");
constexpr float kMinLogDecay = -80.0f;     // exp(-80) ~ 1.8e-35: a full reset for f32 purposes

template <typename TA> struct IsBf16 { static constexpr bool value = false; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

template <typename TA, int DK, int DV, int NW> struct TcCfg {
    static constexpr bool EXACT = IsBf16<TA>::value;  // raw rows are exact bf16 operands
    static constexpr int RB = 16 * NW;               // rows per CTA (NW row warps)
    static constexpr int NRB = DV / RB;              // CTAs per head
    static constexpr int NP = (NW == 8) ? 8 : 4;     // producer warps
    static constexpr int PT = 32 * NP;               // producer threads
    static constexpr int NT = 32 * (NW + NP);
    // 16 warps launch with 128 registers each; the row warps then take 168 from the producer
    // warps, which keep 88 (setmaxnreg; 8 x 168 + 8 x 88 = 16 x 128)
    static constexpr bool REG_SPLIT = (NT == 512);
    static constexpr int REG_ROW = 168, REG_PROD = 88;
    static_assert(!REG_SPLIT || (NW * REG_ROW + NP * REG_PROD == (NW + NP) * 128 &&
                                 NW % 4 == 0 && NP % 4 == 0),
                  "register split within the launch's registers, whole warpgroups");
    static constexpr bool SPLIT_KQ = (NP == 8);      // norm pass: k on 4 warps, q on the others
    // f32 rows of 256: the norm pass reads the raw k, q rows from global memory (no staging
    // slot; the two f32 rows and the hi / lo rings would not fit in shared memory together)
    static constexpr bool DIRECT_KQ = !EXACT && sizeof(TA) == 4 && DK > 128;
    // a warp's 16 x 256 memory block takes about 250 registers: no register split, whole
    // register file for at most 8 warps
    static_assert(DK <= 128 || NT <= 256, "Dk > 128 runs at most 4 row warps");
    static constexpr int NTILE = DK / 8;             // n-tiles of a warp's 16 x Dk memory block
    static constexpr int KST = DK / 16;              // k-steps over Dk
    static constexpr int NBLK = kT / kB;
    static constexpr int PADE = 16 / (int)sizeof(TA);  // 16 bytes of row padding, in elements
    static constexpr int LDV = RB + PADE;            // raw v / z rows
    static constexpr int LDO = RB + 4;               // o rows (f32)
    static constexpr int NOP = EXACT ? 3 : 2;        // operand ring depth
    static constexpr int NVZ = 3;                    // v / z ring depth
    static constexpr bool WHOLE_HEAD = (RB == DV);
    static constexpr int KPIECES = DK * (int)sizeof(TA) / 16;    // 16-byte pieces of a k row
    static constexpr int VPIECES = RB * (int)sizeof(TA) / 16;    // ... of this CTA's v rows
    static constexpr int TPK = KPIECES % 4 == 0 ? 4 : (KPIECES % 2 == 0 ? 2 : 1);  // norm-pass
                                                                  // threads per token
    static_assert(DV % RB == 0 && DK % 16 == 0 && DV % 16 == 0, "shape");
    static_assert(KPIECES >= 1 && VPIECES >= 1, "16-byte copy granularity");
    static_assert(KPIECES % TPK == 0 && (SPLIT_KQ ? PT / 2 : PT) / TPK >= kT,
                  "norm pass covers a chunk at once");
};

// k and q operands, rows padded by 16 bytes (conflict-free ldmatrix and 16-byte accesses).
// bf16: the raw rows, copied in place into a ring of three slots.  Other types: a staging
// slot for the raw rows and a ring of two slots of bf16 hi / lo parts.
// f32 rows of 256 have no staging slot (read from global memory by the norm pass).
template <typename TA, int D, bool EXACT, bool DIRECT> struct TcOps;
template <typename TA, int D> struct TcOps<TA, D, true, false> {
    __nv_bfloat16 k[3][kT][D + 8], q[3][kT][D + 8];
};
template <typename TA, int D> struct TcOps<TA, D, false, false> {
    TA kraw[kT][D + 16 / sizeof(TA)], qraw[kT][D + 16 / sizeof(TA)];
    __nv_bfloat16 khi[2][kT][D + 8], klo[2][kT][D + 8];
    __nv_bfloat16 qhi[2][kT][D + 8], qlo[2][kT][D + 8];
};
template <typename TA, int D> struct TcOps<TA, D, false, true> {
    __nv_bfloat16 khi[2][kT][D + 8], klo[2][kT][D + 8];
    __nv_bfloat16 qhi[2][kT][D + 8], qlo[2][kT][D + 8];
};

// Shared memory; every member 16-byte aligned (vector accesses, ldmatrix rows, cp.async).
// Slots are indexed by chunk: operands c % NOP, v / z c % 3, and everything else the row warps
// read (o, per-token scalars, tables) c % 2.
template <typename TA, int DK, int DV, int NW> struct TcSmem {
    using C = TcCfg<TA, DK, DV, NW>;
    alignas(16) TcOps<TA, DK, C::EXACT, C::DIRECT_KQ> op;
    alignas(16) TA vr[C::NVZ][kT][C::LDV];       // raw v rows of this CTA
    alignas(16) TA zr[C::NVZ][kT][C::LDV];       // raw z (whole-head CTAs with z)
    alignas(16) float ob[2][kT][C::LDO];         // o of the chunk, written by the row warps
    alignas(16) float4 cst[2][kT];               // row-warp scalars: beta, alpha D rk, alpha D rq, W rk
    alignas(16) float4 gts[kT];                  // producer: alpha, beta, alpha D, W of the staged chunk
    alignas(16) float2 nrm[kT];                  // rk, rq from the norm pass
    alignas(16) float cum[kT];                   // block-inclusive sums of the clamped log_decay
    alignas(16) float gamp[C::NBLK];             // producer: Gam of each block of the staged chunk
    alignas(16) float gam[2][C::NBLK];           // Gam of each block
    alignas(16) float nm[C::NBLK][kB][kB];       // N[s][t] = beta_t alpha_t KK[s][t] for s < t, else 0
    // B operands [s][t] (k = s, n = t), bf16 hi/lo, rows padded to 24 (conflict-free ldmatrix):
    alignas(16) __nv_bfloat16 thi[2][C::NBLK][kB][kB + 8], tlo[2][C::NBLK][kB][kB + 8];   // (I + N)^-1
    alignas(16) __nv_bfloat16 phi[2][C::NBLK][kB][kB + 8], plo[2][C::NBLK][kB][kB + 8];   // QX'
    // heads split over a cluster of NRB CTAs: the other CTAs' partial sums of squares of each
    // token's gated output, per chunk parity and sender, and their arrival
    alignas(16) float peer_ss[2][C::NRB][kT];
    alignas(8) uint64_t peer_bar[2];
};

// Named barriers (0 is __syncthreads): chunk parity b full / empty, and producers only.
enum { kBarFull0 = 1, kBarEmpty0 = 3, kBarProd = 5 };


template <typename TA, int DK, int DV, int NW>
__global__ void __launch_bounds__(TcCfg<TA, DK, DV, NW>::NT, 1)
gdn_scan_tc_kernel(const gdn_params p, const ScanSplit sp) {
    using C = TcCfg<TA, DK, DV, NW>;
    using A = Act<TA>;
    using Sm = TcSmem<TA, DK, DV, NW>;
    constexpr int RB = C::RB, NTILE = C::NTILE, KST = C::KST, NP = C::NP, NT = C::NT, PT = C::PT;
    constexpr bool EXACT = C::EXACT;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);

    // segment seg of the sequence (one segment for the plain scan), then head and row block
    const int64_t per_seg = static_cast<int64_t>(p.B) * p.Hv * C::NRB;
    const int gseg = static_cast<int>(blockIdx.x / per_seg);   // segment slot in the grid
    const int64_t local = blockIdx.x - gseg * per_seg;
    // mode 3 runs transitions (first half of the grid) beside offsets (second half)
    const int half = sp.nseg / 2;
    const int mode = sp.mode != 3 ? sp.mode : (gseg < half ? 1 : 2);
    const int seg = (sp.mode == 3 && gseg >= half) ? gseg - half : gseg;
    const int64_t head = local / C::NRB;                   // b * Hv + hv
    const int rblk = static_cast<int>(local % C::NRB);
    const int b = static_cast<int>(head / p.Hv);
    const int hv = static_cast<int>(head - static_cast<int64_t>(b) * p.Hv);
    const int hk = hv / (p.Hv / p.Hk);
    const int r0 = rblk * RB;                              // first memory row of this CTA
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;                // MMA fragment coordinates
    const int S_full = p.S;                                // strides follow the whole sequence
    const int t_begin = seg * sp.seg_len;                  // this segment's first token
    const int S = min(sp.seg_len, S_full - t_begin);       // and its length (>= 1)
    const int nchunks = (S + kT - 1) / kT;
    const bool v_zero = mode == 1;                         // transition: v = 0, start = identity

    int64_t k_base, k_ts, v_base, v_ts, g_base, g_ts;
    if (p.head_major) {
        k_base = (static_cast<int64_t>(b) * p.Hk + hk) * S_full * DK;  k_ts = DK;
        v_base = head * S_full * DV;                                   v_ts = DV;
        g_base = head * S_full;                                       g_ts = 1;
    } else {
        k_base = (static_cast<int64_t>(b) * S_full * p.Hk + hk) * DK;  k_ts = static_cast<int64_t>(p.Hk) * DK;
        v_base = (static_cast<int64_t>(b) * S_full * p.Hv + hv) * DV;  v_ts = static_cast<int64_t>(p.Hv) * DV;
        g_base = static_cast<int64_t>(b) * S_full * p.Hv + hv;        g_ts = p.Hv;
    }
    k_base += t_begin * k_ts;
    v_base += t_begin * v_ts;
    g_base += t_begin * g_ts;
    // offset of this (segment, head) in the per-segment memories of a split scan
    auto seg_head = [&]() {
        return (static_cast<int64_t>(seg) * p.B * p.Hv + head) * (DV * DK);
    };
    // gated RMSNorm in this kernel: over the CTA when it owns the whole head, else over the
    // cluster of the head's NRB CTAs (partial sums exchanged through distributed shared memory)
    const bool fused_norm = p.z != nullptr;
    if (!C::WHOLE_HEAD && fused_norm) {
        if (threadIdx.x == 0) {
            mbar_init(&sm.peer_bar[0], 1);
            mbar_init(&sm.peer_bar[1], 1);
            mbar_init_fence();
        }
        cluster_sync_all();                                // every CTA's barriers initialised
    }
    if constexpr (C::REG_SPLIT) {
        if (warp < NW) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(C::REG_ROW));
        else asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(C::REG_PROD));
    }

    if (warp < NW) {
        // ============================ row warps: the recurrence =============================
        const int wrow = warp * 16;                        // first local row of this warp
        const int m = lane >> 3, r = lane & 7;             // ldmatrix address roles
        // the warp's 16 x D block of the memory as accumulator fragments:
        // sacc[j] = S[wrow+g][8j+2tq], S[wrow+g][8j+2tq+1], S[wrow+g+8][8j+2tq], S[..+8][..+1]
        float sacc[NTILE][4];
        {
            // start memory: the caller's s0 (plain scan), the segment's start, zeros or the
            // identity (transition)
            const float *s0_src = mode != 0 ? nullptr
                                  : sp.s0_seg ? sp.s0_seg + seg_head()
                                  : p.s0 ? p.s0 + head * (DV * DK) : nullptr;
            const float *s0 = s0_src ? s0_src + static_cast<int64_t>(r0 + wrow) * DK : nullptr;
#pragma unroll
            for (int j = 0; j < NTILE; j++) {
                float2 lo = make_float2(0.f, 0.f), hi = lo;
                if (s0) {
                    lo = *reinterpret_cast<const float2 *>(s0 + g * DK + 8 * j + 2 * tq);
                    hi = *reinterpret_cast<const float2 *>(s0 + (g + 8) * DK + 8 * j + 2 * tq);
                } else if (v_zero) {                       // the identity (rows = key dims)
                    const int row = r0 + wrow + g, col = 8 * j + 2 * tq;
                    lo = make_float2(row == col ? 1.f : 0.f, row == col + 1 ? 1.f : 0.f);
                    hi = make_float2(row + 8 == col ? 1.f : 0.f, row + 8 == col + 1 ? 1.f : 0.f);
                }
                sacc[j][0] = lo.x; sacc[j][1] = lo.y; sacc[j][2] = hi.x; sacc[j][3] = hi.y;
            }
        }
        float lam = 1.0f;                                  // true memory = lam * registers
        for (int ch = 0; ch < nchunks; ch++) {
            const int hb = ch & 1, os = ch % C::NOP, vs = ch % C::NVZ;
            const int nt = min(kT, S - ch * kT);
            bar_sync(kBarFull0 + hb, NT);                  // chunk ch staged
            for (int blk = 0; blk * kB < nt; blk++) {
                const int tb = blk * kB;
                const int nb = min(kB, nt - tb);

                // X = S' K^T, Y = S' Q^T for the block's 16 tokens (two n8 tiles each)
                float xa[2][4] = {}, ya[2][4] = {};
#pragma unroll
                for (int kk = 0; kk < KST; kk++) {
                    uint32_t ah[4], al[4];
                    split2(sacc[2 * kk][0], sacc[2 * kk][1], ah[0], al[0]);
                    split2(sacc[2 * kk][2], sacc[2 * kk][3], ah[1], al[1]);
                    split2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1], ah[2], al[2]);
                    split2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3], ah[3], al[3]);
                    if constexpr (EXACT) {
                        // matrices: (tokens 0-7 | 8-15) x (k 0-7 | 8-15): both n8 tiles at once
                        const int trow = tb + 8 * (m >> 1) + r, col = 16 * kk + 8 * (m & 1);
                        uint32_t kb[4], qb[4];
                        ldsm_x4(kb, &sm.op.k[os][trow][col]);
                        ldsm_x4(qb, &sm.op.q[os][trow][col]);
                        mma2(xa[0], ah, al, kb[0], kb[1]);
                        mma2(xa[1], ah, al, kb[2], kb[3]);
                        mma2(ya[0], ah, al, qb[0], qb[1]);
                        mma2(ya[1], ah, al, qb[2], qb[3]);
                    } else {
#pragma unroll
                        for (int nt8 = 0; nt8 < 2; nt8++) {
                            const int trow = tb + 8 * nt8 + r, col = 16 * kk + 8 * (m & 1);
                            uint32_t kb[4], qb[4];
                            ldsm_x4(kb, (m & 2) ? &sm.op.klo[os][trow][col] : &sm.op.khi[os][trow][col]);
                            ldsm_x4(qb, (m & 2) ? &sm.op.qlo[os][trow][col] : &sm.op.qhi[os][trow][col]);
                            mma3(xa[nt8], ah, al, kb[0], kb[1], kb[2], kb[3]);
                            mma3(ya[nt8], ah, al, qb[0], qb[1], qb[2], qb[3]);
                        }
                    }
                }
                // r = beta (v - lam alpha D rk x) and lam alpha D rq y at this lane's positions;
                // exact zeros past the sequence end (those columns meet every other token's
                // terms in the d, O and update MMAs)
                float ra[2][4], oa[2][4];
#pragma unroll
                for (int nt8 = 0; nt8 < 2; nt8++)
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int rr = g + ((e & 2) ? 8 : 0);
                        const int t = 8 * nt8 + 2 * tq + (e & 1);
                        const float4 cs = sm.cst[hb][tb + t];
                        const float vv = v_zero ? 0.f : A::one(&sm.vr[vs][tb + t][wrow + rr]);
                        ra[nt8][e] = (t < nb) ? cs.x * (vv - lam * cs.y * xa[nt8][e]) : 0.f;
                        oa[nt8][e] = lam * cs.z * ya[nt8][e];
                    }
                // d = r T  (A = r, rows x tokens s; B = T[s][t])
                float da[2][4] = {};
                {
                    uint32_t rh[4], rl[4];
                    split2(ra[0][0], ra[0][1], rh[0], rl[0]);
                    split2(ra[0][2], ra[0][3], rh[1], rl[1]);
                    split2(ra[1][0], ra[1][1], rh[2], rl[2]);
                    split2(ra[1][2], ra[1][3], rh[3], rl[3]);
#pragma unroll
                    for (int nt8 = 0; nt8 < 2; nt8++) {
                        uint32_t tbf[4];
                        const int srow = r + ((m & 1) ? 8 : 0);
                        ldsm_x4_t(tbf, (m & 2) ? &sm.tlo[hb][blk][srow][8 * nt8] : &sm.thi[hb][blk][srow][8 * nt8]);
                        mma3(da[nt8], rh, rl, tbf[0], tbf[1], tbf[2], tbf[3]);
                    }
                }
                // O = lam alpha D rq Y + d QX'
                uint32_t dh[4], dl[4];
                split2(da[0][0], da[0][1], dh[0], dl[0]);
                split2(da[0][2], da[0][3], dh[1], dl[1]);
                split2(da[1][0], da[1][1], dh[2], dl[2]);
                split2(da[1][2], da[1][3], dh[3], dl[3]);
#pragma unroll
                for (int nt8 = 0; nt8 < 2; nt8++) {
                    uint32_t pbf[4];
                    const int srow = r + ((m & 1) ? 8 : 0);
                    ldsm_x4_t(pbf, (m & 2) ? &sm.plo[hb][blk][srow][8 * nt8] : &sm.phi[hb][blk][srow][8 * nt8]);
                    mma3(oa[nt8], dh, dl, pbf[0], pbf[1], pbf[2], pbf[3]);
                }
#pragma unroll
                for (int nt8 = 0; nt8 < 2; nt8++) {
                    const int t = 8 * nt8 + 2 * tq;
                    if (t < nb) {
                        sm.ob[hb][tb + t][wrow + g] = oa[nt8][0];
                        sm.ob[hb][tb + t][wrow + g + 8] = oa[nt8][2];
                    }
                    if (t + 1 < nb) {
                        sm.ob[hb][tb + t + 1][wrow + g] = oa[nt8][1];
                        sm.ob[hb][tb + t + 1][wrow + g + 8] = oa[nt8][3];
                    }
                }
                // the rank-16 update: C = d W rk / lam' (A fragment), S' += C K
                const float lam_new = lam * sm.gam[hb][blk];
                const bool fold = !(lam_new >= 0x1p-40f);  // uniform over the row warps
                const float scale = fold ? 1.0f : 1.0f / lam_new;
                float cf[2][4];
#pragma unroll
                for (int nt8 = 0; nt8 < 2; nt8++)
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int t = 8 * nt8 + 2 * tq + (e & 1);
                        cf[nt8][e] = da[nt8][e] * sm.cst[hb][tb + t].w * scale;
                    }
                uint32_t ch_[4], cl_[4];
                split2(cf[0][0], cf[0][1], ch_[0], cl_[0]);
                split2(cf[0][2], cf[0][3], ch_[1], cl_[1]);
                split2(cf[1][0], cf[1][1], ch_[2], cl_[2]);
                split2(cf[1][2], cf[1][3], ch_[3], cl_[3]);
                if (fold) {
#pragma unroll
                    for (int j = 0; j < NTILE; j++)
#pragma unroll
                        for (int e = 0; e < 4; e++) sacc[j][e] *= lam_new;
                }
                // S' += C K : B = K[tokens][cols 8j..8j+7], k = token (transposed ldmatrix)
                if constexpr (EXACT) {
#pragma unroll
                    for (int j = 0; j < NTILE; j += 2) {
                        uint32_t kb[4];
                        const int trow = tb + r + ((m & 1) ? 8 : 0);
                        ldsm_x4_t(kb, &sm.op.k[os][trow][8 * (j + (m >> 1))]);
                        mma2(sacc[j], ch_, cl_, kb[0], kb[1]);
                        mma2(sacc[j + 1], ch_, cl_, kb[2], kb[3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < NTILE; j++) {
                        uint32_t kb[4];
                        const int trow = tb + r + ((m & 1) ? 8 : 0);
                        ldsm_x4_t(kb, (m & 2) ? &sm.op.klo[os][trow][8 * j] : &sm.op.khi[os][trow][8 * j]);
                        mma3(sacc[j], ch_, cl_, kb[0], kb[1], kb[2], kb[3]);
                    }
                }
                lam = fold ? 1.0f : lam_new;
            }
            bar_arrive(kBarEmpty0 + hb, NT);               // slots of chunk ch handed back
        }
        // final memory rows (undo the deferred decay): the caller's state for the plain scan
        // and the last segment, the per-segment end memory for transitions and offsets
        if (mode == 0 && seg != sp.nseg - 1) return;       // a segment before the last
        float *state_dst = mode == 0 ? p.state + head * (DV * DK)
                         : (mode == 2 && sp.mode == 3 ? sp.state_seg2 : sp.state_seg) + seg_head();
        float *so = state_dst + static_cast<int64_t>(r0 + wrow) * DK;
#pragma unroll
        for (int j = 0; j < NTILE; j++) {
            *reinterpret_cast<float2 *>(so + g * DK + 8 * j + 2 * tq) =
                make_float2(lam * sacc[j][0], lam * sacc[j][1]);
            *reinterpret_cast<float2 *>(so + (g + 8) * DK + 8 * j + 2 * tq) =
                make_float2(lam * sacc[j][2], lam * sacc[j][3]);
        }
        return;
    }

    // ============================== producer warps: staging ===============================
    const int pw = warp - NW;                              // 0 .. NP-1
    const int ptid = threadIdx.x - 32 * NW;                // 0 .. PT-1
    const TA *kg = static_cast<const TA *>(p.k) + k_base;
    const TA *qg = static_cast<const TA *>(p.q) + k_base;
    const TA *vg = static_cast<const TA *>(p.v) + v_base + r0;
    const TA *zg = fused_norm ? static_cast<const TA *>(p.z) + v_base + r0 : nullptr;

    // copies of chunk c: raw k, q rows (into the operand ring for bf16, else the staging slot)
    auto issue_kq = [&](int c) {
        if constexpr (C::DIRECT_KQ) return;
        const int t0 = c * kT, nt = min(kT, S - t0);
        for (int i = ptid; i < nt * C::KPIECES; i += PT) {
            const int tt = i / C::KPIECES, pc = i % C::KPIECES;
            const int64_t off = (t0 + tt) * k_ts;
            char *dk = nullptr, *dq = nullptr;             // set below (the DIRECT_KQ branch returns)
            if constexpr (EXACT) {
                dk = reinterpret_cast<char *>(&sm.op.k[c % 3][tt][0]);
                dq = reinterpret_cast<char *>(&sm.op.q[c % 3][tt][0]);
            } else if constexpr (C::DIRECT_KQ) {
                return;
            } else {
                dk = reinterpret_cast<char *>(&sm.op.kraw[tt][0]);
                dq = reinterpret_cast<char *>(&sm.op.qraw[tt][0]);
            }
            cp_async16(dk + 16 * pc, reinterpret_cast<const char *>(kg + off) + 16 * pc);
            cp_async16(dq + 16 * pc, reinterpret_cast<const char *>(qg + off) + 16 * pc);
        }
    };
    auto issue_vz = [&](int c) {
        if (v_zero && !fused_norm) return;                 // a transition reads neither v nor z
        const int t0 = c * kT, nt = min(kT, S - t0);
        const int vs = c % C::NVZ;
        for (int i = ptid; i < nt * C::VPIECES; i += PT) {
            const int tt = i / C::VPIECES, pc = i % C::VPIECES;
            const int64_t off = (t0 + tt) * v_ts;
            cp_async16(reinterpret_cast<char *>(&sm.vr[vs][tt][0]) + 16 * pc,
                       reinterpret_cast<const char *>(vg + off) + 16 * pc);
            if (fused_norm)
                cp_async16(reinterpret_cast<char *>(&sm.zr[vs][tt][0]) + 16 * pc,
                           reinterpret_cast<const char *>(zg + off) + 16 * pc);
        }
    };

    // y of a finished chunk: gated RMSNorm, TPT threads per token, each with FPT float4 column
    // groups of this CTA's RB columns interleaved (a quarter-warp reads 128 contiguous bytes);
    // a split head first sends each token's partial sum of squares to the other CTAs of its
    // cluster and waits for theirs.  Without z: this CTA's raw o rows.
    constexpr int TPT = (RB / 4) % 8 == 0 ? 8 : 4;         // threads per token (norm); RB / 4
                                                           // is a multiple of 4
    constexpr int FPT = RB / (4 * TPT);                    // float4 groups per thread
    constexpr int NIT = kT * TPT / PT;                     // token passes
    static_assert(PT % TPT == 0 && (kT * TPT) % PT == 0, "norm thread groups");
    float4 gn4[FPT];
#pragma unroll
    for (int f = 0; f < FPT; f++)
        gn4[f] = fused_norm ? *reinterpret_cast<const float4 *>(p.gn + r0 + 4 * (ptid % TPT + TPT * f))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    const float inv_d = 1.0f / static_cast<float>(DV);
    bool gave_up = false;                                  // a cluster wait ran out twice
    auto emit = [&](int c) {
        if (p.y == nullptr) return;                        // transitions and offsets: no y
        const int hb = c & 1, vs = c % C::NVZ;
        const int t0 = c * kT, nt = min(kT, S - t0);
        if (fused_norm) {
            float4 x[NIT][FPT];
            float ss[NIT];
            if (!C::WHOLE_HEAD && ptid == 0)               // this chunk's partner bytes
                mbar_arrive_expect_tx(&sm.peer_bar[hb], (C::NRB - 1) * kT * 4);
#pragma unroll
            for (int it = 0; it < NIT; it++) {
                const int tt = ptid / TPT + it * (PT / TPT);
                ss[it] = 0.f;
#pragma unroll
                for (int f = 0; f < FPT; f++) {
                    const int col = 4 * (ptid % TPT + TPT * f);
                    const float4 o4 = *reinterpret_cast<const float4 *>(&sm.ob[hb][tt][col]);
                    const float4 z4 = A::four(&sm.zr[vs][tt][col]);
                    x[it][f] = make_float4(o4.x * silu_fast(z4.x), o4.y * silu_fast(z4.y),
                                           o4.z * silu_fast(z4.z), o4.w * silu_fast(z4.w));
                    ss[it] = fmaf(x[it][f].x, x[it][f].x, fmaf(x[it][f].y, x[it][f].y,
                             fmaf(x[it][f].z, x[it][f].z, fmaf(x[it][f].w, x[it][f].w, ss[it]))));
                }
                ss[it] = group_sum<TPT>(ss[it]);
                if (!C::WHOLE_HEAD && ptid % TPT == 0) {   // every token, also past the end
#pragma unroll
                    for (int pr = 0; pr < C::NRB; pr++)
                        if (pr != rblk) st_async_peer(&sm.peer_ss[hb][rblk][tt], ss[it], &sm.peer_bar[hb], pr);
                }
            }
            // a wait that runs out sets the watchdog word and is tried once more; if that runs
            // out too, this thread stops waiting and stops storing y (the call is then reported
            // as timed out by gdn_device_status)
            if (!C::WHOLE_HEAD && !gave_up &&
                !mbar_wait_bounded(&sm.peer_bar[hb], static_cast<unsigned>((c >> 1) & 1)) &&
                !mbar_wait_bounded(&sm.peer_bar[hb], static_cast<unsigned>((c >> 1) & 1)))
                gave_up = true;
#pragma unroll
            for (int it = 0; it < NIT; it++) {
                const int tt = ptid / TPT + it * (PT / TPT);
                float tot = ss[it];
                if (!C::WHOLE_HEAD) {
#pragma unroll
                    for (int pr = 0; pr < C::NRB; pr++)
                        if (pr != rblk) tot += sm.peer_ss[hb][pr][tt];
                }
                const float rr = rsqrtf(fmaf(tot, inv_d, p.norm_eps));
                if (tt < nt && !gave_up) {
                    float *yr = p.y + v_base + r0 + (t0 + tt) * v_ts;
#pragma unroll
                    for (int f = 0; f < FPT; f++) {
                        const int col = 4 * (ptid % TPT + TPT * f);
                        *reinterpret_cast<float4 *>(yr + col) =
                            make_float4(x[it][f].x * rr * gn4[f].x, x[it][f].y * rr * gn4[f].y,
                                        x[it][f].z * rr * gn4[f].z, x[it][f].w * rr * gn4[f].w);
                    }
                }
            }
        } else {
            constexpr int TPR = RB / 4;                    // threads per token row
            for (int i = ptid; i < nt * TPR; i += PT) {
                const int tt = i / TPR, col = 4 * (i % TPR);
                *reinterpret_cast<float4 *>(p.y + v_base + r0 + (t0 + tt) * v_ts + col) =
                    *reinterpret_cast<const float4 *>(&sm.ob[hb][tt][col]);
            }
        }
    };

    // The gate warp computes a chunk's decay products one chunk ahead, beside the triangular
    // inverse of the previous chunk (kT == 32: one lane per token); its lanes hold the gates
    // of the chunk after that, in flight.
    constexpr int GATE_WARP = NP - 1;
    static_assert(GATE_WARP >= 1, "the gate warp is not the inverse warp");
    float gl = 0.f, gb = 0.f;
    auto load_gates = [&](int c) {
        const int t = c * kT + lane;
        if (t < S) {
            const int64_t gi = g_base + static_cast<int64_t>(t) * g_ts;
            gl = load_gate(p.log_decay, p.gate_dtype, gi);
            gb = load_gate(p.beta, p.gate_dtype, gi);
        }
    };
    auto decay_products = [&](int c) {                     // gates in gl, gb -> gts, cum, gamp
        const bool valid = c * kT + lane < S;
        const float gc = valid ? fmaxf(gl, kMinLogDecay) : 0.f;
        float upto = gc;                                   // block-inclusive prefix sum
#pragma unroll
        for (int off = 1; off < kB; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, upto, off, kB);
            if ((lane & (kB - 1)) >= off) upto += o;
        }
        const float total = __shfl_sync(0xffffffffu, upto, kB - 1, kB);
        sm.gts[lane] = make_float4(expf(gc), valid ? gb : 0.f, expf(upto), expf(total - upto));
        sm.cum[lane] = upto;
        if ((lane & (kB - 1)) == kB - 1) sm.gamp[lane / kB] = expf(total);
    };
    if (pw == GATE_WARP) {
        load_gates(0);
        decay_products(0);
        if (kT < S) load_gates(1);
    }
    issue_vz(0);
    issue_kq(0);
    cp_async_commit();
    const float inv_sqrt_dk = rsqrtf(static_cast<float>(DK));
    // norm-pass roles: token nt_tok, pieces nq, nq + TPK, ...; a quarter-warp of 8 lanes
    // covers 8 tokens (conflict-free 16-byte accesses on the padded rows)
    constexpr int TPW = 32 / C::TPK;                       // tokens per warp in the norm pass
    const bool do_k = !C::SPLIT_KQ || pw < NP / 2;         // this warp's rows: k, q or both
    const bool do_q = !C::SPLIT_KQ || pw >= NP / 2;
    const int n_tok = (C::SPLIT_KQ ? pw % (NP / 2) : pw) * TPW + lane % TPW;
    const int nq = lane / TPW;

    for (int ch = 0; ch < nchunks; ch++) {
        const int hb = ch & 1, os = ch % C::NOP;
        const int t0 = ch * kT;
        const int nt = min(kT, S - t0);
        if (ch >= 2) {                                     // chunk ch-2 is done with parity hb
            bar_sync(kBarEmpty0 + hb, NT);
            emit(ch - 2);
            bar_sync(kBarProd, PT);                        // its z slot is read: refill it
        }
        if (ch + 1 < nchunks) {
            issue_vz(ch + 1);
            if constexpr (EXACT) issue_kq(ch + 1);
        }
        cp_async_commit();
        cp_async_wait<1>();                                // all but chunk ch+1's copies
        bar_sync(kBarProd, PT);

        // ---- norm pass: rk, rq per token; bf16 hi / lo operands for other input types; zero
        //      operand rows past the sequence end
        if (n_tok < kT) {
            float ssk = 0.f, ssq = 0.f;
            const bool valid = n_tok < nt;
#pragma unroll
            for (int i = 0; i < C::KPIECES / C::TPK; i++) {
                const int pc = nq + C::TPK * i;
                if constexpr (EXACT) {
                    uint4 *dk = reinterpret_cast<uint4 *>(&sm.op.k[os][n_tok][8 * pc]);
                    uint4 *dq = reinterpret_cast<uint4 *>(&sm.op.q[os][n_tok][8 * pc]);
                    if (valid) {
                        if (do_k) Piece<TA>::sq(&sm.op.k[os][n_tok][8 * pc], ssk);
                        if (do_q) Piece<TA>::sq(&sm.op.q[os][n_tok][8 * pc], ssq);
                    } else {
                        if (do_k) *dk = make_uint4(0u, 0u, 0u, 0u);
                        if (do_q) *dq = make_uint4(0u, 0u, 0u, 0u);
                    }
                } else {
                    constexpr int E = Piece<TA>::E;
                    if (valid) {
                        const TA *ksrc, *qsrc;
                        if constexpr (C::DIRECT_KQ) {
                            const int64_t off = static_cast<int64_t>(t0 + n_tok) * k_ts + E * pc;
                            ksrc = kg + off;
                            qsrc = qg + off;
                        } else {
                            ksrc = &sm.op.kraw[n_tok][E * pc];
                            qsrc = &sm.op.qraw[n_tok][E * pc];
                        }
                        if (do_k)
                            Piece<TA>::split(ksrc, &sm.op.khi[os][n_tok][E * pc],
                                             &sm.op.klo[os][n_tok][E * pc], ssk);
                        if (do_q)
                            Piece<TA>::split(qsrc, &sm.op.qhi[os][n_tok][E * pc],
                                             &sm.op.qlo[os][n_tok][E * pc], ssq);
                    } else {
#pragma unroll
                        for (int e = 0; e < E; e++) {
                            if (do_k) {
                                sm.op.khi[os][n_tok][E * pc + e] = __float2bfloat16_rn(0.f);
                                sm.op.klo[os][n_tok][E * pc + e] = __float2bfloat16_rn(0.f);
                            }
                            if (do_q) {
                                sm.op.qhi[os][n_tok][E * pc + e] = __float2bfloat16_rn(0.f);
                                sm.op.qlo[os][n_tok][E * pc + e] = __float2bfloat16_rn(0.f);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int off = TPW; off < 32; off <<= 1) {
                ssk += __shfl_xor_sync(0xffffffffu, ssk, off);
                ssq += __shfl_xor_sync(0xffffffffu, ssq, off);
            }
            if (nq == 0) {
                if (do_k) sm.nrm[n_tok].x = valid ? rsqrtf(ssk + p.qk_eps) : 0.f;
                if (do_q) sm.nrm[n_tok].y = valid ? rsqrtf(ssq + p.qk_eps) * inv_sqrt_dk : 0.f;
            }
        }
        bar_sync(kBarProd, PT);                            // staging consumed, norms written
        if constexpr (!EXACT) {
            if (ch + 1 < nchunks) issue_kq(ch + 1);        // overlaps the rest of this chunk
            cp_async_commit();
        }

        // ---- KK and QX of each block by MMA; N and QX'.  The 4 NBLK n8 tiles, ordered
        //      (block, table, tokens t 0-7 | 8-15), go NT8W to a producer warp.
        {
            constexpr int NT8W = 4 * C::NBLK / NP;
            static_assert(NT8W * NP == 4 * C::NBLK, "table tiles per producer warp");
            const int tile0 = pw * NT8W;
            const int blk = tile0 >> 2, nt0 = tile0 & 1;
            const bool isq = (tile0 >> 1) & 1;
            const int tb = blk * kB;
            const int m = lane >> 3, r = lane & 7;
            if (pw == 0) {                                 // the row warps' per-token scalars
                const float4 gt = sm.gts[lane];
                const float2 nr = sm.nrm[lane];
                sm.cst[hb][lane] = make_float4(gt.y, gt.z * nr.x, gt.z * nr.y, gt.w * nr.x);
                if (lane < C::NBLK) sm.gam[hb][lane] = sm.gamp[lane];
            }
            float acc[NT8W][4] = {};
#pragma unroll
            for (int kk = 0; kk < KST; kk++) {
                const int arow = tb + r + ((m & 1) ? 8 : 0), acol = 16 * kk + ((m & 2) ? 8 : 0);
                if constexpr (EXACT) {
                    uint32_t a[4];
                    ldsm_x4(a, &sm.op.k[os][arow][acol]);
#pragma unroll
                    for (int j = 0; j < NT8W; j++) {
                        // matrices (k 0-7 | 8-15) of tokens tb + 8 (nt0 + j) ..; lanes 16-31 mirror
                        const int trow = tb + 8 * (nt0 + j) + r, col = 16 * kk + 8 * (m & 1);
                        uint32_t bb[2];
                        ldsm_x2(bb, isq ? &sm.op.q[os][trow][col] : &sm.op.k[os][trow][col]);
                        mma16816(acc[j], a, bb[0], bb[1]);
                    }
                } else {
                    uint32_t ah[4], al[4];
                    ldsm_x4(ah, &sm.op.khi[os][arow][acol]);
                    ldsm_x4(al, &sm.op.klo[os][arow][acol]);
#pragma unroll
                    for (int j = 0; j < NT8W; j++) {
                        const int trow = tb + 8 * (nt0 + j) + r, col = 16 * kk + 8 * (m & 1);
                        uint32_t bb[4];
                        const __nv_bfloat16 *src =
                            (m & 2) ? (isq ? &sm.op.qlo[os][trow][col] : &sm.op.klo[os][trow][col])
                                    : (isq ? &sm.op.qhi[os][trow][col] : &sm.op.khi[os][trow][col]);
                        ldsm_x4(bb, src);
                        mma3(acc[j], ah, al, bb[0], bb[1], bb[2], bb[3]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < NT8W; j++)
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int s2 = g + ((e & 2) ? 8 : 0);
                    const int t = 8 * (nt0 + j) + 2 * tq + (e & 1);
                    const float4 gt = sm.gts[tb + t];      // alpha, beta of token t
                    const float2 nt_ = sm.nrm[tb + t];     // rk, rq of token t
                    const float dot = acc[j][e] * sm.nrm[tb + s2].x;   // rk_s (k_s . x_t)
                    // prod_{s<r<t} alpha_r: exp of a non-positive sum (fast exp: a few ulp,
                    // about 1e-5 relative at the largest arguments that do not underflow).
                    // Evaluated for every (s, t) and then masked, so no lane branches around
                    // the exponential; the clamps keep the unused ones finite and in range.
                    const float ex = __expf(fminf(sm.cum[tb + max(t - 1, 0)] - sm.cum[tb + s2], 0.f));
                    const float wgt = (s2 < t) ? ex : 0.f;
                    if (isq) {
                        const float val = (s2 < t) ? gt.x * wgt * nt_.y * dot : (s2 == t ? nt_.y * dot : 0.f);
                        split1(val, sm.phi[hb][blk][s2][t], sm.plo[hb][blk][s2][t]);
                    } else {
                        sm.nm[blk][s2][t] = (s2 < t) ? gt.y * gt.x * wgt * nt_.x * dot : 0.f;
                    }
                }
        }
        bar_sync(kBarProd, PT);
        // T = (I + N)^-1 (unit upper triangular): lane s of block blk (producer warp 0, lanes
        // 16 blk + s) builds row s by forward accumulation, T[s][t] = -sum_{s<=r<t} T[s][r] N[r][t].
        // Meanwhile the gate warp prepares the next chunk's decay products.
        static_assert(C::NBLK * kB == 32, "one lane per row of the blocks' inverses");
        if (pw == 0) {
            const int blk = lane / kB, srow = lane % kB;
            float tr[kB], acc[kB];
#pragma unroll
            for (int t = 0; t < kB; t++) { tr[t] = (t == srow) ? 1.f : 0.f; acc[t] = 0.f; }
#pragma unroll
            for (int r = 0; r < kB - 1; r++) {
                if (r > srow) tr[r] = -acc[r];
                float nr[kB];
#pragma unroll
                for (int t4 = 0; t4 < kB / 4; t4++)
                    *reinterpret_cast<float4 *>(&nr[4 * t4]) = *reinterpret_cast<const float4 *>(&sm.nm[blk][r][4 * t4]);
#pragma unroll
                for (int t = r + 1; t < kB; t++) acc[t] = fmaf(tr[r], nr[t], acc[t]);
            }
            if (kB - 1 > srow) tr[kB - 1] = -acc[kB - 1];
#pragma unroll
            for (int t = 0; t < kB; t++) split1(tr[t], sm.thi[hb][blk][srow][t], sm.tlo[hb][blk][srow][t]);
        } else if (pw == GATE_WARP && ch + 1 < nchunks) {
            decay_products(ch + 1);                        // tables of chunk ch are done with them
            if (ch + 2 < nchunks) load_gates(ch + 2);
        }
        bar_arrive(kBarFull0 + hb, NT);                    // chunk ch ready for the row warps
    }
    // y of the last (up to two) chunks
    for (int ch = max(0, nchunks - 2); ch < nchunks; ch++) {
        bar_sync(kBarEmpty0 + (ch & 1), NT);
        emit(ch);
    }
}

// Occupancy of one variant; a variant whose shared memory exceeds the per-CTA limit of this
// device reports 0 (the caller then uses a variant with fewer rows per CTA).  Computed once per
// device (with the kernel's shared-memory attribute set then) and kept: the queries cost more
// host time than a short scan's launch.
template <typename TA, int DK, int DV, int NW>
cudaError_t prepare_tc(int *occupancy) {
    using C = TcCfg<TA, DK, DV, NW>;
    constexpr int kDevices = 64;
    static std::atomic<int> cached[kDevices];              // occupancy + 1; 0 = not yet known
    auto kern = gdn_scan_tc_kernel<TA, DK, DV, NW>;
    const int bytes = static_cast<int>(sizeof(TcSmem<TA, DK, DV, NW>));
    *occupancy = 0;
    int dev = 0, limit = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cacheable = dev >= 0 && dev < kDevices;
    if (cacheable) {
        const int c = cached[dev].load(std::memory_order_acquire);
        if (c > 0) {
            *occupancy = c - 1;
            return cudaSuccess;
        }
    }
    e = cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    if (bytes <= limit) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occupancy, kern, C::NT, bytes);
        if (e != cudaSuccess) return e;
    }
    if (cacheable) cached[dev].store(*occupancy + 1, std::memory_order_release);
    return cudaSuccess;
}

template <typename TA, int DK, int DV, int NW>
cudaError_t launch_tc_cfg(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream) {
    using C = TcCfg<TA, DK, DV, NW>;
    const int bytes = static_cast<int>(sizeof(TcSmem<TA, DK, DV, NW>));
    const int64_t ctas = static_cast<int64_t>(p.B) * p.Hv * C::NRB * sp.nseg;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(C::NT);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (!C::WHOLE_HEAD && p.z != nullptr) {                // a head's CTAs form one cluster
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C::NRB;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, gdn_scan_tc_kernel<TA, DK, DV, NW>, p, sp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

inline int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Rows per CTA among the candidates NWS (row warps, largest first): the fewest warps on the
// busiest SM with every CTA resident at once (a sequential scan must not run in waves); ties go
// to the larger CTA.  A candidate whose shared memory exceeds this device's limit is skipped.
// `best` is the chosen candidate's index, `per_sm_out` the CTAs it gives the busiest SM (at once
// or in waves).
template <typename TA, int DK, int DV, int... NWS>
cudaError_t choose_tc(const gdn_params &p, const ScanSplit &sp, int *best, int64_t *per_sm_out) {
    constexpr int n = sizeof...(NWS);
    constexpr int nws[n] = {NWS...};
    cudaError_t (*const prep[n])(int *) = {prepare_tc<TA, DK, DV, NWS>...};
    const int sms = std::max(1, device_sms());
    const int64_t heads = static_cast<int64_t>(p.B) * p.Hv * sp.nseg;   // (segment, head) pairs
    *best = -1;
    *per_sm_out = 0;
    int64_t best_cost = INT64_MAX;
    for (int i = 0; i < n; i++) {
        int occ = 0;
        const cudaError_t e = prep[i](&occ);
        if (e != cudaSuccess) return e;
        if (occ < 1) continue;
        const int64_t ctas = heads * (DV / (16 * nws[i]));
        const int64_t per_sm = (ctas + sms - 1) / sms;
        const int64_t waves = (per_sm + occ - 1) / occ;
        const int64_t cost = waves * std::min<int64_t>(per_sm, occ) * nws[i];
        if (cost < best_cost) {
            best_cost = cost;
            *best = i;
            *per_sm_out = per_sm;
        }
    }
    return *best < 0 ? cudaErrorInvalidConfiguration : cudaSuccess;
}

template <typename TA, int DK, int DV, int... NWS>
cudaError_t launch_tc_best(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream) {
    cudaError_t (*const launch[])(const gdn_params &, const ScanSplit &, cudaStream_t) = {
        launch_tc_cfg<TA, DK, DV, NWS>...};
    int best = -1;
    int64_t per_sm = 0;
    const cudaError_t e = choose_tc<TA, DK, DV, NWS...>(p, sp, &best, &per_sm);
    if (e != cudaSuccess) return e;
    return launch[best](p, sp, stream);
}

// Value head dims: multiples of 16 up to 128, and 256.  Up to Dk = 128 a CTA takes a whole head
// of Dv <= 112 (Dv / 16 row warps); Dv = 128 and 256 choose their rows per CTA.  Dk = 256 runs
// at most 4 row warps per CTA, so a head of more rows is split over a cluster of CTAs.
template <typename TA, int DK>
cudaError_t launch_tc_dv(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream) {
    if constexpr (DK <= 128) {
        switch (p.Dv) {
            case 16: return launch_tc_best<TA, DK, 16, 1>(p, sp, stream);
            case 32: return launch_tc_best<TA, DK, 32, 2>(p, sp, stream);
            case 48: return launch_tc_best<TA, DK, 48, 3>(p, sp, stream);
            case 64: return launch_tc_best<TA, DK, 64, 4>(p, sp, stream);
            case 80: return launch_tc_best<TA, DK, 80, 5>(p, sp, stream);
            case 96: return launch_tc_best<TA, DK, 96, 6>(p, sp, stream);
            case 112:   // f32 rows of 128 with 7 row warps exceed the shared-memory limit
                if constexpr (sizeof(TA) == 4) return launch_tc_best<TA, DK, 112, 7, 1>(p, sp, stream);
                else return launch_tc_best<TA, DK, 112, 7>(p, sp, stream);
            case 128: return launch_tc_best<TA, DK, 128, 8, 4, 2>(p, sp, stream);
            case 256: return launch_tc_best<TA, DK, 256, 8, 4>(p, sp, stream);
            default: return cudaErrorInvalidValue;
        }
    } else {
        switch (p.Dv) {
            case 16: return launch_tc_best<TA, DK, 16, 1>(p, sp, stream);
            case 32: return launch_tc_best<TA, DK, 32, 2>(p, sp, stream);
            case 48: return launch_tc_best<TA, DK, 48, 3>(p, sp, stream);
            case 64: return launch_tc_best<TA, DK, 64, 4>(p, sp, stream);
            case 80: return launch_tc_best<TA, DK, 80, 1>(p, sp, stream);
            case 96: return launch_tc_best<TA, DK, 96, 3>(p, sp, stream);
            case 112: return launch_tc_best<TA, DK, 112, 1>(p, sp, stream);
            case 128: return launch_tc_best<TA, DK, 128, 4, 2>(p, sp, stream);
            case 256: return launch_tc_best<TA, DK, 256, 4, 2>(p, sp, stream);
            default: return cudaErrorInvalidValue;
        }
    }
}

// Every activation type and value head dim for one key head dim.
template <int DK>
cudaError_t launch_tc_dk(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream) {
    switch (p.act_dtype) {
        case GDN_F32: return launch_tc_dv<float, DK>(p, sp, stream);
        case GDN_BF16: return launch_tc_dv<__nv_bfloat16, DK>(p, sp, stream);
        case GDN_F16: return launch_tc_dv<__half, DK>(p, sp, stream);
        default: return cudaErrorInvalidValue;
    }
}

// This translation unit's watchdog word (set by a cluster-exchange wait that ran out): read
// and clear (synchronises `stream`).
inline cudaError_t read_watchdog(unsigned *flag, cudaStream_t stream) {
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
