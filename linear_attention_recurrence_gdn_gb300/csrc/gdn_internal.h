// gdn_internal.h -- launchers behind the C ABI (arguments already validated by gdn_api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// One decode step: one CTA per (b, hv) head, gated norm fused in the CTA tail.
cudaError_t launch_decode(const gdn_params &p, cudaStream_t stream);

// The decode step per activation type (gdn_decode_{f32,bf16,f16}.cu) and each unit's watchdog
// word (read and cleared; synchronises `stream`).
cudaError_t launch_decode_f32(const gdn_params &p, cudaStream_t stream);
cudaError_t launch_decode_bf16(const gdn_params &p, cudaStream_t stream);
cudaError_t launch_decode_f16(const gdn_params &p, cudaStream_t stream);
cudaError_t decode_watchdog_f32(unsigned *flag, cudaStream_t stream);
cudaError_t decode_watchdog_bf16(unsigned *flag, cudaStream_t stream);
cudaError_t decode_watchdog_f16(unsigned *flag, cudaStream_t stream);

// Reads and clears the decode kernels' watchdog words (synchronises `stream`).
cudaError_t decode_watchdog(unsigned *flag, cudaStream_t stream);

// One CTA whose mbarrier wait runs out after limit_ns, setting the decode watchdog word.
cudaError_t launch_wait_timeout(cudaStream_t stream, uint64_t limit_ns);

// Multi-token scan (S >= 1): state resident on chip across the time axis.
cudaError_t launch_scan(const gdn_params &p, cudaStream_t stream);

// A scan launch over segments of the sequence.  The plain scan is one segment of S tokens in
// mode 0 with no per-segment buffers.  Segment g covers tokens [g * seg_len, min(S, (g + 1) *
// seg_len)); its CTAs are blocks [g * B*Hv*CTAs-per-head, ...) of the grid.
//   mode 0: each segment from its start memory (s0_seg[g], or p.s0 when s0_seg is NULL),
//           writing y; the last segment writes the final memory to p.state;
//   mode 1: each segment's transition M = prod_t alpha_t (I - beta_t k^_t k^_t^T): the rows of
//           the identity carried through the update with v = 0 (p.Dv == p.Dk), into
//           state_seg[g]; no y;
//   mode 2: each segment's offset N (its end memory from zeros), into state_seg[g]; no y;
//   mode 3: both at once when Dk == Dv: grid segments g < nseg / 2 are the transitions of
//           segments g (into state_seg), the others the offsets of segments g - nseg / 2
//           (into state_seg2).
struct ScanSplit {
    int nseg;              // segments in this launch
    int seg_len;           // tokens per segment (the last one may be shorter)
    int mode;
    const float *s0_seg;   // mode 0: [nseg][B*Hv][Dv][Dk] start memories, or NULL
    float *state_seg;      // modes 1, 2, 3: [nseg][B*Hv][Dv][Dk] end memories
    float *state_seg2;     // mode 3: the offsets' end memories
};

// The sequence-split scan: transitions and offsets of segments 0 .. nseg-2 in parallel, their
// composition into every segment's start memory, then every segment's outputs in parallel.
// `ws` holds gdn_scan_split_workspace() bytes.
cudaError_t launch_scan_split(const gdn_params &p, int nseg, float *ws, cudaStream_t stream);
size_t scan_split_workspace_floats(const gdn_params &p, int nseg);

// The scan on tensor cores, one translation unit per key head dim (gdn_scan_tc_dk*.cu), and
// each unit's watchdog word (read and cleared; synchronises `stream`).
cudaError_t launch_scan_tc_dk16(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream);
cudaError_t launch_scan_tc_dk32(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream);
cudaError_t launch_scan_tc_dk48(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream);
cudaError_t launch_scan_tc_dk64(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream);
cudaError_t launch_scan_tc_dk80(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream);
cudaError_t launch_scan_tc_dk96(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream);
cudaError_t launch_scan_tc_dk112(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream);
cudaError_t launch_scan_tc_dk128(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream);
// The block kernel's launch plan for Dk = Dv = 128 (16-bit activations): CTAs per SM and per
// head of the configuration it would choose.
cudaError_t scan_tc_dk128_plan(const gdn_params &p, int64_t *per_sm, int *ctas_per_head);
cudaError_t launch_scan_tc_dk256(const gdn_params &p, const ScanSplit &sp, cudaStream_t stream);
cudaError_t scan_watchdog_dk16(unsigned *flag, cudaStream_t stream);
cudaError_t scan_watchdog_dk32(unsigned *flag, cudaStream_t stream);
cudaError_t scan_watchdog_dk48(unsigned *flag, cudaStream_t stream);
cudaError_t scan_watchdog_dk64(unsigned *flag, cudaStream_t stream);
cudaError_t scan_watchdog_dk80(unsigned *flag, cudaStream_t stream);
cudaError_t scan_watchdog_dk96(unsigned *flag, cudaStream_t stream);
cudaError_t scan_watchdog_dk112(unsigned *flag, cudaStream_t stream);
cudaError_t scan_watchdog_dk128(unsigned *flag, cudaStream_t stream);
cudaError_t scan_watchdog_dk256(unsigned *flag, cudaStream_t stream);

// The chunked scan with the memory in tensor memory (bf16, Dk = Dv = 128, 16-byte aligned
// operands; chosen by GDN_FLAG_SCAN_TMEM), and its watchdog word.
bool scan_umma_supported(const gdn_params &p);
cudaError_t launch_scan_umma(const gdn_params &p, cudaStream_t stream);
cudaError_t scan_umma_watchdog(unsigned *flag, cudaStream_t stream);

// The chunked (WY) scan on tcgen05: bf16 or f16 activations, Dk = Dv = 128, 16-byte aligned
// q, k, v; its watchdog word; the first-attempt limit of its waits (0 = the default), set only
// by the self-test hook (synchronises `stream`).
// General kernel (gdn_general.cu): any Dk, Dv from 1 to 256 whose memory, rows padded to an odd
// stride, fits in the shared memory of one CTA; used for the dims the tiled kernels do not take.
constexpr size_t kGeneralSmemMax = 226 * 1024;
// Head dims of the tiled kernels (decode, the block and chunked scans, the split scan).
inline bool tiled_dim(int d) { return (d >= 16 && d <= 128 && d % 16 == 0) || d == 256; }
inline bool tiled_dims(const gdn_params &p) { return tiled_dim(p.Dk) && tiled_dim(p.Dv); }
size_t general_smem_bytes(int dk, int dv);
bool general_supported(int dk, int dv);
// decode: the memory is read from and written back to `state` (a decode step); else the scan
// starts from s0 (NULL = zeros) and writes `state`.
cudaError_t launch_general(const gdn_params &p, bool decode, cudaStream_t stream);

bool scan_wy_supported(const gdn_params &p);
cudaError_t launch_scan_wy(const gdn_params &p, cudaStream_t stream);
cudaError_t scan_wy_watchdog(unsigned *flag, cudaStream_t stream);
cudaError_t scan_wy_set_first_wait_limit(unsigned long long ns, cudaStream_t stream);

// Reads and clears the scan kernels' watchdog words (synchronises `stream`).
cudaError_t scan_watchdog(unsigned *flag, cudaStream_t stream);

}  // namespace gdn
