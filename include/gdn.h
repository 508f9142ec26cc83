/*
 * gdn.h -- C ABI of libgdn.so, a GB300 (sm_103a) implementation of the Gated DeltaNet (GDN)
 * linear-attention recurrence.
 *
 * WHAT IS COMPUTED
 *   logicaffeine_compile::codegen_cuda::gdn (module description): every value head keeps a
 *   Dv x Dk f32 memory S and, per token,
 *       u = S k^                              (prediction from the OLD memory)
 *       S = alpha S + beta (v - alpha u) k^T  (decay, then correct by the prediction error)
 *       o = S q^                              (read of the UPDATED memory)
 *       y = rmsnorm(o * silu(z)) * GN         (gate first, then normalise over the head)
 *   The kernels evaluate o with the single-pass identity of that page's "The fusion"
 *   section, o[a] = alpha (S_old q^)[a] + coef[a] (k^ . q^), coef[a] = beta (v[a] - alpha u[a]),
 *   so each state row is read once and written once per token.
 *
 *   torch_to_nnef.op.gated_delta, native_gdn_reject_reason: q and k are l2-normalised and the
 *   1/sqrt(head_dim) scale is folded in:
 *       k^ = k / sqrt(sum k^2 + qk_eps),   q^ = q / sqrt(sum q^2 + qk_eps) / sqrt(Dk).
 *   alpha = exp(log_decay); beta is used as given.  rmsnorm: x / sqrt(mean x^2 + norm_eps).
 *   Value head hv reads key head hv / (Hv / Hk) (modelopt.torch.puzzletron.pruning.
 *   gated_delta_net, GDNShape.value_heads_per_group).
 *
 * LAYOUTS  (torch_to_nnef.op.gated_delta, emit_native_gdn_recurrent; all dense row-major)
 *   head_major = 0:  q,k [B,S,Hk,Dk]   v,z,y [B,S,Hv,Dv]   log_decay,beta [B,S,Hv]
 *   head_major = 1:  q,k [B,Hk,S,Dk]   v,z,y [B,Hv,S,Dv]   log_decay,beta [B,Hv,S]
 *   state, s0:       [B,Hv,Dv,Dk] f32, row = value index, column = key index.
 *   gn:              [Dv] f32.
 *
 * HEAD DIMS
 *   Dk and Dv are independent.  Multiples of 16 from 16 to 128, and 256, run the tiled
 *   kernels (tensor cores, bulk copies).  Any other Dk, Dv from 1 to 256 runs a general
 *   kernel (f32 on CUDA cores, plain loads, one CTA per head), provided that the head's
 *   memory fits in its shared memory: Dv * ld * 4 + 8 * Dk4 + 96 <= 226 KB, Dk4 being Dk
 *   rounded up to a multiple of 4 and ld a row stride of Dk4 plus at most 28 floats of bank
 *   padding (e.g. any Dk, Dv up to 232).  Pruned widths of any size are allowed by modelopt
 *   puzzletron.pruning.gated_delta_net (slice_gated_delta_net_state_dict, GDNShape).  Other
 *   dims: GDN_ERR_UNSUPPORTED_DIM.
 *   y is always f32: the promoted type of gated_delta_fake on the same page (the memory is
 *   f32 even for a 16-bit model).
 *
 * OWNERSHIP
 *   The caller owns every buffer and every pointer is a DEVICE pointer (the stream's device),
 *   except under GDN_FLAG_HOST_IO below.  The library allocates nothing, keeps no state
 *   between calls and never copies to the host.  Work is enqueued on `stream` (a cudaStream_t passed as void*, NULL = legacy
 *   default stream) and is asynchronous: results are ready when the stream is.
 *
 * ERRORS
 *   Every entry point validates its arguments on the host BEFORE enqueuing anything and
 *   returns a negative gdn_status on failure, with nothing enqueued and no buffer touched.
 *   A launch failure returns GDN_ERR_CUDA (text from gdn_last_error()).  Faults during
 *   kernel execution surface at the caller's next synchronisation, as usual for CUDA.
 *   There is no fallback path of any kind.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_VERSION 1

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

typedef enum {
    GDN_F32 = 0,
    GDN_BF16 = 1,
    GDN_F16 = 2
} gdn_dtype;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_NULL_PTR = -1,        /* a required pointer is NULL, or z/gn only one given     */
    GDN_ERR_BAD_SHAPE = -2,       /* dims < 0 or heads < 1, Hv % Hk != 0, S != 1 on decode   */
    GDN_ERR_UNSUPPORTED_DIM = -3, /* Dk or Dv above 256, or too large a memory (HEAD DIMS)    */
    GDN_ERR_BAD_DTYPE = -4,       /* unknown dtype, or gate dtype neither F32 nor act dtype  */
    GDN_ERR_MISALIGNED = -5,      /* a pointer is not aligned (16 B; gates: element size)    */
    GDN_ERR_ALIASING = -6,        /* y overlaps an operand, or state partially overlaps s0   */
    GDN_ERR_BAD_ARG = -7,         /* eps negative or not finite; bad flag; size overflow     */
    GDN_ERR_CUDA = -8,            /* the CUDA runtime reported an error                      */
    GDN_ERR_TIMEOUT = -9          /* a kernel gave up waiting for its own async copies       */
} gdn_status;

/* Option bits of gdn_params.flags.
 *   Two scan kernels give the same results within the scan tolerance: the chunked kernel,
 *   which writes the recurrence over 64-token chunks in WY form on tcgen05 tensor cores (bf16
 *   or f16 activations with Dk == Dv == 128 and 16-byte aligned q, k, v; one CTA per head),
 *   and the 16-token block kernel on warp-level MMAs (every shape; a head's rows may spread
 *   over a cluster of CTAs).  By default gdn_scan runs the chunked kernel where it applies,
 *   except for bf16 when the block kernel's launch would split each head over several CTAs
 *   and give no SM more than one CTA (few heads; as measured, the block kernel is then
 *   faster); every other shape runs the block kernel.
 *   At most one of GDN_FLAG_SCAN_TMEM, GDN_FLAG_SCAN_BLOCK16 and GDN_FLAG_SCAN_CHUNKED may be
 *   set.
 *   GDN_FLAG_SCAN_TMEM  gdn_scan only (gdn_decode_step rejects it): run instead the 32-token
 *                       look-ahead kernel that keeps each head's memory in tensor memory, where
 *                       it applies (bf16 activations, Dk == Dv == 128); other shapes run the
 *                       16-token block kernel. */
#define GDN_FLAG_SCAN_TMEM 1
/*   GDN_FLAG_HOST_IO    gdn_decode_step only (gdn_scan rejects it): q, k, v, z, log_decay,
 *                       beta and y may live in pinned host memory that is mapped into the
 *                       device's address space (cudaHostAlloc, or cudaHostRegister with
 *                       cudaHostRegisterMapped, under unified addressing: the host address is
 *                       the device address).  The kernel then reads each head's inputs with
 *                       plain loads one head ahead and writes y with plain stores, so a step
 *                       fed from the host needs no separate copies.  state and gn stay in
 *                       device memory.  Device pointers remain valid with the flag.  Passing
 *                       memory the device cannot address is a fault, as with any bad pointer. */
#define GDN_FLAG_HOST_IO 2
/*   GDN_FLAG_SCAN_BLOCK16  gdn_scan (and gdn_scan_split) only: run the 16-token block kernel
 *                       for every shape, also where the chunked kernel applies. */
#define GDN_FLAG_SCAN_BLOCK16 4
/*   GDN_FLAG_SCAN_CHUNKED  gdn_scan (and gdn_scan_split) only: run the chunked kernel wherever
 *                       it applies, also where the default would pick the block kernel;
 *                       other shapes run the block kernel. */
#define GDN_FLAG_SCAN_CHUNKED 8

/* Operands of one call.  Shape fields follow GDNShape (num_key_heads = Hk, num_value_heads
 * = Hv, key_head_dim = Dk, value_head_dim = Dv) plus batch B and sequence length S. */
typedef struct gdn_params {
    int32_t B, S, Hk, Hv, Dk, Dv;
    int32_t head_major;       /* 0: [B,S,H,W] / [B,S,H] operands; 1: [B,H,S,W] / [B,H,S]     */
    int32_t act_dtype;        /* gdn_dtype of q, k, v, z                                      */
    int32_t gate_dtype;       /* gdn_dtype of log_decay and beta: GDN_F32 or act_dtype        */
    int32_t flags;            /* GDN_FLAG_* bits (0 = defaults); unknown bits are rejected    */
    const void *q, *k;        /* [B,S,Hk,Dk] / [B,Hk,S,Dk]                                    */
    const void *v;            /* [B,S,Hv,Dv] / [B,Hv,S,Dv]                                    */
    const void *log_decay;    /* [B,S,Hv] / [B,Hv,S]                                          */
    const void *beta;         /* [B,S,Hv] / [B,Hv,S]                                          */
    const void *z;            /* like v; NULL together with gn: y = raw o (no gated norm).
                                 With S == 0 every per-token pointer may be NULL              */
    const float *gn;          /* [Dv] f32 gated-norm weight; NULL together with z             */
    const float *s0;          /* scan: initial memory [B,Hv,Dv,Dk]; NULL = zeros.
                                 decode: ignored (the memory is `state`, updated in place)    */
    float *state;             /* decode: memory, read and written in place.
                                 scan: final memory out; may be the same pointer as s0        */
    float *y;                 /* output, like v but f32; must not overlap any operand;
                                 may be NULL only when S == 0 (nothing is written)            */
    float qk_eps;             /* l2-norm eps of q and k (1e-6 in the reference workloads)     */
    float norm_eps;           /* rmsnorm eps (1e-6 in the reference workloads)                */
} gdn_params;

/*
 * gdn_decode_step -- one token (S must be 1) for every (b, hv) head; `state` is read and
 * written in place (one HBM read and one write of each state row).  At S == 1 the two
 * layouts coincide, so head_major only has to be a valid flag.  B == 0 is a no-op.
 * Source: logicaffeine codegen_cuda::gdn, "The fusion" and GDN_KERNELS; torch_to_nnef
 * gated_delta, native_gdn_reject_reason (the fused operator is a single decode step).
 */
GDN_API int gdn_decode_step(const gdn_params *p, void *stream);

/*
 * gdn_scan -- the recurrence over the time axis, t = 0 .. S-1, from s0 (or zeros) to the
 * final memory written to `state`; y receives every token's output.  Each head's memory
 * stays on chip for the whole sequence.  S == 0 copies s0 (or zeros) into `state` and
 * leaves y untouched; B == 0 is a no-op.  `state` may equal `s0` (in-place resume); any
 * other overlap of the two is rejected.
 * Source: torch_to_nnef gated_delta, gated_delta_reference (recurrence over the time axis)
 * and emit_native_gdn_recurrent (operands and outputs); logicaffeine codegen_cuda::gdn.
 */
GDN_API int gdn_scan(const gdn_params *p, void *stream);

/*
 * gdn_scan_split -- gdn_scan with the sequence cut into `segments` ranges of ceil(S / segments)
 * tokens (fewer if S is small), for batches with too few heads to fill the GPU.  The update is
 * affine in the memory (logicaffeine codegen_cuda::gdn, "The fusion"), so a segment maps its
 * start memory S0 to S0 M + N.  M is the product of alpha_t (I - beta_t k^_t k^_t^T) over the
 * segment, and N is the memory it reaches from zeros.  The call computes M and N of every
 * segment but the last in parallel, composes the segments' start memories in order, then runs
 * every segment from its start in parallel, writing y and, for the last, `state`.  The results
 * equal gdn_scan's within the scan tolerance.  It takes about 3x gdn_scan's work, spread over
 * `segments` times as many CTAs, so it pays when B * Hv leaves most of the GPU idle (measured
 * 1.9x faster with 4 segments, 2.1x with 8, on one sequence of 16384 tokens with 8 heads).
 * `workspace`: device memory of at least gdn_scan_split_workspace(p, segments) bytes, 16-byte
 * aligned, overlapping no operand; the caller owns it.  When the sequence yields a single
 * segment (segments == 1, or S == 1) no workspace is needed and gdn_scan runs; so it does for
 * head dims of the general kernel (HEAD DIMS above), whose whole sequence runs in one launch
 * (segments ignored, no workspace).  Errors as gdn_scan, plus GDN_ERR_BAD_ARG for
 * segments < 1, a short workspace or GDN_FLAG_SCAN_TMEM, GDN_ERR_NULL_PTR / MISALIGNED /
 * ALIASING for the workspace (the reason in gdn_last_error()).
 */
GDN_API int gdn_scan_split(const gdn_params *p, int segments, void *workspace,
                           size_t workspace_bytes, void *stream);

/* Workspace bytes gdn_scan_split(p, segments, ...) needs: 0 when it needs none, or when `p`
 * would be rejected by gdn_scan.  (segments - 1) * B * Hv * (Dk + Dv) * Dk + segments * B * Hv
 * * Dv * Dk floats, with segments reduced so that none is empty.  Source: none on the pages
 * (a size query for gdn_scan_split). */
GDN_API size_t gdn_scan_split_workspace(const gdn_params *p, int segments);

/*
 * gdn_scan_split_noalloc -- gdn_scan_split for callers that cannot allocate device memory
 * (code that runs inside another framework's memory pool or arena, or where a cudaMalloc
 * would synchronise the device or is not allowed), so cannot provide the workspace.  It
 * computes the same results as gdn_scan_split with a workspace, but takes its scratch from
 * one fixed device array inside the library, GDN_SCAN_SPLIT_NOALLOC_MAX_BYTES (16 MiB), which
 * every device that loads the library holds until the process exits.  The caller still passes
 * every input and output in `p`.  The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *   - Calls whose scratch, gdn_scan_split_workspace(p, segments), exceeds the maximum return
 *     GDN_ERR_BAD_ARG before anything is enqueued (the sizes in gdn_last_error()); a single
 *     segment needs no scratch and runs gdn_scan.
 *   - The first call that needs scratch on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, which keeps the last call's contents (each
 *     call writes every scratch element before reading it, so nothing needs clearing).  Calls
 *     that overlap on the GPU (on different streams, or from different threads) race on it:
 *     order them on one stream, or synchronise between them.
 *   - Other errors as gdn_scan_split.
 * Source: none on the pages -- the pages have no counterpart; a deployment variant of
 * gdn_scan_split.
 */
#define GDN_SCAN_SPLIT_NOALLOC_MAX_BYTES (16u << 20)
GDN_API int gdn_scan_split_noalloc(const gdn_params *p, int segments, void *stream);

/*
 * gdn_reject_reason -- NULL when gdn_decode_step (is_decode != 0) or gdn_scan (is_decode
 * == 0) would accept `p`, else a short static string naming the first failed check.
 * Host-only; touches no device memory.
 * Source: torch_to_nnef gated_delta, native_gdn_reject_reason (a reason string for logging;
 * this library has no fallback to log it before).
 */
GDN_API const char *gdn_reject_reason(const gdn_params *p, int is_decode);

/* gdn_status_string -- static text for a gdn_status value (unknown codes included).
 * Source: none on the pages -- the library's own status codes. */
GDN_API const char *gdn_status_string(int status);

/* gdn_last_error -- text of the last GDN_ERR_CUDA seen by the calling thread ("" if none), or
 * of the last rejection that gdn_reject_reason cannot name (split-scan arguments).
 * Source: none on the pages -- the library's own error reporting. */
GDN_API const char *gdn_last_error(void);

/*
 * gdn_device_status -- waits for `stream`, then reports whether a kernel of this library,
 * since the last call on this device, gave up a wait on an mbarrier after its time limit
 * (about 2 s; never expected on a healthy GPU): the decode kernel's wait for its own bulk
 * copies (it then abandons its work), or the scan's wait for the partial norm sums of the
 * other CTAs of its cluster (it then carries on with what it has).  Returns GDN_ERR_TIMEOUT
 * then (the outputs of that call are incomplete or invalid) and clears the condition; GDN_OK
 * otherwise; GDN_ERR_CUDA if the runtime reports an error.
 * Source: none on the pages -- failure detection for the asynchronous-copy waits.
 */
GDN_API int gdn_device_status(void *stream);

/*
 * gdn_selftest_wait_timeout -- exercises the failure path above without a GPU fault: launches
 * one CTA on `stream` whose mbarrier wait can never complete (the barrier expects 16 bytes
 * that no copy sends); the wait gives up after `limit_ms` milliseconds, sets the watchdog word
 * and the CTA returns.  The next gdn_device_status on that device then reports
 * GDN_ERR_TIMEOUT (and clears it).  Returns GDN_ERR_BAD_ARG unless 0 < limit_ms <= 2000,
 * GDN_ERR_CUDA on a launch error, GDN_OK otherwise (asynchronous on `stream`).
 * Source: none on the pages -- a test hook for the bounded waits.
 */
GDN_API int gdn_selftest_wait_timeout(void *stream, double limit_ms);

/*
 * gdn_selftest_scan_wait_limit -- exercises the scan's own bounded waits without a GPU fault:
 * sets, for later launches of the chunked scan kernel on the current device, the time limit
 * of the first attempt of each of its mbarrier waits to `limit_us` microseconds (0 restores
 * the default of about 2 s).  A first attempt that runs out sets the watchdog word, so
 * gdn_device_status then reports GDN_ERR_TIMEOUT, and the wait is retried with the full limit;
 * only if that also runs out does the CTA abandon its work.  So with a tiny limit a scan
 * reports the timeout and still computes correct results.  Synchronises `stream`.  Returns
 * GDN_ERR_BAD_ARG unless 0 <= limit_us <= 2e6, GDN_ERR_CUDA on a runtime error, else GDN_OK.
 * Source: none on the pages -- a test hook for the bounded waits.
 */
GDN_API int gdn_selftest_scan_wait_limit(void *stream, double limit_us);

/* gdn_version -- GDN_VERSION of the loaded library.
 * Source: none on the pages -- the library's own version number. */
GDN_API int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
