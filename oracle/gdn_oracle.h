/*
 * gdn_oracle.h -- interface of the fp64 GDN oracle (test infrastructure only).
 *
 * Not part of the product: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  All arrays are host memory, dense row-major, double precision; see
 * gdn_oracle.c for the layouts and for what is computed.
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_LITERAL = 0, ORACLE_FUSED = 1 };

typedef struct {
    int32_t B, S, Hk, Hv, Dk, Dv;
    int32_t head_major;            /* 0: [B,S,H,W] operands, 1: [B,H,S,W] operands          */
    int32_t mode;                  /* ORACLE_LITERAL or ORACLE_FUSED                          */
    const double *q, *k;           /* [B,S,Hk,Dk] or [B,Hk,S,Dk]                              */
    const double *v, *z;           /* [B,S,Hv,Dv] or [B,Hv,S,Dv]; z may be NULL (with gn)    */
    const double *g, *beta;        /* log_decay and beta, [B,S,Hv] or [B,Hv,S]                */
    const double *gn;              /* [Dv] gated-norm weight, NULL together with z            */
    const double *s0;              /* [B,Hv,Dv,Dk] initial memory, NULL = zeros               */
    double *y;                     /* same layout as v                                        */
    double *state;                 /* [B,Hv,Dv,Dk] final memory                               */
    double qk_eps, norm_eps;
    const int64_t *heads;          /* optional subset of flattened heads b*Hv+hv (NULL = all) */
    int64_t n_heads;
    int32_t threads;               /* worker threads over heads (1 = sequential)              */
    int32_t reserved;
} oracle_gdn_args;

/* Returns 0 on success, a negative code on bad arguments.  Only the selected heads' entries
 * of y and state are written. */
int oracle_gdn_run(const oracle_gdn_args *a);

#ifdef __cplusplus
}
#endif

#endif
