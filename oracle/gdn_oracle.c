/*
 * gdn_oracle.c -- fp64 reference oracle for the Gated DeltaNet (GDN) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this file:
 * it is used by the test-suite, by the smoke check and by the CPU-baseline leg of the
 * benchmark.  It shares no code, header, constant or helper with the CUDA library.
 *
 * What it computes (plain definition, double precision throughout, straightforward loops):
 *
 *   Source: "logicaffeine_compile::codegen_cuda::gdn" (module description).  Each value head
 *   holds a D x D memory S and, for every token,
 *       u = S k                        prediction of the memory for this key  (OLD S)
 *       S = alpha S + beta (v - alpha u) k^T
 *       o = S q                        read of the UPDATED memory
 *       o = rmsnorm(o * silu(z)) * GN  gate first, then normalise over the whole head
 *
 *   Source: "torch_to_nnef.op.gated_delta", native_gdn_reject_reason: the fused operator
 *   folds the q/k l2-normalisation and the 1/sqrt(head_dim) output scale.  Readings used
 *   here (the page prints no formula for either):
 *       k^ = k / sqrt(sum k^2 + qk_eps)
 *       q^ = q / sqrt(sum q^2 + qk_eps) / sqrt(Dk)     (scale applied to q; o is linear in q)
 *   alpha = exp(log_decay) (the operand is named log_decay on the same page).
 *   beta is used as given.
 *
 *   Key head of value head hv:  hk = hv / (Hv / Hk)   (contiguous groups of
 *   "value_heads_per_group", modelopt.torch.puzzletron.pruning.gated_delta_net, GDNShape).
 *
 *   State layout [B, Hv, Dv, Dk]: row a is the value index, column j the key index, as the
 *   "The fusion" section of the logicaffeine page indexes S[a][b] with b summed against k, q.
 *
 *   Operand layouts ("torch_to_nnef.op.gated_delta", emit_native_gdn_recurrent):
 *       head_major = 0:  q,k [B,S,Hk,Dk]   v,z,y [B,S,Hv,Dv]   log_decay,beta [B,S,Hv]
 *       head_major = 1:  q,k [B,Hk,S,Dk]   v,z,y [B,Hv,S,Dv]   log_decay,beta [B,Hv,S]
 *   y is always the promoted (here: double) type, per gated_delta_fake on the same page.
 *
 * Two evaluation modes, both from the logicaffeine page:
 *   ORACLE_LITERAL (0): the three literal passes (S k, rank-1 update, S_new q).
 *   ORACLE_FUSED   (1): the single-pass identity of its "The fusion" section,
 *                        o[a] = alpha (S_old q)[a] + coef[a] (k . q),
 *                        coef[a] = beta (v[a] - alpha u[a]).
 *   The two must agree to rounding; the tests check that.
 *
 * Gated norm (same page, module description and GDN_KERNELS):
 *       x[a] = o[a] * z[a] / (1 + exp(-z[a]))            (silu(z) = z * sigmoid(z))
 *       y[a] = x[a] / sqrt(mean_a x[a]^2 + norm_eps) * GN[a]
 *   When z and gn are both NULL the raw o is returned (used to make the q scale visible).
 *
 * Threads: heads (b, hv) are independent; a small pthread pool splits them.  threads = 1 is
 * the plain sequential program.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "gdn_oracle.h"

static int64_t idx_qk(const oracle_gdn_args *a, int64_t b, int64_t t, int64_t h, int64_t j)
{
    if (a->head_major)
        return ((b * a->Hk + h) * a->S + t) * a->Dk + j;
    return ((b * a->S + t) * a->Hk + h) * a->Dk + j;
}

static int64_t idx_v(const oracle_gdn_args *a, int64_t b, int64_t t, int64_t h, int64_t i)
{
    if (a->head_major)
        return ((b * a->Hv + h) * a->S + t) * a->Dv + i;
    return ((b * a->S + t) * a->Hv + h) * a->Dv + i;
}

static int64_t idx_gate(const oracle_gdn_args *a, int64_t b, int64_t t, int64_t h)
{
    if (a->head_major)
        return (b * a->Hv + h) * a->S + t;
    return (b * a->S + t) * a->Hv + h;
}

/* Per-thread work buffers. */
typedef struct {
    double *S;    /* Dv x Dk */
    double *kh;   /* Dk */
    double *qh;   /* Dk */
    double *u;    /* Dv */
    double *o;    /* Dv */
} oracle_work;

/* One value head over the whole time axis. */
static void run_head(const oracle_gdn_args *a, int64_t head, oracle_work *wk)
{
    const int64_t Dk = a->Dk, Dv = a->Dv;
    const int64_t b = head / a->Hv;
    const int64_t hv = head % a->Hv;
    const int64_t hk = hv / (a->Hv / a->Hk);
    double *S = wk->S;

    /* initial memory */
    for (int64_t i = 0; i < Dv * Dk; i++)
        S[i] = a->s0 ? a->s0[head * Dv * Dk + i] : 0.0;

    for (int64_t t = 0; t < a->S; t++) {
        /* l2-normalised key and query, query scaled by 1/sqrt(Dk) */
        double ssk = 0.0, ssq = 0.0;
        for (int64_t j = 0; j < Dk; j++) {
            double kv = a->k[idx_qk(a, b, t, hk, j)];
            double qv = a->q[idx_qk(a, b, t, hk, j)];
            ssk += kv * kv;
            ssq += qv * qv;
        }
        const double rk = 1.0 / sqrt(ssk + a->qk_eps);
        const double rq = 1.0 / sqrt(ssq + a->qk_eps) / sqrt((double)Dk);
        for (int64_t j = 0; j < Dk; j++) {
            wk->kh[j] = a->k[idx_qk(a, b, t, hk, j)] * rk;
            wk->qh[j] = a->q[idx_qk(a, b, t, hk, j)] * rq;
        }
        const double alpha = exp(a->g[idx_gate(a, b, t, hv)]);
        const double beta = a->beta[idx_gate(a, b, t, hv)];

        if (a->mode == ORACLE_LITERAL) {
            /* pass 1: u = S_old k^ */
            for (int64_t i = 0; i < Dv; i++) {
                double acc = 0.0;
                for (int64_t j = 0; j < Dk; j++)
                    acc += S[i * Dk + j] * wk->kh[j];
                wk->u[i] = acc;
            }
            /* pass 2: S = alpha S + beta (v - alpha u) k^T */
            for (int64_t i = 0; i < Dv; i++) {
                const double vi = a->v[idx_v(a, b, t, hv, i)];
                for (int64_t j = 0; j < Dk; j++)
                    S[i * Dk + j] = alpha * S[i * Dk + j] + beta * (vi - alpha * wk->u[i]) * wk->kh[j];
            }
            /* pass 3: o = S_new q^ */
            for (int64_t i = 0; i < Dv; i++) {
                double acc = 0.0;
                for (int64_t j = 0; j < Dk; j++)
                    acc += S[i * Dk + j] * wk->qh[j];
                wk->o[i] = acc;
            }
        } else {
            /* fused single pass: u = S_old k^, w = S_old q^, kq = k^ . q^ */
            double kq = 0.0;
            for (int64_t j = 0; j < Dk; j++)
                kq += wk->kh[j] * wk->qh[j];
            for (int64_t i = 0; i < Dv; i++) {
                double uu = 0.0, ww = 0.0;
                for (int64_t j = 0; j < Dk; j++) {
                    uu += S[i * Dk + j] * wk->kh[j];
                    ww += S[i * Dk + j] * wk->qh[j];
                }
                const double coef = beta * (a->v[idx_v(a, b, t, hv, i)] - alpha * uu);
                for (int64_t j = 0; j < Dk; j++)
                    S[i * Dk + j] = alpha * S[i * Dk + j] + coef * wk->kh[j];
                wk->o[i] = alpha * ww + coef * kq;
            }
        }

        /* gated RMSNorm over the Dv outputs of this (b, t, hv) */
        if (a->z) {
            double ss = 0.0;
            for (int64_t i = 0; i < Dv; i++) {
                const double zi = a->z[idx_v(a, b, t, hv, i)];
                const double x = wk->o[i] * zi / (1.0 + exp(-zi));
                wk->o[i] = x;
                ss += x * x;
            }
            const double r = 1.0 / sqrt(ss / (double)Dv + a->norm_eps);
            for (int64_t i = 0; i < Dv; i++)
                a->y[idx_v(a, b, t, hv, i)] = wk->o[i] * r * a->gn[i];
        } else {
            for (int64_t i = 0; i < Dv; i++)
                a->y[idx_v(a, b, t, hv, i)] = wk->o[i];
        }
    }

    for (int64_t i = 0; i < Dv * Dk; i++)
        a->state[head * Dv * Dk + i] = S[i];
}

typedef struct {
    const oracle_gdn_args *a;
    int64_t n_heads;
    int64_t next;            /* next list position to take */
    pthread_mutex_t lock;
    int failed;
} oracle_pool;

static int64_t head_at(const oracle_gdn_args *a, int64_t pos)
{
    return a->heads ? a->heads[pos] : pos;
}

static void *worker(void *arg)
{
    oracle_pool *pool = (oracle_pool *)arg;
    const oracle_gdn_args *a = pool->a;
    oracle_work wk;
    const size_t dk = (size_t)a->Dk, dv = (size_t)a->Dv;
    double *mem = (double *)malloc(sizeof(double) * (dv * dk + 2 * dk + 2 * dv));
    if (!mem) {
        pthread_mutex_lock(&pool->lock);
        pool->failed = 1;
        pthread_mutex_unlock(&pool->lock);
        return NULL;
    }
    wk.S = mem;
    wk.kh = wk.S + dv * dk;
    wk.qh = wk.kh + dk;
    wk.u = wk.qh + dk;
    wk.o = wk.u + dv;
    for (;;) {
        pthread_mutex_lock(&pool->lock);
        const int64_t pos = pool->next++;
        pthread_mutex_unlock(&pool->lock);
        if (pos >= pool->n_heads)
            break;
        run_head(a, head_at(a, pos), &wk);
    }
    free(mem);
    return NULL;
}

int oracle_gdn_run(const oracle_gdn_args *a)
{
    if (!a || !a->q || !a->k || !a->v || !a->g || !a->beta || !a->y || !a->state)
        return -1;
    if (a->B < 0 || a->S < 0 || a->Hk <= 0 || a->Hv <= 0 || a->Dk <= 0 || a->Dv <= 0)
        return -2;
    if (a->Hv % a->Hk != 0)
        return -2;
    if ((a->z == NULL) != (a->gn == NULL))
        return -3;
    if (a->mode != ORACLE_LITERAL && a->mode != ORACLE_FUSED)
        return -4;

    const int64_t total = (int64_t)a->B * a->Hv;
    const int64_t n = a->heads ? a->n_heads : total;
    for (int64_t i = 0; a->heads && i < n; i++)
        if (a->heads[i] < 0 || a->heads[i] >= total)
            return -2;

    int threads = a->threads > 0 ? a->threads : 1;
    if (threads > 256)
        threads = 256;
    if (threads > n)
        threads = n > 0 ? (int)n : 1;

    oracle_pool pool;
    pool.a = a;
    pool.n_heads = n;
    pool.next = 0;
    pool.failed = 0;
    pthread_mutex_init(&pool.lock, NULL);

    if (threads == 1) {
        worker(&pool);
    } else {
        pthread_t tid[256];
        int started = 0;
        for (int i = 0; i < threads; i++) {
            if (pthread_create(&tid[i], NULL, worker, &pool) != 0)
                break;
            started++;
        }
        if (started == 0)
            worker(&pool);
        for (int i = 0; i < started; i++)
            pthread_join(tid[i], NULL);
    }
    pthread_mutex_destroy(&pool.lock);
    return pool.failed ? -5 : 0;
}
