/*
 * Oracle for deferred-RoPE attention (TEST INFRASTRUCTURE ONLY).
 *
 * Plain, slow, obviously correct fp64 CPU code. Only the tests, the smoke check and the bench's
 * CPU-baseline leg may call it; the product path never does. It shares no code, header or
 * table with the CUDA library.
 *
 * What it computes follows "LazyAttention: Efficient Retrieval-Augmented Generation with
 * Deferred Positional Encoding" (technical summaries, section "Mathematical equivalence"): the
 * deferred form is identical to attention over keys materialised with standard RoPE at their
 * absolute logical positions, because RoPE scores depend only on the position difference n - m.
 * So form A below is that plain definition:
 *   theta_i = base^(-2i/D), i = 0..D/2-1
 *   R(p) x : (x_i, x_{i+D/2}) -> (x_i cos(p theta_i) - x_{i+D/2} sin(p theta_i),
 *                                 x_i sin(p theta_i) + x_{i+D/2} cos(p theta_i))   (half-split)
 *   s_k = scale * (R(m) q) . (R(p_k) k_k),   visible keys only
 *   out = sum_k softmax(s)_k v_k,   lse = max_k s_k + ln sum_k exp(s_k - max)
 * Form B is the lazy form the summaries describe ("Concepto central" / decoding section):
 *   s_k = scale * (R(m - o_k) q) . (R(j_k) k_k)   with p_k = o_k + j_k,
 * i.e. a key stored once at its document-local position j_k and attended at offset o_k.
 * Form S (the stored-key form) is form A with the cache's storage step written out: a key that
 * the cache holds is kept as round(R(j_k) k_k), rounded to the cache's element type (bf16 or
 * fp32; the summaries' "Core concept": the cache holds each document's keys once, rotated only
 * at document-local positions), and attended as R(o_k) round(R(j_k) k_k); a key that is not
 * cached (a question token's own key) enters as R(p_k) k_k. With exact storage S equals A.
 *
 * Visibility: a key flagged causal (a question token's own key) is visible to a query at m only
 * if its position p_k <= m; every other key (a cached document or private-segment key) is
 * visible to every query.
 *
 * Build: gcc -O2 -fPIC -shared -pthread oracle.c -lm (no fast-math).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* R(pos) x for one head vector of length D (half-split pairing), in place. */
static void rope_rotate(double *x, int D, double pos, double base) {
    int h = D / 2;
    for (int i = 0; i < h; ++i) {
        double theta = pow(base, -2.0 * (double)i / (double)D);
        double a = pos * theta;
        double c = cos(a), s = sin(a);
        double x0 = x[i], x1 = x[i + h];
        x[i] = x0 * c - x1 * s;
        x[i + h] = x0 * s + x1 * c;
    }
}

/* x rounded to the nearest bfloat16 (8 significant bits; ties to even under the default
 * rounding mode). Below the smallest normal, 2^-126, the spacing stays 2^-133 (subnormals);
 * results beyond the largest finite value, (2 - 2^-7) 2^127, become +-inf. */
static double round_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e); /* |x| in [2^(e-1), 2^e) */
    if (e < -125) e = -125;
    double q = ldexp(1.0, e - 8); /* spacing of 8-bit significands in that binade */
    double r = nearbyint(x / q) * q;
    if (fabs(r) >= ldexp(1.0, 128)) r = copysign(INFINITY, x);
    return r;
}

/* Storage rounding of a cached element: 0 = none (exact), 1 = bfloat16, 2 = float32. */
static double round_store(double x, int store) {
    if (store == 1) return round_bf16(x);
    if (store == 2) return (double)(float)x;
    return x;
}

double oracle_round_bf16(double x) { return round_bf16(x); }

/* Exposed so tests can pin the rotation itself (norm, composition, D=2 closed form). */
void oracle_rope(int D, double base, double pos, const double *x_in, double *x_out) {
    memcpy(x_out, x_in, sizeof(double) * (size_t)D);
    rope_rotate(x_out, D, pos, base);
}

/* Softmax attention of one query vector over n keys already materialised in `kt` (n x D). */
static void attend_one(int D, double scale, int n, const double *kt, const double *v,
                       const int64_t *key_pos, const uint8_t *key_causal, const double *qt,
                       int64_t m, double *s_buf, double *out, double *lse) {
    double mx = -INFINITY;
    for (int k = 0; k < n; ++k) {
        if (key_causal[k] && key_pos[k] > m) { s_buf[k] = -INFINITY; continue; }
        double acc = 0.0;
        const double *kk = kt + (size_t)k * D;
        for (int d = 0; d < D; ++d) acc += qt[d] * kk[d];
        s_buf[k] = acc * scale;
        if (s_buf[k] > mx) mx = s_buf[k];
    }
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (mx == -INFINITY) { *lse = -INFINITY; return; }
    double l = 0.0;
    for (int k = 0; k < n; ++k) {
        if (s_buf[k] == -INFINITY) continue;
        double w = exp(s_buf[k] - mx);
        l += w;
        const double *vv = v + (size_t)k * D;
        for (int d = 0; d < D; ++d) out[d] += w * vv[d];
    }
    for (int d = 0; d < D; ++d) out[d] /= l;
    *lse = mx + log(l);
}

typedef struct {
    int D, G, n_keys, n_q, tid, nt;
    double base, scale;
    const double *k_raw, *v, *q;
    const int64_t *key_pos, *q_pos;
    const uint8_t *key_causal;
    double *kt, *out, *lse;
    int phase;
    /* form S only (key_off == NULL for form A) */
    const int64_t *key_off, *key_local;
    const uint8_t *key_stored;
    int store;
} job_t;

static void *worker(void *arg) {
    job_t *j = (job_t *)arg;
    if (j->phase == 0) {
        /* materialise every key at its absolute logical position */
        for (int k = j->tid; k < j->n_keys; k += j->nt) {
            double *dst = j->kt + (size_t)k * j->D;
            memcpy(dst, j->k_raw + (size_t)k * j->D, sizeof(double) * (size_t)j->D);
            if (j->key_off && j->key_stored[k]) {
                /* form S: the cache's copy R(j) k in its element type, then the offset */
                rope_rotate(dst, j->D, (double)j->key_local[k], j->base);
                for (int d = 0; d < j->D; ++d) dst[d] = round_store(dst[d], j->store);
                rope_rotate(dst, j->D, (double)j->key_off[k], j->base);
            } else {
                rope_rotate(dst, j->D, (double)j->key_pos[k], j->base);
            }
        }
        return NULL;
    }
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)(j->n_keys > 0 ? j->n_keys : 1));
    double *qt = (double *)malloc(sizeof(double) * (size_t)j->D);
    int items = j->n_q * j->G;
    for (int it = j->tid; it < items; it += j->nt) {
        int i = it / j->G, g = it % j->G;
        memcpy(qt, j->q + ((size_t)i * j->G + g) * j->D, sizeof(double) * (size_t)j->D);
        rope_rotate(qt, j->D, (double)j->q_pos[i], j->base);
        attend_one(j->D, j->scale, j->n_keys, j->kt, j->v, j->key_pos, j->key_causal, qt,
                   j->q_pos[i], s_buf, j->out + ((size_t)i * j->G + g) * j->D,
                   j->lse + (size_t)i * j->G + g);
    }
    free(s_buf);
    free(qt);
    return NULL;
}

/* Materialises every key (phase 0), then attends every (query, head) (phase 1), threaded. */
static int run_jobs(int D, int G, double base, double scale, int n_keys, const double *k_raw,
                    const double *v, const int64_t *key_pos, const uint8_t *key_causal, int n_q,
                    const double *q, const int64_t *q_pos, double *out, double *lse,
                    int n_threads, const int64_t *key_off, const int64_t *key_local,
                    const uint8_t *key_stored, int store) {
    if (D < 2 || (D & 1) || G < 1 || n_keys < 0 || n_q < 0) return -1;
    if (n_threads < 1) n_threads = 1;
    double *kt = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1) * (size_t)D);
    if (!kt) return -1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)n_threads);
    for (int phase = 0; phase < 2; ++phase) {
        for (int t = 0; t < n_threads; ++t) {
            job_t jb = {D, G, n_keys, n_q, t, n_threads, base, scale, k_raw, v, q, key_pos, q_pos,
                        key_causal, kt, out, lse, phase, key_off, key_local, key_stored, store};
            jobs[t] = jb;
            pthread_create(&th[t], NULL, worker, &jobs[t]);
        }
        for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
    }
    free(jobs);
    free(th);
    free(kt);
    return 0;
}

/*
 * Form A for one kv head and its G query heads.
 *   k_raw, v : [n_keys][D]   raw (unrotated) keys and values
 *   key_pos  : [n_keys]      absolute logical position of each key
 *   key_causal:[n_keys]      1 = visible only to queries at m >= key_pos
 *   q        : [n_q][G][D]   raw queries;  q_pos: [n_q] their logical positions
 *   out      : [n_q][G][D];  lse: [n_q][G]  (natural log of the scaled scores' exp-sum)
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attend_materialised(int D, int G, double base, double scale, int n_keys,
                               const double *k_raw, const double *v, const int64_t *key_pos,
                               const uint8_t *key_causal, int n_q, const double *q,
                               const int64_t *q_pos, double *out, double *lse, int n_threads) {
    return run_jobs(D, G, base, scale, n_keys, k_raw, v, key_pos, key_causal, n_q, q, q_pos, out,
                    lse, n_threads, NULL, NULL, NULL, 0);
}

/*
 * Form S for one kv head: as form A, except that a key with key_stored[k] = 1 is the cache's
 * copy round(R(key_local[k]) k_raw[k]) (store: 0 = exact, 1 = bfloat16, 2 = float32), attended
 * at offset key_off[k], i.e. rotated by R(key_off[k]) in fp64 before the dot product. Keys with
 * key_stored[k] = 0 enter as R(key_off[k] + key_local[k]) k_raw[k]. Causal visibility uses the
 * absolute position key_off + key_local.
 */
int oracle_attend_stored(int D, int G, double base, double scale, int n_keys, const double *k_raw,
                         const double *v, const int64_t *key_off, const int64_t *key_local,
                         const uint8_t *key_stored, const uint8_t *key_causal, int n_q,
                         const double *q, const int64_t *q_pos, int store, double *out,
                         double *lse, int n_threads) {
    if (store < 0 || store > 2 || n_keys < 0) return -1;
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_keys > 0 ? n_keys : 1));
    if (!pos) return -1;
    for (int k = 0; k < n_keys; ++k) pos[k] = key_off[k] + key_local[k];
    int rc = run_jobs(D, G, base, scale, n_keys, k_raw, v, pos, key_causal, n_q, q, q_pos, out, lse,
                      n_threads, key_off, key_local, key_stored, store);
    free(pos);
    return rc;
}

/*
 * Form B (the lazy form) for one kv head: key k is stored at document-local position
 * key_local[k] and attended at offset key_off[k]; its absolute position is off + local.
 * The query is rotated by the relative offset m - off, the key by its local position.
 * Single-threaded and O(n_q * G * n_keys * D) trig: small cases only.
 */
int oracle_attend_lazy(int D, int G, double base, double scale, int n_keys, const double *k_raw,
                       const double *v, const int64_t *key_off, const int64_t *key_local,
                       const uint8_t *key_causal, int n_q, const double *q, const int64_t *q_pos,
                       double *out, double *lse) {
    if (D < 2 || (D & 1) || G < 1 || n_keys < 0 || n_q < 0) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
    double *qr = (double *)malloc(sizeof(double) * (size_t)D);
    double *kr = (double *)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < n_q; ++i) {
        for (int g = 0; g < G; ++g) {
            const double *qq = q + ((size_t)i * G + g) * D;
            double mx = -INFINITY;
            for (int k = 0; k < n_keys; ++k) {
                int64_t p = key_off[k] + key_local[k];
                if (key_causal[k] && p > q_pos[i]) { s[k] = -INFINITY; continue; }
                memcpy(qr, qq, sizeof(double) * (size_t)D);
                rope_rotate(qr, D, (double)(q_pos[i] - key_off[k]), base);
                memcpy(kr, k_raw + (size_t)k * D, sizeof(double) * (size_t)D);
                rope_rotate(kr, D, (double)key_local[k], base);
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += qr[d] * kr[d];
                s[k] = acc * scale;
                if (s[k] > mx) mx = s[k];
            }
            double *o = out + ((size_t)i * G + g) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (mx == -INFINITY) { lse[(size_t)i * G + g] = -INFINITY; continue; }
            double l = 0.0;
            for (int k = 0; k < n_keys; ++k) {
                if (s[k] == -INFINITY) continue;
                double w = exp(s[k] - mx);
                l += w;
                for (int d = 0; d < D; ++d) o[d] += w * v[(size_t)k * D + d];
            }
            for (int d = 0; d < D; ++d) o[d] /= l;
            lse[(size_t)i * G + g] = mx + log(l);
        }
    }
    free(s);
    free(qr);
    free(kr);
    return 0;
}
