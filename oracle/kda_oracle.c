/*
 * kda_oracle.c -- fp64 CPU oracle for the Kimi Delta Attention (KDA) token mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker that the
 * CUDA library is compared against.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or constant with the CUDA path and includes nothing from it.
 *
 * Two functions are exported (plain C ABI, host pointers, row-major, fp64):
 *
 *   kda_oracle_recurrent  -- the defining token-by-token recurrence.
 *   kda_oracle_chunkwise  -- the chunkwise schedule of the same recurrence,
 *                            written step by step as the derivation gives it
 *                            (provisional errors, causal key-key system solved
 *                            by forward substitution, state fast-forward,
 *                            causal outputs).  It exists so that a test can
 *                            check the chunk algebra against the recurrence
 *                            by brute force.
 *
 * Sources (pages on Kimi Delta Attention):
 *   "Kimi Unveils Delta Attention and K3 Architecture Updates"
 *       sec. 4 (KDA: forget, predict, correct, write, read), the five-line
 *       recurrence in the d_k x d_v layout at the end of sec. 4.1, and
 *       sec. 6.1-6.5 (chunkwise KDA).
 *   "Kimi Delta Attention: Channel-Wise Memory Control"
 *       sec. "Change one piece of Gated DeltaNet" (key-by-value state, rows
 *       decayed by left multiplication, o_t = S_t^T q_t) and
 *       "The core update in a few lines".
 *   "Linear Attention, From Scratch to Kimi 3" sec. 9 (cu_seqlens: packed
 *       requests whose state never crosses a boundary).
 *
 * Conventions.  State S is d_k x d_v per (sequence, head), row i = key
 * channel i, stored row-major (d_v contiguous).  log_alpha holds g = log(alpha)
 * per (token, head, key channel); beta one write strength per (token, head).
 * The read is taken after the write, and the query is multiplied by `scale`.
 *
 * parity pins: every function here is pinned by the "not gpu" tests (worked
 * examples printed on the pages, closed forms, reductions to DeltaNet and
 * Gated DeltaNet written independently, and brute-force agreement of the two
 * schedules).
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t num_seqs, total_tokens, num_heads, d_k, d_v;
    const double *q, *k, *v, *log_alpha, *beta;
    double scale;
    const double *initial_state;
    const int32_t *cu_seqlens;
    double *out, *final_state;
    int32_t chunk_size; /* 0 = token recurrence */
    atomic_int next_item;
    atomic_int failed;
} job_t;

/* ------------------------------------------------------------------------ */
/* One (sequence, head) pair, token by token.                                */
/* "Kimi Unveils Delta Attention ...", sec. 4: forget each key channel,      */
/* predict from the forgotten state, correct, write, then read.              */
/* ------------------------------------------------------------------------ */
static void recurrent_pair(const job_t *J, int32_t seq, int32_t h, double *S,
                           double *p) {
    const int32_t H = J->num_heads, dk = J->d_k, dv = J->d_v;
    const int32_t t_begin = J->cu_seqlens[seq], t_end = J->cu_seqlens[seq + 1];

    for (int32_t t = t_begin; t < t_end; ++t) {
        const double *q = J->q + ((size_t)t * H + h) * dk;
        const double *k = J->k + ((size_t)t * H + h) * dk;
        const double *v = J->v + ((size_t)t * H + h) * dv;
        const double *g = J->log_alpha + ((size_t)t * H + h) * dk;
        const double beta = J->beta[(size_t)t * H + h];
        double *o = J->out + ((size_t)t * H + h) * dv;

        /* forget: S_bar = Diag(alpha_t) S_{t-1}  (row i scaled by exp(g_i)) */
        for (int32_t i = 0; i < dk; ++i) {
            const double a = exp(g[i]);
            for (int32_t j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a;
        }
        /* predict: p = S_bar^T k */
        for (int32_t j = 0; j < dv; ++j) p[j] = 0.0;
        for (int32_t i = 0; i < dk; ++i)
            for (int32_t j = 0; j < dv; ++j) p[j] += S[(size_t)i * dv + j] * k[i];
        /* correct: e = beta (v - p) */
        for (int32_t j = 0; j < dv; ++j) p[j] = beta * (v[j] - p[j]);
        /* write: S_t = S_bar + k e^T */
        for (int32_t i = 0; i < dk; ++i)
            for (int32_t j = 0; j < dv; ++j) S[(size_t)i * dv + j] += k[i] * p[j];
        /* read after the write: o_t = S_t^T (scale q_t) */
        for (int32_t j = 0; j < dv; ++j) o[j] = 0.0;
        for (int32_t i = 0; i < dk; ++i) {
            const double sq = J->scale * q[i];
            for (int32_t j = 0; j < dv; ++j) o[j] += S[(size_t)i * dv + j] * sq;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* One (sequence, head) pair, chunk by chunk.                                */
/* "Kimi Unveils Delta Attention ...", sec. 6.1-6.5, in the d_k x d_v layout */
/* (the page writes the d_v x d_k transpose; every product below is the      */
/* transpose of the page's, which leaves the numbers unchanged).             */
/* ------------------------------------------------------------------------ */
typedef struct {
    double *G;    /* [C][dk] chunk-local cumulative log decay              */
    double *E;    /* [C][dv] errors (provisional, then resolved in place)  */
    double *tmp;  /* [dk]                                                   */
} chunk_ws_t;

static void chunkwise_pair(const job_t *J, int32_t seq, int32_t h, double *S,
                           chunk_ws_t *ws) {
    const int32_t H = J->num_heads, dk = J->d_k, dv = J->d_v, C = J->chunk_size;
    const int32_t t_begin = J->cu_seqlens[seq], t_end = J->cu_seqlens[seq + 1];
    double *G = ws->G, *E = ws->E, *x = ws->tmp;

#define Q_(t) (J->q + ((size_t)(t) * H + h) * dk)
#define K_(t) (J->k + ((size_t)(t) * H + h) * dk)
#define V_(t) (J->v + ((size_t)(t) * H + h) * dv)
#define G_(t) (J->log_alpha + ((size_t)(t) * H + h) * dk)
#define B_(t) (J->beta[(size_t)(t) * H + h])
#define O_(t) (J->out + ((size_t)(t) * H + h) * dv)

    for (int32_t c0 = t_begin; c0 < t_end; c0 += C) {
        const int32_t L = (t_end - c0 < C) ? (t_end - c0) : C;

        /* sec. 6.1: cumulative decay from the chunk boundary through token i,
           G_i = sum_{r<=i} g_r, so D_{0:i} = Diag(exp(G_i)) and the decay
           carrying a write at j to token i is Diag(exp(G_i - G_j)). */
        for (int32_t i = 0; i < L; ++i)
            for (int32_t d = 0; d < dk; ++d)
                G[(size_t)i * dk + d] =
                    (i ? G[(size_t)(i - 1) * dk + d] : 0.0) + G_(c0 + i)[d];

        /* sec. 6.2: provisional errors against the decayed incoming state,
           e_bar_i = beta_i (v_i - S_c^T (exp(G_i) * k_i)). */
        for (int32_t i = 0; i < L; ++i) {
            for (int32_t d = 0; d < dk; ++d)
                x[d] = exp(G[(size_t)i * dk + d]) * K_(c0 + i)[d];
            for (int32_t j = 0; j < dv; ++j) {
                double pred = 0.0;
                for (int32_t d = 0; d < dk; ++d) pred += S[(size_t)d * dv + j] * x[d];
                E[(size_t)i * dv + j] = B_(c0 + i) * (V_(c0 + i)[j] - pred);
            }
        }

        /* sec. 6.3: restore the causal dependencies.  With
           rho_ij = beta_i <k_j| D_{j+1:i} |k_i>  (j < i),
           e_i = e_bar_i - sum_{j<i} rho_ij e_j, i.e. the unit lower
           triangular system (I + R) E = E_bar solved by forward substitution. */
        for (int32_t i = 1; i < L; ++i) {
            for (int32_t j = 0; j < i; ++j) {
                double dot = 0.0;
                for (int32_t d = 0; d < dk; ++d)
                    dot += K_(c0 + j)[d] *
                           exp(G[(size_t)i * dk + d] - G[(size_t)j * dk + d]) *
                           K_(c0 + i)[d];
                const double rho = B_(c0 + i) * dot;
                for (int32_t m = 0; m < dv; ++m)
                    E[(size_t)i * dv + m] -= rho * E[(size_t)j * dv + m];
            }
        }

        /* sec. 6.5: outputs read the state after their own write,
           o_i = s S_c^T (exp(G_i) q_i) + sum_{j<=i} chi_ij e_j,
           chi_ij = s <k_j| D_{j+1:i} |q_i>. */
        for (int32_t i = 0; i < L; ++i) {
            double *o = O_(c0 + i);
            for (int32_t d = 0; d < dk; ++d)
                x[d] = J->scale * exp(G[(size_t)i * dk + d]) * Q_(c0 + i)[d];
            for (int32_t m = 0; m < dv; ++m) {
                double acc = 0.0;
                for (int32_t d = 0; d < dk; ++d) acc += S[(size_t)d * dv + m] * x[d];
                o[m] = acc;
            }
            for (int32_t j = 0; j <= i; ++j) {
                double dot = 0.0;
                for (int32_t d = 0; d < dk; ++d)
                    dot += K_(c0 + j)[d] *
                           exp(G[(size_t)i * dk + d] - G[(size_t)j * dk + d]) *
                           Q_(c0 + i)[d];
                const double chi = J->scale * dot;
                for (int32_t m = 0; m < dv; ++m) o[m] += chi * E[(size_t)j * dv + m];
            }
        }

        /* sec. 6.4: fast-forward the state by the whole chunk,
           S_{c+1} = D_{0:L-1} S_c + sum_i (exp(G_{L-1} - G_i) k_i) e_i^T. */
        const double *Gl = G + (size_t)(L - 1) * dk;
        for (int32_t d = 0; d < dk; ++d) {
            const double a = exp(Gl[d]);
            for (int32_t m = 0; m < dv; ++m) S[(size_t)d * dv + m] *= a;
        }
        for (int32_t i = 0; i < L; ++i) {
            for (int32_t d = 0; d < dk; ++d) {
                const double kend = exp(Gl[d] - G[(size_t)i * dk + d]) * K_(c0 + i)[d];
                for (int32_t m = 0; m < dv; ++m)
                    S[(size_t)d * dv + m] += kend * E[(size_t)i * dv + m];
            }
        }
    }
#undef Q_
#undef K_
#undef V_
#undef G_
#undef B_
#undef O_
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    const size_t SS = (size_t)J->d_k * J->d_v;
    double *S = (double *)malloc(SS * sizeof(double));
    double *p = (double *)malloc((size_t)J->d_v * sizeof(double));
    chunk_ws_t ws = {0, 0, 0};
    if (J->chunk_size > 0) {
        ws.G = (double *)malloc((size_t)J->chunk_size * J->d_k * sizeof(double));
        ws.E = (double *)malloc((size_t)J->chunk_size * J->d_v * sizeof(double));
        ws.tmp = (double *)malloc((size_t)J->d_k * sizeof(double));
    }
    if (!S || !p || (J->chunk_size > 0 && (!ws.G || !ws.E || !ws.tmp))) {
        atomic_store(&J->failed, 1);
        free(S); free(p); free(ws.G); free(ws.E); free(ws.tmp);
        return NULL;
    }
    const int32_t n_items = J->num_seqs * J->num_heads;
    for (;;) {
        const int32_t item = atomic_fetch_add(&J->next_item, 1);
        if (item >= n_items) break;
        const int32_t seq = item / J->num_heads, h = item % J->num_heads;
        const size_t off = ((size_t)seq * J->num_heads + h) * SS;
        if (J->initial_state)
            memcpy(S, J->initial_state + off, SS * sizeof(double));
        else
            memset(S, 0, SS * sizeof(double));
        if (J->chunk_size > 0)
            chunkwise_pair(J, seq, h, S, &ws);
        else
            recurrent_pair(J, seq, h, S, p);
        if (J->final_state) memcpy(J->final_state + off, S, SS * sizeof(double));
    }
    free(S); free(p); free(ws.G); free(ws.E); free(ws.tmp);
    return NULL;
}

static int run(job_t *J, int32_t num_threads) {
    if (J->num_seqs < 0 || J->num_heads <= 0 || J->d_k <= 0 || J->d_v <= 0 ||
        J->total_tokens < 0 || !J->cu_seqlens)
        return 1;
    if (J->total_tokens > 0 && (!J->q || !J->k || !J->v || !J->log_alpha ||
                                !J->beta || !J->out))
        return 1;
    if (J->cu_seqlens[0] != 0 || J->cu_seqlens[J->num_seqs] != J->total_tokens)
        return 1;
    for (int32_t s = 0; s < J->num_seqs; ++s)
        if (J->cu_seqlens[s + 1] < J->cu_seqlens[s]) return 1;
    atomic_init(&J->next_item, 0);
    atomic_init(&J->failed, 0);
    const int32_t n_items = J->num_seqs * J->num_heads;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > n_items) num_threads = n_items > 0 ? n_items : 1;
    pthread_t *th = (pthread_t *)malloc((size_t)num_threads * sizeof(pthread_t));
    if (!th) return 2;
    int32_t started = 0;
    for (int32_t i = 1; i < num_threads; ++i) {
        if (pthread_create(&th[i], NULL, worker, J) != 0) break;
        ++started;
    }
    worker(J);
    for (int32_t i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    free(th);
    return atomic_load(&J->failed) ? 2 : 0;
}

/* Token-by-token recurrence over packed sequences.  Returns 0 on success,
   1 on an invalid argument, 2 when host memory runs out. */
int kda_oracle_recurrent(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                         int32_t d_k, int32_t d_v, const double *q, const double *k,
                         const double *v, const double *log_alpha, const double *beta,
                         double scale, const double *initial_state,
                         const int32_t *cu_seqlens, double *out, double *final_state,
                         int32_t num_threads) {
    job_t J;
    memset(&J, 0, sizeof(J));
    J.num_seqs = num_seqs; J.total_tokens = total_tokens; J.num_heads = num_heads;
    J.d_k = d_k; J.d_v = d_v; J.q = q; J.k = k; J.v = v; J.log_alpha = log_alpha;
    J.beta = beta; J.scale = scale; J.initial_state = initial_state;
    J.cu_seqlens = cu_seqlens; J.out = out; J.final_state = final_state;
    J.chunk_size = 0;
    return run(&J, num_threads);
}

/* Chunkwise schedule of the same recurrence, chunks of `chunk_size` tokens
   restarting at every sequence start (the last chunk of a sequence may be
   shorter).  Same arguments and return codes. */
int kda_oracle_chunkwise(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                         int32_t d_k, int32_t d_v, const double *q, const double *k,
                         const double *v, const double *log_alpha, const double *beta,
                         double scale, const double *initial_state,
                         const int32_t *cu_seqlens, double *out, double *final_state,
                         int32_t chunk_size, int32_t num_threads) {
    if (chunk_size < 1) return 1;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.num_seqs = num_seqs; J.total_tokens = total_tokens; J.num_heads = num_heads;
    J.d_k = d_k; J.d_v = d_v; J.q = q; J.k = k; J.v = v; J.log_alpha = log_alpha;
    J.beta = beta; J.scale = scale; J.initial_state = initial_state;
    J.cu_seqlens = cu_seqlens; J.out = out; J.final_state = final_state;
    J.chunk_size = chunk_size;
    return run(&J, num_threads);
}
