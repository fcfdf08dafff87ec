/*
 * ssm_oracle.c -- plain CPU oracle of the Mamba2 selective-state scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * bench's CPU-baseline leg may load this library.  It shares no code, header or
 * constant with the CUDA path.
 *
 * What it computes (the recurrence itself, in double precision):
 *   for every sequence i, head h (group g = h / (H/G)), head-dim row p and
 *   token t of the sequence, in token order:
 *     a          = exp(dt[t,h] * A[h])
 *     S[h,p,n]   = a * S[h,p,n] + dt[t,h] * x[t,h,p] * B[t,g,n]      (n < N)
 *     y[t,h,p]   = sum_n S[h,p,n] * C[t,g,n] + D[h] * x[t,h,p]
 *   S starts from slot i when resume[i] is nonzero, else from zero, and the
 *   state after the last token is the new slot i.
 *
 * Sources:
 *   - "The llama journey", Day 14 (the rewritten ssm_scan_f32_group kernel
 *     body): per-token state update with the decay exp(dt*A) of a per-head
 *     scalar A, the x*dt input term, then a dot product with C over the state
 *     for y, using the state that already includes token t.
 *   - "The llama journey", Day 12 (the CPU reference ggml_compute_forward_ssm_scan_f32):
 *     loop order sequence -> token -> head -> row -> state element, and the
 *     tensor table (state [n_seq][n_head][dim][d_state], B/C per group).
 *   - The same kernel's group map: heads are split into G contiguous blocks,
 *     group = head / (H / G).
 *   - "keep the Mamba2 scan state in registers" (gllm PR 90), "What changes":
 *     the per-sequence state slot persists between calls; fresh and resuming
 *     sequences are mixed in one batch.
 *   - The skip term D[h] * x[t,h,p] (absent from the ggml kernel) is part of the
 *     scan definition this library implements; it is added after the dot
 *     product.
 *
 * Readings where the sources leave a step open:
 *   - dt is used as given (no softplus, no bias, no positivity check).
 *   - A zero-length sequence writes no y; a fresh one still zeroes its slot,
 *     a resuming one leaves it unchanged (as copied from state_in).
 *
 * No blocking, fusion or reordering: each (sequence, head) unit runs the loops
 * above in the stated order.  Units are independent, so the only parallelism is
 * running whole units on different threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *state_in;
    double *state_out;
    const double *x, *dt, *A, *B, *C, *D;
    double *y;
    const int32_t *seq_starts, *seq_lens, *resume;
    const uint8_t *head_sel;
    int n_seqs, H, P, N, G;
    long next_unit;        /* shared work counter, guarded by lock */
    pthread_mutex_t lock;
} oracle_job;

/* One (sequence i, head h) unit: the recurrence over the sequence's tokens. */
static void scan_unit(const oracle_job *J, int i, int h)
{
    const int H = J->H, P = J->P, N = J->N, G = J->G;
    const int g = h / (H / G);
    const size_t slot = ((size_t)i * H + h) * (size_t)P * N;
    double *S = J->state_out + slot;

    for (size_t e = 0; e < (size_t)P * N; ++e)
        S[e] = J->resume[i] ? J->state_in[slot + e] : 0.0;

    const long t0 = J->seq_starts[i];
    const long t1 = t0 + J->seq_lens[i];
    for (long t = t0; t < t1; ++t) {
        const double dt_th = J->dt[t * H + h];
        const double a = exp(dt_th * J->A[h]);
        const double *Bt = J->B + ((size_t)t * G + g) * N;
        const double *Ct = J->C + ((size_t)t * G + g) * N;
        for (int p = 0; p < P; ++p) {
            const double x_thp = J->x[((size_t)t * H + h) * P + p];
            const double xdt = dt_th * x_thp;
            double *Sp = S + (size_t)p * N;
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                Sp[n] = a * Sp[n] + xdt * Bt[n];
                acc += Sp[n] * Ct[n];
            }
            J->y[((size_t)t * H + h) * P + p] = acc + J->D[h] * x_thp;
        }
    }
}

static void *worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    const long n_units = (long)J->n_seqs * J->H;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        long u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= n_units)
            break;
        const int i = (int)(u / J->H), h = (int)(u % J->H);
        if (J->head_sel && !J->head_sel[h])
            continue;
        scan_unit(J, i, h);
    }
    return NULL;
}

/*
 * Run the scan.  All arrays are host memory in the layouts of the header
 * comment; state_in is read only for resuming sequences.  head_sel (may be
 * NULL) restricts the work to the heads with a nonzero entry; outputs of the
 * other heads are left untouched.  Returns 0, or -1 on an invalid argument.
 */
int ssm_oracle_scan(const double *state_in, double *state_out,
                    const double *x, const double *dt, const double *A,
                    const double *B, const double *C, const double *D,
                    double *y,
                    const int32_t *seq_starts, const int32_t *seq_lens,
                    const int32_t *resume, const uint8_t *head_sel,
                    int n_seqs, long n_tokens, int H, int P, int N, int G,
                    int n_threads)
{
    if (n_seqs < 0 || n_tokens < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0)
        return -1;
    for (int i = 0; i < n_seqs; ++i) {
        if (seq_lens[i] < 0 || seq_starts[i] < 0 ||
            (long)seq_starts[i] + seq_lens[i] > n_tokens)
            return -1;
    }
    oracle_job J;
    memset(&J, 0, sizeof J);
    J.state_in = state_in; J.state_out = state_out;
    J.x = x; J.dt = dt; J.A = A; J.B = B; J.C = C; J.D = D; J.y = y;
    J.seq_starts = seq_starts; J.seq_lens = seq_lens; J.resume = resume;
    J.head_sel = head_sel;
    J.n_seqs = n_seqs; J.H = H; J.P = P; J.N = N; J.G = G;
    J.next_unit = 0;
    pthread_mutex_init(&J.lock, NULL);

    if (n_threads <= 1) {
        worker(&J);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
        if (!th) {
            pthread_mutex_destroy(&J.lock);
            return -1;
        }
        int started = 0;
        for (int k = 0; k < n_threads; ++k)
            if (pthread_create(&th[k], NULL, worker, &J) == 0)
                ++started;
            else
                break;
        if (started == 0)
            worker(&J);
        for (int k = 0; k < started; ++k)
            pthread_join(th[k], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J.lock);
    return 0;
}
