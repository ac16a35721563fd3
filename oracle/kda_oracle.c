/*
 * kda_oracle.c -- plain fp64 CPU oracle for the KDA (gated delta rule with a
 * per-channel decay gate) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this file; only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header or constant with the CUDA path.
 *
 * What it computes (per v-head h of sequence n, token by token, in the order
 * the sequence is packed):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * i.e. the state is first decayed row-wise by exp(g_t) and then receives the
 * delta-rule write.  The recurrence itself is the one the KDA prefill pages
 * describe by its chunked form (sglang PR 27488 digest "KDA SM100 CuteDSL
 * prefill", section 实现拆解 / implementation breakdown, item 1; and section
 * 关键源码片段, kernel_kkt_inv_uw.py, whose operand KG = k * exp(g_cu) is only
 * consistent with an inclusive cumulative gate, i.e. decay-then-update).
 *
 * State pool semantics follow sglang PR 30169 digest "pool state I/O fused into
 * the h kernel", section 实现拆解 items 1-3: with per-sequence slot indices the
 * state array is a pool read and written in place; index -1 (padding) maps to
 * the last slot (the sentinel).  Without indices the initial state is dense
 * [N,Hv,K,V] and a new dense final state is produced.
 *
 * Layouts (all row-major, fp64):
 *   q, k        [T, Hk, K]
 *   v           [T, Hv, V]
 *   g           [T, Hv, K]   natural-log decay per key channel
 *   beta        [T, Hv]
 *   cu_seqlens  [N+1]        int32 prefix offsets of the packed sequences
 *   state       [N or num_slots, Hv, K, V]   S[k][v]
 *   o           [T, Hv, V]
 * v-head h reads k/q head kh = h / (Hv / Hk) (contiguous groups).
 *
 * Sums over channels run in ascending channel order in fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int num_seqs, Hk, Hv, K, V;
    double scale;
    const double *q, *k, *v, *g, *beta;
    const int *cu_seqlens;
    const double *init;  /* [N,Hv,K,V] gathered initial states or NULL (zeros) */
    double *final_;      /* [N,Hv,K,V] final states */
    double *o;
    long next_item;      /* shared work counter (guarded by mu) */
    long num_items;
    pthread_mutex_t mu;
} job_t;

/* One (sequence, v-head) pair: the token-by-token recurrence. */
static void run_item(const job_t *J, long item, double *S, double *w) {
    const int n = (int)(item / J->Hv), h = (int)(item % J->Hv);
    const int K = J->K, V = J->V, Hk = J->Hk, Hv = J->Hv;
    const int kh = h / (Hv / Hk);
    const size_t sKV = (size_t)K * V;
    const size_t state_off = ((size_t)n * Hv + h) * sKV;

    if (J->init)
        memcpy(S, J->init + state_off, sKV * sizeof(double));
    else
        memset(S, 0, sKV * sizeof(double));

    for (long t = J->cu_seqlens[n]; t < J->cu_seqlens[n + 1]; ++t) {
        const double *qt = J->q + ((size_t)t * Hk + kh) * K;
        const double *kt = J->k + ((size_t)t * Hk + kh) * K;
        const double *vt = J->v + ((size_t)t * Hv + h) * V;
        const double *gt = J->g + ((size_t)t * Hv + h) * K;
        const double bt = J->beta[(size_t)t * Hv + h];
        double *ot = J->o + ((size_t)t * Hv + h) * V;

        /* decay: S <- Diag(exp g_t) S */
        for (int c = 0; c < K; ++c) {
            const double d = exp(gt[c]);
            double *row = S + (size_t)c * V;
            for (int j = 0; j < V; ++j) row[j] *= d;
        }
        /* w = S^T k_t ; u = beta (v - w) */
        for (int j = 0; j < V; ++j) w[j] = 0.0;
        for (int c = 0; c < K; ++c) {
            const double kc = kt[c];
            const double *row = S + (size_t)c * V;
            for (int j = 0; j < V; ++j) w[j] += kc * row[j];
        }
        for (int j = 0; j < V; ++j) w[j] = bt * (vt[j] - w[j]);
        /* S <- S + k_t u^T */
        for (int c = 0; c < K; ++c) {
            const double kc = kt[c];
            double *row = S + (size_t)c * V;
            for (int j = 0; j < V; ++j) row[j] += kc * w[j];
        }
        /* o_t = scale S^T q_t */
        for (int j = 0; j < V; ++j) ot[j] = 0.0;
        for (int c = 0; c < K; ++c) {
            const double qc = qt[c];
            const double *row = S + (size_t)c * V;
            for (int j = 0; j < V; ++j) ot[j] += qc * row[j];
        }
        for (int j = 0; j < V; ++j) ot[j] *= J->scale;
    }
    memcpy(J->final_ + state_off, S, sKV * sizeof(double));
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc((size_t)J->K * J->V * sizeof(double));
    double *w = (double *)malloc((size_t)J->V * sizeof(double));
    if (!S || !w) { free(S); free(w); return (void *)1; }
    for (;;) {
        pthread_mutex_lock(&J->mu);
        long item = J->next_item++;
        pthread_mutex_unlock(&J->mu);
        if (item >= J->num_items) break;
        run_item(J, item, S, w);
    }
    free(S);
    free(w);
    return NULL;
}

/*
 * Returns 0 on success, -1 on an invalid argument (including a slot index
 * outside [-1, num_slots)), -2 on allocation failure.
 *
 * state_in:  dense h0 [N,Hv,K,V] (indices NULL), pool [num_slots,Hv,K,V]
 *            (indices given) or NULL (zero initial state).
 * state_out: dense ht [N,Hv,K,V] (indices NULL; may be NULL) or the updated
 *            pool [num_slots,Hv,K,V] (indices given).  In pool mode every
 *            sequence starts from the pool as it was before the call; final
 *            states are written back in sequence order, and rows that no index
 *            names are copied unchanged.  state_out may alias state_in.
 * nthreads:  worker threads; <= 0 means one per online core.
 */
int kda_oracle_recurrence(int num_seqs, int Hk, int Hv, int K, int V, double scale,
                          const double *q, const double *k, const double *v,
                          const double *g, const double *beta, const int *cu_seqlens,
                          const double *state_in, const int *state_indices,
                          long long num_slots, double *o, double *state_out,
                          int nthreads) {
    if (num_seqs < 0 || Hk <= 0 || Hv <= 0 || K <= 0 || V <= 0 || Hv % Hk != 0)
        return -1;
    if (!cu_seqlens || (num_seqs > 0 && (!q || !k || !v || !g || !beta || !o)))
        return -1;
    if (cu_seqlens[0] != 0) return -1;
    for (int n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    if (state_indices) {
        if (!state_in || !state_out || num_slots <= 0) return -1;
        for (int n = 0; n < num_seqs; ++n)
            if (state_indices[n] < -1 || state_indices[n] >= num_slots) return -1;
    }

    const size_t sKV = (size_t)K * V;
    const size_t per_seq = (size_t)Hv * sKV;
    double *init = NULL, *fin = (double *)malloc((num_seqs ? num_seqs : 1) * per_seq * sizeof(double));
    if (!fin) return -2;
    if (state_in) {
        init = (double *)malloc((num_seqs ? num_seqs : 1) * per_seq * sizeof(double));
        if (!init) { free(fin); return -2; }
        for (int n = 0; n < num_seqs; ++n) {
            long long slot = n;
            if (state_indices) slot = state_indices[n] < 0 ? num_slots - 1 : state_indices[n];
            memcpy(init + (size_t)n * per_seq, state_in + (size_t)slot * per_seq,
                   per_seq * sizeof(double));
        }
    }

    job_t J;
    J.num_seqs = num_seqs; J.Hk = Hk; J.Hv = Hv; J.K = K; J.V = V; J.scale = scale;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.cu_seqlens = cu_seqlens;
    J.init = init; J.final_ = fin; J.o = o;
    J.next_item = 0; J.num_items = (long)num_seqs * Hv;
    pthread_mutex_init(&J.mu, NULL);

    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > J.num_items) nthreads = J.num_items > 0 ? (int)J.num_items : 1;
    pthread_t *tid = (pthread_t *)malloc((size_t)nthreads * sizeof(pthread_t));
    int rc = 0;
    if (!tid) rc = -2;
    int started = 0;
    for (int i = 0; rc == 0 && i < nthreads; ++i) {
        if (pthread_create(&tid[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (rc == 0 && started == 0) worker(&J); /* no thread could start: run inline */
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(tid[i], &ret);
        if (ret) rc = -2;
    }
    free(tid);
    pthread_mutex_destroy(&J.mu);

    if (rc == 0 && state_out) {
        if (state_indices) {
            if (state_out != state_in)
                memcpy(state_out, state_in, (size_t)num_slots * per_seq * sizeof(double));
            for (int n = 0; n < num_seqs; ++n) {
                long long slot = state_indices[n] < 0 ? num_slots - 1 : state_indices[n];
                memcpy(state_out + (size_t)slot * per_seq, fin + (size_t)n * per_seq,
                       per_seq * sizeof(double));
            }
        } else {
            memcpy(state_out, fin, (size_t)num_seqs * per_seq * sizeof(double));
        }
    }
    free(init);
    free(fin);
    return rc;
}
