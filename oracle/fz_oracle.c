/*
 * CPU oracle for gapped seed extension -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-threaded C that states what the GPU path must compute.
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * may load it.  It shares no code, header or table with the CUDA library.
 *
 * What is computed (FastZ: Accelerating Gapped Whole Genome Alignment on
 * GPUs, sections 2.1-2.2 and 3.1; the recurrence figure is not in the text, so
 * the form below is read from its prose: I and D each choose between 2 options,
 * S between 3, five adds and four compares per cell):
 *
 *   window: target t[1..m], query q[1..n]; cell (i, j), anti-diagonal d = i + j
 *   S(0,0) = 0, I(0,0) = D(0,0) = NEG
 *   I(i,j) = max(I(i,j-1) - e, S(i,j-1) - o - e)        (consumes q_j, op I)
 *   D(i,j) = max(D(i-1,j) - e, S(i-1,j) - o - e)        (consumes t_i, op D)
 *   S(i,j) = max(S(i-1,j-1) + M[t_i][q_j], I(i,j), D(i,j))
 *   a gap of k bases costs o + k*e.  Missing predecessors (outside the window
 *   or dead) count as NEG.
 *
 * Y-drop (LASTZ ydrop_one_sided_align as FastZ section 3.4 restates it:
 * prune against scores that are already complete).  Anti-diagonals are
 * processed in order d = 0, 1, 2, ...; best_d = max S over live cells on
 * anti-diagonals < d; a computed cell is live iff at least one predecessor is
 * live and S >= best_d - ydrop (a cell with S < best_d - ydrop is pruned).
 * Dead cells hold NEG in S, I and D.  A cell depends on the two previous
 * anti-diagonals, so the sweep stops when two consecutive anti-diagonals hold
 * no live cell (then no later cell can be live).  ydrop < 0: no pruning.
 *
 * Result: (score, i*, j*) = max S over live cells (origin included, so the
 * score is >= 0); ties go to the smallest d, then the smallest i.
 * Traceback from (i*, j*) in state S: diag if S == S(i-1,j-1) + M, else I if
 * S == I, else D; in state I at (i,j): the gap opens here (back to state S at
 * (i,j-1)) if I(i,j) == S(i,j-1) - o - e, else it extends; D likewise.
 *
 * LOCAL mode: S(i,j) = max(0, S(i-1,j-1) + M, I, D), S = 0 and I = D = NEG on
 * row and column 0, no pruning, result = max S with the same tie rule, no
 * CIGAR (the zero-floored cell H of the DPX intrinsics article, section 1.1,
 * with affine gaps).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define NEG (-(1 << 30))

/* one anti-diagonal: cells i = lo..hi stored from pool offset off */
typedef struct {
    int32_t lo, hi;          /* candidate rows computed on this anti-diagonal (hi < lo: none) */
    int32_t live_lo, live_hi;/* live extent (live_hi < live_lo: no live cell) */
    int64_t off;
} diag_rec;

typedef struct {
    int32_t *S, *I, *D;
    uint8_t *alive;
    int64_t used, cap;
    diag_rec *dg;
    int32_t ndg, dg_cap;
} store;

typedef struct {
    int32_t score, i_end, j_end;
    int32_t d_last;          /* last anti-diagonal that held a live cell */
    int64_t live_cells;      /* live cells of the sweep, origin and border included */
    int32_t n_cigar;         /* CIGAR runs written */
    int32_t status;          /* 0 ok, -1 out of memory, -2 CIGAR buffer too small */
    int32_t max_width;       /* diagnostic: widest candidate row range of one anti-diagonal */
    int32_t narrow_steps;    /* diagnostic: anti-diagonals whose candidate range spans <= 160 rows */
} orc_result;

static void store_free(store* st) {
    free(st->S); free(st->I); free(st->D); free(st->alive); free(st->dg);
    memset(st, 0, sizeof(*st));
}

static int store_reserve(store* st, int64_t more) {
    if (st->used + more <= st->cap) return 0;
    int64_t nc = st->cap ? st->cap : 4096;
    while (nc < st->used + more) nc *= 2;
    int32_t* s = (int32_t*)realloc(st->S, (size_t)nc * sizeof(int32_t));
    if (!s) return -1;
    st->S = s;
    s = (int32_t*)realloc(st->I, (size_t)nc * sizeof(int32_t));
    if (!s) return -1;
    st->I = s;
    s = (int32_t*)realloc(st->D, (size_t)nc * sizeof(int32_t));
    if (!s) return -1;
    st->D = s;
    uint8_t* a = (uint8_t*)realloc(st->alive, (size_t)nc);
    if (!a) return -1;
    st->alive = a;
    st->cap = nc;
    return 0;
}

static int store_push_diag(store* st, int32_t lo, int32_t hi) {
    if (st->ndg == st->dg_cap) {
        int32_t nc = st->dg_cap ? st->dg_cap * 2 : 1024;
        diag_rec* r = (diag_rec*)realloc(st->dg, (size_t)nc * sizeof(diag_rec));
        if (!r) return -1;
        st->dg = r;
        st->dg_cap = nc;
    }
    int64_t w = hi >= lo ? (int64_t)(hi - lo + 1) : 0;
    if (store_reserve(st, w)) return -1;
    diag_rec* r = &st->dg[st->ndg++];
    r->lo = lo;
    r->hi = hi;
    r->live_lo = 1;
    r->live_hi = 0;
    r->off = st->used;
    st->used += w;
    return 0;
}

/* Cell (i, d-i) if it was computed and is live; otherwise returns 0 and NEGs. */
static int cell(const store* st, int32_t d, int32_t i, int32_t* s, int32_t* ii, int32_t* dd) {
    *s = NEG; *ii = NEG; *dd = NEG;
    if (d < 0 || d >= st->ndg) return 0;
    const diag_rec* r = &st->dg[d];
    if (i < r->lo || i > r->hi) return 0;
    int64_t k = r->off + (i - r->lo);
    if (!st->alive[k]) return 0;
    *s = st->S[k]; *ii = st->I[k]; *dd = st->D[k];
    return 1;
}

static int32_t max2(int32_t a, int32_t b) { return a > b ? a : b; }

/*
 * One-sided extension.  t[0..m-1] holds t_1..t_m, q likewise; codes 0..3.
 * sub is the 4x4 matrix, row = target base.  flags bit 0: visit each
 * anti-diagonal in descending i (the result must not depend on it).
 * cigar receives runs (len << 4 | op, op 0 = M, 1 = I, 2 = D) in extension
 * order, from the anchor outward.
 */
int orc_extend(const uint8_t* t, int32_t m, const uint8_t* q, int32_t n, const int32_t* sub,
               int32_t o, int32_t e, int64_t ydrop, int32_t flags, orc_result* res,
               uint32_t* cigar, int32_t cigar_cap) {
    store st;
    memset(&st, 0, sizeof(st));
    memset(res, 0, sizeof(*res));
    const int descending = flags & 1;
    const int32_t oe = o + e;

    /* anti-diagonal 0: the origin */
    if (store_push_diag(&st, 0, 0)) { res->status = -1; return -1; }
    st.S[0] = 0; st.I[0] = NEG; st.D[0] = NEG; st.alive[0] = 1;
    st.dg[0].live_lo = 0; st.dg[0].live_hi = 0;
    int64_t live = 1;
    int32_t best = 0, bi = 0, bj = 0, d_last = 0;

    for (int32_t d = 1; d <= m + n; ++d) {
        /* rows that can have a live predecessor: (i, j-1) and (i-1, j) lie on
           d-1, (i-1, j-1) on d-2; rows outside this range are dead */
        const diag_rec* p1 = &st.dg[d - 1];
        const diag_rec* p2 = d >= 2 ? &st.dg[d - 2] : NULL;
        int32_t lo = INT32_MAX, hi = INT32_MIN;
        if (p1->live_hi >= p1->live_lo) { lo = p1->live_lo; hi = p1->live_hi + 1; }
        if (p2 && p2->live_hi >= p2->live_lo) {
            if (p2->live_lo + 1 < lo) lo = p2->live_lo + 1;
            if (p2->live_hi + 1 > hi) hi = p2->live_hi + 1;
        }
        if (lo < d - n) lo = d - n;
        if (lo < 0) lo = 0;
        if (hi > m) hi = m;
        if (hi > d) hi = d;
        if (lo > hi) break;                      /* d-1 and d-2 hold no live cell */
        if (store_push_diag(&st, lo, hi)) { store_free(&st); res->status = -1; return -1; }
        if (hi - lo + 1 > res->max_width) res->max_width = hi - lo + 1;
        if (hi - lo + 1 <= 160) res->narrow_steps++;
        diag_rec* r = &st.dg[d];
        const int64_t T = (int64_t)best - ydrop;   /* prune threshold of this anti-diagonal */
        int32_t dmax = NEG, dmax_i = -1;
        for (int32_t step = 0; step <= hi - lo; ++step) {
            const int32_t i = descending ? hi - step : lo + step;
            const int32_t j = d - i;
            int32_t sl, il, dl, su, iu, du, sd, id, dd;
            int a_left = j >= 1 ? cell(&st, d - 1, i, &sl, &il, &dl) : (sl = il = dl = NEG, 0);
            int a_up = i >= 1 ? cell(&st, d - 1, i - 1, &su, &iu, &du) : (su = iu = du = NEG, 0);
            int a_diag = (i >= 1 && j >= 1) ? cell(&st, d - 2, i - 1, &sd, &id, &dd) : (sd = id = dd = NEG, 0);
            int32_t I = j >= 1 ? max2(il - e, sl - oe) : NEG;
            int32_t D = i >= 1 ? max2(du - e, su - oe) : NEG;
            int32_t G = (i >= 1 && j >= 1) ? sd + sub[t[i - 1] * 4 + q[j - 1]] : NEG;
            int32_t S = max2(G, max2(I, D));
            int alive = a_left || a_up || a_diag;
            if (alive && ydrop >= 0 && (int64_t)S < T) alive = 0;
            int64_t k = r->off + (i - lo);
            if (alive) {
                st.S[k] = S; st.I[k] = I; st.D[k] = D; st.alive[k] = 1;
                ++live;
                if (i < r->live_lo || r->live_hi < r->live_lo) r->live_lo = i;
                if (i > r->live_hi || r->live_hi < r->live_lo) r->live_hi = i;
                if (S > dmax || (S == dmax && i < dmax_i)) { dmax = S; dmax_i = i; }
            } else {
                st.S[k] = NEG; st.I[k] = NEG; st.D[k] = NEG; st.alive[k] = 0;
            }
        }
        if (r->live_hi < r->live_lo) continue;   /* no live cell on d; d+1 may still be
                                                    reached from d-1 by a diagonal move */
        d_last = d;
        if (dmax > best) { best = dmax; bi = dmax_i; bj = d - dmax_i; }
    }

    res->score = best;
    res->i_end = bi;
    res->j_end = bj;
    res->d_last = d_last;
    res->live_cells = live;

    /* traceback from (bi, bj) in state S; ops collected backwards */
    int32_t cap_ops = bi + bj;
    uint8_t* ops = (uint8_t*)malloc((size_t)(cap_ops > 0 ? cap_ops : 1));
    if (!ops) { store_free(&st); res->status = -1; return -1; }
    int32_t nops = 0, i = bi, j = bj, state = 0; /* 0 = S, 1 = I, 2 = D */
    while (i > 0 || j > 0) {
        int32_t s0, i0, d0;
        cell(&st, i + j, i, &s0, &i0, &d0);
        if (state == 0) {
            int32_t sd, id, dd;
            if (i >= 1 && j >= 1 && cell(&st, i + j - 2, i - 1, &sd, &id, &dd) &&
                s0 == sd + sub[t[i - 1] * 4 + q[j - 1]]) {
                ops[nops++] = 0; --i; --j;
            } else if (j >= 1 && s0 == i0) {
                state = 1;
            } else {
                state = 2;
            }
        } else if (state == 1) {
            int32_t sl, il, dl;
            cell(&st, i + j - 1, i, &sl, &il, &dl);
            ops[nops++] = 1;
            state = (i0 == sl - oe) ? 0 : 1;
            --j;
        } else {
            int32_t su, iu, du;
            cell(&st, i + j - 1, i - 1, &su, &iu, &du);
            ops[nops++] = 2;
            state = (d0 == su - oe) ? 0 : 2;
            --i;
        }
    }
    /* runs in extension order (reverse of the walk) */
    int32_t nr = 0;
    for (int32_t k = nops - 1; k >= 0;) {
        int32_t l = k;
        while (l >= 0 && ops[l] == ops[k]) --l;
        uint32_t len = (uint32_t)(k - l);
        if (nr >= cigar_cap) { free(ops); store_free(&st); res->status = -2; return -2; }
        cigar[nr++] = (len << 4) | ops[k];
        k = l;
    }
    res->n_cigar = nr;
    free(ops);
    store_free(&st);
    return 0;
}

/* LOCAL mode: unpruned, zero-floored, score and end cell only.  Row-major. */
int orc_local(const uint8_t* t, int32_t m, const uint8_t* q, int32_t n, const int32_t* sub,
              int32_t o, int32_t e, orc_result* res) {
    memset(res, 0, sizeof(*res));
    const int32_t oe = o + e;
    int32_t* Sprev = (int32_t*)malloc((size_t)(n + 1) * sizeof(int32_t));
    int32_t* Scur = (int32_t*)malloc((size_t)(n + 1) * sizeof(int32_t));
    int32_t* Dcol = (int32_t*)malloc((size_t)(n + 1) * sizeof(int32_t));
    if (!Sprev || !Scur || !Dcol) { free(Sprev); free(Scur); free(Dcol); res->status = -1; return -1; }
    for (int32_t j = 0; j <= n; ++j) { Sprev[j] = 0; Dcol[j] = NEG; }
    int32_t best = 0, bi = 0, bj = 0;
    for (int32_t i = 1; i <= m; ++i) {
        Scur[0] = 0;
        int32_t I = NEG;
        for (int32_t j = 1; j <= n; ++j) {
            I = max2(I - e, Scur[j - 1] - oe);
            Dcol[j] = max2(Dcol[j] - e, Sprev[j] - oe);
            int32_t G = Sprev[j - 1] + sub[t[i - 1] * 4 + q[j - 1]];
            int32_t S = max2(0, max2(G, max2(I, Dcol[j])));
            Scur[j] = S;
            /* keep the earliest (d, i) among equal maxima */
            if (S > best || (S == best && (i + j < bi + bj || (i + j == bi + bj && i < bi)))) {
                best = S; bi = i; bj = j;
            }
        }
        int32_t* tmp = Sprev; Sprev = Scur; Scur = tmp;
    }
    res->score = best;
    res->i_end = bi;
    res->j_end = bj;
    res->live_cells = (int64_t)m * n;
    res->d_last = m + n;
    free(Sprev); free(Scur); free(Dcol);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Batch driver: window setup per seed and side, and a thread pool over      */
/* independent extensions (the FastZ paper's multicore LASTZ partitions the  */
/* seeds across processes in the same way, section 3.4).                     */
/* ------------------------------------------------------------------------ */
#include <pthread.h>

typedef struct {
    const uint8_t *tseq, *qseq;
    uint64_t t_len, q_len;
    const uint64_t *t_pos, *q_pos;
    const uint32_t* side;
    int64_t n_seeds;
    const int32_t* sub;
    int32_t o, e, max_len, mode;
    int64_t ydrop;
    int32_t flags;
    orc_result* out;          /* 2 per seed: [right, left] */
    uint32_t* cigar;          /* runs */
    const int64_t* cig_off;   /* 2*n_seeds + 1 offsets into cigar */
    int64_t next;             /* work counter */
    pthread_mutex_t mu;
} batch_job;

/* Window of one side, in extension order.  Right: seq[pos], seq[pos+1], ...
   Left: seq[pos-1], seq[pos-2], ...  Length min(max_len, bases available). */
static int32_t window(const uint8_t* seq, uint64_t len, uint64_t pos, int left, int32_t max_len,
                      uint8_t* buf) {
    uint64_t avail = left ? pos : (pos <= len ? len - pos : 0);
    if (pos > len) avail = left ? len : 0;
    int32_t w = avail < (uint64_t)max_len ? (int32_t)avail : max_len;
    for (int32_t k = 0; k < w; ++k) buf[k] = left ? seq[pos - 1 - k] : seq[pos + k];
    return w;
}

static void run_one(batch_job* jb, int64_t x, uint8_t* tb, uint8_t* qb) {
    int64_t s = x >> 1;
    int left = (int)(x & 1);
    orc_result* r = &jb->out[x];
    memset(r, 0, sizeof(*r));
    uint32_t want = left ? 2u : 1u;
    if (!(jb->side[s] & want)) return;
    int32_t m = window(jb->tseq, jb->t_len, jb->t_pos[s], left, jb->max_len, tb);
    int32_t n = window(jb->qseq, jb->q_len, jb->q_pos[s], left, jb->max_len, qb);
    if (jb->mode == 1) {
        orc_local(tb, m, qb, n, jb->sub, jb->o, jb->e, r);
    } else {
        int64_t off = jb->cig_off[x];
        int32_t cap = (int32_t)(jb->cig_off[x + 1] - off);
        orc_extend(tb, m, qb, n, jb->sub, jb->o, jb->e, jb->ydrop, jb->flags, r,
                   jb->cigar + off, cap);
    }
}

static void* worker(void* arg) {
    batch_job* jb = (batch_job*)arg;
    uint8_t* tb = (uint8_t*)malloc((size_t)jb->max_len + 1);
    uint8_t* qb = (uint8_t*)malloc((size_t)jb->max_len + 1);
    for (;;) {
        pthread_mutex_lock(&jb->mu);
        int64_t x = jb->next++;
        pthread_mutex_unlock(&jb->mu);
        if (x >= 2 * jb->n_seeds) break;
        run_one(jb, x, tb, qb);
    }
    free(tb);
    free(qb);
    return NULL;
}

int orc_batch(const uint8_t* tseq, uint64_t t_len, const uint8_t* qseq, uint64_t q_len,
              const uint64_t* t_pos, const uint64_t* q_pos, const uint32_t* side, int64_t n_seeds,
              const int32_t* sub, int32_t o, int32_t e, int64_t ydrop, int32_t max_len, int32_t mode,
              int32_t flags, int32_t nthreads, orc_result* out, uint32_t* cigar, const int64_t* cig_off) {
    batch_job jb;
    memset(&jb, 0, sizeof(jb));
    jb.tseq = tseq; jb.qseq = qseq; jb.t_len = t_len; jb.q_len = q_len;
    jb.t_pos = t_pos; jb.q_pos = q_pos; jb.side = side; jb.n_seeds = n_seeds;
    jb.sub = sub; jb.o = o; jb.e = e; jb.ydrop = ydrop; jb.max_len = max_len; jb.mode = mode;
    jb.flags = flags; jb.out = out; jb.cigar = cigar; jb.cig_off = cig_off;
    pthread_mutex_init(&jb.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    for (int k = 1; k < nthreads; ++k) pthread_create(&th[k], NULL, worker, &jb);
    worker(&jb);
    for (int k = 1; k < nthreads; ++k) pthread_join(th[k], NULL);
    pthread_mutex_destroy(&jb.mu);
    int rc = 0;
    for (int64_t x = 0; x < 2 * n_seeds; ++x)
        if (out[x].status) rc = out[x].status;
    return rc;
}

/*
 * Two more dynamic programs of the DPX intrinsics article (section 1.3: edit
 * distance and dynamic time warping are, like alignment, a minimum over three
 * sources plus an add).  Plain full-table definitions, one row kept at a time.
 *
 * Edit distance (Levenshtein: substitution, insertion and deletion cost 1):
 *   D(i,0) = i, D(0,j) = j,
 *   D(i,j) = min(D(i-1,j) + 1, D(i,j-1) + 1, D(i-1,j-1) + [a_i != b_j]);
 *   result D(m,n).
 */
int32_t orc_edit_distance(const uint8_t* a, int32_t m, const uint8_t* b, int32_t n) {
    int32_t* prev = (int32_t*)malloc(sizeof(int32_t) * ((size_t)n + 1));
    int32_t* cur = (int32_t*)malloc(sizeof(int32_t) * ((size_t)n + 1));
    if (!prev || !cur) { free(prev); free(cur); return -2; }
    for (int32_t j = 0; j <= n; ++j) prev[j] = j;
    for (int32_t i = 1; i <= m; ++i) {
        cur[0] = i;
        for (int32_t j = 1; j <= n; ++j) {
            int32_t v = prev[j] + 1;                                   /* from above: a_i deleted */
            if (cur[j - 1] + 1 < v) v = cur[j - 1] + 1;                /* from the left: b_j inserted */
            const int32_t dg = prev[j - 1] + (a[i - 1] != b[j - 1]);   /* diagonal: match or substitution */
            if (dg < v) v = dg;
            cur[j] = v;
        }
        int32_t* t = prev; prev = cur; cur = t;
    }
    const int32_t r = prev[n];
    free(prev);
    free(cur);
    return r;
}

/*
 * Dynamic time warping of two integer sequences, cost |x_i - y_j| per cell:
 *   D(0,0) = 0, D(i,0) = D(0,j) = infinity for i, j >= 1,
 *   D(i,j) = |x_i - y_j| + min(D(i-1,j), D(i,j-1), D(i-1,j-1));
 *   result D(m,n) (64-bit); -1 when exactly one sequence is empty (no warping
 *   path exists), 0 when both are.
 */
int64_t orc_dtw(const int32_t* x, int32_t m, const int32_t* y, int32_t n) {
    if (m == 0 && n == 0) return 0;
    if (m == 0 || n == 0) return -1;
    const int64_t INF = (int64_t)1 << 62;
    int64_t* prev = (int64_t*)malloc(sizeof(int64_t) * ((size_t)n + 1));
    int64_t* cur = (int64_t*)malloc(sizeof(int64_t) * ((size_t)n + 1));
    if (!prev || !cur) { free(prev); free(cur); return -2; }
    prev[0] = 0;
    for (int32_t j = 1; j <= n; ++j) prev[j] = INF;
    for (int32_t i = 1; i <= m; ++i) {
        cur[0] = INF;
        for (int32_t j = 1; j <= n; ++j) {
            int64_t best = prev[j];
            if (cur[j - 1] < best) best = cur[j - 1];
            if (prev[j - 1] < best) best = prev[j - 1];
            const int64_t c = (int64_t)x[i - 1] - (int64_t)y[j - 1];
            cur[j] = best + (c < 0 ? -c : c);
        }
        int64_t* t = prev; prev = cur; cur = t;
    }
    const int64_t r = prev[n];
    free(prev);
    free(cur);
    return r;
}
