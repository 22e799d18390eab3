/*
 * CPU oracle for the topology-aware expert-routing plan.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
 * statement of what the GPU path must compute, used to check it bit for bit.
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (page title, section / equation / figure):
 *   [TopoEP]  "TopoEP: Topology-Aware Load Balancing for Expert-Parallel MoE
 *             Training" -- §2.1 (Top-k gating), §6.4 (synthetic routing from
 *             biased random logits), §4.1 (system model, Eqs. 3-4), §4.2 (constraints
 *             C1-C5, Eqs. 5-8), §4.3 (two-stage solver, Eqs. 9-10, Fig. 9),
 *             §2.3 (Fig. 3 byte accounting), §5 (receive counts on the GPU).
 *   [Zyphra]  "Expert Coupling in MoE Pretraining" -- sections "Experts Are
 *             Correlated Within a Layer" and "Routing Is Also Correlated
 *             Across Layers".
 *   [MoX]     "MoX: Efficient MoE Routing on Direct-Connect Topologies" --
 *             §2.4 "Partial Reduction on Combine" (combine is a reduction of
 *             the top-K expert outputs into one vector per token); §2 the
 *             per-token destination bitmap.
 *   [Zyphra]  also "Moving Correlated Experts Together" (a deduplicating
 *             dispatcher sends a token to a GPU once, with metadata naming
 *             the local experts that process it).
 *
 * Where the pages leave a step open, the reading taken is stated at the step.
 * Every function is a direct transcription of the step list, with no blocking,
 * fusion or reordering.  Integers only; 64-bit where a product may overflow.
 *
 * Conventions shared with the inputs (not with any other code):
 *   pair p = t*k + j; each rank routes its own local tokens [TopoEP §2.1],
 *   the ranks' blocks lying one after the other: source rank src(t) = the s
 *   with off[s] <= t < off[s+1] for the caller's offsets off[0..R]
 *   (0 = off[0] <= ... <= off[R] = T), or t / (T/R) for equal blocks when no
 *   offsets are given (T % R == 0); domain dom(r) = r / ranks_per_node;
 *   main(e) = e / (E/R) with local index e % (E/R) unless a main_rank map is
 *   given, in which case the local index of e is the number of experts e' < e
 *   with the same main rank; an instance (r, l) is packed as r*n_local + l,
 *   n_local = E/R + n_slot, l < E/R a main, l >= E/R replica slot l - E/R.
 *
 * Return codes: 0 ok, -1 bad argument, -2 an id outside [0, E).
 *
 * Floating point (gating, permute and combine only): bf16 values are 16-bit
 * patterns, widened to float by appending 16 zero bits and narrowed by
 * round-to-nearest-even; products and sums are separate float operations
 * (built with -ffp-contract=off, so no multiply-add is fused).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL -1
#define ORC_ERANGE -2

/* ------------------------------------------------------------------------ */
/* Problem description                                                        */
/* ------------------------------------------------------------------------ */

typedef struct {
    int T, E, k, R, rpn, n_slot;
    int64_t S_tok;   /* bytes of one routed activation [TopoEP §4.1] */
    int64_t W;       /* ||W_e|| bytes, equal for all experts [TopoEP §4.1] */
    int64_t c_intra; /* c_{s,r} for s != r in the same NVLink domain */
    int64_t c_inter; /* c_{s,r} across domains */
    int max_iters;   /* 0 = refine until no feasible candidate */
    int M, E_R, n_local;
    int *main_of;    /* [E] main(e) */
    int *main_l;     /* [E] local index of e on main(e) */
} Problem;

static int dom(const Problem *P, int r) { return r / P->rpn; }

/* Communication-time matrix C of [TopoEP §4.1]: c_{r,r} = 0, cheaper inside
 * an NVLink domain than across domains (two-level integer reading). */
static int64_t cost(const Problem *P, int s, int r) {
    if (s == r) return 0;
    if (dom(P, s) == dom(P, r)) return P->c_intra;
    return P->c_inter;
}

/* src[t] for t < T: the source rank of every token, from the offsets off
 * (R+1 values) or, when off is NULL, from equal blocks of T/R tokens.  An
 * offset table that is not 0 = off[0] <= off[1] <= ... <= off[R] = T, or
 * equal blocks that do not divide T, are argument errors. */
static int token_sources(int T, int R, const int64_t *off, int32_t *src) {
    if (T < 0 || R < 1) return ORC_EINVAL;
    if (!off) {
        if (T % R != 0) return ORC_EINVAL;
        for (int t = 0; t < T; t++) src[t] = t / (T / R);
        return ORC_OK;
    }
    if (off[0] != 0 || off[R] != T) return ORC_EINVAL;
    for (int s = 0; s < R; s++) {
        if (off[s + 1] < off[s]) return ORC_EINVAL;
        for (int64_t t = off[s]; t < off[s + 1]; t++) src[t] = s;
    }
    return ORC_OK;
}

static int32_t *sources_or_null(int T, int R, const int64_t *off) {
    int32_t *src = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    if (src && token_sources(T, R, off, src) != ORC_OK) {
        free(src);
        return NULL;
    }
    return src;
}

static int problem_init(Problem *P, int T, int E, int k, int R, int rpn,
                        int n_slot, int64_t S_tok, int64_t W, int64_t c_intra,
                        int64_t c_inter, int max_iters, const int32_t *main_rank) {
    memset(P, 0, sizeof *P);
    if (T < 0 || E < 1 || k < 1 || R < 1 || rpn < 1 || n_slot < 0) return ORC_EINVAL;
    if (R % rpn != 0 || E % R != 0) return ORC_EINVAL;
    if (S_tok < 0 || W < 0 || c_intra < 1 || c_inter < c_intra || max_iters < 0) return ORC_EINVAL;
    P->T = T; P->E = E; P->k = k; P->R = R; P->rpn = rpn; P->n_slot = n_slot;
    P->S_tok = S_tok; P->W = W; P->c_intra = c_intra; P->c_inter = c_inter;
    P->max_iters = max_iters;
    P->M = R / rpn; P->E_R = E / R; P->n_local = P->E_R + n_slot;
    P->main_of = (int *)malloc(sizeof(int) * E);
    P->main_l = (int *)malloc(sizeof(int) * E);
    int *owned = (int *)calloc(R, sizeof(int));
    for (int e = 0; e < E; e++) {
        int r = main_rank ? main_rank[e] : e / P->E_R;
        if (r < 0 || r >= R) { free(owned); return ORC_EINVAL; }
        P->main_of[e] = r;
        P->main_l[e] = owned[r]++;   /* ascending e within the rank */
    }
    for (int r = 0; r < R; r++)
        if (owned[r] != P->E_R) { free(owned); return ORC_EINVAL; }
    free(owned);
    return ORC_OK;
}

static void problem_free(Problem *P) {
    free(P->main_of);
    free(P->main_l);
}

/* ------------------------------------------------------------------------ */
/* O1  Routing matrix Omega  [TopoEP §4.1, Eq. 3]                             */
/* omega_{s,e} = number of token-expert assignments from source rank s that  */
/* select expert e.                                                           */
/* ------------------------------------------------------------------------ */

int oracle_hist(int T, int E, int k, int R, int n_layers, const int64_t *rank_offsets,
                const int32_t *ids, int32_t *hist) {
    if (T < 0 || E < 1 || k < 1 || R < 1 || n_layers < 0) return ORC_EINVAL;
    int32_t *src = sources_or_null(T, R, rank_offsets);
    if (!src) return ORC_EINVAL;
    int rc = ORC_OK;
    for (int l = 0; l < n_layers; l++) {
        const int32_t *id = ids + (int64_t)l * T * k;
        int32_t *h = hist + (int64_t)l * R * E;
        memset(h, 0, sizeof(int32_t) * (size_t)R * E);
        for (int t = 0; t < T; t++) {
            int s = src[t];
            for (int j = 0; j < k; j++) {
                int e = id[(int64_t)t * k + j];
                if (e < 0 || e >= E) { rc = ORC_ERANGE; continue; }
                h[(int64_t)s * E + e] += 1;
            }
        }
    }
    free(src);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* O0  Top-k gating [TopoEP §2.1: for each token a trainable router selects  */
/* the Top-k experts; §6.4: synthetic routing uses random logits with a      */
/* fixed expert-specific bias], followed by O1 on the selected ids.          */
/* Readings: score_{t,e} = logit_{t,e} + bias_e as one float addition (no    */
/* addition without a bias); the k experts of the largest scores, in         */
/* descending order; equal scores (-0 equals +0) go to the lower expert      */
/* index; a NaN score ranks below every number, NaNs among themselves by     */
/* index.  scores[t][j] is the raw logit of the j-th selected expert.        */
/* logits are float32, or bf16 patterns widened by appending 16 zero bits.   */
/* ------------------------------------------------------------------------ */

/* Does score a of expert ia rank above score b of expert ib? */
static int gate_above(float a, int ia, float b, int ib) {
    int na = a != a, nb = b != b;
    if (na != nb) return nb;             /* a number ranks above a NaN */
    if (!na && a != b) return a > b;
    return ia < ib;
}

int oracle_gate(int T, int E, int k, int R, int n_layers, const int64_t *rank_offsets, int is_bf16,
                const void *logits, const float *bias, int32_t *ids, float *scores, int32_t *hist) {
    if (T < 0 || E < 1 || k < 1 || k > E || R < 1 || n_layers < 0) return ORC_EINVAL;
    float *raw = (float *)malloc(sizeof(float) * (size_t)E);
    float *sc = (float *)malloc(sizeof(float) * (size_t)E);
    char *taken = (char *)malloc((size_t)E);
    if (!raw || !sc || !taken) { free(raw); free(sc); free(taken); return ORC_EINVAL; }
    for (int64_t t = 0; t < (int64_t)n_layers * T; t++) {
        for (int e = 0; e < E; e++) {
            if (is_bf16) {
                uint32_t w = (uint32_t)((const uint16_t *)logits)[t * E + e] << 16;
                memcpy(&raw[e], &w, 4);
            } else {
                raw[e] = ((const float *)logits)[t * E + e];
            }
            sc[e] = bias ? raw[e] + bias[e] : raw[e];
            taken[e] = 0;
        }
        for (int j = 0; j < k; j++) {
            int best = -1;
            for (int e = 0; e < E; e++)
                if (!taken[e] && (best < 0 || gate_above(sc[e], e, sc[best], best))) best = e;
            taken[best] = 1;
            ids[t * k + j] = best;
            scores[t * k + j] = raw[best];
        }
    }
    free(raw); free(sc); free(taken);
    return oracle_hist(T, E, k, R, n_layers, rank_offsets, ids, hist);
}

/* ------------------------------------------------------------------------ */
/* O2  Expert co-selection and cross-layer transition counts                  */
/* [Zyphra, "Experts Are Correlated Within a Layer", "Routing Is Also         */
/* Correlated Across Layers"].  With n_t^l the count vector of token t's      */
/* choices at layer l:  co_l = sum_t n_t^l (n_t^l)^T,                         */
/* tr_l = sum_t n_t^l (n_t^{l+1})^T.  The diagonal of co is kept (the page    */
/* masks it only in a plot).  tr may be NULL.                                 */
/* ------------------------------------------------------------------------ */

int oracle_cooccur(int L, int T, int E, int k, const int32_t *ids, int64_t *co,
                   int64_t *tr) {
    if (L < 0 || T < 0 || E < 1 || k < 1) return ORC_EINVAL;
    int rc = ORC_OK;
    memset(co, 0, sizeof(int64_t) * (size_t)L * E * E);
    if (tr && L > 1) memset(tr, 0, sizeof(int64_t) * (size_t)(L - 1) * E * E);
    for (int l = 0; l < L; l++) {
        const int32_t *a = ids + (int64_t)l * T * k;
        for (int t = 0; t < T; t++)
            for (int j = 0; j < k; j++) {
                int x = a[(int64_t)t * k + j];
                if (x < 0 || x >= E) { rc = ORC_ERANGE; continue; }
                for (int i = 0; i < k; i++) {
                    int y = a[(int64_t)t * k + i];
                    if (y < 0 || y >= E) continue;
                    co[((int64_t)l * E + x) * E + y] += 1;
                }
            }
        if (!tr || l == L - 1) continue;
        const int32_t *b = ids + (int64_t)(l + 1) * T * k;
        for (int t = 0; t < T; t++)
            for (int j = 0; j < k; j++) {
                int x = a[(int64_t)t * k + j];
                if (x < 0 || x >= E) continue;
                for (int i = 0; i < k; i++) {
                    int y = b[(int64_t)t * k + i];
                    if (y < 0 || y >= E) { rc = ORC_ERANGE; continue; }
                    tr[((int64_t)l * E + x) * E + y] += 1;
                }
            }
    }
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Plan state for one layer                                                   */
/* ------------------------------------------------------------------------ */

typedef struct {
    const Problem *P;
    const int32_t *hist;  /* [R][E] omega */
    int32_t *slot_expert; /* [R][n_slot], -1 empty  (x for replicas) */
    int32_t *q;           /* [R_src][R_dst][n_local] */
    int32_t *U;           /* [R][n_local] instance loads */
    int32_t *Lr;          /* [R] rank loads */
    int *used;            /* [R] occupied replica slots */
    int *host;            /* [R][E] local index of e on r, or -1  (x) */
    int64_t stage1_replicas;
    int64_t refine_iters;
} Plan;

static int32_t *Q(Plan *S, int s, int r, int l) {
    const Problem *P = S->P;
    return &S->q[((int64_t)s * P->R + r) * P->n_local + l];
}

static void place_replica(Plan *S, int r, int e) {
    const Problem *P = S->P;
    int slot = S->used[r]++;
    S->slot_expert[(int64_t)r * P->n_slot + slot] = e;
    S->host[(int64_t)r * P->E + e] = P->E_R + slot;
}

/* O3  Domain demand D_{d,e} = sum over sources s in domain d of omega_{s,e}
 * [TopoEP §4.1, Eq. 4]. */
static void demand(const Plan *S, int64_t *D) {
    const Problem *P = S->P;
    memset(D, 0, sizeof(int64_t) * (size_t)P->M * P->E);
    for (int s = 0; s < P->R; s++)
        for (int e = 0; e < P->E; e++)
            D[(int64_t)dom(P, s) * P->E + e] += S->hist[(int64_t)s * P->E + e];
}

typedef struct { int64_t b; int e; } Cand;

static int cand_cmp(const void *x, const void *y) {
    const Cand *a = (const Cand *)x, *c = (const Cand *)y;
    if (a->b != c->b) return a->b > c->b ? -1 : 1;   /* benefit descending */
    return a->e < c->e ? -1 : (a->e > c->e);          /* then expert ascending */
}

/* O4  Stage 1, inter-node placement [TopoEP §4.3, Eq. 9; C4 of §4.2].
 * For each domain d, every expert whose main lies outside d with benefit
 * b_{d,e} = 2 D_{d,e} S_tok - ||W|| > 0 is a candidate; candidates are taken
 * in descending benefit (ties: lower expert id first) and each is placed on
 * the rank of d with a free slot that has the fewest occupied slots (ties:
 * lower rank).  At most one stage-1 replica per (domain, expert).  A domain
 * stops when none of its ranks has a free slot. */
static void stage1_place(Plan *S, const int64_t *D) {
    const Problem *P = S->P;
    Cand *c = (Cand *)malloc(sizeof(Cand) * (size_t)(P->E ? P->E : 1));
    for (int d = 0; d < P->M; d++) {
        int n = 0;
        for (int e = 0; e < P->E; e++) {
            if (dom(P, P->main_of[e]) == d) continue;
            int64_t b = 2 * D[(int64_t)d * P->E + e] * P->S_tok - P->W;
            if (b > 0) { c[n].b = b; c[n].e = e; n++; }
        }
        qsort(c, (size_t)n, sizeof(Cand), cand_cmp);
        for (int i = 0; i < n; i++) {
            int best = -1;
            for (int r = d * P->rpn; r < (d + 1) * P->rpn; r++) {
                if (S->used[r] >= P->n_slot) continue;
                if (best < 0 || S->used[r] < S->used[best]) best = r;
            }
            if (best < 0) break;
            place_replica(S, best, c[i].e);
            S->stage1_replicas++;
        }
    }
    free(c);
}

/* Sort helper: ranks ordered by (c_{s,r}, r) ascending. */
static const Problem *g_sortP;
static int g_sort_s;
static int rank_cost_cmp(const void *x, const void *y) {
    int a = *(const int *)x, b = *(const int *)y;
    int64_t ca = cost(g_sortP, g_sort_s, a), cb = cost(g_sortP, g_sort_s, b);
    if (ca != cb) return ca < cb ? -1 : 1;
    return a < b ? -1 : (a > b);
}

/* O5  Stage-1 routing [TopoEP §4.3, "Given the resulting placement ..."].
 * For every (s, e) with omega_{s,e} > 0: the candidate instances are those
 * of e inside dom(s) if any exist, else every instance of e.  omega_{s,e} is
 * divided as evenly as integers allow: each of the n instances gets
 * floor(omega / n) and the first (omega mod n) of them, in ascending
 * (c_{s,r}, r) order, get one more.  Then U_{e,r} = sum_s q_{s,e,r} and
 * L_r = sum of U over r's instances. */
static void stage1_route(Plan *S) {
    const Problem *P = S->P;
    int *I = (int *)malloc(sizeof(int) * (size_t)P->R);
    for (int s = 0; s < P->R; s++)
        for (int e = 0; e < P->E; e++) {
            int w = S->hist[(int64_t)s * P->E + e];
            if (w == 0) continue;
            int n = 0;
            for (int r = 0; r < P->R; r++)
                if (S->host[(int64_t)r * P->E + e] >= 0 && dom(P, r) == dom(P, s)) I[n++] = r;
            if (n == 0)
                for (int r = 0; r < P->R; r++)
                    if (S->host[(int64_t)r * P->E + e] >= 0) I[n++] = r;
            g_sortP = P; g_sort_s = s;
            qsort(I, (size_t)n, sizeof(int), rank_cost_cmp);
            int base = w / n, rem = w % n;
            for (int i = 0; i < n; i++)
                *Q(S, s, I[i], S->host[(int64_t)I[i] * P->E + e]) = base + (i < rem ? 1 : 0);
        }
    free(I);
    memset(S->U, 0, sizeof(int32_t) * (size_t)P->R * P->n_local);
    for (int s = 0; s < P->R; s++)
        for (int r = 0; r < P->R; r++)
            for (int l = 0; l < P->n_local; l++)
                S->U[(int64_t)r * P->n_local + l] += *Q(S, s, r, l);
    for (int r = 0; r < P->R; r++) {
        int64_t sum = 0;
        for (int l = 0; l < P->n_local; l++) sum += S->U[(int64_t)r * P->n_local + l];
        S->Lr[r] = (int32_t)sum;
    }
}

/* Source order for assignments that move from r_b to r_t: ascending
 * (c_{s,r_t} - c_{s,r_b}, s), i.e. the moves that save the most token cost
 * first.  (Reading: the pages do not say which assignments move.) */
static int g_rt, g_rb;
static int src_move_cmp(const void *x, const void *y) {
    int a = *(const int *)x, b = *(const int *)y;
    int64_t ka = cost(g_sortP, a, g_rt) - cost(g_sortP, a, g_rb);
    int64_t kb = cost(g_sortP, b, g_rt) - cost(g_sortP, b, g_rb);
    if (ka != kb) return ka < kb ? -1 : 1;
    return a < b ? -1 : (a > b);
}

typedef struct {
    int ok;
    int64_t delta, Lt, cost;
    int e, rt, lb, lt, is_new;
} Move;

/* Lexicographic candidate order of [TopoEP §4.3, after Eq. 10]: transfer
 * amount (larger first), target load (smaller first), communication cost
 * (smaller first); remaining ties by expert id, then target rank, ascending. */
static int move_better(const Move *a, const Move *b) {
    if (!b->ok) return 1;
    if (a->delta != b->delta) return a->delta > b->delta;
    if (a->Lt != b->Lt) return a->Lt < b->Lt;
    if (a->cost != b->cost) return a->cost < b->cost;
    if (a->e != b->e) return a->e < b->e;
    return a->rt < b->rt;
}

/* O6  Stage 2, intra-node refinement [TopoEP §4.3, Eq. 10, Fig. 9].
 * Each domain independently: take the busiest rank r_b (ties: lowest r);
 * for every expert e with load on r_b and every other rank r_t of the domain
 * that hosts e or has a free slot, the transfer amount is
 *     delta = min(U_{e,r_b}, floor((L_{r_b} - L_{r_t}) / 2)),
 * feasible when delta >= 1.  The assignments moved are taken from sources in
 * the order of src_move_cmp, m_s = min(q_{s,e,r_b}, still to move).  The cost
 * of a candidate is the change it makes to T_token + T_replica of Eq. 7:
 *     2 S_tok sum_s m_s (c_{s,r_t} - c_{s,r_b}) + [r_t lacks e] c_{main(e),r_t} ||W||.
 * The best candidate (move_better) is committed -- a new replica in r_t's
 * next free slot if needed, the m_s moved in q, U and L updated -- and the
 * loop repeats until the busiest rank has no feasible candidate (or the
 * optional iteration cap).  Each commit lowers sum_r L_r^2 by
 * 2 delta (gap - delta) >= 2, so the loop ends. */
static void stage2_refine(Plan *S) {
    const Problem *P = S->P;
    int *order = (int *)malloc(sizeof(int) * (size_t)P->R);
    int64_t *m = (int64_t *)malloc(sizeof(int64_t) * (size_t)P->R);
    for (int d = 0; d < P->M; d++) {
        int r0 = d * P->rpn, r1 = r0 + P->rpn;
        int64_t iters = 0;
        for (;;) {
            if (P->max_iters > 0 && iters >= P->max_iters) break;
            int rb = r0;
            for (int r = r0; r < r1; r++)
                if (S->Lr[r] > S->Lr[rb]) rb = r;
            Move best; memset(&best, 0, sizeof best);
            for (int lb = 0; lb < P->n_local; lb++) {
                int64_t Ub = S->U[(int64_t)rb * P->n_local + lb];
                if (Ub <= 0) continue;
                int e = lb < P->E_R ? -1 : S->slot_expert[(int64_t)rb * P->n_slot + (lb - P->E_R)];
                if (lb < P->E_R) {
                    for (int x = 0; x < P->E; x++)
                        if (P->main_of[x] == rb && P->main_l[x] == lb) e = x;
                }
                for (int rt = r0; rt < r1; rt++) {
                    if (rt == rb) continue;
                    int lt = S->host[(int64_t)rt * P->E + e];
                    int is_new = lt < 0;
                    if (is_new && S->used[rt] >= P->n_slot) continue;
                    int64_t gap = (int64_t)S->Lr[rb] - S->Lr[rt];
                    int64_t half = gap / 2;    /* gap >= 0: floor */
                    int64_t delta = Ub < half ? Ub : half;
                    if (delta < 1) continue;
                    for (int s = 0; s < P->R; s++) order[s] = s;
                    g_sortP = P; g_rt = rt; g_rb = rb;
                    qsort(order, (size_t)P->R, sizeof(int), src_move_cmp);
                    int64_t left = delta, tok = 0;
                    for (int i = 0; i < P->R; i++) {
                        int s = order[i];
                        int64_t have = *Q(S, s, rb, lb);
                        int64_t take = have < left ? have : left;
                        left -= take;
                        tok += take * (cost(P, s, rt) - cost(P, s, rb));
                    }
                    Move mv;
                    mv.ok = 1; mv.delta = delta; mv.Lt = S->Lr[rt];
                    mv.cost = 2 * P->S_tok * tok + (is_new ? cost(P, P->main_of[e], rt) * P->W : 0);
                    mv.e = e; mv.rt = rt; mv.lb = lb; mv.lt = lt; mv.is_new = is_new;
                    if (move_better(&mv, &best)) best = mv;
                }
            }
            if (!best.ok) break;
            /* commit */
            int rt = best.rt, lb = best.lb, lt = best.lt;
            if (best.is_new) {
                place_replica(S, rt, best.e);
                lt = S->host[(int64_t)rt * P->E + best.e];
            }
            for (int s = 0; s < P->R; s++) order[s] = s;
            g_sortP = P; g_rt = rt; g_rb = rb;
            qsort(order, (size_t)P->R, sizeof(int), src_move_cmp);
            int64_t left = best.delta;
            for (int i = 0; i < P->R; i++) {
                int s = order[i];
                int64_t have = *Q(S, s, rb, lb);
                m[s] = have < left ? have : left;
                left -= m[s];
            }
            for (int s = 0; s < P->R; s++) {
                *Q(S, s, rb, lb) -= (int32_t)m[s];
                *Q(S, s, rt, lt) += (int32_t)m[s];
            }
            S->U[(int64_t)rb * P->n_local + lb] -= (int32_t)best.delta;
            S->U[(int64_t)rt * P->n_local + lt] += (int32_t)best.delta;
            S->Lr[rb] -= (int32_t)best.delta;
            S->Lr[rt] += (int32_t)best.delta;
            iters++;
        }
        S->refine_iters += iters;
    }
    free(order);
    free(m);
}

/* Plan statistics (per layer, int64[8]):
 *   0 L_max            max_r L_r after refinement            [TopoEP §4.2, Eq. 5]
 *   1 L_max_static     max_r of the load with mains only (no replicas)
 *   2 n_replicas       occupied replica slots after refinement
 *   3 n_stage1         replicas created by inter-node placement
 *   4 refine_iters     refinement commits, all domains
 *   5 T_token          2 S_tok sum_{s,e,r} c_{s,r} q_{s,e,r}   [Eq. 7]
 *   6 T_replica        sum_{replicas} c_{main(e),r} ||W||      [Eq. 7]
 *   7 sum_L            sum_r L_r (= T k)                                   */
static void plan_stats(Plan *S, int64_t *st) {
    const Problem *P = S->P;
    int64_t lmax = 0, sum = 0;
    for (int r = 0; r < P->R; r++) {
        if (S->Lr[r] > lmax) lmax = S->Lr[r];
        sum += S->Lr[r];
    }
    int64_t smax = 0;
    for (int r = 0; r < P->R; r++) {
        int64_t load = 0;
        for (int e = 0; e < P->E; e++) {
            if (P->main_of[e] != r) continue;
            for (int s = 0; s < P->R; s++) load += S->hist[(int64_t)s * P->E + e];
        }
        if (load > smax) smax = load;
    }
    int64_t nrep = 0, trep = 0;
    for (int r = 0; r < P->R; r++)
        for (int j = 0; j < P->n_slot; j++) {
            int e = S->slot_expert[(int64_t)r * P->n_slot + j];
            if (e < 0) continue;
            nrep++;
            trep += cost(P, P->main_of[e], r) * P->W;
        }
    int64_t ttok = 0;
    for (int s = 0; s < P->R; s++)
        for (int r = 0; r < P->R; r++)
            for (int l = 0; l < P->n_local; l++)
                ttok += cost(P, s, r) * (int64_t)*Q(S, s, r, l);
    ttok *= 2 * P->S_tok;
    st[0] = lmax; st[1] = smax; st[2] = nrep; st[3] = S->stage1_replicas;
    st[4] = S->refine_iters; st[5] = ttok; st[6] = trep; st[7] = sum;
}

int oracle_plan(int T, int E, int k, int R, int rpn, int n_slot, int64_t S_tok,
                int64_t W, int64_t c_intra, int64_t c_inter, int max_iters,
                const int32_t *main_rank, int n_layers, const int32_t *hist,
                int32_t *slot_expert, int32_t *route_cnt, int32_t *inst_load,
                int32_t *rank_load, int64_t *stats) {
    Problem P;
    int rc = problem_init(&P, T, E, k, R, rpn, n_slot, S_tok, W, c_intra, c_inter,
                          max_iters, main_rank);
    if (rc != ORC_OK || n_layers < 0) { problem_free(&P); return ORC_EINVAL; }
    int64_t *D = (int64_t *)malloc(sizeof(int64_t) * (size_t)P.M * E);
    int *used = (int *)malloc(sizeof(int) * (size_t)R);
    int *host = (int *)malloc(sizeof(int) * (size_t)R * E);
    for (int l = 0; l < n_layers; l++) {
        Plan S;
        S.P = &P;
        S.hist = hist + (int64_t)l * R * E;
        S.slot_expert = slot_expert + (int64_t)l * R * n_slot;
        S.q = route_cnt + (int64_t)l * R * R * P.n_local;
        S.U = inst_load + (int64_t)l * R * P.n_local;
        S.Lr = rank_load + (int64_t)l * R;
        S.used = used; S.host = host;
        S.stage1_replicas = 0; S.refine_iters = 0;
        for (int64_t i = 0; i < (int64_t)R * n_slot; i++) S.slot_expert[i] = -1;
        memset(S.q, 0, sizeof(int32_t) * (size_t)R * R * P.n_local);
        memset(used, 0, sizeof(int) * (size_t)R);
        for (int64_t i = 0; i < (int64_t)R * E; i++) host[i] = -1;
        for (int e = 0; e < E; e++) host[(int64_t)P.main_of[e] * E + e] = P.main_l[e];  /* C5 */
        demand(&S, D);
        stage1_place(&S, D);
        stage1_route(&S);
        stage2_refine(&S);
        plan_stats(&S, stats + (int64_t)l * 8);
    }
    free(D); free(used); free(host);
    problem_free(&P);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* O7  Rerouting of each (token, slot) pair to an expert instance             */
/* [TopoEP §1 and Fig. 5, "token rerouting"; the rule is not given].          */
/* Reading: within source s the pairs that select e are taken in ascending  */
/* pair order; the instances of e are listed in ascending (r, l); the o-th    */
/* such pair goes to the instance whose running range of q_{s,e,.} holds o.  */
/* ------------------------------------------------------------------------ */

int oracle_reroute(int T, int E, int k, int R, int rpn, int n_slot,
                   const int32_t *main_rank, const int64_t *rank_offsets, int n_layers,
                   const int32_t *ids, const int32_t *slot_expert, const int32_t *route_cnt,
                   int32_t *dst_inst) {
    Problem P;
    int rc = problem_init(&P, T, E, k, R, rpn, n_slot, 0, 0, 1, 1, 0, main_rank);
    if (rc != ORC_OK || n_layers < 0) { problem_free(&P); return ORC_EINVAL; }
    /* first token of each source */
    int64_t *beg = (int64_t *)malloc(sizeof(int64_t) * (size_t)(R + 1));
    int32_t *src = sources_or_null(T, R, rank_offsets);
    if (!beg || !src) { free(beg); free(src); problem_free(&P); return ORC_EINVAL; }
    for (int s = 0; s <= R; s++) beg[s] = rank_offsets ? rank_offsets[s] : (int64_t)s * (T / R);
    free(src);
    int64_t npairs = (int64_t)T * k;
    int32_t *occ = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int *host = (int *)malloc(sizeof(int) * (size_t)R * E);
    rc = ORC_OK;
    for (int l = 0; l < n_layers; l++) {
        const int32_t *id = ids + l * npairs;
        const int32_t *se = slot_expert + (int64_t)l * R * n_slot;
        const int32_t *q = route_cnt + (int64_t)l * R * R * P.n_local;
        int32_t *dst = dst_inst + l * npairs;
        for (int64_t i = 0; i < (int64_t)R * E; i++) host[i] = -1;
        for (int e = 0; e < E; e++) host[(int64_t)P.main_of[e] * E + e] = P.main_l[e];
        for (int r = 0; r < R; r++)
            for (int j = 0; j < n_slot; j++) {
                int e = se[(int64_t)r * n_slot + j];
                if (e >= 0 && e < E) host[(int64_t)r * E + e] = P.E_R + j;
            }
        for (int s = 0; s < R; s++) {
            memset(occ, 0, sizeof(int32_t) * (size_t)E);
            for (int64_t p = beg[s] * k; p < beg[s + 1] * k; p++) {
                int e = id[p];
                dst[p] = -1;
                if (e < 0 || e >= E) { rc = ORC_ERANGE; continue; }
                int64_t o = occ[e]++;
                int64_t pre = 0;
                for (int r = 0; r < R; r++) {
                    int li = host[(int64_t)r * E + e];
                    if (li < 0) continue;
                    int64_t c = q[((int64_t)s * R + r) * P.n_local + li];
                    if (o < pre + c) { dst[p] = r * P.n_local + li; break; }
                    pre += c;
                }
            }
        }
    }
    free(occ); free(host); free(beg);
    problem_free(&P);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* O8  Dispatch layout [TopoEP §5: receive counts derived on the GPU;        */
/* §2.3 Fig. 3 and §6 Fig. 16 for the byte / locality accounting].            */
/*   sorted_pairs: stable ascending sort of the pair indices by dst_inst     */
/*                 (gather form: sorted_pairs[pos] = p);                      */
/*   seg_off:      exclusive prefix of the per-instance pair counts, [R*n_local+1]; */
/*   send_counts:  [R][R] pairs from source s to destination rank r;         */
/*   layout_stats: int64[8] = pairs local (s = r), intra-domain, inter-domain;  */
/*                 their dispatch bytes (count * S_tok); pairs served by a    */
/*                 replica (l >= E/R); 0.                                     */
/* A dst_inst outside [0, R*n_local) is an argument error.                    */
/* ------------------------------------------------------------------------ */

int oracle_layout(int T, int E, int k, int R, int rpn, int n_slot, int64_t S_tok,
                  const int64_t *rank_offsets, int n_layers, const int32_t *dst_inst,
                  int32_t *sorted_pairs, int32_t *seg_off, int64_t *send_counts,
                  int64_t *layout_stats) {
    if (T < 0 || E < 1 || k < 1 || R < 1 || rpn < 1 || n_slot < 0) return ORC_EINVAL;
    if (R % rpn != 0 || E % R != 0 || n_layers < 0) return ORC_EINVAL;
    int E_R = E / R, n_local = E_R + n_slot, nkeys = R * n_local;
    int32_t *src = sources_or_null(T, R, rank_offsets);
    if (!src) return ORC_EINVAL;
    int64_t npairs = (int64_t)T * k;
    int64_t *count = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nkeys + 1));
    for (int l = 0; l < n_layers; l++) {
        const int32_t *key = dst_inst + l * npairs;
        int32_t *out = sorted_pairs + l * npairs;
        int32_t *off = seg_off + (int64_t)l * (nkeys + 1);
        int64_t *sc = send_counts + (int64_t)l * R * R;
        int64_t *st = layout_stats + (int64_t)l * 8;
        for (int64_t p = 0; p < npairs; p++)
            if (key[p] < 0 || key[p] >= nkeys) { free(count); free(src); return ORC_EINVAL; }
        /* counting sort: count, exclusive prefix, stable placement */
        memset(count, 0, sizeof(int64_t) * (size_t)(nkeys + 1));
        for (int64_t p = 0; p < npairs; p++) count[key[p]]++;
        int64_t run = 0;
        for (int i = 0; i < nkeys; i++) {
            off[i] = (int32_t)run;
            run += count[i];
        }
        off[nkeys] = (int32_t)run;
        for (int i = 0; i < nkeys; i++) count[i] = off[i];
        for (int64_t p = 0; p < npairs; p++) out[count[key[p]]++] = (int32_t)p;
        /* send counts and locality */
        memset(sc, 0, sizeof(int64_t) * (size_t)R * R);
        memset(st, 0, sizeof(int64_t) * 8);
        for (int64_t p = 0; p < npairs; p++) {
            int s = src[p / k];
            int r = key[p] / n_local, li = key[p] % n_local;
            sc[(int64_t)s * R + r]++;
            if (s == r) st[0]++;
            else if (s / rpn == r / rpn) st[1]++;
            else st[2]++;
            if (li >= E_R) st[6]++;
        }
        st[3] = st[0] * S_tok;
        st[4] = st[1] * S_tok;
        st[5] = st[2] * S_tok;
        st[7] = 0;
    }
    free(count);
    free(src);
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Dispatch pack and combine (TopoEP Fig. 1: dispatch sends each token's
 * activation to the ranks hosting its selected experts; [MoX] §2.4: combine
 * reduces the token's top-K expert outputs into one vector).
 *
 * Readings: the send buffer is in layout order -- row pos of y holds the
 * activation of the token of pair sorted[pos]; combine weights each expert
 * output by the caller's gate weight w[t][j] and sums in slot order j = 0..k-1
 * in float, rounding once to bf16.
 * ------------------------------------------------------------------------- */

static float bf16_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))   /* NaN: quiet */
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7fffu + ((u >> 16) & 1u);                              /* to nearest, ties even */
    return (uint16_t)(u >> 16);
}

/* y[l][pos][:] = x[l][sorted[l][pos] / k][:]   (x: [L][T][H], y: [L][T*k][H]) */
int oracle_permute(int L, int T, int k, int H, const uint16_t *x, const int32_t *sorted,
                   uint16_t *y) {
    if (L < 0 || T < 0 || k < 1 || H < 1) return ORC_EINVAL;
    const int64_t npairs = (int64_t)T * k;
    for (int l = 0; l < L; l++)
        for (int64_t pos = 0; pos < npairs; pos++) {
            const int32_t p = sorted[(int64_t)l * npairs + pos];
            if (p < 0 || p >= npairs) return ORC_EINVAL;
            const int t = p / k;
            memcpy(y + ((int64_t)l * npairs + pos) * H, x + ((int64_t)l * T + t) * H,
                   sizeof(uint16_t) * (size_t)H);
        }
    return ORC_OK;
}

/* out[l][t][:] = bf16( sum_{j<k} w[l][t][j] * y[l][pos(t, j)][:] ), where
 * pos(t, j) is the position of pair t*k + j in sorted[l] (sorted is a
 * permutation of the pairs). */
int oracle_combine(int L, int T, int k, int H, const uint16_t *y, const int32_t *sorted,
                   const float *w, uint16_t *out) {
    if (L < 0 || T < 0 || k < 1 || H < 1) return ORC_EINVAL;
    const int64_t npairs = (int64_t)T * k;
    int64_t *pos_of = (int64_t *)malloc(sizeof(int64_t) * (size_t)(npairs > 0 ? npairs : 1));
    if (!pos_of) return ORC_EINVAL;
    for (int l = 0; l < L; l++) {
        for (int64_t p = 0; p < npairs; p++) pos_of[p] = -1;
        for (int64_t pos = 0; pos < npairs; pos++) {
            const int32_t p = sorted[(int64_t)l * npairs + pos];
            if (p < 0 || p >= npairs || pos_of[p] >= 0) { free(pos_of); return ORC_EINVAL; }
            pos_of[p] = pos;
        }
        for (int t = 0; t < T; t++)
            for (int h = 0; h < H; h++) {
                float acc = 0.0f;
                for (int j = 0; j < k; j++) {
                    const int64_t pos = pos_of[(int64_t)t * k + j];
                    const float v = bf16_to_float(y[((int64_t)l * npairs + pos) * H + h]);
                    const float prod = w[((int64_t)l * T + t) * k + j] * v;
                    acc = acc + prod;
                }
                out[((int64_t)l * T + t) * H + h] = float_to_bf16(acc);
            }
    }
    free(pos_of);
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Deduplicated dispatch layout ([Zyphra] "Moving Correlated Experts
 * Together"; [MoX] §2 destination bitmap).  One row per (token, destination
 * rank) instead of one per pair.
 *
 * Readings: rows are ordered by destination rank, then by token (so by
 * source, tokens being source-blocked); a row carries its token and the mask
 * of the token's slots whose instance is on that rank; the destination rank of
 * a pair is dst_inst / n_local.
 *
 * Outputs per layer: seg[R+1] row offsets per destination rank; row_token and
 * row_slots [T*k] (the first seg[R] rows used); tok_dst[T][RW] bitmap of each
 * token's destination ranks, RW = ceil(R / 64) 64-bit words; send[R][R] rows
 * from source s to rank r; stats {rows, pairs, rows to another rank, pairs to
 * another rank}.
 * ------------------------------------------------------------------------- */
int oracle_dedup(int T, int k, int R, int n_local, const int64_t *rank_offsets, int n_layers,
                 const int32_t *dst_inst, int32_t *seg, int32_t *row_token, uint64_t *row_slots,
                 uint64_t *tok_dst, int64_t *send, int64_t *stats) {
    if (T < 0 || k < 1 || k > 64 || R < 1 || n_local < 1 || n_layers < 0) return ORC_EINVAL;
    const int64_t npairs = (int64_t)T * k;
    const int RW = (R + 63) / 64;
    int32_t *src = sources_or_null(T, R, rank_offsets);
    if (!src) return ORC_EINVAL;
    int64_t *fill = (int64_t *)malloc(sizeof(int64_t) * (size_t)(R + 1));
    uint64_t *mask = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)R);
    if (!fill || !mask) { free(fill); free(mask); free(src); return ORC_EINVAL; }
    for (int l = 0; l < n_layers; l++) {
        const int32_t *d = dst_inst + (int64_t)l * npairs;
        int32_t *sg = seg + (int64_t)l * (R + 1);
        int32_t *rt = row_token + (int64_t)l * npairs;
        uint64_t *rs = row_slots + (int64_t)l * npairs;
        uint64_t *td = tok_dst + (int64_t)l * T * RW;
        int64_t *sc = send + (int64_t)l * R * R;
        int64_t *st = stats + (int64_t)l * 4;
        for (int64_t p = 0; p < npairs; p++)
            if (d[p] < 0 || d[p] >= R * n_local) { free(fill); free(mask); free(src); return ORC_EINVAL; }
        /* rows per destination rank */
        for (int r = 0; r <= R; r++) fill[r] = 0;
        for (int t = 0; t < T; t++)
            for (int j = 0; j < k; j++) {
                const int r = d[(int64_t)t * k + j] / n_local;
                int first = 1;
                for (int i = 0; i < j; i++)
                    if (d[(int64_t)t * k + i] / n_local == r) first = 0;
                if (first) fill[r]++;
            }
        int64_t run = 0;
        for (int r = 0; r < R; r++) {
            const int64_t c = fill[r];
            sg[r] = (int32_t)run;
            fill[r] = run;
            run += c;
        }
        sg[R] = (int32_t)run;
        memset(sc, 0, sizeof(int64_t) * (size_t)R * R);
        memset(st, 0, sizeof(int64_t) * 4);
        memset(td, 0, sizeof(uint64_t) * (size_t)T * RW);
        /* rows in token order within each rank */
        for (int t = 0; t < T; t++) {
            const int s = src[t];
            for (int r = 0; r < R; r++) mask[r] = 0;
            for (int j = 0; j < k; j++) mask[d[(int64_t)t * k + j] / n_local] |= (uint64_t)1 << j;
            for (int r = 0; r < R; r++) {
                if (!mask[r]) continue;
                rt[fill[r]] = t;
                rs[fill[r]] = mask[r];
                fill[r]++;
                td[(int64_t)t * RW + r / 64] |= (uint64_t)1 << (r % 64);
                sc[(int64_t)s * R + r]++;
                st[0]++;
                if (r != s) st[2]++;
            }
            for (int j = 0; j < k; j++)
                if (d[(int64_t)t * k + j] / n_local != s) st[3]++;
        }
        st[1] = npairs;
    }
    free(fill);
    free(mask);
    free(src);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Token-shuffle targets [Zyphra, "Moving Tokens Toward Their Next Experts": */
/* the experts a token selected at one layer predict which GPU holds most of */
/* its next experts, and the token is moved there before the next router].   */
/* Readings: the prediction for layer l+1 uses layer l's ids and the         */
/* transition counts tr_l (O2); the rank of an expert is its main rank       */
/* (main_rank map, or e / (E/R) when NULL);                                  */
/*   M_l[a][r]   = sum over experts b on rank r of tr_l[a][b],               */
/*   score_r(t)  = sum over the token's slots j of M_l[ids_l[t][j]][r],       */
/*   target_l[t] = the rank of the largest score; on a tie the token's own    */
/*                 source rank src(t) if it is among the largest, else the    */
/*                 lowest such rank.                                          */
/* stats_l = {next-layer pairs whose expert is on target_l[t], next-layer    */
/* pairs whose expert is on src(t), tokens with target != src, pairs}.       */
/* ------------------------------------------------------------------------ */

int oracle_shuffle(int L, int T, int E, int k, int R, const int32_t *ids, const int64_t *tr,
                   const int32_t *main_rank, const int64_t *rank_offsets, int32_t *target,
                   int64_t *stats) {
    if (L < 0 || T < 0 || E < 1 || k < 1 || R < 1 || (!main_rank && E % R != 0)) return ORC_EINVAL;
    int rc = ORC_OK;
    int32_t *src = sources_or_null(T, R, rank_offsets);
    if (!src) return ORC_EINVAL;
    int32_t *rank_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int64_t *M = (int64_t *)malloc(sizeof(int64_t) * (size_t)E * R);
    int64_t *score = (int64_t *)malloc(sizeof(int64_t) * (size_t)R);
    if (!rank_of || !M || !score) { free(rank_of); free(M); free(score); free(src); return ORC_EINVAL; }
    for (int e = 0; e < E; e++) {
        rank_of[e] = main_rank ? main_rank[e] : e / (E / R);
        if (rank_of[e] < 0 || rank_of[e] >= R) { free(rank_of); free(M); free(score); free(src); return ORC_EINVAL; }
    }
    for (int l = 0; l + 1 < L; l++) {
        const int64_t *t_l = tr + (int64_t)l * E * E;
        const int32_t *cur = ids + (int64_t)l * T * k, *nxt = ids + (int64_t)(l + 1) * T * k;
        int64_t *st = stats + (int64_t)l * 4;
        memset(M, 0, sizeof(int64_t) * (size_t)E * R);
        for (int a = 0; a < E; a++)
            for (int b = 0; b < E; b++) M[(int64_t)a * R + rank_of[b]] += t_l[(int64_t)a * E + b];
        memset(st, 0, sizeof(int64_t) * 4);
        for (int t = 0; t < T; t++) {
            int s = src[t];
            for (int r = 0; r < R; r++) score[r] = 0;
            for (int j = 0; j < k; j++) {
                int a = cur[(int64_t)t * k + j];
                if (a < 0 || a >= E) { rc = ORC_ERANGE; continue; }
                for (int r = 0; r < R; r++) score[r] += M[(int64_t)a * R + r];
            }
            int64_t mx = score[0];
            for (int r = 1; r < R; r++)
                if (score[r] > mx) mx = score[r];
            int best = s;
            if (score[s] != mx) {
                best = 0;
                while (score[best] != mx) best++;
            }
            target[(int64_t)l * T + t] = best;
            if (best != s) st[2]++;
            for (int j = 0; j < k; j++) {
                int b = nxt[(int64_t)t * k + j];
                if (b < 0 || b >= E) { rc = ORC_ERANGE; continue; }
                if (rank_of[b] == best) st[0]++;
                if (rank_of[b] == s) st[1]++;
                st[3]++;
            }
        }
    }
    free(rank_of); free(M); free(score); free(src);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Correlated expert placement [Zyphra, "Moving Correlated Experts           */
/* Together": the co-selection counts form a graph over experts, which is    */
/* partitioned across GPUs with a fixed number of experts per GPU so that    */
/* frequently co-selected experts share a GPU].  The pages give no           */
/* algorithm.  Readings: the weight of a pair is w(a,b) = co[a][b] +         */
/* co[b][a] (a != b; the diagonal is ignored).  Greedy construction: ranks   */
/* r = 0..R-1 in turn take E/R experts: first the unassigned expert with the */
/* largest total weight, then repeatedly the unassigned expert with the      */
/* largest weight to the rank's members.  Refinement: while some swap of two */
/* experts on different ranks raises the within-rank weight, apply the best  */
/* one (gain C[a][rb] - C[a][ra] + C[b][ra] - C[b][rb] - 2 w(a,b), with      */
/* C[x][r] the weight of x to rank r's members), at most max_iters swaps     */
/* when max_iters > 0 and never more than 2^20 (a bound on time).  Every     */
/* choice takes the lowest index on ties (a before b for swaps, a < b).      */
/* stats = {within-rank weight of the contiguous map e / (E/R), after the    */
/* greedy construction, final, swaps}.                                       */
/* ------------------------------------------------------------------------ */

static int64_t place_within(int E, const int64_t *w, const int32_t *part) {
    int64_t s = 0;
    for (int a = 0; a < E; a++)
        for (int b = a + 1; b < E; b++)
            if (part[a] == part[b]) s += w[(int64_t)a * E + b];
    return s;
}

int oracle_place(int L, int E, int R, int max_iters, const int64_t *co, int32_t *main_rank,
                 int64_t *stats) {
    if (L < 0 || E < 1 || R < 1 || E % R != 0 || max_iters < 0) return ORC_EINVAL;
    int per = E / R;
    int64_t *w = (int64_t *)malloc(sizeof(int64_t) * (size_t)E * E);
    int64_t *C = (int64_t *)malloc(sizeof(int64_t) * (size_t)E * R);
    int32_t *part = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!w || !C || !part) { free(w); free(C); free(part); return ORC_EINVAL; }
    for (int l = 0; l < L; l++) {
        const int64_t *c = co + (int64_t)l * E * E;
        int32_t *mr = main_rank + (int64_t)l * E;
        int64_t *st = stats + (int64_t)l * 4;
        for (int a = 0; a < E; a++)
            for (int b = 0; b < E; b++)
                w[(int64_t)a * E + b] = a == b ? 0 : c[(int64_t)a * E + b] + c[(int64_t)b * E + a];
        for (int e = 0; e < E; e++) part[e] = e / per;
        st[0] = place_within(E, w, part);
        /* greedy construction */
        for (int e = 0; e < E; e++) part[e] = -1;
        for (int r = 0; r < R; r++) {
            int seed = -1;
            int64_t best = 0;
            for (int a = 0; a < E; a++) {
                if (part[a] >= 0) continue;
                int64_t tot = 0;
                for (int b = 0; b < E; b++) tot += w[(int64_t)a * E + b];
                if (seed < 0 || tot > best) { seed = a; best = tot; }
            }
            part[seed] = r;
            for (int n = 1; n < per; n++) {
                int pick = -1;
                int64_t bc = 0;
                for (int b = 0; b < E; b++) {
                    if (part[b] >= 0) continue;
                    int64_t conn = 0;
                    for (int m = 0; m < E; m++)
                        if (part[m] == r) conn += w[(int64_t)m * E + b];
                    if (pick < 0 || conn > bc) { pick = b; bc = conn; }
                }
                part[pick] = r;
            }
        }
        st[1] = place_within(E, w, part);
        /* swap refinement */
        for (int x = 0; x < E; x++) {
            for (int r = 0; r < R; r++) C[(int64_t)x * R + r] = 0;
            for (int m = 0; m < E; m++) C[(int64_t)x * R + part[m]] += w[(int64_t)x * E + m];
        }
        int64_t swaps = 0;
        while ((max_iters == 0 || swaps < max_iters) && swaps < (1 << 20)) {
            int ba = -1, bb = -1;
            int64_t bg = 0;
            for (int a = 0; a < E; a++)
                for (int b = a + 1; b < E; b++) {
                    int pa = part[a], pb = part[b];
                    if (pa == pb) continue;
                    int64_t g = C[(int64_t)a * R + pb] - C[(int64_t)a * R + pa] + C[(int64_t)b * R + pa] -
                                C[(int64_t)b * R + pb] - 2 * w[(int64_t)a * E + b];
                    if (g > bg) { bg = g; ba = a; bb = b; }
                }
            if (ba < 0) break;
            int pa = part[ba], pb = part[bb];
            for (int x = 0; x < E; x++) {
                C[(int64_t)x * R + pa] += w[(int64_t)x * E + bb] - w[(int64_t)x * E + ba];
                C[(int64_t)x * R + pb] += w[(int64_t)x * E + ba] - w[(int64_t)x * E + bb];
            }
            part[ba] = pb;
            part[bb] = pa;
            swaps++;
        }
        st[2] = place_within(E, w, part);
        st[3] = swaps;
        for (int e = 0; e < E; e++) mr[e] = part[e];
    }
    free(w); free(C); free(part);
    return ORC_OK;
}
