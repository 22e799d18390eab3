/*
 * topo.h -- C ABI of the GB300 topology-aware expert-routing plan library
 * (libtopoep.so, sm_103a).
 *
 * The library turns one MoE layer's Top-k routing result (T tokens x k int32
 * expert ids) into a deterministic, topology-aware expert-parallel plan, as
 * defined in "TopoEP: Topology-Aware Load Balancing for Expert-Parallel MoE
 * Training" (§4.1 system model, §4.2 constraints C1-C5, §4.3 two-stage solver)
 * and, for the correlation statistics, "Expert Coupling in MoE Pretraining".
 *
 * Model.  R expert-parallel ranks form M = R / ranks_per_node NVLink domains
 * (dom(r) = r / ranks_per_node).  Each rank routes its own local tokens
 * (TopoEP §2.1): the tokens of a layer are the ranks' blocks one after the
 * other, token t belonging to source rank src(t) = the s with
 * rank_offsets[s] <= t < rank_offsets[s+1] (equal blocks of T / R tokens
 * when rank_offsets is NULL).  Pair p = t*k + j is the
 * j-th expert choice of token t.  Expert e has its main instance on rank
 * main(e) (= e / (E/R) by default, or main_rank[e]) with local index l < E/R
 * (ascending e among the rank's mains); each rank also has n_slot replica
 * slots, local indices E/R .. E/R+n_slot-1.  n_local = E/R + n_slot.  An
 * instance is packed as r*n_local + l.  The per-byte communication cost is
 * c(s,r) = 0 if s == r, c_intra inside a domain, c_inter across domains.
 *
 * Conventions for every call.
 *   - Pointers named "device" are device memory; the caller allocates every
 *     buffer, including the workspace ws.  The library never allocates,
 *     frees or synchronises; each call only enqueues kernels on `stream`.
 *   - n_layers independent problems (layers or microbatches) are handled per
 *     call; array arguments are stacked with layer as the slowest dimension.
 *   - Outputs are fully overwritten.
 *   - k <= 64; the shared-memory budget bounds E (about 2000 for R = 128).
 *   - Host-detectable problems return a negative code before anything is
 *     enqueued.  Problems only the device can see (an id outside [0, E), a
 *     workspace that does not hold what the call needs) set a sticky error
 *     word in ws; outputs are then unspecified.  Read it with
 *     topo_read_error after synchronising.  No kernel traps or asserts.
 *   - All results are integers and are bit-for-bit deterministic.
 *   - Thread safety: calls on distinct workspaces are independent.
 */
#ifndef TOPO_H
#define TOPO_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return / error-word codes. */
#define TOPO_OK 0
#define TOPO_EINVAL (-1)   /* bad argument: dimension, divisibility, NULL, range */
#define TOPO_ENOSPC (-2)   /* ws_bytes smaller than topo_workspace_bytes() */
#define TOPO_ECUDA (-3)    /* a CUDA runtime call or launch failed */
#define TOPO_ERANGE (-4)   /* device: an expert id outside [0, E) */
#define TOPO_ESTATE (-5)   /* device: ws does not hold the index this call needs */
#define TOPO_EMAP (-6)     /* device: main_rank is not a balanced map onto [0, R) */
#define TOPO_EOFFSETS (-7) /* device: rank_offsets is not 0 = o[0] <= o[1] <= ... <= o[R] = T */
#define TOPO_ETIMEOUT (-8) /* device: a bounded wait inside a kernel expired */

/* Workspace needs per call (argument `which_call` of topo_workspace_bytes). */
#define TOPO_CALL_HIST 0
#define TOPO_CALL_PLAN 1
#define TOPO_CALL_REROUTE 2
#define TOPO_CALL_LAYOUT 3
#define TOPO_CALL_COOCCUR 4
#define TOPO_CALL_CHAIN 5   /* hist -> plan -> reroute -> dispatch_layout on one ws */
#define TOPO_CALL_REROUTE_LAYOUT 6
#define TOPO_CALL_PACK 7    /* topo_permute, topo_combine */
#define TOPO_CALL_DEDUP 8   /* topo_dedup_layout */
#define TOPO_DEDUP_STATS 4  /* int64 deduplicated-layout statistics per layer */
#define TOPO_CALL_GATE 9    /* topo_gate_hist (the chain's workspace) */
#define TOPO_DTYPE_F32 0    /* logits as float32 */
#define TOPO_DTYPE_BF16 1   /* logits as bf16 bit patterns */
#define TOPO_GATE_MAX_E 1024
#define TOPO_SHUFFLE_STATS 4
#define TOPO_SHUFFLE_MAX_RANKS 256
#define TOPO_PLACE_STATS 4

#define TOPO_STATS 8        /* int64 plan statistics per layer */
#define TOPO_LAYOUT_STATS 8 /* int64 layout statistics per layer */

/* Problem configuration (TopoEP §4.1: N_slot, C, S_tok, ||W_e||, main(e)). */
typedef struct {
    int32_t T;                /* tokens per layer; T >= 0, T*k <= 2^31-1; T % R == 0
                                 when rank_offsets is NULL */
    int32_t E;                /* logical experts; E % R == 0, E < 2^26 */
    int32_t k;                /* expert choices per token (Top-k), 1..64 */
    int32_t R;                /* expert-parallel ranks; R % ranks_per_node == 0 */
    int32_t ranks_per_node;   /* ranks per NVLink domain, 1..32 */
    int32_t n_slot;           /* replica slots per rank (C3), >= 0; R*n_slot <= 2^20
                                 and E/R + n_slot <= 32767 */
    int64_t tok_bytes;        /* S_tok: bytes of one routed activation, >= 0,
                                 tok_bytes * c_inter < 2^31 */
    int64_t expert_bytes;     /* ||W_e||: parameter bytes of one expert, >= 0,
                                 expert_bytes * c_inter < 2^40 (so every cost
                                 product is exact in int64) */
    int32_t c_intra;          /* integer per-byte cost inside a domain, >= 1 */
    int32_t c_inter;          /* integer per-byte cost across domains, >= c_intra */
    int32_t max_refine_iters; /* cap on refinement commits per domain, >= 0; 0 = none */
    int32_t reserved;         /* must be 0 */
    const int32_t *main_rank; /* device [E] main rank of each expert, or NULL for
                                 e / (E/R); each rank must own exactly E/R mains */
    const int64_t *rank_offsets; /* device int64 [R+1] token offsets of the source
                                 ranks' blocks (the same for every layer), or NULL
                                 for equal blocks of T / R tokens.  Must satisfy
                                 0 = o[0] <= o[1] <= ... <= o[R] = T; a source may
                                 be empty.  Checked on the device by the calls that
                                 read tokens (topo_hist, topo_gate_hist,
                                 topo_dedup_layout; TOPO_EOFFSETS).  The calls of one
                                 chain must be given the same pointer. */
} topo_cfg;
/* A cfg that breaks one of these rules, or whose E, R, ranks_per_node and
 * n_slot exceed the kernels' shared memory (227 KB per CTA), is invalid:
 * topo_workspace_bytes returns 0 and every call returns TOPO_EINVAL. */

/* Plan outputs (TopoEP §4.2 decision variables x and q, loads U and L).
 * All device pointers, caller-allocated, layer-major. */
typedef struct {
    int32_t *slot_expert;  /* [L][R][n_slot] expert in each replica slot, -1 empty
                              (x_{e,r} for replicas; mains are implicit, C5);
                              may be NULL when n_slot == 0 */
    int32_t *route_cnt;    /* [L][R][R][n_local] q: assignments from source s
                              executed on instance (r, l) */
    int32_t *inst_load;    /* [L][R][n_local] U: load of each instance */
    int32_t *rank_load;    /* [L][R] L_r: load of each rank */
    int64_t *stats;        /* [L][TOPO_STATS]: 0 L_max, 1 L_max of the static
                              placement, 2 replicas, 3 replicas from inter-node
                              placement, 4 refinement commits, 5 T_token,
                              6 T_replica (Eq. 7 in the integer cost units),
                              7 sum_r L_r */
} topo_plan_t;

/* Bytes of workspace a call needs.  One workspace of
 * topo_workspace_bytes(cfg, n_layers, TOPO_CALL_CHAIN) serves the whole chain
 * hist -> plan -> reroute -> dispatch_layout; TOPO_CALL_COOCCUR needs only the
 * header (cfg may then be NULL).  Returns 0 for an invalid cfg. */
size_t topo_workspace_bytes(const topo_cfg *cfg, int32_t n_layers, int32_t which_call);

 /* Clear the workspace header (error word and the indices' fingerprints;
 * nothing else).  Call once on a fresh workspace and after reading an error.
 * ws: device, at least TOPO_CALL_COOCCUR bytes. */
int topo_ws_reset(void *ws, size_t ws_bytes, cudaStream_t stream);

/* Routing matrix Omega [TopoEP §4.1, Eq. 3]:
 *   hist[l][s][e] = #pairs of layer l whose token belongs to source rank s
 *                   and whose expert is e.
 * ids:  device int32 [n_layers][T][k].
 * hist: device int32 [n_layers][R][E].
 * ws:   device; also receives the per-tile expert-count index that
 *       topo_reroute and topo_dispatch_layout read for these ids.
 * Device errors: TOPO_ERANGE (the id is skipped), TOPO_EOFFSETS (nothing is
 * counted). */
int topo_hist(const topo_cfg *cfg, int32_t n_layers, const int32_t *ids, int32_t *hist,
              void *ws, size_t ws_bytes, cudaStream_t stream);

/* Top-k gating fused with the routing matrix [TopoEP §2.1: per token the
 * router selects the Top-k experts; §6.4: synthetic routing from random
 * logits with a fixed expert-specific bias; Omega as in topo_hist].
 * Readings: score[t][e] = logit[t][e] + bias[e] (one float addition; no bias
 * when bias is NULL); ids[t] = the k experts of the largest scores, in
 * descending order; equal scores (-0 equals +0) go to the lower expert; a NaN
 * score ranks below every number.
 * logits: device [n_layers][T][E], float32 (TOPO_DTYPE_F32) or bf16 bit
 *         patterns (TOPO_DTYPE_BF16), aligned to its element size.
 * bias:   device float32 [E] or NULL.
 * ids:    device int32 [n_layers][T][k] (written).
 * scores: device float32 [n_layers][T][k], the raw logits of the selected
 *         experts, or NULL.
 * hist:   device int32 [n_layers][R][E] (written, as topo_hist for ids).
 * ws:     >= topo_workspace_bytes(cfg, n_layers, TOPO_CALL_GATE); receives the
 *         tile index of ids, so topo_reroute / topo_reroute_layout may follow.
 * Requires k <= E <= TOPO_GATE_MAX_E (else TOPO_EINVAL).  No device errors. */
int topo_gate_hist(const topo_cfg *cfg, int32_t n_layers, const void *logits, int32_t logits_dtype,
                   const float *bias, int32_t *ids, float *scores, int32_t *hist, void *ws,
                   size_t ws_bytes, cudaStream_t stream);

/* Token-shuffle targets ["Expert Coupling in MoE Pretraining", "Moving Tokens
 * Toward Their Next Experts": a token's experts at one layer predict the GPU
 * holding most of its next experts, and the token is moved there before the
 * next router runs].  For each layer l < L-1 and token t:
 *   M_l[a][r]   = sum of tr[l][a][b] over experts b with main rank r,
 *   score_r     = sum over the token's slots j of M_l[ids[l][t][j]][r],
 *   target[l][t] = the best rank; a tie keeps the token on its source rank
 *                 src(t) if that rank is among the best, else the lowest.
 * ids:       device int32 [L][T][k].
 * tr:        device int64 [L-1][E][E] (topo_cooccur's transitions, or counts
 *            gathered elsewhere); the sums must fit int64.
 * main_rank: device int32 [E] (experts per rank need not be equal here) or
 *            NULL for e / (E/R).
 * rank_offsets: device int64 [R+1] source blocks as in topo_cfg, or NULL for
 *            equal blocks of T / R tokens.
 * target:    device int32 [L-1][T] (written).
 * stats:     device int64 [L-1][TOPO_SHUFFLE_STATS]: next-layer pairs whose
 *            expert is on the target, next-layer pairs on the source rank,
 *            tokens whose target is not their source, next-layer pairs.
 * ws:        >= topo_shuffle_workspace_bytes(L, E, R).
 * Requires T % R == 0 without rank_offsets, 1 <= R <= TOPO_SHUFFLE_MAX_RANKS,
 * 1 <= k <= 64, and E % R == 0 without a map.  Device errors: TOPO_ERANGE (an
 * id outside [0, E), skipped), TOPO_EMAP (a map entry outside [0, R),
 * skipped), TOPO_EOFFSETS (rank_offsets out of order). */
size_t topo_shuffle_workspace_bytes(int32_t L, int32_t E, int32_t R);
int topo_shuffle_targets(int32_t L, int32_t T, int32_t E, int32_t k, int32_t R, const int32_t *ids,
                         const int64_t *tr, const int32_t *main_rank, const int64_t *rank_offsets,
                         int32_t *target, int64_t *stats, void *ws, size_t ws_bytes,
                         cudaStream_t stream);

/* Correlated expert placement ["Expert Coupling in MoE Pretraining", "Moving
 * Correlated Experts Together": the co-selection graph partitioned across
 * GPUs with a fixed number of experts per GPU, co-selected experts kept
 * together].  Readings (the pages give no algorithm): w(a,b) = co[a][b] +
 * co[b][a] for a != b; greedy construction, ranks r = 0..R-1 in turn taking
 * E/R experts -- the unassigned expert of largest total weight, then
 * repeatedly the unassigned expert of largest weight to the rank's members;
 * then, while the best swap of two experts on different ranks raises the
 * within-rank weight, apply it (at most max_iters swaps when max_iters > 0,
 * and never more than 2^20).
 * Lowest index on every tie.
 * co:        device int64 [L][E][E] (topo_cooccur's co-selection counts).
 * main_rank: device int32 [L][E] (written): a map for topo_cfg.main_rank.
 * stats:     device int64 [L][TOPO_PLACE_STATS]: within-rank weight of the
 *            contiguous map e / (E/R), after the greedy construction, final;
 *            swaps applied.
 * Requires E % R == 0, E <= 1024 and E * (R + 1.5) * 8 bytes of shared memory
 * within the device limit (else TOPO_EINVAL).  No device errors. */
int topo_place_experts(int32_t L, int32_t E, int32_t R, int32_t max_iters, const int64_t *co,
                       int32_t *main_rank, int64_t *stats, cudaStream_t stream);

/* Expert co-selection and cross-layer transition counts ["Expert Coupling in
 * MoE Pretraining": within-layer correlation, cross-layer correlation]:
 *   co[l][a][b] = sum_t n_t^l[a] * n_t^l[b]
 *   tr[l][a][b] = sum_t n_t^l[a] * n_t^{l+1}[b]      (l < L-1)
 * where n_t^l is the count vector of token t's ids at layer l (the diagonal
 * of co is each expert's load).
 * ids: device int32 [L][T][k]; co: device int64 [L][E][E];
 * tr: device int64 [L-1][E][E] or NULL.  ws: >= TOPO_CALL_COOCCUR bytes.
 * Device errors: TOPO_ERANGE. */
int topo_cooccur(int32_t L, int32_t T, int32_t E, int32_t k, const int32_t *ids, int64_t *co,
                 int64_t *tr, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Workspace that lets topo_cooccur run on the tensor cores: the counts are
 * the contractions co_l = C_l^T C_l and tr_l = C_l^T C_{l+1} of the T x E
 * count matrices, computed by tcgen05.mma on count tiles (exact: counts are
 * small integers and every per-tile sum stays below 2^24 in the float32
 * accumulator) when E <= 128 and k <= 16.  It holds the header and int32
 * partial matrices of about 152 token chunks; with a smaller workspace
 * (TOPO_CALL_COOCCUR bytes) topo_cooccur counts with integer shared-memory
 * atomics instead, with the same results.  Device errors of the tensor-core
 * path: TOPO_ERANGE (the id is dropped), TOPO_ETIMEOUT (a bounded wait for
 * the tensor core expired; outputs unspecified). */
size_t topo_cooccur_workspace_bytes(int32_t L, int32_t T, int32_t E, int32_t k);

/* Two-stage topology-aware replication plan [TopoEP §4.3, Eqs. 9-10], one per
 * layer of hist (device int32 [n_layers][R][E]), following these rules:
 *  1. Demand D_{d,e} = sum of hist rows of domain d (Eq. 4).
 *  2. Inter-node placement (Eq. 9): per domain, experts whose main is outside
 *     the domain with b = 2 D S_tok - ||W|| > 0, in descending b (ties: lower
 *     e), each placed on the domain's rank with the fewest used slots (ties:
 *     lower rank); the domain stops when its slots are full.
 *  3. Routing: each (s, e) is split over e's instances in dom(s), or over all
 *     of e's instances if dom(s) has none: floor share each, the remainder one
 *     apiece to the first instances in ascending (c(s,r), r).
 *  4. Intra-node refinement (Eq. 10): per domain, repeatedly take the busiest
 *     rank r_b (ties: lower rank) and, over its experts e and the other ranks
 *     r_t of the domain that host e or have a free slot, the move of
 *     delta = min(U, floor((L_b - L_t)/2)) >= 1 assignments that is best by
 *     (delta desc, L_t asc, cost asc, e asc, r_t asc), where the moved
 *     assignments come from sources in ascending (c(s,r_t) - c(s,r_b), s) and
 *     cost is the resulting change of T_token + T_replica (Eq. 7); stop when
 *     r_b has no such move or after max_refine_iters commits.
 * Outputs: *plan (all fields required).  ws: TOPO_CALL_PLAN bytes.
 * Device errors: TOPO_EMAP. */
int topo_plan(const topo_cfg *cfg, int32_t n_layers, const int32_t *hist, const topo_plan_t *plan,
              void *ws, size_t ws_bytes, cudaStream_t stream);

/* Rerouting of every (token, slot) pair to an expert instance [TopoEP §1,
 * Fig. 5 "token rerouting"; the rule is this library's reading]: within
 * source s, the pairs selecting e are taken in ascending pair order and fill
 * e's instances in ascending rank order, q[s][r][l] pairs each.
 *   dst_inst[l][p] = r*n_local + l_inst.
 * ids: device int32 [n_layers][T][k], the same ids (same pointer) that
 * topo_hist indexed into this ws.  plan: from topo_plan (or any plan whose
 * route_cnt rows sum to hist).  dst_inst: device int32 [n_layers][T*k].
 * ws: TOPO_CALL_REROUTE bytes; receives the routing index that
 * topo_dispatch_layout reads.  Device errors: TOPO_ESTATE (no index for these
 * ids in ws), TOPO_ERANGE. */
int topo_reroute(const topo_cfg *cfg, int32_t n_layers, const int32_t *ids, const topo_plan_t *plan,
                 int32_t *dst_inst, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Dispatch layout [TopoEP §5: receive counts derived on the GPU; §2.3 Fig. 3
 * byte accounting]:
 *   sorted_pairs[l][pos]: pair indices stably sorted by dst_inst (gather form);
 *   seg_off[l][i]: start of instance i's segment, [n_layers][R*n_local + 1];
 *   send_counts[l][s][r]: pairs from source s to rank r, int64 [n_layers][R][R];
 *   layout_stats[l][8]: pairs with s == r, same domain, other domain; their
 *     dispatch bytes (pairs * tok_bytes); pairs served by a replica; 0.
 * dst_inst must be topo_reroute's output for this plan on this ws: topo_reroute
 * already ranked every pair and left its position in ws, so this call only
 * scatters (checked: TOPO_ESTATE otherwise).  All output pointers required. */
int topo_dispatch_layout(const topo_cfg *cfg, int32_t n_layers, const int32_t *dst_inst,
                         const topo_plan_t *plan, int32_t *sorted_pairs, int32_t *seg_off,
                         int64_t *send_counts, int64_t *layout_stats, void *ws, size_t ws_bytes,
                         cudaStream_t stream);

/* topo_reroute followed by topo_dispatch_layout in one pass over the pairs:
 * the same dst_inst, sorted_pairs, seg_off, send_counts and layout_stats, with
 * each pair read once and no per-pair positions kept in ws.  Same arguments
 * and requirements as the two calls (ids indexed by topo_hist on this ws).
 * Device errors: TOPO_ESTATE, TOPO_ERANGE. */
int topo_reroute_layout(const topo_cfg *cfg, int32_t n_layers, const int32_t *ids,
                        const topo_plan_t *plan, int32_t *dst_inst, int32_t *sorted_pairs,
                        int32_t *seg_off, int64_t *send_counts, int64_t *layout_stats, void *ws,
                        size_t ws_bytes, cudaStream_t stream);

/* Deduplicated dispatch layout ["Expert Coupling in MoE Pretraining",
 * "Moving Correlated Experts Together": a token goes to a destination rank
 * once, with metadata naming the local experts that process it; "MoX:
 * Efficient MoE Routing on Direct-Connect Topologies" §2: a per-token
 * destination bitmap].  Readings: one row per (token, destination rank), the
 * destination rank of a pair being dst_inst / n_local; rows ordered by rank,
 * then by token; a row's metadata is the mask of the token's slots on that
 * rank (bit j = slot j).
 * dst_inst:  device int32 [n_layers][T*k] (topo_reroute, topo_reroute_layout).
 * seg:       device int32 [n_layers][R+1] row offsets per destination rank.
 * row_token: device int32 [n_layers][T*k]; row_slots: device uint64
 *            [n_layers][T*k] (the first seg[R] entries of a layer are used).
 * tok_dst:   device uint64 [n_layers][T][ceil(R/64)] destination-rank bitmap.
 * send:      device int64 [n_layers][R][R] rows from source s to rank r.
 * stats:     device int64 [n_layers][TOPO_DEDUP_STATS]: rows, pairs, rows to
 *            another rank, pairs to another rank.
 * Requires k <= 16 and R <= 1024 (else TOPO_EINVAL).
 * ws: >= topo_workspace_bytes(cfg, n_layers, TOPO_CALL_DEDUP) bytes.
 * Device errors: TOPO_ESTATE for a dst_inst value outside [0, R*n_local),
 * TOPO_EOFFSETS. */
int topo_dedup_layout(const topo_cfg *cfg, int32_t n_layers, const int32_t *dst_inst, int32_t *seg,
                      int32_t *row_token, uint64_t *row_slots, uint64_t *tok_dst, int64_t *send,
                      int64_t *stats, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Dispatch pack [TopoEP Fig. 1: dispatch sends each token's activation to the
 * ranks hosting its selected experts].  Reading: the send buffer holds the
 * pairs' rows in layout order, so each destination instance's rows are one
 * contiguous segment (seg_off):
 *   y[l][pos][:] = x[l][sorted_pairs[l][pos] / k][:]
 * x:  device bf16 (16-bit patterns) [n_layers][T][H], 16-byte aligned.
 * y:  device bf16 [n_layers][T*k][H], 16-byte aligned.
 * H:  elements per row, a positive multiple of 8 (16-byte rows).
 * sorted_pairs: device int32 [n_layers][T*k] from topo_dispatch_layout or
 *     topo_reroute_layout (a permutation of the pairs).
 * ws: >= topo_workspace_bytes(cfg, n_layers, TOPO_CALL_PACK) bytes (the
 *     inverse permutation).  Rows are copied bit for bit.
 * Device errors: TOPO_ESTATE when sorted_pairs is not a permutation (the
 * affected tokens are skipped). */
int topo_permute(const topo_cfg *cfg, int32_t n_layers, int32_t H, const uint16_t *x,
                 const int32_t *sorted_pairs, uint16_t *y, void *ws, size_t ws_bytes,
                 cudaStream_t stream);

/* Combine ["MoX: Efficient MoE Routing on Direct-Connect Topologies" §2.4:
 * combine reduces the token's top-K expert outputs into one vector].
 * Reading: the reduction is the gate-weighted sum of the expert outputs, in
 * float, in slot order, rounded once to bf16 (nearest, ties to even):
 *   out[l][t][:] = bf16( sum_{j=0..k-1} w[l][t][j] * y[l][pos(t, j)][:] )
 * where pos(t, j) is the position of pair t*k + j in sorted_pairs[l] and
 * each product and each sum is one float operation (no fused multiply-add).
 * y: device bf16 [n_layers][T*k][H]; w: device float [n_layers][T][k];
 * out: device bf16 [n_layers][T][H]; alignment, H and ws as topo_permute.
 * Device errors: TOPO_ESTATE as topo_permute. */
int topo_combine(const topo_cfg *cfg, int32_t n_layers, int32_t H, const uint16_t *y,
                 const int32_t *sorted_pairs, const float *w, uint16_t *out, void *ws,
                 size_t ws_bytes, cudaStream_t stream);

/* topo_hist without a caller-supplied workspace.  No passage of the pages
 * has a counterpart: it computes exactly what topo_hist computes (Omega), for
 * callers that cannot hand the library device memory on the step path -- C
 * or C++ hosts with no device allocator of their own, and processes that
 * reserve the device's memory up front, where a cudaMalloc during a step
 * would fail or would make a caching allocator release memory and
 * synchronise the device.
 *
 * Scratch: one fixed array of TOPO_HIST_NOALLOC_SCRATCH_BYTES per device,
 * compiled into the library; the call allocates nothing.  It holds a 256-byte
 * error header and the per-tile expert counts, n_layers * R *
 * tiles_per_source * E int32.  Shapes that need more return TOPO_ENOSPC
 * before anything runs.  Each call clears the header on `stream` before its
 * kernels (every tile count is rewritten).
 *
 * The first call on a device looks the array's address up (with that device
 * current) and caches it; make that first call before any stream capture.
 * All calls on one device share the array: calls that overlap in time (on
 * different streams, or from several host threads without ordering) race on
 * it and give undefined results.  The tile index left in the array is not
 * usable by topo_reroute or topo_dispatch_layout.
 *
 * ids:  device int32 [n_layers][T][k].   hist: device int32 [n_layers][R][E].
 * err:  device int32, or NULL; receives the call's device error word
 *       (TOPO_OK, or TOPO_ERANGE when an id lies outside [0, E), which is
 *       skipped), in stream order.
 * Returns TOPO_EINVAL / TOPO_ENOSPC on the host, TOPO_ECUDA if the lookup or a
 * launch fails. */
#define TOPO_HIST_NOALLOC_SCRATCH_BYTES (16u << 20)
int topo_hist_noalloc(const topo_cfg *cfg, int32_t n_layers, const int32_t *ids, int32_t *hist,
                      int32_t *err, cudaStream_t stream);

/* Synchronous: copies the error word out of ws (device) and returns it
 * (TOPO_OK or a negative code; TOPO_ECUDA if the copy fails).  Call after
 * the stream that used ws has been synchronised. */
int topo_read_error(const void *ws);

/* Static description of a code. */
const char *topo_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* TOPO_H */
