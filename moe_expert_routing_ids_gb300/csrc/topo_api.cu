// C-ABI entry points: argument validation, workspace layout, launches.
#include <cuda_runtime.h>

#include <climits>
#include <cstddef>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

using namespace topo;

namespace topo {

cudaError_t ensure_smem(const void *fn, size_t bytes) {
    // the default limit, 48 KB, covers a kernel's static and dynamic shared
    // memory together; beyond it the kernel must opt in
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, size_t> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    size_t &have = done[{fn, dev}];
    if (have >= bytes) return cudaSuccess;
    cudaFuncAttributes a;
    if ((e = cudaFuncGetAttributes(&a, fn)) != cudaSuccess) return e;
    if (a.sharedSizeBytes + bytes > 48 * 1024)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) have = bytes;
    return e;
}

}  // namespace topo

namespace {

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

// Validates cfg and fills the geometry (including the workspace layout).
int make_geo(const topo_cfg *c, int32_t n_layers, Geo *g) {
    if (!c || n_layers < 0) return TOPO_EINVAL;
    if (c->T < 0 || c->E < 1 || c->k < 1 || c->R < 1 || c->ranks_per_node < 1 || c->n_slot < 0)
        return TOPO_EINVAL;
    if (c->ranks_per_node > kMaxRanksPerNode) return TOPO_EINVAL;
    if (c->R % c->ranks_per_node || c->E % c->R) return TOPO_EINVAL;
    if (!c->rank_offsets && c->T % c->R) return TOPO_EINVAL;
    if ((int64_t)c->T * c->k > INT32_MAX) return TOPO_EINVAL;
    if (c->tok_bytes < 0 || c->expert_bytes < 0 || c->c_intra < 1 || c->c_inter < c->c_intra)
        return TOPO_EINVAL;
    if (c->max_refine_iters < 0 || c->reserved != 0) return TOPO_EINVAL;
    // keep every int64 cost product exact: S_tok*c < 2^31, ||W||*c < 2^40
    if (c->tok_bytes * (int64_t)c->c_inter >= (int64_t(1) << 31)) return TOPO_EINVAL;
    if (c->expert_bytes * (int64_t)c->c_inter >= (int64_t(1) << 40)) return TOPO_EINVAL;
    if ((int64_t)c->R * c->n_slot > (1 << 20)) return TOPO_EINVAL;
    if (c->k > kMaxK) return TOPO_EINVAL;
    // shared-memory capacity of the kernels (227 KB per CTA on sm_103a)
    const int64_t E = c->E, R = c->R, rpn = c->ranks_per_node;
    const int64_t nl = E / R + c->n_slot;
    if (nl > 32767) return TOPO_EINVAL;
    if ((2 * (R * nl + 3) + E + 4 + 2 * E) * 4 + 2560 > kSmemMax) return TOPO_EINVAL;       // row index
    if ((E * ((R + 31) / 32) + E + 4 + R * nl) * 4 + 8192 > kSmemMax) return TOPO_EINVAL;   // instance list
    if ((((2 * rpn + 4 * rpn * nl + (rpn * E + 1) / 2 + 3) & ~int64_t(3)) + rpn * nl * (rpn | 1)) * 4 >
        kSmemMax - 4096)
        return TOPO_EINVAL;                                                                 // refinement
    if (E >= (1 << 26)) return TOPO_EINVAL;
    int64_t npow = 2;                                                                       // placement sort
    while (npow < E) npow <<= 1;
    if (npow * 8 > kSmemMax) return TOPO_EINVAL;
    std::memset(g, 0, sizeof *g);
    g->T = c->T; g->E = c->E; g->k = c->k; g->R = c->R; g->rpn = c->ranks_per_node;
    g->n_slot = c->n_slot; g->M = c->R / c->ranks_per_node; g->E_R = c->E / c->R;
    g->n_local = (int32_t)nl; g->L = n_layers;
    g->c_intra = c->c_intra; g->c_inter = c->c_inter; g->max_iters = c->max_refine_iters;
    g->S_tok = c->tok_bytes; g->W = c->expert_bytes;
    g->roff = c->rank_offsets;
    // tokens per source: exact for equal blocks; with rank_offsets the
    // average, which only steers the tile size below
    g->tpr = c->rank_offsets ? (c->T + c->R - 1) / c->R : c->T / c->R;
    g->pps = (int64_t)g->tpr * c->k;
    g->npairs = (int64_t)c->T * c->k;
    g->kp = (c->k & 1) ? c->k : c->k + 1;
    g->kmagic = c->k == 1 ? 0u : (uint32_t)(((uint64_t(1) << 32) + c->k - 1) / c->k);
    // Tile geometry: RW rounds of 32 tokens per warp, within the shared-memory
    // budget of two rank CTAs per SM and about kTilePairsTarget pairs; among
    // the admissible RW take the one with the least work per source counting
    // a fixed per-tile cost of 1.5 rounds.
    const int64_t tables = E * (8 + 8 * kRankWarps) + (int64_t)kRankEntCap * 12;
    const int64_t round_bytes = (int64_t)kRankThreads * g->kp * 4;
    int64_t rw_max = kTilePairsTarget / ((int64_t)kRankThreads * c->k);
    const int64_t rw_smem = (kRankSmemTarget - tables) / round_bytes;
    if (rw_smem < rw_max) rw_max = rw_smem;
    if (rw_max < 1) {
        rw_max = 1;
        if (tables + round_bytes > kSmemMax - 1024) return TOPO_EINVAL;
    }
    const int64_t rw_need = (g->tpr + kRankThreads - 1) / kRankThreads;
    if (rw_max > rw_need && rw_need > 0) rw_max = rw_need;
    int64_t best_rw = 1;
    double best_cost = -1.0;
    for (int64_t rw = 1; rw <= rw_max; ++rw) {
        const int64_t tps = g->tpr == 0 ? 1 : (g->tpr + kRankThreads * rw - 1) / (kRankThreads * rw);
        const double cost = (double)tps * ((double)rw + 1.5);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_rw = rw; }
    }
    g->RW = (int32_t)best_rw;
    g->TT = kRankThreads * g->RW;
    g->tps = g->tpr == 0 ? 1 : (g->tpr + g->TT - 1) / g->TT;
    // tiles per layer: a source of n tokens holds ceil(n / TT) tiles, at most
    // n / TT + 1, so ceil(T / TT) + R bound them for any offsets
    g->ntl = c->rank_offsets ? (int32_t)((c->T + (int64_t)g->TT - 1) / g->TT + c->R) : c->R * g->tps;
    if ((int64_t)n_layers * g->ntl > INT32_MAX) return TOPO_EINVAL;
    g->n_inst_cap = c->E + c->R * c->n_slot;
    g->n_keys = c->R * g->n_local;
    const size_t L = (size_t)n_layers;
    const size_t tiles = L * (size_t)g->ntl;
    size_t off = sizeof(WsHeader);
    g->off_first = off; off = align_up(off + (size_t)(R + 1) * 4);
    g->off_tile = off;  off = align_up(off + tiles * E * 4);
    g->off_pos = off;   off = align_up(off + tiles * g->TT * c->k * 4);
    g->off_main = off;  off = align_up(off + 3 * E * 4);
    g->off_rep = off;   off = align_up(off + L * E * g->M * 4);
    g->off_iexp = off;  off = align_up(off + L * g->n_keys * 4);
    g->off_ioff = off;  off = align_up(off + L * (E + 1) * 4);
    g->off_ilist = off; off = align_up(off + L * g->n_keys * 4);
    g->off_roff = off;  off = align_up(off + L * R * (E + 1) * 4);
    g->off_rent = off;  off = align_up(off + L * R * g->n_inst_cap * 16);
    g->off_soff = off;  off = align_up(off + L * R * g->n_keys * 4);
    g->off_ccnt = off;  off = align_up(off + L * g->n_keys * 4);
    g->off_lseg = off;  off = align_up(off + L * (g->n_keys + 1) * 4);
    g->off_lsend = off; off = align_up(off + L * R * R * 8);
    g->off_lstat = off; off = align_up(off + L * TOPO_LAYOUT_STATS * 8);
    g->total = off;
    return TOPO_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? TOPO_OK : TOPO_ECUDA; }

// The per-call table of each source's first tile lives in the workspace.
void bind_ws(Geo &g, void *ws) { g.tfirst = ws_at<int32_t>(ws, g.off_first); }

uint64_t hist_fingerprint(const Geo &g, const int32_t *ids) {
    uint64_t h = fp_mix(0x48495354ull, (uint64_t)g.T);
    h = fp_mix(h, (uint64_t)g.E);
    h = fp_mix(h, (uint64_t)g.k);
    h = fp_mix(h, (uint64_t)g.R);
    h = fp_mix(h, (uint64_t)g.L);
    h = fp_mix(h, (uint64_t)g.tps);
    h = fp_mix(h, (uint64_t)(uintptr_t)g.roff);
    return fp_mix(h, (uint64_t)(uintptr_t)ids);
}

// Part of the routing-index fingerprint that does not depend on ws contents;
// the device mixes it with the stored hist fingerprint.
uint64_t route_fingerprint(const Geo &g, const topo_plan_t &p, const int32_t *dst,
                           const int32_t *main_rank) {
    uint64_t h = fp_mix(0x524f5554ull, (uint64_t)g.n_slot);
    h = fp_mix(h, (uint64_t)g.rpn);
    h = fp_mix(h, (uint64_t)(uintptr_t)p.slot_expert);
    h = fp_mix(h, (uint64_t)(uintptr_t)p.route_cnt);
    h = fp_mix(h, (uint64_t)(uintptr_t)p.inst_load);
    h = fp_mix(h, (uint64_t)(uintptr_t)main_rank);
    return fp_mix(h, (uint64_t)(uintptr_t)dst);
}

// slot_expert may be NULL only when there are no slots (a zero-size array).
bool plan_ok(const topo_plan_t *p, const Geo &g) {
    return p && (p->slot_expert || g.n_slot == 0 || g.L == 0) && p->route_cnt && p->inst_load &&
           p->rank_load && p->stats;
}

// Workspace of topo_permute / topo_combine: header + the inverse permutation.
size_t pack_ws_bytes(Geo &g) {
    g.off_pack_inv = sizeof(WsHeader);
    return align_up(g.off_pack_inv + (size_t)g.L * (size_t)g.npairs * 4);
}

int pack_args(const topo_cfg *cfg, int32_t n_layers, int32_t H, const void *in, const int32_t *sorted,
              const void *out, void *ws, size_t ws_bytes, Geo *g) {
    int rc = make_geo(cfg, n_layers, g);
    if (rc) return rc;
    if (H < 8 || H % 8) return TOPO_EINVAL;
    if (!ws) return TOPO_EINVAL;
    if (ws_bytes < pack_ws_bytes(*g)) return TOPO_ENOSPC;
    if (n_layers == 0 || g->npairs == 0) return TOPO_OK;
    if (!in || !sorted || !out) return TOPO_EINVAL;
    if (((uintptr_t)in | (uintptr_t)out) & 15) return TOPO_EINVAL;
    return TOPO_OK;
}

}  // namespace

extern "C" {

size_t topo_workspace_bytes(const topo_cfg *cfg, int32_t n_layers, int32_t which_call) {
    if (which_call == TOPO_CALL_COOCCUR) return sizeof(WsHeader);
    if (which_call < TOPO_CALL_HIST || which_call > TOPO_CALL_GATE) return 0;
    Geo g;
    if (make_geo(cfg, n_layers, &g) != TOPO_OK) return 0;
    if (which_call == TOPO_CALL_PACK) return pack_ws_bytes(g);
    if (which_call == TOPO_CALL_DEDUP) return dedup_ws_bytes(g, nullptr, nullptr, nullptr);
    return g.total;
}

int topo_ws_reset(void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!ws || ws_bytes < sizeof(WsHeader)) return TOPO_EINVAL;
    return cuda_rc(cudaMemsetAsync(ws, 0, sizeof(WsHeader), stream));
}

int topo_hist(const topo_cfg *cfg, int32_t n_layers, const int32_t *ids, int32_t *hist, void *ws,
              size_t ws_bytes, cudaStream_t stream) {
    Geo g;
    int rc = make_geo(cfg, n_layers, &g);
    if (rc) return rc;
    if (!hist || !ws || (!ids && g.npairs > 0 && n_layers > 0)) return TOPO_EINVAL;
    if (ws_bytes < g.total) return TOPO_ENOSPC;
    if (n_layers == 0) return TOPO_OK;
    bind_ws(g, ws);
    return cuda_rc(launch_hist(g, ids, hist, ws, hist_fingerprint(g, ids), stream));
}

int topo_gate_hist(const topo_cfg *cfg, int32_t n_layers, const void *logits, int32_t logits_dtype,
                   const float *bias, int32_t *ids, float *scores, int32_t *hist, void *ws,
                   size_t ws_bytes, cudaStream_t stream) {
    Geo g;
    int rc = make_geo(cfg, n_layers, &g);
    if (rc) return rc;
    if (logits_dtype != TOPO_DTYPE_F32 && logits_dtype != TOPO_DTYPE_BF16) return TOPO_EINVAL;
    if (cfg->k > cfg->E || cfg->E > TOPO_GATE_MAX_E) return TOPO_EINVAL;
    if (!hist || !ws || (g.npairs > 0 && n_layers > 0 && (!logits || !ids))) return TOPO_EINVAL;
    const uintptr_t esz = logits_dtype == TOPO_DTYPE_BF16 ? 2 : 4;
    if (((uintptr_t)logits % esz) || ((uintptr_t)bias | (uintptr_t)ids | (uintptr_t)scores) % 4)
        return TOPO_EINVAL;
    if (ws_bytes < g.total) return TOPO_ENOSPC;
    if (n_layers == 0) return TOPO_OK;
    bind_ws(g, ws);
    return cuda_rc(launch_gate(g, logits, logits_dtype == TOPO_DTYPE_BF16, bias, ids, scores, hist, ws,
                               hist_fingerprint(g, ids), stream));
}

int topo_place_experts(int32_t L, int32_t E, int32_t R, int32_t max_iters, const int64_t *co,
                       int32_t *main_rank, int64_t *stats, cudaStream_t stream) {
    if (L < 0 || E < 1 || E > kPlaceMaxE || R < 1 || E % R != 0 || max_iters < 0) return TOPO_EINVAL;
    if (place_smem_bytes(E, R) > kSmemMax) return TOPO_EINVAL;
    if (L == 0) return TOPO_OK;
    if (!co || !main_rank || !stats) return TOPO_EINVAL;
    return cuda_rc(launch_place(L, E, R, max_iters, co, main_rank, stats, stream));
}

size_t topo_shuffle_workspace_bytes(int32_t L, int32_t E, int32_t R) {
    if (L < 0 || E < 1 || R < 1 || R > TOPO_SHUFFLE_MAX_RANKS || E >= (1 << 26)) return 0;
    return shuffle_ws_bytes(L, E, R);
}

int topo_shuffle_targets(int32_t L, int32_t T, int32_t E, int32_t k, int32_t R, const int32_t *ids,
                         const int64_t *tr, const int32_t *main_rank, const int64_t *rank_offsets,
                         int32_t *target, int64_t *stats, void *ws, size_t ws_bytes,
                         cudaStream_t stream) {
    static_assert(TOPO_SHUFFLE_MAX_RANKS == kShuffleMaxRanks, "rank limit");
    if (L < 0 || T < 0 || E < 1 || E >= (1 << 26) || k < 1 || k > kMaxK || R < 1 ||
        R > TOPO_SHUFFLE_MAX_RANKS || (!rank_offsets && T % R != 0) || (!main_rank && E % R != 0))
        return TOPO_EINVAL;
    if ((int64_t)L * T * k > ((int64_t)1 << 40)) return TOPO_EINVAL;
    if (!ws) return TOPO_EINVAL;
    if (ws_bytes < shuffle_ws_bytes(L, E, R)) return TOPO_ENOSPC;
    if (L < 2) return TOPO_OK;
    if (!tr || !stats || (T > 0 && (!ids || !target))) return TOPO_EINVAL;
    return cuda_rc(launch_shuffle(L, T, E, k, R, ids, tr, main_rank, rank_offsets, target, stats, ws, stream));
}

int topo_plan(const topo_cfg *cfg, int32_t n_layers, const int32_t *hist, const topo_plan_t *plan,
              void *ws, size_t ws_bytes, cudaStream_t stream) {
    Geo g;
    int rc = make_geo(cfg, n_layers, &g);
    if (rc) return rc;
    if (!hist || !ws || !plan_ok(plan, g)) return TOPO_EINVAL;
    if (ws_bytes < g.total) return TOPO_ENOSPC;
    if (n_layers == 0) return TOPO_OK;
    return cuda_rc(launch_plan(g, cfg->main_rank, hist, *plan, ws, stream));
}

int topo_reroute(const topo_cfg *cfg, int32_t n_layers, const int32_t *ids, const topo_plan_t *plan,
                 int32_t *dst_inst, void *ws, size_t ws_bytes, cudaStream_t stream) {
    Geo g;
    int rc = make_geo(cfg, n_layers, &g);
    if (rc) return rc;
    if (!ws || !plan_ok(plan, g) || ((!ids || !dst_inst) && g.npairs > 0 && n_layers > 0))
        return TOPO_EINVAL;
    if (ws_bytes < g.total) return TOPO_ENOSPC;
    if (n_layers == 0) return TOPO_OK;
    bind_ws(g, ws);
    return cuda_rc(launch_reroute(g, cfg->main_rank, ids, *plan, dst_inst, ws, hist_fingerprint(g, ids),
                                  route_fingerprint(g, *plan, dst_inst, cfg->main_rank), stream));
}

int topo_dispatch_layout(const topo_cfg *cfg, int32_t n_layers, const int32_t *dst_inst,
                         const topo_plan_t *plan, int32_t *sorted_pairs, int32_t *seg_off,
                         int64_t *send_counts, int64_t *layout_stats, void *ws, size_t ws_bytes,
                         cudaStream_t stream) {
    Geo g;
    int rc = make_geo(cfg, n_layers, &g);
    if (rc) return rc;
    if (!ws || !plan_ok(plan, g) || !seg_off || !send_counts || !layout_stats) return TOPO_EINVAL;
    if ((!dst_inst || !sorted_pairs) && g.npairs > 0 && n_layers > 0) return TOPO_EINVAL;
    if (ws_bytes < g.total) return TOPO_ENOSPC;
    if (n_layers == 0) return TOPO_OK;
    bind_ws(g, ws);
    return cuda_rc(launch_layout(g, sorted_pairs, seg_off, send_counts, layout_stats, ws,
                                 route_fingerprint(g, *plan, dst_inst, cfg->main_rank), stream));
}

int topo_reroute_layout(const topo_cfg *cfg, int32_t n_layers, const int32_t *ids,
                        const topo_plan_t *plan, int32_t *dst_inst, int32_t *sorted_pairs,
                        int32_t *seg_off, int64_t *send_counts, int64_t *layout_stats, void *ws,
                        size_t ws_bytes, cudaStream_t stream) {
    Geo g;
    int rc = make_geo(cfg, n_layers, &g);
    if (rc) return rc;
    if (!ws || !plan_ok(plan, g) || !seg_off || !send_counts || !layout_stats) return TOPO_EINVAL;
    if ((!ids || !dst_inst || !sorted_pairs) && g.npairs > 0 && n_layers > 0) return TOPO_EINVAL;
    if (ws_bytes < g.total) return TOPO_ENOSPC;
    if (n_layers == 0) return TOPO_OK;
    bind_ws(g, ws);
    return cuda_rc(launch_reroute_layout(g, cfg->main_rank, ids, *plan, dst_inst, sorted_pairs, seg_off,
                                         send_counts, layout_stats, ws, hist_fingerprint(g, ids),
                                         stream));
}

size_t topo_cooccur_workspace_bytes(int32_t L, int32_t T, int32_t E, int32_t k) {
    if (L < 0 || T < 0 || E < 1 || k < 1) return 0;
    return cooccur_mma_ws_bytes(L, T, E, k);
}

int topo_cooccur(int32_t L, int32_t T, int32_t E, int32_t k, const int32_t *ids, int64_t *co,
                 int64_t *tr, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (L < 0 || T < 0 || E < 1 || k < 1 || !ws) return TOPO_EINVAL;
    if ((int64_t)T * k > INT32_MAX || (int64_t)E * E > INT32_MAX) return TOPO_EINVAL;
    if (L > 0 && !co) return TOPO_EINVAL;
    if (L > 0 && T > 0 && !ids) return TOPO_EINVAL;
    if (ws_bytes < sizeof(WsHeader)) return TOPO_ENOSPC;
    if (L == 0) return TOPO_OK;
    if (cooccur_mma_applies(L, T, E, k) && ws_bytes >= cooccur_mma_ws_bytes(L, T, E, k))
        return cuda_rc(launch_cooccur_mma(L, T, E, k, ids, co, L > 1 ? tr : nullptr, ws, stream));
    return cuda_rc(launch_cooccur(L, T, E, k, ids, co, L > 1 ? tr : nullptr, ws, stream));
}

int topo_dedup_layout(const topo_cfg *cfg, int32_t n_layers, const int32_t *dst_inst, int32_t *seg,
                      int32_t *row_token, uint64_t *row_slots, uint64_t *tok_dst, int64_t *send,
                      int64_t *stats, void *ws, size_t ws_bytes, cudaStream_t stream) {
    Geo g;
    int rc = make_geo(cfg, n_layers, &g);
    if (rc) return rc;
    if (cfg->k > kDedupMaxK || cfg->R > kDedupMaxRanks) return TOPO_EINVAL;
    if (!ws) return TOPO_EINVAL;
    if (ws_bytes < dedup_ws_bytes(g, nullptr, nullptr, nullptr)) return TOPO_ENOSPC;
    if (n_layers == 0) return TOPO_OK;
    if (!seg || !send || !stats || (g.npairs > 0 && (!dst_inst || !row_token || !row_slots || !tok_dst)))
        return TOPO_EINVAL;
    return cuda_rc(launch_dedup(g, dst_inst, seg, row_token, row_slots, tok_dst, send, stats, ws,
                                stream));
}

int topo_permute(const topo_cfg *cfg, int32_t n_layers, int32_t H, const uint16_t *x,
                 const int32_t *sorted_pairs, uint16_t *y, void *ws, size_t ws_bytes,
                 cudaStream_t stream) {
    Geo g;
    const int rc = pack_args(cfg, n_layers, H, x, sorted_pairs, y, ws, ws_bytes, &g);
    if (rc || n_layers == 0 || g.npairs == 0) return rc;
    return cuda_rc(launch_permute(g, H, x, sorted_pairs, y, ws, stream));
}

int topo_combine(const topo_cfg *cfg, int32_t n_layers, int32_t H, const uint16_t *y,
                 const int32_t *sorted_pairs, const float *w, uint16_t *out, void *ws,
                 size_t ws_bytes, cudaStream_t stream) {
    Geo g;
    const int rc = pack_args(cfg, n_layers, H, y, sorted_pairs, out, ws, ws_bytes, &g);
    if (rc || n_layers == 0 || g.npairs == 0) return rc;
    if (!w) return TOPO_EINVAL;
    return cuda_rc(launch_combine(g, H, y, sorted_pairs, w, out, ws, stream));
}

int topo_read_error(const void *ws) {
    if (!ws) return TOPO_EINVAL;
    int32_t e = 0;
    if (cudaMemcpy(&e, ws, sizeof e, cudaMemcpyDeviceToHost) != cudaSuccess) return TOPO_ECUDA;
    return e;
}

const char *topo_strerror(int code) {
    switch (code) {
        case TOPO_OK: return "ok";
        case TOPO_EINVAL: return "invalid argument";
        case TOPO_ENOSPC: return "workspace too small";
        case TOPO_ECUDA: return "CUDA runtime error";
        case TOPO_ERANGE: return "expert id outside [0, E)";
        case TOPO_ESTATE: return "workspace does not hold the index this call needs";
        case TOPO_EMAP: return "main_rank is not a balanced map onto the ranks";
        case TOPO_EOFFSETS: return "rank_offsets is not an ordered partition of the tokens";
        case TOPO_ETIMEOUT: return "a bounded wait inside a kernel expired";
        default: return "unknown error";
    }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// topo_hist_noalloc: topo_hist with its scratch in a fixed per-device array,
// for callers that cannot give the library device memory during a step.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TOPO_HIST_NOALLOC_SCRATCH_BYTES];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kNoAllocMaxDevices];

// Address of the scratch array on the current device, looked up once per
// device (the lookup may load the module, so it belongs before any capture).
cudaError_t noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int topo_hist_noalloc(const topo_cfg *cfg, int32_t n_layers, const int32_t *ids,
                                 int32_t *hist, int32_t *err, cudaStream_t stream) {
    Geo g;
    int rc = make_geo(cfg, n_layers, &g);
    if (rc) return rc;
    if (!hist || (!ids && g.npairs > 0 && n_layers > 0)) return TOPO_EINVAL;
    // Compact layout: header, the sources' first tiles, tile counts (the
    // histogram kernels touch no other region).
    const size_t tiles = (size_t)n_layers * g.ntl;
    g.off_first = sizeof(WsHeader);
    g.off_tile = align_up(g.off_first + (size_t)(g.R + 1) * 4);
    g.total = align_up(g.off_tile + tiles * g.E * sizeof(int32_t));
    if (g.total > TOPO_HIST_NOALLOC_SCRATCH_BYTES) return TOPO_ENOSPC;
    void *ws = nullptr;
    cudaError_t e = noalloc_scratch(&ws);
    if (e != cudaSuccess) return TOPO_ECUDA;
    bind_ws(g, ws);
    e = cudaMemsetAsync(ws, 0, sizeof(WsHeader), stream);     // error word starts at 0
    if (e == cudaSuccess && n_layers > 0)
        e = launch_hist(g, ids, hist, ws, hist_fingerprint(g, ids), stream);
    if (e == cudaSuccess && err)
        e = cudaMemcpyAsync(err, static_cast<char *>(ws) + offsetof(WsHeader, error), sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, stream);
    return cuda_rc(e);
}
