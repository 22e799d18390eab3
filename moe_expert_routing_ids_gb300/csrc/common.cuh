// Internal definitions shared by the library's kernels and its C-ABI layer.
#pragma once

#include <cstddef>
#include <cstdint>

#include "topo.h"

namespace topo {

// Pair-scan tiling.  A tile is TT consecutive tokens of one source rank
// (TT = 32 * kRankWarps * RW, RW rounds of 32 tokens per warp), so tiles never
// straddle a source and every token's k pairs sit in one tile.  hist, reroute
// and layout share the tiling: the tile index topo_hist leaves is per tile.
// Tiles are numbered source by source within a layer (see tile_ref).
constexpr int kRankWarps = 8;
constexpr int kRankThreads = kRankWarps * 32;
constexpr int kTilePairsTarget = 16384;            // pairs per tile aimed for
constexpr int kRankSmemTarget = 110 * 1024;        // two rank CTAs per SM
constexpr int kSmemMax = 227 * 1024;               // per CTA on sm_103a
constexpr int kMaxK = 64;
constexpr int kRankEntCap = 1024;                 // routing entries of a row kept in shared memory
constexpr int kDedupMaxK = 16;                     // slots per token the dedup layout takes
constexpr int kDedupMaxRanks = 1024;               // ranks the dedup layout takes
constexpr int kMaxRanksPerNode = 32;               // one warp lane per rank of a domain

// Workspace header, 256 bytes at offset 0 of every workspace.
struct WsHeader {
    int32_t error;       // first device error code, 0 if none
    int32_t pad0;
    uint64_t hist_fp;    // fingerprint of the tile index written by topo_hist
    uint64_t route_fp;   // fingerprint of the routing index written by topo_reroute
    uint64_t pad[29];
};
static_assert(sizeof(WsHeader) == 256, "header size");

// Geometry of one call, derived on the host and passed by value to kernels.
struct Geo {
    int32_t T, E, k, R, rpn, n_slot, M, E_R, n_local, L;
    int32_t tps;            // tiles per source rank (equal blocks)
    int32_t tpr;            // tokens per source rank (equal blocks)
    int32_t ntl;            // tiles per layer: R * tps, or ceil(T / TT) + R with
                            //   rank_offsets (a bound: sources hold whole tiles)
    const int64_t *roff;    // device [R+1] token offsets of the sources, or null
                            //   for equal blocks of tpr tokens
    const int32_t *tfirst;  // device [R+1] first tile of each source (rank_offsets
                            //   only; set per call from the workspace)
    int32_t TT, RW;         // tokens per tile, rounds of 32 tokens per warp
    int32_t kp;             // shared-memory stride of a token's ids (k, made odd)
    uint32_t kmagic;        // ceil(2^32 / k) for k >= 2: i / k == umulhi(i, kmagic), i < 2^26
    int32_t n_inst_cap;     // E + R * n_slot: most instances a layer can hold
    int32_t n_keys;         // R * n_local
    int32_t c_intra, c_inter, max_iters;
    int64_t pps;            // pairs per source rank
    int64_t npairs;         // pairs per layer = T * k
    int64_t S_tok, W;
    // workspace regions (byte offsets)
    size_t off_tile;        // int32 [L][R][tps][E]   tile counts -> exclusive prefix
    size_t off_pos;         // int32 [L][R][tps][TT*k] layout position of each pair,
                            //        in (warp, round, slot, lane) order within a tile
    size_t off_main;        // int32 [2E + R*E_R]     main(e), local index, mains[r][j]
    size_t off_rep;         // int32 [L][E][M]        stage-1 replica instance per domain
    size_t off_iexp;        // int32 [L][n_keys]      expert held by each instance
    size_t off_ioff;        // int32 [L][E+1]         start of each expert's instances in ilist
    size_t off_ilist;       // int32 [L][n_keys]      instances grouped by expert, ascending rank
    size_t off_roff;        // int32 [L][R][E+1]      per-(s,e) entry offsets in row s
    size_t off_rent;        // int4  [L][R][n_inst_cap] (inst, cum_start, cum_end, out_base)
    size_t off_soff;        // int32 [L][R][n_keys]   column prefix of q over sources
    size_t off_ccnt;        // int32 [L][n_keys]      column totals of q
    size_t off_lseg;        // int32 [L][n_keys+1]    segment offsets
    size_t off_lsend;       // int64 [L][R][R]        send counts
    size_t off_lstat;       // int64 [L][8]           layout statistics
    size_t off_pack_inv;    // int32 [L][T*k]         position of each pair (pack workspace)
    size_t off_first;       // int32 [R+1]            first tile of each source (rank_offsets)
    size_t total;
};

__host__ __device__ inline int dom_of(int r, int rpn) { return r / rpn; }

__host__ __device__ inline int64_t cost_sr(const Geo &g, int s, int r) {
    if (s == r) return 0;
    return (s / g.rpn == r / g.rpn) ? g.c_intra : g.c_inter;
}

// Source blocks and tiles.  Token t of a layer belongs to the source s with
// off[s] <= t < off[s+1], where off = rank_offsets, or s * tpr for equal
// blocks.  Tiles of TT tokens never straddle a source and are numbered source
// by source: tile = s * tps + t for equal blocks; with rank_offsets, source s
// owns tiles [first[s], first[s+1]) (first[] built per call by
// launch_tile_first), and tiles from first[R] to ntl are empty.
struct TileRef {
    int s, t;          // source, tile within the source (s < 0: an empty tile)
    int tok0, ntok;    // first token (within the layer) and token count
    bool last;         // the source's last tile
};

// roff: the offsets or null; tpr: tokens per source for equal blocks.
__device__ __forceinline__ TileRef tile_ref(const int64_t *roff, int R, int tpr, const int32_t *first,
                                            int TT, int tps, int tile) {
    TileRef r;
    if (!roff) {
        r.s = tile / tps;
        r.t = tile - r.s * tps;
        r.tok0 = r.s * tpr + r.t * TT;
        r.ntok = max(0, min(TT, tpr - r.t * TT));
        r.last = r.t + 1 == tps;
        return r;
    }
    // the last source whose first tile is <= tile (binary search over first[])
    const int nt = __ldg(first + R);
    if (tile >= nt) {
        r.s = -1; r.t = 0; r.tok0 = 0; r.ntok = 0; r.last = true;
        return r;
    }
    int lo = 0, hi = R - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(first + mid) <= tile) lo = mid;
        else hi = mid - 1;
    }
    r.s = lo;
    r.t = tile - __ldg(first + lo);
    const int64_t b = __ldg(roff + lo), e = __ldg(roff + lo + 1);
    r.tok0 = (int)b + r.t * TT;
    r.ntok = max(0, min(TT, (int)(e - r.tok0)));
    r.last = tile + 1 == __ldg(first + lo + 1);
    return r;
}

__device__ __forceinline__ TileRef tile_ref(const Geo &g, const int32_t *first, int TT, int tps, int tile) {
    return tile_ref(g.roff, g.R, g.tpr, first, TT, tps, tile);
}

// Tiles [*b, *e) of source s.
__device__ __forceinline__ void source_tiles(const int64_t *roff, const int32_t *first, int tps, int s,
                                             int *b, int *e) {
    if (!roff) {
        *b = s * tps;
        *e = *b + tps;
    } else {
        *b = __ldg(first + s);
        *e = __ldg(first + s + 1);
    }
}

__device__ __forceinline__ void source_tiles(const Geo &g, const int32_t *first, int tps, int s, int *b,
                                             int *e) {
    source_tiles(g.roff, first, tps, s, b, e);
}

// Record the first device error in the header (sticky).
// First error wins; once the word is set, later reporters only read it (no
// atomic traffic on one address when every thread of a launch reports).
__device__ inline void set_error(WsHeader *h, int code) {
    if (*reinterpret_cast<volatile int32_t *>(&h->error) == 0) atomicCAS(&h->error, 0, code);
}

// 64-bit fingerprint mixing (splitmix64 finaliser).
__host__ __device__ inline uint64_t fp_mix(uint64_t h, uint64_t v) {
    uint64_t z = h + 0x9e3779b97f4a7c15ull + v;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

// i / k for 0 <= i < 2^26 without a hardware divide (k = 1 is the identity;
// its reciprocal does not fit in 32 bits).
__device__ __forceinline__ int div_k(const Geo &g, int i) {
    return g.k == 1 ? i : (int)__umulhi((unsigned)i, g.kmagic);
}

template <typename T>
__host__ __device__ inline T *ws_at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device, once per (kernel, device): later calls, including calls
// made while a stream is being captured into a CUDA graph, launch only.
cudaError_t ensure_smem(const void *fn, size_t bytes);

// n / d for n < 2^32 by a multiply-high with m = floor(2^32 / d) (2^32 - 1 for
// d = 1), which gives the quotient or one less, and one correction step (the
// reciprocal-multiplication method of Granlund and Montgomery, "Division by
// Invariant Integers using Multiplication", with the correction in place of
// the rounding analysis).
struct FastDiv {
    unsigned d, m;
};

inline FastDiv make_fast_div(unsigned d) {
    FastDiv v;
    v.d = d;
    v.m = d <= 1 ? 0xffffffffu : (unsigned)((1ull << 32) / d);
    return v;
}

__device__ __forceinline__ unsigned fast_quot(unsigned n, FastDiv v) {
    unsigned q = __umulhi(n, v.m);
    q += (n - q * v.d) >= v.d;
    return q;
}

// Routing-index entry of one (source, instance) pair with a nonzero count:
// the instance code r * n_local + l, the source's occurrences of the expert
// routed there [cum_start, cum_end), and the layout position of occurrence
// cum_start minus cum_start.
struct Entry {
    int32_t code;
    int32_t cum_start;
    int32_t cum_end;
    int32_t out_base;
};
static_assert(sizeof(Entry) == 16, "entry size");

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

// Prep of the rerouting calls (instance index, routing index, layout
// offsets), from the plan alone; defined in k_prep.cu.  The segment offsets,
// send counts and layout statistics go to seg_off / send_counts /
// layout_stats when given (the fused call's outputs), else to the workspace.
cudaError_t launch_prep(const Geo &g, const int32_t *main_rank, const topo_plan_t &p, void *ws,
                        int32_t *seg_off, int64_t *send_counts, int64_t *layout_stats, cudaStream_t st);
cudaError_t launch_main_tables(const Geo &g, const int32_t *main_rank, void *ws, int64_t *stats,
                               int n_stats, cudaStream_t st);
// first[s] = first tile of source s for tiles of TT tokens over g.roff, and
// first[R] = the tile count; checks that the offsets partition [0, T] in
// order (TOPO_EOFFSETS in hdr otherwise, with every tile left empty).
// Defined in k_hist.cu.
cudaError_t launch_tile_first(const Geo &g, int TT, int32_t *first, WsHeader *hdr, cudaStream_t st);

// Programmatic dependent launch.  A kernel launched with launch_pdl may
// start while the previous kernel of the stream is still finishing: it must
// call pdl_wait() before reading anything earlier kernels wrote (or writing
// anything they read); pdl_wait() returns once those kernels have completed
// and their writes are visible.  pdl_trigger() lets the next kernel start
// launching; both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// Kernel launchers (defined in the kernel translation units).  Each returns
// the cudaError_t of its launches.
// ---------------------------------------------------------------------------
cudaError_t launch_hist(const Geo &g, const int32_t *ids, int32_t *hist, void *ws, uint64_t fp,
                        cudaStream_t st);
// Column prefix of the tile counts in ws (the tile index) and Omega; records
// the hist fingerprint fp.  Shared by topo_hist and topo_gate_hist.
cudaError_t launch_hist_prefix(const Geo &g, int32_t *hist, void *ws, uint64_t fp, cudaStream_t st);
// Top-k gating of logits [L][T][E] (float32, or bf16 patterns) plus bias,
// writing ids, the selected raw logits (scores may be null) and the tile
// counts, then launch_hist_prefix.
cudaError_t launch_gate(const Geo &g, const void *logits, bool bf16, const float *bias, int32_t *ids,
                        float *scores, int32_t *hist, void *ws, uint64_t fp, cudaStream_t st);
// Token-shuffle targets: ranks at most kShuffleMaxRanks.
constexpr int kShuffleMaxRanks = 256;
size_t shuffle_ws_bytes(int L, int E, int R);
cudaError_t launch_shuffle(int L, int T, int E, int k, int R, const int32_t *ids, const int64_t *tr,
                           const int32_t *main_rank, const int64_t *rank_offsets, int32_t *target,
                           int64_t *stats, void *ws, cudaStream_t st);
// Correlated expert placement: one CTA per layer, E <= kPlaceMaxE and the
// shared tables within kSmemMax.
constexpr int kPlaceMaxE = 1024;
size_t place_smem_bytes(int E, int R);
cudaError_t launch_place(int L, int E, int R, int max_iters, const int64_t *co, int32_t *main_rank,
                         int64_t *stats, cudaStream_t st);
cudaError_t launch_plan(const Geo &g, const int32_t *main_rank, const int32_t *hist,
                        const topo_plan_t &p, void *ws, cudaStream_t st);
cudaError_t launch_reroute(const Geo &g, const int32_t *main_rank, const int32_t *ids,
                           const topo_plan_t &p, int32_t *dst, void *ws, uint64_t hist_fp,
                           uint64_t route_part, cudaStream_t st);
cudaError_t launch_layout(const Geo &g, int32_t *sorted, int32_t *seg_off, int64_t *send_counts,
                          int64_t *layout_stats, void *ws, uint64_t route_part, cudaStream_t st);
cudaError_t launch_reroute_layout(const Geo &g, const int32_t *main_rank, const int32_t *ids,
                                  const topo_plan_t &p, int32_t *dst, int32_t *sorted,
                                  int32_t *seg_off, int64_t *send_counts, int64_t *layout_stats,
                                  void *ws, uint64_t hist_fp, cudaStream_t st);
// Shared-memory bytes of the rank kernel for this geometry.
size_t row_index_smem(const Geo &g);
size_t rank_smem_bytes(const Geo &g);
cudaError_t launch_cooccur(int L, int T, int E, int k, const int32_t *ids, int64_t *co, int64_t *tr,
                           void *ws, cudaStream_t st);
// Tensor-core co-occurrence (k_cooccur_mma.cu): E <= 128 and k <= 16, units
// of at most kMaxCoocTokens tokens (a cell's sum stays below 2^24), about
// kCoocUnitsTarget units per call; int32 partials per unit in the workspace.
constexpr int kMaxCoocTokens = 65536;
constexpr int kCoocUnitsTarget = 152;
bool cooccur_mma_applies(int L, int T, int E, int k);
void cooccur_mma_units(int L, int T, int *nchunks, int *chunk);
size_t cooccur_mma_ws_bytes(int L, int T, int E, int k);
cudaError_t launch_cooccur_mma(int L, int T, int E, int k, const int32_t *ids, int64_t *co, int64_t *tr,
                               void *ws, cudaStream_t st);
size_t dedup_ws_bytes(const Geo &g, size_t *off_tile, size_t *off_src, size_t *off_first);
cudaError_t launch_dedup(const Geo &g, const int32_t *dst, int32_t *seg, int32_t *row_token,
                         uint64_t *row_slots, uint64_t *tok_dst, int64_t *send, int64_t *stats, void *ws,
                         cudaStream_t st);
cudaError_t launch_permute(const Geo &g, int H, const uint16_t *x, const int32_t *sorted, uint16_t *y,
                           void *ws, cudaStream_t st);
cudaError_t launch_combine(const Geo &g, int H, const uint16_t *y, const int32_t *sorted, const float *w,
                           uint16_t *out, void *ws, cudaStream_t st);

}  // namespace topo
