// Rerouting of every (token, slot) pair to an expert instance and the
// dispatch layout (TopoEP §1 / Fig. 5 token rerouting; §5 receive counts
// derived on the GPU).
//
// Reading used for the pair -> instance rule: within source s, the pairs that
// select e are taken in pair order; the o-th of them (its occurrence index)
// goes to the instance of e whose running range of q[s][.] over e's instances
// in ascending rank order holds o.  The layout is the stable sort of pairs by
// instance, so a pair's position is  seg_off[i] + sum_{s'<s} q[s'][i] +
// (o - start of i's range)  =  out_base(s, i) + o.
//
// Everything therefore follows from one number per pair, o, computed once by
// k_route_tiles:
//   * topo_hist's tile index gives the occurrences before the tile;
//   * inside a tile (TT tokens, 8 warps, lane = token) each warp counts its
//     rounds per expert (shared atomics), the warps' counts are prefixed, and
//     each round of 32 tokens is ranked with a per-expert token bitmask:
//     every lane ORs its bit into mask[e] for each of its k ids, then a pair's
//     rank in the round is popc(mask[e] & lanes below) -- the earlier tokens
//     of the round holding e.  Top-k ids of one token are distinct, so no
//     token meets the same expert twice in a round; a tile where one does is
//     redone by the warp match_any path below, which is exact in any case.
// The routing index (per (s, e) entries {instance, cum_start, cum_end,
// out_base}) is built by the prep kernels (k_prep.cu) from the plan alone.
#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {

namespace {

// ---------------------------------------------------------------------------
// Tile kernels
// ---------------------------------------------------------------------------

struct TileGeo {
    int l, s, t;
    int ntok;        // tokens in this tile (0: an empty tile, s < 0 possible)
    bool last;       // the source's last tile
    int64_t row;     // the tile's row of the tile index: l * ntl + tile
    int64_t p0;      // first pair of the tile within its layer
    int64_t slot0;   // base of the tile in the position array (TT * k entries)
};

__device__ __forceinline__ TileGeo tile_geo(const Geo &g) {
    TileGeo tg;
    tg.l = blockIdx.x / g.ntl;
    const int tile = blockIdx.x - tg.l * g.ntl;
    const TileRef r = tile_ref(g, g.tfirst, g.TT, g.tps, tile);
    tg.s = r.s;
    tg.t = r.t;
    tg.ntok = r.ntok;
    tg.last = r.last;
    tg.row = blockIdx.x;
    tg.p0 = (int64_t)r.tok0 * g.k;
    tg.slot0 = (int64_t)blockIdx.x * g.TT * g.k;
    return tg;
}

__device__ __forceinline__ bool check_fp(const WsHeader *hdr, uint64_t want, bool routed,
                                         uint64_t part, int *flag) {
    if (threadIdx.x == 0) {
        const uint64_t have = routed ? hdr->route_fp : hdr->hist_fp;
        const uint64_t exp = routed ? fp_mix(hdr->hist_fp, part) : want;
        *flag = (have == exp && have != 0);
    }
    __syncthreads();
    return *flag != 0;
}

// Position-array index of pair (token t of the tile, slot j).
__device__ __forceinline__ int64_t pos_index(const Geo &g, const TileGeo &tg, int t, int j) {
    return tg.slot0 + ((int64_t)(t >> 5) * g.k + j) * 32 + (t & 31);
}

// Exact ranking of one tile with warp match_any, pair-major, ids read from
// global memory.  Used for k > KMAX and for tiles where a token repeats an
// expert.  cntw: [kRankWarps][E] shared.
template <bool kFused>
__device__ void rank_tile_exact(const Geo &g, const TileGeo &tg, const int32_t *ids_layer,
                                const int32_t *tile_base, const int32_t *ro, const Entry *re,
                                int *cntw, int32_t *dst_layer, int32_t *pos_ws,
                                int32_t *sorted_layer, bool &bad_id, bool &bad_state) {
    const int E = g.E, k = g.k;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int n = tg.ntok * k;
    const int seg = ((n + kRankWarps - 1) / kRankWarps + 31) & ~31;
    const int beg = w * seg, end = min(n, beg + seg);
    __syncthreads();
    for (int i = threadIdx.x; i < kRankWarps * E; i += blockDim.x) cntw[i] = 0;
    __syncthreads();
    int *mine = cntw + w * E;
    for (int b = beg; b < end; b += 32) {
        const int idx = b + lane;
        int e = idx < end ? __ldg(ids_layer + tg.p0 + idx) : -1;
        if ((unsigned)e >= (unsigned)E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (peers & lt_mask) == 0) mine[e] += __popc(peers);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = __ldg(tile_base + e);
        for (int x = 0; x < kRankWarps; ++x) {
            const int c = cntw[x * E + e];
            cntw[x * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int b = beg; b < end; b += 32) {
        const int idx = b + lane;
        const bool valid = idx < end;
        int e = valid ? __ldg(ids_layer + tg.p0 + idx) : -1;
        if (valid && (unsigned)e >= (unsigned)E) { bad_id = true; e = -1; }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int occ = e >= 0 ? mine[e] + __popc(peers & lt_mask) : 0;
        __syncwarp();
        if (e >= 0 && (peers & lt_mask) == 0) mine[e] += __popc(peers);
        if (valid) {
            int code = -1, ob = 0;
            if (e >= 0) {
                const int f = __ldg(ro + e), en = __ldg(ro + e + 1);
                for (int j = f; j < en; ++j) {
                    if (occ < __ldg(&re[j].cum_end)) {
                        code = __ldg(&re[j].code);
                        ob = __ldg(&re[j].out_base);
                        break;
                    }
                }
                if (code < 0) bad_state = true;
            }
            const int t = idx / k, j = idx - t * k;
            dst_layer[tg.p0 + idx] = code;
            const int64_t pos = code >= 0 ? (int64_t)ob + occ : -1;
            if (kFused) {
                if (pos >= 0 && pos < g.npairs) sorted_layer[pos] = (int32_t)(tg.p0 + idx);
                else if (code >= 0) bad_state = true;
            } else {
                pos_ws[pos_index(g, tg, t, j)] = (int32_t)pos;
            }
        }
        __syncwarp();
    }
}

// Shared-memory layout of k_route_tiles.
struct RankSmem {
    int *ec;         // [E] code of the expert's only routing entry in this row;
                     //     -1: several entries; -2: none
    int *ro;         // [E+1] entry offsets of the row
    int *ent_ce;     // [kRankEntCap] entries' cum_end, code, out_base (when the
    int *ent_code;   //     row has at most kRankEntCap entries)
    int *ent_ob;
    int *base;       // [kRankWarps][E] per-warp running base: the layout position
                     //     of the next pair (single entry) or its occurrence index
    unsigned *msk;   // [kRankWarps][E] per-warp token bitmask of the round
    int32_t *keys;   // [TT][kp] ids, then the instance codes, in place
};

__device__ __forceinline__ RankSmem rank_smem(const Geo &g, int *sm) {
    RankSmem r;
    int *p = sm;
    r.ec = p; p += g.E;
    r.ro = p; p += g.E + 1;
    r.ent_ce = p; p += kRankEntCap;
    r.ent_code = p; p += kRankEntCap;
    r.ent_ob = p; p += kRankEntCap;
    r.base = p; p += kRankWarps * g.E;
    r.msk = reinterpret_cast<unsigned *>(p); p += kRankWarps * g.E;
    r.keys = reinterpret_cast<int32_t *>(p);
    return r;
}

// Instance code and layout position for occurrence occ of expert e with
// several entries in this row (entries in rank order, running ranges), from
// shared memory when the row's entries fit there.
__device__ __forceinline__ int route_walk(int occ, int e, const RankSmem &S, bool row_in_smem,
                                          const Entry *re, int *pos) {
    const int b = S.ro[e], en = S.ro[e + 1];
    if (row_in_smem) {
        for (int j = b; j < en; ++j)
            if (occ < S.ent_ce[j]) {
                *pos = S.ent_ob[j] + occ;
                return S.ent_code[j];
            }
        return -1;
    }
    for (int j = b; j < en; ++j) {
        if (occ < __ldg(&re[j].cum_end)) {
            *pos = __ldg(&re[j].out_base) + occ;
            return __ldg(&re[j].code);
        }
    }
    return -1;
}

// One CTA per tile.  kFused: write the layout (sorted pairs) directly;
// otherwise store each pair's layout position in the workspace for
// topo_dispatch_layout.  K > 0: k known at compile time; K == 0: any k up to
// KMAX.  Each lane visits its token's slots starting at lane % k, so a hot
// expert that Top-k puts in the same slot of many tokens does not serialise
// one shared atomic across the warp (the order inside a round is free: a
// round is ranked only after all its slots are in the bitmasks).
template <int K, int KMAX, bool kFused>
__global__ void __launch_bounds__(kRankThreads, 2)
k_route_tiles(const int32_t *__restrict__ ids, const int32_t *__restrict__ tile_idx,
              const int32_t *__restrict__ roff, const Entry *__restrict__ rent, int32_t *dst,
              int32_t *pos_ws, int32_t *sorted, WsHeader *hdr, Geo g, uint64_t hist_fp,
              uint64_t route_part) {
    pdl_wait();                                  // the previous kernel's outputs
    constexpr int KB = K > 0 ? K : KMAX;
    extern __shared__ int sm[];
    __shared__ int ok;
    if (!check_fp(hdr, hist_fp, false, 0, &ok)) {
        if (threadIdx.x == 0) set_error(hdr, TOPO_ESTATE);
        return;
    }
    if (!kFused && blockIdx.x == 0 && threadIdx.x == 0) hdr->route_fp = fp_mix(hist_fp, route_part);
    const TileGeo tg = tile_geo(g);
    if (tg.ntok == 0) {                          // an empty tile: no pairs, no tables
        pdl_trigger();
        return;
    }
    const int E = g.E;
    const int k = K > 0 ? K : g.k;
    const int kp = K > 0 ? ((K & 1) ? K : K + 1) : g.kp;
    const RankSmem S = rank_smem(g, sm);
    const int p0i = (int)tg.p0;                        // pair indices fit in int32
    const unsigned npairs_u = (unsigned)g.npairs;
    const int32_t *ids_layer = ids + (int64_t)tg.l * g.npairs;
    int32_t *dst_layer = dst + (int64_t)tg.l * g.npairs;
    int32_t *sorted_layer = kFused ? sorted + (int64_t)tg.l * g.npairs : nullptr;
    const int32_t *tbase = tile_idx + tg.row * E;
    const int32_t *ro = roff + ((int64_t)tg.l * g.R + tg.s) * (E + 1);
    const Entry *re = rent + ((int64_t)tg.l * g.R + tg.s) * g.n_inst_cap;
    bool bad_id = false, bad_state = false;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned bit = 1u << lane, lt_mask = bit - 1u;
    const int rot = lane % k;                        // first slot this lane visits
    const int n = tg.ntok * k;
    auto div = [&](int i) { return K > 0 ? i / K : div_k(g, i); };

    // stage: ids token-major with an odd stride (conflict-free per lane) by
    // asynchronous 4-byte copies, all in flight at once; the per-expert
    // routing table; zeroed per-warp tables
    const bool fast = k <= KB;
    if (fast) {
        const int32_t *src = ids_layer + tg.p0;
        for (int i = threadIdx.x; i < n; i += kRankThreads) {
            const int t = div(i);
            cp_async4(&S.keys[t * kp + (i - t * k)], src + i);
        }
    }
    const int n_ent = __ldg(ro + E);
    const bool row_in_smem = n_ent <= kRankEntCap;
    // every per-expert value of the tile requested at once (the tile's
    // occurrence range [tb, te) parked in warp 0's base and mask words), the
    // row's entries staged, the other warps' words zeroed; then one barrier
    if (row_in_smem)
        for (int j = threadIdx.x; j < n_ent; j += kRankThreads) {
            S.ent_ce[j] = __ldg(&re[j].cum_end);
            S.ent_code[j] = __ldg(&re[j].code);
            S.ent_ob[j] = __ldg(&re[j].out_base);
        }
    if (threadIdx.x == 0) S.ro[E] = n_ent;
    for (int e = threadIdx.x; e < E; e += kRankThreads) {
        S.ro[e] = __ldg(ro + e);
        S.base[e] = __ldg(tbase + e);
        S.msk[e] = tg.last ? 0u : (unsigned)__ldg(tbase + E + e);
#pragma unroll
        for (int x = 1; x < kRankWarps; ++x) {
            S.base[x * E + e] = 0;
            S.msk[x * E + e] = 0;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kRankThreads) {
        const int b = S.ro[e], en = S.ro[e + 1];
        const int ne = en - b;
        auto ce = [&](int j) { return row_in_smem ? S.ent_ce[j] : __ldg(&re[j].cum_end); };
        auto cd = [&](int j) { return row_in_smem ? S.ent_code[j] : __ldg(&re[j].code); };
        auto ob = [&](int j) { return row_in_smem ? S.ent_ob[j] : __ldg(&re[j].out_base); };
        int code = ne == 1 ? cd(b) : (ne == 0 ? -2 : -1);
        // per-warp base: tile base (+ out_base when the expert has one entry);
        // pass 1 then adds each warp's count into the following warps' bases
        const int tb = S.base[e];
        int b0 = tb + (ne == 1 ? ob(b) : 0);
        if (ne > 1) {
            // several entries: when the tile's occurrences [tb, te) all fall in
            // one entry, the tile ranks e like a single-entry expert
            const int te = !tg.last ? (int)S.msk[e] : ce(en - 1);
            int j = b;
            while (j < en && tb >= ce(j)) ++j;
            if (j < en && te <= ce(j)) {
                code = cd(j);
                b0 = tb + ob(j);
            }
        }
        S.ec[e] = code;
        S.base[e] = b0;
        S.msk[e] = 0;
    }
    if (fast) cp_async_wait_all();
    __syncthreads();

    bool dup = !fast;
    if (fast) {
        int *mybase = S.base + w * E;
        unsigned *mymsk = S.msk + w * E;
        // pass 1: per-warp counts over its rounds, added into the next warp's
        // base (shifted by one so pass 2 is a plain prefix)
        if (w + 1 < kRankWarps) {
            int *nextbase = S.base + (w + 1) * E;
            for (int r = 0; r < g.RW; ++r) {
                const int t = (w * g.RW + r) * 32 + lane;
                if (t < tg.ntok) {
                    int j = rot;
#pragma unroll
                    for (int jj = 0; jj < KB; ++jj) {
                        if (jj < k) {
                            const int e = S.keys[t * kp + j];
                            if ((unsigned)e < (unsigned)E) atomicAdd(&nextbase[e], 1);
                            j = (j + 1 == k) ? 0 : j + 1;
                        }
                    }
                }
            }
        }
        __syncthreads();
        // pass 2: inclusive prefix over warps (the expert's words all read first)
        for (int e = threadIdx.x; e < E; e += kRankThreads) {
            int v[kRankWarps];
#pragma unroll
            for (int x = 0; x < kRankWarps; ++x) v[x] = S.base[x * E + e];
            int run = 0;
#pragma unroll
            for (int x = 0; x < kRankWarps; ++x) {
                run += v[x];
                S.base[x * E + e] = run;
            }
        }
        __syncthreads();
        // pass 3: rank each round of 32 tokens with per-expert token bitmasks
        for (int r = 0; r < g.RW; ++r) {
            const int t = (w * g.RW + r) * 32 + lane;
            const bool vt = t < tg.ntok;
            int ek[KB];
            {
                int j = rot;
#pragma unroll
                for (int jj = 0; jj < KB; ++jj) {
                    ek[jj] = -1;
                    if (jj < k) {
                        if (vt) {
                            const int e = S.keys[t * kp + j];
                            if ((unsigned)e < (unsigned)E) ek[jj] = e;
                            else bad_id = true;
                        }
                        j = (j + 1 == k) ? 0 : j + 1;
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < KB; ++jj)
                if (ek[jj] >= 0) dup |= (atomicOr(&mymsk[ek[jj]], bit) & bit) != 0;
            __syncwarp();
            int nb[KB];
            unsigned lead = 0;
            {
                int j = rot;
#pragma unroll
                for (int jj = 0; jj < KB; ++jj) {
                    nb[jj] = 0;
                    if (jj >= k) continue;
                    int code = -1, pos = -1;
                    if (ek[jj] >= 0) {
                        const unsigned m = mymsk[ek[jj]];
                        const int b = mybase[ek[jj]];
                        const int rk = __popc(m & lt_mask);
                        if (rk == 0) {
                            lead |= 1u << jj;
                            nb[jj] = b + __popc(m);
                        }
                        code = S.ec[ek[jj]];
                        if (code >= 0) pos = b + rk;
                        else if (code == -1) code = route_walk(b + rk, ek[jj], S, row_in_smem, re, &pos);
                        if (code < 0) bad_state = true;
                    }
                    if (vt) {
                        S.keys[t * kp + j] = code;
                        if (kFused && code >= 0) {
                            if ((unsigned)pos < npairs_u) sorted_layer[pos] = p0i + t * k + j;
                            else bad_state = true;
                        }
                    }
                    if (!kFused)
                        pos_ws[tg.slot0 + ((t >> 5) * k + j) * 32 + lane] =
                            (vt && code >= 0) ? pos : -1;
                    j = (j + 1 == k) ? 0 : j + 1;
                }
            }
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < KB; ++jj)
                if ((lead >> jj) & 1u) {
                    mybase[ek[jj]] = nb[jj];
                    mymsk[ek[jj]] = 0;
                }
            __syncwarp();
        }
    }
    if (__syncthreads_or(dup)) {
        // a token repeats an expert (or k > KB): redo the tile exactly
        rank_tile_exact<kFused>(g, tg, ids_layer, tbase, ro, re, S.base, dst_layer, pos_ws,
                                sorted_layer, bad_id, bad_state);
    } else {
        // instance codes out, pair order, coalesced
        for (int i = threadIdx.x; i < n; i += kRankThreads) {
            const int t = div(i);
            dst_layer[tg.p0 + i] = S.keys[t * kp + (i - t * k)];
        }
    }
    if (bad_id) set_error(hdr, TOPO_ERANGE);
    if (bad_state) set_error(hdr, TOPO_ESTATE);
    pdl_trigger();
}

// Layout from the positions topo_reroute stored: sorted[pos] = pair.
__global__ void __launch_bounds__(256)
k_layout_scatter(const int32_t *__restrict__ pos_ws, int32_t *sorted, WsHeader *hdr, Geo g,
                 uint64_t route_part) {
    pdl_wait();                                  // the previous kernel's outputs
    __shared__ int ok;
    if (!check_fp(hdr, 0, true, route_part, &ok)) {
        if (threadIdx.x == 0) set_error(hdr, TOPO_ESTATE);
        return;
    }
    const TileGeo tg = tile_geo(g);
    const int k = g.k;
    const int n = g.TT * k;
    int32_t *out = sorted + (int64_t)tg.l * g.npairs;
    if (tg.ntok == 0) {
        pdl_trigger();
        return;
    }
    bool bad = false;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int wr = div_k(g, i >> 5);   // (i / 32) / k
        const int t = wr * 32 + (i & 31);
        if (t >= tg.ntok) continue;
        const int v = __ldcs(pos_ws + tg.slot0 + i);
        const int j = (i >> 5) - wr * k;
        if (v < 0 || v >= g.npairs) { bad = true; continue; }
        out[v] = (int32_t)(tg.p0 + (int64_t)t * k + j);
    }
    if (bad) set_error(hdr, TOPO_ESTATE);
    pdl_trigger();
}

// Copy the small layout outputs the prep kernels left in the workspace
// (topo_dispatch_layout, after topo_reroute).
__global__ void __launch_bounds__(256)
k_lay_copy(const int32_t *__restrict__ lseg, const int64_t *__restrict__ lsend,
           const int64_t *__restrict__ lstat, int32_t *seg_off, int64_t *send_counts,
           int64_t *layout_stats, const WsHeader *hdr, Geo g, uint64_t route_part) {
    pdl_wait();                                  // the previous kernel's outputs
    __shared__ int ok;
    if (!check_fp(hdr, 0, true, route_part, &ok)) return;
    const int64_t nseg = (int64_t)g.L * (g.n_keys + 1);
    const int64_t nsend = (int64_t)g.L * g.R * g.R;
    const int64_t nst = (int64_t)g.L * TOPO_LAYOUT_STATS;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nseg + nsend + nst;
         i += stride) {
        if (i < nseg) seg_off[i] = lseg[i];
        else if (i < nseg + nsend) send_counts[i - nseg] = lsend[i - nseg];
        else layout_stats[i - nseg - nsend] = lstat[i - nseg - nsend];
    }
    pdl_trigger();
}

template <bool kFused>
using RouteKernel = void (*)(const int32_t *, const int32_t *, const int32_t *, const Entry *,
                             int32_t *, int32_t *, int32_t *, WsHeader *, Geo, uint64_t, uint64_t);

template <bool kFused>
RouteKernel<kFused> pick_route_kernel(int k) {
    switch (k) {
        case 1: return k_route_tiles<1, 1, kFused>;
        case 2: return k_route_tiles<2, 2, kFused>;
        case 4: return k_route_tiles<4, 4, kFused>;
        case 6: return k_route_tiles<6, 6, kFused>;
        case 8: return k_route_tiles<8, 8, kFused>;
        case 10: return k_route_tiles<10, 10, kFused>;
        case 16: return k_route_tiles<16, 16, kFused>;
        default: return k_route_tiles<0, 16, kFused>;
    }
}

template <bool kFused>
cudaError_t launch_tiles(const Geo &g, const int32_t *ids, int32_t *dst, int32_t *sorted, void *ws,
                         uint64_t hist_fp, uint64_t route_part, cudaStream_t st) {
    RouteKernel<kFused> kern = pick_route_kernel<kFused>(g.k);
    const size_t smem = rank_smem_bytes(g);
    cudaError_t e;
    if ((e = ensure_smem((const void *)kern, smem)) != cudaSuccess) return e;
    const int64_t tiles = (int64_t)g.L * g.ntl;
    return launch_pdl(kern, dim3((unsigned)tiles), dim3(kRankThreads), smem, st,
        ids, ws_at<int32_t>(ws, g.off_tile), ws_at<int32_t>(ws, g.off_roff),
        ws_at<Entry>(ws, g.off_rent), dst, ws_at<int32_t>(ws, g.off_pos), sorted,
        ws_at<WsHeader>(ws, 0), g, hist_fp, route_part);
}

cudaError_t launch_copy(const Geo &g, int32_t *seg_off, int64_t *send_counts, int64_t *layout_stats,
                        void *ws, uint64_t route_part, cudaStream_t st) {
    const int64_t n = (int64_t)g.L * (g.n_keys + 1 + (int64_t)g.R * g.R + TOPO_LAYOUT_STATS);
    const int64_t want = (n + 255) / 256;
    const int blocks = (int)(want < 1024 ? want : 1024);
    return launch_pdl(k_lay_copy, dim3(blocks), dim3(256), 0, st, ws_at<int32_t>(ws, g.off_lseg),
                      ws_at<int64_t>(ws, g.off_lsend), ws_at<int64_t>(ws, g.off_lstat), seg_off, send_counts,
                      layout_stats, ws_at<WsHeader>(ws, 0), g, route_part);
}

}  // namespace

size_t rank_smem_bytes(const Geo &g) {
    return ((size_t)2 * g.E + 1 + 3 * (size_t)kRankEntCap) * 4 + (size_t)kRankWarps * g.E * 8 +
           (size_t)g.TT * g.kp * 4;
}

cudaError_t launch_reroute(const Geo &g, const int32_t *main_rank, const int32_t *ids,
                           const topo_plan_t &p, int32_t *dst, void *ws, uint64_t hist_fp,
                           uint64_t route_part, cudaStream_t st) {
    cudaError_t e;
    if ((e = launch_prep(g, main_rank, p, ws, nullptr, nullptr, nullptr, st)) != cudaSuccess) return e;
    return launch_tiles<false>(g, ids, dst, nullptr, ws, hist_fp, route_part, st);
}

cudaError_t launch_layout(const Geo &g, int32_t *sorted, int32_t *seg_off, int64_t *send_counts,
                          int64_t *layout_stats, void *ws, uint64_t route_part, cudaStream_t st) {
    cudaError_t e;
    const int64_t tiles = (int64_t)g.L * g.ntl;
    if ((e = launch_pdl(k_layout_scatter, dim3((unsigned)tiles), dim3(256), 0, st, ws_at<int32_t>(ws, g.off_pos),
                        sorted, ws_at<WsHeader>(ws, 0), g, route_part)) != cudaSuccess)
        return e;
    return launch_copy(g, seg_off, send_counts, layout_stats, ws, route_part, st);
}

cudaError_t launch_reroute_layout(const Geo &g, const int32_t *main_rank, const int32_t *ids,
                                  const topo_plan_t &p, int32_t *dst, int32_t *sorted,
                                  int32_t *seg_off, int64_t *send_counts, int64_t *layout_stats,
                                  void *ws, uint64_t hist_fp, cudaStream_t st) {
    cudaError_t e;
    // the prep writes the layout's offsets, send counts and statistics
    // straight to the outputs
    if ((e = launch_prep(g, main_rank, p, ws, seg_off, send_counts, layout_stats, st)) != cudaSuccess)
        return e;
    return launch_tiles<true>(g, ids, dst, sorted, ws, hist_fp, 0, st);
}

}  // namespace topo
