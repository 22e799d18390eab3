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
// out_base}) is built by the prep kernels from the plan alone.
#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {

cudaError_t launch_main_tables(const Geo &g, const int32_t *main_rank, void *ws, int64_t *stats,
                               int n_stats, cudaStream_t st);

namespace {

struct Entry {
    int32_t code;       // instance r * n_local + l
    int32_t cum_start;  // first occurrence index routed here
    int32_t cum_end;    // one past the last
    int32_t out_base;   // layout position minus occurrence index
};
static_assert(sizeof(Entry) == 16, "entry size");

// Exclusive scan of a[0..n) in place by one CTA; returns the total.
__device__ int block_excl_scan(int *a, int n, int *warp_tot) {
    __shared__ int carry;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const int v = i < n ? a[i] : 0;
        int x = v;
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[w] = x;
        __syncthreads();
        int pre = carry;
        for (int j = 0; j < w; ++j) pre += warp_tot[j];
        if (i < n) a[i] = pre + x - v;
        __syncthreads();
        if (threadIdx.x == 0) {
            int t = 0;
            for (int j = 0; j < nw; ++j) t += warp_tot[j];
            carry += t;
        }
        __syncthreads();
    }
    return carry;
}

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

// Start copying n words from global to shared memory (all threads of the CTA
// take part); 16-byte copies when both sides are 16-byte aligned.  Completes
// at the next cp_async_wait_all.
__device__ __forceinline__ void stage_words(void *dst, const void *src, int n) {
    if ((((uintptr_t)dst | (uintptr_t)src) & 15) == 0) {
        const int n4 = n >> 2;
        for (int i = threadIdx.x; i < n4; i += blockDim.x)
            cp_async16(static_cast<int4 *>(dst) + i, static_cast<const int4 *>(src) + i);
        for (int i = (n4 << 2) + threadIdx.x; i < n; i += blockDim.x)
            cp_async4(static_cast<int *>(dst) + i, static_cast<const int *>(src) + i);
    } else {
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            cp_async4(static_cast<int *>(dst) + i, static_cast<const int *>(src) + i);
    }
}

// ---------------------------------------------------------------------------
// Prep: instance index, routing index, layout offsets (from the plan only)
// ---------------------------------------------------------------------------

// Instance index of a layer: the expert of every instance (iexp) and a
// bitmask over ranks of the instances of every expert (imask, zeroed before).
// One thread per instance.  tab == nullptr: the contiguous main map (main of
// e is e / (E/R)).
__global__ void __launch_bounds__(256)
k_inst_index(const int32_t *__restrict__ slot_expert, const int32_t *__restrict__ tab, int32_t *iexp,
             unsigned *imask, WsHeader *hdr, Geo g) {
    const int l = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (l == 0 && i == 0) hdr->route_fp = 0;
    if (i >= g.n_keys) return;
    const int E = g.E, R = g.R, nl = g.n_local, ER = g.E_R, ns = g.n_slot;
    const int RW = (R + 31) / 32;
    const int r = i / nl, li = i - r * nl;
    int e = li < ER ? (tab ? __ldg(tab + 2 * E + r * ER + li) : r * ER + li)
                    : __ldg(slot_expert + ((int64_t)l * R + r) * ns + (li - ER));
    bool bad = false;
    if (e >= E || e < -1) { bad = true; e = -1; }
    iexp[(int64_t)l * g.n_keys + i] = e;
    if (e >= 0) {
        const unsigned bit = 1u << (r & 31);
        const unsigned old = atomicOr(&imask[((int64_t)l * E + e) * RW + (r >> 5)], bit);
        if (old & bit) bad = true;                             // expert twice on one rank
    }
    if (bad) set_error(hdr, TOPO_ESTATE);
}

// Exclusive scan of one (count, sum) pair per thread over the CTA; returns
// the totals.  blockDim.x is a multiple of 32, at most 1024.
__device__ __forceinline__ int2 block_excl_scan2(int &a, int &b, int2 *warp_tot) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = a, y = b;
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, x, o), v = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) { x += u; y += v; }
    }
    if (lane == 31) warp_tot[w] = make_int2(x, y);
    __syncthreads();
    int px = 0, py = 0, tx = 0, ty = 0;
    for (int j = 0; j < nw; ++j) {
        const int2 t = warp_tot[j];
        if (j < w) { px += t.x; py += t.y; }
        tx += t.x; ty += t.y;
    }
    a = px + x - a;
    b = py + y - b;
    __syncthreads();
    return make_int2(tx, ty);
}

// First index in a[0..n) whose value is greater than (upper) or not less than
// (lower) v; a is non-decreasing.
__device__ __forceinline__ int upper_idx(const int *a, int n, int v) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int m = (lo + hi) >> 1;
        if (a[m] <= v) lo = m + 1; else hi = m;
    }
    return lo;
}
__device__ __forceinline__ int lower_idx(const int *a, int n, int v) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int m = (lo + hi) >> 1;
        if (a[m] < v) lo = m + 1; else hi = m;
    }
    return lo;
}

// Routing index of one source row: per expert, its nonzero instances in rank
// order with running occurrence ranges.  One CTA per (source, layer).  The
// row of q and the layer's rank masks are staged in shared memory; the CTA
// lays out the layer's instances grouped by expert in rank order (an
// instance's place is its expert's offset plus the number of lower ranks in
// the mask).  That list is cut into equal chunks, one per thread, and one
// scan of (nonzero count, occurrence sum) over the chunks gives every entry
// its place in the row and its occurrence range -- the cost does not depend
// on how many instances a hot expert has.
__global__ void __launch_bounds__(256)
k_row_index(const int32_t *__restrict__ q, const int32_t *__restrict__ iexp,
            const unsigned *__restrict__ imask, int32_t *roff, Entry *rent, Geo g) {
    extern __shared__ __align__(16) int smi[];
    __shared__ int warp_tot[32];
    __shared__ int2 warp_tot2[32];
    __shared__ int cbase[256], vbase[256];
    const int s = blockIdx.x, l = blockIdx.y, E = g.E, R = g.R, nk = g.n_keys, nl = g.n_local;
    const int RW = (R + 31) / 32;
    int *qrow = smi;                                            // [nk], 16-byte aligned
    unsigned *msk = reinterpret_cast<unsigned *>(qrow + ((nk + 3) & ~3));   // [E][RW]
    int *ilist = reinterpret_cast<int *>(msk + E * RW);         // [nk]
    int *ioff = ilist + nk;                                     // [E+1]
    int *ro_s = ioff + E + 1;                                   // [E]
    int *vst = ro_s + E;                                        // [E]
    stage_words(qrow, q + ((int64_t)l * R + s) * nk, nk);
    stage_words(msk, imask + (int64_t)l * E * RW, E * RW);
    cp_async_wait_all();
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
        for (int w = 0; w < RW; ++w) c += __popc(msk[e * RW + w]);
        ioff[e] = c;
    }
    __syncthreads();
    const int n_inst = block_excl_scan(ioff, E, warp_tot);
    if (threadIdx.x == 0) ioff[E] = n_inst;
    const int32_t *ie = iexp + (int64_t)l * nk;
    for (int i0 = threadIdx.x; i0 < nk; i0 += 4 * blockDim.x) {
        int ev[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * blockDim.x;
            ev[u] = i < nk ? __ldg(ie + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = ev[u];
            if (e < 0) continue;
            const int i = i0 + u * blockDim.x;
            const int r = i / nl;
            const unsigned *m = msk + e * RW;
            int j = ioff[e] + __popc(m[r >> 5] & ((1u << (r & 31)) - 1u));
            for (int w = 0; w < (r >> 5); ++w) j += __popc(m[w]);
            ilist[j] = i;
        }
    }
    __syncthreads();
    // Chunk of this thread: odd length so a warp's chunk starts fall in
    // distinct banks.  An expert placed twice on one rank (flagged by the
    // instance index) can leave a list slot unwritten: codes are range-checked
    // before use.
    const int ch = ((n_inst + blockDim.x - 1) / blockDim.x) | 1;
    const int j0 = min(n_inst, (int)threadIdx.x * ch), j1 = min(n_inst, j0 + ch);
    int c = 0, vs = 0;
    {
        int er = lower_idx(ioff, E, j0);                        // first segment starting at >= j0
        for (int j = j0; j < j1; ++j) {
            for (; er < E && ioff[er] == j; ++er) { ro_s[er] = c; vst[er] = vs; }
            const int code = ilist[j];
            const int v = (unsigned)code < (unsigned)nk ? qrow[code] : 0;
            if (v > 0) { ++c; vs += v; }
        }
    }
    const int2 tot = block_excl_scan2(c, vs, warp_tot2);
    cbase[threadIdx.x] = c;
    vbase[threadIdx.x] = vs;
    __syncthreads();
    int32_t *ro = roff + ((int64_t)l * R + s) * (E + 1);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int j = ioff[e];
        int a = tot.x, b = tot.y;
        if (j < n_inst) {
            const int t = j / ch;
            a = ro_s[e] + cbase[t];
            b = vst[e] + vbase[t];
        }
        ro[e] = a;
        vst[e] = b;
    }
    if (threadIdx.x == 0) ro[E] = tot.x;
    __syncthreads();
    Entry *re = rent + ((int64_t)l * R + s) * g.n_inst_cap;
    if (j0 < j1) {
        int e = upper_idx(ioff, E + 1, j0) - 1;                  // segment holding j0
        for (int j = j0; j < j1; ++j) {
            while (ioff[e + 1] <= j) ++e;
            const int code = ilist[j];
            const int v = (unsigned)code < (unsigned)nk ? qrow[code] : 0;
            if (v <= 0) continue;
            const int run = vs - vst[e];
            re[c++] = Entry{code, run, run + v, 0};
            vs += v;
        }
    }
}

// Column prefix of q over sources (stored only where q != 0) and column
// totals.  A CTA covers 32 columns; its 8 warps each scan one chunk of the
// sources (16 loads in flight per lane), and the chunks are prefixed through
// shared memory.
__global__ void __launch_bounds__(256)
k_lay_cols(const int32_t *__restrict__ q, int32_t *soff, int32_t *ccnt, Geo g) {
    __shared__ int part[8][33];
    const int l = blockIdx.y;
    const int lane = threadIdx.x & 31, ch = threadIdx.x >> 5;
    const int i = blockIdx.x * 32 + lane;
    const int chunk = (g.R + 7) / 8;
    const int s0 = ch * chunk, s1 = min(g.R, s0 + chunk);
    const bool col = i < g.n_keys;
    const int32_t *Q = q + (int64_t)l * g.R * g.n_keys + i;
    int32_t *S = soff + (int64_t)l * g.R * g.n_keys + i;
    int sum = 0;
    for (int a = s0; a < s1; a += 16) {
        int v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = (col && a + u < s1) ? __ldg(Q + (int64_t)(a + u) * g.n_keys) : 0;
#pragma unroll
        for (int u = 0; u < 16; ++u) sum += v[u];
    }
    part[ch][lane] = sum;
    __syncthreads();
    int run = 0;
    for (int x = 0; x < ch; ++x) run += part[x][lane];
    if (ch == 7) {
        int tot = run + sum;
        if (col) ccnt[(int64_t)l * g.n_keys + i] = tot;
    }
    for (int a = s0; a < s1; a += 16) {
        int v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = (col && a + u < s1) ? __ldg(Q + (int64_t)(a + u) * g.n_keys) : 0;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if (v[u]) S[(int64_t)(a + u) * g.n_keys] = run;
            run += v[u];
        }
    }
}

// Segment offsets (exclusive prefix of the column totals); zeroes the layout
// statistics.  One CTA per layer: each thread sums a contiguous run of the
// totals, the runs' sums are scanned once, then each run is written out.
__global__ void __launch_bounds__(1024)
k_lay_seg(const int32_t *__restrict__ ccnt, int32_t *lseg, int64_t *lstat, Geo g) {
    __shared__ int warp_tot[32];
    __shared__ int sums[1024];
    const int l = blockIdx.x;
    if (threadIdx.x < TOPO_LAYOUT_STATS) lstat[l * TOPO_LAYOUT_STATS + threadIdx.x] = 0;
    const int32_t *c = ccnt + (int64_t)l * g.n_keys;
    int32_t *o = lseg + (int64_t)l * (g.n_keys + 1);
    const int n = g.n_keys;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int a0 = threadIdx.x * per, a1 = min(n, a0 + per);
    int v[16];
    int local = 0;
    if (per <= 16) {
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = a0 + u < a1 ? __ldg(c + a0 + u) : 0;
#pragma unroll
        for (int u = 0; u < 16; ++u) local += v[u];
    } else {
        for (int a = a0; a < a1; ++a) local += __ldg(c + a);
    }
    sums[threadIdx.x] = local;
    __syncthreads();
    const int total = block_excl_scan(sums, blockDim.x, warp_tot);
    int run = sums[threadIdx.x];
    if (per <= 16) {
#pragma unroll
        for (int u = 0; u < 16; ++u)
            if (a0 + u < a1) {
                o[a0 + u] = run;
                run += v[u];
            }
    } else {
        for (int a = a0; a < a1; ++a) {
            o[a] = run;
            run += __ldg(c + a);
        }
    }
    if (threadIdx.x == 0) o[n] = total;
}

// Per-entry output bases; send counts and locality statistics from the
// routing index.  One CTA per (source, layer).
__global__ void __launch_bounds__(256)
k_lay_entries(const int32_t *__restrict__ roff, Entry *rent, const int32_t *__restrict__ soff,
              const int32_t *__restrict__ lseg, int64_t *lsend, int64_t *lstat, Geo g) {
    extern __shared__ long long sc[];            // [R]
    __shared__ long long red[4][32];
    const int s = blockIdx.x, l = blockIdx.y, R = g.R, nl = g.n_local;
    for (int r = threadIdx.x; r < R; r += blockDim.x) sc[r] = 0;
    __syncthreads();
    const int32_t *ro = roff + ((int64_t)l * R + s) * (g.E + 1);
    Entry *re = rent + ((int64_t)l * R + s) * g.n_inst_cap;
    const int32_t *so = soff + ((int64_t)l * R + s) * g.n_keys;
    const int32_t *seg = lseg + (int64_t)l * (g.n_keys + 1);
    const int n = ro[g.E];
    long long loc = 0, intra = 0, inter = 0, repl = 0;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        Entry x = re[j];
        x.out_base = seg[x.code] + so[x.code] - x.cum_start;
        re[j] = x;
        const int r = x.code / nl, li = x.code % nl;
        const long long v = x.cum_end - x.cum_start;
        atomicAdd(reinterpret_cast<unsigned long long *>(&sc[r]), (unsigned long long)v);
        if (r == s) loc += v;
        else if (r / g.rpn == s / g.rpn) intra += v;
        else inter += v;
        if (li >= g.E_R) repl += v;
    }
    long long vals[4] = {loc, intra, inter, repl};
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int k = 0; k < 4; ++k) {
        long long v = vals[k];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[k][w] = v;
    }
    __syncthreads();
    int64_t *sc_out = lsend + ((int64_t)l * R + s) * R;
    for (int r = threadIdx.x; r < R; r += blockDim.x) sc_out[r] = sc[r];
    if (threadIdx.x < 4) {
        long long t = 0;
        for (int x = 0; x < (int)(blockDim.x >> 5); ++x) t += red[threadIdx.x][x];
        int64_t *st = lstat + l * TOPO_LAYOUT_STATS;
        const int slot = threadIdx.x == 3 ? 6 : threadIdx.x;
        atomicAdd(reinterpret_cast<unsigned long long *>(&st[slot]), (unsigned long long)t);
        if (threadIdx.x < 3)
            atomicAdd(reinterpret_cast<unsigned long long *>(&st[3 + threadIdx.x]),
                      (unsigned long long)(t * g.S_tok));
    }
}

// ---------------------------------------------------------------------------
// Tile kernels
// ---------------------------------------------------------------------------

struct TileGeo {
    int l, s, t;
    int ntok;        // tokens in this tile
    int64_t p0;      // first pair of the tile within its layer
    int64_t slot0;   // base of the tile in the position array (TT * k entries)
};

__device__ __forceinline__ TileGeo tile_geo(const Geo &g) {
    TileGeo tg;
    const int tile = blockIdx.x;
    tg.t = tile % g.tps;
    tg.s = (tile / g.tps) % g.R;
    tg.l = tile / (g.tps * g.R);
    const int tok0 = tg.t * g.TT;
    tg.ntok = max(0, min(g.TT, g.tpr - tok0));
    tg.p0 = ((int64_t)tg.s * g.tpr + tok0) * g.k;
    tg.slot0 = (int64_t)tile * g.TT * g.k;
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
    constexpr int KB = K > 0 ? K : KMAX;
    extern __shared__ int sm[];
    __shared__ int ok;
    if (!check_fp(hdr, hist_fp, false, 0, &ok)) {
        if (threadIdx.x == 0) set_error(hdr, TOPO_ESTATE);
        return;
    }
    if (!kFused && blockIdx.x == 0 && threadIdx.x == 0) hdr->route_fp = fp_mix(hist_fp, route_part);
    const TileGeo tg = tile_geo(g);
    const int E = g.E;
    const int k = K > 0 ? K : g.k;
    const int kp = K > 0 ? ((K & 1) ? K : K + 1) : g.kp;
    const RankSmem S = rank_smem(g, sm);
    const int32_t *ids_layer = ids + (int64_t)tg.l * g.npairs;
    int32_t *dst_layer = dst + (int64_t)tg.l * g.npairs;
    int32_t *sorted_layer = kFused ? sorted + (int64_t)tg.l * g.npairs : nullptr;
    const int32_t *tbase = tile_idx + (((int64_t)tg.l * g.R + tg.s) * g.tps + tg.t) * E;
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
    if (row_in_smem)
        for (int j = threadIdx.x; j < n_ent; j += kRankThreads) {
            S.ent_ce[j] = __ldg(&re[j].cum_end);
            S.ent_code[j] = __ldg(&re[j].code);
            S.ent_ob[j] = __ldg(&re[j].out_base);
        }
    if (threadIdx.x == 0) S.ro[E] = n_ent;
    for (int e = threadIdx.x; e < E; e += kRankThreads) {
        const int b = __ldg(ro + e), en = __ldg(ro + e + 1);
        const int ne = en - b;
        const int code = ne == 1 ? __ldg(&re[b].code) : (ne == 0 ? -2 : -1);
        S.ec[e] = code;
        S.ro[e] = b;
        // per-warp base: tile base (+ out_base when the expert has one entry);
        // pass 1 then adds each warp's count into the following warps' bases
        const int b0 = __ldg(tbase + e) + (ne == 1 ? __ldg(&re[b].out_base) : 0);
#pragma unroll
        for (int x = 0; x < kRankWarps; ++x) {
            S.base[x * E + e] = x == 0 ? b0 : 0;
            S.msk[x * E + e] = 0;
        }
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
        // pass 2: inclusive prefix over warps
        for (int e = threadIdx.x; e < E; e += kRankThreads) {
            int run = 0;
#pragma unroll
            for (int x = 0; x < kRankWarps; ++x) {
                run += S.base[x * E + e];
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
                        if (kFused) {
                            if (code >= 0 && pos >= 0 && pos < g.npairs)
                                sorted_layer[pos] = (int32_t)(tg.p0 + t * k + j);
                            else if (code >= 0)
                                bad_state = true;
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
}

// Layout from the positions topo_reroute stored: sorted[pos] = pair.
__global__ void __launch_bounds__(256)
k_layout_scatter(const int32_t *__restrict__ pos_ws, int32_t *sorted, WsHeader *hdr, Geo g,
                 uint64_t route_part) {
    __shared__ int ok;
    if (!check_fp(hdr, 0, true, route_part, &ok)) {
        if (threadIdx.x == 0) set_error(hdr, TOPO_ESTATE);
        return;
    }
    const TileGeo tg = tile_geo(g);
    const int k = g.k;
    const int n = g.TT * k;
    int32_t *out = sorted + (int64_t)tg.l * g.npairs;
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
}

// Copy the small layout outputs computed by the prep kernels.
__global__ void __launch_bounds__(256)
k_lay_copy(const int32_t *__restrict__ lseg, const int64_t *__restrict__ lsend,
           const int64_t *__restrict__ lstat, int32_t *seg_off, int64_t *send_counts,
           int64_t *layout_stats, const WsHeader *hdr, Geo g, uint64_t route_part, int check) {
    __shared__ int ok;
    if (check && !check_fp(hdr, 0, true, route_part, &ok)) return;
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
}

// Prep shared by topo_reroute and topo_reroute_layout.
cudaError_t launch_prep(const Geo &g, const int32_t *main_rank, const topo_plan_t &p, void *ws,
                        cudaStream_t st) {
    cudaError_t e;
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    if (main_rank && (e = launch_main_tables(g, main_rank, ws, nullptr, 0, st)) != cudaSuccess) return e;
    const int RW = (g.R + 31) / 32;
    if ((e = cudaMemsetAsync(ws_at<unsigned>(ws, g.off_imask), 0, (size_t)g.L * g.E * RW * 4, st)) !=
        cudaSuccess)
        return e;
    k_inst_index<<<dim3((g.n_keys + 255) / 256, g.L), 256, 0, st>>>(
        p.slot_expert, main_rank ? ws_at<int32_t>(ws, g.off_main) : nullptr,
        ws_at<int32_t>(ws, g.off_iexp), ws_at<unsigned>(ws, g.off_imask), hdr, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem_row = row_index_smem(g);
    if ((e = ensure_smem((const void *)k_row_index, smem_row)) != cudaSuccess) return e;
    k_row_index<<<dim3(g.R, g.L), 256, smem_row, st>>>(
        p.route_cnt, ws_at<int32_t>(ws, g.off_iexp), ws_at<unsigned>(ws, g.off_imask),
        ws_at<int32_t>(ws, g.off_roff), ws_at<Entry>(ws, g.off_rent), g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_lay_cols<<<dim3((g.n_keys + 31) / 32, g.L), 256, 0, st>>>(
        p.route_cnt, ws_at<int32_t>(ws, g.off_soff), ws_at<int32_t>(ws, g.off_ccnt), g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_lay_seg<<<g.L, 1024, 0, st>>>(ws_at<int32_t>(ws, g.off_ccnt), ws_at<int32_t>(ws, g.off_lseg),
                                    ws_at<int64_t>(ws, g.off_lstat), g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem_e = (size_t)g.R * 8;
    if ((e = ensure_smem((const void *)k_lay_entries, smem_e)) != cudaSuccess) return e;
    k_lay_entries<<<dim3(g.R, g.L), 256, smem_e, st>>>(
        ws_at<int32_t>(ws, g.off_roff), ws_at<Entry>(ws, g.off_rent), ws_at<int32_t>(ws, g.off_soff),
        ws_at<int32_t>(ws, g.off_lseg), ws_at<int64_t>(ws, g.off_lsend),
        ws_at<int64_t>(ws, g.off_lstat), g);
    return cudaGetLastError();
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
    const int64_t tiles = (int64_t)g.L * g.R * g.tps;
    kern<<<(unsigned)tiles, kRankThreads, smem, st>>>(
        ids, ws_at<int32_t>(ws, g.off_tile), ws_at<int32_t>(ws, g.off_roff),
        ws_at<Entry>(ws, g.off_rent), dst, ws_at<int32_t>(ws, g.off_pos), sorted,
        ws_at<WsHeader>(ws, 0), g, hist_fp, route_part);
    return cudaGetLastError();
}

cudaError_t launch_copy(const Geo &g, int32_t *seg_off, int64_t *send_counts, int64_t *layout_stats,
                        void *ws, uint64_t route_part, int check, cudaStream_t st) {
    const int64_t n = (int64_t)g.L * (g.n_keys + 1 + (int64_t)g.R * g.R + TOPO_LAYOUT_STATS);
    const int64_t want = (n + 255) / 256;
    const int blocks = (int)(want < 1024 ? want : 1024);
    k_lay_copy<<<blocks, 256, 0, st>>>(ws_at<int32_t>(ws, g.off_lseg), ws_at<int64_t>(ws, g.off_lsend),
                                       ws_at<int64_t>(ws, g.off_lstat), seg_off, send_counts,
                                       layout_stats, ws_at<WsHeader>(ws, 0), g, route_part, check);
    return cudaGetLastError();
}

}  // namespace

size_t row_index_smem(const Geo &g) {
    return ((size_t)((g.n_keys + 3) & ~3) + (size_t)g.E * ((g.R + 31) / 32) + g.n_keys + 3 * (size_t)g.E + 1) * 4;
}

size_t rank_smem_bytes(const Geo &g) {
    return ((size_t)2 * g.E + 1 + 3 * (size_t)kRankEntCap) * 4 + (size_t)kRankWarps * g.E * 8 +
           (size_t)g.TT * g.kp * 4;
}

cudaError_t launch_reroute(const Geo &g, const int32_t *main_rank, const int32_t *ids,
                           const topo_plan_t &p, int32_t *dst, void *ws, uint64_t hist_fp,
                           uint64_t route_part, cudaStream_t st) {
    cudaError_t e;
    if ((e = launch_prep(g, main_rank, p, ws, st)) != cudaSuccess) return e;
    return launch_tiles<false>(g, ids, dst, nullptr, ws, hist_fp, route_part, st);
}

cudaError_t launch_layout(const Geo &g, int32_t *sorted, int32_t *seg_off, int64_t *send_counts,
                          int64_t *layout_stats, void *ws, uint64_t route_part, cudaStream_t st) {
    cudaError_t e;
    const int64_t tiles = (int64_t)g.L * g.R * g.tps;
    k_layout_scatter<<<(unsigned)tiles, 256, 0, st>>>(ws_at<int32_t>(ws, g.off_pos), sorted,
                                                      ws_at<WsHeader>(ws, 0), g, route_part);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_copy(g, seg_off, send_counts, layout_stats, ws, route_part, 1, st);
}

cudaError_t launch_reroute_layout(const Geo &g, const int32_t *main_rank, const int32_t *ids,
                                  const topo_plan_t &p, int32_t *dst, int32_t *sorted,
                                  int32_t *seg_off, int64_t *send_counts, int64_t *layout_stats,
                                  void *ws, uint64_t hist_fp, cudaStream_t st) {
    cudaError_t e;
    if ((e = launch_prep(g, main_rank, p, ws, st)) != cudaSuccess) return e;
    if ((e = launch_tiles<true>(g, ids, dst, sorted, ws, hist_fp, 0, st)) != cudaSuccess) return e;
    return launch_copy(g, seg_off, send_counts, layout_stats, ws, 0, 0, st);
}

}  // namespace topo
