// Rerouting of every (token, slot) pair to an expert instance and the
// dispatch layout (TopoEP §1 / Fig. 5 token rerouting; §5 receive counts
// derived on the GPU).
//
// Both pair scans need, for pair p of source s selecting expert e, its
// occurrence index o = number of earlier pairs of s that select e.  The tile
// index left by topo_hist gives o up to the start of p's tile; inside the
// tile a CTA ranks pairs with warp match_any: each warp owns a contiguous
// slice, counts per expert (pass 1), the slices are prefixed per expert
// (pass 2), and pass 3 walks the slice again in pair order adding
// popc(peers below the lane).  Everything is an integer count, so the result
// is exact and the same on every run.
//
// The instance a pair goes to follows from o: within (s, e) the instances of
// e are filled in ascending rank order, q[s][r][l] pairs each.  The routing
// index stores, per (s, e), the nonzero instances with their running ranges
// [cum_start, cum_end) and -- for the layout -- the output position of the
// range's first pair, out_base, so that a pair's position is out_base + o.
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
    int32_t out_base;   // layout position of occurrence 0 of this (s, e) range
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

// Instances of each expert in ascending rank order, and the expert of each
// instance.  One CTA per layer.
__global__ void __launch_bounds__(512)
k_inst_index(const int32_t *__restrict__ slot_expert, const int32_t *__restrict__ tab, int32_t *iexp,
             int32_t *ioff, int32_t *ilist, WsHeader *hdr, Geo g) {
    extern __shared__ unsigned smem_u[];
    __shared__ int warp_tot[32];
    const int l = blockIdx.x;
    const int E = g.E, R = g.R, nl = g.n_local, ER = g.E_R, ns = g.n_slot;
    const int RW = (R + 31) / 32;
    unsigned *mask = smem_u;                                   // [E][RW]
    int *cnt = reinterpret_cast<int *>(mask + (size_t)E * RW); // [E]
    const int32_t *mains = tab + 2 * E;
    const int32_t *SE = slot_expert + (int64_t)l * R * ns;
    if (l == 0 && threadIdx.x == 0) hdr->route_fp = 0;
    for (int i = threadIdx.x; i < E * RW; i += blockDim.x) mask[i] = 0;
    __syncthreads();
    bool bad = false;
    for (int i = threadIdx.x; i < g.n_keys; i += blockDim.x) {
        const int r = i / nl, li = i % nl;
        int e = li < ER ? mains[r * ER + li] : SE[(int64_t)r * ns + (li - ER)];
        if (e >= E) { bad = true; e = -1; }
        if (e < -1) { bad = true; e = -1; }
        iexp[(int64_t)l * g.n_keys + i] = e;
        if (e >= 0) {
            const unsigned bit = 1u << (r & 31);
            const unsigned old = atomicOr(&mask[e * RW + (r >> 5)], bit);
            if (old & bit) bad = true;                         // expert twice on one rank
        }
    }
    if (bad) set_error(hdr, TOPO_ESTATE);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
        for (int w = 0; w < RW; ++w) c += __popc(mask[e * RW + w]);
        cnt[e] = c;
    }
    __syncthreads();
    const int total = block_excl_scan(cnt, E, warp_tot);
    int32_t *off = ioff + (int64_t)l * (E + 1);
    for (int e = threadIdx.x; e < E; e += blockDim.x) off[e] = cnt[e];
    if (threadIdx.x == 0) off[E] = total;
    for (int i = threadIdx.x; i < g.n_keys; i += blockDim.x) {
        const int e = iexp[(int64_t)l * g.n_keys + i];
        if (e < 0) continue;
        const int r = i / nl;
        const unsigned bit = 1u << (r & 31);
        if (!(mask[e * RW + (r >> 5)] & bit)) continue;
        int below = 0;
        for (int w = 0; w < (r >> 5); ++w) below += __popc(mask[e * RW + w]);
        below += __popc(mask[e * RW + (r >> 5)] & (bit - 1));
        ilist[(int64_t)l * g.n_inst_cap + cnt[e] + below] = i;
    }
}

// Routing index of one source row: per expert, its nonzero instances in
// rank order with running occurrence ranges.  One CTA per (source, layer).
__global__ void __launch_bounds__(256)
k_row_index(const int32_t *__restrict__ q, const int32_t *__restrict__ ioff,
            const int32_t *__restrict__ ilist, int32_t *roff, Entry *rent, Geo g) {
    extern __shared__ int cnt[];                    // [E]
    __shared__ int warp_tot[32];
    const int s = blockIdx.x, l = blockIdx.y, E = g.E;
    const int32_t *row = q + ((int64_t)l * g.R + s) * g.n_keys;
    const int32_t *off = ioff + (int64_t)l * (E + 1);
    const int32_t *lst = ilist + (int64_t)l * g.n_inst_cap;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
        for (int i = off[e]; i < off[e + 1]; ++i) c += row[lst[i]] > 0;
        cnt[e] = c;
    }
    __syncthreads();
    const int total = block_excl_scan(cnt, E, warp_tot);
    int32_t *ro = roff + ((int64_t)l * g.R + s) * (E + 1);
    Entry *re = rent + ((int64_t)l * g.R + s) * g.n_inst_cap;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        ro[e] = cnt[e];
        int pos = cnt[e], run = 0;
        for (int i = off[e]; i < off[e + 1]; ++i) {
            const int code = lst[i];
            const int v = row[code];
            if (v <= 0) continue;
            re[pos++] = Entry{code, run, run + v, 0};
            run += v;
        }
    }
    if (threadIdx.x == 0) ro[E] = total;
}

// ---------------------------------------------------------------------------
// Tile scan shared by rerouting and layout.
// ---------------------------------------------------------------------------

struct TileGeo {
    int l, s, t;
    int64_t p0;   // first pair of the tile within its layer
    int n;        // pairs in the tile
};

__device__ __forceinline__ TileGeo tile_geo(const Geo &g) {
    TileGeo tg;
    const int tile = blockIdx.x;
    tg.t = tile % g.tps;
    tg.s = (tile / g.tps) % g.R;
    tg.l = tile / (g.tps * g.R);
    tg.p0 = (int64_t)tg.s * g.pps + (int64_t)tg.t * kTile;
    int64_t p1 = tg.p0 + kTile;
    const int64_t pend = (int64_t)(tg.s + 1) * g.pps;
    if (p1 > pend) p1 = pend;
    tg.n = p1 > tg.p0 ? (int)(p1 - tg.p0) : 0;
    return tg;
}

// Copy n int32 from global to shared with 16-byte loads where aligned.
__device__ __forceinline__ void stage_tile(const int32_t *a, int n, int32_t *dst) {
    int head = (int)(((16 - ((uintptr_t)a & 15)) & 15) >> 2);
    if (head > n) head = n;
    for (int i = threadIdx.x; i < head; i += blockDim.x) dst[i] = __ldg(a + i);
    const int4 *v = reinterpret_cast<const int4 *>(a + head);
    const int nv = (n - head) >> 2;
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        const int4 x = __ldg(v + i);
        int32_t *o = dst + head + 4 * i;
        o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
    }
    for (int i = head + nv * 4 + threadIdx.x; i < n; i += blockDim.x) dst[i] = __ldg(a + i);
}

// Occurrence ranking inside a staged tile.  key_of(idx) gives the expert of
// the tile's idx-th pair, or -1 for a pair that is skipped.  cntw: [warps][E].
// On return cntw[w][e] holds, for warp w, the occurrence index of the first
// pair of e in w's slice (tile base included); emit(idx, e, occ) is then
// called for every pair in pair order within each warp.
template <typename KeyOf, typename Emit>
__device__ __forceinline__ void rank_tile(int n, int E, const int32_t *tile_base, int *cntw,
                                          KeyOf key_of, Emit emit) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int i = threadIdx.x; i < kScanWarps * E; i += blockDim.x) cntw[i] = 0;
    __syncthreads();
    int *mine = cntw + w * E;
    const int beg = w * kWarpSeg;
    for (int r = 0; r < kWarpSeg / 32 && beg + r * 32 < n; ++r) {
        const int idx = beg + r * 32 + lane;
        const int e = idx < n ? key_of(idx) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (peers & lt_mask) == 0) mine[e] += __popc(peers);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = tile_base[e];
        for (int x = 0; x < kScanWarps; ++x) {
            const int c = cntw[x * E + e];
            cntw[x * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int r = 0; r < kWarpSeg / 32 && beg + r * 32 < n; ++r) {
        const int idx = beg + r * 32 + lane;
        const int e = idx < n ? key_of(idx) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int occ = e >= 0 ? mine[e] + __popc(peers & lt_mask) : 0;
        __syncwarp();
        if (e >= 0 && (peers & lt_mask) == 0) mine[e] += __popc(peers);
        if (idx < n) emit(idx, e, occ);
        __syncwarp();
    }
}

__device__ __forceinline__ bool check_fp(const WsHeader *hdr, uint64_t want, bool mix_hist,
                                         uint64_t part, int *flag) {
    if (threadIdx.x == 0) {
        const uint64_t have = mix_hist ? hdr->route_fp : hdr->hist_fp;
        const uint64_t exp = mix_hist ? fp_mix(hdr->hist_fp, part) : want;
        *flag = (have == exp && have != 0);
    }
    __syncthreads();
    return *flag != 0;
}

__global__ void __launch_bounds__(kScanThreads)
k_reroute_tiles(const int32_t *__restrict__ ids, const int32_t *__restrict__ tile_idx,
                const int32_t *__restrict__ roff, const Entry *__restrict__ rent, int32_t *dst,
                WsHeader *hdr, Geo g, uint64_t hist_fp, uint64_t route_part) {
    extern __shared__ int smem_i[];
    __shared__ int ok;
    int32_t *tile = smem_i;                    // [kTile]
    int *cntw = smem_i + kTile;                // [warps][E]
    if (!check_fp(hdr, hist_fp, false, 0, &ok)) {
        if (threadIdx.x == 0) set_error(hdr, TOPO_ESTATE);
        return;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) hdr->route_fp = fp_mix(hist_fp, route_part);
    const TileGeo tg = tile_geo(g);
    const int E = g.E;
    stage_tile(ids + (int64_t)tg.l * g.npairs + tg.p0, tg.n, tile);
    __syncthreads();
    const int32_t *base = tile_idx + (((int64_t)tg.l * g.R + tg.s) * g.tps + tg.t) * E;
    const int32_t *ro = roff + ((int64_t)tg.l * g.R + tg.s) * (E + 1);
    const Entry *re = rent + ((int64_t)tg.l * g.R + tg.s) * g.n_inst_cap;
    int32_t *out = dst + (int64_t)tg.l * g.npairs + tg.p0;
    bool bad_id = false, bad_state = false;
    rank_tile(
        tg.n, E, base, cntw,
        [&](int idx) {
            const int e = tile[idx];
            return (unsigned)e < (unsigned)E ? e : -1;
        },
        [&](int idx, int e, int occ) {
            int code = -1;
            if (e < 0) {
                bad_id = true;
            } else {
                const int b = __ldg(ro + e), en = __ldg(ro + e + 1);
                for (int j = b; j < en; ++j) {
                    const int ce = __ldg(&re[j].cum_end);
                    if (occ < ce) { code = __ldg(&re[j].code); break; }
                }
                if (code < 0) bad_state = true;
            }
            out[idx] = code;
        });
    if (bad_id) set_error(hdr, TOPO_ERANGE);
    if (bad_state) set_error(hdr, TOPO_ESTATE);
}

// Column prefix of q over sources (only where q != 0) and column totals.
__global__ void __launch_bounds__(256)
k_lay_cols(const int32_t *__restrict__ q, int32_t *soff, int32_t *ccnt, const WsHeader *hdr, Geo g,
           uint64_t route_part) {
    __shared__ int ok;
    if (!check_fp(hdr, 0, true, route_part, &ok)) return;
    const int l = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= g.n_keys) return;
    const int32_t *Q = q + (int64_t)l * g.R * g.n_keys + i;
    int32_t *S = soff + (int64_t)l * g.R * g.n_keys + i;
    int run = 0;
    int s = 0;
    for (; s + 4 <= g.R; s += 4) {
        const int v0 = Q[(int64_t)s * g.n_keys], v1 = Q[(int64_t)(s + 1) * g.n_keys];
        const int v2 = Q[(int64_t)(s + 2) * g.n_keys], v3 = Q[(int64_t)(s + 3) * g.n_keys];
        if (v0) S[(int64_t)s * g.n_keys] = run;
        run += v0;
        if (v1) S[(int64_t)(s + 1) * g.n_keys] = run;
        run += v1;
        if (v2) S[(int64_t)(s + 2) * g.n_keys] = run;
        run += v2;
        if (v3) S[(int64_t)(s + 3) * g.n_keys] = run;
        run += v3;
    }
    for (; s < g.R; ++s) {
        const int v = Q[(int64_t)s * g.n_keys];
        if (v) S[(int64_t)s * g.n_keys] = run;
        run += v;
    }
    ccnt[(int64_t)l * g.n_keys + i] = run;
}

// Segment offsets (exclusive prefix of column totals); zeroes layout stats.
__global__ void __launch_bounds__(1024)
k_lay_seg(const int32_t *__restrict__ ccnt, int32_t *seg_off, int64_t *layout_stats,
          const WsHeader *hdr, Geo g, uint64_t route_part) {
    __shared__ int ok;
    __shared__ int warp_tot[32];
    __shared__ int carry;
    if (!check_fp(hdr, 0, true, route_part, &ok)) return;
    const int l = blockIdx.x;
    if (threadIdx.x < TOPO_LAYOUT_STATS) layout_stats[l * TOPO_LAYOUT_STATS + threadIdx.x] = 0;
    const int32_t *c = ccnt + (int64_t)l * g.n_keys;
    int32_t *o = seg_off + (int64_t)l * (g.n_keys + 1);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < g.n_keys; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const int v = i < g.n_keys ? c[i] : 0;
        int x = v;
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= d) x += y;
        }
        if (lane == 31) warp_tot[w] = x;
        __syncthreads();
        int pre = carry;
        for (int j = 0; j < w; ++j) pre += warp_tot[j];
        if (i < g.n_keys) o[i] = pre + x - v;
        __syncthreads();
        if (threadIdx.x == 0) {
            int t = 0;
            for (int j = 0; j < nw; ++j) t += warp_tot[j];
            carry += t;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) o[g.n_keys] = carry;
}

// Per-entry output bases; send counts and locality statistics from the
// routing index.  One CTA per (source, layer).
__global__ void __launch_bounds__(256)
k_lay_entries(const int32_t *__restrict__ roff, Entry *rent, const int32_t *__restrict__ soff,
              const int32_t *__restrict__ seg_off, int64_t *send_counts, int64_t *layout_stats,
              const WsHeader *hdr, Geo g, uint64_t route_part) {
    extern __shared__ long long sc[];            // [R]
    __shared__ int ok;
    __shared__ long long red[4][32];
    if (!check_fp(hdr, 0, true, route_part, &ok)) return;
    const int s = blockIdx.x, l = blockIdx.y, R = g.R, nl = g.n_local;
    for (int r = threadIdx.x; r < R; r += blockDim.x) sc[r] = 0;
    __syncthreads();
    const int32_t *ro = roff + ((int64_t)l * R + s) * (g.E + 1);
    Entry *re = rent + ((int64_t)l * R + s) * g.n_inst_cap;
    const int32_t *so = soff + ((int64_t)l * R + s) * g.n_keys;
    const int32_t *seg = seg_off + (int64_t)l * (g.n_keys + 1);
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
    int64_t *sc_out = send_counts + ((int64_t)l * R + s) * R;
    for (int r = threadIdx.x; r < R; r += blockDim.x) sc_out[r] = sc[r];
    if (threadIdx.x < 4) {
        long long t = 0;
        for (int x = 0; x < (int)(blockDim.x >> 5); ++x) t += red[threadIdx.x][x];
        int64_t *st = layout_stats + l * TOPO_LAYOUT_STATS;
        const int slot = threadIdx.x == 3 ? 6 : threadIdx.x;
        atomicAdd(reinterpret_cast<unsigned long long *>(&st[slot]), (unsigned long long)t);
        if (threadIdx.x < 3)
            atomicAdd(reinterpret_cast<unsigned long long *>(&st[3 + threadIdx.x]),
                      (unsigned long long)(t * g.S_tok));
    }
}

__global__ void __launch_bounds__(kScanThreads)
k_layout_tiles(const int32_t *__restrict__ dst, const int32_t *__restrict__ tile_idx,
               const int32_t *__restrict__ iexp, const int32_t *__restrict__ roff,
               const Entry *__restrict__ rent, int32_t *sorted, WsHeader *hdr, Geo g,
               uint64_t route_part) {
    extern __shared__ int smem_i[];
    __shared__ int ok;
    int32_t *tile = smem_i;
    int *cntw = smem_i + kTile;
    if (!check_fp(hdr, 0, true, route_part, &ok)) {
        if (threadIdx.x == 0) set_error(hdr, TOPO_ESTATE);
        return;
    }
    const TileGeo tg = tile_geo(g);
    const int E = g.E;
    stage_tile(dst + (int64_t)tg.l * g.npairs + tg.p0, tg.n, tile);
    __syncthreads();
    const int32_t *base = tile_idx + (((int64_t)tg.l * g.R + tg.s) * g.tps + tg.t) * E;
    const int32_t *ro = roff + ((int64_t)tg.l * g.R + tg.s) * (E + 1);
    const Entry *re = rent + ((int64_t)tg.l * g.R + tg.s) * g.n_inst_cap;
    const int32_t *ie = iexp + (int64_t)tg.l * g.n_keys;
    int32_t *out = sorted + (int64_t)tg.l * g.npairs;
    const int n_keys = g.n_keys;
    const int64_t npairs = g.npairs;
    bool bad = false;
    rank_tile(
        tg.n, E, base, cntw,
        [&](int idx) {
            const int code = tile[idx];
            return (unsigned)code < (unsigned)n_keys ? __ldg(ie + code) : -1;
        },
        [&](int idx, int e, int occ) {
            const int code = tile[idx];
            if (e < 0) { bad = true; return; }
            const int b = __ldg(ro + e), en = __ldg(ro + e + 1);
            for (int j = b; j < en; ++j) {
                if (__ldg(&re[j].code) != code) continue;
                const int cs = __ldg(&re[j].cum_start), ce = __ldg(&re[j].cum_end);
                if (occ < cs || occ >= ce) break;
                const int64_t pos = (int64_t)__ldg(&re[j].out_base) + occ;
                if (pos < 0 || pos >= npairs) break;          // plan inconsistent with the pairs
                out[pos] = (int32_t)(tg.p0 + idx);
                return;
            }
            bad = true;
        });
    if (bad) set_error(hdr, TOPO_ESTATE);
}

size_t tile_smem_bytes(const Geo &g) { return (size_t)kTile * 4 + (size_t)kScanWarps * g.E * 4; }

cudaError_t set_smem(const void *fn, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

size_t route_smem_bytes(const Geo &g) {
    const size_t a = tile_smem_bytes(g);
    const size_t b = (size_t)g.E * ((g.R + 31) / 32) * 4 + (size_t)g.E * 4;
    return a > b ? a : b;
}

cudaError_t launch_reroute(const Geo &g, const int32_t *main_rank, const int32_t *ids,
                           const topo_plan_t &p, int32_t *dst, void *ws, uint64_t hist_fp,
                           uint64_t route_part, cudaStream_t st) {
    cudaError_t e;
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    if ((e = launch_main_tables(g, main_rank, ws, nullptr, 0, st)) != cudaSuccess) return e;
    const size_t smem_inst = (size_t)g.E * ((g.R + 31) / 32) * 4 + (size_t)g.E * 4;
    if ((e = set_smem((const void *)k_inst_index, smem_inst)) != cudaSuccess) return e;
    k_inst_index<<<g.L, 512, smem_inst, st>>>(p.slot_expert, ws_at<int32_t>(ws, g.off_main),
                                              ws_at<int32_t>(ws, g.off_iexp),
                                              ws_at<int32_t>(ws, g.off_ioff),
                                              ws_at<int32_t>(ws, g.off_ilist), hdr, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem_row = (size_t)g.E * 4;
    if ((e = set_smem((const void *)k_row_index, smem_row)) != cudaSuccess) return e;
    k_row_index<<<dim3(g.R, g.L), 256, smem_row, st>>>(
        p.route_cnt, ws_at<int32_t>(ws, g.off_ioff), ws_at<int32_t>(ws, g.off_ilist),
        ws_at<int32_t>(ws, g.off_roff), ws_at<Entry>(ws, g.off_rent), g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem_t = tile_smem_bytes(g);
    if ((e = set_smem((const void *)k_reroute_tiles, smem_t)) != cudaSuccess) return e;
    const int64_t tiles = (int64_t)g.L * g.R * g.tps;
    k_reroute_tiles<<<(unsigned)tiles, kScanThreads, smem_t, st>>>(
        ids, ws_at<int32_t>(ws, g.off_tile), ws_at<int32_t>(ws, g.off_roff),
        ws_at<Entry>(ws, g.off_rent), dst, hdr, g, hist_fp, route_part);
    return cudaGetLastError();
}

cudaError_t launch_layout(const Geo &g, const int32_t *dst, const topo_plan_t &p, int32_t *sorted,
                          int32_t *seg_off, int64_t *send_counts, int64_t *layout_stats, void *ws,
                          uint64_t route_part, cudaStream_t st) {
    cudaError_t e;
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    k_lay_cols<<<dim3((g.n_keys + 255) / 256, g.L), 256, 0, st>>>(
        p.route_cnt, ws_at<int32_t>(ws, g.off_soff), ws_at<int32_t>(ws, g.off_ccnt), hdr, g, route_part);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_lay_seg<<<g.L, 1024, 0, st>>>(ws_at<int32_t>(ws, g.off_ccnt), seg_off, layout_stats, hdr, g,
                                    route_part);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem_e = (size_t)g.R * 8;
    if ((e = set_smem((const void *)k_lay_entries, smem_e)) != cudaSuccess) return e;
    k_lay_entries<<<dim3(g.R, g.L), 256, smem_e, st>>>(
        ws_at<int32_t>(ws, g.off_roff), ws_at<Entry>(ws, g.off_rent), ws_at<int32_t>(ws, g.off_soff),
        seg_off, send_counts, layout_stats, hdr, g, route_part);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem_t = tile_smem_bytes(g);
    if ((e = set_smem((const void *)k_layout_tiles, smem_t)) != cudaSuccess) return e;
    const int64_t tiles = (int64_t)g.L * g.R * g.tps;
    k_layout_tiles<<<(unsigned)tiles, kScanThreads, smem_t, st>>>(
        dst, ws_at<int32_t>(ws, g.off_tile), ws_at<int32_t>(ws, g.off_iexp),
        ws_at<int32_t>(ws, g.off_roff), ws_at<Entry>(ws, g.off_rent), sorted, hdr, g, route_part);
    return cudaGetLastError();
}

}  // namespace topo
