// Deduplicated dispatch layout ("Expert Coupling in MoE Pretraining", "Moving
// Correlated Experts Together": a token is sent to a destination rank once,
// with metadata naming the local experts that process it; "MoX: Efficient MoE
// Routing on Direct-Connect Topologies" §2: a per-token destination bitmap).
//
// One row per (token, destination rank), ordered by rank, then by token.  A
// row carries its token and the mask of the token's slots whose instance is
// on that rank (the first slot with a rank stands for the row).  Tiles of
// kDdTile tokens inside one source, one CTA per tile; thread x takes the
// tile's (token, slot) elements x, x + kDdTile, ... of the tile's contiguous
// run of k * tokens ints (coalesced loads, all issued before any use):
//   k_dd_count  per-rank lane masks of the tile's 32-token groups (shared
//               atomicOr of the token's lane bit: a token with several
//               slots on one rank sets it once) -> rows per (tile, rank);
//               the token bitmaps; the pairs sent to another rank
//   k_dd_prefix per (layer, source, rank): tile counts -> exclusive prefix,
//               total -> send counts
//   k_dd_seg    per layer: per-source bases of every rank, the rank segment
//               offsets, and the row statistics
//   k_dd_fill   the same lane masks, prefixed over ranks and groups (CTA
//               scan), give each row its place in (rank, token) order inside
//               the tile; every slot ORs its bit into the row staged in
//               shared memory, and consecutive threads write consecutive
//               rows, so runs of one rank leave as contiguous stores
#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

constexpr int kDdTile = 256;              // tokens per tile = threads per CTA
constexpr int kDdWarps = kDdTile / 32;    // 32-token groups of a tile
constexpr int kDdSegThreads = kDedupMaxRanks;
constexpr int kDdFillCtas = 6;            // resident fill CTAs per SM the registers must allow

struct DdGeo {
    int T, k, R, nl, tpr, tps, RW, L;
    int ntl;                   // tiles per layer (R * tps, or ceil(T / kDdTile) + R)
    const int64_t *roff;       // source offsets or null (equal blocks)
    const int32_t *first;      // first tile of each source (with roff)
    int64_t npairs;
    FastDiv dk, dnl;
};

struct DdTile {
    int l, s, tok0, ntok;      // tok0: first token of the tile within the layer
};

__device__ __forceinline__ DdTile dd_tile(const DdGeo &g) {
    DdTile d;
    d.l = (int)(blockIdx.x / g.ntl);
    const int tile = (int)(blockIdx.x - (unsigned)d.l * g.ntl);
    const TileRef r = tile_ref(g.roff, g.R, g.tpr, g.first, kDdTile, g.tps, tile);
    d.s = r.s;
    d.tok0 = r.tok0;
    d.ntok = r.ntok;
    return d;
}

// The tile's pairs are one contiguous run of ntok * k ints; thread x takes the
// elements e = u * kDdTile + x, u < KB (coalesced), all loads issued first.
template <int KB>
__device__ __forceinline__ void dd_load(const int32_t *__restrict__ src, int n, int *v) {
#pragma unroll
    for (int u = 0; u < KB; ++u) {
        const int e = u * kDdTile + threadIdx.x;
        v[u] = e < n ? __ldg(src + e) : 0;
    }
}

// Exclusive scan of one int per thread over the CTA; returns the thread's
// prefix and writes the total.  Every thread of the CTA must call it.
__device__ __forceinline__ int dd_block_scan(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < nw) warp_tot[lane] = t;
    }
    __syncthreads();
    total = warp_tot[nw - 1];
    const int r = (w ? warp_tot[w - 1] : 0) + x - v;
    __syncthreads();                                      // warp_tot reusable after return
    return r;
}

// Element e of a tile with destination instance v: token i = e / k, slot
// j = e % k, rank r = v / nl.  False for an instance outside [0, R*nl).
__device__ __forceinline__ bool dd_elem(int e, int v, const DdGeo &g, int &i, int &j, int &r) {
    i = (int)fast_quot((unsigned)e, g.dk);
    j = e - i * g.k;
    if ((unsigned)v >= (unsigned)(g.R * g.nl)) return false;
    r = (int)fast_quot((unsigned)v, g.dnl);
    return true;
}

// Rows per (tile, rank): lm[(i / 32) * R + r] gets bit i % 32 for every slot
// of token i on rank r, so a token with several slots on one rank sets one
// bit and the popcounts of a rank's words are its rows in the tile.  The
// token bitmaps are built in shared memory (32-bit words, little-endian
// halves of the 64-bit output words) and stored as the tile's contiguous run.
template <int KB>
__global__ void __launch_bounds__(kDdTile)
k_dd_count(const int32_t *__restrict__ dst, int32_t *__restrict__ tile_cnt,
           unsigned long long *__restrict__ tok_dst, int64_t *stats, WsHeader *hdr, DdGeo g) {
    extern __shared__ unsigned ddc[];
    unsigned *lm = ddc;                                    // [kDdWarps][R] lane masks
    unsigned *bm = ddc + kDdWarps * g.R;                   // [kDdTile][2*RW] token bitmaps
    __shared__ int red[kDdWarps];
    __shared__ int any_bad;
    const DdTile d = dd_tile(g);
    if (d.s < 0) return;                                   // past the last source's tiles
    const int tid = threadIdx.x, lane = tid & 31;
    const int n = d.ntok * g.k;
    const int64_t tokb = d.tok0;
    int v[KB];
    dd_load<KB>(dst + (int64_t)d.l * g.npairs + tokb * g.k, n, v);
    for (int x = tid; x < kDdWarps * g.R; x += kDdTile) lm[x] = 0;
    for (int x = tid; x < kDdTile * 2 * g.RW; x += kDdTile) bm[x] = 0;
    if (tid == 0) any_bad = 0;
    __syncthreads();
    int pr = 0;
    bool bad = false;
#pragma unroll
    for (int u = 0; u < KB; ++u) {
        const int e = u * kDdTile + tid;
        int i, j, r;
        if (e >= n) continue;
        if (dd_elem(e, v[u], g, i, j, r)) {
            atomicOr(&lm[(i >> 5) * g.R + r], 1u << (i & 31));
            atomicOr(&bm[i * 2 * g.RW + (r >> 5)], 1u << (r & 31));
            pr += r != d.s;
        } else {
            bad = true;
        }
    }
    if (bad) any_bad = 1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pr += __shfl_xor_sync(0xffffffffu, pr, o);
    if (lane == 0) red[tid >> 5] = pr;
    __syncthreads();
    int32_t *out = tile_cnt + (int64_t)blockIdx.x * g.R;
    for (int r = tid; r < g.R; r += kDdTile) {
        int c = 0;
#pragma unroll
        for (int x = 0; x < kDdWarps; ++x) c += __popc(lm[x * g.R + r]);
        out[r] = c;
    }
    // the tile's bitmaps are one contiguous run of ntok * RW words
    unsigned long long *td = tok_dst + ((int64_t)d.l * g.T + tokb) * g.RW;
    const int nw = d.ntok * g.RW;
    for (int x = tid; x < nw; x += kDdTile)
        td[x] = (unsigned long long)bm[2 * x] | ((unsigned long long)bm[2 * x + 1] << 32);
    if (tid == 0) {
        long long sum = 0;
#pragma unroll
        for (int w = 0; w < kDdWarps; ++w) sum += red[w];
        if (sum) atomicAdd(reinterpret_cast<unsigned long long *>(stats + (int64_t)d.l * 4 + 3),
                           (unsigned long long)sum);
        if (any_bad) set_error(hdr, TOPO_ESTATE);
    }
}

// One thread per (layer, source, rank): tile counts -> exclusive prefix over
// the source's tiles (32 loads in flight per thread); the total -> send count.
__global__ void __launch_bounds__(256)
k_dd_prefix(int32_t *tile_cnt, int64_t *send, DdGeo g, int64_t ncols) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= ncols) return;
    const int r = (int)(c % g.R);
    const int64_t ls = c / g.R;                            // l * R + s
    const int l = (int)(ls / g.R), s = (int)(ls - (int64_t)l * g.R);
    int tb, te;
    source_tiles(g.roff, g.first, g.tps, s, &tb, &te);
    const int nt = te - tb;
    int32_t *col = tile_cnt + ((int64_t)l * g.ntl + tb) * g.R + r;
    int run = 0;
    for (int t0 = 0; t0 < nt; t0 += 32) {
        int v[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) v[u] = t0 + u < nt ? col[(int64_t)(t0 + u) * g.R] : 0;
#pragma unroll
        for (int u = 0; u < 32; ++u)
            if (t0 + u < nt) {
                col[(int64_t)(t0 + u) * g.R] = run;
                run += v[u];
            }
    }
    send[c] = run;
}

// One CTA per layer, one thread per rank r: src_base[l][s][r] = rows to rank
// r from sources before s (32 loads in flight); seg[l][r] = rows to ranks
// before r (CTA scan); stats[l][0..2] = rows, pairs, rows to another rank.
__global__ void __launch_bounds__(kDdSegThreads)
k_dd_seg(const int64_t *__restrict__ send, int32_t *__restrict__ src_base, int32_t *seg, int64_t *stats,
         DdGeo g) {
    __shared__ int warp_tot[32];
    const int l = blockIdx.x, r = threadIdx.x;
    int run = 0, local = 0;
    if (r < g.R) {
        const int64_t *col = send + (int64_t)l * g.R * g.R + r;
        int32_t *sb = src_base + (int64_t)l * g.R * g.R + r;
        for (int s0 = 0; s0 < g.R; s0 += 32) {
            int v[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) v[u] = s0 + u < g.R ? (int)col[(int64_t)(s0 + u) * g.R] : 0;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                if (s0 + u < g.R) {
                    sb[(int64_t)(s0 + u) * g.R] = run;
                    run += v[u];
                    if (s0 + u == r) local = v[u];
                }
        }
    }
    int total;
    const int pre = dd_block_scan(run, warp_tot, total);
    int loc_total;
    dd_block_scan(local, warp_tot, loc_total);
    if (r < g.R) seg[(int64_t)l * (g.R + 1) + r] = pre;
    if (r == 0) {
        seg[(int64_t)l * (g.R + 1) + g.R] = total;
        stats[(int64_t)l * 4 + 0] = total;
        stats[(int64_t)l * 4 + 1] = g.npairs;
        stats[(int64_t)l * 4 + 2] = total - loc_total;
    }
}

template <int KB>
__global__ void __launch_bounds__(kDdTile, kDdFillCtas)
k_dd_fill(const int32_t *__restrict__ dst, const int32_t *__restrict__ tile_pre,
          const int32_t *__restrict__ src_base, const int32_t *__restrict__ seg,
          int32_t *__restrict__ row_token, unsigned long long *__restrict__ row_slots, DdGeo g) {
    extern __shared__ __align__(16) unsigned ddf[];
    // [kDdWarps][R] (lane mask, tile position) pairs: a slot reads both of its
    // group's words with one 64-bit load
    uint2 *lmb = reinterpret_cast<uint2 *>(ddf);
    int *dlt = reinterpret_cast<int *>(lmb + kDdWarps * g.R);   // [R] global - tile position
    // staged rows [kDdTile*KB]: token | slots << 8 | rank << (8 + k) when the
    // rank fits the word's remaining 24 - k bits (every slot of a row ORs the
    // same rank in); otherwise the rank goes to srk
    unsigned *srow = reinterpret_cast<unsigned *>(dlt + g.R);
    unsigned short *srk = reinterpret_cast<unsigned short *>(srow + kDdTile * KB);
    const bool rk_in_row = g.R <= (1 << (24 - g.k));
    const int rk_shift = 8 + g.k;
    __shared__ int warp_tot[32];
    const DdTile d = dd_tile(g);
    if (d.s < 0) return;                                   // past the last source's tiles
    const int tid = threadIdx.x;
    const int n = d.ntok * g.k;
    const int64_t tokb = d.tok0;
    int v[KB];
    dd_load<KB>(dst + (int64_t)d.l * g.npairs + tokb * g.k, n, v);
    for (int x = tid; x < kDdWarps * g.R; x += kDdTile) lmb[x].x = 0u;
#pragma unroll
    for (int u = 0; u < KB; ++u) srow[u * kDdTile + tid] = 0;
    __syncthreads();
    // element -> packed rank | token << 10 | slot << 18; -1 for padding and
    // invalid elements (those are flagged by k_dd_count)
    int pk[KB];
#pragma unroll
    for (int u = 0; u < KB; ++u) {
        const int e = u * kDdTile + tid;
        int i = 0, j = 0, r = -1;
        pk[u] = -1;
        if (e < n && dd_elem(e, v[u], g, i, j, r)) {
            pk[u] = r | (i << 10) | (j << 18);
            atomicOr(&lmb[(i >> 5) * g.R + r].x, 1u << (i & 31));
        }
    }
    __syncthreads();
    // tile positions: ranks in consecutive chunks of q per thread, scanned over the CTA
    const int q = (g.R + kDdTile - 1) / kDdTile;
    const int r0 = min(tid * q, g.R), r1 = min(r0 + q, g.R);
    int mine = 0;
    for (int r = r0; r < r1; ++r)
#pragma unroll
        for (int x = 0; x < kDdWarps; ++x) mine += __popc(lmb[x * g.R + r].x);
    int nrows;
    int run = dd_block_scan(mine, warp_tot, nrows);
    const int64_t tile = blockIdx.x;
    for (int r = r0; r < r1; ++r) {
        dlt[r] = __ldg(seg + (int64_t)d.l * (g.R + 1) + r) +
                 __ldg(src_base + ((int64_t)d.l * g.R + d.s) * g.R + r) +
                 __ldg(tile_pre + tile * g.R + r) - run;
#pragma unroll
        for (int x = 0; x < kDdWarps; ++x) {
            lmb[x * g.R + r].y = (unsigned)run;
            run += __popc(lmb[x * g.R + r].x);
        }
    }
    __syncthreads();
    // a row's position: its rank's tile base for the token's 32-group, plus
    // the group's earlier tokens with that rank; every slot ORs its bit in
#pragma unroll
    for (int u = 0; u < KB; ++u)
        if (pk[u] >= 0) {
            const int r = pk[u] & 1023, i = (pk[u] >> 10) & 255, j = pk[u] >> 18;
            const int x = (i >> 5) * g.R + r;
            const uint2 mb = lmb[x];
            const int p = (int)mb.y + __popc(mb.x & ((1u << (i & 31)) - 1u));
            if (rk_in_row) {
                atomicOr(&srow[p], (unsigned)i | (1u << (j + 8)) | ((unsigned)r << rk_shift));
            } else {
                atomicOr(&srow[p], (unsigned)i | (1u << (j + 8)));
                srk[p] = (unsigned short)r;
            }
        }
    __syncthreads();
    // consecutive threads write consecutive rows: runs of one rank are contiguous
    int32_t *rt = row_token + (int64_t)d.l * g.npairs;
    unsigned long long *rs = row_slots + (int64_t)d.l * g.npairs;
    const unsigned slot_mask = (1u << g.k) - 1u;             // k <= 16
    for (int p = tid; p < nrows; p += kDdTile) {
        const unsigned v = srow[p];
        const int r = rk_in_row ? (int)(v >> rk_shift) : (int)srk[p];
        const int64_t pos = (int64_t)dlt[r] + p;
        if (pos >= 0 && pos < g.npairs) {
            rt[pos] = (int32_t)(tokb + (v & 255u));
            rs[pos] = (v >> 8) & slot_mask;
        }
    }
}

template <int KB>
size_t dd_fill_smem(const DdGeo &g) {
    return (size_t)2 * kDdWarps * g.R * 4 + (size_t)g.R * 4 + (size_t)kDdTile * KB * 4 +
           (size_t)kDdTile * KB * 2;
}

template <int KB>
cudaError_t run_dedup(const DdGeo &g, const int32_t *dst, int32_t *seg, int32_t *row_token,
                      uint64_t *row_slots, uint64_t *tok_dst, int64_t *send, int64_t *stats,
                      int32_t *tile_cnt, int32_t *src_base, WsHeader *hdr, cudaStream_t st) {
    cudaError_t e;
    const int64_t ntiles = (int64_t)g.L * g.ntl;
    unsigned long long *ts = reinterpret_cast<unsigned long long *>(tok_dst);
    unsigned long long *rs = reinterpret_cast<unsigned long long *>(row_slots);
    if ((e = cudaMemsetAsync(stats, 0, (size_t)g.L * 4 * 8, st)) != cudaSuccess) return e;
    const size_t smc = (size_t)kDdWarps * g.R * 4 + (size_t)kDdTile * 2 * g.RW * 4;
    if ((e = ensure_smem((const void *)k_dd_count<KB>, smc)) != cudaSuccess) return e;
    k_dd_count<KB><<<(unsigned)ntiles, kDdTile, smc, st>>>(dst, tile_cnt, ts, stats, hdr, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t ncols = (int64_t)g.L * g.R * g.R;
    k_dd_prefix<<<(unsigned)((ncols + 255) / 256), 256, 0, st>>>(tile_cnt, send, g, ncols);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_dd_seg<<<g.L, kDdSegThreads, 0, st>>>(send, src_base, seg, stats, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smf = dd_fill_smem<KB>(g);
    if ((e = ensure_smem((const void *)k_dd_fill<KB>, smf)) != cudaSuccess) return e;
    k_dd_fill<KB><<<(unsigned)ntiles, kDdTile, smf, st>>>(dst, tile_cnt, src_base, seg, row_token, rs, g);
    return cudaGetLastError();
}

}  // namespace

namespace {

int dd_tps(const Geo &g) {
    const int tps = (g.tpr + kDdTile - 1) / kDdTile;
    return tps > 0 ? tps : 1;
}

int64_t dd_ntl(const Geo &g) {
    return g.roff ? ((int64_t)g.T + kDdTile - 1) / kDdTile + g.R : (int64_t)g.R * dd_tps(g);
}

}  // namespace

size_t dedup_ws_bytes(const Geo &g, size_t *off_tile, size_t *off_src, size_t *off_first) {
    const size_t f = sizeof(WsHeader);
    const size_t a = (f + (size_t)(g.R + 1) * 4 + 255) & ~size_t(255);
    const size_t b = (a + (size_t)g.L * dd_ntl(g) * g.R * 4 + 255) & ~size_t(255);
    const size_t c = (b + (size_t)g.L * g.R * g.R * 4 + 255) & ~size_t(255);
    if (off_tile) *off_tile = a;
    if (off_src) *off_src = b;
    if (off_first) *off_first = f;
    return c;
}


cudaError_t launch_dedup(const Geo &g, const int32_t *dst, int32_t *seg, int32_t *row_token,
                         uint64_t *row_slots, uint64_t *tok_dst, int64_t *send, int64_t *stats, void *ws,
                         cudaStream_t st) {
    DdGeo d;
    d.T = g.T; d.k = g.k; d.R = g.R; d.nl = g.n_local; d.tpr = g.tpr; d.L = g.L;
    d.tps = dd_tps(g);
    const int64_t ntl = dd_ntl(g);
    if ((int64_t)g.L * ntl > INT32_MAX) return cudaErrorInvalidValue;
    d.ntl = (int)ntl;
    d.roff = g.roff;
    d.RW = (g.R + 63) / 64;
    d.npairs = g.npairs;
    d.dk = make_fast_div((unsigned)(g.k > 0 ? g.k : 1));
    d.dnl = make_fast_div((unsigned)g.n_local);
    size_t off_tile = 0, off_src = 0, off_first = 0;
    dedup_ws_bytes(g, &off_tile, &off_src, &off_first);
    int32_t *tile_cnt = ws_at<int32_t>(ws, off_tile);
    int32_t *src_base = ws_at<int32_t>(ws, off_src);
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    d.first = ws_at<int32_t>(ws, off_first);
    if (g.roff) {
        const cudaError_t e = launch_tile_first(g, kDdTile, ws_at<int32_t>(ws, off_first), hdr, st);
        if (e != cudaSuccess) return e;
    }
#define TOPO_DD(KB) run_dedup<KB>(d, dst, seg, row_token, row_slots, tok_dst, send, stats, tile_cnt, src_base, hdr, st)
    if (g.k <= 1) return TOPO_DD(1);
    if (g.k <= 2) return TOPO_DD(2);
    if (g.k <= 4) return TOPO_DD(4);
    if (g.k <= 8) return TOPO_DD(8);
    if (g.k <= 10) return TOPO_DD(10);
    if (g.k <= kDedupMaxK) return TOPO_DD(16);
#undef TOPO_DD
    return cudaErrorInvalidValue;
}

}  // namespace topo
