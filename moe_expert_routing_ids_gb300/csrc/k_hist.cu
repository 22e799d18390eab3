// Routing matrix Omega (TopoEP §4.1, Eq. 3) and the per-tile expert index.
//
// k_hist_tiles: one CTA per tile of TT tokens inside one source rank's block.
// The tile's ids are all requested up front with 16-byte loads, then counted
// into a shared-memory histogram (integer shared atomics, no float), and the
// CTA stores its counts.  k_hist_prefix: one thread per (layer, source,
// expert) column turns the source's tile counts into exclusive prefixes --
// the index that lets the rerouting kernel rank pairs in one pass -- and
// writes the source's row of Omega.
#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

constexpr int kHistThreads = 512;
constexpr int kHistVec = 6;          // 16-byte loads in flight per thread

// Count one id; an id outside [0, E) goes to the spare counter E (dropped)
// and raises `bad`, without a branch.
__device__ __forceinline__ void count_id(int e, int E, int *cnt, bool &bad) {
    const bool ok = (unsigned)e < (unsigned)E;
    bad |= !ok;
    atomicAdd(&cnt[ok ? e : E], 1);
}

__device__ __forceinline__ void count4(const int4 &x, int E, int *cnt, bool &bad) {
    count_id(x.x, E, cnt, bad);
    count_id(x.y, E, cnt, bad);
    count_id(x.z, E, cnt, bad);
    count_id(x.w, E, cnt, bad);
}

__global__ void __launch_bounds__(kHistThreads, 3)
k_hist_tiles(const int32_t *__restrict__ ids, int32_t *__restrict__ tile_cnt, WsHeader *hdr, Geo g) {
    extern __shared__ int cnt[];                     // [E + 1]: E = the spare counter
    const int E = g.E;
    const int l = blockIdx.x / g.ntl;
    const int tile = blockIdx.x - l * g.ntl;
    for (int e = threadIdx.x; e <= E; e += blockDim.x) cnt[e] = 0;
    pdl_wait();                                    // the ids (and the tile table) may come
                                                   // from the previous kernels
    const TileRef tr = tile_ref(g, g.tfirst, g.TT, g.tps, tile);
    if (tr.s < 0) {                                // past the last source's tiles
        pdl_trigger();
        return;
    }
    const int ntok = tr.ntok;
    const int32_t *a = ids + (int64_t)l * g.npairs + (int64_t)tr.tok0 * g.k;
    const int n = ntok * g.k;
    int head = (int)(((16 - ((uintptr_t)a & 15)) & 15) >> 2);
    if (head > n) head = n;
    const int4 *v = reinterpret_cast<const int4 *>(a + head);
    const int nv = (n - head) >> 2;
    // all of this thread's vectors requested before any is counted; vectors
    // past the end read as the spare id E
    int4 x[kHistVec];
#pragma unroll
    for (int u = 0; u < kHistVec; ++u) {
        const int i = threadIdx.x + u * kHistThreads;
        x[u] = i < nv ? __ldg(v + i) : make_int4(E, E, E, E);
    }
    __syncthreads();                               // histogram zeroed
    bool bad = false;
    for (int i = threadIdx.x; i < head; i += blockDim.x) count_id(__ldg(a + i), E, cnt, bad);
    for (int j = head + nv * 4 + threadIdx.x; j < n; j += blockDim.x) count_id(__ldg(a + j), E, cnt, bad);
    const int nmine = nv > (int)threadIdx.x ? (nv - (int)threadIdx.x + kHistThreads - 1) / kHistThreads : 0;
#pragma unroll
    for (int u = 0; u < kHistVec; ++u)
        if (u < nmine) count4(x[u], E, cnt, bad);
    for (int i = threadIdx.x + kHistVec * kHistThreads; i < nv; i += kHistThreads) count4(__ldg(v + i), E, cnt, bad);
    if (bad) set_error(hdr, TOPO_ERANGE);
    __syncthreads();
    int32_t *mine = tile_cnt + ((int64_t)l * g.ntl + tile) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) mine[e] = cnt[e];
    pdl_trigger();
}

// first[s] for tiles of TT tokens over the source offsets, one CTA: the
// sources' tile counts ceil(len / TT), scanned in chunks of the block; the
// offsets are checked (0 first, T last, never decreasing).  On a bad table
// every first[] is 0, so every tile is empty, and TOPO_EOFFSETS is raised.
constexpr int kFirstThreads = 1024;

__global__ void __launch_bounds__(kFirstThreads)
k_tile_first(const int64_t *__restrict__ off, int32_t *first, WsHeader *hdr, int R, int T, int TT) {
    __shared__ int wsum[kFirstThreads / 32];
    __shared__ int carry, bad;
    pdl_wait();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        carry = 0;
        bad = (__ldg(off) != 0 || __ldg(off + R) != (int64_t)T);
    }
    __syncthreads();
    for (int s0 = 0; s0 < R; s0 += kFirstThreads) {
        const int s = s0 + threadIdx.x;
        int c = 0;
        if (s < R) {
            const int64_t len = __ldg(off + s + 1) - __ldg(off + s);
            if (len < 0 || len > T) bad = 1;
            else c = (int)((len + TT - 1) / TT);
        }
        int inc = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, d);
            if (lane >= d) inc += y;
        }
        if (lane == 31) wsum[w] = inc;
        __syncthreads();
        int before = carry;
        for (int x = 0; x < w; ++x) before += wsum[x];
        if (s < R) first[s] = before + inc - c;
        __syncthreads();
        if (threadIdx.x == kFirstThreads - 1) carry = before + inc;
        __syncthreads();
    }
    if (threadIdx.x == 0) first[R] = carry;
    __syncthreads();
    if (bad) {
        for (int s = threadIdx.x; s <= R; s += kFirstThreads) first[s] = 0;
        if (threadIdx.x == 0) set_error(hdr, TOPO_EOFFSETS);
    }
    pdl_trigger();
}

// One thread per (layer, source, group of V experts): exclusive prefix of
// the source's tile counts in place, and the source's totals into Omega.  V =
// 4 (16-byte loads and stores) when E is a multiple of 4, else 1.  The column
// is read in chunks of kPrefixChunk tiles, every load of a chunk issued before
// any of its stores, so no load waits behind a store.
constexpr int kPrefixChunk = 16;

template <int V>
struct IntV;
template <>
struct IntV<1> {
    using T = int;
    __device__ static void add(int &a, int b) { a += b; }
};
template <>
struct IntV<4> {
    using T = int4;
    __device__ static void add(int4 &a, int4 b) { a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w; }
};

template <int V>
__global__ void __launch_bounds__(256)
k_hist_prefix(int32_t *tile_cnt, int32_t *__restrict__ hist, WsHeader *hdr, Geo g, uint64_t fp,
              int64_t n_cols) {
    using Vt = typename IntV<V>::T;
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // column group
    pdl_wait();
    if (c == 0) {
        hdr->hist_fp = fp;
        hdr->route_fp = 0;                      // any routing index is now stale
    }
    if (c >= n_cols) return;
    const int EV = g.E / V;
    const unsigned row = (unsigned)(c / EV);      // l * R + s
    const int ev = (int)(c - (int64_t)row * EV);
    const int l = (int)(row / (unsigned)g.R), s = (int)(row - (unsigned)l * g.R);
    int tb, te;
    source_tiles(g, g.tfirst, g.tps, s, &tb, &te);
    Vt *col = reinterpret_cast<Vt *>(tile_cnt + ((int64_t)l * g.ntl + tb) * g.E) + ev;
    const int nt = te - tb;
    Vt run;
    memset(&run, 0, sizeof run);
    for (int u0 = 0; u0 < nt; u0 += kPrefixChunk) {
        const int m = min(kPrefixChunk, nt - u0);
        Vt v[kPrefixChunk];
#pragma unroll
        for (int q = 0; q < kPrefixChunk; ++q) {
            if (q < m) v[q] = col[(int64_t)(u0 + q) * EV];
            else memset(&v[q], 0, sizeof(Vt));
        }
#pragma unroll
        for (int q = 0; q < kPrefixChunk; ++q) {
            if (q < m) col[(int64_t)(u0 + q) * EV] = run;
            IntV<V>::add(run, v[q]);
        }
    }
    reinterpret_cast<Vt *>(hist)[c] = run;
    pdl_trigger();
}

}  // namespace

cudaError_t launch_tile_first(const Geo &g, int TT, int32_t *first, WsHeader *hdr, cudaStream_t st) {
    return launch_pdl(k_tile_first, dim3(1), dim3(kFirstThreads), 0, st, g.roff, first, hdr, g.R, g.T, TT);
}

cudaError_t launch_hist(const Geo &g, const int32_t *ids, int32_t *hist, void *ws, uint64_t fp,
                        cudaStream_t st) {
    const int64_t tiles = (int64_t)g.L * g.ntl;
    if (tiles == 0) return cudaSuccess;
    if (tiles > INT32_MAX) return cudaErrorInvalidValue;
    const size_t smem = ((size_t)g.E + 1) * sizeof(int);
    cudaError_t e = ensure_smem((const void *)k_hist_tiles, smem);
    if (e != cudaSuccess) return e;
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    if (g.roff && (e = launch_tile_first(g, g.TT, ws_at<int32_t>(ws, g.off_first), hdr, st)) != cudaSuccess)
        return e;
    if ((e = launch_pdl(k_hist_tiles, dim3((unsigned)tiles), dim3(kHistThreads), smem, st, ids,
                        ws_at<int32_t>(ws, g.off_tile), hdr, g)) != cudaSuccess)
        return e;
    return launch_hist_prefix(g, hist, ws, fp, st);
}

cudaError_t launch_hist_prefix(const Geo &g, int32_t *hist, void *ws, uint64_t fp, cudaStream_t st) {
    const int64_t cols = (int64_t)g.L * g.R * g.E;
    if (cols == 0) return cudaSuccess;
    // 16-byte groups need E % 4 == 0 and a 16-byte aligned Omega (the tile
    // index region is 256-byte aligned)
    if (g.E % 4 == 0 && ((uintptr_t)hist & 15) == 0)
        return launch_pdl(k_hist_prefix<4>, dim3((unsigned)((cols / 4 + 255) / 256)), dim3(256), 0, st,
                          ws_at<int32_t>(ws, g.off_tile), hist, ws_at<WsHeader>(ws, 0), g, fp, cols / 4);
    return launch_pdl(k_hist_prefix<1>, dim3((unsigned)((cols + 255) / 256)), dim3(256), 0, st,
                      ws_at<int32_t>(ws, g.off_tile), hist, ws_at<WsHeader>(ws, 0), g, fp, cols);
}

}  // namespace topo
