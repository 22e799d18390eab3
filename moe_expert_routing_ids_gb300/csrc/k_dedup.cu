// Deduplicated dispatch layout ("Expert Coupling in MoE Pretraining", "Moving
// Correlated Experts Together": a token is sent to a destination rank once,
// with metadata naming the local experts that process it; "MoX: Efficient MoE
// Routing on Direct-Connect Topologies" §2: a per-token destination bitmap).
//
// One row per (token, destination rank), ordered by rank, then by token.  A
// row carries its token and the mask of the token's slots whose instance is
// on that rank (the first slot with a rank stands for the row).  Tiles of
// kDdTile tokens inside one source, one warp per tile:
//   k_dd_count  distinct ranks per token -> rows per (tile, rank), the
//               token bitmaps, and the statistics
//   k_dd_prefix per (layer, source, rank): tile counts -> exclusive prefix,
//               total -> send counts
//   k_dd_seg    per layer: per-source bases of every rank and the rank
//               segment offsets
//   k_dd_fill   rows ranked in token order inside each round of 32 tokens with
//               a per-rank lane bitmask (popc of the lanes below), written at
//               segment + source base + tile prefix + rank
#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

constexpr int kDdTile = 256;          // tokens per warp tile
constexpr int kDdWarps = 8;
constexpr int kDdMaxRW = kDedupMaxRanks / 64;   // 64-bit words of a token bitmap

struct DdGeo {
    int T, k, R, nl, tpr, tps, RW, L;
    int64_t npairs;
};

// Ranks of a token's k slots and, for the first slot of each rank, the mask
// of all its slots with that rank (0 for the other slots).  KB >= k is the
// compile-time slot count; slots k..KB-1 are empty.
template <int KB>
__device__ __forceinline__ void token_rows(const int32_t *d, int k, int nl, int R, int *rk,
                                           unsigned long long *msk, bool &bad) {
#pragma unroll
    for (int j = 0; j < KB; ++j) {
        rk[j] = -1;
        if (j < k) {
            const int v = __ldg(d + j);
            if ((unsigned)v < (unsigned)(R * nl)) rk[j] = v / nl;
            else bad = true;
        }
    }
#pragma unroll
    for (int j = 0; j < KB; ++j) {
        bool first = rk[j] >= 0;
#pragma unroll
        for (int i = 0; i < j; ++i) first = first && rk[i] != rk[j];
        unsigned long long m = 0;
        if (first) {
#pragma unroll
            for (int i = j; i < KB; ++i) m |= (unsigned long long)(rk[i] == rk[j]) << i;
        }
        msk[j] = m;
    }
}

__device__ __forceinline__ int tile_tokens(const DdGeo &g, int t, int &tok0) {
    tok0 = t * kDdTile;
    return max(0, min(kDdTile, g.tpr - tok0));
}

template <int KB>
__global__ void __launch_bounds__(kDdWarps * 32)
k_dd_count(const int32_t *__restrict__ dst, int32_t *tile_cnt, unsigned long long *tok_dst,
           int64_t *stats, WsHeader *hdr, DdGeo g, int64_t ntiles) {
    extern __shared__ int ddc[];                           // [kDdWarps][R]
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tile = (int64_t)blockIdx.x * kDdWarps + w;
    int *cnt = ddc + w * g.R;
    for (int r = lane; r < g.R; r += 32) cnt[r] = 0;
    __syncwarp();
    if (tile >= ntiles) return;                            // whole warp (no block barrier below)
    const int t = (int)(tile % g.tps), s = (int)((tile / g.tps) % g.R), l = (int)(tile / ((int64_t)g.tps * g.R));
    int tok0;
    const int ntok = tile_tokens(g, t, tok0);
    long long rows = 0, rows_remote = 0, pairs_remote = 0;
    bool bad = false;
    for (int r0 = 0; r0 < ntok; r0 += 32) {
        const int i = r0 + lane;
        if (i >= ntok) continue;
        const int64_t tok = (int64_t)s * g.tpr + tok0 + i;
        int rk[KB];
        unsigned long long m[KB];
        token_rows<KB>(dst + (int64_t)l * g.npairs + tok * g.k, g.k, g.nl, g.R, rk, m, bad);
        unsigned long long bits[kDdMaxRW];
#pragma unroll
        for (int x = 0; x < kDdMaxRW; ++x) bits[x] = 0;
#pragma unroll
        for (int j = 0; j < KB; ++j) {
            if (rk[j] >= 0 && rk[j] != s) ++pairs_remote;
            if (!m[j]) continue;
            atomicAdd(&cnt[rk[j]], 1);
            ++rows;
            if (rk[j] != s) ++rows_remote;
#pragma unroll
            for (int x = 0; x < kDdMaxRW; ++x)
                if (x == (rk[j] >> 6)) bits[x] |= 1ull << (rk[j] & 63);
        }
        unsigned long long *td = tok_dst + ((int64_t)l * g.T + tok) * g.RW;
#pragma unroll
        for (int x = 0; x < kDdMaxRW; ++x)
            if (x < g.RW) td[x] = bits[x];
    }
    __syncwarp();
    int32_t *out = tile_cnt + tile * g.R;
    for (int r = lane; r < g.R; r += 32) out[r] = cnt[r];
    for (int o = 16; o > 0; o >>= 1) {
        rows += __shfl_xor_sync(0xffffffffu, rows, o);
        rows_remote += __shfl_xor_sync(0xffffffffu, rows_remote, o);
        pairs_remote += __shfl_xor_sync(0xffffffffu, pairs_remote, o);
    }
    if (lane == 0) {
        unsigned long long *st = reinterpret_cast<unsigned long long *>(stats + (int64_t)l * 4);
        atomicAdd(&st[0], (unsigned long long)rows);
        atomicAdd(&st[2], (unsigned long long)rows_remote);
        atomicAdd(&st[3], (unsigned long long)pairs_remote);
    }
    if (bad) set_error(hdr, TOPO_ESTATE);
}

// One thread per (layer, source, rank): tile counts -> exclusive prefix over
// the source's tiles; the total -> send count.
__global__ void __launch_bounds__(256)
k_dd_prefix(int32_t *tile_cnt, int64_t *send, DdGeo g, int64_t ncols) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= ncols) return;
    const int r = (int)(c % g.R);
    const int64_t ls = c / g.R;                            // l * R + s
    int32_t *col = tile_cnt + ls * g.tps * g.R + r;
    int run = 0;
    for (int t = 0; t < g.tps; ++t) {
        const int v = col[(int64_t)t * g.R];
        col[(int64_t)t * g.R] = run;
        run += v;
    }
    send[c] = run;
}

// One CTA per layer: src_base[l][s][r] = rows to rank r from sources before s;
// seg[l][r] = rows to ranks before r; stats[l][1] = pairs.
__global__ void __launch_bounds__(1024)
k_dd_seg(const int64_t *__restrict__ send, int32_t *src_base, int32_t *seg, int64_t *stats, DdGeo g) {
    __shared__ int tot[1024];
    __shared__ int carry;
    const int l = blockIdx.x;
    if (threadIdx.x == 0) {
        carry = 0;
        stats[(int64_t)l * 4 + 1] = g.npairs;
    }
    for (int r0 = 0; r0 < g.R; r0 += blockDim.x) {
        const int r = r0 + threadIdx.x;
        int run = 0;
        if (r < g.R)
            for (int s = 0; s < g.R; ++s) {
                const int64_t i = ((int64_t)l * g.R + s) * g.R + r;
                src_base[i] = run;
                run += (int)send[i];
            }
        tot[threadIdx.x] = r < g.R ? run : 0;
        __syncthreads();
        if (threadIdx.x == 0) {                            // prefix of this chunk of ranks
            int c = carry;
            for (int x = 0; x < (int)blockDim.x && r0 + x < g.R; ++x) {
                const int v = tot[x];
                seg[(int64_t)l * (g.R + 1) + r0 + x] = c;
                c += v;
            }
            carry = c;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) seg[(int64_t)l * (g.R + 1) + g.R] = carry;
}

template <int KB>
__global__ void __launch_bounds__(kDdWarps * 32)
k_dd_fill(const int32_t *__restrict__ dst, const int32_t *__restrict__ tile_pre,
          const int32_t *__restrict__ src_base, const int32_t *__restrict__ seg, int32_t *row_token,
          unsigned long long *row_slots, DdGeo g, int64_t ntiles) {
    extern __shared__ int ddf[];                           // [kDdWarps][3][R]
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tile = (int64_t)blockIdx.x * kDdWarps + w;
    if (tile >= ntiles) return;                            // whole warp
    int *gb = ddf + w * 3 * g.R;                           // row position base per rank
    unsigned *msk = reinterpret_cast<unsigned *>(gb + g.R);
    int *base = gb + 2 * g.R;                              // rows already placed in this tile
    const int t = (int)(tile % g.tps), s = (int)((tile / g.tps) % g.R), l = (int)(tile / ((int64_t)g.tps * g.R));
    for (int r = lane; r < g.R; r += 32) {
        gb[r] = __ldg(seg + (int64_t)l * (g.R + 1) + r) +
                __ldg(src_base + ((int64_t)l * g.R + s) * g.R + r) + __ldg(tile_pre + tile * g.R + r);
        msk[r] = 0;
        base[r] = 0;
    }
    __syncwarp();
    int tok0;
    const int ntok = tile_tokens(g, t, tok0);
    const unsigned bit = 1u << lane, lt = bit - 1u;
    int32_t *rt = row_token + (int64_t)l * g.npairs;
    unsigned long long *rs = row_slots + (int64_t)l * g.npairs;
    for (int r0 = 0; r0 < ntok; r0 += 32) {
        const int i = r0 + lane;
        const bool vt = i < ntok;
        const int64_t tok = (int64_t)s * g.tpr + tok0 + i;
        int rk[KB];
        unsigned long long m[KB];
        bool bad = false;
        if (vt) {
            token_rows<KB>(dst + (int64_t)l * g.npairs + tok * g.k, g.k, g.nl, g.R, rk, m, bad);
        } else {
#pragma unroll
            for (int j = 0; j < KB; ++j) { rk[j] = -1; m[j] = 0; }
        }
#pragma unroll
        for (int j = 0; j < KB; ++j)
            if (m[j]) atomicOr(&msk[rk[j]], bit);
        __syncwarp();
        int nb[KB];
        unsigned lead = 0;
#pragma unroll
        for (int j = 0; j < KB; ++j) {
            nb[j] = 0;
            if (!m[j]) continue;
            const unsigned mm = msk[rk[j]];
            const int b = base[rk[j]];
            const int rank = __popc(mm & lt);
            if (rank == 0) {
                lead |= 1u << j;
                nb[j] = b + __popc(mm);
            }
            const int64_t pos = (int64_t)gb[rk[j]] + b + rank;
            if (pos >= 0 && pos < g.npairs) {
                rt[pos] = (int32_t)tok;
                rs[pos] = m[j];
            }
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < KB; ++j)
            if ((lead >> j) & 1u) {
                base[rk[j]] = nb[j];
                msk[rk[j]] = 0;
            }
        __syncwarp();
    }
}

template <int KB>
cudaError_t run_dedup(const DdGeo &g, const int32_t *dst, int32_t *seg, int32_t *row_token,
                      uint64_t *row_slots, uint64_t *tok_dst, int64_t *send, int64_t *stats,
                      int32_t *tile_cnt, int32_t *src_base, WsHeader *hdr, cudaStream_t st) {
    cudaError_t e;
    const int64_t ntiles = (int64_t)g.L * g.R * g.tps;
    const unsigned blocks = (unsigned)((ntiles + kDdWarps - 1) / kDdWarps);
    unsigned long long *ts = reinterpret_cast<unsigned long long *>(tok_dst);
    unsigned long long *rs = reinterpret_cast<unsigned long long *>(row_slots);
    if ((e = cudaMemsetAsync(stats, 0, (size_t)g.L * 4 * 8, st)) != cudaSuccess) return e;
    const size_t smc = (size_t)kDdWarps * g.R * 4;
    if ((e = ensure_smem((const void *)k_dd_count<KB>, smc)) != cudaSuccess) return e;
    k_dd_count<KB><<<blocks, kDdWarps * 32, smc, st>>>(dst, tile_cnt, ts, stats, hdr, g, ntiles);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t ncols = (int64_t)g.L * g.R * g.R;
    k_dd_prefix<<<(unsigned)((ncols + 255) / 256), 256, 0, st>>>(tile_cnt, send, g, ncols);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_dd_seg<<<g.L, 1024, 0, st>>>(send, src_base, seg, stats, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smf = (size_t)kDdWarps * 3 * g.R * 4;
    if ((e = ensure_smem((const void *)k_dd_fill<KB>, smf)) != cudaSuccess) return e;
    k_dd_fill<KB><<<blocks, kDdWarps * 32, smf, st>>>(dst, tile_cnt, src_base, seg, row_token, rs, g,
                                                      ntiles);
    return cudaGetLastError();
}

}  // namespace

size_t dedup_ws_bytes(const Geo &g, size_t *off_tile, size_t *off_src) {
    const int tps = (g.tpr + kDdTile - 1) / kDdTile;
    const size_t a = sizeof(WsHeader);
    const size_t b = (a + (size_t)g.L * g.R * (tps > 0 ? tps : 1) * g.R * 4 + 255) & ~size_t(255);
    const size_t c = (b + (size_t)g.L * g.R * g.R * 4 + 255) & ~size_t(255);
    if (off_tile) *off_tile = a;
    if (off_src) *off_src = b;
    return c;
}


cudaError_t launch_dedup(const Geo &g, const int32_t *dst, int32_t *seg, int32_t *row_token,
                         uint64_t *row_slots, uint64_t *tok_dst, int64_t *send, int64_t *stats, void *ws,
                         cudaStream_t st) {
    DdGeo d;
    d.T = g.T; d.k = g.k; d.R = g.R; d.nl = g.n_local; d.tpr = g.tpr; d.L = g.L;
    d.tps = (g.tpr + kDdTile - 1) / kDdTile;
    if (d.tps < 1) d.tps = 1;
    d.RW = (g.R + 63) / 64;
    d.npairs = g.npairs;
    size_t off_tile = 0, off_src = 0;
    dedup_ws_bytes(g, &off_tile, &off_src);
    int32_t *tile_cnt = ws_at<int32_t>(ws, off_tile);
    int32_t *src_base = ws_at<int32_t>(ws, off_src);
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
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
