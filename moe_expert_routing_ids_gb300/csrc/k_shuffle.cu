// Token-shuffle targets ("Expert Coupling in MoE Pretraining", "Moving Tokens
// Toward Their Next Experts": the experts a token selected at one layer
// predict which GPU holds most of its next experts; the token is moved there
// before the next router runs).
//
//   M_l[a][r]   = sum of tr_l[a][b] over the experts b whose main rank is r
//   score_r(t)  = sum over the token's slots j of M_l[ids_l[t][j]][r]
//   target_l[t] = the best rank; a tie keeps the token on its source rank if
//                 that rank is among the best, else the lowest best rank.
//
// k_sh_table: one CTA per (layer, expert a) sums the row tr_l[a][.] by rank
// (shared 64-bit atomics).  k_sh_target: a group of G lanes (G = the power of
// two >= R, at most 32) scores one token, lane i holding ranks i, i + G, ...;
// each slot's id is one broadcast load and its M row one contiguous read, so
// a warp's groups read whole rows.  The best rank is a group shuffle
// reduction; the next layer's slots on the target and on the source are
// counted per lane and summed per CTA.
#include <climits>

#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

constexpr int kShThreads = 256;
constexpr size_t kShSmemTable = 96 * 1024;   // largest M table staged in shared memory

struct ShGeo {
    int L, T, E, k, R, tpr, er;      // er = E / R for the contiguous main map
    const int32_t *main_rank;
};

__device__ __forceinline__ int sh_rank(const ShGeo &g, int b) {
    return g.main_rank ? __ldg(g.main_rank + b) : b / g.er;
}

__global__ void __launch_bounds__(128)
k_sh_table(const int64_t *__restrict__ tr, int64_t *__restrict__ M, WsHeader *hdr, ShGeo g) {
    extern __shared__ unsigned long long acc[];              // [R]
    const int row = blockIdx.x;                              // l * E + a
    for (int r = threadIdx.x; r < g.R; r += blockDim.x) acc[r] = 0;
    __syncthreads();
    const int64_t *src = tr + (int64_t)row * g.E;
    bool bad = false;
    for (int b = threadIdx.x; b < g.E; b += blockDim.x) {
        const int r = sh_rank(g, b);
        if ((unsigned)r >= (unsigned)g.R) {
            bad = true;
            continue;
        }
        atomicAdd(&acc[r], (unsigned long long)__ldg(src + b));
    }
    if (bad) set_error(hdr, TOPO_EMAP);
    __syncthreads();
    int64_t *dst = M + (int64_t)row * g.R;
    for (int r = threadIdx.x; r < g.R; r += blockDim.x) dst[r] = (int64_t)acc[r];
}

// RPL: ranks per lane (R <= G * RPL).  SMEM: the layer's table is staged in
// shared memory (E * R * 8 bytes).
template <int G, int RPL, bool SMEM>
__global__ void __launch_bounds__(kShThreads)
k_sh_target(const int32_t *__restrict__ ids, const int64_t *__restrict__ M, int32_t *__restrict__ target,
            int64_t *stats, WsHeader *hdr, ShGeo g, int blocks_per_layer) {
    extern __shared__ long long tab[];                       // [E][R] when SMEM
    __shared__ long long red[4][kShThreads / 32];
    const int l = blockIdx.x / blocks_per_layer;
    const int blk = blockIdx.x - l * blocks_per_layer;
    const int64_t *Ml = M + (int64_t)l * g.E * g.R;
    if (SMEM) {
        for (int x = threadIdx.x; x < g.E * g.R; x += kShThreads) tab[x] = __ldg(Ml + x);
        __syncthreads();
    }
    const long long *tp = SMEM ? tab : reinterpret_cast<const long long *>(Ml);
    const int lane = threadIdx.x & 31, gl = lane & (G - 1);
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    const int gpw = 32 / G;                                   // tokens per warp
    const int warp = threadIdx.x >> 5;
    const int64_t t = ((int64_t)blk * (kShThreads / 32) + warp) * gpw + lane / G;
    long long on_tgt = 0, on_src = 0, moved = 0, pairs = 0;
    bool bad = false;
    if (t < g.T) {
        const int32_t *cur = ids + ((int64_t)l * g.T + t) * g.k;
        const int32_t *nxt = ids + ((int64_t)(l + 1) * g.T + t) * g.k;
        long long sc[RPL];
#pragma unroll
        for (int i = 0; i < RPL; ++i) sc[i] = 0;
        for (int j = 0; j < g.k; ++j) {
            const int a = __ldg(cur + j);                    // the same address across the group
            if ((unsigned)a >= (unsigned)g.E) {
                bad = true;
                continue;
            }
            const long long *row = tp + (int64_t)a * g.R;
#pragma unroll
            for (int i = 0; i < RPL; ++i) {
                const int r = gl + i * G;
                if (r < g.R) sc[i] += SMEM ? row[r] : __ldg(row + r);
            }
        }
        // the best (score, rank) of the lane, then of the group; lower rank on ties
        long long best = sc[0];
        int br = gl < g.R ? gl : 0;
#pragma unroll
        for (int i = 1; i < RPL; ++i) {
            const int r = gl + i * G;
            if (r < g.R && sc[i] > best) {
                best = sc[i];
                br = r;
            }
        }
        if (gl >= g.R) best = LLONG_MIN;
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) {
            const long long ob = __shfl_xor_sync(gmask, best, o, G);
            const int orr = __shfl_xor_sync(gmask, br, o, G);
            if (ob > best || (ob == best && orr < br)) {
                best = ob;
                br = orr;
            }
        }
        // the source rank's own score, from the lane that holds it
        const int s = (int)(t / g.tpr);
        long long mine = 0;
#pragma unroll
        for (int i = 0; i < RPL; ++i)
            if (gl + i * G == s) mine = sc[i];
        const long long ssc = __shfl_sync(gmask, mine, s % G, G);
        const int tg = ssc == best ? s : br;
        if (gl == 0) target[(int64_t)l * g.T + t] = tg;
        // next-layer slots on the target and on the source
        for (int j = gl; j < g.k; j += G) {
            const int b = __ldg(nxt + j);
            if ((unsigned)b >= (unsigned)g.E) {
                bad = true;
                continue;
            }
            const int rb = sh_rank(g, b);
            on_tgt += rb == tg;
            on_src += rb == s;
            ++pairs;
        }
        if (gl == 0) moved = tg != s;
    }                                   // a group past the end skips its shuffles as a whole
    if (bad) set_error(hdr, TOPO_ERANGE);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        on_tgt += __shfl_xor_sync(0xffffffffu, on_tgt, o);
        on_src += __shfl_xor_sync(0xffffffffu, on_src, o);
        moved += __shfl_xor_sync(0xffffffffu, moved, o);
        pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
    }
    if (lane == 0) {
        red[0][warp] = on_tgt;
        red[1][warp] = on_src;
        red[2][warp] = moved;
        red[3][warp] = pairs;
    }
    __syncthreads();
    if (threadIdx.x < 4) {
        long long v = 0;
        for (int w = 0; w < kShThreads / 32; ++w) v += red[threadIdx.x][w];
        if (v) atomicAdd(reinterpret_cast<unsigned long long *>(stats + (int64_t)l * 4 + threadIdx.x),
                         (unsigned long long)v);
    }
}

template <int G, int RPL>
cudaError_t run_target(const ShGeo &g, const int32_t *ids, const int64_t *M, int32_t *target, int64_t *stats,
                       WsHeader *hdr, cudaStream_t st) {
    const int tok_per_block = (kShThreads / 32) * (32 / G);
    const int bpl = (g.T + tok_per_block - 1) / tok_per_block;
    const int64_t blocks = (int64_t)(g.L - 1) * bpl;
    if (blocks == 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    const size_t tab = (size_t)g.E * g.R * 8;
    cudaError_t e;
    if (tab <= kShSmemTable) {
        if ((e = ensure_smem((const void *)k_sh_target<G, RPL, true>, tab)) != cudaSuccess) return e;
        k_sh_target<G, RPL, true><<<(unsigned)blocks, kShThreads, tab, st>>>(ids, M, target, stats, hdr, g,
                                                                              bpl);
    } else {
        k_sh_target<G, RPL, false><<<(unsigned)blocks, kShThreads, 0, st>>>(ids, M, target, stats, hdr, g,
                                                                             bpl);
    }
    return cudaGetLastError();
}

}  // namespace

size_t shuffle_ws_bytes(int L, int E, int R) {
    const size_t table = (size_t)(L > 1 ? L - 1 : 0) * E * R * 8;
    return sizeof(WsHeader) + ((table + 255) & ~size_t(255));
}

cudaError_t launch_shuffle(int L, int T, int E, int k, int R, const int32_t *ids, const int64_t *tr,
                           const int32_t *main_rank, int32_t *target, int64_t *stats, void *ws,
                           cudaStream_t st) {
    if (L < 2) return cudaSuccess;
    ShGeo g;
    g.L = L; g.T = T; g.E = E; g.k = k; g.R = R;
    g.tpr = R > 0 && T > 0 ? T / R : 1;
    g.er = main_rank ? 1 : E / R;
    g.main_rank = main_rank;
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    int64_t *M = ws_at<int64_t>(ws, sizeof(WsHeader));
    cudaError_t e = cudaMemsetAsync(stats, 0, (size_t)(L - 1) * 4 * 8, st);
    if (e != cudaSuccess) return e;
    k_sh_table<<<(unsigned)((L - 1) * E), 128, (size_t)R * 8, st>>>(tr, M, hdr, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (T == 0) return cudaSuccess;
    if (R <= 4) return run_target<4, 1>(g, ids, M, target, stats, hdr, st);
    if (R <= 8) return run_target<8, 1>(g, ids, M, target, stats, hdr, st);
    if (R <= 16) return run_target<16, 1>(g, ids, M, target, stats, hdr, st);
    if (R <= 32) return run_target<32, 1>(g, ids, M, target, stats, hdr, st);
    if (R <= 64) return run_target<32, 2>(g, ids, M, target, stats, hdr, st);
    if (R <= 128) return run_target<32, 4>(g, ids, M, target, stats, hdr, st);
    if (R <= kShuffleMaxRanks) return run_target<32, 8>(g, ids, M, target, stats, hdr, st);
    return cudaErrorInvalidValue;
}

}  // namespace topo
