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
// (shared 64-bit atomics), writes it as int64 and as int32, and flags the call
// when some entry is too large for k int32 additions.  For R <= 16,
// k_sh_target_t: one thread per token (below), int32 scores unless flagged.
// Otherwise k_sh_target: a group of G lanes (G = the power of
// two >= R, at most 32) scores kShIter tokens in turn, lane i holding ranks
// i, i + G, ...; the group's lanes load a token's ids together (the next
// token's already in flight) and pass each to all lanes by shuffle, and each
// id's M row is one contiguous read, so a warp's groups read whole rows.  The
// best rank is a group shuffle reduction; the next layer's slots on the target
// and on the source are counted per lane and summed per CTA.
#include <climits>

#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

constexpr int kShThreads = 256;
constexpr size_t kShSmemTable = 96 * 1024;   // largest M table staged in shared memory
constexpr int kShIter = 16;                  // tokens per group per CTA
constexpr int kShIterT = 8;                  // tokens per thread per CTA (one thread per token)

struct ShGeo {
    int L, T, E, k, R;
    FastDiv tpr, er;                 // tokens per source; E / R for the contiguous main map
    const int32_t *main_rank;
    const int64_t *roff;             // source offsets [R+1], or null for equal blocks
};

// Source rank of token t: t / tpr for equal blocks, else the last s with
// roff[s] <= t (an empty source never holds a token).
__device__ __forceinline__ int sh_src(const ShGeo &g, int64_t t) {
    if (!g.roff) return (int)fast_quot((unsigned)t, g.tpr);
    int lo = 0, hi = g.R - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(g.roff + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The offsets must run from 0 to T without decreasing.
__global__ void k_sh_check_offsets(const int64_t *__restrict__ roff, int R, int T, WsHeader *hdr) {
    bool bad = threadIdx.x == 0 && (__ldg(roff) != 0 || __ldg(roff + R) != (int64_t)T);
    for (int s = threadIdx.x; s < R; s += blockDim.x) bad |= __ldg(roff + s + 1) < __ldg(roff + s);
    if (bad) set_error(hdr, TOPO_EOFFSETS);
}

__device__ __forceinline__ int sh_rank(const ShGeo &g, int b) {
    return g.main_rank ? __ldg(g.main_rank + b) : (int)fast_quot((unsigned)b, g.er);
}

__global__ void __launch_bounds__(128)
k_sh_table(const int64_t *__restrict__ tr, int64_t *__restrict__ M, int32_t *__restrict__ M32, int *wide,
           WsHeader *hdr, ShGeo g) {
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
    int32_t *dst32 = M32 + (int64_t)row * g.R;
    const long long lim = INT_MAX / g.k;                     // k int32 additions cannot overflow
    for (int r = threadIdx.x; r < g.R; r += blockDim.x) {
        const long long v = (long long)acc[r];
        dst[r] = v;
        const bool fits = v <= lim && v >= -lim;
        dst32[r] = fits ? (int32_t)v : 0;
        if (!fits) atomicOr(wide, 1);
    }
}

// A group's lanes hold a token's slots j = lane, lane + G, ... (KQ registers).
template <int G, int KQ>
__device__ __forceinline__ void sh_load_ids(const int32_t *row, int k, int gl, int *v) {
#pragma unroll
    for (int q = 0; q < KQ; ++q) {
        const int j = gl + q * G;
        v[q] = j < k ? __ldg(row + j) : -1;
    }
}

// RPL: ranks per lane (R <= G * RPL).  KQ: slots per lane (k <= G * KQ).
// SMEM: the layer's table is staged in shared memory (E * R * 8 bytes).
// Each group scores kShIter tokens, the ids of the next one in flight.
template <int G, int RPL, int KQ, bool SMEM>
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
    constexpr int kGroups = kShThreads / G;                   // groups per CTA
    const int grp = threadIdx.x / G;
    const int64_t tok0 = (int64_t)blk * kGroups * kShIter;
    int on_tgt = 0, on_src = 0, moved = 0, pairs = 0;           // per thread: < kShIter * KQ
    bool bad = false;
    const int32_t *cur0 = ids + (int64_t)l * g.T * g.k;
    const int32_t *nxt0 = ids + (int64_t)(l + 1) * g.T * g.k;
    int ca[KQ], cb[KQ];                                       // this token's ids: layer l, l + 1
    int64_t t = tok0 + grp;
    if (t < g.T) {
        sh_load_ids<G, KQ>(cur0 + t * g.k, g.k, gl, ca);
        sh_load_ids<G, KQ>(nxt0 + t * g.k, g.k, gl, cb);
    }
    for (int it = 0; it < kShIter && t < g.T; ++it, t += kGroups) {   // t uniform in the group
        int a_cur[KQ], a_nxt[KQ];
#pragma unroll
        for (int q = 0; q < KQ; ++q) {
            a_cur[q] = ca[q];
            a_nxt[q] = cb[q];
        }
        const int64_t tn = t + kGroups;
        if (it + 1 < kShIter && tn < g.T) {                   // the next token's ids in flight
            sh_load_ids<G, KQ>(cur0 + tn * g.k, g.k, gl, ca);
            sh_load_ids<G, KQ>(nxt0 + tn * g.k, g.k, gl, cb);
        }
        long long sc[RPL];
#pragma unroll
        for (int i = 0; i < RPL; ++i) sc[i] = 0;
#pragma unroll
        for (int q = 0; q < KQ; ++q)
            for (int jj = 0; jj < G; ++jj) {
                if (q * G + jj >= g.k) break;
                const int a = __shfl_sync(gmask, a_cur[q], jj, G);
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
        const int s = sh_src(g, t);
        long long mine = 0;
#pragma unroll
        for (int i = 0; i < RPL; ++i)
            if (gl + i * G == s) mine = sc[i];
        const long long ssc = __shfl_sync(gmask, mine, s % G, G);
        const int tg = ssc == best ? s : br;
        if (gl == 0) {
            target[(int64_t)l * g.T + t] = tg;
            moved += tg != s;
        }
        // next-layer slots on the target and on the source
#pragma unroll
        for (int q = 0; q < KQ; ++q) {
            const int b = a_nxt[q];
            if (gl + q * G >= g.k) continue;
            if ((unsigned)b >= (unsigned)g.E) {
                bad = true;
                continue;
            }
            const int rb = sh_rank(g, b);
            on_tgt += rb == tg;
            on_src += rb == s;
            ++pairs;
        }
    }
    if (bad) set_error(hdr, TOPO_ERANGE);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {                       // a warp's sums stay far below 2^31
        on_tgt += __shfl_xor_sync(0xffffffffu, on_tgt, o);
        on_src += __shfl_xor_sync(0xffffffffu, on_src, o);
        moved += __shfl_xor_sync(0xffffffffu, moved, o);
        pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
    }
    const int warp = threadIdx.x >> 5;
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

// One thread per token, for R <= 2 * RB <= 16 and k <= KV: the token's R
// scores live in registers; the table rows are padded to P = 2 * RB entries
// and read in 16-byte chunks, lane i starting at chunk i mod the chunk count,
// so that the 8 lanes of a quarter-warp read different bank groups.  The
// scores are int32 when the table kernel found every entry small enough for
// k additions (flag *wide clear), else int64: half or all of the reads.
template <int RB, int KV, typename S>
__device__ __forceinline__ void sh_thread_tokens(const int32_t *__restrict__ ids, const S *tab,
                                                 int32_t *__restrict__ target, int l, int64_t tok0,
                                                 const ShGeo &g, int &on_tgt, int &on_src, int &moved,
                                                 int &pairs, bool &bad) {
    constexpr int P = 2 * RB;
    constexpr int CPR = 16 / (int)sizeof(S);                 // ranks per 16-byte chunk
    constexpr int NCH = P / CPR;
    const int lane = threadIdx.x & 31;
    const uint4 *tab4 = reinterpret_cast<const uint4 *>(tab);
    const int32_t *cur0 = ids + (int64_t)l * g.T * g.k;
    const int32_t *nxt0 = ids + (int64_t)(l + 1) * g.T * g.k;
    // 16-byte id loads when every token's slots start 16-byte aligned
    const bool vec = (g.k & 3) == 0 && ((reinterpret_cast<uintptr_t>(ids) & 15) == 0);
    for (int it = 0; it < kShIterT; ++it) {
        const int64_t t = tok0 + (int64_t)it * kShThreads + threadIdx.x;
        if (t >= g.T) break;
        int a[KV], b[KV];
        if (vec) {
#pragma unroll
            for (int j = 0; j < KV; j += 4) {
                int4 x = make_int4(-1, -1, -1, -1), y = x;
                if (j < g.k) {
                    x = __ldg(reinterpret_cast<const int4 *>(cur0 + t * g.k + j));
                    y = __ldg(reinterpret_cast<const int4 *>(nxt0 + t * g.k + j));
                }
                a[j] = x.x; a[j + 1] = x.y; a[j + 2] = x.z; a[j + 3] = x.w;
                b[j] = y.x; b[j + 1] = y.y; b[j + 2] = y.z; b[j + 3] = y.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < KV; ++j) {
                a[j] = j < g.k ? __ldg(cur0 + t * g.k + j) : -1;
                b[j] = j < g.k ? __ldg(nxt0 + t * g.k + j) : -1;
            }
        }
        S acc[P];
#pragma unroll
        for (int c = 0; c < P; ++c) acc[c] = 0;
#pragma unroll
        for (int j = 0; j < KV; ++j) {
            if (j >= g.k) break;
            if ((unsigned)a[j] >= (unsigned)g.E) {
                bad = true;
                continue;
            }
            const uint4 *row = tab4 + a[j] * NCH;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const uint4 v = row[(c + lane) % NCH];
                if constexpr (sizeof(S) == 8) {
                    acc[c * CPR] += (S)(((unsigned long long)v.y << 32) | v.x);
                    acc[c * CPR + 1] += (S)(((unsigned long long)v.w << 32) | v.z);
                } else {
                    acc[c * CPR] += (S)(int)v.x;
                    acc[c * CPR + 1] += (S)(int)v.y;
                    acc[c * CPR + 2] += (S)(int)v.z;
                    acc[c * CPR + 3] += (S)(int)v.w;
                }
            }
        }
        const int s = sh_src(g, t);
        S best = 0, ssc = 0;
        int br = -1;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int r0 = ((c + lane) % NCH) * CPR;
#pragma unroll
            for (int h = 0; h < CPR; ++h) {
                const int r = r0 + h;
                const S v = acc[c * CPR + h];
                if (r < g.R) {
                    if (br < 0 || v > best || (v == best && r < br)) {
                        best = v;
                        br = r;
                    }
                    if (r == s) ssc = v;
                }
            }
        }
        const int tg = ssc == best ? s : br;
        target[(int64_t)l * g.T + t] = tg;
        moved += tg != s;
#pragma unroll
        for (int j = 0; j < KV; ++j) {
            if (j >= g.k) break;
            if ((unsigned)b[j] >= (unsigned)g.E) {
                bad = true;
                continue;
            }
            const int rb = sh_rank(g, b[j]);
            on_tgt += rb == tg;
            on_src += rb == s;
            ++pairs;
        }
    }
}

template <int RB, int KV>
__global__ void __launch_bounds__(kShThreads, 3)
k_sh_target_t(const int32_t *__restrict__ ids, const int64_t *__restrict__ M, const int32_t *__restrict__ M32,
              const int *__restrict__ wide, int32_t *__restrict__ target, int64_t *stats, WsHeader *hdr, ShGeo g,
              int blocks_per_layer) {
    extern __shared__ uint4 tabs[];                          // [E][2 * RB] scores of the chosen width
    __shared__ long long red[4][kShThreads / 32];
    constexpr int P = 2 * RB;
    const int l = blockIdx.x / blocks_per_layer;
    const int blk = blockIdx.x - l * blocks_per_layer;
    const bool w64 = __ldg(wide) != 0;                       // uniform over the launch
    if (w64) {
        long long *tab = reinterpret_cast<long long *>(tabs);
        const int64_t *Ml = M + (int64_t)l * g.E * g.R;
        for (int x = threadIdx.x; x < g.E * P; x += kShThreads) {
            const int a = x / P, r = x - a * P;
            tab[x] = r < g.R ? __ldg(Ml + (int64_t)a * g.R + r) : 0;
        }
    } else {
        int *tab = reinterpret_cast<int *>(tabs);
        const int32_t *Ml = M32 + (int64_t)l * g.E * g.R;
        for (int x = threadIdx.x; x < g.E * P; x += kShThreads) {
            const int a = x / P, r = x - a * P;
            tab[x] = r < g.R ? __ldg(Ml + (int64_t)a * g.R + r) : 0;
        }
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    int on_tgt = 0, on_src = 0, moved = 0, pairs = 0;
    bool bad = false;
    const int64_t tok0 = (int64_t)blk * kShThreads * kShIterT;
    if (w64)
        sh_thread_tokens<RB, KV, long long>(ids, reinterpret_cast<const long long *>(tabs), target, l, tok0, g,
                                            on_tgt, on_src, moved, pairs, bad);
    else
        sh_thread_tokens<RB, KV, int>(ids, reinterpret_cast<const int *>(tabs), target, l, tok0, g, on_tgt,
                                      on_src, moved, pairs, bad);
    if (bad) set_error(hdr, TOPO_ERANGE);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        on_tgt += __shfl_xor_sync(0xffffffffu, on_tgt, o);
        on_src += __shfl_xor_sync(0xffffffffu, on_src, o);
        moved += __shfl_xor_sync(0xffffffffu, moved, o);
        pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
    }
    const int warp = threadIdx.x >> 5;
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

template <int RB, int KV>
cudaError_t run_target_t(const ShGeo &g, const int32_t *ids, const int64_t *M, const int32_t *M32,
                         const int *wide, int32_t *target, int64_t *stats, WsHeader *hdr, cudaStream_t st) {
    const int tok_per_block = kShThreads * kShIterT;
    const int bpl = (g.T + tok_per_block - 1) / tok_per_block;
    const int64_t blocks = (int64_t)(g.L - 1) * bpl;
    if (blocks == 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    const size_t tab = (size_t)g.E * RB * 16;                // room for the int64 table
    cudaError_t e = ensure_smem((const void *)k_sh_target_t<RB, KV>, tab);
    if (e != cudaSuccess) return e;
    k_sh_target_t<RB, KV><<<(unsigned)blocks, kShThreads, tab, st>>>(ids, M, M32, wide, target, stats, hdr, g,
                                                                      bpl);
    return cudaGetLastError();
}

template <int G, int RPL, int KQ>
cudaError_t run_target_kq(const ShGeo &g, const int32_t *ids, const int64_t *M, int32_t *target,
                          int64_t *stats, WsHeader *hdr, cudaStream_t st) {
    const int tok_per_block = (kShThreads / G) * kShIter;
    const int bpl = (g.T + tok_per_block - 1) / tok_per_block;
    const int64_t blocks = (int64_t)(g.L - 1) * bpl;
    if (blocks == 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    const size_t tab = (size_t)g.E * g.R * 8;
    cudaError_t e;
    if (tab <= kShSmemTable) {
        if ((e = ensure_smem((const void *)k_sh_target<G, RPL, KQ, true>, tab)) != cudaSuccess) return e;
        k_sh_target<G, RPL, KQ, true><<<(unsigned)blocks, kShThreads, tab, st>>>(ids, M, target, stats, hdr,
                                                                                  g, bpl);
    } else {
        k_sh_target<G, RPL, KQ, false><<<(unsigned)blocks, kShThreads, 0, st>>>(ids, M, target, stats, hdr,
                                                                                 g, bpl);
    }
    return cudaGetLastError();
}

// KQ = 1 when a group's lanes cover the token's slots, else enough for k <= 64.
template <int G, int RPL>
cudaError_t run_target(const ShGeo &g, const int32_t *ids, const int64_t *M, int32_t *target, int64_t *stats,
                       WsHeader *hdr, cudaStream_t st) {
    if (g.k <= G) return run_target_kq<G, RPL, 1>(g, ids, M, target, stats, hdr, st);
    return run_target_kq<G, RPL, (kMaxK + G - 1) / G>(g, ids, M, target, stats, hdr, st);
}

}  // namespace

// Workspace: header, the int32 "wide" flag (own 256 bytes), the int64 table,
// its int32 copy.
size_t shuffle_ws_bytes(int L, int E, int R) {
    const size_t n = (size_t)(L > 1 ? L - 1 : 0) * E * R;
    return sizeof(WsHeader) + 256 + ((n * 8 + 255) & ~size_t(255)) + ((n * 4 + 255) & ~size_t(255));
}

cudaError_t launch_shuffle(int L, int T, int E, int k, int R, const int32_t *ids, const int64_t *tr,
                           const int32_t *main_rank, const int64_t *rank_offsets, int32_t *target,
                           int64_t *stats, void *ws, cudaStream_t st) {
    if (L < 2) return cudaSuccess;
    ShGeo g;
    g.L = L; g.T = T; g.E = E; g.k = k; g.R = R;
    g.tpr = make_fast_div((unsigned)(R > 0 && T / R > 0 ? T / R : 1));
    g.er = make_fast_div((unsigned)(main_rank ? 1 : E / R));
    g.main_rank = main_rank;
    g.roff = rank_offsets;
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    if (rank_offsets) {
        k_sh_check_offsets<<<1, 256, 0, st>>>(rank_offsets, R, T, hdr);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t n = (size_t)(L - 1) * E * R;
    int *wide = ws_at<int>(ws, sizeof(WsHeader));
    int64_t *M = ws_at<int64_t>(ws, sizeof(WsHeader) + 256);
    int32_t *M32 = ws_at<int32_t>(ws, sizeof(WsHeader) + 256 + ((n * 8 + 255) & ~size_t(255)));
    cudaError_t e = cudaMemsetAsync(stats, 0, (size_t)(L - 1) * 4 * 8, st);
    if (e != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(wide, 0, sizeof(int), st)) != cudaSuccess) return e;
    k_sh_table<<<(unsigned)((L - 1) * E), 128, (size_t)R * 8, st>>>(tr, M, M32, wide, hdr, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (T == 0) return cudaSuccess;
    if (R <= 16 && k <= 16 && (size_t)E * 128 <= kShSmemTable) {   // one thread per token
        const int rb = (R + 1) / 2;
        if (k <= 8) {
            if (rb <= 2) return run_target_t<2, 8>(g, ids, M, M32, wide, target, stats, hdr, st);
            if (rb <= 4) return run_target_t<4, 8>(g, ids, M, M32, wide, target, stats, hdr, st);
            return run_target_t<8, 8>(g, ids, M, M32, wide, target, stats, hdr, st);
        }
        if (rb <= 2) return run_target_t<2, 16>(g, ids, M, M32, wide, target, stats, hdr, st);
        if (rb <= 4) return run_target_t<4, 16>(g, ids, M, M32, wide, target, stats, hdr, st);
        return run_target_t<8, 16>(g, ids, M, M32, wide, target, stats, hdr, st);
    }
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
