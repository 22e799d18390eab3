// Correlated expert placement ("Expert Coupling in MoE Pretraining", "Moving
// Correlated Experts Together": the co-selection counts form a graph over
// experts, partitioned across GPUs with a fixed number of experts per GPU so
// that frequently co-selected experts share a GPU).
//
// w(a,b) = co[a][b] + co[b][a] for a != b.  Greedy construction: ranks
// r = 0..R-1 in turn take E/R experts, first the unassigned expert of largest
// total weight, then repeatedly the unassigned expert of largest weight to the
// rank's members.  Refinement: while the best swap of two experts on different
// ranks gains, apply it (gain C[a][rb] - C[a][ra] + C[b][ra] - C[b][rb] -
// 2 w(a,b), C[x][r] = weight of x to rank r's members).  Lowest index on ties.
//
// One CTA of kPlThreads per layer.  Each choice takes the best key (value
// desc, index asc): the greedy choices are warp argmaxes made by one warp,
// the swap choice a block argmax over all pairs.  When every pair weight lies
// in [0, 2^36) -- always so for co-selection counts -- the greedy sums stay
// below 2^47 and a key packs into 64 bits (value << 16 | 0xffff - index), so
// that a warp argmax is two 32-bit max reductions.  The symmetrised weights are
// staged in shared memory when E <= kPlSmemE (else read through L1/L2), with
// the connection array and the C table.
#include <climits>

#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

constexpr int kPlThreads = 1024;
constexpr int kPlWarps = kPlThreads / 32;
constexpr int kPlSmemE = 128;         // up to this E the weights are staged in shared memory
constexpr long long kPlaceSwapCap = 1 << 20;   // swaps at most (each raises the weight; a bound on time)
constexpr long long kPlPackedW = 1ll << 36;    // pair weights below this: packed greedy keys

struct PlKey {
    long long v;
    int i;                            // ranks above any key with a larger i at equal v
};

__device__ __forceinline__ bool pl_better(const PlKey &a, const PlKey &b) {
    return a.v > b.v || (a.v == b.v && a.i < b.i);
}

// Block-wide best key; every thread gets the result.  scratch: kPlWarps keys.
__device__ __forceinline__ PlKey pl_block_best(PlKey k, PlKey *scratch) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        PlKey q;
        q.v = __shfl_xor_sync(0xffffffffu, k.v, o);
        q.i = __shfl_xor_sync(0xffffffffu, k.i, o);
        if (pl_better(q, k)) k = q;
    }
    __syncthreads();                                  // scratch free
    if (lane == 0) scratch[w] = k;
    __syncthreads();
    k = scratch[0];
    for (int x = 1; x < kPlWarps; ++x)
        if (pl_better(scratch[x], k)) k = scratch[x];
    return k;
}

// Best key over a warp (every lane gets it).
__device__ __forceinline__ PlKey pl_warp_best(PlKey k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        PlKey q;
        q.v = __shfl_xor_sync(0xffffffffu, k.v, o);
        q.i = __shfl_xor_sync(0xffffffffu, k.i, o);
        if (pl_better(q, k)) k = q;
    }
    return k;
}

// Index of the best packed key over a warp (every lane gets it); key 0: none.
__device__ __forceinline__ int pl_warp_best_packed(unsigned long long key) {
    const unsigned hi = __reduce_max_sync(0xffffffffu, (unsigned)(key >> 32));
    const unsigned lo = __reduce_max_sync(0xffffffffu, (unsigned)(key >> 32) == hi ? (unsigned)key : 0u);
    return 0xffff - (int)(lo & 0xffffu);
}

// Pair weights: from the staged matrix W (E x E) when present, else from co.
struct PlW {
    const int64_t *co;
    const long long *W;
    int E;
    __device__ __forceinline__ long long operator()(int a, int b) const {
        if (W) return W[a * E + b];
        return a == b ? 0 : __ldg(co + (int64_t)a * E + b) + __ldg(co + (int64_t)b * E + a);
    }
};

// Within-rank weight of the map in part (block sum; every thread gets it).
__device__ long long pl_within(const PlW &wt, int E, FastDiv fe, const int *part, long long *red) {
    long long s = 0;
    for (int x = threadIdx.x; x < E * E; x += kPlThreads) {
        const int a = (int)fast_quot((unsigned)x, fe), b = x - a * E;
        if (a < b && part[a] == part[b]) s += wt(a, b);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    long long t = 0;
    for (int x = 0; x < kPlWarps; ++x) t += red[x];
    return t;
}

__global__ void __launch_bounds__(kPlThreads)
k_place(const int64_t *__restrict__ co_all, int32_t *__restrict__ main_rank, int64_t *__restrict__ stats,
        int E, int R, int max_iters, FastDiv fe, int staged) {
    extern __shared__ long long psm[];
    long long *W = psm;                               // [E][E] when staged
    long long *conn = psm + (staged ? (size_t)E * E : 0);   // [E] greedy connection
    long long *tot = conn + E;                        // [E] total weight
    long long *C = tot + E;                           // [E][R]
    int *part = reinterpret_cast<int *>(C + (size_t)E * R);   // [E]
    __shared__ PlKey scratch[kPlWarps];
    __shared__ long long red[kPlWarps];
    const int l = blockIdx.x;
    const int64_t *co = co_all + (int64_t)l * E * E;
    const int per = E / R;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (staged)
        for (int x = threadIdx.x; x < E * E; x += kPlThreads) {
            const int a = (int)fast_quot((unsigned)x, fe), b = x - a * E;
            W[x] = a == b ? 0 : __ldg(co + (int64_t)a * E + b) + __ldg(co + (int64_t)b * E + a);
        }
    const PlW wt{co, staged ? W : nullptr, E};

    // contiguous map, and every expert's total weight (a warp per row)
    for (int e = threadIdx.x; e < E; e += kPlThreads) part[e] = e / per;
    __syncthreads();
    const long long w_contig = pl_within(wt, E, fe, part, red);
    bool wide = false;                                // a weight outside [0, kPlPackedW)
    for (int a = w; a < E; a += kPlWarps) {
        long long s = 0;
        for (int b = lane; b < E; b += 32) {
            const long long v = wt(a, b);
            wide |= v < 0 || v >= kPlPackedW;
            s += v;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) tot[a] = s;
    }
    for (int e = threadIdx.x; e < E; e += kPlThreads) part[e] = -1;
    const bool packed = !__syncthreads_or(wide);     // uniform; also the barrier

    // greedy construction by one warp: each choice is a warp argmax over the
    // unassigned experts of val (tot, then the connection to the rank)
    auto choose = [&](const long long *val) -> int {
        if (packed) {
            unsigned long long key = 0;
            for (int a = lane; a < E; a += 32)
                if (part[a] < 0) {
                    const unsigned long long q = ((unsigned long long)val[a] << 16) | (unsigned)(0xffff - a);
                    key = q > key ? q : key;
                }
            return pl_warp_best_packed(key);
        }
        PlKey k{LLONG_MIN, INT_MAX};
        for (int a = lane; a < E; a += 32)
            if (part[a] < 0) {
                const PlKey q{val[a], a};
                if (pl_better(q, k)) k = q;
            }
        return pl_warp_best(k).i;
    };
    if (w == 0) {
        for (int r = 0; r < R; ++r) {
            int pick = choose(tot);
            __syncwarp();
            if (lane == 0) part[pick] = r;
            for (int b = lane; b < E; b += 32) conn[b] = wt(pick, b);
            __syncwarp();
            for (int n = 1; n < per; ++n) {
                pick = choose(conn);
                __syncwarp();
                if (lane == 0) part[pick] = r;
                for (int b = lane; b < E; b += 32) conn[b] += wt(pick, b);
                __syncwarp();
            }
        }
    }
    __syncthreads();
    const long long w_greedy = pl_within(wt, E, fe, part, red);

    // refinement: C[x][r], then best-gain swaps
    for (int x = threadIdx.x; x < E; x += kPlThreads) {
        long long *cx = C + (size_t)x * R;
        for (int r = 0; r < R; ++r) cx[r] = 0;
        for (int m = 0; m < E; ++m) cx[part[m]] += wt(x, m);
    }
    __syncthreads();
    long long swaps = 0;
    while ((max_iters == 0 || swaps < max_iters) && swaps < kPlaceSwapCap) {
        PlKey k{0, INT_MAX};                          // only a positive gain is taken
        for (int x = threadIdx.x; x < E * E; x += kPlThreads) {
            const int a = (int)fast_quot((unsigned)x, fe), b = x - a * E;
            if (a >= b) continue;
            const int pa = part[a], pb = part[b];
            if (pa == pb) continue;
            const long long g = C[(size_t)a * R + pb] - C[(size_t)a * R + pa] + C[(size_t)b * R + pa] -
                                C[(size_t)b * R + pb] - 2 * wt(a, b);
            const PlKey q{g, x};
            if (g > 0 && pl_better(q, k)) k = q;
        }
        const PlKey best = pl_block_best(k, scratch);
        if (best.i == INT_MAX) break;                 // no swap gains
        const int ba = best.i / E, bb = best.i - ba * E;
        const int pa = part[ba], pb = part[bb];
        __syncthreads();                              // every thread has read part
        for (int x = threadIdx.x; x < E; x += kPlThreads) {
            const long long da = wt(x, ba), db = wt(x, bb);
            C[(size_t)x * R + pa] += db - da;
            C[(size_t)x * R + pb] += da - db;
        }
        if (threadIdx.x == 0) {
            part[ba] = pb;
            part[bb] = pa;
        }
        ++swaps;
        __syncthreads();
    }
    const long long w_final = pl_within(wt, E, fe, part, red);
    for (int e = threadIdx.x; e < E; e += kPlThreads) main_rank[(int64_t)l * E + e] = part[e];
    if (threadIdx.x == 0) {
        stats[(int64_t)l * 4 + 0] = w_contig;
        stats[(int64_t)l * 4 + 1] = w_greedy;
        stats[(int64_t)l * 4 + 2] = w_final;
        stats[(int64_t)l * 4 + 3] = swaps;
    }
}

}  // namespace

size_t place_smem_bytes(int E, int R) {       // without the staged weights
    return (size_t)2 * E * 8 + (size_t)E * R * 8 + (size_t)E * 4;
}

cudaError_t launch_place(int L, int E, int R, int max_iters, const int64_t *co, int32_t *main_rank,
                         int64_t *stats, cudaStream_t st) {
    if (L == 0) return cudaSuccess;
    size_t smem = place_smem_bytes(E, R);
    const int staged = E <= kPlSmemE && smem + (size_t)E * E * 8 <= kSmemMax;
    if (staged) smem += (size_t)E * E * 8;
    cudaError_t e = ensure_smem((const void *)k_place, smem);
    if (e != cudaSuccess) return e;
    k_place<<<L, kPlThreads, smem, st>>>(co, main_rank, stats, E, R, max_iters,
                                         make_fast_div((unsigned)E), staged);
    return cudaGetLastError();
}

}  // namespace topo
