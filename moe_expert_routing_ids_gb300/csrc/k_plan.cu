// Two-stage topology-aware replication plan (TopoEP §4.3, Eqs. 9-10).
//
//   k_main_tables   main(e), its local index, and the experts of each rank
//   k_plan_place    one CTA per (domain, layer): demand D (Eq. 4), benefit
//                   b = 2 D S_tok - ||W|| (Eq. 9) and the inter-node placement
//   k_plan_route    one CTA per (source, layer): the even split of omega_{s,e}
//                   over the chosen instances; U and L by integer atomics
//   k_plan_refine   one warp per (domain, layer): intra-node refinement (Eq. 10)
//
// Inter-node placement in closed form: every rank of a domain starts with no
// used slot, so placing candidates one by one on the rank with the fewest used
// slots (ties: lower rank) is a round robin -- the i-th candidate in
// descending-benefit order lands on rank d*rpn + i % rpn, slot i / rpn, while
// i < rpn * n_slot.  The kernel ranks candidates and applies that directly.
//
// Refinement cost in closed form: with a two-level cost matrix only three
// sources change cost when assignments move from r_b to r_t in one domain --
// r_t's own tokens (-c_intra), r_b's own tokens (+c_intra), everyone else 0 --
// so a candidate's cost needs only q[r_t][r_b][l], q[r_b][r_b][l] and U, which
// the warp keeps in shared memory for the domain's own sources.
#include <cuda_runtime.h>

#include <climits>

#include "common.cuh"

namespace topo {
namespace {

__device__ __forceinline__ int64_t block_sum64(int64_t v, int64_t *red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    int64_t t = 0;
    for (int i = 0; i < nw; ++i) t += red[i];
    return t;
}

// main(e), local index of e on main(e), and mains[r][j] (ascending e).
__global__ void k_main_tables(const int32_t *__restrict__ main_rank, int32_t *tab, int64_t *stats,
                              int n_stats, WsHeader *hdr, Geo g) {
    extern __shared__ int own[];
    __shared__ int bad;
    pdl_wait();
    pdl_trigger();
    const int E = g.E, R = g.R, ER = g.E_R;
    int32_t *main_of = tab, *main_l = tab + E, *mains = tab + 2 * E;
    for (int i = threadIdx.x; i < n_stats; i += blockDim.x) stats[i] = 0;
    if (threadIdx.x == 0) {
        bad = 0;
        if (stats) hdr->route_fp = 0;   // a new plan makes any routing index stale
    }
    for (int r = threadIdx.x; r < R; r += blockDim.x) own[r] = 0;
    __syncthreads();
    if (main_rank) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            int r = main_rank[e];
            if (r < 0 || r >= R) bad = 1;
            else atomicAdd(&own[r], 1);
        }
        __syncthreads();
        for (int r = threadIdx.x; r < R; r += blockDim.x)
            if (own[r] != ER) bad = 1;
        __syncthreads();
        if (!bad) {
            for (int e = threadIdx.x; e < E; e += blockDim.x) {
                const int r = main_rank[e];
                int li = 0;
                for (int x = 0; x < e; ++x) li += (main_rank[x] == r);
                main_of[e] = r;
                main_l[e] = li;
                mains[r * ER + li] = e;
            }
            return;
        }
        if (threadIdx.x == 0) set_error(hdr, TOPO_EMAP);
    }
    // contiguous map (also the in-bounds fallback after TOPO_EMAP)
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        main_of[e] = e / ER;
        main_l[e] = e % ER;
        mains[e] = e;
    }
}

__global__ void __launch_bounds__(512)
k_plan_place(const int32_t *__restrict__ hist, const int32_t *__restrict__ tab, int32_t *slot_expert,
             int32_t *rep, int32_t *inst_load, int32_t *rank_load, int64_t *stats, Geo g, int npow) {
    // candidates sorted by (benefit desc, expert asc) in shared memory:
    // keyv[i] the benefit (LLONG_MIN: not a candidate), kid[i] the expert
    extern __shared__ long long keyv[];          // [npow], then int kid[npow]
    int *kid = reinterpret_cast<int *>(keyv + npow);
    __shared__ int ncand;
    __shared__ int64_t red[32];
    __shared__ int stat_load[kMaxRanksPerNode];
    pdl_wait();
    pdl_trigger();
    const int d = blockIdx.x, l = blockIdx.y;
    const int E = g.E, R = g.R, rpn = g.rpn, ns = g.n_slot, nl = g.n_local;
    const int32_t *main_of = tab, *mains = tab + 2 * E;
    const int32_t *H = hist + (int64_t)l * R * E;
    if (threadIdx.x == 0) ncand = 0;
    if (threadIdx.x < rpn) stat_load[threadIdx.x] = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < npow; e += blockDim.x) {
        long long key = LLONG_MIN;
        if (e < E) {
            int64_t D = 0;
#pragma unroll 8
            for (int j = 0; j < rpn; ++j) D += H[(int64_t)(d * rpn + j) * E + e];
            const int64_t b = 2 * D * g.S_tok - g.W;
            if ((main_of[e] / rpn != d) && b > 0) {
                key = (long long)b;
                atomicAdd(&ncand, 1);
            }
        }
        keyv[e] = key;
        kid[e] = e;
    }
    int32_t *SE = slot_expert + (int64_t)l * R * ns;
    for (int i = threadIdx.x; i < rpn * ns; i += blockDim.x) SE[(int64_t)d * rpn * ns + i] = -1;
    for (int e = threadIdx.x; e < E; e += blockDim.x) rep[((int64_t)l * E + e) * g.M + d] = -1;
    __syncthreads();
    const int cap = rpn * ns;
    const int placed = ncand < cap ? ncand : cap;
    int64_t repcost = 0;
    if (npow <= 256) {
        // few experts: each candidate counts the candidates ahead of it
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const long long b = keyv[e];
            if (b == LLONG_MIN) continue;
            int rank = 0;
            for (int x = 0; x < E; ++x) {
                const long long bx = keyv[x];
                rank += (bx > b) || (bx == b && x < e);
            }
            if (rank < cap) {
                const int r = d * rpn + rank % rpn, slot = rank / rpn;
                SE[(int64_t)r * ns + slot] = e;
                rep[((int64_t)l * E + e) * g.M + d] = r * nl + g.E_R + slot;
                repcost += cost_sr(g, main_of[e], r) * g.W;
            }
        }
    } else {
    // bitonic sort, descending by benefit, ascending by expert on ties
    for (int size = 2; size <= npow; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < (npow >> 1); i += blockDim.x) {
                const int a = 2 * i - (i & (stride - 1)), b = a + stride;
                const long long ka = keyv[a], kb = keyv[b];
                const int ia = kid[a], ib = kid[b];
                const bool a_first = ka > kb || (ka == kb && ia < ib);   // a precedes b
                const bool desc = (a & size) == 0;
                if (desc != a_first) {
                    keyv[a] = kb; keyv[b] = ka;
                    kid[a] = ib; kid[b] = ia;
                }
            }
            __syncthreads();
        }
    }
    for (int rank = threadIdx.x; rank < placed; rank += blockDim.x) {
        const int e = kid[rank];
        const int r = d * rpn + rank % rpn, slot = rank / rpn;
        SE[(int64_t)r * ns + slot] = e;
        rep[((int64_t)l * E + e) * g.M + d] = r * nl + g.E_R + slot;
        repcost += cost_sr(g, main_of[e], r) * g.W;
    }
    }
    // static loads of the domain's ranks (mains only): each thread sums one
    // main over a strided group of sources, the groups meet in shared atomics
    const int nm = rpn * g.E_R;
    const int groups = nm < (int)blockDim.x ? (int)blockDim.x / nm : 1;
    for (int i = threadIdx.x; i < nm * groups; i += blockDim.x) {
        const int jm = i % nm, grp = i / nm;
        const int j = jm / g.E_R, r = d * rpn + j;
        const int e = mains[r * g.E_R + jm % g.E_R];
        int load = 0;
#pragma unroll 8
        for (int s = grp; s < R; s += groups) load += H[(int64_t)s * E + e];
        atomicAdd(&stat_load[j], load);
    }
    // zeroed U, L
    for (int i = threadIdx.x; i < rpn * nl; i += blockDim.x)
        inst_load[((int64_t)l * R + d * rpn) * nl + i] = 0;
    for (int j = threadIdx.x; j < rpn; j += blockDim.x) rank_load[(int64_t)l * R + d * rpn + j] = 0;
    const int64_t tot = block_sum64(repcost, red);
    if (threadIdx.x < rpn)
        atomicMax(reinterpret_cast<unsigned long long *>(&stats[l * TOPO_STATS + 1]),
                  (unsigned long long)stat_load[threadIdx.x]);
    if (threadIdx.x == 0) {
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats[l * TOPO_STATS + 3]),
                  (unsigned long long)placed);
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats[l * TOPO_STATS + 6]),
                  (unsigned long long)tot);
    }
}

__global__ void __launch_bounds__(256)
k_plan_route(const int32_t *__restrict__ hist, const int32_t *__restrict__ tab,
             const int32_t *__restrict__ rep, int32_t *q, int32_t *inst_load, int32_t *rank_load,
             int64_t *stats, Geo g) {
    extern __shared__ int lr[];                  // [R] this row's load per destination rank
    __shared__ int64_t red[32];
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x, l = blockIdx.y;
    const int E = g.E, R = g.R, rpn = g.rpn, nl = g.n_local, M = g.M;
    const int32_t *main_of = tab, *main_l = tab + E;
    const int32_t *REP = rep + (int64_t)l * E * M;
    int32_t *row = q + ((int64_t)l * R + s) * R * nl;
    int32_t *U = inst_load + (int64_t)l * R * nl;
    int32_t *Lr = rank_load + (int64_t)l * R;
    for (int i = threadIdx.x; i < R * nl; i += blockDim.x) row[i] = 0;
    for (int r = threadIdx.x; r < R; r += blockDim.x) lr[r] = 0;
    __syncthreads();
    const int ds = s / rpn;
    int64_t tok = 0, wsum = 0;
    const int32_t *H = hist + ((int64_t)l * R + s) * E;
    auto emit = [&](int r, int li, int amt) {
        if (amt <= 0) return;
        row[r * nl + li] = amt;
        atomicAdd(&U[r * nl + li], amt);
        atomicAdd(&lr[r], amt);
        tok += cost_sr(g, s, r) * amt;
    };
    // two experts per thread and pass, their table entries requested together
    for (int e0 = threadIdx.x; e0 < E; e0 += 2 * blockDim.x) {
        int ew[2], wv[2], me[2], ml[2], rc[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            ew[u] = e0 + u * (int)blockDim.x;
            const bool in = ew[u] < E;
            wv[u] = in ? __ldg(H + ew[u]) : 0;
            me[u] = in ? __ldg(main_of + ew[u]) : 0;
            ml[u] = in ? __ldg(main_l + ew[u]) : 0;
            rc[u] = in ? __ldg(REP + (int64_t)ew[u] * M + ds) : -1;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int w = wv[u];
            if (w == 0) continue;
            wsum += w;
            const int dm = me[u] / rpn;
            if (dm == ds) { emit(me[u], ml[u], w); continue; }
            if (rc[u] >= 0) { emit(rc[u] / nl, rc[u] % nl, w); continue; }
            // no instance in dom(s): every instance of e, in rank (= domain)
            // order; all are cross-domain, so (c, r) order is rank order
            const int32_t *re = REP + (int64_t)ew[u] * M;
            int n = 1;
            for (int d = 0; d < M; ++d) n += (d != dm && __ldg(re + d) >= 0);
            const int base = w / n, rem = w % n;
            int i = 0;
            for (int d = 0; d < M; ++d) {
                int r, li;
                if (d == dm) { r = me[u]; li = ml[u]; }
                else {
                    const int c = __ldg(re + d);
                    if (c < 0) continue;
                    r = c / nl; li = c % nl;
                }
                emit(r, li, base + (i < rem ? 1 : 0));
                ++i;
            }
        }
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x)
        if (lr[r]) atomicAdd(&Lr[r], lr[r]);
    const int64_t t = block_sum64(tok, red);
    const int64_t ws = block_sum64(wsum, red);
    if (threadIdx.x == 0) {
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats[l * TOPO_STATS + 5]),
                  (unsigned long long)(2 * g.S_tok * t));
        atomicAdd(reinterpret_cast<unsigned long long *>(&stats[l * TOPO_STATS + 7]),
                  (unsigned long long)ws);
    }
}

__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// Candidate key, lexicographic, larger is better; a == 0: no candidate.
//   a = delta << 32 | ~L_t          (more moved first, then the lighter target)
//   b = order-preserving map of -cost (cheaper first)
//   c = ~(e << 5 | j_t)              (lower expert, then lower target rank)
struct Key {
    unsigned long long a, b;
    unsigned c;
};

__device__ __forceinline__ bool key_gt(const Key &x, const Key &y) {
    if (x.a != y.a) return x.a > y.a;
    if (x.b != y.b) return x.b > y.b;
    return x.c > y.c;
}

// Lanes holding the warp's largest key: five 32-bit redux steps, each
// keeping only the lanes that tie on every word so far.
__device__ __forceinline__ unsigned warp_argmax_lanes(const Key &k) {
    unsigned live = 0xffffffffu;
    const unsigned words[5] = {(unsigned)(k.a >> 32), (unsigned)k.a, (unsigned)(k.b >> 32),
                               (unsigned)k.b, k.c};
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        const bool in = (live >> (threadIdx.x & 31)) & 1u;
        const unsigned m = __reduce_max_sync(0xffffffffu, in ? words[i] : 0u);
        live = __ballot_sync(0xffffffffu, in && words[i] == m);
    }
    return live;
}

constexpr int kRefineMaxWarps = 8;

// One CTA per (domain, layer) refines the domain (TopoEP §4.3, Eq. 10).
// Candidates (instance at the busiest rank x other rank of the domain) are
// spread over the CTA's warps; each warp reduces with redux/ballot steps, the
// warps' winners meet in shared memory (skipped with one warp, which then
// runs barrier-free), and warp 0 commits.  The domain's columns of q (every
// source, the domain's ranks) live in shared memory when they fit
// (colcache), else in global memory -- updated there by atomic adds that do
// not wait, and re-read past L1 -- with the domain's own sources mirrored in
// shared memory for the candidate costs.
__global__ void __launch_bounds__(kRefineMaxWarps * 32)
k_plan_refine(const int32_t *__restrict__ tab, int32_t *slot_expert, int32_t *q, int32_t *inst_load,
              int32_t *rank_load, int64_t *stats, Geo g, int colcache) {
    extern __shared__ int sm[];
    pdl_wait();
    pdl_trigger();
    __shared__ Key kbuf[kRefineMaxWarps];
    __shared__ int cbuf[kRefineMaxWarps];
    __shared__ int lbuf[kRefineMaxWarps];
    const int d = blockIdx.x, l = blockIdx.y, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nthr = blockDim.x, nwarp = nthr >> 5;
    const int E = g.E, R = g.R, rpn = g.rpn, ns = g.n_slot, nl = g.n_local, ER = g.E_R;
    const int32_t *main_of = tab, *mains = tab + 2 * E;
    int *Lr = sm;                               // [rpn]
    int *used = Lr + rpn;                       // [rpn]
    int *U = used + rpn;                        // [rpn][nl]
    int *xe = U + rpn * nl;                     // [rpn][nl] expert of each instance
    int *xc = xe + rpn * nl;                    // [rpn][nl] main rank of that expert, or
                                                //   -1 - main rank when it is in another domain
    // colcache: qc[s][j][l] for every source s; else qc[js][j][l] for the
    // domain's own sources only
    int *qc = xc + rpn * nl;
    const int nsrc = colcache ? R : rpn;
    short *hl = reinterpret_cast<short *>(qc + nsrc * rpn * nl);   // [rpn][E] local index or -1
    const int r0 = d * rpn;
    const int src0 = colcache ? 0 : r0;         // source index of qc's first row
    int32_t *Q = q + (int64_t)l * R * R * nl;
    int32_t *SE = slot_expert + (int64_t)l * R * ns;

    for (int j = tid; j < rpn; j += nthr) {
        Lr[j] = rank_load[(int64_t)l * R + r0 + j];
        int u = 0;
        while (u < ns && SE[(int64_t)(r0 + j) * ns + u] >= 0) ++u;
        used[j] = u;
    }
    for (int i = tid; i < rpn * E; i += nthr) hl[i] = -1;
    __syncthreads();
    for (int i = tid; i < rpn * nl; i += nthr) {
        const int j = i / nl, li = i % nl, r = r0 + j;
        U[i] = inst_load[((int64_t)l * R + r) * nl + li];
        const int e = li < ER ? mains[r * ER + li] : SE[(int64_t)r * ns + (li - ER)];
        xe[i] = e;
        if (e >= 0) {
            hl[j * E + e] = (short)li;
            const int m = main_of[e];
            xc[i] = (m / rpn == d) ? m : -1 - m;
        } else {
            xc[i] = 0;
        }
    }
    for (int i = tid; i < nsrc * rpn * nl; i += nthr) {
        const int sr = i / (rpn * nl), rest = i % (rpn * nl);
        qc[i] = Q[(int64_t)(src0 + sr) * R * nl + (int64_t)r0 * nl + rest];
    }
    __syncthreads();

    auto qcell = [&](int s, int j, int li) -> int * { return &qc[((s - src0) * rpn + j) * nl + li]; };
    // per-byte cost of a replica on rank r0 + jt of the expert whose main class is xcv
    auto repl_cost = [&](int xcv, int jt) -> int64_t {
        if (xcv < 0) return g.c_inter;
        return xcv == r0 + jt ? 0 : g.c_intra;
    };

    int iters = 0;
    int64_t tokd = 0, repd = 0;
    const int ncand = nl * rpn;
    // this thread's first candidate (lb, jt) and the stride in (lb, jt) form
    const int c_lb0 = tid / rpn, c_jt0 = tid % rpn;
    const int s_lb = nthr / rpn, s_jt = nthr % rpn;
    constexpr int kHardCap = 1 << 24;   // commits provably end; guards a corrupted state only
    while ((g.max_iters == 0 || iters < g.max_iters) && iters < kHardCap) {
        // busiest rank, lowest index on ties (every warp computes it)
        const int myL = lane < rpn ? Lr[lane] : -1;
        const int Lb = __reduce_max_sync(0xffffffffu, myL);
        const int jb = __ffs(__ballot_sync(0xffffffffu, myL == Lb)) - 1;
        Key best{0ull, 0ull, 0u};
        int bc = 0;                              // packed (lb << 5 | jt) of best
        int blt = -1;                            // its local index on jt, -1: a new replica
        int lb = c_lb0, jt = c_jt0;
        for (int c = tid; c < ncand; c += nthr) {
            if (jt != jb) {
                const int Ub = U[jb * nl + lb];
                const int e = xe[jb * nl + lb];
                const int xcv = xc[jb * nl + lb];
                const int Lt = Lr[jt];
                const int usedt = used[jt];
                const int q_rt = *qcell(r0 + jt, jb, lb);
                const int q_rb = *qcell(r0 + jb, jb, lb);
                if (Ub > 0 && e >= 0) {
                    const int lt = hl[jt * E + e];
                    const bool is_new = lt < 0;
                    const int half = (Lb - Lt) >> 1;
                    const int delta = Ub < half ? Ub : half;
                    if (delta >= 1 && (!is_new || usedt < ns)) {
                        const int m_rt = q_rt < delta ? q_rt : delta;
                        const int rest = delta - m_rt;
                        const int others = Ub - q_rt - q_rb;
                        const int m_o = others < rest ? others : rest;
                        const int m_rb = rest - m_o;
                        const int64_t cst = 2 * g.S_tok * g.c_intra * (int64_t)(m_rb - m_rt) +
                                            (is_new ? repl_cost(xcv, jt) * g.W : 0);
                        Key k;
                        k.a = ((unsigned long long)delta << 32) | (unsigned long long)(0xffffffffu - (unsigned)Lt);
                        k.b = ~((unsigned long long)cst ^ 0x8000000000000000ull);
                        k.c = ~(((unsigned)e << 5) | (unsigned)jt);
                        if (key_gt(k, best)) {
                            best = k;
                            bc = (lb << 5) | jt;
                            blt = lt;
                        }
                    }
                }
            }
            lb += s_lb;
            jt += s_jt;
            if (jt >= rpn) { jt -= rpn; ++lb; }
        }
        const unsigned win = warp_argmax_lanes(best);
        const int wl = __ffs(win) - 1;
        Key wk;
        wk.a = __shfl_sync(0xffffffffu, best.a, wl);
        wk.b = __shfl_sync(0xffffffffu, best.b, wl);
        wk.c = __shfl_sync(0xffffffffu, best.c, wl);
        int wc = __shfl_sync(0xffffffffu, bc, wl);
        int wlt = __shfl_sync(0xffffffffu, blt, wl);
        if (nwarp > 1) {
            if (lane == 0) {
                kbuf[w] = wk;
                cbuf[w] = wc;
                lbuf[w] = wlt;
            }
            __syncthreads();
            wk = kbuf[0];
            wc = cbuf[0];
            wlt = lbuf[0];
            for (int x = 1; x < nwarp; ++x)
                if (key_gt(kbuf[x], wk)) {
                    wk = kbuf[x];
                    wc = cbuf[x];
                    wlt = lbuf[x];
                }
        }
        if (wk.a == 0) break;                   // uniform: every thread saw the same keys
        if (w == 0) {
            const int delta = (int)(wk.a >> 32);
            const int blb = wc >> 5, bjt = wc & 31;
            const int e = (int)((~wk.c) >> 5);
            const int xcv = xc[jb * nl + blb];
            const int rb = r0 + jb, rt = r0 + bjt;
            const bool is_new = wlt < 0;
            const int lt = is_new ? ER + used[bjt] : wlt;
            const int m_rt = min(*qcell(rt, jb, blb), delta);
            int remaining = delta - m_rt;
            __syncwarp();
            if (is_new) {
                repd += repl_cost(xcv, bjt) * g.W;
                if (lane == 0) {
                    used[bjt] += 1;
                    hl[bjt * E + e] = (short)lt;
                    xe[bjt * nl + lt] = e;
                    xc[bjt * nl + lt] = xcv;
                    SE[(int64_t)rt * ns + (lt - ER)] = e;
                }
            }
            // other sources, ascending, skipping r_t and r_b: a block of 256
            // sources' q values is requested at once, then scanned 32 at a time
            for (int base = 0; base < R && remaining > 0; base += 256) {
                int v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int s = base + 32 * u + lane;
                    const bool in = s < R && s != rt && s != rb;
                    const bool cached = colcache || (s >= r0 && s < r0 + rpn);
                    v[u] = in ? (cached ? *qcell(s, jb, blb) : __ldcg(&Q[((int64_t)s * R + rb) * nl + blb]))
                              : 0;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (remaining <= 0 || base + 32 * u >= R) break;   // no source left to take from
                    const int s = base + 32 * u + lane;
                    const int incl = warp_incl_scan(v[u]);
                    const int excl = incl - v[u];
                    int take = remaining - excl;
                    take = take < 0 ? 0 : (take > v[u] ? v[u] : take);
                    if (take > 0) {
                        if (colcache || (s >= r0 && s < r0 + rpn)) {
                            *qcell(s, jb, blb) -= take;
                            *qcell(s, bjt, lt) += take;
                        }
                        if (!colcache) {   // no return value: the lane does not wait
                            atomicAdd(&Q[((int64_t)s * R + rb) * nl + blb], -take);
                            atomicAdd(&Q[((int64_t)s * R + rt) * nl + lt], take);
                        }
                    }
                    const int tot = __shfl_sync(0xffffffffu, incl, 31);
                    remaining -= tot < remaining ? tot : remaining;
                }
            }
            const int m_rb = remaining;
            __syncwarp();
            if (lane == 0) {
                if (m_rt > 0) {
                    *qcell(rt, jb, blb) -= m_rt;
                    *qcell(rt, bjt, lt) += m_rt;
                    if (!colcache) {
                        atomicAdd(&Q[((int64_t)rt * R + rb) * nl + blb], -m_rt);
                        atomicAdd(&Q[((int64_t)rt * R + rt) * nl + lt], m_rt);
                    }
                }
                if (m_rb > 0) {
                    *qcell(rb, jb, blb) -= m_rb;
                    *qcell(rb, bjt, lt) += m_rb;
                    if (!colcache) {
                        atomicAdd(&Q[((int64_t)rb * R + rb) * nl + blb], -m_rb);
                        atomicAdd(&Q[((int64_t)rb * R + rt) * nl + lt], m_rb);
                    }
                }
                U[jb * nl + blb] -= delta;
                U[bjt * nl + lt] += delta;
                Lr[jb] -= delta;
                Lr[bjt] += delta;
            }
            tokd += 2 * g.S_tok * g.c_intra * (int64_t)(m_rb - m_rt);
            __syncwarp();
        }
        ++iters;
        if (nwarp > 1) __syncthreads();
    }
    // write back the domain's state and statistics
    if (nwarp > 1) __syncthreads();
    if (colcache)
        for (int i = tid; i < R * rpn * nl; i += nthr) {
            const int sr = i / (rpn * nl), rest = i % (rpn * nl);
            Q[(int64_t)sr * R * nl + (int64_t)r0 * nl + rest] = qc[i];
        }
    for (int j = tid; j < rpn; j += nthr) rank_load[(int64_t)l * R + r0 + j] = Lr[j];
    for (int i = tid; i < rpn * nl; i += nthr) inst_load[((int64_t)l * R + r0) * nl + i] = U[i];
    if (w == 0) {
        int lmax = lane < rpn ? Lr[lane] : 0, nused = lane < rpn ? used[lane] : 0;
        for (int o = 16; o > 0; o >>= 1) {
            lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
            nused += __shfl_xor_sync(0xffffffffu, nused, o);
        }
        if (lane == 0) {
            int64_t *st = stats + l * TOPO_STATS;
            atomicMax(reinterpret_cast<unsigned long long *>(&st[0]), (unsigned long long)lmax);
            atomicAdd(reinterpret_cast<unsigned long long *>(&st[2]), (unsigned long long)nused);
            atomicAdd(reinterpret_cast<unsigned long long *>(&st[4]), (unsigned long long)iters);
            atomicAdd(reinterpret_cast<unsigned long long *>(&st[5]), (unsigned long long)tokd);
            atomicAdd(reinterpret_cast<unsigned long long *>(&st[6]), (unsigned long long)repd);
        }
    }
}

}  // namespace

// Shared memory of the refinement kernel; colcache: all sources' columns.
size_t refine_smem_bytes(const Geo &g, bool colcache) {
    const size_t nsrc = colcache ? (size_t)g.R : (size_t)g.rpn;
    return (2 * (size_t)g.rpn + 3 * (size_t)g.rpn * g.n_local + nsrc * g.rpn * g.n_local) * 4 +
           (size_t)g.rpn * g.E * 2;
}

// Warps of the refinement CTA: about two candidates per lane, at most 8.
int refine_warps(const Geo &g) {
    const int ncand = g.n_local * g.rpn;
    int w = (ncand + 31) / 32;                      // one warp per 32 candidates (measured best)
    return w < 1 ? 1 : (w > kRefineMaxWarps ? kRefineMaxWarps : w);
}

bool refine_colcache(const Geo &g) { return refine_smem_bytes(g, true) <= 160 * 1024; }

cudaError_t launch_main_tables(const Geo &g, const int32_t *main_rank, void *ws, int64_t *stats,
                               int n_stats, cudaStream_t st) {
    return launch_pdl(k_main_tables, dim3(1), dim3(1024), (size_t)g.R * 4, st, main_rank,
                      ws_at<int32_t>(ws, g.off_main), stats, n_stats, ws_at<WsHeader>(ws, 0), g);
}

cudaError_t launch_plan(const Geo &g, const int32_t *main_rank, const int32_t *hist,
                        const topo_plan_t &p, void *ws, cudaStream_t st) {
    cudaError_t e;
    const int32_t *tab = ws_at<int32_t>(ws, g.off_main);
    int32_t *rep = ws_at<int32_t>(ws, g.off_rep);
    if ((e = launch_main_tables(g, main_rank, ws, p.stats, g.L * TOPO_STATS, st)) != cudaSuccess)
        return e;
    int npow = 2;
    while (npow < g.E) npow <<= 1;
    const size_t smem_place = (size_t)npow * 12;
    if ((e = ensure_smem((const void *)k_plan_place, smem_place)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_plan_place, dim3(g.M, g.L), dim3(512), smem_place, st, hist, tab,
                        p.slot_expert, rep, p.inst_load, p.rank_load, p.stats, g, npow)) != cudaSuccess)
        return e;
    if ((e = ensure_smem((const void *)k_plan_route, (size_t)g.R * 4)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_plan_route, dim3(g.R, g.L), dim3(256), (size_t)g.R * 4, st, hist, tab, rep,
                        p.route_cnt, p.inst_load, p.rank_load, p.stats, g)) != cudaSuccess)
        return e;
    const bool cc = refine_colcache(g);
    const size_t smem_ref = refine_smem_bytes(g, cc);
    if ((e = ensure_smem((const void *)k_plan_refine, smem_ref)) != cudaSuccess) return e;
    return launch_pdl(k_plan_refine, dim3(g.M, g.L), dim3(refine_warps(g) * 32), smem_ref, st, tab,
                      p.slot_expert, p.route_cnt, p.inst_load, p.rank_load, p.stats, g, cc ? 1 : 0);
}

}  // namespace topo
