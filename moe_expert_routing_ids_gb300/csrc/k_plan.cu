// Two-stage topology-aware replication plan (TopoEP §4.3, Eqs. 9-10).
//
//   k_main_tables   main(e), its local index, and the experts of each rank
//   k_plan_place    one CTA per (domain, layer): demand D (Eq. 4), benefit
//                   b = 2 D S_tok - ||W|| (Eq. 9) and the inter-node placement
//   k_plan_route    one CTA per (source, layer): the even split of omega_{s,e}
//                   over the chosen instances; U and L by integer atomics
//   k_plan_refine   one CTA per (domain, layer): intra-node refinement (Eq. 10)
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
#include <type_traits>

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
    // Candidates ranked by (benefit desc, expert asc).  With S_tok > 0 the
    // benefit 2 D S_tok - ||W|| rises strictly with the demand D < 2^31, so
    // one unsigned key D << 32 | ~e orders them the same way (0: not a
    // candidate); keys are distinct.
    extern __shared__ __align__(16) unsigned long long keyv[];   // [npow]
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
        unsigned long long key = 0;
        if (e < E) {
            int64_t D = 0;
#pragma unroll 8
            for (int j = 0; j < rpn; ++j) D += H[(int64_t)(d * rpn + j) * E + e];
            const int64_t b = 2 * D * g.S_tok - g.W;
            if ((main_of[e] / rpn != d) && b > 0) {
                key = ((unsigned long long)D << 32) | (0xffffffffu - (unsigned)e);
                atomicAdd(&ncand, 1);
            }
        }
        keyv[e] = key;
    }
    int32_t *SE = slot_expert + (int64_t)l * R * ns;
    for (int i = threadIdx.x; i < rpn * ns; i += blockDim.x) SE[(int64_t)d * rpn * ns + i] = -1;
    for (int e = threadIdx.x; e < E; e += blockDim.x) rep[((int64_t)l * E + e) * g.M + d] = -1;
    __syncthreads();
    const int cap = rpn * ns;
    const int placed = ncand < cap ? ncand : cap;
    int64_t repcost = 0;
    auto place_one = [&](int rank, int e) {
        const int r = d * rpn + rank % rpn, slot = rank / rpn;
        SE[(int64_t)r * ns + slot] = e;
        rep[((int64_t)l * E + e) * g.M + d] = r * nl + g.E_R + slot;
        repcost += cost_sr(g, main_of[e], r) * g.W;
    };
    if (npow <= 512) {
        // each candidate counts the keys above its own, two per load
        const ulonglong2 *kv2 = reinterpret_cast<const ulonglong2 *>(keyv);
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const unsigned long long key = keyv[e];
            if (key == 0) continue;
            int rank = 0;
#pragma unroll 4
            for (int x = 0; x < (npow >> 1); ++x) {
                const ulonglong2 v = kv2[x];
                rank += (v.x > key) + (v.y > key);
            }
            if (rank < cap) place_one(rank, e);
        }
    } else {
        // bitonic sort in shared memory, descending
        for (int size = 2; size <= npow; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = threadIdx.x; i < (npow >> 1); i += blockDim.x) {
                    const int a = 2 * i - (i & (stride - 1)), b = a + stride;
                    const unsigned long long ka = keyv[a], kb = keyv[b];
                    if (((a & size) == 0) != (ka > kb)) {
                        keyv[a] = kb;
                        keyv[b] = ka;
                    }
                }
                __syncthreads();
            }
        }
        for (int rank = threadIdx.x; rank < placed; rank += blockDim.x)
            place_one(rank, (int)(0xffffffffu - (unsigned)keyv[rank]));
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

constexpr int kRouteRowMax = 16;     // domains whose replica row a thread holds in registers

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
    const bool rep_vec = (M & 3) == 0 && ((uintptr_t)REP & 15) == 0;
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
            if (M <= kRouteRowMax) {
                // the expert's row of stage-1 replicas in registers (16-byte
                // loads when the rows are 16-byte aligned)
                int rr[kRouteRowMax];
                if (rep_vec) {
#pragma unroll
                    for (int q4 = 0; q4 < kRouteRowMax / 4; ++q4) {
                        const int4 v = 4 * q4 < M ? __ldg(reinterpret_cast<const int4 *>(re) + q4)
                                                  : make_int4(-1, -1, -1, -1);
                        rr[4 * q4] = v.x;
                        rr[4 * q4 + 1] = v.y;
                        rr[4 * q4 + 2] = v.z;
                        rr[4 * q4 + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int dd = 0; dd < kRouteRowMax; ++dd) rr[dd] = dd < M ? __ldg(re + dd) : -1;
                }
                int n = 1;
#pragma unroll
                for (int dd = 0; dd < kRouteRowMax; ++dd) n += (dd != dm && rr[dd] >= 0);
                const int base = w / n, rem = w % n;
                int i = 0;
#pragma unroll
                for (int dd = 0; dd < kRouteRowMax; ++dd) {
                    int r, li;
                    if (dd == dm) {
                        r = me[u];
                        li = ml[u];
                    } else {
                        if (rr[dd] < 0) continue;
                        r = rr[dd] / nl;
                        li = rr[dd] % nl;
                    }
                    emit(r, li, base + (i < rem ? 1 : 0));
                    ++i;
                }
                continue;
            }
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

// Lanes holding the warp's largest key: up to five 32-bit redux steps, each
// keeping only the lanes that tie on every word so far, ending once one lane
// is left.
__device__ __forceinline__ unsigned warp_argmax_lanes(const Key &k) {
    unsigned live = 0xffffffffu;
    const unsigned words[5] = {(unsigned)(k.a >> 32), (unsigned)k.a, (unsigned)(k.b >> 32),
                               (unsigned)k.b, k.c};
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        const bool in = (live >> (threadIdx.x & 31)) & 1u;
        const unsigned m = __reduce_max_sync(0xffffffffu, in ? words[i] : 0u);
        live = __ballot_sync(0xffffffffu, in && words[i] == m);
        if ((live & (live - 1)) == 0) break;    // one lane left (uniform)
    }
    return live;
}

constexpr int kRefineMaxWarps = 8;
constexpr int kRefineCpl = 4;        // candidates a thread evaluates in one batch
constexpr int kScanPerLane = 8;      // sources a lane takes per block of the commit scan
constexpr int kRefineSmem = kSmemMax - 4096;   // dynamic shared memory beside the kernel's static arrays

// Where the refinement CTA keeps the domain's cells of q:
//   kQAll     every source's rows, int32, in shared memory
//   kQAll16   every source's rows as 16-bit counts (exact while each source's
//             cells in the domain sum to at most 65535, checked at load: a
//             move keeps its source and stays in the domain, so no cell can
//             exceed that sum); a CTA failing the check falls back to kQOwn
//   kQOwnFetch the domain's own sources' rows in shared memory, the rest in
//             global memory (atomic adds that do not wait, reads past L1),
//             the busiest rank's rows fetched into shared memory each iteration
//   kQOwn     the same, the commit reading the rows from global memory
enum RefineQ : int { kQOwn = 0, kQAll = 1, kQOwnFetch = 2, kQAll16 = 3 };

// Row stride (elements) of the refinement CTA's q table: the sources it holds,
// made odd in 32-bit words so that one source's cells down the rows meet
// distinct banks.
__host__ __device__ __forceinline__ int refine_row_stride(const Geo &g, int qmode) {
    if (qmode == kQAll16) return 2 * (((g.R + 1) / 2) | 1);
    return (qmode == kQAll ? g.R : g.rpn) | 1;
}

// Offset (in ints, 16-byte aligned) of the q table in the refinement CTA's
// shared memory, after the per-rank and per-instance arrays and hl.
__host__ __device__ __forceinline__ int refine_q_offset(const Geo &g) {
    const int head = 2 * g.rpn + 4 * g.rpn * g.n_local + (g.rpn * g.E + 1) / 2;
    return (head + 3) & ~3;
}

// Ints the q table takes (16-byte multiple).
__host__ __device__ __forceinline__ int refine_q_ints(const Geo &g, int qmode) {
    const int64_t el = (int64_t)g.rpn * g.n_local * refine_row_stride(g, qmode);
    const int64_t ints = qmode == kQAll16 ? (el + 1) / 2 : el;
    return (int)((ints + 3) & ~int64_t(3));
}

// Shared-memory state of one refinement CTA.  The domain's cells of q are held
// transposed -- row (j, li) of the domain's instance over sources -- so that
// the commit reads and updates one row across the warp.
struct RefState {
    int *Lr;        // [rpn] rank loads
    int *used;      // [rpn] used slots
    int *U;         // [rpn][nl] instance loads
    int *xe;        // [rpn][nl] expert of each instance, -1: none
    int *xc;        // [rpn][nl] main rank of that expert, or -1 - main rank when it is in another domain
    int *dirty;     // [rpn][nl] row changed: written back to q at the end
    short *hl;      // [rpn][E] local index of expert e on rank j, or -1
    void *qc;       // [rpn][nl][RS] q of sources src0 .. src0 + RS - 1 (int32, or uint16 in kQAll16)
    int *pf;        // [nl][R] the busiest rank's rows of q, fetched each iteration (kQOwnFetch)
    int RS, src0, r0;
    int32_t *Q;     // this layer's q [R][R][nl]
    int32_t *SE;    // this layer's slot experts [R][n_slot]
};

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;\n" ::: "memory");
}

// The domain's int32 cells of q for sources [s_begin, s_end) into the
// transposed table: 4-byte asynchronous copies, all issued here;
// cp_async_wait_all() completes them.
__device__ void load_q(const RefState &x, const Geo &g, int s_begin, int s_end) {
    const int nl = g.n_local, n = g.rpn * nl, nthr = blockDim.x;
    int *qc = static_cast<int *>(x.qc);
    const int64_t total = (int64_t)(s_end - s_begin) * n;
    int s = (int)threadIdx.x / n, i = (int)threadIdx.x % n;
    const int ds = nthr / n, di = nthr % n;
    for (int64_t f = threadIdx.x; f < total; f += nthr) {
        cp_async4(&qc[(size_t)i * x.RS + s], x.Q + ((int64_t)(s_begin + s) * g.R + x.r0) * nl + i);
        s += ds;
        i += di;
        if (i >= n) { i -= n; ++s; }
    }
}

// Every source's cells of the domain into the 16-bit table (kQAll16).  Only a
// rank's first E_R + used[j] instances can hold tokens (an instance without an
// expert routes nothing), and for one (source, rank) they are contiguous in q:
// those runs, rounded up to whole 16-byte pieces, go by asynchronous copies
// into an int32 staging area (sources in chunks that fit), then into the
// table (zeroed by the caller), summing each source's cells.  Returns true (to every thread)
// when every source's sum fits 16 bits.
__device__ bool load_q16(const RefState &x, const Geo &g, int *stage, int stage_ints) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int R = g.R, rpn = g.rpn, nl = g.n_local, ER = g.E_R;
    uint16_t *qc = static_cast<uint16_t *>(x.qc);
    __shared__ int run0[kMaxRanksPerNode + 1];   // staging offset of rank j's run in a source's piece
    __shared__ int over;
    int *ssum = stage;                          // [R] per-source sums, then the staging pieces
    int *pieces = stage + ((R + 3) & ~3);
    const int piece_room = stage_ints - ((R + 3) & ~3);
    const bool vec = (nl & 3) == 0 && ((uintptr_t)x.Q & 15) == 0;
    if (tid == 0) {
        int o = 0;
        for (int j = 0; j < rpn; ++j) {
            run0[j] = o;
            o += (ER + x.used[j] + 3) & ~3;
        }
        run0[rpn] = o;
        over = 0;
    }
    for (int s = tid; s < R; s += nthr) ssum[s] = 0;
    __syncthreads();
    const int SP = run0[rpn];                   // ints per source in the staging area
    const int chunk = SP > 0 ? piece_room / SP : R;
    if (chunk < 1) return false;                // no room: the caller falls back
    for (int c0 = 0; c0 < R; c0 += chunk) {
        const int cs = min(chunk, R - c0);
        // a thread per (source, rank) run: its copies, then (after the wait)
        // its cells into the table and its sum
        for (int f = tid; f < cs * rpn; f += nthr) {
            const int sl = f / rpn, j = f - sl * rpn;
            const int live = ER + x.used[j];
            const int32_t *src = x.Q + ((int64_t)(c0 + sl) * R + x.r0 + j) * nl;
            int *dst = pieces + sl * SP + run0[j];
            if (vec) {
#pragma unroll 4
                for (int li = 0; li < live; li += 4) cp_async16(dst + li, src + li);
            } else {
#pragma unroll 4
                for (int li = 0; li < live; ++li) cp_async4(dst + li, src + li);
            }
        }
        cp_async_wait_all();
        __syncthreads();
        for (int f = tid; f < cs * rpn; f += nthr) {
            const int sl = f / rpn, j = f - sl * rpn, s = c0 + sl;
            const int live = ER + x.used[j];
            const int *p = pieces + sl * SP + run0[j];
            uint16_t *col = qc + (size_t)j * nl * x.RS + s;
            int sum = 0;
#pragma unroll 4
            for (int li = 0; li < live; ++li) {
                const int v = p[li];
                sum += v;
                col[(size_t)li * x.RS] = (uint16_t)v;
            }
            atomicAdd(&ssum[s], sum);
        }
        __syncthreads();
    }
    for (int s = tid; s < R; s += nthr)
        if ((unsigned)ssum[s] > 65535u) over = 1;
    __syncthreads();
    return over == 0;
}

// The refinement loop (TopoEP §4.3, Eq. 10) over the state in shared memory.
//
// A rank's instances are its E_R mains and then its slots, filled from the
// first (placement fills slots in order; a new replica takes the first empty
// one), so only the busiest rank's first E_R + used[jb] instances can be
// moved: the candidates of an iteration are those rows times the other ranks.
// They take as many warps as they fill (kRefineCpl per thread); with one warp
// no winners meet in shared memory.  With kQOwnFetch the warps not evaluating
// fetch the busiest rank's rows of q meanwhile (pf), so the commit reads them
// from shared memory.  kOneWarp: a CTA of one warp (no barriers, one stride).
template <int kMode, bool kOneWarp>
__device__ __forceinline__ void refine_loop(const RefState &x, const Geo &g, int *iters_out, int64_t *tokd_out,
                                            int64_t *repd_out) {
    using QT = typename std::conditional<kMode == kQAll16, uint16_t, int>::type;
    __shared__ Key kbuf[kRefineMaxWarps];
    __shared__ int cbuf[kRefineMaxWarps];
    __shared__ int lbuf[kRefineMaxWarps];
    __shared__ int s_done;
    __shared__ int2 s_step[kRefineMaxWarps + 1];   // (lb, jt) stride of nact * 32 candidates
    constexpr bool kAll = kMode == kQAll || kMode == kQAll16;
    const int tid = threadIdx.x, lane = tid & 31, w = kOneWarp ? 0 : tid >> 5;
    const int nthr = kOneWarp ? 32 : blockDim.x, nwarp = kOneWarp ? 1 : nthr >> 5;
    const int E = g.E, R = g.R, rpn = g.rpn, ns = g.n_slot, nl = g.n_local, ER = g.E_R;
    int *Lr = x.Lr, *used = x.used, *U = x.U, *xe = x.xe, *xc = x.xc, *pf = x.pf;
    QT *qc = static_cast<QT *>(x.qc);
    short *hl = x.hl;
    const int RS = x.RS, r0 = x.r0, src0 = x.src0;
    int32_t *Q = x.Q;
    const int64_t tok_cost = 2 * g.S_tok * g.c_intra;     // per token moved off or onto its own rank
    const int64_t w_intra = (int64_t)g.c_intra * g.W, w_inter = (int64_t)g.c_inter * g.W;
    // this thread's first candidate (lb, jt): candidate c is (c / rpn, c % rpn)
    const int c_lb0 = tid / rpn, c_jt0 = tid % rpn;
    const int2 step1 = make_int2(32 / rpn, 32 % rpn);
    if (!kOneWarp) {
        if (tid == 0) s_done = 0;
        if (tid <= kRefineMaxWarps) s_step[tid] = make_int2(tid * 32 / rpn, tid * 32 % rpn);
        __syncthreads();
    }
    int iters = 0;
    int64_t tokd = 0, repd = 0;
    constexpr int kHardCap = 1 << 24;   // commits provably end; guards a corrupted state only
    while ((g.max_iters == 0 || iters < g.max_iters) && iters < kHardCap) {
        // busiest rank, lowest index on ties (every warp computes it)
        const int myL = lane < rpn ? Lr[lane] : -1;
        const int myU = !kOneWarp && lane < rpn ? used[lane] : 0;
        const int Lb = __reduce_max_sync(0xffffffffu, myL);
        const int jb = __ffs(__ballot_sync(0xffffffffu, myL == Lb)) - 1;
        const int col_b = r0 + jb - src0;
        // (one warp: a single batch covers every row, so no bound is needed)
        const int live = kOneWarp ? nl : ER + __shfl_sync(0xffffffffu, myU, jb);
        const int ncand = live * rpn;
        int nact = kOneWarp ? 1 : (ncand + 32 * kRefineCpl - 1) / (32 * kRefineCpl);
        nact = nact < 1 ? 1 : (nact > nwarp ? nwarp : nact);
        const int stride = nact * 32;
        Key wk{0ull, 0ull, 0u};
        int wc = 0, wlt = -1;
        if (w < nact) {
            Key best{0ull, 0ull, 0u};
            int bc = 0;                          // packed (lb << 5 | jt) of best
            int blt = -1;                        // its local index on jt, -1: a new replica
            const int2 step = kOneWarp ? step1 : s_step[nact];
            const int s_lb = step.x, s_jt = step.y;
            int lb = c_lb0, jt = c_jt0;
            for (int c0 = tid; c0 < ncand; c0 += kRefineCpl * stride) {
                // every load of the batch issued before any is used
                int cl[kRefineCpl], cj[kRefineCpl], ub[kRefineCpl], ev[kRefineCpl], xv[kRefineCpl];
                int lt[kRefineCpl], ldt[kRefineCpl], ut[kRefineCpl], qt[kRefineCpl], qb[kRefineCpl];
#pragma unroll
                for (int i = 0; i < kRefineCpl; ++i) {
                    const bool ok = c0 + i * stride < ncand && jt != jb;
                    const int row = jb * nl + lb;
                    cl[i] = lb;
                    cj[i] = jt;
                    ub[i] = ok ? U[row] : 0;     // 0: no candidate
                    ev[i] = ok ? xe[row] : -1;
                    xv[i] = ok ? xc[row] : 0;
                    qt[i] = ok ? (int)qc[row * RS + (r0 + jt - src0)] : 0;
                    qb[i] = ok ? (int)qc[row * RS + col_b] : 0;
                    ldt[i] = Lr[jt];
                    ut[i] = used[jt];
                    lb += s_lb;
                    jt += s_jt;
                    if (jt >= rpn) { jt -= rpn; ++lb; }
                }
#pragma unroll
                for (int i = 0; i < kRefineCpl; ++i)
                    lt[i] = (ub[i] > 0 && ev[i] >= 0) ? hl[cj[i] * E + ev[i]] : -1;
#pragma unroll
                for (int i = 0; i < kRefineCpl; ++i) {
                    const bool is_new = lt[i] < 0;
                    const int half = (Lb - ldt[i]) >> 1;
                    const int delta = ub[i] < half ? ub[i] : half;
                    if (ub[i] > 0 && ev[i] >= 0 && delta >= 1 && (!is_new || ut[i] < ns)) {
                        const int m_rt = qt[i] < delta ? qt[i] : delta;
                        const int rest = delta - m_rt;
                        const int others = ub[i] - qt[i] - qb[i];
                        const int m_o = others < rest ? others : rest;
                        const int m_rb = rest - m_o;
                        const int64_t repl = !is_new ? 0 : xv[i] < 0 ? w_inter : xv[i] == r0 + cj[i] ? 0 : w_intra;
                        const int64_t cst = tok_cost * (int64_t)(m_rb - m_rt) + repl;
                        Key k;
                        k.a = ((unsigned long long)delta << 32) |
                              (unsigned long long)(0xffffffffu - (unsigned)ldt[i]);
                        k.b = ~((unsigned long long)cst ^ 0x8000000000000000ull);
                        k.c = ~(((unsigned)ev[i] << 5) | (unsigned)cj[i]);
                        if (key_gt(k, best)) {
                            best = k;
                            bc = (cl[i] << 5) | cj[i];
                            blt = lt[i];
                        }
                    }
                }
            }
            const unsigned win = warp_argmax_lanes(best);
            const int wl = __ffs(win) - 1;
            wk.a = __shfl_sync(0xffffffffu, best.a, wl);
            wk.c = __shfl_sync(0xffffffffu, best.c, wl);
            wc = __shfl_sync(0xffffffffu, bc, wl);
            wlt = __shfl_sync(0xffffffffu, blt, wl);
            if (nact > 1) {
                wk.b = __shfl_sync(0xffffffffu, best.b, wl);
                if (lane == 0) {
                    kbuf[w] = wk;
                    cbuf[w] = wc;
                    lbuf[w] = wlt;
                }
            }
        } else if (kMode == kQOwnFetch) {
            // rows li < live of r_b over every source, from global memory
            const int rb = r0 + jb, n = live * R;
            for (int i0 = tid - stride; i0 < n; i0 += (nthr - stride) * 8) {
                int v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * (nthr - stride);
                    const int li = i / R, s = i - li * R;
                    v[u] = i < n ? __ldcg(&Q[((int64_t)s * R + rb) * nl + li]) : 0;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * (nthr - stride);
                    if (i < n) pf[i] = v[u];
                }
            }
        }
        const bool fetched = kMode == kQOwnFetch && nact < nwarp;   // else the commit reads q itself
        // winners and rows in place; and no warp still reads this iteration's
        // loads when warp 0 commits
        if (nwarp > 1) __syncthreads();
        if (w == 0 && nact > 1) {
            // the warps' winners, tree over the first nact
            Key kk[kRefineMaxWarps];
            int cc[kRefineMaxWarps], ll[kRefineMaxWarps];
#pragma unroll
            for (int v = 0; v < kRefineMaxWarps; ++v) {
                if (v < nact) {
                    kk[v] = kbuf[v];
                    cc[v] = cbuf[v];
                    ll[v] = lbuf[v];
                } else {
                    kk[v] = Key{0ull, 0ull, 0u};
                    cc[v] = 0;
                    ll[v] = -1;
                }
            }
#pragma unroll
            for (int st = 1; st < kRefineMaxWarps; st <<= 1)
#pragma unroll
                for (int v = 0; v + st < kRefineMaxWarps; v += 2 * st)
                    if (v + st < nact && key_gt(kk[v + st], kk[v])) {
                        kk[v] = kk[v + st];
                        cc[v] = cc[v + st];
                        ll[v] = ll[v + st];
                    }
            wk = kk[0];
            wc = cc[0];
            wlt = ll[0];
        }
        if (w == 0 && wk.a != 0) {
            const int delta = (int)(wk.a >> 32);
            const int blb = wc >> 5, bjt = wc & 31;
            const int e = (int)((~wk.c) >> 5);
            const int rowb = jb * nl + blb;
            const int xcv = xc[rowb];
            const int rb = r0 + jb, rt = r0 + bjt;
            const bool is_new = wlt < 0;
            const int lt = is_new ? ER + used[bjt] : wlt;
            const int rowt = bjt * nl + lt;
            QT *qB = qc + rowb * RS, *qT = qc + rowt * RS;       // indexed by source - src0
            const int *pB = pf + blb * R;                        // fetched row, by source
            const int m_rt = min((int)qB[rt - src0], delta);
            int remaining = delta - m_rt;
            __syncwarp();
            if (is_new) {
                repd += xcv < 0 ? w_inter : xcv == rt ? 0 : w_intra;
                if (lane == 0) {
                    used[bjt] += 1;
                    hl[bjt * E + e] = (short)lt;
                    xe[rowt] = e;
                    xc[rowt] = xcv;
                    x.SE[(int64_t)rt * ns + (lt - ER)] = e;
                }
            }
            // other sources, ascending, skipping r_t and r_b: blocks of up to
            // 32 * kScanPerLane sources, each lane holding a run of consecutive
            // ones, so one warp scan of the runs' sums places every take
            for (int base = 0; base < R && remaining > 0; base += 32 * kScanPerLane) {
                const int nb = min(32 * kScanPerLane, R - base);
                const int per = (nb + 31) >> 5;
                const int s0 = base + lane * per;
                int v[kScanPerLane];
                int sum = 0;
#pragma unroll
                for (int u = 0; u < kScanPerLane; ++u) {
                    const int s = s0 + u;
                    const bool in = u < per && s < base + nb && s != rt && s != rb;
                    const bool cached = kAll || (s >= r0 && s < r0 + rpn);
                    v[u] = !in ? 0
                           : cached ? (int)qB[s - src0]
                           : fetched ? pB[s]
                                     : __ldcg(&Q[((int64_t)s * R + rb) * nl + blb]);
                    sum += v[u];
                }
                const int incl = warp_incl_scan(sum);
                int left = remaining - (incl - sum);     // still to take where this lane's run starts
#pragma unroll
                for (int u = 0; u < kScanPerLane; ++u) {
                    const int take = left <= 0 ? 0 : (left < v[u] ? left : v[u]);
                    left -= v[u];
                    if (take > 0) {
                        const int s = s0 + u;
                        if (kAll || (s >= r0 && s < r0 + rpn)) {
                            qB[s - src0] -= take;
                            qT[s - src0] += take;
                        }
                        if (!kAll) {   // no return value: the lane does not wait
                            atomicAdd(&Q[((int64_t)s * R + rb) * nl + blb], -take);
                            atomicAdd(&Q[((int64_t)s * R + rt) * nl + lt], take);
                        }
                    }
                }
                const int tot = __shfl_sync(0xffffffffu, incl, 31);
                remaining -= tot < remaining ? tot : remaining;
            }
            const int m_rb = remaining;
            // r_t's and r_b's cells, the loads: three lanes, disjoint cells
            if (lane == 0 && m_rt > 0) {
                qB[rt - src0] -= m_rt;
                qT[rt - src0] += m_rt;
                if (!kAll) {
                    atomicAdd(&Q[((int64_t)rt * R + rb) * nl + blb], -m_rt);
                    atomicAdd(&Q[((int64_t)rt * R + rt) * nl + lt], m_rt);
                }
            }
            if (lane == 1 && m_rb > 0) {
                qB[rb - src0] -= m_rb;
                qT[rb - src0] += m_rb;
                if (!kAll) {
                    atomicAdd(&Q[((int64_t)rb * R + rb) * nl + blb], -m_rb);
                    atomicAdd(&Q[((int64_t)rb * R + rt) * nl + lt], m_rb);
                }
            }
            if (lane == 2) {
                U[rowb] -= delta;
                U[rowt] += delta;
                Lr[jb] -= delta;
                Lr[bjt] += delta;
                x.dirty[rowb] = 1;
                x.dirty[rowt] = 1;
            }
            tokd += tok_cost * (int64_t)(m_rb - m_rt);
            __syncwarp();
        }
        bool done;
        if (!kOneWarp) {
            if (tid == 0 && wk.a == 0) s_done = 1;
            __syncthreads();
            done = s_done;
        } else {
            done = wk.a == 0;                    // uniform across the warp
        }
        if (done) break;
        ++iters;
    }
    *iters_out = iters;
    *tokd_out = tokd;
    *repd_out = repd;
}

// Writes the changed rows of the table back to q: warp 0 lists them (over xe,
// no longer needed), then a thread per row writes it.
template <typename QT>
__device__ void write_rows(const RefState &x, const Geo &g) {
    __shared__ int n_dirty;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int R = g.R, nl = g.n_local, n = g.rpn * nl;
    int *list = x.xe;
    const QT *qc = static_cast<const QT *>(x.qc);
    if (w == 0) {
        int cnt = 0;
        for (int base = 0; base < n; base += 32) {
            const int row = base + lane;
            const bool dv = row < n && x.dirty[row];
            const unsigned b = __ballot_sync(0xffffffffu, dv);
            if (dv) list[cnt + __popc(b & ((1u << lane) - 1u))] = row;
            cnt += __popc(b);
        }
        if (lane == 0) n_dirty = cnt;
    }
    __syncthreads();
    for (int k = tid; k < n_dirty; k += blockDim.x) {
        const int row = list[k], j = row / nl, li = row - j * nl;
        int32_t *dst = x.Q + (int64_t)(x.r0 + j) * nl + li;
        const QT *src = qc + (size_t)row * x.RS;
#pragma unroll 4
        for (int s = 0; s < R; ++s) dst[(int64_t)s * R * nl] = (int32_t)src[s];
    }
}

// One CTA per (domain, layer) refines the domain (TopoEP §4.3, Eq. 10).
// Candidates (instance at the busiest rank x other rank of the domain) are
// spread over the CTA's warps, a few per thread with their loads batched; each
// warp reduces with redux/ballot steps, the warps' winners meet in shared
// memory, and warp 0 commits.  qmode says where q lives (RefineQ); smem_ints:
// the dynamic shared memory, whose tail past the table stages kQAll16's load.
__global__ void __launch_bounds__(kRefineMaxWarps * 32)
k_plan_refine(const int32_t *__restrict__ tab, int32_t *slot_expert, int32_t *q, int32_t *inst_load,
              int32_t *rank_load, int64_t *stats, Geo g, int qmode, int smem_ints) {
    extern __shared__ __align__(16) int sm[];
    const int d = blockIdx.x, l = blockIdx.y, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nthr = blockDim.x;
    const int E = g.E, R = g.R, rpn = g.rpn, ns = g.n_slot, nl = g.n_local, ER = g.E_R;
    const int32_t *main_of = tab, *mains = tab + 2 * E;
    RefState x;
    x.Lr = sm;
    x.used = x.Lr + rpn;
    x.U = x.used + rpn;
    x.xe = x.U + rpn * nl;
    x.xc = x.xe + rpn * nl;
    x.dirty = x.xc + rpn * nl;
    x.hl = reinterpret_cast<short *>(x.dirty + rpn * nl);
    x.qc = sm + refine_q_offset(g);
    x.r0 = d * rpn;
    x.Q = q + (int64_t)l * R * R * nl;
    x.SE = slot_expert + (int64_t)l * R * ns;
    const int r0 = x.r0;

    // Before the wait, what the main tables and the placement kernel wrote:
    // this grid starts only once every CTA of the routing kernel has passed
    // its own wait, so those kernels have completed and their writes are
    // visible (read past L1).  used[j]: the slots before the first empty one.
    for (int i = tid; i < rpn * E; i += nthr) x.hl[i] = -1;
    for (int j = tid; j < rpn; j += nthr) x.used[j] = ns;
    __syncthreads();
    for (int i = tid; i < rpn * ns; i += nthr) {
        const int j = i / ns, u = i - j * ns;
        if (__ldcg(&x.SE[(int64_t)(r0 + j) * ns + u]) < 0) atomicMin(&x.used[j], u);
    }
    for (int i = tid; i < rpn * nl; i += nthr) {
        const int j = i / nl, li = i - j * nl, r = r0 + j;
        x.dirty[i] = 0;
        const int e = li < ER ? __ldcg(&mains[r * ER + li]) : __ldcg(&x.SE[(int64_t)r * ns + (li - ER)]);
        x.xe[i] = e;
        if (e >= 0) {
            x.hl[j * E + e] = (short)li;
            const int m = __ldcg(&main_of[e]);
            x.xc[i] = (m / rpn == d) ? m : -1 - m;
        } else {
            x.xc[i] = 0;
        }
    }
    if (qmode == kQAll16) {                     // the 16-bit table's empty rows stay zero
        int4 *z = static_cast<int4 *>(x.qc);
        const int nz = refine_q_ints(g, kQAll16) / 4;
        for (int i = tid; i < nz; i += nthr) z[i] = make_int4(0, 0, 0, 0);
    }
    // the routing kernel's output: q, U and L
    pdl_wait();
    pdl_trigger();
    for (int j = tid; j < rpn; j += nthr) x.Lr[j] = rank_load[(int64_t)l * R + r0 + j];
    for (int i = tid; i < rpn * nl; i += nthr) x.U[i] = inst_load[((int64_t)l * R + r0) * nl + i];
    __syncthreads();                            // used[] complete for load_q16
    int mode = qmode;
    if (mode == kQAll16) {
        x.RS = refine_row_stride(g, kQAll16);
        x.src0 = 0;
        const int q_end = refine_q_offset(g) + refine_q_ints(g, kQAll16);
        if (!load_q16(x, g, sm + q_end, smem_ints - q_end)) mode = kQOwn;   // uniform
    }
    if (mode != kQAll16) {
        const bool all_src = mode == kQAll;
        x.RS = refine_row_stride(g, mode);
        x.src0 = all_src ? 0 : r0;
        x.pf = static_cast<int *>(x.qc) + rpn * nl * x.RS;
        if (all_src) load_q(x, g, 0, R);
        else load_q(x, g, r0, r0 + rpn);
        cp_async_wait_all();
        __syncthreads();
    }

    int iters;
    int64_t tokd, repd;
    if (mode == kQAll16) refine_loop<kQAll16, false>(x, g, &iters, &tokd, &repd);
    else if (mode == kQAll && nthr == 32) refine_loop<kQAll, true>(x, g, &iters, &tokd, &repd);
    else if (mode == kQAll) refine_loop<kQAll, false>(x, g, &iters, &tokd, &repd);
    else if (mode == kQOwnFetch) refine_loop<kQOwnFetch, false>(x, g, &iters, &tokd, &repd);
    else refine_loop<kQOwn, false>(x, g, &iters, &tokd, &repd);

    // write back the domain's state and statistics; q's changed rows only
    // (in the other modes q in global memory is already current)
    __syncthreads();
    if (mode == kQAll16) write_rows<uint16_t>(x, g);
    else if (mode == kQAll) write_rows<int>(x, g);
    for (int j = tid; j < rpn; j += nthr) rank_load[(int64_t)l * R + r0 + j] = x.Lr[j];
    for (int i = tid; i < rpn * nl; i += nthr) inst_load[((int64_t)l * R + r0) * nl + i] = x.U[i];
    if (w == 0) {
        int lmax = lane < rpn ? x.Lr[lane] : 0, nused = lane < rpn ? x.used[lane] : 0;
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

// Shared memory (bytes) of the refinement kernel in each q mode; kQAll16 takes
// all the kernel may have, its tail staging the load.
size_t refine_smem_bytes(const Geo &g, int qmode) {
    if (qmode == kQAll16) return kRefineSmem;
    const size_t pf = qmode == kQOwnFetch ? (size_t)g.n_local * g.R : 0;
    return ((size_t)refine_q_offset(g) + (size_t)refine_q_ints(g, qmode) + pf) * 4;
}

int refine_qmode(const Geo &g) {
    if (refine_smem_bytes(g, kQAll) <= 200 * 1024) return kQAll;
    // the 16-bit table, the per-source sums and at least one source's pieces
    const size_t q16 = ((size_t)refine_q_offset(g) + refine_q_ints(g, kQAll16) + ((g.R + 3) & ~3) +
                        (size_t)g.rpn * ((g.n_local + 3) & ~3)) * 4;
    if (q16 <= (size_t)kRefineSmem && refine_smem_bytes(g, kQOwn) <= (size_t)kRefineSmem) return kQAll16;
    if (refine_smem_bytes(g, kQOwnFetch) <= 220 * 1024) return kQOwnFetch;
    return kQOwn;
}

// Warps of the refinement CTA: one when a single warp holds every candidate
// of an iteration at kRefineCpl per thread (no barriers then); else 8 -- all
// of them load the table (or fetch rows of q), and each iteration's
// candidates take as many as they fill.
int refine_warps(const Geo &g, int qmode) {
    if (qmode == kQAll && g.n_local * g.rpn <= 32 * kRefineCpl) return 1;
    return kRefineMaxWarps;
}

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
    const size_t smem_place = (size_t)npow * 8;
    if ((e = ensure_smem((const void *)k_plan_place, smem_place)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_plan_place, dim3(g.M, g.L), dim3(512), smem_place, st, hist, tab,
                        p.slot_expert, rep, p.inst_load, p.rank_load, p.stats, g, npow)) != cudaSuccess)
        return e;
    if ((e = ensure_smem((const void *)k_plan_route, (size_t)g.R * 4)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_plan_route, dim3(g.R, g.L), dim3(256), (size_t)g.R * 4, st, hist, tab, rep,
                        p.route_cnt, p.inst_load, p.rank_load, p.stats, g)) != cudaSuccess)
        return e;
    const int qmode = refine_qmode(g);
    const size_t smem_ref = refine_smem_bytes(g, qmode);
    if ((e = ensure_smem((const void *)k_plan_refine, smem_ref)) != cudaSuccess) return e;
    return launch_pdl(k_plan_refine, dim3(g.M, g.L), dim3(refine_warps(g, qmode) * 32), smem_ref, st, tab,
                      p.slot_expert, p.route_cnt, p.inst_load, p.rank_load, p.stats, g, qmode,
                      (int)(smem_ref / 4));
}

}  // namespace topo
