// Prep of the rerouting calls, from the plan alone: the instance index of
// every layer, the routing index of every (source, layer) row (TopoEP §4.2
// routing counts q turned into per-expert occurrence ranges over the
// expert's instances in ascending rank order) and the dispatch-layout offsets
// (segment starts, column prefixes of q, send counts, locality statistics).
#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

constexpr int kPrepBThreads = 1024;

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

// Instance index of a layer: the expert of every instance (iexp).  One thread
// per instance.  tab == nullptr: the contiguous main map (main of e is
// e / (E/R)).
__device__ __forceinline__ void inst_index(const int32_t *__restrict__ slot_expert,
                                           const int32_t *__restrict__ tab, int32_t *iexp, WsHeader *hdr,
                                           const Geo &g, int bx) {
    const int l = blockIdx.y;
    const int i = bx * blockDim.x + threadIdx.x;
    if (l == 0 && i == 0) hdr->route_fp = 0;
    if (i >= g.n_keys) return;
    const int E = g.E, R = g.R, nl = g.n_local, ER = g.E_R, ns = g.n_slot;
    const int r = i / nl, li = i - r * nl;
    int e = li < ER ? (tab ? __ldg(tab + 2 * E + r * ER + li) : r * ER + li)
                    : __ldg(slot_expert + ((int64_t)l * R + r) * ns + (li - ER));
    if (e >= E || e < -1) {
        set_error(hdr, TOPO_ESTATE);
        e = -1;
    }
    iexp[(int64_t)l * g.n_keys + i] = e;
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

// Instances of a layer grouped by expert, in ascending rank order (ilist),
// and each expert's start in it (ioff).  Every CTA stages the layer's
// instance experts and builds each expert's bitmask over ranks in shared
// memory (an expert twice on one rank raises ESTATE); an instance's place is
// its expert's start plus the number of lower ranks in the mask.  Every CTA
// prefixes the mask popcounts itself; CTA 0 stores the offsets.
__device__ __forceinline__ void inst_list(const int32_t *__restrict__ iexp, int32_t *ioff_g, int32_t *ilist,
                                          WsHeader *hdr, const Geo &g, int bx, int *sml) {
    __shared__ int warp_tot[32];
    const int l = blockIdx.y, E = g.E, nk = g.n_keys, nl = g.n_local;
    const int RW = (g.R + 31) / 32;
    unsigned *msk = reinterpret_cast<unsigned *>(sml);          // [E][RW]
    int *ioff = reinterpret_cast<int *>(msk + E * RW);          // [E+1]
    int *ie = ioff + ((E + 4) & ~3);                            // [nk] the layer's instance experts
    stage_words(ie, iexp + (int64_t)l * nk, nk);
    for (int i = threadIdx.x; i < E * RW; i += blockDim.x) msk[i] = 0u;
    cp_async_wait_all();
    __syncthreads();
    bool dup = false;
    for (int i = threadIdx.x; i < nk; i += blockDim.x) {
        const int e = ie[i];
        if (e < 0) continue;
        const int r = i / nl;
        const unsigned bit = 1u << (r & 31);
        dup |= (atomicOr(&msk[e * RW + (r >> 5)], bit) & bit) != 0;   // expert twice on one rank
    }
    if (dup && bx == 0) set_error(hdr, TOPO_ESTATE);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
        for (int w = 0; w < RW; ++w) c += __popc(msk[e * RW + w]);
        ioff[e] = c;
    }
    __syncthreads();
    const int n_inst = block_excl_scan(ioff, E, warp_tot);
    if (bx == 0) {
        int32_t *o = ioff_g + (int64_t)l * (E + 1);
        for (int e = threadIdx.x; e < E; e += blockDim.x) o[e] = ioff[e];
        if (threadIdx.x == 0) o[E] = n_inst;
    }
    const int i = bx * blockDim.x + threadIdx.x;
    if (i >= nk) return;
    const int e = ie[i];
    if (e < 0) return;
    const int r = i / nl;
    const unsigned *m = msk + e * RW;
    int j = ioff[e] + __popc(m[r >> 5] & ((1u << (r & 31)) - 1u));
    for (int w = 0; w < (r >> 5); ++w) j += __popc(m[w]);
    ilist[(int64_t)l * nk + j] = i;
}

// Routing index of one source row: per expert, its nonzero instances in rank
// order with running occurrence ranges.  One CTA per (source, layer).  The
// row of q and the layer's instance list are staged in shared memory; the
// list is cut into equal chunks, one per thread, and one scan of (nonzero
// count, occurrence sum) over the chunks gives every entry its place in the
// row and its occurrence range -- the cost does not depend on how many
// instances a hot expert has.
__global__ void __launch_bounds__(256)
k_row_index(const int32_t *__restrict__ q, const int32_t *__restrict__ ioff_g,
            const int32_t *__restrict__ ilist_g, int32_t *roff, Entry *rent, Geo g) {
    pdl_wait();                                  // the previous kernel's outputs
    extern __shared__ __align__(16) int smi[];
    __shared__ int2 warp_tot2[32];
    __shared__ int cbase[256], vbase[256];
    const int s = blockIdx.x, l = blockIdx.y, E = g.E, R = g.R, nk = g.n_keys;
    const int nk4 = (nk + 3) & ~3;
    int *qrow = smi;                                            // [nk]
    int *ilist = qrow + nk4;                                    // [nk]
    int *ioff = ilist + nk4;                                    // [E+1]
    int *ro_s = ioff + ((E + 4) & ~3);                          // [E]
    int *vst = ro_s + E;                                        // [E]
    stage_words(qrow, q + ((int64_t)l * R + s) * nk, nk);
    stage_words(ilist, ilist_g + (int64_t)l * nk, nk);
    stage_words(ioff, ioff_g + (int64_t)l * (E + 1), E + 1);
    cp_async_wait_all();
    __syncthreads();
    const int n_inst = min(ioff[E], nk);
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
    pdl_trigger();
}

// Column prefix of q over sources (stored only where q != 0) and column
// totals.  A CTA covers 32 columns; its 8 warps each scan one chunk of the
// sources (16 loads in flight per lane), and the chunks are prefixed through
// shared memory.
__device__ __forceinline__ void lay_cols(const int32_t *__restrict__ q, int32_t *soff, int32_t *ccnt,
                                         const Geo &g, int bx) {
    __shared__ int part[8][33];
    const int l = blockIdx.y;
    const int lane = threadIdx.x & 31, ch = threadIdx.x >> 5;
    const int i = bx * 32 + lane;
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
__device__ __forceinline__ void lay_seg(const int32_t *__restrict__ ccnt, int32_t *lseg, int64_t *lstat,
                                        const Geo &g) {
    __shared__ int warp_tot[32];
    __shared__ int sums[1024];
    const int l = blockIdx.y;
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

// The prep's first two steps each pair two independent jobs in one launch:
// blocks [0, n_a) build the instance index (or list), the rest the column
// prefixes of q (or, one block per layer, the segment offsets), which need q
// alone.
__global__ void __launch_bounds__(256)
k_prep_a(const int32_t *__restrict__ slot_expert, const int32_t *__restrict__ tab, int32_t *iexp,
         WsHeader *hdr, const int32_t *__restrict__ q, int32_t *soff, int32_t *ccnt, Geo g, int n_a) {
    pdl_wait();                                  // the previous kernel's outputs
    if ((int)blockIdx.x < n_a) inst_index(slot_expert, tab, iexp, hdr, g, blockIdx.x);
    else lay_cols(q, soff, ccnt, g, blockIdx.x - n_a);
    pdl_trigger();
}

__global__ void __launch_bounds__(kPrepBThreads)
k_prep_b(const int32_t *__restrict__ iexp, int32_t *ioff_g, int32_t *ilist, WsHeader *hdr,
         const int32_t *__restrict__ ccnt, int32_t *lseg, int64_t *lstat, Geo g, int n_a) {
    extern __shared__ __align__(16) int sml[];
    pdl_wait();                                  // the previous kernel's outputs
    if ((int)blockIdx.x < n_a) inst_list(iexp, ioff_g, ilist, hdr, g, blockIdx.x, sml);
    else lay_seg(ccnt, lseg, lstat, g);
    pdl_trigger();
}

// Per-entry output bases; send counts and locality statistics from the
// routing index.  One CTA per (source, layer).
__global__ void __launch_bounds__(256)
k_lay_entries(const int32_t *__restrict__ roff, Entry *rent, const int32_t *__restrict__ soff,
              const int32_t *__restrict__ lseg, int64_t *lsend, int64_t *lstat, Geo g) {
    pdl_wait();                                  // the previous kernel's outputs
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
    pdl_trigger();
}

}  // namespace

// Shared memory of the instance list: rank masks, offsets, the instance experts.
size_t inst_list_smem(const Geo &g) {
    return ((size_t)g.E * ((g.R + 31) / 32) + (((size_t)g.E + 4) & ~(size_t)3) + g.n_keys) * 4;
}

size_t row_index_smem(const Geo &g) {
    const size_t nk4 = ((size_t)g.n_keys + 3) & ~(size_t)3;
    return (2 * nk4 + (((size_t)g.E + 4) & ~(size_t)3) + 2 * (size_t)g.E) * 4;
}

// Prep shared by topo_reroute and topo_reroute_layout.
cudaError_t launch_prep(const Geo &g, const int32_t *main_rank, const topo_plan_t &p, void *ws,
                        int32_t *seg_off, int64_t *send_counts, int64_t *layout_stats, cudaStream_t st) {
    cudaError_t e;
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    int32_t *lseg = seg_off ? seg_off : ws_at<int32_t>(ws, g.off_lseg);
    int64_t *lsend = send_counts ? send_counts : ws_at<int64_t>(ws, g.off_lsend);
    int64_t *lstat = layout_stats ? layout_stats : ws_at<int64_t>(ws, g.off_lstat);
    if (main_rank && (e = launch_main_tables(g, main_rank, ws, nullptr, 0, st)) != cudaSuccess) return e;
    const int na = (g.n_keys + 255) / 256, nb = (g.n_keys + 31) / 32;
    if ((e = launch_pdl(k_prep_a, dim3(na + nb, g.L), dim3(256), 0, st, p.slot_expert,
                        main_rank ? ws_at<int32_t>(ws, g.off_main) : nullptr, ws_at<int32_t>(ws, g.off_iexp), hdr,
                        p.route_cnt, ws_at<int32_t>(ws, g.off_soff), ws_at<int32_t>(ws, g.off_ccnt), g, na)) !=
        cudaSuccess)
        return e;
    const int nl_blocks = (g.n_keys + kPrepBThreads - 1) / kPrepBThreads;
    const size_t smem_list = inst_list_smem(g);
    if ((e = ensure_smem((const void *)k_prep_b, smem_list)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_prep_b, dim3(nl_blocks + 1, g.L), dim3(kPrepBThreads), smem_list, st,
                        ws_at<int32_t>(ws, g.off_iexp), ws_at<int32_t>(ws, g.off_ioff),
                        ws_at<int32_t>(ws, g.off_ilist), hdr, ws_at<int32_t>(ws, g.off_ccnt), lseg, lstat, g,
                        nl_blocks)) != cudaSuccess)
        return e;
    const size_t smem_row = row_index_smem(g);
    if ((e = ensure_smem((const void *)k_row_index, smem_row)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_row_index, dim3(g.R, g.L), dim3(256), smem_row, st,
        p.route_cnt, ws_at<int32_t>(ws, g.off_ioff), ws_at<int32_t>(ws, g.off_ilist),
        ws_at<int32_t>(ws, g.off_roff), ws_at<Entry>(ws, g.off_rent), g)) != cudaSuccess)
        return e;
    const size_t smem_e = (size_t)g.R * 8;
    if ((e = ensure_smem((const void *)k_lay_entries, smem_e)) != cudaSuccess) return e;
    return launch_pdl(k_lay_entries, dim3(g.R, g.L), dim3(256), smem_e, st,
        ws_at<int32_t>(ws, g.off_roff), ws_at<Entry>(ws, g.off_rent), ws_at<int32_t>(ws, g.off_soff),
        lseg, lsend, lstat, g);
}

}  // namespace topo
