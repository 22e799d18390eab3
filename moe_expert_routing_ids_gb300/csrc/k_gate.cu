// Top-k gating fused with the routing matrix ("TopoEP: Topology-Aware Load
// Balancing for Expert-Parallel MoE Training" §2.1: per token the router
// selects the Top-k experts; §6.4: synthetic routing from random logits with a
// fixed expert-specific bias; Omega of the selection, §4.1 Eq. 3).
//
// score = logit + bias (one float addition); the k largest scores in
// descending order, equal scores (-0 equals +0) to the lower expert, NaN below
// every number.  One CTA per tile of TT tokens of one source (the tiles of
// topo_hist); a group of G lanes per token at a time (G = 16, two tokens per
// warp, for 128 < E <= 512 and k <= 16, so that the sort, scan and ranking
// below serve two tokens at once; else G = 32).  Lane l of a group holds VPL
// scores of the token: with 16-byte loads, chunk c = u * G + l of VEC
// consecutive experts; otherwise experts u * G + l.
//
// Selection: the k-th largest of the G lane maxima (a bitonic sort across the
// group) is a lower bound tau of the k-th largest score, since k lanes each
// hold a score >= tau.  Every score >= tau is a candidate -- typically a
// little more than k -- and each candidate's place is the number of
// candidates ranking above it.  When that shortcut cannot be taken (k > G,
// more than kGateCand candidates, or fewer than k because of NaN or padding)
// the group runs k rounds of an exact argmax instead.  The selected ids are
// counted in shared memory and stored as the tile's counts; k_hist_prefix
// then builds Omega and the tile index exactly as topo_hist does.
#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

constexpr int kGateThreads = 256;
constexpr int kGateCand = 64;               // candidate buffer per token group

// Does (a, ia) rank above (b, ib)?  NaN below every number; ties by index.
__device__ __forceinline__ bool g_above(float a, int ia, float b, int ib) {
    const bool na = a != a, nb = b != b;
    if (na != nb) return nb;
    if (!na && a != b) return a > b;
    return ia < ib;
}

template <bool BF>
__device__ __forceinline__ float g_widen(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// The raw logit of expert e of a token row (read again for a selected expert;
// the row was just streamed, so it is normally still in L2).
template <bool BF>
__device__ __forceinline__ float g_raw(const void *row, int e) {
    if (BF) return g_widen<BF>(__ldg(reinterpret_cast<const unsigned short *>(row) + e));
    return __ldg(reinterpret_cast<const float *>(row) + e);
}

// Raw logits of this lane's VPL slots of one token row (invalid slots 0); gl
// is the lane's index in its group of G lanes.
template <int VPL, int G, bool BF, int VEC>
__device__ __forceinline__ void g_load(const void *row, int E, int gl, float *x) {
    if (VEC > 1) {
#pragma unroll
        for (int c = 0; c < VPL / VEC; ++c) {
            const int ch = c * G + gl;
            if (ch * VEC < E) {
                if (BF) {
                    const uint4 w = __ldcs(reinterpret_cast<const uint4 *>(row) + ch);
                    const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        x[c * VEC + 2 * h] = __uint_as_float(q[h] << 16);
                        x[c * VEC + 2 * h + 1] = __uint_as_float(q[h] & 0xffff0000u);
                    }
                } else {
                    const float4 w = __ldcs(reinterpret_cast<const float4 *>(row) + ch);
                    x[c * VEC] = w.x;
                    x[c * VEC + 1] = w.y;
                    x[c * VEC + 2] = w.z;
                    x[c * VEC + 3] = w.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < VEC; ++i) x[c * VEC + i] = 0.f;
            }
        }
    } else {
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int e = u * G + gl;
            x[u] = 0.f;
            if (e < E) {
                if (BF) x[u] = g_widen<BF>(__ldcs(reinterpret_cast<const unsigned short *>(row) + e));
                else x[u] = __ldcs(reinterpret_cast<const float *>(row) + e);
            }
        }
    }
}

template <int VPL, int G, int VEC>
__device__ __forceinline__ int g_expert(int u, int gl) {
    return VEC > 1 ? ((u / VEC) * G + gl) * VEC + (u % VEC) : u * G + gl;
}

// Order key of a candidate score (never NaN) and its expert: the float's
// sign-magnitude bits made monotone (-0 taken as +0), then the complement of
// the expert, so that a larger key ranks above and every key is distinct.
__device__ __forceinline__ unsigned long long g_key(float v, int e) {
    uint32_t bits = __float_as_uint(v);
    if (bits == 0x80000000u) bits = 0u;
    const uint32_t k32 = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
    return ((unsigned long long)k32 << 32) | (uint32_t)~e;
}

// G lanes per token (32 / G tokens per warp at a time); FULL: E == G * VPL,
// every slot of every lane holds an expert.
template <int VPL, int G, bool BF, int VEC, bool FULL>
__global__ void __launch_bounds__(kGateThreads, 3)
k_gate_tiles(const void *__restrict__ logits, const float *__restrict__ bias, int32_t *__restrict__ ids,
             float *__restrict__ scores, int32_t *__restrict__ tile_cnt, Geo g) {
    constexpr int kGroups = kGateThreads / G;                  // token groups per CTA
    extern __shared__ __align__(16) int gsm[];
    const int E = g.E, k = g.k;
    const int E4 = (E + 3) & ~3;
    float *sb = reinterpret_cast<float *>(gsm);                   // [E4] bias
    float *stash = sb + E4;                                       // [groups][G * VPL] scores by expert
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(stash + kGroups * G * VPL);
    int *cnt = reinterpret_cast<int *>(keys + kGroups * kGateCand);   // [E]
    const int l = blockIdx.x / g.ntl;
    const int tile = blockIdx.x - l * g.ntl;
    const int lane = threadIdx.x & 31, gl = lane & (G - 1);
    const int grp = threadIdx.x / G;
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    for (int e = threadIdx.x; e < E; e += kGateThreads) cnt[e] = 0;
    if (bias)
        for (int e = threadIdx.x; e < E4; e += kGateThreads) sb[e] = e < E ? __ldg(bias + e) : 0.f;
    float *wst = stash + grp * G * VPL;
    unsigned long long *wk = keys + grp * kGateCand;
    unsigned valid = FULL ? (VPL >= 32 ? 0xffffffffu : (1u << VPL) - 1u) : 0u;   // slots inside [0, E)
    if (!FULL)
#pragma unroll
        for (int u = 0; u < VPL; ++u) valid |= (unsigned)(g_expert<VPL, G, VEC>(u, gl) < E) << u;
    // bitonic directions of this lane, one bit per compare-exchange stage
    unsigned kmax = 0;
    {
        int st = 0;
#pragma unroll
        for (int size = 2; size <= G; size <<= 1)
#pragma unroll
            for (int stride = size >> 1; stride > 0; stride >>= 1, ++st)
                kmax |= (unsigned)(((gl & stride) == 0) == ((gl & size) == 0)) << st;
    }
    __syncthreads();                                              // cnt zeroed, bias staged

    const TileRef tr = tile_ref(g, g.tfirst, g.TT, g.tps, tile);
    if (tr.s < 0) return;                                         // past the last source's tiles
    const int ntok = tr.ntok;
    const int64_t row0 = (int64_t)l * g.T + tr.tok0;              // token row of the tile
    const size_t esz = BF ? 2 : 4;
    const char *base = reinterpret_cast<const char *>(logits);
    for (int i = grp; i < ntok; i += kGroups) {                  // i uniform in the group
        const void *row = base + (size_t)(row0 + i) * E * esz;
        float sc[VPL];                                            // scores, in place of the logits
        g_load<VPL, G, BF, VEC>(row, E, gl, sc);
        if (bias) {                                               // same chunking as the loads
            if (VEC > 1) {
#pragma unroll
                for (int c = 0; c < VPL / VEC; ++c) {
                    const int ch = c * G + gl;
                    if (FULL || ch * VEC < E)
#pragma unroll
                        for (int h = 0; h < VEC / 4; ++h) {
                            const float4 bb = reinterpret_cast<const float4 *>(sb)[ch * (VEC / 4) + h];
                            sc[c * VEC + 4 * h] += bb.x;
                            sc[c * VEC + 4 * h + 1] += bb.y;
                            sc[c * VEC + 4 * h + 2] += bb.z;
                            sc[c * VEC + 4 * h + 3] += bb.w;
                        }
                }
            } else {
#pragma unroll
                for (int u = 0; u < VPL; ++u)
                    if ((valid >> u) & 1u) sc[u] += sb[u * G + gl];
            }
        }
        float m = -__int_as_float(0x7f800000);                    // -inf
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            if ((valid >> u) & 1u) m = fmaxf(m, sc[u]);           // a NaN never wins fmaxf
        // tau = k-th largest lane maximum of the group (bitonic sort, descending)
        float tau = -__int_as_float(0x7f800000);
        if (k <= G) {
            float y = m;
            int st = 0;
#pragma unroll
            for (int size = 2; size <= G; size <<= 1)
#pragma unroll
                for (int stride = size >> 1; stride > 0; stride >>= 1, ++st) {
                    const float o = __shfl_xor_sync(gmask, y, stride, G);
                    y = ((kmax >> st) & 1u) ? fmaxf(y, o) : fminf(y, o);
                }
            tau = __shfl_sync(gmask, y, k - 1, G);
        }
        unsigned cm = 0;
#pragma unroll
        for (int u = 0; u < VPL; ++u) cm |= (unsigned)(((valid >> u) & 1u) && sc[u] >= tau) << u;
        const int c = __popc(cm);
        int incl = c;
#pragma unroll
        for (int o = 1; o < G; o <<= 1) {
            const int y = __shfl_up_sync(gmask, incl, o, G);
            if (gl >= o) incl += y;
        }
        const int n = __shfl_sync(gmask, incl, G - 1, G);
        const int64_t tok = row0 + i;
        int32_t *out_id = ids + tok * k;
        float *out_sc = scores ? scores + tok * k : nullptr;
        if (k <= G && n >= k && n <= kGateCand) {
            // the lane's scores by expert, so that its few candidates are read by index
            if (c) {
                if (VEC > 1) {
#pragma unroll
                    for (int q = 0; q < VPL / VEC; ++q) {
                        const int ch = q * G + gl;
                        if (FULL || ch * VEC < E)
#pragma unroll
                            for (int h = 0; h < VEC / 4; ++h)
                                reinterpret_cast<float4 *>(wst)[ch * (VEC / 4) + h] =
                                    make_float4(sc[q * VEC + 4 * h], sc[q * VEC + 4 * h + 1],
                                                sc[q * VEC + 4 * h + 2], sc[q * VEC + 4 * h + 3]);
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < VPL; ++u) wst[u * G + gl] = sc[u];
                }
                int off = incl - c;
                unsigned mm = cm;
                while (mm) {
                    const int u = __ffs(mm) - 1;
                    mm &= mm - 1u;
                    const int e = g_expert<VPL, G, VEC>(u, gl);
                    wk[off++] = g_key(wst[e], e);
                }
            }
            __syncwarp(gmask);
            for (int q = gl; q < n; q += G) {
                const unsigned long long key = wk[q];
                int rank = 0;
#pragma unroll 4
                for (int j = 0; j < n; ++j) rank += wk[j] > key;
                if (rank < k) {
                    const int e = (int)~(uint32_t)key;
                    out_id[rank] = e;
                    if (out_sc) out_sc[rank] = g_raw<BF>(row, e);
                    atomicAdd(&cnt[e], 1);
                }
            }
            __syncwarp(gmask);
        } else {
            // exact: k rounds of a group argmax over the slots not yet taken
            unsigned taken = 0;
            for (int j = 0; j < k; ++j) {
                float bv = 0.f;
                int bi = -1;
#pragma unroll
                for (int u = 0; u < VPL; ++u) {
                    const int e = g_expert<VPL, G, VEC>(u, gl);
                    if (((valid & ~taken) >> u) & 1u && (bi < 0 || g_above(sc[u], e, bv, bi))) {
                        bv = sc[u];
                        bi = e;
                    }
                }
#pragma unroll
                for (int o = G / 2; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(gmask, bv, o, G);
                    const int oi = __shfl_xor_sync(gmask, bi, o, G);
                    if (oi >= 0 && (bi < 0 || g_above(ov, oi, bv, bi))) {
                        bv = ov;
                        bi = oi;
                    }
                }
#pragma unroll
                for (int u = 0; u < VPL; ++u)
                    if (g_expert<VPL, G, VEC>(u, gl) == bi) taken |= 1u << u;
                if (gl == 0) {
                    out_id[j] = bi;
                    if (out_sc) out_sc[j] = g_raw<BF>(row, bi);
                    atomicAdd(&cnt[bi], 1);
                }
            }
        }
    }
    __syncthreads();
    int32_t *mine = tile_cnt + ((int64_t)l * g.ntl + tile) * E;
    for (int e = threadIdx.x; e < E; e += kGateThreads) mine[e] = cnt[e];
}

template <int VPL, int G, bool BF, int VEC>
cudaError_t run_gate(const Geo &g, const void *logits, const float *bias, int32_t *ids, float *scores,
                     int32_t *tile_cnt, cudaStream_t st) {
    constexpr int kGroups = kGateThreads / G;
    const int64_t tiles = (int64_t)g.L * g.ntl;
    const size_t smem = (size_t)((g.E + 3) & ~3) * 4 + (size_t)kGroups * G * VPL * 4 +
                        (size_t)kGroups * kGateCand * 8 + (size_t)g.E * 4;
    const bool full = g.E == G * VPL;
    const void *fn = full ? (const void *)k_gate_tiles<VPL, G, BF, VEC, true>
                          : (const void *)k_gate_tiles<VPL, G, BF, VEC, false>;
    cudaError_t e = ensure_smem(fn, smem);
    if (e != cudaSuccess) return e;
    if (full)
        k_gate_tiles<VPL, G, BF, VEC, true><<<(unsigned)tiles, kGateThreads, smem, st>>>(
            logits, bias, ids, scores, tile_cnt, g);
    else
        k_gate_tiles<VPL, G, BF, VEC, false><<<(unsigned)tiles, kGateThreads, smem, st>>>(
            logits, bias, ids, scores, tile_cnt, g);
    return cudaGetLastError();
}

template <int VPL, int G, bool BF>
cudaError_t gate_vec(const Geo &g, const void *logits, const float *bias, int32_t *ids, float *scores,
                     int32_t *tile_cnt, bool vec, cudaStream_t st) {
    constexpr int V = BF ? 8 : 4;
    if (vec && VPL % V == 0)
        return run_gate<VPL, G, BF, (VPL % V == 0 ? V : 1)>(g, logits, bias, ids, scores, tile_cnt, st);
    return run_gate<VPL, G, BF, 1>(g, logits, bias, ids, scores, tile_cnt, st);
}

// 16 lanes per token for 128 < E <= 512 with k <= 16 (two tokens per warp:
// the per-token sort, scan and ranking are shared), else 32.
template <bool BF>
cudaError_t gate_vpl(const Geo &g, const void *logits, const float *bias, int32_t *ids, float *scores,
                     int32_t *tile_cnt, bool vec, cudaStream_t st) {
    if (g.E > 128 && g.E <= 512 && g.k <= 16) {
        const int vpl = (g.E + 15) / 16;
        if (vpl <= 16) return gate_vec<16, 16, BF>(g, logits, bias, ids, scores, tile_cnt, vec, st);
        return gate_vec<32, 16, BF>(g, logits, bias, ids, scores, tile_cnt, vec, st);
    }
    const int vpl = (g.E + 31) / 32;
    if (vpl <= 1) return gate_vec<1, 32, BF>(g, logits, bias, ids, scores, tile_cnt, vec, st);
    if (vpl <= 2) return gate_vec<2, 32, BF>(g, logits, bias, ids, scores, tile_cnt, vec, st);
    if (vpl <= 4) return gate_vec<4, 32, BF>(g, logits, bias, ids, scores, tile_cnt, vec, st);
    if (vpl <= 8) return gate_vec<8, 32, BF>(g, logits, bias, ids, scores, tile_cnt, vec, st);
    if (vpl <= 16) return gate_vec<16, 32, BF>(g, logits, bias, ids, scores, tile_cnt, vec, st);
    if (vpl <= 32) return gate_vec<32, 32, BF>(g, logits, bias, ids, scores, tile_cnt, vec, st);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gate(const Geo &g, const void *logits, bool bf16, const float *bias, int32_t *ids,
                        float *scores, int32_t *hist, void *ws, uint64_t fp, cudaStream_t st) {
    const int64_t tiles = (int64_t)g.L * g.ntl;
    if (tiles == 0) return cudaSuccess;
    if (tiles > INT32_MAX) return cudaErrorInvalidValue;
    const size_t esz = bf16 ? 2 : 4;
    const bool vec = ((uintptr_t)logits & 15) == 0 && ((size_t)g.E * esz) % 16 == 0;
    int32_t *tile_cnt = ws_at<int32_t>(ws, g.off_tile);
    cudaError_t e;
    if (g.roff &&
        (e = launch_tile_first(g, g.TT, ws_at<int32_t>(ws, g.off_first), ws_at<WsHeader>(ws, 0), st)) != cudaSuccess)
        return e;
    e = bf16 ? gate_vpl<true>(g, logits, bias, ids, scores, tile_cnt, vec, st)
                         : gate_vpl<false>(g, logits, bias, ids, scores, tile_cnt, vec, st);
    if (e != cudaSuccess) return e;
    return launch_hist_prefix(g, hist, ws, fp, st);
}

}  // namespace topo
