// Dispatch pack and combine of hidden rows in layout order.
//
// Dispatch (TopoEP Fig. 1) sends each token's activation to the ranks hosting
// its selected experts; combine ("MoX: Efficient MoE Routing on Direct-Connect
// Topologies", §2.4) reduces the token's top-K expert outputs back into one
// vector.  With the dispatch layout, the send buffer is the rows of the pairs
// in layout order:  y[pos] = x[token of sorted_pairs[pos]], and combine is
// out[t] = sum over slots j of w[t][j] * y[position of pair (t, j)].
//
// Both are row moves (bf16 rows of H elements, 16-byte aligned), so both run
// token-major: one warp per token, 16-byte vectors, one 512-byte chunk of the
// row per warp instruction.
//   k_invert   position of every pair (the inverse of sorted_pairs)
//   k_permute  reads each token row once and writes it to its k positions
//   k_combine  gathers the token's k rows, weights and sums them in float in
//              slot order (separate multiply and add, no fused multiply-add),
//              rounds once to bf16 (nearest, ties to even)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

// inv[l][p] = pos for p = sorted[l][pos]; inv starts at -1, so a value that
// is not a permutation of the pairs leaves a -1 the row kernels report.
__global__ void __launch_bounds__(256)
k_invert(const int32_t *__restrict__ sorted, int32_t *inv, WsHeader *hdr, int64_t npairs,
         int64_t total) {
    bool bad = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t l = i / npairs, pos = i - l * npairs;
        const int32_t p = __ldg(sorted + i);
        if ((uint64_t)p < (uint64_t)npairs) inv[l * npairs + p] = (int32_t)pos;
        else bad = true;
    }
    if (bad) set_error(hdr, TOPO_ESTATE);
}

// Positions of token t's k pairs, lane j holding slot j (and j + 32); false
// if one is missing.
__device__ __forceinline__ bool token_positions(const int32_t *inv_tok, int k, int64_t npairs,
                                                int &pa, int &pb) {
    const int lane = threadIdx.x & 31;
    pa = lane < k ? __ldg(inv_tok + lane) : 0;
    pb = lane + 32 < k ? __ldg(inv_tok + lane + 32) : 0;
    const bool ok = (uint64_t)pa < (uint64_t)npairs && (uint64_t)pb < (uint64_t)npairs;
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ int slot_pos(int j, int pa, int pb) {
    const int a = __shfl_sync(0xffffffffu, pa, j & 31);
    const int b = __shfl_sync(0xffffffffu, pb, j & 31);
    return j < 32 ? a : b;
}

// One warp per (layer, token): x row -> its k positions in y.  The chunk
// loop is warp-uniform (every lane takes part in the shuffles); only the
// loads and stores are predicated.
template <int KB>
__global__ void __launch_bounds__(256)
k_permute(const int4 *__restrict__ x, const int32_t *__restrict__ inv, int4 *y, WsHeader *hdr,
          int T, int k, int nv, int64_t npairs, int64_t ntok) {
    const int64_t tok = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (tok >= ntok) return;                           // whole warp
    const int lane = threadIdx.x & 31;
    const int64_t l = tok / T;
    int pa, pb;
    if (!token_positions(inv + tok * k, k, npairs, pa, pb)) {
        if (lane == 0) set_error(hdr, TOPO_ESTATE);
        return;
    }
    constexpr int KD = KB > 0 ? KB : 1;
    int64_t dst[KD];
    if (KB > 0) {
#pragma unroll
        for (int j = 0; j < KD; ++j) dst[j] = (l * npairs + slot_pos(j, pa, pb)) * nv;
    }
    const int4 *src = x + tok * nv;
    constexpr int U = 4;                               // vectors in flight per lane
    for (int c0 = 0; c0 < nv; c0 += 32 * U) {
        int4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + 32 * u + lane;
            if (c < nv) v[u] = __ldg(src + c);
        }
        for (int j = 0; j < (KB > 0 ? KD : k); ++j) {
            const int64_t d = KB > 0 ? dst[KB > 0 ? j : 0] : (l * npairs + slot_pos(j, pa, pb)) * nv;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + 32 * u + lane;
                if (c < nv) __stcs(y + d + c, v[u]);
            }
        }
    }
}

__device__ __forceinline__ float bf_lo(unsigned u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(unsigned u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ void acc8(float (&a)[8], float w, const int4 &v) {
    const unsigned q[4] = {(unsigned)v.x, (unsigned)v.y, (unsigned)v.z, (unsigned)v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a[2 * i] = __fadd_rn(a[2 * i], __fmul_rn(w, bf_lo(q[i])));
        a[2 * i + 1] = __fadd_rn(a[2 * i + 1], __fmul_rn(w, bf_hi(q[i])));
    }
}

__device__ __forceinline__ unsigned pack2(float lo, float hi) {
    const unsigned a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const unsigned b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return a | (b << 16);
}

// One warp per (layer, token): out row = sum_j w_j * y[pos_j] in slot order.
// Warp-uniform chunk loop as in k_permute.
template <int KB>
__global__ void __launch_bounds__(256)
k_combine(const int4 *__restrict__ y, const int32_t *__restrict__ inv, const float *__restrict__ w,
          int4 *out, WsHeader *hdr, int T, int k, int nv, int64_t npairs, int64_t ntok) {
    const int64_t tok = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (tok >= ntok) return;                           // whole warp
    const int lane = threadIdx.x & 31;
    const int64_t l = tok / T;
    int pa, pb;
    if (!token_positions(inv + tok * k, k, npairs, pa, pb)) {
        if (lane == 0) set_error(hdr, TOPO_ESTATE);
        return;
    }
    const float wa = lane < k ? __ldg(w + tok * k + lane) : 0.f;
    const float wb = lane + 32 < k ? __ldg(w + tok * k + lane + 32) : 0.f;
    constexpr int KD = KB > 0 ? KB : 1;
    int64_t src[KD];
    float wt[KD];
    if (KB > 0) {
#pragma unroll
        for (int j = 0; j < KD; ++j) {
            src[j] = (l * npairs + slot_pos(j, pa, pb)) * nv;
            const float x0 = __shfl_sync(0xffffffffu, wa, j & 31);
            const float x1 = __shfl_sync(0xffffffffu, wb, j & 31);
            wt[j] = j < 32 ? x0 : x1;
        }
    }
    int4 *o = out + tok * nv;
    for (int c0 = 0; c0 < nv; c0 += 32) {
        const int c = c0 + lane;
        const bool in = c < nv;
        float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (KB > 0) {
            int4 v[KD];
#pragma unroll
            for (int j = 0; j < KD; ++j)                       // all k rows requested first
                v[j] = in ? __ldg(y + src[j] + c) : make_int4(0, 0, 0, 0);
#pragma unroll
            for (int j = 0; j < KD; ++j) acc8(a, wt[j], v[j]);
        } else {
            for (int j = 0; j < k; ++j) {
                const int64_t s = (l * npairs + slot_pos(j, pa, pb)) * nv;
                const float x0 = __shfl_sync(0xffffffffu, wa, j & 31);
                const float x1 = __shfl_sync(0xffffffffu, wb, j & 31);
                const int4 v = in ? __ldg(y + s + c) : make_int4(0, 0, 0, 0);
                acc8(a, j < 32 ? x0 : x1, v);
            }
        }
        if (in) {
            int4 r;
            r.x = (int)pack2(a[0], a[1]);
            r.y = (int)pack2(a[2], a[3]);
            r.z = (int)pack2(a[4], a[5]);
            r.w = (int)pack2(a[6], a[7]);
            o[c] = r;
        }
    }
}

cudaError_t launch_invert(const Geo &g, const int32_t *sorted, void *ws, cudaStream_t st) {
    cudaError_t e;
    const int64_t total = (int64_t)g.L * g.npairs;
    int32_t *inv = ws_at<int32_t>(ws, g.off_pack_inv);
    if ((e = cudaMemsetAsync(inv, 0xff, (size_t)total * 4, st)) != cudaSuccess) return e;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 64) blocks = 152 * 64;
    k_invert<<<(unsigned)blocks, 256, 0, st>>>(sorted, inv, ws_at<WsHeader>(ws, 0), g.npairs, total);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_permute(const Geo &g, int H, const uint16_t *x, const int32_t *sorted, uint16_t *y,
                           void *ws, cudaStream_t st) {
    cudaError_t e;
    if ((e = launch_invert(g, sorted, ws, st)) != cudaSuccess) return e;
    const int64_t ntok = (int64_t)g.L * g.T;
    if (ntok == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((ntok + 7) / 8);
    const int nv = H / 8;
    const int4 *xv = reinterpret_cast<const int4 *>(x);
    int4 *yv = reinterpret_cast<int4 *>(y);
    const int32_t *inv = ws_at<int32_t>(ws, g.off_pack_inv);
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    switch (g.k) {
        case 2: k_permute<2><<<blocks, 256, 0, st>>>(xv, inv, yv, hdr, g.T, g.k, nv, g.npairs, ntok); break;
        case 4: k_permute<4><<<blocks, 256, 0, st>>>(xv, inv, yv, hdr, g.T, g.k, nv, g.npairs, ntok); break;
        case 6: k_permute<6><<<blocks, 256, 0, st>>>(xv, inv, yv, hdr, g.T, g.k, nv, g.npairs, ntok); break;
        case 8: k_permute<8><<<blocks, 256, 0, st>>>(xv, inv, yv, hdr, g.T, g.k, nv, g.npairs, ntok); break;
        case 10: k_permute<10><<<blocks, 256, 0, st>>>(xv, inv, yv, hdr, g.T, g.k, nv, g.npairs, ntok); break;
        default: k_permute<0><<<blocks, 256, 0, st>>>(xv, inv, yv, hdr, g.T, g.k, nv, g.npairs, ntok); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_combine(const Geo &g, int H, const uint16_t *y, const int32_t *sorted, const float *w,
                           uint16_t *out, void *ws, cudaStream_t st) {
    cudaError_t e;
    if ((e = launch_invert(g, sorted, ws, st)) != cudaSuccess) return e;
    const int64_t ntok = (int64_t)g.L * g.T;
    if (ntok == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((ntok + 7) / 8);
    const int nv = H / 8;
    const int4 *yv = reinterpret_cast<const int4 *>(y);
    int4 *ov = reinterpret_cast<int4 *>(out);
    const int32_t *inv = ws_at<int32_t>(ws, g.off_pack_inv);
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    switch (g.k) {
        case 2: k_combine<2><<<blocks, 256, 0, st>>>(yv, inv, w, ov, hdr, g.T, g.k, nv, g.npairs, ntok); break;
        case 4: k_combine<4><<<blocks, 256, 0, st>>>(yv, inv, w, ov, hdr, g.T, g.k, nv, g.npairs, ntok); break;
        case 6: k_combine<6><<<blocks, 256, 0, st>>>(yv, inv, w, ov, hdr, g.T, g.k, nv, g.npairs, ntok); break;
        case 8: k_combine<8><<<blocks, 256, 0, st>>>(yv, inv, w, ov, hdr, g.T, g.k, nv, g.npairs, ntok); break;
        case 10: k_combine<10><<<blocks, 256, 0, st>>>(yv, inv, w, ov, hdr, g.T, g.k, nv, g.npairs, ntok); break;
        default: k_combine<0><<<blocks, 256, 0, st>>>(yv, inv, w, ov, hdr, g.T, g.k, nv, g.npairs, ntok); break;
    }
    return cudaGetLastError();
}

}  // namespace topo
