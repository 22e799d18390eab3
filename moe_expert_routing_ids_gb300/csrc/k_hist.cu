// Routing matrix Omega (TopoEP §4.1, Eq. 3) and the per-tile expert index.
//
// One CTA per tile of TT tokens inside one source rank's block.  The tile's
// ids are streamed once with 16-byte loads and counted into a shared-memory
// histogram (integer shared atomics, no float).  Each CTA stores its counts;
// the last CTA of a source (one release fence + counter by thread 0, no
// waiting) turns the source's tile counts into exclusive prefixes -- the index
// that lets the rerouting kernel rank pairs in one pass -- and writes the
// source's row of Omega.
#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

constexpr int kHistThreads = 512;

__device__ __forceinline__ void count_id(int e, int E, int *cnt, bool &bad) {
    if ((unsigned)e < (unsigned)E)
        atomicAdd(&cnt[e], 1);
    else
        bad = true;
}

__global__ void __launch_bounds__(kHistThreads)
k_hist_tiles(const int32_t *__restrict__ ids, int32_t *__restrict__ hist, int32_t *tile_cnt,
             int32_t *done, WsHeader *hdr, Geo g, uint64_t fp) {
    extern __shared__ int cnt[];
    __shared__ int is_last;
    const int E = g.E;
    const int tile = blockIdx.x;
    const int t = tile % g.tps;
    const int s = (tile / g.tps) % g.R;
    const int l = tile / (g.tps * g.R);
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();

    const int tok0 = t * g.TT;
    const int ntok = max(0, min(g.TT, g.tpr - tok0));
    bool bad = false;
    if (ntok > 0) {
        const int32_t *a = ids + (int64_t)l * g.npairs + ((int64_t)s * g.tpr + tok0) * g.k;
        const int n = ntok * g.k;
        int head = (int)(((16 - ((uintptr_t)a & 15)) & 15) >> 2);
        if (head > n) head = n;
        for (int i = threadIdx.x; i < head; i += blockDim.x) count_id(__ldg(a + i), E, cnt, bad);
        const int4 *v = reinterpret_cast<const int4 *>(a + head);
        const int nv = (n - head) >> 2;
        int i = threadIdx.x;
        for (; i + 3 * (int)blockDim.x < nv; i += 4 * blockDim.x) {
            int4 x0 = __ldg(v + i), x1 = __ldg(v + i + blockDim.x);
            int4 x2 = __ldg(v + i + 2 * blockDim.x), x3 = __ldg(v + i + 3 * blockDim.x);
            count_id(x0.x, E, cnt, bad); count_id(x0.y, E, cnt, bad);
            count_id(x0.z, E, cnt, bad); count_id(x0.w, E, cnt, bad);
            count_id(x1.x, E, cnt, bad); count_id(x1.y, E, cnt, bad);
            count_id(x1.z, E, cnt, bad); count_id(x1.w, E, cnt, bad);
            count_id(x2.x, E, cnt, bad); count_id(x2.y, E, cnt, bad);
            count_id(x2.z, E, cnt, bad); count_id(x2.w, E, cnt, bad);
            count_id(x3.x, E, cnt, bad); count_id(x3.y, E, cnt, bad);
            count_id(x3.z, E, cnt, bad); count_id(x3.w, E, cnt, bad);
        }
        for (; i < nv; i += blockDim.x) {
            int4 x = __ldg(v + i);
            count_id(x.x, E, cnt, bad); count_id(x.y, E, cnt, bad);
            count_id(x.z, E, cnt, bad); count_id(x.w, E, cnt, bad);
        }
        for (int j = head + nv * 4 + threadIdx.x; j < n; j += blockDim.x)
            count_id(__ldg(a + j), E, cnt, bad);
    }
    if (bad) set_error(hdr, TOPO_ERANGE);
    __syncthreads();

    int32_t *mine = tile_cnt + (((int64_t)l * g.R + s) * g.tps + t) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) mine[e] = cnt[e];
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();                        // release this CTA's counts (cumulative)
        const int old = atomicAdd(&done[l * g.R + s], 1);
        is_last = (old == g.tps - 1);
        if (is_last) __threadfence();           // acquire the other CTAs' counts
    }
    __syncthreads();
    if (!is_last) return;
    // Last tile of source s: exclusive prefix over the source's tiles, and the
    // source's row of Omega.
    int32_t *first = tile_cnt + ((int64_t)l * g.R + s) * g.tps * E;
    int32_t *hrow = hist + ((int64_t)l * g.R + s) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int u = 0; u < g.tps; ++u) {
            const int c = __ldcg(first + (int64_t)u * E + e);
            first[(int64_t)u * E + e] = run;
            run += c;
        }
        hrow[e] = run;
    }
    if (threadIdx.x == 0) {
        hdr->hist_fp = fp;
        hdr->route_fp = 0;                      // any routing index is now stale
    }
}

}  // namespace

cudaError_t launch_hist(const Geo &g, const int32_t *ids, int32_t *hist, void *ws, uint64_t fp,
                        cudaStream_t st) {
    const int64_t tiles = (int64_t)g.L * g.R * g.tps;
    if (tiles == 0) return cudaSuccess;
    if (tiles > INT32_MAX) return cudaErrorInvalidValue;
    cudaError_t e0 = cudaMemsetAsync(ws_at<int32_t>(ws, g.off_done), 0, (size_t)g.L * g.R * 4, st);
    if (e0 != cudaSuccess) return e0;
    const size_t smem = (size_t)g.E * sizeof(int);
    cudaError_t e1 = ensure_smem((const void *)k_hist_tiles, smem);
    if (e1 != cudaSuccess) return e1;
    k_hist_tiles<<<(unsigned)tiles, kHistThreads, smem, st>>>(
        ids, hist, ws_at<int32_t>(ws, g.off_tile), ws_at<int32_t>(ws, g.off_done),
        ws_at<WsHeader>(ws, 0), g, fp);
    return cudaGetLastError();
}

}  // namespace topo
