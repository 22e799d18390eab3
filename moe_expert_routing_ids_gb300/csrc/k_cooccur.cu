// Expert co-selection and cross-layer transition counts ("Expert Coupling in
// MoE Pretraining": within-layer correlation, cross-layer correlation).
//
//   co[l][a][b] = sum_t n_t^l[a] n_t^l[b],   tr[l][a][b] = sum_t n_t^l[a] n_t^{l+1}[b]
//
// Each CTA takes a block of tokens of one layer and counts into int32
// shared-memory matrices: co only on and above the diagonal (for i < j the
// unordered pair {x_i, x_j} adds 1 at (min, max), or 2 on the diagonal when
// the two ids repeat; i == j adds 1 on the diagonal), tr in full.  A cluster
// of kCl CTAs of the same layer then sums its shared matrices through
// distributed shared memory -- each CTA reduces one slice of the entries over
// the cluster -- and adds the slice to the int64 outputs (zeroed first), the
// co slice mirrored below the diagonal.  Integer adds only: exact and
// order-independent.  Large E splits the matrix rows over a third grid
// dimension.
//
// For k in {2, 4, 6, 8, 10} and E <= 159 (both (E+1)^2 matrices in one CTA's
// shared memory) k_cooccur_fast does the same with exact-k loops and no
// per-pair checks, 1024 threads per CTA, and the cluster size that keeps the
// most CTAs resident.  It is bound by the shared-memory atomics: random
// columns put about 3.5 lanes of a warp on one bank.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace topo {
namespace {

constexpr int kCl = 8;                    // CTAs per cluster
constexpr int kCoThreads = 512;
constexpr size_t kCoSmemCap = 200 * 1024;   // shared matrices per CTA

// Sums the cluster's shared matrices slice by slice and adds them to the
// int64 outputs (co mirrored below the diagonal).
__device__ void cluster_reduce(cg::cluster_group &cl, int *sm, int64_t *co, int64_t *tr, bool has_tr,
                               int l, int E, int a0, int nrow, int nent) {
    cl.sync();
    // cluster reduction: this CTA owns entries [e0, e1) of both matrices
    const int me = (int)cl.block_rank();
    const int per = (nent + kCl - 1) / kCl;
    const int e0 = me * per, e1 = min(nent, e0 + per);
    int64_t *CO = co + (int64_t)l * E * E;
    int64_t *TR = has_tr ? tr + (int64_t)l * E * E : nullptr;
    for (int i = e0 + threadIdx.x; i < e1; i += blockDim.x) {
        const int a = i / E, b = i % E;
        if (a >= nrow) continue;
        int vc = 0, vt = 0;
#pragma unroll
        for (int c = 0; c < kCl; ++c) {
            const int *peer = cl.map_shared_rank(sm, c);
            vc += peer[i];
            if (has_tr) vt += peer[nent + i];
        }
        const int ga = a0 + a;
        if (vc) {
            atomicAdd(reinterpret_cast<unsigned long long *>(&CO[(int64_t)ga * E + b]),
                      (unsigned long long)vc);
            if (ga != b)
                atomicAdd(reinterpret_cast<unsigned long long *>(&CO[(int64_t)b * E + ga]),
                          (unsigned long long)vc);
        }
        if (vt)
            atomicAdd(reinterpret_cast<unsigned long long *>(&TR[(int64_t)ga * E + b]),
                      (unsigned long long)vt);
    }
    cl.sync();   // peers' shared memory must outlive the reads above
}

template <int KMAX>
__global__ void __launch_bounds__(kCoThreads)
k_cooccur(const int32_t *__restrict__ ids, int64_t *co, int64_t *tr, WsHeader *hdr, int L, int T,
          int E, int k, int rows, int tok_per_cta) {
    extern __shared__ int sm[];
    cg::cluster_group cl = cg::this_cluster();
    const int l = blockIdx.y;
    const int a0 = blockIdx.z * rows;
    const int a1 = min(E, a0 + rows);
    const int nrow = a1 - a0;
    const bool has_tr = (tr != nullptr) && (l + 1 < L);
    int *sco = sm;                         // [rows][E]
    int *str = sm + (size_t)rows * E;      // [rows][E]
    const int nent = rows * E;
    for (int i = threadIdx.x; i < 2 * nent; i += blockDim.x) sm[i] = 0;
    __syncthreads();

    const int t0 = blockIdx.x * tok_per_cta;
    const int t1 = min(T, t0 + tok_per_cta);
    bool bad = false;
    for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
        int x[KMAX], y[KMAX];
        const int32_t *pa = ids + ((int64_t)l * T + t) * k;
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
            x[i] = -1;
            if (i < k) {
                const int v = __ldg(pa + i);
                if ((unsigned)v < (unsigned)E) x[i] = v;
                else bad = true;
            }
        }
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
            if (i >= k || x[i] < 0) continue;
            const int xi = x[i];
            if (xi >= a0 && xi < a1) atomicAdd(&sco[(xi - a0) * E + xi], 1);
#pragma unroll
            for (int j = i + 1; j < KMAX; ++j) {
                if (j >= k || x[j] < 0) continue;
                const int xj = x[j];
                const int lo = min(xi, xj), hi = max(xi, xj);
                if (lo >= a0 && lo < a1) atomicAdd(&sco[(lo - a0) * E + hi], lo == hi ? 2 : 1);
            }
        }
        if (has_tr) {
            const int32_t *pb = ids + ((int64_t)(l + 1) * T + t) * k;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                y[j] = -1;
                if (j < k) {
                    const int v = __ldg(pb + j);
                    if ((unsigned)v < (unsigned)E) y[j] = v;
                    else bad = true;
                }
            }
#pragma unroll
            for (int i = 0; i < KMAX; ++i) {
                if (i >= k || x[i] < a0 || x[i] >= a1) continue;
                int *rowp = str + (x[i] - a0) * E;
#pragma unroll
                for (int j = 0; j < KMAX; ++j)
                    if (j < k && y[j] >= 0) atomicAdd(&rowp[y[j]], 1);
            }
        }
    }
    if (bad) set_error(hdr, TOPO_ERANGE);
    cluster_reduce(cl, sm, co, tr, has_tr, l, E, a0, nrow, nent);
}


// Exact k = K and E small enough for both full matrices in shared memory
// (row stride S = E + 1).  An id outside [0, E) is counted at the spare index
// E, which the reduction drops, so the pair loops carry no checks.  One
// thread per token.  Cluster size is a launch parameter (cs CTAs of one
// layer reduce through distributed shared memory).
template <int K>
__global__ void __launch_bounds__(1024)
k_cooccur_fast(const int32_t *__restrict__ ids, int64_t *co, int64_t *tr, WsHeader *hdr, int L, int T,
               int E, int tok_per_cta) {
    extern __shared__ int sm[];
    cg::cluster_group cl = cg::this_cluster();
    const int l = blockIdx.y;
    const int S = E + 1, nent = S * S;
    const bool has_tr = (tr != nullptr) && (l + 1 < L);
    int *sco = sm;
    int *str = sm + nent;
    for (int i = threadIdx.x; i < 2 * nent; i += blockDim.x) sm[i] = 0;
    __syncthreads();
    const int t0 = blockIdx.x * tok_per_cta;
    const int t1 = min(T, t0 + tok_per_cta);
    bool bad = false;
    for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
        int x[K];
        const int32_t *pa = ids + ((int64_t)l * T + t) * K;
#pragma unroll
        for (int i = 0; i < K; ++i) x[i] = __ldg(pa + i);
#pragma unroll
        for (int i = 0; i < K; ++i)
            if ((unsigned)x[i] >= (unsigned)E) { bad = true; x[i] = E; }
#pragma unroll
        for (int i = 0; i < K; ++i) {
            atomicAdd(&sco[x[i] * (S + 1)], 1);
#pragma unroll
            for (int j = i + 1; j < K; ++j) {
                const int lo = min(x[i], x[j]), hi = max(x[i], x[j]);
                atomicAdd(&sco[lo * S + hi], 1 + (lo == hi));
            }
        }
        if (has_tr) {
            int y[K];
            const int32_t *pb = pa + (int64_t)T * K;
#pragma unroll
            for (int j = 0; j < K; ++j) y[j] = __ldg(pb + j);
#pragma unroll
            for (int j = 0; j < K; ++j)
                if ((unsigned)y[j] >= (unsigned)E) { bad = true; y[j] = E; }
#pragma unroll
            for (int i = 0; i < K; ++i) {
                int *rowp = str + x[i] * S;
#pragma unroll
                for (int j = 0; j < K; ++j) atomicAdd(&rowp[y[j]], 1);
            }
        }
    }
    if (bad) set_error(hdr, TOPO_ERANGE);
    cl.sync();
    // this CTA sums entries [e0, e1) over the cluster; co is upper-triangular
    const int cs = (int)cl.num_blocks(), me = (int)cl.block_rank();
    const int per = (nent + cs - 1) / cs;
    const int e0 = me * per, e1 = min(nent, e0 + per);
    int64_t *CO = co + (int64_t)l * E * E;
    int64_t *TR = has_tr ? tr + (int64_t)l * E * E : nullptr;
    for (int i = e0 + threadIdx.x; i < e1; i += blockDim.x) {
        const int a = i / S, b = i - a * S;
        if (a == E || b == E) continue;
        int vc = 0, vt = 0;
        for (int c = 0; c < cs; ++c) {
            const int *peer = cl.map_shared_rank(sm, c);
            vc += peer[i];
            if (has_tr) vt += peer[nent + i];
        }
        if (vc) {
            atomicAdd(reinterpret_cast<unsigned long long *>(&CO[(int64_t)a * E + b]),
                      (unsigned long long)vc);
            if (a != b)
                atomicAdd(reinterpret_cast<unsigned long long *>(&CO[(int64_t)b * E + a]),
                          (unsigned long long)vc);
        }
        if (vt)
            atomicAdd(reinterpret_cast<unsigned long long *>(&TR[(int64_t)a * E + b]),
                      (unsigned long long)vt);
    }
    cl.sync();   // peers' shared memory must outlive the reads above
}

template <int K>
cudaError_t launch_fast(int L, int T, int E, const int32_t *ids, int64_t *co, int64_t *tr,
                        WsHeader *hdr, cudaStream_t st) {
    const size_t smem = 2 * (size_t)(E + 1) * (E + 1) * 4;
    const void *fn = (const void *)k_cooccur_fast<K>;
    cudaError_t e;
    if ((e = ensure_smem(fn, smem)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(1024);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the cluster size that keeps the most CTAs resident at once, a whole
    // number of clusters per layer, at least 1024 tokens per CTA
    int best_cs = 1, best_cpl = 1;
    long best = 0;
    const int max_ctas = (T + 1023) / 1024;
    for (int cs : {8, 6, 4, 2, 1}) {
        attr[0].val.clusterDim.x = cs;
        cfg.gridDim = dim3(cs, L, 1);
        int n_cl = 0;
        if (cudaOccupancyMaxActiveClusters(&n_cl, fn, &cfg) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        int cpl = n_cl / L;                                    // clusters per layer
        while (cpl > 1 && cpl * cs > max_ctas) --cpl;
        if (cpl < 1) cpl = 1;
        const long ctas = (long)cpl * cs * L;
        if (ctas > best) { best = ctas; best_cs = cs; best_cpl = cpl; }
    }
    const int ctas = best_cpl * best_cs;
    attr[0].val.clusterDim.x = best_cs;
    cfg.gridDim = dim3(ctas, L, 1);
    const int tok_per_cta = (T + ctas - 1) / ctas;
    if ((e = cudaLaunchKernelEx(&cfg, k_cooccur_fast<K>, ids, co, tr, hdr, L, T, E, tok_per_cta)) !=
        cudaSuccess)
        return e;
    return cudaGetLastError();
}

// Any k: the same counts with the ids re-read from global memory (L1) in
// rolled loops; used only when k > 16.
__global__ void __launch_bounds__(kCoThreads)
k_cooccur_any(const int32_t *__restrict__ ids, int64_t *co, int64_t *tr, WsHeader *hdr, int L, int T,
              int E, int k, int rows, int tok_per_cta) {
    extern __shared__ int sm[];
    cg::cluster_group cl = cg::this_cluster();
    const int l = blockIdx.y;
    const int a0 = blockIdx.z * rows;
    const int a1 = min(E, a0 + rows);
    const int nrow = a1 - a0;
    const bool has_tr = (tr != nullptr) && (l + 1 < L);
    int *sco = sm;
    int *str = sm + (size_t)rows * E;
    const int nent = rows * E;
    for (int i = threadIdx.x; i < 2 * nent; i += blockDim.x) sm[i] = 0;
    __syncthreads();
    const int t0 = blockIdx.x * tok_per_cta;
    const int t1 = min(T, t0 + tok_per_cta);
    bool bad = false;
    for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
        const int32_t *pa = ids + ((int64_t)l * T + t) * k;
        const int32_t *pb = has_tr ? ids + ((int64_t)(l + 1) * T + t) * k : nullptr;
#pragma unroll 1
        for (int i = 0; i < k; ++i) {
            const int xi = __ldg(pa + i);
            if ((unsigned)xi >= (unsigned)E) { bad = true; continue; }
            if (xi >= a0 && xi < a1) atomicAdd(&sco[(xi - a0) * E + xi], 1);
#pragma unroll 1
            for (int j = i + 1; j < k; ++j) {
                const int xj = __ldg(pa + j);
                if ((unsigned)xj >= (unsigned)E) continue;
                const int lo = min(xi, xj), hi = max(xi, xj);
                if (lo >= a0 && lo < a1) atomicAdd(&sco[(lo - a0) * E + hi], lo == hi ? 2 : 1);
            }
            if (!has_tr || xi < a0 || xi >= a1) continue;
#pragma unroll 1
            for (int j = 0; j < k; ++j) {
                const int yj = __ldg(pb + j);
                if ((unsigned)yj < (unsigned)E) atomicAdd(&str[(xi - a0) * E + yj], 1);
            }
        }
        if (has_tr)
            for (int j = 0; j < k; ++j)
                if ((unsigned)__ldg(pb + j) >= (unsigned)E) bad = true;
    }
    if (bad) set_error(hdr, TOPO_ERANGE);
    cluster_reduce(cl, sm, co, tr, has_tr, l, E, a0, nrow, nent);
}

}  // namespace

cudaError_t launch_cooccur(int L, int T, int E, int k, const int32_t *ids, int64_t *co, int64_t *tr,
                           void *ws, cudaStream_t st) {
    cudaError_t e;
    if ((e = cudaMemsetAsync(co, 0, (size_t)L * E * E * 8, st)) != cudaSuccess) return e;
    if (tr && L > 1 && (e = cudaMemsetAsync(tr, 0, (size_t)(L - 1) * E * E * 8, st)) != cudaSuccess)
        return e;
    if (T == 0) return cudaSuccess;
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    if (2 * (size_t)(E + 1) * (E + 1) * 4 <= kCoSmemCap) {
        switch (k) {
            case 2: return launch_fast<2>(L, T, E, ids, co, tr, hdr, st);
            case 4: return launch_fast<4>(L, T, E, ids, co, tr, hdr, st);
            case 6: return launch_fast<6>(L, T, E, ids, co, tr, hdr, st);
            case 8: return launch_fast<8>(L, T, E, ids, co, tr, hdr, st);
            case 10: return launch_fast<10>(L, T, E, ids, co, tr, hdr, st);
            default: break;
        }
    }
    int rows = (int)(kCoSmemCap / (2 * (size_t)E * 4));
    if (rows < 1) return cudaErrorInvalidValue;
    if (rows > E) rows = E;
    const int chunks = (E + rows - 1) / rows;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // clusters per (layer, row chunk): fill the SMs once, at least one cluster
    int cpl = (sms / kCl) / (L * chunks);
    if (cpl < 1) cpl = 1;
    const int max_ctas = (T + 255) / 256;            // keep >= 256 tokens per CTA
    while (cpl > 1 && cpl * kCl > max_ctas) --cpl;
    const int ctas = cpl * kCl;
    const int tok_per_cta = (T + ctas - 1) / ctas;
    const size_t smem = 2 * (size_t)rows * E * 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, L, chunks);
    cfg.blockDim = dim3(kCoThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (k <= 8) {
        if ((e = ensure_smem((const void *)k_cooccur<8>, smem)) != cudaSuccess) return e;
        e = cudaLaunchKernelEx(&cfg, k_cooccur<8>, ids, co, tr, hdr, L, T, E, k, rows, tok_per_cta);
    } else if (k <= 16) {
        if ((e = ensure_smem((const void *)k_cooccur<16>, smem)) != cudaSuccess) return e;
        e = cudaLaunchKernelEx(&cfg, k_cooccur<16>, ids, co, tr, hdr, L, T, E, k, rows, tok_per_cta);
    } else {
        if ((e = ensure_smem((const void *)k_cooccur_any, smem)) != cudaSuccess) return e;
        e = cudaLaunchKernelEx(&cfg, k_cooccur_any, ids, co, tr, hdr, L, T, E, k, rows, tok_per_cta);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace topo
