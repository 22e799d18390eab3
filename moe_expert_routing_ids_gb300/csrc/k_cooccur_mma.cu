// Expert co-selection and transition counts on the tensor cores ("Expert
// Coupling in MoE Pretraining": within-layer and cross-layer correlation).
//
// With C_l the T x E count matrix of layer l (C_l[t][e] = times token t
// selected e), co_l = C_l^T C_l and tr_l = C_l^T C_{l+1}: dense contractions
// over the tokens.  One CTA per (layer, chunk of tokens) -- a "unit" -- builds
// the count tiles of layers l and l+1 in shared memory, 128 experts x 128
// tokens per K-block, and issues tcgen05.mma (D[a][b] += sum_t A[a][t] B[b][t],
// M = N = 128) with the two accumulators in tensor memory: co (A = B = the
// layer-l tile) and tr (A = layer l, B = layer l+1).  Counts are small
// integers (at most k <= 16 per token), exact in bf16 and in e4m3; products
// and sums are integers, exact in the float32 accumulator while a cell stays
// below 2^24, which bounds a unit's tokens (kMaxChunkTokens * 16 * 16 <=
// 2^24).  The epilogue reads the accumulators back (tcgen05.ld), converts
// them to int32 partials per unit, and k_cooc_reduce sums a layer's partials
// into the int64 outputs.  Shared-memory layout of a tile: one 128-byte row
// of e4m3 counts per expert (a K-block of 128 tokens), in the K-major
// 128-byte swizzle layout (8-row atoms of 1024 bytes).
//
// Three stages: the builders fill stage s while the tensor core still works
// on the others; tcgen05.commit arrives on stage s's mbarrier once the MMAs
// that read it are done.  Every mbarrier wait is bounded: on expiry the kernel
// records TOPO_ETIMEOUT, waits (bounded) for its own MMAs, frees its tensor
// memory and returns.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace topo {
namespace {

constexpr int kMmaKB = 256;                   // tokens per K-block: two 128-token swizzle atoms along K
constexpr int kMmaThreads = 2 * kMmaKB;       // one thread per (layer, token) of a K-block
constexpr int kMmaRows = 128;                 // M: experts (E <= 128, the rest zero rows)
constexpr int kMmaK = 32;                     // K of one kind::f8f6f4 MMA
constexpr int kMmaStages = 3;
constexpr uint32_t kAtomRows = 128 * 128;     // one layer's 128 rows x 128 tokens (16 KB)
constexpr uint32_t kStage = 4 * kAtomRows;    // [K-atom][layer][row][128 B] (64 KB)
constexpr uint32_t kAtom = 1024;              // 8 rows x 128 B: one swizzle atom
constexpr int kTmemCols = 256;                // co: columns [0, 128), tr: [128, 256)
constexpr uint64_t kWaitNs = 200000000ull;    // longest mbarrier wait: 0.2 s of %globaltimer
constexpr uint8_t kE4m3One = 0x38;            // 1.0 in e4m3: sign 0, exponent 7 (the bias), mantissa 0

// Instruction descriptor of kind::f8f6f4: D float32 (bits 4-5 = 1), A and B
// e4m3 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f8(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kMmaRows >> 4) << 24);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout: start address >> 4 (bits 0-13), leading offset >> 4
// (bits 16-29; 1, unused: a row's K extent is one atom), stride offset >> 4
// (bits 32-45) = 1024 bytes between 8-row groups, version 1 (bit 46), layout
// type 2 = 128-byte swizzle (bits 61-63).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(kAtom >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the completion of the phase with the given parity: non-blocking
// tests with a short sleep between them, for at most kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    const uint64_t start = globaltimer_ns();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
        if (globaltimer_ns() - start > kWaitNs) return false;
        __nanosleep(32);
    }
}

__device__ __forceinline__ void mma_f8(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(da), "l"(db), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrive on bar once every tcgen05 operation this thread issued is complete.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive float32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
          "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
          "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
          "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

constexpr int kMaxKIds = 16;

// KT: k at compile time (0: any k <= 16).  Token ids in registers.
// A token's ids into registers: 16-byte loads when vec (the row is 16-byte
// aligned and KT is a multiple of 4), else one load per slot.  Slots past k,
// and tokens that are not valid, read as -1 (no expert).
template <int KT>
__device__ __forceinline__ void load_token(const int32_t *src, int k, bool valid, bool vec,
                                           int (&v)[KT > 0 ? KT : kMaxKIds]) {
    constexpr int KB = KT > 0 ? KT : kMaxKIds;
    if (KT > 0 && KT % 4 == 0 && vec) {
#pragma unroll
        for (int q = 0; q < KB / 4; ++q) {
            int4 a = valid ? __ldg(reinterpret_cast<const int4 *>(src) + q) : make_int4(-1, -1, -1, -1);
            v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < KB; ++j) v[j] = (valid && j < k) ? __ldg(src + j) : -1;
}

// True when the token's k ids are pairwise different (the Top-k case).  For
// eight ids below 128 the comparisons run four bytes at a time: packed words
// A (ids 0-3) and B (ids 4-7) against their byte rotations cover every pair.
template <int KT>
__device__ __forceinline__ bool distinct_ids(const int (&v)[KT > 0 ? KT : kMaxKIds], int k) {
    constexpr int KB = KT > 0 ? KT : kMaxKIds;
    if (KT == 8) {
        unsigned hi = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) hi |= (unsigned)v[j];
        if (hi < 128u) {
            // x ^ y has a zero byte exactly where two packed ids are equal; a
            // zero byte of z shows in (z - 0x01..) & ~z & 0x80.. (ids < 128)
            const unsigned A = (unsigned)v[0] | ((unsigned)v[1] << 8) | ((unsigned)v[2] << 16) | ((unsigned)v[3] << 24);
            const unsigned B = (unsigned)v[4] | ((unsigned)v[5] << 8) | ((unsigned)v[6] << 16) | ((unsigned)v[7] << 24);
            auto zb = [](unsigned z) { return (z - 0x01010101u) & ~z & 0x80808080u; };
            const unsigned r1 = __funnelshift_l(B, B, 8), r2 = __funnelshift_l(B, B, 16), r3 = __funnelshift_l(B, B, 24);
            const unsigned eq = zb(A ^ __funnelshift_l(A, A, 8)) | zb(A ^ __funnelshift_l(A, A, 16)) |
                                zb(B ^ r1) | zb(B ^ r2) | zb(A ^ B) | zb(A ^ r1) | zb(A ^ r2) | zb(A ^ r3);
            return eq == 0u;
        }
    }
    bool d = true;
#pragma unroll
    for (int i = 0; i < KB; ++i)
#pragma unroll
        for (int j = i + 1; j < KB; ++j)
            if (j < k) d &= v[i] != v[j];
    return d;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

constexpr int kBuildWarps = kMmaThreads / 32;     // builder warps; the next warp issues MMAs

// One CTA per unit (layer l, chunk of tokens).  Warp-specialized: the
// builder warps (thread x * kMmaKB + tt fills token column tt of layer l + x)
// each own one column per stage -- they clear the bytes they set in that
// stage kMmaStages K-blocks ago and set the new ones, so no thread touches
// another's bytes and no tile is zeroed between uses -- and report a filled
// stage on its `full` barrier (one arrival per warp).  The issuer warp waits
// on `full`, issues per 32-token step one MMA of N = 256 (B = the layer-l rows
// followed by the layer-(l+1) rows: co in TMEM columns 0-127, tr in 128-255;
// N = 128 for the last layer) and commits to the stage's `empty` barrier, which
// the builders wait on before reusing the stage.  No CTA-wide barrier runs
// inside the loop.
template <int KT>
__global__ void __launch_bounds__(kMmaThreads + 32, 1)
k_cooccur_mma(const int32_t *__restrict__ ids, int32_t *__restrict__ part, WsHeader *hdr, int L, int T,
              int E, int k, int nchunks, int chunk, int want_tr, int vec) {
    constexpr int KB = KT > 0 ? KT : kMaxKIds;
    extern __shared__ __align__(1024) unsigned char smc[];
    __shared__ __align__(8) uint64_t full[kMmaStages];
    __shared__ __align__(8) uint64_t empty[kMmaStages];
    __shared__ __align__(8) uint64_t mbar_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int timed_out;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int l = unit / nchunks, c = unit - l * nchunks;
    const bool has_tr = want_tr && l + 1 < L;
    const int t0 = c * chunk, t1 = min(T, t0 + chunk);
    const int nkb = t1 > t0 ? (t1 - t0 + kMmaKB - 1) / kMmaKB : 0;
    const int kk = KT > 0 ? KT : k;
    int32_t *pu = part + (int64_t)unit * 2 * kMmaRows * kMmaRows;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int s = 0; s < kMmaStages; ++s) {
            mbar_init(&full[s], kBuildWarps);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&mbar_done, 1);
        timed_out = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    {   // all tiles start at zero
        uint4 *z = reinterpret_cast<uint4 *>(smc);
        for (int i = tid; i < (int)(kMmaStages * kStage / 16); i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    bool bad = false;

    if (warp < kBuildWarps) {
        // ------------------------------------------------------------ builders
        const int x = tid / kMmaKB, tt = tid % kMmaKB;
        const bool builds = x == 0 || has_tr;
        const int32_t *lay = ids + (int64_t)(l + x) * T * kk;
        // byte of (layer x, expert e, token tt) in a stage laid out [K-atom]
        // [layer][row][128 B]: tokens 128a .. 128a+127 in K-atom a; row e is
        // 128 bytes with its 16-byte chunks permuted by XOR with e % 8 (the
        // 128-byte swizzle); the two layers' rows of one K-atom are contiguous,
        // one operand of 256 rows.  off = colb + 128 e + (((cb ^ e) & 7) << 4).
        const int cc = tt & 127;
        const uint32_t colb = (uint32_t)(tt >> 7) * 2u * kAtomRows + (uint32_t)x * kAtomRows + (uint32_t)(cc & 15);
        const int cb = cc >> 4;
        int nxt[KB];
        load_token<KT>(lay + (int64_t)(t0 + tt) * kk, kk, builds && t0 + tt < t1, vec, nxt);
        uint32_t set[kMmaStages][KB];     // bytes this thread set in each stage (all ones: none)
#pragma unroll
        for (int s = 0; s < kMmaStages; ++s)
#pragma unroll
            for (int j = 0; j < KB; ++j) set[s][j] = 0xffffffffu;
        bool stop = false;
        for (int kb0 = 0; kb0 < nkb && !stop; kb0 += kMmaStages)
#pragma unroll
        for (int s = 0; s < kMmaStages; ++s) {     // s compile-time: set[s][] stays in registers
            const int kb = kb0 + s;
            if (kb >= nkb || stop) break;
            int cur[KB];
#pragma unroll
            for (int j = 0; j < KB; ++j) cur[j] = nxt[j];
            {   // the next K-block's ids in flight during this one
                const int tok = t0 + (kb + 1) * kMmaKB + tt;
                load_token<KT>(lay + (int64_t)tok * kk, kk, builds && kb + 1 < nkb && tok < t1, vec, nxt);
            }
            // stage s is free once the MMAs of K-block kb - kMmaStages are done
            if (kb >= kMmaStages) {
                bool ok = lane == 0 ? mbar_wait(&empty[s], (uint32_t)((kb - kMmaStages) / kMmaStages) & 1u) : true;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) atomicExch(&timed_out, 1);
                    stop = true;
                    break;
                }
            }
            unsigned char *stage = smc + (size_t)s * kStage;
            if (builds) {
#pragma unroll
                for (int j = 0; j < KB; ++j)
                    if (set[s][j] != 0xffffffffu) stage[set[s][j]] = 0;
                if (t0 + kb * kMmaKB + tt < t1) {
                    if (distinct_ids<KT>(cur, kk)) {
                        // the Top-k case: every id once, count 1
#pragma unroll
                        for (int j = 0; j < KB; ++j) {
                            const int e = cur[j];
                            const bool ok = j < kk && (unsigned)e < (unsigned)E;
                            bad |= j < kk && !ok;                 // dropped and reported
                            const uint32_t off = colb + (uint32_t)e * 128u + ((uint32_t)((cb ^ e) & 7) << 4);
                            if (ok) stage[off] = kE4m3One;
                            set[s][j] = ok ? off : 0xffffffffu;
                        }
                    } else {
                        // a repeated id: its count, written once, at its first slot
#pragma unroll
                        for (int j = 0; j < KB; ++j) {
                            set[s][j] = 0xffffffffu;
                            if (j >= kk) continue;
                            const int e = cur[j];
                            if ((unsigned)e >= (unsigned)E) {
                                bad = true;
                                continue;
                            }
                            int cnt = 0;
                            bool first = true;
#pragma unroll
                            for (int i = 0; i < KB; ++i)
                                if (i < kk && cur[i] == e) {
                                    ++cnt;
                                    if (i < j) first = false;
                                }
                            if (!first) continue;
                            const uint32_t off = colb + (uint32_t)e * 128u + ((uint32_t)((cb ^ e) & 7) << 4);
                            stage[off] = (uint8_t)__nv_cvt_float_to_fp8((float)cnt, __NV_SATFINITE, __NV_E4M3);
                            set[s][j] = off;
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < KB; ++j) set[s][j] = 0xffffffffu;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[s]);
        }
    } else if (lane == 0) {
        // -------------------------------------------------------------- issuer
        const uint32_t idesc = idesc_f8(has_tr ? 2 * kMmaRows : kMmaRows);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % kMmaStages;
            if (!mbar_wait(&full[s], (uint32_t)(kb / kMmaStages) & 1u)) {
                atomicExch(&timed_out, 1);
                break;
            }
            tc_fence_after();
            const uint32_t ua = smem_u32(smc + (size_t)s * kStage);
#pragma unroll
            for (int q = 0; q < kMmaKB / kMmaK; ++q) {
                // a 32-token step: its K-atom, then (q % 4) * 32 bytes into the
                // rows (the hardware applies the swizzle to the start it is given)
                const uint64_t d = smem_desc(ua + (uint32_t)(q >> 2) * 2u * kAtomRows + (uint32_t)(q & 3) * kMmaK);
                mma_f8(tmem, d, d, idesc, (kb > 0 || q > 0) ? 1u : 0u);
            }
            mma_commit(&empty[s]);
        }
        if (nkb > 0) mma_commit(&mbar_done);      // every MMA issued so far
    }
    // every MMA this CTA issued is complete once mbar_done arrives
    bool done = true;
    __syncthreads();
    if (nkb > 0) done = mbar_wait(&mbar_done, 0);
    const bool fail = __syncthreads_or(!done || timed_out);
    tc_fence_after();
    if (!fail && warp < 4) {
        const int row = warp * 32 + lane;
        for (int m = 0; m < 2; ++m) {
            int32_t *dst = pu + ((int64_t)m * kMmaRows + row) * kMmaRows;
            if (m == 1 && !has_tr) break;
            for (int cb2 = 0; cb2 < kMmaRows; cb2 += 32) {
                uint32_t v[32];
                if (nkb > 0) {
                    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(m * kMmaRows + cb2), v);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0u;     // float +0
                }
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    int4 q;
                    q.x = (int)__uint_as_float(v[i]);
                    q.y = (int)__uint_as_float(v[i + 1]);
                    q.z = (int)__uint_as_float(v[i + 2]);
                    q.w = (int)__uint_as_float(v[i + 3]);
                    *reinterpret_cast<int4 *>(dst + cb2 + i) = q;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    if (tid == 0 && fail) set_error(hdr, TOPO_ETIMEOUT);
    if (bad) set_error(hdr, TOPO_ERANGE);
}

// co[l][a][b] (and tr) = sum of the layer's unit partials, as int64.
__global__ void __launch_bounds__(256)
k_cooc_reduce(const int32_t *__restrict__ part, int64_t *co, int64_t *tr, int L, int E, int nchunks) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nco = (int64_t)L * E * E;
    const int64_t ntr = tr ? (int64_t)(L - 1) * E * E : 0;
    if (i >= nco + ntr) return;
    const int m = i < nco ? 0 : 1;
    const int64_t j = m ? i - nco : i;
    const int l = (int)(j / ((int64_t)E * E));
    const int ab = (int)(j - (int64_t)l * E * E);
    const int a = ab / E, b = ab - a * E;
    const int32_t *p = part + ((int64_t)l * nchunks * 2 + m) * kMmaRows * kMmaRows + a * kMmaRows + b;
    int64_t s = 0;
    for (int c = 0; c < nchunks; ++c) s += __ldg(p + (int64_t)c * 2 * kMmaRows * kMmaRows);
    (m ? tr : co)[j] = s;
}

}  // namespace

// Units: about one per SM of a 152-SM part over all layers, each at most
// kMaxCoocTokens tokens in whole K-blocks.
void cooccur_mma_units(int L, int T, int *nchunks, int *chunk) {
    const int kb = (T + kMmaKB - 1) / kMmaKB;
    int n = (kCoocUnitsTarget + L - 1) / (L > 0 ? L : 1);
    if (n < 1) n = 1;
    if (n > kb) n = kb > 0 ? kb : 1;
    const int min_n = (T + kMaxCoocTokens - 1) / kMaxCoocTokens;
    if (n < min_n) n = min_n;
    int per = (kb + n - 1) / n;
    if (per < 1) per = 1;
    *chunk = per * kMmaKB;
    *nchunks = T > 0 ? (T + *chunk - 1) / *chunk : 1;
}

size_t cooccur_mma_ws_bytes(int L, int T, int E, int k) {
    if (!cooccur_mma_applies(L, T, E, k)) return sizeof(WsHeader);
    int nchunks, chunk;
    cooccur_mma_units(L, T, &nchunks, &chunk);
    return sizeof(WsHeader) + (size_t)L * nchunks * 2 * kMmaRows * kMmaRows * 4;
}

bool cooccur_mma_applies(int L, int T, int E, int k) {
    return L > 0 && T > 0 && E <= kMmaRows && k <= kMaxKIds && (int64_t)L * (T + kMmaKB - 1) / kMmaKB < INT32_MAX;
}

template <int KT>
cudaError_t run_cooccur_mma(int units, int L, int T, int E, int k, const int32_t *ids, int32_t *part,
                            WsHeader *hdr, int nchunks, int chunk, bool want_tr, cudaStream_t st) {
    const size_t smem = (size_t)kMmaStages * kStage;
    cudaError_t e = ensure_smem((const void *)k_cooccur_mma<KT>, smem);
    if (e != cudaSuccess) return e;
    const int vec = ((uintptr_t)ids & 15) == 0 && k % 4 == 0;
    k_cooccur_mma<KT><<<units, kMmaThreads + 32, smem, st>>>(ids, part, hdr, L, T, E, k, nchunks, chunk, want_tr,
                                                             vec);
    return cudaGetLastError();
}

cudaError_t launch_cooccur_mma(int L, int T, int E, int k, const int32_t *ids, int64_t *co, int64_t *tr,
                               void *ws, cudaStream_t st) {
    int nchunks, chunk;
    cooccur_mma_units(L, T, &nchunks, &chunk);
    int32_t *part = ws_at<int32_t>(ws, sizeof(WsHeader));
    WsHeader *hdr = ws_at<WsHeader>(ws, 0);
    const int units = L * nchunks;
    const bool want_tr = tr != nullptr;
    cudaError_t e;
    switch (k) {
        case 2: e = run_cooccur_mma<2>(units, L, T, E, k, ids, part, hdr, nchunks, chunk, want_tr, st); break;
        case 4: e = run_cooccur_mma<4>(units, L, T, E, k, ids, part, hdr, nchunks, chunk, want_tr, st); break;
        case 6: e = run_cooccur_mma<6>(units, L, T, E, k, ids, part, hdr, nchunks, chunk, want_tr, st); break;
        case 8: e = run_cooccur_mma<8>(units, L, T, E, k, ids, part, hdr, nchunks, chunk, want_tr, st); break;
        case 10: e = run_cooccur_mma<10>(units, L, T, E, k, ids, part, hdr, nchunks, chunk, want_tr, st); break;
        default: e = run_cooccur_mma<0>(units, L, T, E, k, ids, part, hdr, nchunks, chunk, want_tr, st); break;
    }
    if (e != cudaSuccess) return e;
    const int64_t n = (int64_t)L * E * E + (tr ? (int64_t)(L - 1) * E * E : 0);
    k_cooc_reduce<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(part, co, tr, L, E, nchunks);
    return cudaGetLastError();
}

}  // namespace topo
