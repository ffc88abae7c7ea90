// gram.cu — the Gram engine of the max-min diversity path.
//
// The method ("Issue 9-014: Tile Diversity Shader Inner Loop For L2 Cache
// Locality", Current Behavior): every iteration, each sequence folds the
// cosine distance of its newest pick p to every candidate c into its running
// minimum and takes the unmasked candidate with the largest running minimum
// (lowest index on ties).  The newest pick is itself a table row, so every
// distance the run needs is an entry of the table's Gram matrix: d(p, c) =
// 1 - G[p][c] with G = E E^T of the unit rows.  The product stores these
// distances (the matrix 1 - G, rounded once from the fp32 G entry, exactly
// as the fold would compute it), so the fold is one min per candidate.  When the sequences make many
// more picks than the table has rows (B * L >> N), computing G once on the
// tensor cores (the BMU kernel's pipeline with a store epilogue, see
// tc_bmu.cu) and then streaming one row of G per sequence and iteration moves
// far less work than the per-iteration contraction: the iterations become a
// pure HBM/L2 stream, and the sequences are independent of one another, so
// the walk needs no grid-wide synchronisation at all.
//
// gram_walk_kernel: one CTA per sequence, all L iterations.  Per iteration
// the CTA streams the distance row of its newest pick (16-byte loads, one
// batch in flight per thread), folds it into the running minimum (kept in
// shared memory when a row of it fits, else in global memory; only vectors
// whose minima fell are written back), and reduces (max, lowest
// index) over the block: per thread in ascending column order, then two
// redux instructions per warp and one shared-memory stage.  The winner is
// masked by the thread that owns its column in the next iteration's fold, so
// the reduction's one barrier is the only block-wide barrier per iteration.
// gram_walk_cluster_kernel: the same walk for rows of running minima longer
// than one CTA's shared memory, spread over a cluster of CTAs.
#include <climits>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dseq {

namespace {


__device__ __forceinline__ float4 ld_nc_v4(const float4 *p) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ float4 ld_cg_v4(const float4 *p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// A running minimum and a candidate are ranked by an ordered 32-bit key of
// the value (the float's bits mapped so that unsigned order is float order,
// -inf lowest) and then by the lower column: every reduction is a max of the
// key followed by a min of the column among the lanes that hold that max,
// two warp-wide redux instructions.  A thread or CTA without a candidate
// holds (-inf, INT_MAX), which never wins; INT_MAX as the winner means that
// every candidate is masked.
__device__ __forceinline__ uint32_t ord_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ void warp_argmax(uint32_t &key, uint32_t &col) {
    const uint32_t mx = __reduce_max_sync(0xffffffffu, key);
    col = __reduce_min_sync(0xffffffffu, key == mx ? col : 0xffffffffu);
    key = mx;
}

// The fold of one 16-byte vector (four candidates) of the distance row
// d(p, .) into the running minima: m <- min(m, d).
__device__ __forceinline__ float4 fold4(float4 m, float4 d) {
    return make_float4(fminf(m.x, d.x), fminf(m.y, d.y), fminf(m.z, d.z), fminf(m.w, d.w));
}
// The thread's running (max, column) over the vectors it folds, in
// ascending column order: a vector's max is compared once, and only when it
// beats the best so far is its lowest column holding that max looked up.
__device__ __forceinline__ void track4(float4 nm, int c0, float &best, int &best_c) {
    const float mx = fmaxf(fmaxf(nm.x, nm.y), fmaxf(nm.z, nm.w));
    if (mx > best) {
        best = mx;
        best_c = c0 + (nm.x == mx ? 0 : nm.y == mx ? 1 : nm.z == mx ? 2 : 3);
    }
}

__global__ void gram_walk_init_kernel(GramWalkArgs a, const int32_t *__restrict__ starts,
                                      const uint8_t *__restrict__ mask) {
    const int64_t total = (int64_t)a.B * a.Np;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int b = (int)(i / a.Np);
        const int64_t c = i - (int64_t)b * a.Np;
        const bool live = c < a.N && c != starts[b] && !(mask && mask[c]);
        a.m[i] = live ? INFINITY : -INFINITY;
    }
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < a.B; b += stride)
        a.cur[b] = starts[b];
}

// Running minima of columns [4 v0, 4 v1) at the start of a fresh run: +inf,
// -inf for masked rows, the start and the row padding.
__device__ __forceinline__ void init_minima(float4 *s_m4, int v0, int v1, int64_t N, int p,
                                            const uint8_t *mask, int kThreads) {
    for (int v = v0 + (int)threadIdx.x; v < v1; v += kThreads) {
        float m4[4];
#pragma unroll
        for (int z = 0; z < 4; ++z) {
            const int64_t c = 4 * (int64_t)v + z;
            m4[z] = (c < N && c != p && !(mask && mask[c])) ? INFINITY : -INFINITY;
        }
        s_m4[v - v0] = make_float4(m4[0], m4[1], m4[2], m4[3]);
    }
}

// kSmem: the sequence's running minima live in shared memory for the whole
// walk (loaded from and stored back to a.m around it); otherwise they are
// read in global memory every iteration and written back where they fell.
// kBatch: 16-byte vectors of the G row each thread has in flight at once;
// the host picks it so that one batch covers a whole row where it can (one
// round trip to memory per iteration).
// The block argmax takes one barrier per iteration: every warp publishes its
// (key, column) in one of two alternating slots, and after the barrier every
// warp reduces all slots itself, so all threads know the winner without a
// second barrier (a warp cannot reach the slots of iteration t + 2 before
// every warp has passed the barrier of iteration t + 1).
template <bool kSmem, int kThreads, int kBatch, int kMinBlocks, bool kTrace>
__global__ void __launch_bounds__(kThreads, kMinBlocks) gram_walk_kernel(GramWalkArgs a) {
    constexpr int kWarps = kThreads / 32;
    static_assert(kThreads % 32 == 0, "whole warps: the reductions use every lane");
    static_assert(kWarps <= 32, "one warp reduces the per-warp slots");
    extern __shared__ float4 s_m4[];
    __shared__ uint32_t red_k[2][kWarps];
    __shared__ uint32_t red_c[2][kWarps];
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = (int)(a.Np / 4);
    float4 *m_g = reinterpret_cast<float4 *>(a.m + (int64_t)b * a.Np);
    int p;
    if (kSmem && a.starts) {
        p = a.starts[b];
        init_minima(s_m4, 0, nv, a.N, p, a.mask, kThreads);
        __syncthreads();
    } else {
        if (kSmem) {
            for (int v = threadIdx.x; v < nv; v += kThreads) s_m4[v] = ld_cg_v4(m_g + v);
            __syncthreads();
        }
        p = a.cur[b];
    }
    const int slot = kTrace ? a.trace_slot[b] : -1;
    int pending = -1;  // the last pick, masked in the next fold
    for (int t = 0; t < a.L; ++t) {
        const float4 *g4 = reinterpret_cast<const float4 *>(a.G + (int64_t)p * a.Np);
        float best = -INFINITY;
        int best_c = INT_MAX;
        // the last pick is masked by the thread whose vectors hold it, before
        // that thread folds them (no other thread reads that vector)
        if (pending >= 0 && (pending >> 2) % kThreads == (int)threadIdx.x) {
            if (kSmem)
                reinterpret_cast<float *>(s_m4)[pending] = -INFINITY;
            else
                a.m[(int64_t)b * a.Np + pending] = -INFINITY;
        }
        for (int v0 = threadIdx.x; v0 < nv; v0 += kBatch * kThreads) {
            float4 gv[kBatch], mv[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int v = v0 + u * kThreads;
                gv[u] = v < nv ? ld_nc_v4(g4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                if (!kSmem)
                    mv[u] = v < nv ? ld_cg_v4(m_g + v)
                                   : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int v = v0 + u * kThreads;
                if (v >= nv) break;
                const float4 m0 = kSmem ? s_m4[v] : mv[u];
                const float4 nm = fold4(m0, gv[u]);
                // only vectors whose minima fell are written back: each
                // vector otherwise passes through L1 three times (the load of
                // G, the read and the write of m), and L1 ran 80 % busy
                // (page-1 walk 3.135 -> 3.089 ms; in the cluster walk, whose
                // iterations wait on DRAM, the test cost more than it saved)
                if (nm.x != m0.x || nm.y != m0.y || nm.z != m0.z || nm.w != m0.w) {
                    if (kSmem)
                        s_m4[v] = nm;
                    else
                        m_g[v] = nm;
                }
                track4(nm, 4 * v, best, best_c);
            }
        }
        uint32_t key = ord_key(best), col = (uint32_t)best_c;
        warp_argmax(key, col);
        const int par = t & 1;
        if (lane == 0) {
            red_k[par][warp] = key;
            red_c[par][warp] = col;
        }
        __syncthreads();
        key = lane < kWarps ? red_k[par][lane] : 0u;
        col = lane < kWarps ? red_c[par][lane] : 0xffffffffu;
        warp_argmax(key, col);
        const int w = col == (uint32_t)INT_MAX ? -1 : (int)col;
        if (threadIdx.x == 0) {
            a.picks[(int64_t)b * a.L + t] = w;
            if (w < 0) atomicOr(a.status, kStatusNoWinner);
        }
        if (kTrace && slot >= 0) {
            // the running minima after this fold, before the pick is masked
            float *dst = a.trace + ((int64_t)slot * a.L + t) * a.N;
            const float *src = kSmem ? reinterpret_cast<const float *>(s_m4) : a.m + (int64_t)b * a.Np;
            if (!kSmem) __syncthreads();  // every thread's global stores of this fold made
            for (int64_t c = threadIdx.x; c < a.N; c += kThreads) dst[c] = src[c];
            __syncthreads();  // every copy read the pre-mask values
        }
        if (w < 0) break;
        pending = w;
        p = w;
    }
    // the state left for a resumed run: the last pick masked, minima in a.m
    __syncthreads();
    if (threadIdx.x == 0 && pending >= 0) {
        if (kSmem)
            reinterpret_cast<float *>(s_m4)[pending] = -INFINITY;
        else
            a.m[(int64_t)b * a.Np + pending] = -INFINITY;
        a.cur[b] = p;
    }
    __syncthreads();
    if (kSmem)
        for (int v = threadIdx.x; v < nv; v += kThreads) m_g[v] = s_m4[v];
}

// The walk with the running minima in registers: thread i holds vectors i,
// i + kThreads, ... of the sequence's row of minima (kBatch of them), so a
// fold reads and writes no memory but the distance row itself.  Shared
// memory would pass every vector through L1 two more times (the read and
// the write of its minima), and the walk is bound by L1 there: page-1 walk
// 3.09 ms with the minima in shared memory (192 threads x 11 vectors, 5
// CTAs per SM), 2.54 ms in registers (128 x 17, 3 CTAs per SM at 167
// registers).  One batch covers the row (nv <= kBatch * kThreads).
template <int kThreads, int kBatch, int kMinBlocks, bool kTrace>
__global__ void __launch_bounds__(kThreads, kMinBlocks) gram_walk_kernel_regs(GramWalkArgs a) {
    constexpr int kWarps = kThreads / 32;
    static_assert(kThreads % 32 == 0, "whole warps: the reductions use every lane");
    static_assert(kWarps <= 32, "one warp reduces the per-warp slots");
    __shared__ uint32_t red_k[2][kWarps];
    __shared__ uint32_t red_c[2][kWarps];
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = (int)(a.Np / 4);
    float4 *m_g = reinterpret_cast<float4 *>(a.m + (int64_t)b * a.Np);
    float4 mr[kBatch];
    int p;
    if (a.starts) {
        p = a.starts[b];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = threadIdx.x + u * kThreads;
            float m4[4];
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const int64_t c = 4 * (int64_t)v + z;
                m4[z] = (v < nv && c < a.N && c != p && !(a.mask && a.mask[c])) ? INFINITY : -INFINITY;
            }
            mr[u] = make_float4(m4[0], m4[1], m4[2], m4[3]);
        }
    } else {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = threadIdx.x + u * kThreads;
            mr[u] = v < nv ? ld_cg_v4(m_g + v) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
        p = a.cur[b];
    }
    const int slot = kTrace ? a.trace_slot[b] : -1;
    int pending = -1;  // the last pick, masked before the next fold
    for (int t = 0; t < a.L; ++t) {
        const float4 *g4 = reinterpret_cast<const float4 *>(a.G + (int64_t)p * a.Np);
        float4 gv[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = threadIdx.x + u * kThreads;
            gv[u] = v < nv ? ld_nc_v4(g4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // the last pick is masked by the thread that holds it
        if (pending >= 0 && (pending >> 2) % kThreads == (int)threadIdx.x) {
            const int up = (pending >> 2) / kThreads, z = pending & 3;
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (u == up) {
                    if (z == 0) mr[u].x = -INFINITY;
                    else if (z == 1) mr[u].y = -INFINITY;
                    else if (z == 2) mr[u].z = -INFINITY;
                    else mr[u].w = -INFINITY;
                }
        }
        float best = -INFINITY;
        int best_c = INT_MAX;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            mr[u] = fold4(mr[u], gv[u]);
            track4(mr[u], 4 * ((int)threadIdx.x + u * kThreads), best, best_c);
        }
        uint32_t key = ord_key(best), col = (uint32_t)best_c;
        warp_argmax(key, col);
        const int par = t & 1;
        if (lane == 0) {
            red_k[par][warp] = key;
            red_c[par][warp] = col;
        }
        __syncthreads();
        key = lane < kWarps ? red_k[par][lane] : 0u;
        col = lane < kWarps ? red_c[par][lane] : 0xffffffffu;
        warp_argmax(key, col);
        const int w = col == (uint32_t)INT_MAX ? -1 : (int)col;
        if (threadIdx.x == 0) {
            a.picks[(int64_t)b * a.L + t] = w;
            if (w < 0) atomicOr(a.status, kStatusNoWinner);
        }
        if (kTrace && slot >= 0) {
            // the running minima after this fold, before the pick is masked
            float *dst = a.trace + ((int64_t)slot * a.L + t) * a.N;
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t c0 = 4 * (int64_t)((int)threadIdx.x + u * kThreads);
                const float m4[4] = {mr[u].x, mr[u].y, mr[u].z, mr[u].w};
#pragma unroll
                for (int z = 0; z < 4; ++z)
                    if (c0 + z < a.N) dst[c0 + z] = m4[z];
            }
        }
        if (w < 0) break;
        pending = w;
        p = w;
    }
    // the state left for a resumed run: the last pick masked, minima in a.m
    if (pending >= 0 && (pending >> 2) % kThreads == (int)threadIdx.x) {
        const int up = (pending >> 2) / kThreads, z = pending & 3;
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (u == up) {
                if (z == 0) mr[u].x = -INFINITY;
                else if (z == 1) mr[u].y = -INFINITY;
                else if (z == 2) mr[u].z = -INFINITY;
                else mr[u].w = -INFINITY;
            }
    }
    if (threadIdx.x == 0 && pending >= 0) a.cur[b] = p;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        const int v = threadIdx.x + u * kThreads;
        if (v < nv) m_g[v] = mr[u];
    }
}

__device__ __forceinline__ void st_async_u64(uint32_t cluster_addr, uint64_t v, uint32_t cluster_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(
                     cluster_addr),
                 "l"(v), "r"(cluster_bar)
                 : "memory");
}

// The walk for tables whose running-minimum row does not fit one CTA's
// shared memory: a cluster of kC CTAs walks one sequence, each CTA holding a
// contiguous kC-th of the row of running minima in its shared memory and
// streaming the same part of each row G[p][.].  Per iteration each CTA
// reduces its part to one (key, column) candidate and sends it, with one
// 8-byte asynchronous store per CTA, into a slot of every CTA of the cluster;
// each store completes bytes on the receiving CTA's mbarrier for that
// iteration, so a CTA waits only until the kC candidates have landed in its
// own shared memory (no cluster-wide barrier, and no release of the CTA's
// global stores, in the loop), then reduces them to the same winner as every
// other CTA.  Slots and mbarriers alternate between iterations: a CTA sends
// the candidate of iteration t + 2 only after it has received all those of
// t + 1, which each CTA sends after it has read the slots of t, so a slot is
// never overwritten before it is read and a phase of an mbarrier always
// completes before the next phase's bytes arrive (bytes may land before the
// receiver's expect_tx of that phase: the transaction count may go negative
// until the arrival).  Only G is streamed: the running minima never leave
// the cluster's shared memory during the walk.
template <int kC, int kThreads, int kBatch, int kMinBlocks, bool kTrace>
__global__ void __launch_bounds__(kThreads, kMinBlocks) gram_walk_cluster_kernel(GramWalkArgs a) {
    constexpr int kWarps = kThreads / 32;
    static_assert(kThreads % 32 == 0, "whole warps: the reductions use every lane");
    static_assert(kC <= 32 && kWarps <= 32, "one warp reduces the candidates");
    extern __shared__ float4 s_m4[];
    __shared__ uint32_t red_k[kWarps];
    __shared__ uint32_t red_c[kWarps];
    __shared__ __align__(8) uint64_t cand[2][kC];
    __shared__ __align__(8) uint64_t bar[2];
    __shared__ int abort_flag;
    const int rank = (int)cluster_ctarank();
    const int b = blockIdx.x / kC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = (int)(a.Np / 4);
    const int wv = (nv + kC - 1) / kC;  // vectors per CTA
    const int v0 = rank * wv, v1 = min(nv, v0 + wv);
    const int my_v = v1 - v0;
    // the launch must be the shape the kernel is written for (it addresses
    // the other CTAs' shared memory): otherwise report and leave uniformly
    if (cluster_nctarank() != (uint32_t)kC || blockDim.x != kThreads || gridDim.x != (unsigned)(a.B * kC)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, kStatusInternal);
        return;
    }
    float4 *m_g = reinterpret_cast<float4 *>(a.m + (int64_t)b * a.Np);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    int p;
    if (a.starts) {
        p = a.starts[b];
        init_minima(s_m4, v0, v1, a.N, p, a.mask, kThreads);
    } else {
        for (int v = threadIdx.x; v < my_v; v += kThreads) s_m4[v] = ld_cg_v4(m_g + v0 + v);
        p = a.cur[b];
    }
    // every CTA's mbarriers set up before any candidate is sent
    cluster_sync_all();
    const int slot = kTrace ? a.trace_slot[b] : -1;
    int pending = -1;
    int t = 0;
    for (; t < a.L; ++t) {
        const int par = t & 1;
        if (threadIdx.x == 0) mbar_arrive_expect_tx(&bar[par], kC * 8);
        const float4 *g4 = reinterpret_cast<const float4 *>(a.G + (int64_t)p * a.Np) + v0;
        float best = -INFINITY;
        int best_c = INT_MAX;
        // the last pick is masked by the thread of the CTA whose vectors
        // hold it, before that thread folds them
        if (pending >= 0 && (pending >> 2) >= v0 && (pending >> 2) < v1 &&
            ((pending >> 2) - v0) % kThreads == (int)threadIdx.x)
            reinterpret_cast<float *>(s_m4)[pending - 4 * v0] = -INFINITY;
        for (int w0 = threadIdx.x; w0 < my_v; w0 += kBatch * kThreads) {
            float4 gv[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int v = w0 + u * kThreads;
                gv[u] = v < my_v ? ld_nc_v4(g4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int v = w0 + u * kThreads;
                if (v >= my_v) break;
                const float4 nm = fold4(s_m4[v], gv[u]);
                s_m4[v] = nm;
                track4(nm, 4 * (v0 + v), best, best_c);
            }
        }
        uint32_t key = ord_key(best), col = (uint32_t)best_c;
        warp_argmax(key, col);
        if (lane == 0) {
            red_k[warp] = key;
            red_c[warp] = col;
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            key = lane < kWarps ? red_k[lane] : 0u;
            col = lane < kWarps ? red_c[lane] : 0xffffffffu;
            warp_argmax(key, col);
            // this CTA's candidate into slot [par][rank] of every CTA (lane r
            // sends CTA r's copy)
            if (lane < kC)
                st_async_u64(mapa_shared(smem_u32(&cand[par][rank]), (uint32_t)lane),
                             ((uint64_t)key << 32) | col,
                             mapa_shared(smem_u32(&bar[par]), (uint32_t)lane));
        }
        // warp 0 waits (bounded) for the kC candidates; the barrier hands
        // them to the other warps and makes a timeout the whole CTA's
        // decision, so that every thread leaves the loop at the same
        // iteration
        bool ok = true;
        if (warp == 0)
            ok = mbar_wait_bounded(&bar[par], (uint32_t)(t >> 1) & 1u, &abort_flag, a.status,
                                   a.timeout_ns, kStatusBarrierTimeout);
        if (__syncthreads_or(!ok)) break;
        {
            const uint64_t k = lane < kC ? cand[par][lane] : 0ull;
            key = (uint32_t)(k >> 32);
            col = lane < kC ? (uint32_t)k : 0xffffffffu;
            warp_argmax(key, col);
        }
        const int w = col == (uint32_t)INT_MAX ? -1 : (int)col;
        if (rank == 0 && threadIdx.x == 0) {
            a.picks[(int64_t)b * a.L + t] = w;
            if (w < 0) atomicOr(a.status, kStatusNoWinner);
        }
        if (kTrace && slot >= 0) {
            // this CTA's part of the running minima after the fold, before the
            // pick is masked
            float *dst = a.trace + ((int64_t)slot * a.L + t) * a.N;
            const float *src = reinterpret_cast<const float *>(s_m4);
            for (int64_t c = threadIdx.x; c < 4 * (int64_t)my_v; c += kThreads)
                if (4 * (int64_t)v0 + c < a.N) dst[4 * (int64_t)v0 + c] = src[c];
            __syncthreads();
        }
        if (w < 0) break;
        pending = w;
        p = w;
    }
    // the state left for a resumed run: the last pick masked, minima in a.m
    __syncthreads();
    if (threadIdx.x == 0 && pending >= 0 && (pending >> 2) >= v0 && (pending >> 2) < v1)
        reinterpret_cast<float *>(s_m4)[pending - 4 * v0] = -INFINITY;
    if (rank == 0 && threadIdx.x == 0) a.cur[b] = p;
    __syncthreads();
    for (int v = threadIdx.x; v < my_v; v += kThreads) m_g[v0 + v] = s_m4[v];
    // no CTA leaves while another may still send into its shared memory.
    // After a timeout, the last candidates sent to a CTA that gave up were
    // sent before their senders' own bounded wait, so they landed long
    // before every CTA of the cluster reaches this barrier.
    cluster_sync_all();
}

}  // namespace

void launch_gram_walk_init(const GramWalkArgs &a, const int32_t *starts, const uint8_t *mask,
                           cudaStream_t st) {
    gram_walk_init_kernel<<<2048, 256, 0, st>>>(a, starts, mask);
}

static size_t gram_walk_smem_bytes(int64_t Np) { return (size_t)Np * sizeof(float); }

// Every walk kernel takes kTrace only where the run keeps a trace: compiled
// into the untraced kernel, the branch that writes it cost the register walk
// 12 % (page 1: 2.85 ms with it, 2.54 without) though it never ran.
template <bool kSmem, int kThreads, int kBatch, int kMinBlocks>
cudaError_t launch_walk_variant(const GramWalkArgs &a, size_t smem, cudaStream_t st) {
    auto kernel = a.trace_slot ? gram_walk_kernel<kSmem, kThreads, kBatch, kMinBlocks, true>
                               : gram_walk_kernel<kSmem, kThreads, kBatch, kMinBlocks, false>;
    // the limit covers dynamic and static shared memory together: a row of
    // exactly 48 KB plus the reduction slots is already above the default
    if (smem > 0) {
        cudaError_t err =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    kernel<<<(unsigned)a.B, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int kThreads, int kBatch, int kMinBlocks>
cudaError_t launch_walk_regs(const GramWalkArgs &a, cudaStream_t st) {
    if (a.trace_slot)
        gram_walk_kernel_regs<kThreads, kBatch, kMinBlocks, true><<<(unsigned)a.B, kThreads, 0, st>>>(a);
    else
        gram_walk_kernel_regs<kThreads, kBatch, kMinBlocks, false><<<(unsigned)a.B, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <int kC, int kThreads, int kBatch, int kMinBlocks>
cudaError_t launch_cluster_variant(const GramWalkArgs &a, cudaStream_t st) {
    const int64_t nv = a.Np / 4;
    const size_t smem = (size_t)((nv + kC - 1) / kC) * sizeof(float4);
    auto kernel = a.trace_slot ? gram_walk_cluster_kernel<kC, kThreads, kBatch, kMinBlocks, true>
                               : gram_walk_cluster_kernel<kC, kThreads, kBatch, kMinBlocks, false>;
    if ((int64_t)a.B * kC > INT_MAX) return cudaErrorInvalidConfiguration;
    cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.B * kC));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// The default place: one CTA per sequence up to 64 KB of running minima,
// the cluster beyond.  Walk times (B = 3584, L = 256, D = 256; one CTA /
// cluster / global memory): N = 16384 10.3 / 11.0 / 10.4 ms, 18432 12.0 /
// 11.9 / 11.3, 20480 16.3 / 12.3 / 13.7, 24576 18.4 / 13.6 / 15.8: past
// 64 KB a one-CTA row no longer lets 3 CTAs share an SM.  A forced one-CTA
// walk (option walk = 1) takes rows up to kGramWalkSmemMax.
constexpr size_t kGramWalkOneCtaDefault = 64 * 1024;

int gram_walk_place(int64_t Np) {
    const size_t row = (size_t)Np * sizeof(float);
    return row <= kGramWalkOneCtaDefault ? 1 : row <= kGramWalkClusterMax ? 2 : 3;
}

cudaError_t launch_gram_walk(const GramWalkArgs &a, cudaStream_t st) {
    const size_t smem = gram_walk_smem_bytes(a.Np);
    const int64_t nv = a.Np / 4;  // 16-byte vectors per row
    // rows of running minima spread over a cluster of 8 CTAs: as many CTAs
    // per SM as the part each CTA holds allows, one batch of loads per part
    if (a.place == 2) {
        const int64_t wv = (nv + 7) / 8;
        if (wv <= 8 * 128) return launch_cluster_variant<8, 128, 8, 6>(a, st);
        if (wv <= 16 * 128) return launch_cluster_variant<8, 128, 16, 4>(a, st);
        return launch_cluster_variant<8, 256, 16, 2>(a, st);
    }
    if (a.place == 3) return launch_walk_variant<false, 256, 6, 3>(a, 0, st);
    // rows of up to 2,176 vectors: the minima in registers, one batch per
    // row (page 1: 128 threads x 17, 3 CTAs per SM); longer rows in shared
    // memory, as many CTAs per SM as shared memory and registers allow
    if (nv <= 4 * 128) return launch_walk_regs<128, 4, 8>(a, st);
    if (nv <= 9 * 128) return launch_walk_regs<128, 9, 5>(a, st);
    if (nv <= 17 * 128) return launch_walk_regs<128, 17, 3>(a, st);
    if (nv <= 9 * 256) return launch_walk_variant<true, 256, 9, 4>(a, smem, st);
    return launch_walk_variant<true, 256, 12, 3>(a, smem, st);
}

}  // namespace dseq
