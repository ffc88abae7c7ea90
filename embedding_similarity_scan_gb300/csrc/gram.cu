// gram.cu — the Gram engine of the max-min diversity path.
//
// The method ("Issue 9-014: Tile Diversity Shader Inner Loop For L2 Cache
// Locality", Current Behavior): every iteration, each sequence folds the
// cosine distance of its newest pick p to every candidate c into its running
// minimum and takes the unmasked candidate with the largest running minimum
// (lowest index on ties).  The newest pick is itself a table row, so every
// distance the run needs is an entry of the table's Gram matrix: d(p, c) =
// 1 - G[p][c] with G = E E^T of the unit rows.  When the sequences make many
// more picks than the table has rows (B * L >> N), computing G once on the
// tensor cores (the BMU kernel's pipeline with a store epilogue, see
// tc_bmu.cu) and then streaming one row of G per sequence and iteration moves
// far less work than the per-iteration contraction: the iterations become a
// pure HBM/L2 stream, and the sequences are independent of one another, so
// the walk needs no grid-wide synchronisation at all.
//
// gram_walk_kernel: one CTA per sequence, all L iterations.  Per iteration
// the CTA streams G[p][0 .. N) (16-byte loads, several in flight per thread),
// folds d = 1 - g into the running minimum (kept in shared memory when a row
// of it fits, else in global memory), and reduces (max, lowest index) over
// the block: per thread in ascending column order with a strict '>', then
// warp shuffles and one shared-memory stage with the index as tie-break.
// The winner is masked by the thread that owns its column in the next
// iteration's fold, so the only block-wide barriers are the two of the
// reduction.
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

// (value, index) max with the lower index on equal values
__device__ __forceinline__ void take_better(float &v, int &c, float ov, int oc) {
    if (ov > v || (ov == v && oc < c)) {
        v = ov;
        c = oc;
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

// kSmem: the sequence's running minima live in shared memory for the whole
// walk (loaded from and stored back to a.m around it); otherwise they are
// read and written in global memory every iteration.
// kBatch: 16-byte vectors of the G row each thread has in flight at once;
// the host picks it so that one batch covers a whole row where it can (one
// round trip to memory per iteration).
// The block argmax takes one barrier per iteration: every warp publishes its
// (max, lowest index) in one of two alternating slots, and after the barrier
// every warp reduces all slots itself, so all threads know the winner
// without a second barrier (a warp cannot reach the slots of iteration t + 2
// before every warp has passed the barrier of iteration t + 1).
template <bool kSmem, int kThreads, int kBatch, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks) gram_walk_kernel(GramWalkArgs a) {
    constexpr int kWarps = kThreads / 32;
    static_assert(kWarps <= 32, "one warp reduces the per-warp slots");
    extern __shared__ float4 s_m4[];
    __shared__ float red_v[2][kWarps];
    __shared__ int red_c[2][kWarps];
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = (int)(a.Np / 4);
    float4 *m_g = reinterpret_cast<float4 *>(a.m + (int64_t)b * a.Np);
    int p;
    if (kSmem && a.starts) {
        // a fresh run: the running minima start here (+inf, -inf for masked
        // rows, the start and the row padding)
        p = a.starts[b];
        for (int v = threadIdx.x; v < nv; v += kThreads) {
            float m4[4];
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const int64_t c = 4 * (int64_t)v + z;
                m4[z] = (c < a.N && c != p && !(a.mask && a.mask[c])) ? INFINITY : -INFINITY;
            }
            s_m4[v] = make_float4(m4[0], m4[1], m4[2], m4[3]);
        }
        __syncthreads();
    } else {
        if (kSmem) {
            for (int v = threadIdx.x; v < nv; v += kThreads) s_m4[v] = ld_cg_v4(m_g + v);
            __syncthreads();
        }
        p = a.cur[b];
    }
    const int slot = a.trace_slot ? a.trace_slot[b] : -1;
    int pending = -1;  // the last pick, masked in the next fold
    for (int t = 0; t < a.L; ++t) {
        const float4 *g4 = reinterpret_cast<const float4 *>(a.G + (int64_t)p * a.Np);
        float best = -INFINITY;
        int best_c = INT_MAX;
        const int pv = pending >> 2;
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
                if (kSmem) mv[u] = s_m4[v];
                float m4[4] = {mv[u].x, mv[u].y, mv[u].z, mv[u].w};
                const float g[4] = {gv[u].x, gv[u].y, gv[u].z, gv[u].w};
                bool changed = false;
                if (v == pv) {
                    m4[pending & 3] = -INFINITY;
                    changed = true;
                }
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    const float d = fmaf(g[z], -1.0f, 1.0f);
                    const float nm = fminf(m4[z], d);
                    changed |= nm != m4[z];
                    m4[z] = nm;
                    if (nm > best) {
                        best = nm;
                        best_c = 4 * v + z;
                    }
                }
                if (changed) {
                    const float4 w = make_float4(m4[0], m4[1], m4[2], m4[3]);
                    if (kSmem)
                        s_m4[v] = w;
                    else
                        m_g[v] = w;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            take_better(best, best_c, __shfl_xor_sync(0xffffffffu, best, o),
                        __shfl_xor_sync(0xffffffffu, best_c, o));
        const int par = t & 1;
        if (lane == 0) {
            red_v[par][warp] = best;
            red_c[par][warp] = best_c;
        }
        __syncthreads();
        best = lane < kWarps ? red_v[par][lane] : -INFINITY;
        best_c = lane < kWarps ? red_c[par][lane] : INT_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            take_better(best, best_c, __shfl_xor_sync(0xffffffffu, best, o),
                        __shfl_xor_sync(0xffffffffu, best_c, o));
        const int w = best_c == INT_MAX ? -1 : best_c;
        if (threadIdx.x == 0) {
            a.picks[(int64_t)b * a.L + t] = w;
            if (w < 0) atomicOr(a.status, kStatusNoWinner);
        }
        if (slot >= 0) {
            // the running minima after this fold, before the pick is masked
            float *dst = a.trace + ((int64_t)slot * a.L + t) * a.N;
            const float *src = kSmem ? reinterpret_cast<const float *>(s_m4) : a.m + (int64_t)b * a.Np;
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

// The walk for tables whose running-minimum row does not fit one CTA's
// shared memory: a cluster of kC CTAs walks one sequence, each CTA holding a
// contiguous kC-th of the row of running minima in its shared memory and
// streaming the same part of each row G[p][.].  Per iteration each CTA
// reduces its part to one (max, lowest column) candidate, writes it into a
// slot of every CTA of the cluster (distributed shared memory), and after
// one cluster barrier every CTA reduces the kC candidates to the same
// winner.  The slots alternate between iterations, so one cluster barrier
// per iteration suffices (no CTA can reach the slots of iteration t + 2
// before all have passed the barrier of t + 1).  Only G is streamed: the
// running minima never leave the cluster's shared memory during the walk.
template <int kC, int kThreads, int kBatch, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks) gram_walk_cluster_kernel(GramWalkArgs a) {
    constexpr int kWarps = kThreads / 32;
    extern __shared__ float4 s_m4[];
    __shared__ float red_v[kWarps];
    __shared__ int red_c[kWarps];
    __shared__ float slot_v[2][kC];
    __shared__ int slot_c[2][kC];
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
    int p;
    if (a.starts) {
        // a fresh run: the running minima start here
        p = a.starts[b];
        for (int v = threadIdx.x; v < my_v; v += kThreads) {
            float m4[4];
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const int64_t c = 4 * (int64_t)(v0 + v) + z;
                m4[z] = (c < a.N && c != p && !(a.mask && a.mask[c])) ? INFINITY : -INFINITY;
            }
            s_m4[v] = make_float4(m4[0], m4[1], m4[2], m4[3]);
        }
    } else {
        for (int v = threadIdx.x; v < my_v; v += kThreads) s_m4[v] = ld_cg_v4(m_g + v0 + v);
        p = a.cur[b];
    }
    // every CTA's shared memory set up before any remote write
    cluster_sync_all();
    const int slot = a.trace_slot ? a.trace_slot[b] : -1;
    int pending = -1;
    for (int t = 0; t < a.L; ++t) {
        const float4 *g4 = reinterpret_cast<const float4 *>(a.G + (int64_t)p * a.Np) + v0;
        float best = -INFINITY;
        int best_c = INT_MAX;
        const int pv = pending >= 0 ? (pending >> 2) - v0 : -1;
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
                const float4 mv = s_m4[v];
                float m4[4] = {mv.x, mv.y, mv.z, mv.w};
                const float g[4] = {gv[u].x, gv[u].y, gv[u].z, gv[u].w};
                bool changed = false;
                if (v == pv) {
                    m4[pending & 3] = -INFINITY;
                    changed = true;
                }
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    const float d = fmaf(g[z], -1.0f, 1.0f);
                    const float nm = fminf(m4[z], d);
                    changed |= nm != m4[z];
                    m4[z] = nm;
                    if (nm > best) {
                        best = nm;
                        best_c = 4 * (v0 + v) + z;
                    }
                }
                if (changed) s_m4[v] = make_float4(m4[0], m4[1], m4[2], m4[3]);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            take_better(best, best_c, __shfl_xor_sync(0xffffffffu, best, o),
                        __shfl_xor_sync(0xffffffffu, best_c, o));
        if (lane == 0) {
            red_v[warp] = best;
            red_c[warp] = best_c;
        }
        __syncthreads();
        const int par = t & 1;
        if (threadIdx.x < 32) {
            best = lane < kWarps ? red_v[lane] : -INFINITY;
            best_c = lane < kWarps ? red_c[lane] : INT_MAX;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                take_better(best, best_c, __shfl_xor_sync(0xffffffffu, best, o),
                            __shfl_xor_sync(0xffffffffu, best_c, o));
            // this CTA's candidate into slot [par][rank] of every CTA (lane r
            // writes CTA r's copy)
            if (lane < kC) {
                const uint32_t av = mapa_shared(smem_u32(&slot_v[par][rank]), (uint32_t)lane);
                const uint32_t ac = mapa_shared(smem_u32(&slot_c[par][rank]), (uint32_t)lane);
                asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(av), "f"(best) : "memory");
                asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(ac), "r"(best_c) : "memory");
            }
        }
        cluster_sync_all();
        best = -INFINITY;
        best_c = INT_MAX;
#pragma unroll
        for (int r = 0; r < kC; ++r) take_better(best, best_c, slot_v[par][r], slot_c[par][r]);
        const int w = best_c == INT_MAX ? -1 : best_c;
        if (rank == 0 && threadIdx.x == 0) {
            a.picks[(int64_t)b * a.L + t] = w;
            if (w < 0) atomicOr(a.status, kStatusNoWinner);
        }
        if (slot >= 0) {
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
    // no CTA leaves while another may still write into its slots
    cluster_sync_all();
}

}  // namespace

void launch_gram_walk_init(const GramWalkArgs &a, const int32_t *starts, const uint8_t *mask,
                           cudaStream_t st) {
    gram_walk_init_kernel<<<2048, 256, 0, st>>>(a, starts, mask);
}

static size_t gram_walk_smem_bytes(int64_t Np) { return (size_t)Np * sizeof(float); }

template <bool kSmem, int kThreads, int kBatch, int kMinBlocks>
cudaError_t launch_walk_variant(const GramWalkArgs &a, size_t smem, cudaStream_t st) {
    auto kernel = gram_walk_kernel<kSmem, kThreads, kBatch, kMinBlocks>;
    if (smem > 48 * 1024) {
        cudaError_t err =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    kernel<<<(unsigned)a.B, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int kC, int kThreads, int kBatch, int kMinBlocks>
cudaError_t launch_cluster_variant(const GramWalkArgs &a, cudaStream_t st) {
    const int64_t nv = a.Np / 4;
    const size_t smem = (size_t)((nv + kC - 1) / kC) * sizeof(float4);
    auto kernel = gram_walk_cluster_kernel<kC, kThreads, kBatch, kMinBlocks>;
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

int gram_walk_place(int64_t Np) {
    const size_t row = (size_t)Np * sizeof(float);
    return row <= kGramWalkSmemMax ? 1 : row <= kGramWalkClusterMax ? 2 : 3;
}

cudaError_t launch_gram_walk(const GramWalkArgs &a, cudaStream_t st) {
    const size_t smem = gram_walk_smem_bytes(a.Np);
    const int64_t nv = a.Np / 4;  // 16-byte vectors per row
    // rows of running minima spread over a cluster of 8 CTAs
    if (a.place == 2) return launch_cluster_variant<8, 256, 16, 2>(a, st);
    if (a.place == 3) return launch_walk_variant<false, 256, 6, 3>(a, 0, st);
    // one batch per row: as few threads as cover the row with at most 17
    // vectors each, so that more CTAs (sequences) fit an SM
    if (nv <= 4 * 128) return launch_walk_variant<true, 128, 4, 8>(a, smem, st);
    if (nv <= 9 * 128) return launch_walk_variant<true, 128, 9, 6>(a, smem, st);
    if (nv <= 17 * 128) return launch_walk_variant<true, 128, 17, 5>(a, smem, st);
    if (nv <= 9 * 256) return launch_walk_variant<true, 256, 9, 4>(a, smem, st);
    return launch_walk_variant<true, 256, 12, 3>(a, smem, st);
}

}  // namespace dseq
