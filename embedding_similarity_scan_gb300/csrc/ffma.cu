// ffma.cu — the FP32-FFMA variant of both scans: a SIMT contraction on
// 128 x 128 output tiles (8 x 8 per thread, 256 threads, one CTA per SM)
// fed by a four-stage cp.async ring, with the min-fold / argmax (diversity)
// or argmin (BMU) fused into its epilogue, so the similarity block is never
// written out.  One launch per iteration plus a small commit launch; kept as
// the plain fp32 variant of the library and as a cross-check of the
// tensor-core path.
//
// Every output is one fmaf chain over k in ascending order, so the results
// do not depend on the tiling.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dseq {

namespace {

constexpr int kTile = 128;               // outputs per CTA side
constexpr int kBk = 32;                  // k per stage
constexpr int kStages = 4;
constexpr int kRow = kBk + 4;            // shared row stride (floats): per-row float4 reads hit distinct banks
constexpr int kStageFloats = 2 * kTile * kRow;
constexpr int kFfmaThreads = 256;
constexpr size_t kFfmaSmem = (size_t)kStages * kStageFloats * sizeof(float);  // 147,456 B

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int o) {
    return __shfl_xor_sync(0xffffffffu, v, o);
}

// Asynchronous global->shared copies; a copy with live == false reads
// nothing and fills its bytes with zeros.
__device__ __forceinline__ void cp_async16(float *dst, const float *src, bool live) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(live ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(float *dst, const float *src, bool live) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src), "r"(live ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// One operand of the tile: rows row0 .. row0+127 of a row-major matrix
// (rows x K, leading dimension ld floats); rows and columns outside it read
// as zero.  vec: rows start on 16-byte boundaries and K % 4 == 0.
struct TileOperand {
    const float *p;
    int64_t row0, rows, ld;
    int K;
    bool vec;
};

__device__ __forceinline__ void stage_operand(float *dst, const TileOperand &o, int k0, int tid) {
    if (o.vec) {
#pragma unroll
        for (int u = 0; u < kTile * (kBk / 4) / kFfmaThreads; ++u) {
            const int ch = tid + u * kFfmaThreads, r = ch / (kBk / 4), c = ch % (kBk / 4);
            const int64_t row = o.row0 + r;
            const int k = k0 + 4 * c;
            const bool live = row < o.rows && k < o.K;
            cp_async16(dst + r * kRow + 4 * c, live ? o.p + row * o.ld + k : o.p, live);
        }
    } else {
        for (int u = 0; u < kTile * kBk / kFfmaThreads; ++u) {
            const int el = tid + u * kFfmaThreads, r = el / kBk, c = el % kBk;
            const int64_t row = o.row0 + r;
            const int k = k0 + c;
            const bool live = row < o.rows && k < o.K;
            cp_async4(dst + r * kRow + c, live ? o.p + row * o.ld + k : o.p, live);
        }
    }
}

// acc[i][j] = sum_k A[a.row0 + ty + 16 i][k] * B[b.row0 + tx + 16 j][k],
// one fmaf per k in ascending order.  sm: kStages stages of [A | B] tiles.
__device__ __forceinline__ void ffma_tile(float (&acc)[8][8], float *sm, const TileOperand &A,
                                          const TileOperand &B, int tid, int tx, int ty) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
    const int kt_n = (A.K + kBk - 1) / kBk;
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < kt_n) {
            stage_operand(sm + s * kStageFloats, A, s * kBk, tid);
            stage_operand(sm + s * kStageFloats + kTile * kRow, B, s * kBk, tid);
        }
        cp_async_commit();
    }
    for (int kt = 0; kt < kt_n; ++kt) {
        cp_async_wait<kStages - 2>();  // stage kt has landed (this thread's copies)
        __syncthreads();               // ... everyone's; and stage kt-1 is no longer read
        const int nk = kt + kStages - 1;
        if (nk < kt_n) {
            float *dst = sm + (nk % kStages) * kStageFloats;
            stage_operand(dst, A, nk * kBk, tid);
            stage_operand(dst + kTile * kRow, B, nk * kBk, tid);
        }
        cp_async_commit();
        const float *As = sm + (kt % kStages) * kStageFloats, *Bs = As + kTile * kRow;
#pragma unroll
        for (int k4 = 0; k4 < kBk / 4; ++k4) {
            float4 x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = *reinterpret_cast<const float4 *>(As + (ty + 16 * i) * kRow + 4 * k4);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 y = *reinterpret_cast<const float4 *>(Bs + (tx + 16 * j) * kRow + 4 * k4);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc[i][j] = fmaf(x[i].x, y.x, acc[i][j]);
                    acc[i][j] = fmaf(x[i].y, y.y, acc[i][j]);
                    acc[i][j] = fmaf(x[i].z, y.z, acc[i][j]);
                    acc[i][j] = fmaf(x[i].w, y.w, acc[i][j]);
                }
            }
        }
    }
    cp_async_wait<0>();
}

// --------------------------------------------------------------------------
// diversity

__global__ void ffma_dseq_init_kernel(FfmaDseqArgs a, const int32_t *__restrict__ starts,
                                      const uint8_t *__restrict__ mask) {
    const int64_t total = (int64_t)a.Bp * a.Nf;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(i / a.Nf);
        const int64_t c = i - (int64_t)b * a.Nf;
        bool live = b < a.B && c < a.N;
        if (live && mask && mask[c]) live = false;
        if (live && c == starts[b]) live = false;
        a.m[i] = live ? INFINITY : -INFINITY;
    }
    const int64_t qtotal = (int64_t)a.Bp * a.Dp;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < qtotal;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(i / a.Dp);
        const int k = (int)(i - (int64_t)b * a.Dp);
        a.q[i] = b < a.B ? a.e_unit[(int64_t)starts[b] * a.Dp + k] : 0.0f;
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.Bp;
         i += (int64_t)gridDim.x * blockDim.x)
        a.keys[i] = 0ull;
}

// S = Q * E^T on a 128 x 128 tile, then d = 1 - S (unit rows), m = min(m, d)
// (stored only where it decreased), and the per-row (max m, lowest index)
// folded into keys[b] by atomicMax.  Masked and padding columns hold -inf.
__global__ void __launch_bounds__(kFfmaThreads, 1) ffma_dseq_fold_kernel(FfmaDseqArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int64_t b0 = (int64_t)blockIdx.y * kTile, c0 = (int64_t)blockIdx.x * kTile;
    const TileOperand A{a.q, b0, (int64_t)a.Bp, (int64_t)a.Dp, a.Dp, true};
    const TileOperand B{a.e_unit, c0, a.N, (int64_t)a.Dp, a.Dp, true};
    float acc[8][8];
    ffma_tile(acc, sm, A, B, tid, tx, ty);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t b = b0 + ty + 16 * i;
        float *mrow = a.m + b * a.Nf + c0;
        float best = -INFINITY;
        uint32_t best_c = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = tx + 16 * j;
            const float d = 1.0f - acc[i][j];
            float mv = mrow[c];
            if (d < mv) {
                mv = d;
                mrow[c] = d;
            }
            if (mv > best) {
                best = mv;
                best_c = (uint32_t)(c0 + c);
            }
        }
        unsigned long long key = best > -INFINITY ? max_key(best, best_c) : 0ull;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            const unsigned long long other = shfl_xor_u64(key, o);
            key = other > key ? other : key;
        }
        if (tx == 0 && key != 0ull) atomicMax(a.keys + b, key);
    }
}

// One warp per sequence: read the winner, record it, copy the traced row of
// m, mask the winner and load its unit row as the next query.
__global__ void ffma_dseq_commit_kernel(FfmaDseqArgs a, int t) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= a.B) return;
    const unsigned long long key = a.keys[b];
    __syncwarp();
    if (key == 0ull) {
        if (lane == 0) {
            atomicOr(a.status, kStatusNoWinner);
            a.picks[(int64_t)b * a.L + t] = -1;
        }
        return;
    }
    const uint32_t w = max_key_index(key);
    if (lane == 0) {
        a.keys[b] = 0ull;
        a.picks[(int64_t)b * a.L + t] = (int32_t)w;
    }
    float *mrow = a.m + (int64_t)b * a.Nf;
    if (a.trace_slot) {
        const int slot = a.trace_slot[b];
        if (slot >= 0) {
            float *dst = a.trace + ((int64_t)slot * a.L + t) * a.N;
            for (int64_t c = lane; c < a.N; c += 32) dst[c] = mrow[c];
        }
    }
    __syncwarp();
    if (lane == 0) mrow[w] = -INFINITY;
    const float *src = a.e_unit + (int64_t)w * a.Dp;
    float *q = a.q + (int64_t)b * a.Dp;
    for (int k = lane; k < a.Dp; k += 32) q[k] = src[k];
}

// --------------------------------------------------------------------------
// BMU: score = |w|^2 - 2 <x, w>, per-row (min score, lowest index) folded
// into keys[i] by atomicMin.  A one-dimensional grid: tile t covers samples
// (t / m_tiles) and neurons (t % m_tiles).
__global__ void __launch_bounds__(kFfmaThreads, 1) ffma_bmu_kernel(BmuArgs a, int64_t m_tiles, int vec) {
    extern __shared__ __align__(16) float sm[];
    __shared__ float wn_s[kTile];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int64_t i0 = (int64_t)(blockIdx.x / m_tiles) * kTile, j0 = (int64_t)(blockIdx.x % m_tiles) * kTile;
    if (tid < kTile) wn_s[tid] = j0 + tid < a.M ? a.wn[j0 + tid] : 0.0f;
    const TileOperand A{a.X, i0, a.n, (int64_t)a.D, a.D, vec != 0};
    const TileOperand B{a.W, j0, a.M, (int64_t)a.D, a.D, vec != 0};
    float acc[8][8];
    ffma_tile(acc, sm, A, B, tid, tx, ty);  // its barriers also publish wn_s
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = i0 + ty + 16 * i;
        float best = INFINITY;
        uint32_t best_j = 0xffffffffu;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = tx + 16 * j;
            const float s = fmaf(-2.0f, acc[i][j], wn_s[c]);
            if (j0 + c < a.M && (s < best || best_j == 0xffffffffu)) {
                best = s;
                best_j = (uint32_t)(j0 + c);
            }
        }
        unsigned long long key = best_j != 0xffffffffu ? min_key(best, best_j) : ~0ull;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            const unsigned long long other = shfl_xor_u64(key, o);
            key = other < key ? other : key;
        }
        if (tx == 0 && row < a.n && key != ~0ull) atomicMin(a.keys + row, key);
    }
}

}  // namespace

cudaError_t ffma_configure() {
    cudaError_t e = cudaFuncSetAttribute(ffma_dseq_fold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kFfmaSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(ffma_bmu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFfmaSmem);
    return e;
}

void launch_ffma_dseq_init(const FfmaDseqArgs &a, const int32_t *starts, const uint8_t *mask,
                           cudaStream_t st) {
    ffma_dseq_init_kernel<<<1024, 256, 0, st>>>(a, starts, mask);
}

void launch_ffma_dseq_iteration(const FfmaDseqArgs &a, int t, cudaStream_t st) {
    dim3 grid((unsigned)(a.Nf / kTile), (unsigned)(a.Bp / kTile));
    ffma_dseq_fold_kernel<<<grid, kFfmaThreads, kFfmaSmem, st>>>(a);
    ffma_dseq_commit_kernel<<<(a.B + 7) / 8, 256, 0, st>>>(a, t);
}

void launch_ffma_bmu(const BmuArgs &a, cudaStream_t st) {
    const int64_t m_tiles = (a.M + kTile - 1) / kTile, n_tiles = (a.n + kTile - 1) / kTile;
    const int vec = (a.D % 4 == 0 && (reinterpret_cast<uintptr_t>(a.X) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.W) & 15) == 0) ? 1 : 0;
    ffma_bmu_kernel<<<(unsigned)(m_tiles * n_tiles), kFfmaThreads, kFfmaSmem, st>>>(a, m_tiles, vec);
}

}  // namespace dseq
