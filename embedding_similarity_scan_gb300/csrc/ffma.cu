// ffma.cu — the FP32-FFMA variant of both scans: a shared-memory tiled
// SIMT contraction (64 x 64 outputs per CTA, 4 x 4 per thread) with the
// min-fold / argmax (diversity) or argmin (BMU) fused into its epilogue, so
// the similarity block is never written out.  One launch per iteration plus
// a small commit launch; kept as the plain fp32 reference path of the
// library and as a cross-check of the tensor-core path.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dseq {

namespace {

constexpr int kT = 64;   // outputs per CTA side
constexpr int kK = 16;   // K per shared-memory phase

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int o) {
    return __shfl_xor_sync(0xffffffffu, v, o);
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

// S = Q * E^T on a 64 x 64 tile, then d = 1 - S (unit rows), m = min(m, d),
// and the per-row (max m, lowest index) folded into keys[b] by atomicMax.
__global__ void __launch_bounds__(256) ffma_dseq_fold_kernel(FfmaDseqArgs a) {
    __shared__ __align__(16) float As[kK][kT + 4];
    __shared__ __align__(16) float Bs[kK][kT + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int64_t b0 = (int64_t)blockIdx.y * kT, c0 = (int64_t)blockIdx.x * kT;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    const int lr = tid >> 2, lk = (tid & 3) * 4;
    for (int k0 = 0; k0 < a.Dp; k0 += kK) {
        const float4 av = *reinterpret_cast<const float4 *>(a.q + (b0 + lr) * a.Dp + k0 + lk);
        float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c0 + lr < a.N)
            bv = *reinterpret_cast<const float4 *>(a.e_unit + (c0 + lr) * a.Dp + k0 + lk);
        As[lk + 0][lr] = av.x;
        As[lk + 1][lr] = av.y;
        As[lk + 2][lr] = av.z;
        As[lk + 3][lr] = av.w;
        Bs[lk + 0][lr] = bv.x;
        Bs[lk + 1][lr] = bv.y;
        Bs[lk + 2][lr] = bv.z;
        Bs[lk + 3][lr] = bv.w;
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kK; ++kk) {
            const float4 x = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
            const float4 y = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
            const float xa[4] = {x.x, x.y, x.z, x.w};
            const float ya[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], ya[j], acc[i][j]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t b = b0 + ty * 4 + i;
        float *mrow = a.m + b * a.Nf + c0 + tx * 4;
        float4 mv = *reinterpret_cast<float4 *>(mrow);
        float mm[4] = {mv.x, mv.y, mv.z, mv.w};
        float best = -INFINITY;
        uint32_t best_c = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float d = 1.0f - acc[i][j];
            mm[j] = fminf(mm[j], d);
            if (mm[j] > best) {
                best = mm[j];
                best_c = (uint32_t)(c0 + tx * 4 + j);
            }
        }
        *reinterpret_cast<float4 *>(mrow) = make_float4(mm[0], mm[1], mm[2], mm[3]);
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
// into keys[i] by atomicMin.

__global__ void __launch_bounds__(256) ffma_bmu_kernel(BmuArgs a) {
    __shared__ __align__(16) float As[kK][kT + 4];
    __shared__ __align__(16) float Bs[kK][kT + 4];
    __shared__ float wn_s[kT];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int64_t i0 = (int64_t)blockIdx.y * kT, j0 = (int64_t)blockIdx.x * kT;
    if (tid < kT) wn_s[tid] = j0 + tid < a.M ? a.wn[j0 + tid] : 0.0f;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
    const int lr = tid >> 2, lk = (tid & 3) * 4;
    for (int k0 = 0; k0 < a.D; k0 += kK) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k0 + lk + u;
            As[lk + u][lr] = (i0 + lr < a.n && k < a.D) ? a.X[(i0 + lr) * a.D + k] : 0.0f;
            Bs[lk + u][lr] = (j0 + lr < a.M && k < a.D) ? a.W[(j0 + lr) * a.D + k] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kK; ++kk) {
            const float4 x = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
            const float4 y = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
            const float xa[4] = {x.x, x.y, x.z, x.w};
            const float ya[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], ya[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t row = i0 + ty * 4 + i;
        float best = INFINITY;
        uint32_t best_j = 0xffffffffu;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t col = j0 + tx * 4 + j;
            const float s = fmaf(-2.0f, acc[i][j], wn_s[tx * 4 + j]);
            if (col < a.M && (s < best || best_j == 0xffffffffu)) {
                best = s;
                best_j = (uint32_t)col;
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

void launch_ffma_dseq_init(const FfmaDseqArgs &a, const int32_t *starts, const uint8_t *mask,
                           cudaStream_t st) {
    ffma_dseq_init_kernel<<<1024, 256, 0, st>>>(a, starts, mask);
}

void launch_ffma_dseq_iteration(const FfmaDseqArgs &a, int t, cudaStream_t st) {
    dim3 grid((unsigned)(a.Nf / kT), (unsigned)(a.Bp / kT));
    ffma_dseq_fold_kernel<<<grid, 256, 0, st>>>(a);
    ffma_dseq_commit_kernel<<<(a.B + 7) / 8, 256, 0, st>>>(a, t);
}

void launch_ffma_bmu(const BmuArgs &a, cudaStream_t st) {
    dim3 grid((unsigned)((a.M + kT - 1) / kT), (unsigned)((a.n + kT - 1) / kT));
    ffma_bmu_kernel<<<grid, 256, 0, st>>>(a);
}

}  // namespace dseq
