// som.cu — the neighbourhood update that follows the BMU search in a SOM
// epoch ("From 80x to 385x: A Best-Matching-Unit Search at the L2 Roof",
// section 3 Background: every sample's closest neuron is found, then that
// neuron and its neighbours are updated; section 6 gives the update's share
// of the epoch).  Because the update comes after a search over all samples
// it is the batch map:
//
//   W_j = sum_i h(j, bmu_i) x_i / sum_i h(j, bmu_i),   W_j kept when the sum is 0,
//
// on a side_x x side_y grid (neuron j at column j % side_x, row j / side_x),
// with h(a, b) = g(|dx|) g(|dy|), g(k) = exp(-k^2 / (2 sigma^2)) for k <= R
// and 0 beyond (sigma = 0: g(0) = 1, g(k > 0) = 0).
//
// Grouping the samples by BMU turns the sum into a smoothing of the
// per-neuron sums S_k = sum_{bmu_i = k} x_i and counts n_k, and the product
// form of h makes that smoothing separable.  Three passes over the map:
//   accumulate  S (f64 atomics) and n (u32 atomics), one warp per sample,
//               into buffers the zero kernel cleared;
//   rows        T = sum_dx g(|dx|) S[k + dx] along each map row, and the
//               same for the counts (fp32 out);
//   columns     num = sum_dy g(|dy|) T[k + dy * side_x], den likewise from
//               the row-smoothed counts; W_j = num / den where den > 0.
// Every map-sized array is laid out neuron-major (j * D + d), so a warp's
// 32 consecutive threads touch 32 consecutive dimensions of one neuron and
// every tap of the stencils is a coalesced 128-byte (fp32) or 256-byte
// (f64) row segment; the 2R re-reads of each segment hit L1 (rows) or L2
// (columns, one map row apart).
#include "common.cuh"
#include "internal.h"

namespace dseq {

namespace {

constexpr int kSomThreads = 256;

__global__ void som_zero_kernel(double *__restrict__ S, int64_t nS, unsigned *__restrict__ cnt,
                                int64_t M) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nS + M; e += stride) {
        if (e < nS)
            S[e] = 0.0;
        else
            cnt[e - nS] = 0u;
    }
}

// one warp per sample: S[bmu_i] += x_i, n[bmu_i] += 1
__global__ void som_accumulate_kernel(SomArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < a.n;
         i += warps) {
        const int32_t c = a.bmu[i];
        if (c < 0 || (int64_t)c >= a.M) {
            if (lane == 0) atomicOr(a.status, kStatusBadIndex);
            continue;
        }
        const float *x = a.X + i * (int64_t)a.D;
        double *s = a.S + (int64_t)c * a.D;
        bool bad = false;
        for (int d = lane; d < a.D; d += 32) {
            const float v = __ldg(x + d);
            bad |= !isfinite(v);
            atomicAdd(s + d, (double)v);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.status, kStatusNonFinite);
        if (lane == 0) atomicAdd(a.cnt + c, 1u);
    }
}

// rows: T[j, d] = sum_dx g(|dx|) S[j + dx, d]; the counts ride along as
// M extra elements past the M x D data elements
__global__ void som_rows_kernel(SomArgs a) {
    __shared__ float g[kSomMaxRadius + 1];
    for (int k = threadIdx.x; k <= a.R; k += blockDim.x) g[k] = a.g[k];
    __syncthreads();
    const int64_t nT = a.M * (int64_t)a.D;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nT + a.M; e += stride) {
        const bool data = e < nT;
        const int64_t j = data ? e / a.D : e - nT;
        const int64_t col = j % a.side_x;
        const int lo = (int)max((int64_t)-a.R, -col);
        const int hi = (int)min((int64_t)a.R, (int64_t)a.side_x - 1 - col);
        float acc = 0.0f;
        if (data) {
            const double *src = a.S + e;
            for (int dx = lo; dx <= hi; ++dx)
                acc = fmaf(g[dx < 0 ? -dx : dx], (float)src[(int64_t)dx * a.D], acc);
            a.T[e] = acc;
        } else {
            for (int dx = lo; dx <= hi; ++dx)
                acc = fmaf(g[dx < 0 ? -dx : dx], (float)a.cnt[j + dx], acc);
            a.Tc[j] = acc;
        }
    }
}

// columns and the division, in place on W; nothing is written when an
// earlier pass flagged an error, so W is left as it was
__global__ void som_cols_kernel(SomArgs a) {
    __shared__ float g[kSomMaxRadius + 1];
    for (int k = threadIdx.x; k <= a.R; k += blockDim.x) g[k] = a.g[k];
    __syncthreads();
    if (*(volatile int *)a.status != 0) return;
    const int64_t nT = a.M * (int64_t)a.D;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t row_elems = (int64_t)a.side_x * a.D;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nT; e += stride) {
        const int64_t j = e / a.D;
        const int64_t row = j / a.side_x;
        const int lo = (int)max((int64_t)-a.R, -row);
        const int hi = (int)min((int64_t)a.R, (int64_t)a.side_y - 1 - row);
        float num = 0.0f, den = 0.0f;
        for (int dy = lo; dy <= hi; ++dy) {
            const float w = g[dy < 0 ? -dy : dy];
            num = fmaf(w, a.T[e + (int64_t)dy * row_elems], num);
            den = fmaf(w, a.Tc[j + (int64_t)dy * a.side_x], den);
        }
        if (den > 0.0f) a.W[e] = num / den;
    }
}

int grid_for(int64_t work, int per_block, int sms) {
    const int64_t blocks = (work + per_block - 1) / per_block;
    return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)sms * 16));
}

}  // namespace

void launch_som_update(const SomArgs &a, int sms, cudaStream_t st) {
    const int64_t nT = a.M * (int64_t)a.D;
    som_zero_kernel<<<grid_for(nT + a.M, kSomThreads, sms), kSomThreads, 0, st>>>(a.S, nT, a.cnt,
                                                                                  a.M);
    if (a.n > 0)
        som_accumulate_kernel<<<grid_for(a.n, kSomThreads / 32, sms), kSomThreads, 0, st>>>(a);
    som_rows_kernel<<<grid_for(nT + a.M, kSomThreads, sms), kSomThreads, 0, st>>>(a);
    som_cols_kernel<<<grid_for(nT, kSomThreads, sms), kSomThreads, 0, st>>>(a);
}

}  // namespace dseq
