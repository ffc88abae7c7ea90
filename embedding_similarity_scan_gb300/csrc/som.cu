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
// form of h makes that smoothing separable.  The kernels:
//   prepare     max |x| over all samples (its exponent fixes the fixed-point
//               scale below) and the counts n_k (32-bit atomics);
//   scan        each neuron's offset in the samples grouped by BMU (an
//               exclusive scan of n_k per tile of kSomScanTile neurons, then
//               one over the tiles' totals);
//   scatter     order[offset(bmu_i) + r] = i (a counting sort), and the rows
//               of S of neurons whose samples straddle a chunk boundary
//               cleared;
//   accumulate  S, one warp per chunk of kSomChunk grouped samples: the
//               sums of each run of samples of one neuron in registers; a
//               neuron whose samples all lie in the chunk gets its row stored,
//               one that straddles chunks gets its part added with 64-bit
//               integer atomics.  The samples' BMUs are very uneven (a few
//               neurons hold thousands of samples, most none), so the work
//               is dealt by samples, not by neurons.  Each x becomes the
//               integer trunc(x 2^F), F chosen so that no sum of n samples
//               can overflow, so the sums are exact and independent of the
//               order the samples are grouped and added in: the update is
//               bitwise reproducible.  The truncation costs at most
//               2^-F <= max|x| n 2^-61 per sample.  Rows of S of neurons
//               without samples are never written: the rows pass reads S only
//               where n_k > 0;
//   rows        T = sum_dx g(|dx|) S[k + dx] along each map row, and the same
//               for the counts, from a shared-memory tile with an R-wide halo
//               (fp32 out; the tile's loads are issued in batches so that
//               several are in flight per thread);
//   columns     num = sum_dy g(|dy|) T[k + dy side_x], den likewise from the
//               row-smoothed counts, again from a tile; W_j = num / den where
//               den > 0, in place.
// No step uses 64-bit floating point: GB300's FP64 rate is a small fraction
// of its fp32 rate, and a conversion from or to double runs at that rate.
// Every map-sized array is neuron-major (j * D + d); a warp covers 32
// consecutive dimensions of one neuron, so each load is a full 128-byte
// (fp32) or 256-byte (int64) segment.
#include "common.cuh"
#include "internal.h"
#include "numeric.cuh"

namespace dseq {

namespace {

constexpr int kSomThreads = 256;
constexpr int kRowTile = 128;  // neurons along a map row per CTA (rows pass)
constexpr int kColTile = 64;   // neurons along a map column per CTA (columns pass)

// Exponent bound E of the largest |x| (|x| < 2^(E+1)) and the fixed-point
// scale F = 61 - E - ceil(log2 n): every |x| 2^F < 2^(62 - ceil(log2 n)), so
// a sum of n of them stays below 2^62.
__device__ __forceinline__ int fixed_scale(unsigned maxbits, int64_t n) {
    const int ef = (int)(maxbits >> 23);
    const int E = ef == 0 ? -126 : ef - 127;
    const int L = n <= 1 ? 0 : 64 - __clzll((unsigned long long)(n - 1));
    return 61 - E - L;
}

__global__ void som_prepare_kernel(SomArgs a) {
    const int64_t nX = a.n * (int64_t)a.D;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    unsigned mx = 0;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nX; e += stride)
        mx = max(mx, __float_as_uint(__ldg(a.X + e)) & 0x7fffffffu);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.n; i += stride) {
        const int32_t c = a.bmu[i];
        if (c < 0 || (int64_t)c >= a.M)
            atomicOr(a.status, kStatusBadIndex);
        else
            atomicAdd(a.cnt + c, 1u);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0 && mx) atomicMax(a.maxbits, mx);
}

// Exclusive scan of v over a block of 1024 threads: returns this thread's
// prefix (the sum of v over the threads before it).
__device__ __forceinline__ unsigned block_exclusive_scan(unsigned v, unsigned *warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        unsigned w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_sums[lane] = w;  // inclusive over the warps
    }
    __syncthreads();
    const unsigned prefix = (warp ? warp_sums[warp - 1] : 0u) + incl - v;
    __syncthreads();  // warp_sums may be reused by the caller's next scan
    return prefix;
}

// Offsets of each neuron's samples within its tile of kSomScanTile neurons
// (4 per thread), and the tile's total.
__global__ void __launch_bounds__(1024) som_scan_kernel(SomArgs a) {
    __shared__ unsigned warp_sums[32];
    const int64_t base = (int64_t)blockIdx.x * kSomScanTile + 4 * (int64_t)threadIdx.x;
    unsigned c[4], s = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        c[j] = base + j < a.M ? a.cnt[base + j] : 0u;
        s += c[j];
    }
    unsigned p = block_exclusive_scan(s, warp_sums);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (base + j < a.M) a.off[base + j] = p;
        p += c[j];
    }
    if (threadIdx.x == 1023) a.tile_sum[blockIdx.x] = p;
}

// Exclusive scan of the tiles' totals (one CTA, 1024 tiles per round).
__global__ void __launch_bounds__(1024) som_scan_tiles_kernel(SomArgs a, int64_t tiles) {
    __shared__ unsigned warp_sums[32];
    __shared__ unsigned carry_s;
    unsigned carry = 0;
    for (int64_t t0 = 0; t0 < tiles; t0 += 1024) {
        const int64_t t = t0 + threadIdx.x;
        const unsigned v = t < tiles ? a.tile_sum[t] : 0u;
        const unsigned p = block_exclusive_scan(v, warp_sums);
        if (t < tiles) a.tile_off[t] = carry + p;
        if (threadIdx.x == 1023) carry_s = p + v;
        __syncthreads();
        carry += carry_s;
        __syncthreads();
    }
}

__device__ __forceinline__ unsigned neuron_start(const SomArgs &a, int64_t k) {
    return a.tile_off[k / kSomScanTile] + a.off[k];
}

// order[start(bmu_i) + r] = i, r the sample's place among its neuron's
// samples (arrival order; the sums do not depend on it); and the rows of S of
// neurons whose samples straddle a chunk boundary cleared (one warp per
// neuron), since the accumulate kernel adds into those with atomics.
__global__ void som_scatter_kernel(SomArgs a) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.n; i += stride) {
        const int32_t c = a.bmu[i];
        if (c < 0 || (int64_t)c >= a.M) continue;  // flagged by the prepare kernel
        a.order[neuron_start(a, c) + atomicAdd(a.cursor + c, 1u)] = (int32_t)i;
    }
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t k = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); k < a.M; k += warps) {
        const unsigned count = a.cnt[k];
        if (count == 0) continue;
        const unsigned st = neuron_start(a, k);
        if (st / kSomChunk == (st + count - 1) / kSomChunk) continue;
        long long *srow = a.S + k * (int64_t)a.D;
        for (int d = lane; d < a.D; d += 32) srow[d] = 0;
    }
}

constexpr int kAccBatch = 8;  // dimensions per lane and pass (32 * 8 = 256)

// The sums of one run of a neuron's samples [r0, r1) (grouped positions):
// stored when the run is all of the neuron's samples, otherwise added.
__device__ __forceinline__ void flush_run(const SomArgs &a, int32_t k, unsigned r0, unsigned r1,
                                          const long long (&acc)[kAccBatch], int d0, int lane) {
    const unsigned st = neuron_start(a, k);
    const bool whole = r0 == st && r1 == st + a.cnt[k];
    long long *srow = a.S + (int64_t)k * a.D;
#pragma unroll
    for (int u = 0; u < kAccBatch; ++u) {
        const int d = d0 + 32 * u + lane;
        if (d >= a.D) break;
        if (whole)
            srow[d] = acc[u];
        else
            atomicAdd(reinterpret_cast<unsigned long long *>(srow + d), (unsigned long long)acc[u]);
    }
}

// One warp per chunk of kSomChunk grouped samples: S_k += fixed(x_i) over the
// chunk's runs of samples of one neuron, the next sample's row loaded while
// the current one is added.
__global__ void som_accumulate_kernel(SomArgs a, int64_t tiles) {
    const unsigned maxbits = *a.maxbits;
    if (maxbits >= 0x7f800000u) {  // an infinity or NaN among the samples
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, kStatusNonFinite);
        return;
    }
    const int F = fixed_scale(maxbits, a.n);
    const int lane = threadIdx.x & 31;
    const unsigned total = a.tile_off[tiles - 1] + a.tile_sum[tiles - 1];  // grouped samples
    const int64_t chunks = ((int64_t)total + kSomChunk - 1) / kSomChunk;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t ch = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); ch < chunks; ch += warps) {
        const unsigned s0 = (unsigned)(ch * kSomChunk);
        const unsigned m = min((unsigned)kSomChunk, total - s0);
        const int32_t my_i = lane < (int)m ? a.order[s0 + lane] : 0;
        const int32_t my_k = lane < (int)m ? a.bmu[my_i] : -1;
        for (int d0 = 0; d0 < a.D; d0 += 32 * kAccBatch) {
            long long acc[kAccBatch];
#pragma unroll
            for (int u = 0; u < kAccBatch; ++u) acc[u] = 0;
            float v[kAccBatch], vn[kAccBatch];
            {
                const float *x = a.X + (int64_t)__shfl_sync(0xffffffffu, my_i, 0) * a.D;
#pragma unroll
                for (int u = 0; u < kAccBatch; ++u) {
                    const int d = d0 + 32 * u + lane;
                    v[u] = d < a.D ? __ldg(x + d) : 0.0f;
                }
            }
            int32_t k_run = __shfl_sync(0xffffffffu, my_k, 0);
            unsigned run0 = s0;
            for (unsigned j = 0; j < m; ++j) {
                const int32_t i_next = __shfl_sync(0xffffffffu, my_i, min(j + 1, m - 1));
                const int32_t k = __shfl_sync(0xffffffffu, my_k, j);
                if (j + 1 < m) {
                    const float *x = a.X + (int64_t)i_next * a.D;
#pragma unroll
                    for (int u = 0; u < kAccBatch; ++u) {
                        const int d = d0 + 32 * u + lane;
                        vn[u] = d < a.D ? __ldg(x + d) : 0.0f;
                    }
                }
                if (k != k_run) {  // the run of k_run ended before sample j
                    flush_run(a, k_run, run0, s0 + j, acc, d0, lane);
#pragma unroll
                    for (int u = 0; u < kAccBatch; ++u) acc[u] = 0;
                    k_run = k;
                    run0 = s0 + j;
                }
#pragma unroll
                for (int u = 0; u < kAccBatch; ++u) {
                    acc[u] += to_fixed(v[u], F);
                    v[u] = vn[u];
                }
            }
            flush_run(a, k_run, run0, s0 + m, acc, d0, lane);
        }
    }
}

// Loads rows [0, span) of a (span x 32) tile, kLoadBatch rows per warp in
// flight: fetch(r) returns the value for tile row r and this lane.
constexpr int kLoadBatch = 4;
template <class Fetch>
__device__ __forceinline__ void load_tile(float *tile, int span, int warp, int lane, Fetch fetch) {
    constexpr int kWarps = kSomThreads / 32;
    for (int base = warp; base < span; base += kWarps * kLoadBatch) {
        float v[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int r = base + kWarps * u;
            v[u] = r < span ? fetch(r) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int r = base + kWarps * u;
            if (r < span) tile[r * 32 + lane] = v[u];
        }
    }
}

// Rows pass.  CTA = (dimension chunk of 32, kRowTile neurons of one map
// row).  The tile holds the neurons [x0 - R, x0 + kRowTile + R) of the row,
// zero outside the map (a zero term leaves a sum unchanged, so this equals
// clipping the window at the map's edge).  Chunk-0 CTAs also smooth the
// counts of their neurons.
__global__ void __launch_bounds__(kSomThreads) som_rows_kernel(SomArgs a) {
    extern __shared__ float tile[];  // (kRowTile + 2R) x 32, counts (span), g[2R + 1]
    const int R = a.R, span = kRowTile + 2 * R;
    float *tc = tile + span * 32;
    float *g = tc + span;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = (a.D + 31) / 32;
    const int ntx = (a.side_x + kRowTile - 1) / kRowTile;
    const int64_t b = blockIdx.x;
    const int chunk = (int)(b % nch);
    const int64_t rest = b / nch;
    const int x0 = (int)(rest % ntx) * kRowTile;
    const int64_t row0 = (rest / ntx) * a.side_x;
    // the whole window, g[k] = weight of offset k - R
    for (int k = threadIdx.x; k <= 2 * R; k += blockDim.x) g[k] = a.g[k < R ? R - k : k - R];
    const int d = chunk * 32 + lane;
    float s1, s2;
    fixed_unscale(fixed_scale(*a.maxbits, a.n), s1, s2);
    load_tile(tile, span, warp, lane, [&](int r) {
        const int xg = x0 - R + r;
        // neurons without samples have no row of S (their sums are zero)
        return (xg >= 0 && xg < a.side_x && d < a.D && a.cnt[row0 + xg] != 0u)
                   ? from_fixed(a.S[(row0 + xg) * a.D + d], s1, s2) : 0.0f;
    });
    if (chunk == 0)
        for (int r = threadIdx.x; r < span; r += blockDim.x) {
            const int xg = x0 - R + r;
            tc[r] = (xg >= 0 && xg < a.side_x) ? (float)a.cnt[row0 + xg] : 0.0f;
        }
    __syncthreads();
    // each warp: kRowTile / 8 consecutive outputs, all taps of one weight at once
    {
        constexpr int V = kRowTile / (kSomThreads / 32);
        const int xb = warp * V;
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.0f;
        const float *t = tile + xb * 32 + lane;
        for (int k = 0; k <= 2 * R; ++k) {
            const float w = g[k];
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] = fmaf(w, t[(k + v) * 32], acc[v]);
        }
        if (d < a.D)
#pragma unroll
            for (int v = 0; v < V; ++v)
                if (x0 + xb + v < a.side_x) a.T[(row0 + x0 + xb + v) * a.D + d] = acc[v];
    }
    if (chunk == 0)
        for (int xi = threadIdx.x; xi < kRowTile && x0 + xi < a.side_x; xi += blockDim.x) {
            float acc = 0.0f;
            for (int k = 0; k <= 2 * R; ++k) acc = fmaf(g[k], tc[xi + k], acc);
            a.Tc[row0 + x0 + xi] = acc;
        }
}

// Columns pass and the division, in place on W.  CTA = (dimension chunk of
// 32, one map column, kColTile neurons down it); the denominators of the
// tile's neurons are smoothed once into shared memory.  Nothing is written
// when an earlier kernel flagged an error, so W is then left as it was.
__global__ void __launch_bounds__(kSomThreads) som_cols_kernel(SomArgs a) {
    extern __shared__ float tile[];  // (kColTile + 2R) x 32, counts (span), den, g[2R + 1]
    const int R = a.R, span = kColTile + 2 * R;
    float *tc = tile + span * 32;
    float *den = tc + span;
    float *g = den + kColTile;
    if (*(volatile int *)a.status != 0) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = (a.D + 31) / 32;
    const int64_t b = blockIdx.x;
    const int chunk = (int)(b % nch);
    const int64_t rest = b / nch;
    const int x = (int)(rest % a.side_x);
    const int y0 = (int)(rest / a.side_x) * kColTile;
    // the whole window, g[k] = weight of offset k - R
    for (int k = threadIdx.x; k <= 2 * R; k += blockDim.x) g[k] = a.g[k < R ? R - k : k - R];
    const int d = chunk * 32 + lane;
    load_tile(tile, span, warp, lane, [&](int r) {
        const int yg = y0 - R + r;
        return (yg >= 0 && yg < a.side_y && d < a.D)
                   ? a.T[((int64_t)yg * a.side_x + x) * a.D + d] : 0.0f;
    });
    for (int r = threadIdx.x; r < span; r += blockDim.x) {
        const int yg = y0 - R + r;
        tc[r] = (yg >= 0 && yg < a.side_y) ? a.Tc[(int64_t)yg * a.side_x + x] : 0.0f;
    }
    __syncthreads();
    for (int yi = threadIdx.x; yi < kColTile; yi += blockDim.x) {
        float acc = 0.0f;
        for (int k = 0; k <= 2 * R; ++k) acc = fmaf(g[k], tc[yi + k], acc);
        den[yi] = acc;
    }
    __syncthreads();
    {
        constexpr int V = kColTile / (kSomThreads / 32);
        const int yb = warp * V;
        float num[V];
#pragma unroll
        for (int v = 0; v < V; ++v) num[v] = 0.0f;
        const float *t = tile + yb * 32 + lane;
        for (int k = 0; k <= 2 * R; ++k) {
            const float w = g[k];
#pragma unroll
            for (int v = 0; v < V; ++v) num[v] = fmaf(w, t[(k + v) * 32], num[v]);
        }
        if (d < a.D)
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int yy = y0 + yb + v;
                const float dn = den[yb + v];
                if (yy < a.side_y && dn > 0.0f) a.W[((int64_t)yy * a.side_x + x) * a.D + d] = num[v] / dn;
            }
    }
}

int grid_for(int64_t work, int per_block, int sms) {
    const int64_t blocks = (work + per_block - 1) / per_block;
    return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)sms * 16));
}

size_t rows_smem(int R) { return ((size_t)(kRowTile + 2 * R) * 33 + 2 * R + 1) * sizeof(float); }
size_t cols_smem(int R) {
    return ((size_t)(kColTile + 2 * R) * 33 + kColTile + 2 * R + 1) * sizeof(float);
}

}  // namespace

cudaError_t launch_som_update(const SomArgs &a, int sms, cudaStream_t st) {
    static bool attrs_set[64] = {};  // the attribute is per function and device
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return de;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attrs_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(som_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)rows_smem(kSomMaxRadius));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(som_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)cols_smem(kSomMaxRadius));
        if (e != cudaSuccess) return e;
        attrs_set[dev] = true;
    }
    const int nch = (a.D + 31) / 32;
    const int64_t tiles = (a.M + kSomScanTile - 1) / kSomScanTile;
    som_prepare_kernel<<<grid_for(a.n * (int64_t)a.D, kSomThreads, sms), kSomThreads, 0, st>>>(a);
    som_scan_kernel<<<(unsigned)tiles, 1024, 0, st>>>(a);
    som_scan_tiles_kernel<<<1, 1024, 0, st>>>(a, tiles);
    som_scatter_kernel<<<grid_for(std::max<int64_t>(a.n, a.M * 32), kSomThreads, sms), kSomThreads, 0, st>>>(a);
    som_accumulate_kernel<<<grid_for((a.n + kSomChunk - 1) / kSomChunk, kSomThreads / 32, sms),
                            kSomThreads, 0, st>>>(a, tiles);
    const int64_t ntx = (a.side_x + kRowTile - 1) / kRowTile;
    som_rows_kernel<<<(unsigned)(nch * ntx * a.side_y), kSomThreads, rows_smem(a.R), st>>>(a);
    const int64_t nty = (a.side_y + kColTile - 1) / kColTile;
    som_cols_kernel<<<(unsigned)(nch * a.side_x * nty), kSomThreads, cols_smem(a.R), st>>>(a);
    return cudaGetLastError();
}

}  // namespace dseq
