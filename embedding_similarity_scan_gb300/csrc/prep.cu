// prep.cu — one-pass preparation kernels: candidate-table normalisation and
// fp16 hi/lo split, BMU operand scaling and split, squared norms, the BMU key
// initialisation / finalisation, and the row gather of global-mask
// compaction.
//
// The split: a float x with |x| <= 1 becomes hi = fp16(x) and
// lo = fp16((x - hi) * 2^12).  x - hi is exact in fp32; scaling the residual
// by 2^12 keeps it in fp16's normal range, so hi + lo * 2^-12 carries about
// 22 significant bits, and a product of two split values needs three fp16
// products (hi*hi, hi*lo, lo*hi) for fp32-level accuracy.  The tensor-core
// kernels fold the 2^-12 into a pre-scaled copy of hi on one side (the
// diversity queries, the BMU codebook: hi * 2^12), so all three products land
// in one fp32 accumulator scaled by 2^12.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "numeric.cuh"

namespace dseq {

namespace {

__device__ __forceinline__ void split_f16(float x, __half &hi, __half &lo) {
    hi = __float2half_rn(x);
    const float r = x - __half2float(hi);
    lo = __float2half_rn(r * 4096.0f);
}

__global__ void table_prepare_kernel(const float *__restrict__ E, int64_t N, int D, int Dp,
                                     float *__restrict__ e_unit, __half *__restrict__ e_split,
                                     float *__restrict__ nrm, int *status) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= N) return;
    const float *src = E + row * (int64_t)D;
    int bad;
    const float mx = row_absmax(src, D, lane, bad);
    if (bad || !(mx > 0.0f)) {
        if (lane == 0) atomicOr(status, kStatusNonFinite);
        return;
    }
    const int e = scale_exponent(mx);
    const float scale = ldexpf(1.0f, -e);
    KahanSum ss;
    for (int k = lane; k < D; k += 32) {
        const float v = src[k] * scale;
        ss.add(v * v);
    }
    const float sum = warp_sum_f(ss.total());
    const float len = sqrtf(sum);  // norm of the scaled row, in [2^-1, sqrt(D))
    const float inv = scale / len;
    if (lane == 0) nrm[row] = ldexpf(len, e);
    float *dst = e_unit + row * (int64_t)Dp;
    __half *sp = e_split + row * (int64_t)(2 * Dp);
    for (int k = lane; k < Dp; k += 32) {
        const float u = k < D ? src[k] * inv : 0.0f;
        dst[k] = u;
        __half hi, lo;
        split_f16(u, hi, lo);
        sp[k] = hi;
        sp[Dp + k] = lo;
    }
}

__global__ void table_prepare_f16_kernel(const float *__restrict__ E, int64_t N, int D, int Dp,
                                         __half *__restrict__ e_f16, float *__restrict__ rn,
                                         int *status) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= N) return;
    const float *src = E + row * (int64_t)D;
    float mx = 0.0f;
    int bad = 0;
    for (int k = lane; k < D; k += 32) {
        const float v = src[k];
        if (!isfinite(v)) bad = 1;
        mx = fmaxf(mx, fabsf(v));
    }
    mx = warp_max_f(mx);
    bad = warp_or_i(bad);
    if (bad || !(mx > 0.0f)) {
        if (lane == 0) atomicOr(status, kStatusNonFinite);
        return;
    }
    // a power-of-two scale keeps the row inside fp16's range without changing
    // its direction; the cosine uses the norm of the stored (rounded) row
    int e = 0;
    frexpf(mx, &e);
    const float scale = ldexpf(1.0f, -e);
    __half *dst = e_f16 + row * (int64_t)Dp;
    KahanSum ss;
    for (int k = lane; k < Dp; k += 32) {
        const __half h = __float2half_rn(k < D ? src[k] * scale : 0.0f);
        dst[k] = h;
        const float hv = __half2float(h);
        ss.add(hv * hv);
    }
    const float sum = warp_sum_f(ss.total());
    if (lane == 0) {
        if (!(sum > 0.0f)) atomicOr(status, kStatusNonFinite);
        rn[row] = 1.0f / sqrtf(sum);
    }
}

// The stored fp16 rows as fp32 (exact), the Gram engine's operand on fp16
// storage: their split has zero low parts, so every product is exact.
__global__ void f16_rows_kernel(const __half *__restrict__ e_f16, int64_t total,
                                float *__restrict__ out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride)
        out[i] = __half2float(e_f16[i]);
}

// inv_scale[r] *= rn[r] for both operand sides: the product's rescaling then
// also divides by the stored rows' norms
__global__ void scale_rows_kernel(float *__restrict__ a, float *__restrict__ b,
                                  const float *__restrict__ rn, int64_t N) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N; i += stride) {
        a[i] *= rn[i];
        b[i] *= rn[i];
    }
}

__global__ void bmu_prepare_kernel(const float *__restrict__ A, int64_t rows, int D, int Dp,
                                   int triple, __half *__restrict__ split,
                                   float *__restrict__ norm2, float *__restrict__ inv_scale,
                                   int *status) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float *src = A + row * (int64_t)D;
    int bad;
    const float mx = row_absmax(src, D, lane, bad);
    if (bad) {
        if (lane == 0) atomicOr(status, kStatusNonFinite);
        return;
    }
    // scale = 2^-e with mx = f * 2^e, f in [0.5, 1): max |row * scale| < 1.
    const int e = scale_exponent(mx);
    const float scale = ldexpf(1.0f, -e);
    const int w = triple ? 3 * Dp : 2 * Dp;
    __half *sp = split + row * (int64_t)w;
    KahanSum ss;
    for (int k = lane; k < Dp; k += 32) {
        const float u = k < D ? src[k] * scale : 0.0f;
        ss.add(u * u);
        __half hi, lo;
        split_f16(u, hi, lo);
        if (triple) {
            sp[k] = __float2half_rn(__half2float(hi) * 4096.0f);  // exact: power-of-two scale
            sp[Dp + k] = hi;
            sp[2 * Dp + k] = lo;
        } else {
            sp[k] = hi;
            sp[Dp + k] = lo;
        }
    }
    const float sum = warp_sum_f(ss.total());
    if (lane == 0) {
        norm2[row] = ldexpf(sum, 2 * e);
        inv_scale[row] = ldexpf(1.0f, e);
    }
}

template <typename T>
__global__ void gather_rows_kernel(const T *__restrict__ src, T *__restrict__ dst,
                                   const int32_t *__restrict__ map, int64_t rows, int64_t vecs) {
    const int64_t total = rows * vecs;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / vecs, k = i - r * vecs;
        dst[i] = src[(int64_t)map[r] * vecs + k];
    }
}

__global__ void row_sqnorm_kernel(const float *__restrict__ A, int64_t rows, int D,
                                  float *__restrict__ out, int *status) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float *src = A + row * (int64_t)D;
    int bad;
    const float mx = row_absmax(src, D, lane, bad);
    const int e = scale_exponent(mx);
    const float scale = ldexpf(1.0f, -e);
    KahanSum ss;
    for (int k = lane; k < D; k += 32) {
        const float u = src[k] * scale;
        ss.add(u * u);
    }
    const float sum = warp_sum_f(ss.total());
    if (lane == 0) {
        if (bad) atomicOr(status, kStatusNonFinite);
        out[row] = ldexpf(sum, 2 * e);
    }
}

__global__ void fill_u64_kernel(unsigned long long *p, int64_t n, unsigned long long v) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = v;
}

__global__ void bmu_finalize_kernel(const unsigned long long *__restrict__ keys,
                                    const float *__restrict__ xn, int64_t n,
                                    int32_t *__restrict__ idx, float *__restrict__ dist,
                                    int *status) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const unsigned long long k = keys[i];
        if (k == ~0ull) {
            atomicOr(status, kStatusNoWinner);
            idx[i] = -1;
            dist[i] = 0.0f;
            continue;
        }
        const float s = float_unorder((uint32_t)(k >> 32));
        idx[i] = (int32_t)(uint32_t)(k & 0xffffffffull);
        dist[i] = fmaxf(0.0f, xn[i] + s);
    }
}

inline unsigned blocks_for_rows(int64_t rows, int warps_per_block) {
    return (unsigned)((rows + warps_per_block - 1) / warps_per_block);
}

}  // namespace

void launch_table_prepare(const float *E, int64_t N, int D, int Dp, float *e_unit,
                          __half *e_split, float *nrm, int *status, cudaStream_t st) {
    table_prepare_kernel<<<blocks_for_rows(N, 8), 256, 0, st>>>(E, N, D, Dp, e_unit, e_split,
                                                                  nrm, status);
}

void launch_table_prepare_f16(const float *E, int64_t N, int D, int Dp, __half *e_f16,
                              float *rn, int *status, cudaStream_t st) {
    table_prepare_f16_kernel<<<blocks_for_rows(N, 8), 256, 0, st>>>(E, N, D, Dp, e_f16, rn,
                                                                       status);
}

void launch_f16_rows(const __half *e_f16, int64_t N, int Dp, float *out, cudaStream_t st) {
    const int64_t total = N * (int64_t)Dp;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, 152 * 16);
    f16_rows_kernel<<<(unsigned)std::max<int64_t>(1, blocks), 256, 0, st>>>(e_f16, total, out);
}

void launch_scale_rows(float *a, float *b, const float *rn, int64_t N, cudaStream_t st) {
    const int64_t blocks = std::min<int64_t>((N + 255) / 256, 152 * 4);
    scale_rows_kernel<<<(unsigned)std::max<int64_t>(1, blocks), 256, 0, st>>>(a, b, rn, N);
}

void launch_gather_rows(const void *src, void *dst, const int32_t *map, int64_t rows,
                        int64_t row_bytes, cudaStream_t st) {
    const bool wide = row_bytes % 16 == 0;
    const int64_t vecs = wide ? row_bytes / 16 : row_bytes / 4;
    const int64_t total = rows * vecs;
    if (total <= 0) return;
    const unsigned blocks = (unsigned)((total + 255) / 256 < 8192 ? (total + 255) / 256 : 8192);
    if (wide)
        gather_rows_kernel<uint4><<<blocks, 256, 0, st>>>(static_cast<const uint4 *>(src),
                                                          static_cast<uint4 *>(dst), map, rows, vecs);
    else
        gather_rows_kernel<uint32_t><<<blocks, 256, 0, st>>>(static_cast<const uint32_t *>(src),
                                                             static_cast<uint32_t *>(dst), map, rows, vecs);
}

void launch_bmu_prepare(const float *A, int64_t rows, int D, int Dp, int triple, __half *split,
                        float *norm2, float *inv_scale, int *status, cudaStream_t st) {
    bmu_prepare_kernel<<<blocks_for_rows(rows, 8), 256, 0, st>>>(A, rows, D, Dp, triple, split,
                                                                   norm2, inv_scale, status);
}

void launch_row_sqnorm(const float *A, int64_t rows, int D, float *out, int *status,
                       cudaStream_t st) {
    row_sqnorm_kernel<<<blocks_for_rows(rows, 8), 256, 0, st>>>(A, rows, D, out, status);
}

void launch_bmu_keys_init(unsigned long long *keys, int64_t n, cudaStream_t st) {
    fill_u64_kernel<<<(unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0, st>>>(
        keys, n, ~0ull);
}

void launch_bmu_finalize(const BmuArgs &a, cudaStream_t st) {
    bmu_finalize_kernel<<<(unsigned)((a.n + 255) / 256 < 4096 ? (a.n + 255) / 256 : 4096), 256, 0,
                          st>>>(a.keys, a.xn, a.n, a.idx, a.dist, a.status);
}

}  // namespace dseq
