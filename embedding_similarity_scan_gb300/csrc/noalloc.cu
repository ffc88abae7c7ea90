// noalloc.cu — bmu_search_noalloc: the tensor-core best-matching-unit search
// for callers that cannot allocate device memory.
//
// bmu_search keeps a workspace that it grows with cudaMalloc.  Some callers
// cannot let a library do that: code running inside a framework whose
// pooling allocator has already reserved nearly all of the GPU's memory (a
// cudaMalloc there fails, or takes memory the pool counts on), and
// latency-critical loops that cannot absorb the device-wide synchronisation
// cudaMalloc and cudaFree may imply.  This variant runs the same kernels on
// a fixed scratch array that lives in the library image itself: a
// file-scope __device__ array of kNoAllocScratchBytes, which every GPU that
// loads the library holds until the process exits.  The caller passes
// device-resident inputs and outputs; the entry point calls no cudaMalloc,
// cudaFree or allocating library routine.
#include <cstdio>
#include <mutex>

#include "../../include/dseq.h"
#include "internal.h"

namespace {

// Upper bound of the scratch one call may use: the split operands, norms,
// scales, per-sample keys and the status word.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_bmu_scratch[kNoAllocScratchBytes];

// Device address of g_bmu_scratch per device.  In host code the array's name
// only stands in for the symbol, so the address comes from
// cudaGetSymbolAddress, taken once per device with that device current.
std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};

int scratch_address(int dev, unsigned char **out) {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (dev < 0 || dev >= 64) return dseq::host::fail_msg(DSEQ_ECUDA, "device ordinal out of range");
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_bmu_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            char msg[256];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the scratch array failed: %s",
                     cudaGetErrorString(e));
            return dseq::host::fail_msg(DSEQ_ECUDA, msg);
        }
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<unsigned char *>(g_scratch_addr[dev]);
    return DSEQ_OK;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" int bmu_search_noalloc(const float *X, int64_t n, const float *W, int64_t M,
                                  int32_t D, int32_t *idx, float *dist, void *cuda_stream) {
    using namespace dseq;
    host::clear_error();
    if (!X || !W || !idx || !dist) return host::fail_msg(DSEQ_EINVAL, "NULL pointer argument");
    if (n < 1 || n >= (int64_t(1) << 31) || M < 1 || M >= (int64_t(1) << 31))
        return host::fail_msg(DSEQ_EINVAL, "n or M out of range");
    if (D < 1 || D > 16384) return host::fail_msg(DSEQ_EINVAL, "D out of range");
    {
        // all four on the current device (nothing can be staged); memory of
        // another device is rejected with its own message
        const void *ptrs[4] = {X, W, idx, dist};
        const char *names[4] = {"X", "W", "idx", "dist"};
        for (int i = 0; i < 4; ++i) {
            bool on_device = false;
            const int r = host::locate_ptr(ptrs[i], names[i], on_device);
            if (r != DSEQ_OK) return r;
            if (!on_device)
                return host::fail_msg(DSEQ_EINVAL,
                                      "bmu_search_noalloc needs X, W, idx and dist in device memory");
        }
    }
    const int Dp = (D + kKBlock - 1) / kKBlock * kKBlock;
    // scratch layout, every piece 256-byte aligned
    const size_t off_xs = 0;
    const size_t off_ws = off_xs + align256((size_t)n * kBmuPartsX * Dp * sizeof(__half));
    const size_t off_xn = off_ws + align256((size_t)M * kBmuPartsW * Dp * sizeof(__half));
    const size_t off_wn = off_xn + align256((size_t)n * sizeof(float));
    const size_t off_xi = off_wn + align256((size_t)M * sizeof(float));
    const size_t off_wi = off_xi + align256((size_t)n * sizeof(float));
    const size_t off_k = off_wi + align256((size_t)M * sizeof(float));
    const size_t off_st = off_k + align256((size_t)n * sizeof(unsigned long long));
    const size_t need = off_st + 256;
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "bmu_search_noalloc needs %zu bytes of scratch for n=%lld, M=%lld, D=%d; "
                 "its fixed scratch holds %zu bytes",
                 need, (long long)n, (long long)M, D, kNoAllocScratchBytes);
        return host::fail_msg(DSEQ_EINVAL, msg);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return host::fail_msg(DSEQ_ECUDA, cudaGetErrorString(e));
    unsigned char *base = nullptr;
    int r = scratch_address(dev, &base);
    if (r != DSEQ_OK) return r;
    int sms = 0;
    if ((r = host::sm_count(dev, &sms)) != DSEQ_OK) return r;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);

    BmuArgs a;
    memset(&a, 0, sizeof a);
    a.X = X;
    a.W = W;
    a.x_split = reinterpret_cast<const __half *>(base + off_xs);
    a.w_split = reinterpret_cast<const __half *>(base + off_ws);
    a.xn = reinterpret_cast<const float *>(base + off_xn);
    a.wn = reinterpret_cast<const float *>(base + off_wn);
    a.x_inv_scale = reinterpret_cast<const float *>(base + off_xi);
    a.w_inv_scale = reinterpret_cast<const float *>(base + off_wi);
    a.keys = reinterpret_cast<unsigned long long *>(base + off_k);
    a.idx = idx;
    a.dist = dist;
    a.status = reinterpret_cast<int *>(base + off_st);
    a.n = n;
    a.M = M;
    a.D = D;
    a.Dp = Dp;
    a.timeout_ns = 10000ull * 1000000ull;

    // the scratch keeps the previous call's contents: reset what must start
    // from a known value (status word, keys); the rest is overwritten
    e = cudaMemsetAsync(a.status, 0, sizeof(int), st);
    if (e != cudaSuccess) return host::fail_msg(DSEQ_ECUDA, cudaGetErrorString(e));
    launch_bmu_keys_init(a.keys, n, st);
    launch_bmu_prepare(X, n, D, Dp, 0, const_cast<__half *>(a.x_split), const_cast<float *>(a.xn),
                       const_cast<float *>(a.x_inv_scale), a.status, st);
    launch_bmu_prepare(W, M, D, Dp, 1, const_cast<__half *>(a.w_split), const_cast<float *>(a.wn),
                       const_cast<float *>(a.w_inv_scale), a.status, st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return host::fail_msg(DSEQ_ECUDA, cudaGetErrorString(e));
    // CTA pairs on whole pairs of sample blocks, as bmu_search by default
    TcPlan plan{};
    plan.pair = 1;
    plan.n_beta = (int)((n + kUnitRows - 1) / kUnitRows);
    plan.n_beta += plan.n_beta & 1;
    plan.set_uniform(256, M);
    const int64_t pair_units = plan.units() / 2;
    const int64_t pairs = sms / 2 > 0 ? sms / 2 : 1;
    plan.grid = 2 * (int)(pair_units < pairs ? (pair_units > 0 ? pair_units : 1) : pairs);
    CUtensorMap tx, tw;
    if ((r = host::encode_map(tx, a.x_split, kBmuPartsX * Dp, n, kUnitRows)) != DSEQ_OK) return r;
    if ((r = host::encode_map(tw, a.w_split, kBmuPartsW * Dp, M, plan.tile_n / 2)) != DSEQ_OK) return r;
    e = launch_tc_bmu(a, plan, tx, tw, 0, st);
    if (e != cudaSuccess) return host::fail_msg(DSEQ_ECUDA, cudaGetErrorString(e));
    launch_bmu_finalize(a, st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return host::fail_msg(DSEQ_ECUDA, cudaGetErrorString(e));
    return host::read_device_status(a.status, st);
}
