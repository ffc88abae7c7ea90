// api.cu — the C ABI of libdseq.so: argument checks, pointer-kind detection
// and staging, device workspace, tensor-map encoding, work planning
// (chunk widths, global-mask compaction, BMU slices), and the launches of
// the kernels in tc_dseq.cu, tc_bmu.cu, ffma.cu, prep.cu and som.cu.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/dseq.h"
#include "internal.h"

using namespace dseq;

namespace {

// --------------------------------------------------------------------------
// errors and statistics (per calling thread)
thread_local std::string g_err;
constexpr int kNoShift = 1 << 30;

struct Stats {
    int64_t units = 0, tile_n = 0, tile_n2 = 0, n_wide = 0, grid = 0, launches = 0, kernel_ns = 0,
            update_ns = 0, gram = 0, gram_ns = 0, walk_ns = 0, walk = 0;
};
thread_local Stats g_stats;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_code(cudaError_t e) {
    return e == cudaErrorMemoryAllocation ? DSEQ_ENOMEM
           : (e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorLaunchOutOfResources)
               ? DSEQ_ELAUNCH
               : DSEQ_ECUDA;
}

#define CUDA_TRY(expr)                                                                        \
    do {                                                                                      \
        cudaError_t e_ = (expr);                                                              \
        if (e_ != cudaSuccess) {                                                              \
            cudaGetLastError();                                                               \
            return fail(cuda_code(e_), "%s failed: %s (%s:%d)", #expr, cudaGetErrorString(e_), \
                        __FILE__, __LINE__);                                                  \
        }                                                                                     \
    } while (0)

#define TRY(expr)              \
    do {                       \
        int r_ = (expr);       \
        if (r_ != DSEQ_OK) return r_; \
    } while (0)

// --------------------------------------------------------------------------
// options
struct Options {
    int64_t engine = 0;
    int64_t tile_n = 0;
    int64_t tile_n2 = 0;
    int64_t grid = 0;
    int64_t timeout_ms = 10000;
    int64_t fault_skip_arrive = 0;
    int64_t fault_skip_copy = 0;
    int64_t timeline = 0;
    int64_t pair = 1;
    int64_t storage = 0;
    int64_t criterion = 0;
    int64_t resume = 0;
    int64_t slice = 0;
    int64_t compact = 1;
    int64_t isolate_epilogue = 0;
    int64_t gram = 2;
    int64_t walk = 0;
};

// Test and measurement options (fault injection, the epilogue-isolated
// kernel) change results on purpose; a process must opt in to them through
// the environment variable DSEQ_ENABLE_TEST_OPTIONS=1 before setting one to a
// non-zero value.
bool test_options_enabled() {
    const char *v = std::getenv("DSEQ_ENABLE_TEST_OPTIONS");
    return v && std::strcmp(v, "1") == 0;
}
std::mutex g_opt_mu;
Options g_defaults;

int set_opt(Options &o, const char *name, int64_t v) {
    if (!name) return fail(DSEQ_EINVAL, "option name is NULL");
    const std::string n(name);
    if (n == "engine") {
        if (v != 0 && v != 1) return fail(DSEQ_EINVAL, "engine must be 0 or 1");
        o.engine = v;
    } else if (n == "tile_n") {
        if (v != 0 && (v < 32 || v > 256 || v % 32)) return fail(DSEQ_EINVAL, "tile_n must be 0 or a multiple of 32 in [32, 256]");
        o.tile_n = v;
    } else if (n == "tile_n2") {
        if (v != 0 && (v < 32 || v > 256 || v % 32)) return fail(DSEQ_EINVAL, "tile_n2 must be 0 or a multiple of 32 in [32, 256]");
        o.tile_n2 = v;
    } else if (n == "grid") {
        if (v < 0 || v > 65535) return fail(DSEQ_EINVAL, "grid out of range");
        o.grid = v;
    } else if (n == "timeout_ms") {
        if (v < 1 || v > 3600000) return fail(DSEQ_EINVAL, "timeout_ms out of range");
        o.timeout_ms = v;
    } else if (n == "resume") {
        if (v != 0 && v != 1) return fail(DSEQ_EINVAL, "resume must be 0 or 1");
        o.resume = v;
    } else if (n == "criterion") {
        if (v != 0 && v != 1) return fail(DSEQ_EINVAL, "criterion must be 0 (max-min) or 1 (centroid)");
        o.criterion = v;
    } else if (n == "storage") {
        if (v != 0 && v != 1) return fail(DSEQ_EINVAL, "storage must be 0 (split) or 1 (fp16)");
        o.storage = v;
    } else if (n == "pair") {
        if (v != 0 && v != 1) return fail(DSEQ_EINVAL, "pair must be 0 or 1");
        o.pair = v;
    } else if (n == "timeline") {
        if (v != 0 && v != 1) return fail(DSEQ_EINVAL, "timeline must be 0 or 1");
        o.timeline = v;
    } else if (n == "fault_skip_arrive" || n == "fault_skip_copy" || n == "isolate_epilogue") {
        if (v != 0 && v != 1) return fail(DSEQ_EINVAL, "%s must be 0 or 1", name);
        if (v != 0 && !test_options_enabled())
            return fail(DSEQ_EINVAL,
                        "%s is a test option that changes results; set DSEQ_ENABLE_TEST_OPTIONS=1 "
                        "in the environment to use it", name);
        (n == "fault_skip_arrive" ? o.fault_skip_arrive
         : n == "fault_skip_copy" ? o.fault_skip_copy
                                  : o.isolate_epilogue) = v;
    } else if (n == "compact") {
        if (v != 0 && v != 1) return fail(DSEQ_EINVAL, "compact must be 0 or 1");
        o.compact = v;
    } else if (n == "walk") {
        if (v < 0 || v > 3) return fail(DSEQ_EINVAL, "walk must be 0 (chosen), 1 (one CTA), 2 (cluster) or 3 (global memory)");
        o.walk = v;
    } else if (n == "gram") {
        if (v < 0 || v > 2) return fail(DSEQ_EINVAL, "gram must be 0 (never), 1 (always) or 2 (auto)");
        o.gram = v;
    } else if (n == "slice") {
        if (v < 0 || v > (int64_t(1) << 24)) return fail(DSEQ_EINVAL, "slice out of range");
        o.slice = v;
    } else {
        return fail(DSEQ_EINVAL, "unknown option '%s'", name);
    }
    return DSEQ_OK;
}

int64_t get_opt(const Options &o, const char *name) {
    if (!name) return -1;
    const std::string n(name);
    if (n == "engine") return o.engine;
    if (n == "tile_n") return o.tile_n;
    if (n == "tile_n2") return o.tile_n2;
    if (n == "grid") return o.grid;
    if (n == "timeout_ms") return o.timeout_ms;
    if (n == "fault_skip_arrive") return o.fault_skip_arrive;
    if (n == "slice") return o.slice;
    if (n == "compact") return o.compact;
    if (n == "fault_skip_copy") return o.fault_skip_copy;
    if (n == "timeline") return o.timeline;
    if (n == "pair") return o.pair;
    if (n == "storage") return o.storage;
    if (n == "criterion") return o.criterion;
    if (n == "resume") return o.resume;
    if (n == "isolate_epilogue") return o.isolate_epilogue;
    if (n == "gram") return o.gram;
    if (n == "walk") return o.walk;
    return -1;
}

// --------------------------------------------------------------------------
// device memory helpers
//
// Buffer cache: a context's buffers, when it is destroyed, and a call's
// staging buffers, once the call has synchronised, are idle; instead of
// cudaFree they go to a per-device cache (up to "cache_mb" in total per
// device; by default half of the device's memory), from which later
// allocations of a similar size are served.  A create / run / destroy cycle
// then maps and unmaps no device memory after the first: cudaMalloc of
// large buffers and cudaFree, which also synchronises the device, cost
// about a millisecond per page-1 cycle, and 60 ms per cycle at N = 131072,
// where G alone is 68.7 GB (its cudaFree 25-33 ms, the product 9 ms slower
// on freshly mapped pages).  A buffer released while work using it may
// still be queued keeps cudaFree.  A failed cudaMalloc empties the device's
// cache and retries once.
struct BufCache {
    std::mutex mu;
    std::multimap<size_t, void *> idle;  // bytes -> buffer
    size_t held = 0;
};
BufCache g_cache[64];
std::atomic<int64_t> g_cache_limit{-1};  // bytes; -1: half of each device's memory
std::atomic<size_t> g_dev_total[64];

// the cache's limit on device `dev`, in bytes
size_t cache_limit(int dev) {
    const int64_t l = g_cache_limit.load();
    if (l >= 0) return (size_t)l;
    size_t total = g_dev_total[dev].load();
    if (total == 0) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        total = prop.totalGlobalMem;
        g_dev_total[dev].store(total);
    }
    return total / 2;
}

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return dev >= 0 && dev < 64 ? dev : -1;
}

// a cached buffer of at least n bytes and not much larger, or nullptr
void *cache_take(int dev, size_t n, size_t &bytes) {
    if (dev < 0) return nullptr;
    BufCache &c = g_cache[dev];
    std::lock_guard<std::mutex> lk(c.mu);
    auto it = c.idle.lower_bound(n);
    if (it == c.idle.end() || it->first > 2 * n + (size_t(1) << 20)) return nullptr;
    void *p = it->second;
    bytes = it->first;
    c.held -= bytes;
    c.idle.erase(it);
    return p;
}

// keeps an idle buffer for reuse, or frees it when the cache is full
void cache_put(int dev, void *p, size_t bytes) {
    if (dev >= 0) {
        BufCache &c = g_cache[dev];
        std::lock_guard<std::mutex> lk(c.mu);
        if (c.held + bytes <= cache_limit(dev)) {
            c.idle.emplace(bytes, p);
            c.held += bytes;
            return;
        }
    }
    cudaFree(p);
}

// bytes the device's cache holds (free for this library's next allocations)
size_t cache_held(int dev) {
    if (dev < 0) return 0;
    BufCache &c = g_cache[dev];
    std::lock_guard<std::mutex> lk(c.mu);
    return c.held;
}

// frees the device's cached buffers down to `keep` bytes (largest first);
// keep = SIZE_MAX: down to the cache's limit
void cache_trim(int dev, size_t keep) {
    BufCache &c = g_cache[dev];
    std::lock_guard<std::mutex> lk(c.mu);
    if (c.held == 0) return;
    if (keep == SIZE_MAX) keep = cache_limit(dev);
    while (c.held > keep && !c.idle.empty()) {
        auto it = std::prev(c.idle.end());
        cudaFree(it->second);
        c.held -= it->first;
        c.idle.erase(it);
    }
}

struct DevBuf {
    void *p = nullptr;
    size_t bytes = 0;
    int dev = -1;
    int ensure(size_t n) {
        if (n <= bytes) return DSEQ_OK;
        release();
        const int d = current_device();
        size_t got = 0;
        if ((p = cache_take(d, n, got)) != nullptr) {
            bytes = got;
            dev = d;
            return DSEQ_OK;
        }
        cudaError_t e = cudaMalloc(&p, n);
        if (e != cudaSuccess && d >= 0) {
            cudaGetLastError();
            cache_trim(d, 0);
            e = cudaMalloc(&p, n);
        }
        if (e != cudaSuccess) {
            cudaGetLastError();
            p = nullptr;
            return fail(DSEQ_ENOMEM, "cudaMalloc of %zu bytes failed: %s", n, cudaGetErrorString(e));
        }
        bytes = n;
        dev = d;
        return DSEQ_OK;
    }
    // frees the buffer (cudaFree: safe while work using it may be queued)
    void release() {
        if (p) cudaFree(p);
        p = nullptr;
        bytes = 0;
    }
    // hands an idle buffer (no queued work uses it) to the cache
    void recycle() {
        if (p) cache_put(dev, p, bytes);
        p = nullptr;
        bytes = 0;
    }
    template <class T>
    T *as() const {
        return static_cast<T *>(p);
    }
};

// Where an array argument lives.  Device memory must belong to the current
// device (the one the call's kernels run on): a pointer into another GPU's
// memory would reach the kernels as plain loads and stores, which fault
// without peer access, so it is rejected before any work is enqueued.
// Managed memory counts as device memory; anything else as host memory.
int locate(const void *p, const char *what, bool &on_device) {
    on_device = false;
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return DSEQ_OK;
    }
    if (at.type == cudaMemoryTypeManaged) {
        on_device = true;
        return DSEQ_OK;
    }
    if (at.type != cudaMemoryTypeDevice) return DSEQ_OK;
    int cur = -1;
    CUDA_TRY(cudaGetDevice(&cur));
    if (at.device != cur)
        return fail(DSEQ_EINVAL, "%s is memory of device %d, but the current device is %d", what,
                    at.device, cur);
    on_device = true;
    return DSEQ_OK;
}

bool is_device_ptr(const void *p) {
    bool dev = false;
    return locate(p, "array", dev) == DSEQ_OK && dev;
}

// input array: the device pointer itself, or a staged device copy of host data
template <class T>
int stage_in(const T *src, size_t count, DevBuf &buf, const T *&dev, cudaStream_t st,
             const char *what) {
    bool on_device;
    TRY(locate(src, what, on_device));
    if (on_device) {
        dev = src;
        return DSEQ_OK;
    }
    TRY(buf.ensure(count * sizeof(T)));
    CUDA_TRY(cudaMemcpyAsync(buf.p, src, count * sizeof(T), cudaMemcpyHostToDevice, st));
    dev = buf.as<T>();
    return DSEQ_OK;
}

// host copy of a small argument array (for validation)
template <class T>
int to_host(const T *src, size_t count, std::vector<T> &out, cudaStream_t st,
            const char *what) {
    out.resize(count);
    if (count == 0) return DSEQ_OK;
    bool on_device;
    TRY(locate(src, what, on_device));
    if (on_device) {
        CUDA_TRY(cudaMemcpyAsync(out.data(), src, count * sizeof(T), cudaMemcpyDeviceToHost, st));
        CUDA_TRY(cudaStreamSynchronize(st));
    } else {
        std::memcpy(out.data(), src, count * sizeof(T));
    }
    return DSEQ_OK;
}

struct DeviceInfo {
    int sms = 0, l2 = 0;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

int device_info(int dev, DeviceInfo &info) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (dev < 0 || dev >= 64) return fail(DSEQ_ECUDA, "device ordinal %d out of range", dev);
    if (g_dev[dev].sms == 0) {
        CUDA_TRY(cudaDeviceGetAttribute(&g_dev[dev].sms, cudaDevAttrMultiProcessorCount, dev));
        CUDA_TRY(cudaDeviceGetAttribute(&g_dev[dev].l2, cudaDevAttrL2CacheSize, dev));
    }
    info = g_dev[dev];
    return DSEQ_OK;
}

// --------------------------------------------------------------------------
// tensor maps (driver entry point fetched at run time: no link against libcuda)
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int get_encoder(EncodeTiledFn &fn) {
    static std::mutex mu;
    static EncodeTiledFn cached = nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!cached) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        CUDA_TRY(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                  cudaEnableDefault, &q));
        if (q != cudaDriverEntryPointSuccess || !p)
            return fail(DSEQ_ECUDA, "cuTensorMapEncodeTiled entry point not found");
        cached = reinterpret_cast<EncodeTiledFn>(p);
    }
    fn = cached;
    return DSEQ_OK;
}

// 2-D fp16 map over a row-major [rows][cols] buffer, box = 32 columns (64 B,
// 64-byte swizzle) x box_rows rows; out-of-range rows read as zero.
int encode_f16_map(CUtensorMap &map, const void *base, int64_t cols, int64_t rows, int box_rows) {
    EncodeTiledFn fn;
    TRY(get_encoder(fn));
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kKBlock, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DSEQ_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return DSEQ_OK;
}

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Relative time of one work unit w candidate columns wide, from the phase
// timeline of the persistent kernel on GB300.  Split storage: a unit costs
// the same for any width up to 128 (the 128 query rows x 3 parts streamed
// from L2 bound it), and above that grows with the width rounded up to a
// multiple of 64 (a 224-wide MMA takes as long as a 256-wide one).  FP16
// storage: nearly flat (the epilogue bounds it).
double unit_cost(int w, bool f16) {
    if (f16) return 0.87 + 0.13 * w / 256.0;
    const int w64 = (w + 63) / 64 * 64;
    return std::max(0.77, w64 / 256.0);
}

// Chunk widths of the diversity plan: chunks j < n_wide are w1 columns wide,
// the rest w2 <= w1, covering ncols.  Units (blocks x chunks, chunk-major)
// are dealt round-robin to `workers`; the widths and split are those that
// minimise the most loaded worker's summed unit_cost (ties: fewer units,
// then wider tiles).  forced_w1 / forced_w2 > 0 pin a width (w1 alone pins a
// uniform plan).
void choose_widths(TcPlan &plan, int64_t blocks, int64_t ncols, int workers, bool f16,
                   int forced_w1, int forced_w2) {
    double best_cost = 1e300;
    int64_t best_units = INT64_MAX;
    int best_w1 = 256, best_w2 = 256, best_nw = 0, best_nn = 0;
    for (int w1 = 256; w1 >= 32; w1 -= 32) {
        if (forced_w1 > 0 && w1 != forced_w1) continue;
        for (int w2 = w1; w2 >= 32; w2 -= 32) {
            if (forced_w2 > 0 ? w2 != forced_w2 : (forced_w1 > 0 && w2 != w1)) continue;
            const int64_t max_wide = (ncols + w1 - 1) / w1;
            // all-narrow splits are the uniform plan of width w2; the narrow
            // chunks only balance the last rounds, so at most 64 of them are
            // considered (this bounds the search for very wide tables)
            const int64_t lo_wide =
                w2 == w1 ? max_wide : std::max<int64_t>(1, max_wide - (64 * w2 + w1 - 1) / w1);
            for (int64_t nw = lo_wide; nw <= max_wide; ++nw) {
                const int64_t rest = std::max<int64_t>(0, ncols - nw * w1);
                const int64_t nn = (rest + w2 - 1) / w2;
                const int64_t units = blocks * (nw + nn), wide = blocks * nw;
                const double c1 = unit_cost(w1, f16), c2 = unit_cost(w2, f16);
                double worst = 0.0;
                for (int k = 0; k < workers && k < units; ++k) {
                    const int64_t n_all = (units - 1 - k) / workers + 1;
                    const int64_t n_wide = k < wide ? (wide - 1 - k) / workers + 1 : 0;
                    worst = std::max(worst, n_wide * c1 + (n_all - n_wide) * c2);
                }
                const bool better = worst < best_cost - 1e-9 ||
                                    (worst < best_cost + 1e-9 && units < best_units);
                if (better) {
                    best_cost = worst;
                    best_units = units;
                    best_w1 = w1;
                    best_w2 = w2;
                    best_nw = (int)nw;
                    best_nn = (int)nn;
                }
            }
        }
    }
    plan.tile_n = best_w1;
    plan.tile_n2 = best_nn == 0 ? best_w1 : best_w2;
    plan.n_wide = best_nw;
    plan.n_chunk = best_nw + best_nn;
}

int read_status(int *status_dev, cudaStream_t st) {
    int s = 0;
    CUDA_TRY(cudaMemcpyAsync(&s, status_dev, sizeof(int), cudaMemcpyDeviceToHost, st));
    CUDA_TRY(cudaStreamSynchronize(st));
    if (s == 0) return DSEQ_OK;
    if (s & kStatusNonFinite) return fail(DSEQ_ENONFINITE, "non-finite value or zero-norm row in input");
    if (s & kStatusBadIndex) return fail(DSEQ_EINVAL, "BMU index out of range [0, M)");
    if (s & (kStatusBarrierTimeout | kStatusPipeTimeout))
        return fail(DSEQ_ETIMEOUT, "device wait timed out (status 0x%x)", s);
    return fail(DSEQ_EINTERNAL, "device consistency check failed (status 0x%x)", s);
}

// CUDA events of finished timers, kept per thread and device for reuse
// (creating and destroying them cost several microseconds a call)
struct EventPool {
    std::vector<std::pair<int, cudaEvent_t>> idle;
    ~EventPool() {
        for (auto &e : idle) cudaEventDestroy(e.second);
    }
};
thread_local EventPool g_events;

int event_take(cudaEvent_t &ev) {
    const int dev = current_device();
    for (size_t i = g_events.idle.size(); i-- > 0;)
        if (g_events.idle[i].first == dev) {
            ev = g_events.idle[i].second;
            g_events.idle.erase(g_events.idle.begin() + (std::ptrdiff_t)i);
            return DSEQ_OK;
        }
    CUDA_TRY(cudaEventCreate(&ev));
    return DSEQ_OK;
}

struct EventTimer {
    cudaEvent_t a = nullptr, b = nullptr;
    int dev = -1;
    ~EventTimer() {
        for (cudaEvent_t e : {a, b})
            if (e) {
                if (g_events.idle.size() < 16)
                    g_events.idle.emplace_back(dev, e);
                else
                    cudaEventDestroy(e);
            }
    }
    int start(cudaStream_t st) {
        dev = current_device();
        if (!a) TRY(event_take(a));
        if (!b) TRY(event_take(b));
        CUDA_TRY(cudaEventRecord(a, st));
        return DSEQ_OK;
    }
    int stop(cudaStream_t st) {
        CUDA_TRY(cudaEventRecord(b, st));
        return DSEQ_OK;
    }
    int64_t ns() {
        float ms = 0.f;
        if (!a || !b || cudaEventElapsedTime(&ms, a, b) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return (int64_t)(ms * 1.0e6);
    }
};

}  // namespace

// ----------------------------------------------------------------------------
// Host helpers shared with the allocation-free entry point (noalloc.cu).
namespace dseq {
namespace host {
int fail_msg(int code, const char *msg) { return fail(code, "%s", msg); }
void clear_error() {
    g_err.clear();
    g_stats = Stats();
}
int locate_ptr(const void *p, const char *what, bool &on_device) {
    return locate(p, what, on_device);
}
int sm_count(int dev, int *sms) {
    DeviceInfo info;
    TRY(device_info(dev, info));
    *sms = info.sms;
    return DSEQ_OK;
}
int encode_map(CUtensorMap &map, const void *base, int64_t cols, int64_t rows, int box_rows) {
    return encode_f16_map(map, base, cols, rows, box_rows);
}
int read_device_status(int *status_dev, cudaStream_t st) { return read_status(status_dev, st); }
}  // namespace host
}  // namespace dseq

// ----------------------------------------------------------------------------
struct dseq_ctx {
    int device = 0;
    int64_t N = 0;
    int32_t D = 0, Dp = 0;
    Options opt;
    DevBuf e_unit, e_split, e_f16, rn, nrm;
    // run workspace
    DevBuf m, held, keys, q, q_rn, csum, c_exp, status, barrier, starts, mask, picks, trace_slot, timeline;
    // global-mask compaction: the unmasked rows' tables and the index maps
    DevBuf col_map, comp_of, e_split_c, e_f16_c, rn_c;
    // Gram engine: G (N x Np), the table split twice for the Gram product,
    // the sequences' newest rows
    DevBuf gram, g_xs, g_ws, g_xn, g_wn, g_xi, g_wi, g_cur, g_u16;
    int64_t timeline_iters = 0, timeline_grid = 0;
    int csum_shift = kNoShift;  // fixed-point scale of the centroid sums, set on first use
    // state left on the device by the last successful run, for "resume"
    bool has_state = false;
    int64_t state_picks = 0;  // picks per sequence made so far
    int64_t state_sig = -1;   // engine / pair / storage / criterion of that run
    TcPlan state_plan{};
    bool state_gram = false;  // the last run used the Gram engine
    int state_walk = 0;       // and kept its running minima there (gram_walk_place)
    std::vector<int32_t> state_starts;
    std::vector<uint8_t> state_mask;
    ~dseq_ctx() {
        DevBuf *all[] = {&e_unit, &e_split, &e_f16,  &rn,      &nrm,    &m,
                         &held,   &keys,    &q,      &q_rn,    &csum,   &c_exp,  &status, &barrier,
                         &starts, &mask,    &picks,  &trace_slot, &timeline,
                         &col_map, &comp_of, &e_split_c, &e_f16_c, &rn_c,
                         &gram, &g_xs, &g_ws, &g_xn, &g_wn, &g_xi, &g_wi, &g_cur, &g_u16};
        // idle: calls on a context do not overlap, and each one synchronised;
        // the largest first, so that the cache keeps the costliest to map
        std::sort(std::begin(all), std::end(all),
                  [](const DevBuf *x, const DevBuf *y) { return x->bytes > y->bytes; });
        for (DevBuf *b : all) b->recycle();
    }
};

extern "C" {

const char *dseq_last_error(void) { return g_err.c_str(); }

int64_t dseq_last_stat(const char *name) {
    if (!name) return -1;
    const std::string n(name);
    if (n == "units") return g_stats.units;
    if (n == "tile_n") return g_stats.tile_n;
    if (n == "tile_n2") return g_stats.tile_n2;
    if (n == "n_wide") return g_stats.n_wide;
    if (n == "grid") return g_stats.grid;
    if (n == "launches") return g_stats.launches;
    if (n == "kernel_ns") return g_stats.kernel_ns;
    if (n == "update_ns") return g_stats.update_ns;
    if (n == "gram") return g_stats.gram;
    if (n == "gram_ns") return g_stats.gram_ns;
    if (n == "walk_ns") return g_stats.walk_ns;
    if (n == "walk") return g_stats.walk;
    return -1;
}

int dseq_set_option(dseq_ctx *ctx, const char *name, int64_t value) {
    g_err.clear();
    if (name && std::string(name) == "cache_mb") {
        if (ctx) return fail(DSEQ_EINVAL, "cache_mb is a process-wide option (ctx must be NULL)");
        if (value < -1 || value > (int64_t(1) << 24)) return fail(DSEQ_EINVAL, "cache_mb out of range");
        g_cache_limit.store(value < 0 ? -1 : value << 20);
        for (int d = 0; d < 64; ++d) cache_trim(d, SIZE_MAX);
        return DSEQ_OK;
    }
    if (ctx) return set_opt(ctx->opt, name, value);
    std::lock_guard<std::mutex> lk(g_opt_mu);
    return set_opt(g_defaults, name, value);
}

int64_t dseq_get_option(dseq_ctx *ctx, const char *name) {
    if (name && std::string(name) == "cache_mb") return ctx ? -1 : g_cache_limit.load() >> 20;
    if (ctx) return get_opt(ctx->opt, name);
    std::lock_guard<std::mutex> lk(g_opt_mu);
    return get_opt(g_defaults, name);
}

int dseq_create(const float *table, int64_t N, int32_t D, int table_on_device, void *cuda_stream,
                dseq_ctx **out) {
    (void)table_on_device;
    g_err.clear();
    if (!out) return fail(DSEQ_EINVAL, "out is NULL");
    *out = nullptr;
    if (!table) return fail(DSEQ_EINVAL, "table is NULL");
    if (N < 1 || N >= (int64_t(1) << 31)) return fail(DSEQ_EINVAL, "N=%lld out of range", (long long)N);
    if (D < 1 || D > 16384) return fail(DSEQ_EINVAL, "D=%d out of range", D);
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    dseq_ctx *ctx = new dseq_ctx();
    {
        std::lock_guard<std::mutex> lk(g_opt_mu);
        ctx->opt = g_defaults;
    }
    auto bail = [&](int code) {
        delete ctx;
        return code;
    };
    cudaError_t e = cudaGetDevice(&ctx->device);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete ctx;
        return fail(DSEQ_ECUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    }
    ctx->N = N;
    ctx->D = D;
    ctx->Dp = (int32_t)round_up(D, kKBlock);
    int r;
    if ((r = ctx->e_unit.ensure((size_t)N * ctx->Dp * sizeof(float))) != DSEQ_OK) return bail(r);
    if ((r = ctx->e_split.ensure((size_t)N * 2 * ctx->Dp * sizeof(__half))) != DSEQ_OK) return bail(r);
    if ((r = ctx->e_f16.ensure((size_t)N * ctx->Dp * sizeof(__half))) != DSEQ_OK) return bail(r);
    if ((r = ctx->rn.ensure((size_t)N * sizeof(float))) != DSEQ_OK) return bail(r);
    if ((r = ctx->nrm.ensure((size_t)N * sizeof(float))) != DSEQ_OK) return bail(r);
    if ((r = ctx->status.ensure(sizeof(int))) != DSEQ_OK) return bail(r);
    DevBuf staged;
    const float *tdev = nullptr;
    if ((r = stage_in(table, (size_t)N * D, staged, tdev, st, "table")) != DSEQ_OK) return bail(r);
    e = cudaMemsetAsync(ctx->status.p, 0, sizeof(int), st);
    if (e == cudaSuccess) {
        launch_table_prepare(tdev, N, D, ctx->Dp, ctx->e_unit.as<float>(),
                             ctx->e_split.as<__half>(), ctx->nrm.as<float>(),
                             ctx->status.as<int>(), st);
        launch_table_prepare_f16(tdev, N, D, ctx->Dp, ctx->e_f16.as<__half>(),
                                 ctx->rn.as<float>(), ctx->status.as<int>(), st);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return bail(fail(cuda_code(e), "table preparation failed: %s", cudaGetErrorString(e)));
    }
    if ((r = read_status(ctx->status.as<int>(), st)) != DSEQ_OK) return bail(r);
    staged.recycle();  // the stream was synchronised by read_status
    *out = ctx;
    return DSEQ_OK;
}

void dseq_destroy(dseq_ctx *ctx) { delete ctx; }

int dseq_get_timeline(dseq_ctx *ctx, int64_t *out, int64_t capacity, int32_t *iters,
                      int32_t *grid) {
    g_err.clear();
    if (!ctx || !iters || !grid) return fail(DSEQ_EINVAL, "NULL argument");
    *iters = (int32_t)ctx->timeline_iters;
    *grid = (int32_t)ctx->timeline_grid;
    const int64_t n = ctx->timeline_iters * ctx->timeline_grid * kTimelineSlots;
    if (n == 0 || !out) return DSEQ_OK;
    if (capacity < n) return fail(DSEQ_EINVAL, "timeline needs %lld slots", (long long)n);
    CUDA_TRY(cudaMemcpy(out, ctx->timeline.p, (size_t)n * sizeof(int64_t), cudaMemcpyDeviceToHost));
    return DSEQ_OK;
}

// Whether the Gram engine is expected to beat the per-iteration contraction
// for this run, and fits in free_bytes of device memory.  The estimate
// takes the split contraction at about 500 TFLOP/s (fp32-equivalent) and
// HBM at about 5.5 TB/s: the Gram product costs 2 N^2 D, the walk one row
// of G per sequence-iteration (and the running minima when a row of them
// does not fit on chip), the scan 2 B N D per iteration.
static bool gram_pays(int64_t N, int64_t Dp, int64_t B, int64_t L, size_t free_bytes) {
    const int64_t Np = round_up(N, 32);
    const double need = (double)N * Np * 4.0 + (double)N * 5.0 * Dp * 2.0 + (double)B * Np * 4.0 +
                        (256.0 * 1024 * 1024);
    if (need > 0.8 * (double)free_bytes) return false;
    const double rt = 5.0e14, rb = 5.5e12;
    // running minima on chip (one CTA's registers or shared memory, or a
    // cluster's) cost no traffic; in global memory they are read and
    // written every iteration
    const bool smem = gram_walk_place(Np) != 3;
    const double t_gram = 2.0 * N * Np * Dp / rt + N * Np * 4.0 / rb +
                          (double)L * B * Np * 4.0 * (smem ? 1.0 : 2.2) / rb + 3.0e-5;
    const double t_scan = 2.0 * B * N * Dp * (double)L / rt;
    return t_gram < 0.9 * t_scan;
}

static int run_impl(dseq_ctx *ctx, const int32_t *starts, int32_t B, int32_t L,
                    const uint8_t *mask, int32_t *picks, const int32_t *trace_seqs,
                    int32_t n_trace, float *trace_mindist, void *cuda_stream) {
    g_err.clear();
    g_stats = Stats();
    if (!ctx) return fail(DSEQ_EINVAL, "ctx is NULL");
    if (!starts) return fail(DSEQ_EINVAL, "starts is NULL");
    if (!picks && L > 0) return fail(DSEQ_EINVAL, "picks is NULL");
    if (B < 1) return fail(DSEQ_EINVAL, "B=%d must be >= 1", B);
    if (L < 0) return fail(DSEQ_EINVAL, "L=%d must be >= 0", L);
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    int cur = -1;
    CUDA_TRY(cudaGetDevice(&cur));
    if (cur != ctx->device) return fail(DSEQ_EINVAL, "context belongs to device %d, current is %d", ctx->device, cur);
    const int64_t N = ctx->N;

    // ---- validate on the host ----
    std::vector<int32_t> h_starts;
    TRY(to_host(starts, (size_t)B, h_starts, st, "starts"));
    std::vector<uint8_t> h_mask;
    if (mask) TRY(to_host(mask, (size_t)N, h_mask, st, "mask"));
    // resume: continue the last run on this context from the state it left
    // on the device (same sequences, mask and mode; picks continue)
    const bool resume = ctx->opt.resume != 0;
    const int64_t sig = ctx->opt.compact * 10000 + ctx->opt.engine * 1000 + ctx->opt.pair * 100 +
                        ctx->opt.storage * 10 + ctx->opt.criterion;
    if (resume) {
        if (!ctx->has_state) return fail(DSEQ_EINVAL, "resume: no earlier run state on this context");
        if (sig != ctx->state_sig) return fail(DSEQ_EINVAL, "resume: engine, pair, storage, criterion or compact differ from the earlier run");
        if (h_starts != ctx->state_starts) return fail(DSEQ_EINVAL, "resume: starts differ from the earlier run");
        if (h_mask != ctx->state_mask) return fail(DSEQ_EINVAL, "resume: mask differs from the earlier run");
    }
    const int64_t done_before = resume ? ctx->state_picks : 0;
    int64_t n_masked = 0;
    if (mask)
        for (int64_t c = 0; c < N; ++c) n_masked += h_mask[c] != 0;
    {
        std::vector<uint8_t> seen((size_t)N, 0);
        for (int32_t b = 0; b < B; ++b) {
            const int32_t s = h_starts[b];
            if (s < 0 || s >= N) return fail(DSEQ_EINVAL, "starts[%d]=%d out of range [0, %lld)", b, s, (long long)N);
            if (seen[s]) return fail(DSEQ_EINVAL, "start %d repeated", s);
            seen[s] = 1;
            const int64_t avail = N - n_masked - ((mask && h_mask[s]) ? 0 : 1) - done_before;
            if (L > avail) return fail(DSEQ_EINVAL, "L=%d exceeds the %lld candidates left to sequence %d", L, (long long)avail, b);
        }
    }
    if (ctx->opt.isolate_epilogue &&
        (ctx->opt.engine != 0 || ctx->opt.criterion != 0 || resume))
        return fail(DSEQ_EINVAL, "isolate_epilogue runs the tensor-core max-min kernel only, without resume");
    if (!resume) ctx->has_state = false;
    std::vector<int32_t> h_slot;
    // CTA pairs work on pairs of 128-sequence blocks: pad B to 256 there
    const bool pair = ctx->opt.engine == 0 && ctx->opt.pair != 0;
    const int64_t Bp = round_up(B, pair ? 2 * kUnitRows : kUnitRows);
    if (n_trace > 0) {
        if (!trace_seqs || !trace_mindist) return fail(DSEQ_EINVAL, "trace arrays are NULL");
        bool trace_dev;
        TRY(locate(trace_mindist, "trace_mindist", trace_dev));
        if (!trace_dev) return fail(DSEQ_EINVAL, "trace_mindist must be device memory");
        std::vector<int32_t> h_tr;
        TRY(to_host(trace_seqs, (size_t)n_trace, h_tr, st, "trace_seqs"));
        h_slot.assign((size_t)Bp, -1);
        for (int32_t k = 0; k < n_trace; ++k) {
            const int32_t b = h_tr[k];
            if (b < 0 || b >= B || h_slot[b] >= 0) return fail(DSEQ_EINVAL, "trace_seqs[%d]=%d invalid or repeated", k, b);
            h_slot[b] = k;
        }
    } else if (n_trace < 0) {
        return fail(DSEQ_EINVAL, "n_trace < 0");
    }
    if (L == 0) return DSEQ_OK;

    // ---- stage the small inputs and outputs ----
    TRY(ctx->starts.ensure((size_t)B * sizeof(int32_t)));
    CUDA_TRY(cudaMemcpyAsync(ctx->starts.p, h_starts.data(), (size_t)B * sizeof(int32_t), cudaMemcpyHostToDevice, st));
    const uint8_t *d_mask = nullptr;
    if (mask) {
        TRY(ctx->mask.ensure((size_t)N));
        CUDA_TRY(cudaMemcpyAsync(ctx->mask.p, h_mask.data(), (size_t)N, cudaMemcpyHostToDevice, st));
        d_mask = ctx->mask.as<uint8_t>();
    }
    const int32_t *d_slot = nullptr;
    if (n_trace > 0) {
        TRY(ctx->trace_slot.ensure((size_t)Bp * sizeof(int32_t)));
        CUDA_TRY(cudaMemcpyAsync(ctx->trace_slot.p, h_slot.data(), (size_t)Bp * sizeof(int32_t), cudaMemcpyHostToDevice, st));
        d_slot = ctx->trace_slot.as<int32_t>();
    }
    bool picks_on_dev;
    TRY(locate(picks, "picks", picks_on_dev));
    int32_t *d_picks = picks;
    if (!picks_on_dev) {
        TRY(ctx->picks.ensure((size_t)B * L * sizeof(int32_t)));
        d_picks = ctx->picks.as<int32_t>();
    }
    TRY(ctx->keys.ensure((size_t)Bp * sizeof(unsigned long long)));
    // cross-CTA counters of the persistent kernel: [1..2] done, [3..4] committed
    TRY(ctx->barrier.ensure(8 * sizeof(unsigned)));
    CUDA_TRY(cudaMemsetAsync(ctx->status.p, 0, sizeof(int), st));

    DeviceInfo info;
    TRY(device_info(ctx->device, info));
    EventTimer timer;

    // the Gram engine (max-min; split or fp16 storage: with fp16 storage G
    // holds the distances between the stored rows) when it pays, or when
    // asked; a resumed run continues on the engine of the run it resumes
    bool use_gram = false;
    if (resume) {
        use_gram = ctx->state_gram;
    } else if (ctx->opt.engine == 0 && ctx->opt.criterion == 0 &&
               ctx->opt.isolate_epilogue == 0 && ctx->opt.timeline == 0 && ctx->opt.gram != 0) {
        if (ctx->opt.gram == 1) {
            use_gram = true;
        } else {
            // the context already holds buffers for G and the running
            // minima of this shape: memory is not the question any more
            const int64_t Np = round_up(N, 32);
            size_t free_b = 0, total_b = 0;
            if (ctx->gram.bytes >= (size_t)N * Np * sizeof(float) &&
                ctx->m.bytes >= (size_t)B * Np * sizeof(float)) {
                free_b = SIZE_MAX / 2;
            } else if (cudaMemGetInfo(&free_b, &total_b) != cudaSuccess) {
                cudaGetLastError();
                free_b = 0;
            } else {
                free_b += cache_held(current_device());  // ours to reuse
            }
            use_gram = gram_pays(N, ctx->Dp, B, L, free_b);
        }
    }

    if (use_gram) {
        // ---- Gram engine: G = E E^T on the tensor cores, then the walk ----
        const int64_t Np = round_up(N, 32);
        // where the running minima live: chosen from the row length, or the
        // "walk" option (a one-CTA row must fit its shared memory, the
        // largest place a forced one-CTA walk has)
        int place = ctx->opt.walk > 0 ? (int)ctx->opt.walk : gram_walk_place(Np);
        if (resume) place = ctx->state_walk;
        if (place == 1 && (size_t)Np * sizeof(float) > kGramWalkSmemMax)
            return fail(DSEQ_EINVAL, "walk=1: a row of %lld running minima does not fit one CTA's shared memory", (long long)Np);
        if (place == 2 && (size_t)Np * sizeof(float) > kGramWalkClusterMax)
            return fail(DSEQ_EINVAL, "walk=2: a row of %lld running minima does not fit a cluster's shared memory", (long long)Np);
        const int Dp = ctx->Dp;
        TRY(ctx->gram.ensure((size_t)N * Np * sizeof(float)));
        TRY(ctx->g_xs.ensure((size_t)N * kBmuPartsX * Dp * sizeof(__half)));
        TRY(ctx->g_ws.ensure((size_t)N * kBmuPartsW * Dp * sizeof(__half)));
        TRY(ctx->g_xn.ensure((size_t)N * sizeof(float)));
        TRY(ctx->g_wn.ensure((size_t)N * sizeof(float)));
        TRY(ctx->g_xi.ensure((size_t)N * sizeof(float)));
        TRY(ctx->g_wi.ensure((size_t)N * sizeof(float)));
        TRY(ctx->g_cur.ensure((size_t)B * sizeof(int32_t)));
        if (ctx->opt.storage != 0) TRY(ctx->g_u16.ensure((size_t)N * Dp * sizeof(float)));
        TRY(ctx->m.ensure((size_t)B * Np * sizeof(float)));
        BmuArgs ga;
        std::memset(&ga, 0, sizeof ga);
        ga.x_split = ctx->g_xs.as<__half>();
        ga.w_split = ctx->g_ws.as<__half>();
        ga.xn = ctx->g_xn.as<float>();
        ga.wn = ctx->g_wn.as<float>();
        ga.x_inv_scale = ctx->g_xi.as<float>();
        ga.w_inv_scale = ctx->g_wi.as<float>();
        ga.status = ctx->status.as<int>();
        ga.n = N;
        ga.M = N;
        ga.D = Dp;
        ga.Dp = Dp;
        ga.timeout_ns = (uint64_t)ctx->opt.timeout_ms * 1000000ull;
        ga.gram = ctx->gram.as<float>();
        ga.gram_ld = Np;
        TcPlan gp{};
        gp.pair = 1;
        gp.n_beta = (int)((N + kUnitRows - 1) / kUnitRows);
        gp.n_beta += gp.n_beta & 1;
        gp.set_uniform(256, N);
        gp.grid = 2 * (int)std::max<int64_t>(1, std::min<int64_t>(info.sms / 2, (int64_t)(gp.n_beta / 2) * gp.n_chunk));
        CUtensorMap tx, tw;
        TRY(encode_f16_map(tx, ga.x_split, kBmuPartsX * Dp, N, kUnitRows));
        TRY(encode_f16_map(tw, ga.w_split, kBmuPartsW * Dp, N, gp.tile_n / 2));
        GramWalkArgs wa;
        std::memset(&wa, 0, sizeof wa);
        wa.G = ctx->gram.as<float>();
        wa.m = ctx->m.as<float>();
        wa.cur = ctx->g_cur.as<int32_t>();
        wa.picks = d_picks;
        wa.trace_slot = d_slot;
        wa.trace = trace_mindist;
        wa.status = ctx->status.as<int>();
        wa.N = N;
        wa.Np = Np;
        wa.B = B;
        wa.L = L;
        wa.place = place;
        wa.timeout_ns = (uint64_t)ctx->opt.timeout_ms * 1000000ull;
        ctx->state_walk = place;
        EventTimer mid;
        TRY(timer.start(st));
        // the table's unit rows, split twice (the sample and codebook sides);
        // with fp16 storage the stored rows themselves (exact in the split,
        // so every product is exact), their inverse norms folded into the
        // product's per-row rescaling
        const float *unit = ctx->e_unit.as<float>();
        if (ctx->opt.storage != 0) {
            launch_f16_rows(ctx->e_f16.as<__half>(), N, Dp, ctx->g_u16.as<float>(), st);
            unit = ctx->g_u16.as<float>();
        }
        launch_bmu_prepare(unit, N, Dp, Dp, 0, ctx->g_xs.as<__half>(),
                           ctx->g_xn.as<float>(), ctx->g_xi.as<float>(), ga.status, st);
        launch_bmu_prepare(unit, N, Dp, Dp, 1, ctx->g_ws.as<__half>(),
                           ctx->g_wn.as<float>(), ctx->g_wi.as<float>(), ga.status, st);
        if (ctx->opt.storage != 0)
            launch_scale_rows(ctx->g_xi.as<float>(), ctx->g_wi.as<float>(), ctx->rn.as<float>(), N, st);
        CUDA_TRY(cudaGetLastError());
        CUDA_TRY(launch_tc_gram(ga, gp, tx, tw, st));
        TRY(mid.start(st));
        if (!resume) {
            if (place != 3) {
                // the walk sets up its running minima on chip itself
                wa.starts = ctx->starts.as<int32_t>();
                wa.mask = d_mask;
            } else {
                launch_gram_walk_init(wa, ctx->starts.as<int32_t>(), d_mask, st);
            }
        }
        CUDA_TRY(cudaGetLastError());
        CUDA_TRY(launch_gram_walk(wa, st));
        TRY(timer.stop(st));
        TRY(mid.stop(st));
        g_stats.gram = 1;
        g_stats.walk = place;
        g_stats.units = B;
        g_stats.grid = B;
        g_stats.launches = ((resume || place != 3) ? 4 : 5) + (ctx->opt.storage != 0 ? 2 : 0);
        {
            const int rs = read_status(ctx->status.as<int>(), st);
            if (rs != DSEQ_OK) {
                ctx->has_state = false;
                return rs;
            }
        }
        // timer: the whole engine; mid: from the end of the Gram product
        g_stats.walk_ns = mid.ns();
        g_stats.gram_ns = std::max<int64_t>(0, timer.ns() - g_stats.walk_ns);
    } else if (ctx->opt.engine == 0) {
        // ---- tensor-core persistent kernel ----
        const bool f16 = ctx->opt.storage == 1;
        // a global mask that removes at least 1/16 of the table: scan only
        // the unmasked rows (option "compact"); picks are mapped back to
        // table rows, ties still go to the lowest table row (the map is
        // increasing), and results are identical to the full scan
        const bool compact = mask && ctx->opt.compact != 0 && n_masked * 16 >= N;
        int64_t Nk = N;
        if (compact) {
            std::vector<int32_t> h_map, h_comp((size_t)N, -1);
            h_map.reserve((size_t)(N - n_masked));
            for (int64_t c = 0; c < N; ++c)
                if (!h_mask[c]) {
                    h_comp[c] = (int32_t)h_map.size();
                    h_map.push_back((int32_t)c);
                }
            Nk = (int64_t)h_map.size();
            TRY(ctx->col_map.ensure((size_t)Nk * sizeof(int32_t)));
            TRY(ctx->comp_of.ensure((size_t)N * sizeof(int32_t)));
            CUDA_TRY(cudaMemcpyAsync(ctx->col_map.p, h_map.data(), (size_t)Nk * sizeof(int32_t), cudaMemcpyHostToDevice, st));
            CUDA_TRY(cudaMemcpyAsync(ctx->comp_of.p, h_comp.data(), (size_t)N * sizeof(int32_t), cudaMemcpyHostToDevice, st));
            const int32_t *d_map = ctx->col_map.as<int32_t>();
            if (f16) {
                TRY(ctx->e_f16_c.ensure((size_t)Nk * ctx->Dp * sizeof(__half)));
                TRY(ctx->rn_c.ensure((size_t)Nk * sizeof(float)));
                launch_gather_rows(ctx->e_f16.p, ctx->e_f16_c.p, d_map, Nk, (int64_t)ctx->Dp * sizeof(__half), st);
                launch_gather_rows(ctx->rn.p, ctx->rn_c.p, d_map, Nk, sizeof(float), st);
            } else {
                TRY(ctx->e_split_c.ensure((size_t)Nk * 2 * ctx->Dp * sizeof(__half)));
                launch_gather_rows(ctx->e_split.p, ctx->e_split_c.p, d_map, Nk,
                                   (int64_t)2 * ctx->Dp * sizeof(__half), st);
            }
            CUDA_TRY(cudaGetLastError());
        }
        TcPlan plan{};
        plan.n_beta = (int)(Bp / kUnitRows);
        plan.pair = pair ? 1 : 0;
        // The persistent grid: the "grid" option as given, else as many CTAs
        // of this kernel variant as can be co-resident (its own occupancy:
        // thread count and shared memory).  A grid beyond that is refused by
        // the cooperative launch and reported as DSEQ_ELAUNCH.
        int grid_cap = 0;
        if (ctx->opt.grid > 0) {
            grid_cap = (int)ctx->opt.grid;
        } else if (!resume) {
            grid_cap = tc_dseq_max_grid(pair, f16, ctx->opt.criterion != 0);
            if (grid_cap < (pair ? 2 : 1))
                return fail(DSEQ_ELAUNCH, "no %s of this kernel variant fits on the device",
                            pair ? "CTA pair" : "CTA");
        }
        if (resume) {
            plan = ctx->state_plan;  // the running-minimum layout depends on it
        } else if (pair) {
            // whole clusters of two
            grid_cap = std::max(2, grid_cap / 2 * 2);
            choose_widths(plan, plan.n_beta / 2, Nk, grid_cap / 2, ctx->opt.storage == 1,
                          (int)ctx->opt.tile_n, (int)ctx->opt.tile_n2);
            plan.grid = 2 * (int)std::min<int64_t>(grid_cap / 2, (int64_t)(plan.n_beta / 2) * plan.n_chunk);
        } else {
            choose_widths(plan, plan.n_beta, Nk, grid_cap, ctx->opt.storage == 1,
                          (int)ctx->opt.tile_n, (int)ctx->opt.tile_n2);
            plan.grid = (int)std::min<int64_t>(grid_cap, plan.units());
        }
        TRY(ctx->m.ensure((size_t)plan.n_beta * kUnitRows * plan.columns() * sizeof(float)));
        // split storage: queries [hi*2^12 | hi | lo], table [hi | lo];
        // fp16 storage: one fp16 part each, plus inverse norms
        // (the centroid query on fp16 storage is not an fp16 row: it keeps
        // (hi*2^12, lo))
        const int qparts = f16 ? (ctx->opt.criterion ? 2 : 1) : 3, eparts = f16 ? 1 : 2;
        const __half *t_split = compact ? ctx->e_split_c.as<__half>() : ctx->e_split.as<__half>();
        const __half *t_f16 = compact ? ctx->e_f16_c.as<__half>() : ctx->e_f16.as<__half>();
        const float *t_rn = compact ? ctx->rn_c.as<float>() : ctx->rn.as<float>();
        TRY(ctx->q.ensure((size_t)Bp * qparts * ctx->Dp * sizeof(__half)));
        TRY(ctx->q_rn.ensure((size_t)Bp * sizeof(float)));
        CUtensorMap tq, te;
        TRY(encode_f16_map(tq, ctx->q.p, qparts * ctx->Dp, Bp, kUnitRows));
        TRY(encode_f16_map(te, f16 ? (const void *)t_f16 : (const void *)t_split, eparts * ctx->Dp, Nk,
                           pair ? plan.tile_n / 2 : plan.tile_n));
        TcDseqArgs a{};
        a.e_split = t_split;
        a.q_split = ctx->q.as<__half>();
        a.e_f16 = f16 ? t_f16 : nullptr;
        a.rn = t_rn;
        a.e_split_full = ctx->e_split.as<__half>();
        a.e_f16_full = ctx->e_f16.as<__half>();
        a.rn_full = ctx->rn.as<float>();
        a.col_map = compact ? ctx->col_map.as<int32_t>() : nullptr;
        a.comp_of = compact ? ctx->comp_of.as<int32_t>() : nullptr;
        a.n_table = N;
        a.q_rn = ctx->q_rn.as<float>();
        a.centroid = (int)ctx->opt.criterion;
        if (a.centroid) {
            TRY(ctx->csum.ensure((size_t)Bp * ctx->Dp * sizeof(long long)));
            TRY(ctx->c_exp.ensure((size_t)Bp * sizeof(int)));
            a.csum = ctx->csum.as<long long>();
            a.c_exp = ctx->c_exp.as<int>();
            TRY(ctx->held.ensure((size_t)plan.n_beta * kUnitRows * plan.columns() / 32 * sizeof(unsigned)));
            a.held = ctx->held.as<unsigned>();
            if (ctx->csum_shift == kNoShift) {
                // every raw-row entry is below the largest row norm 2^e and a
                // sequence holds at most N rows: F = 62 - e - ceil(log2 N)
                std::vector<float> h_nrm;
                TRY(to_host(ctx->nrm.as<float>(), (size_t)N, h_nrm, st, "norms"));
                float mx = 0.0f;
                for (float v : h_nrm) mx = std::max(mx, v);
                int e = 0;
                std::frexp(mx, &e);
                int L = 0;
                while ((int64_t(1) << L) < N) ++L;
                ctx->csum_shift = 62 - e - L;
            }
            a.csum_shift = ctx->csum_shift;
        }
        a.e_unit = ctx->e_unit.as<float>();
        a.nrm = ctx->nrm.as<float>();
        a.m = ctx->m.as<float>();
        a.keys = ctx->keys.as<unsigned long long>();
        a.picks = d_picks;
        a.trace_slot = d_slot;
        a.trace = trace_mindist;
        a.status = ctx->status.as<int>();
        a.barrier = ctx->barrier.as<unsigned>();
        a.N = Nk;
        a.B = B;
        a.L = L;
        a.Dp = ctx->Dp;
        a.timeout_ns = (uint64_t)ctx->opt.timeout_ms * 1000000ull;
        a.fault_skip_arrive = (int)ctx->opt.fault_skip_arrive;
        a.isolate_epilogue = (int)ctx->opt.isolate_epilogue;
        // the split table stays L2-resident across iterations only if it is a
        // small part of L2; larger tables stream through once per iteration
        a.keep_table = (double)Nk * eparts * ctx->Dp * sizeof(__half) <= info.l2 / 3.0 ? 1 : 0;
        a.timeline = nullptr;
        ctx->timeline_iters = ctx->timeline_grid = 0;
        if (ctx->opt.timeline) {
            TRY(ctx->timeline.ensure((size_t)L * plan.grid * kTimelineSlots * sizeof(unsigned long long)));
            CUDA_TRY(cudaMemsetAsync(ctx->timeline.p, 0, (size_t)L * plan.grid * kTimelineSlots * sizeof(unsigned long long), st));
            a.timeline = ctx->timeline.as<unsigned long long>();
            ctx->timeline_iters = L;
            ctx->timeline_grid = plan.grid;
        }
        CUDA_TRY(cudaMemsetAsync(ctx->barrier.p, 0, 8 * sizeof(unsigned), st));
        if (!resume) launch_tc_dseq_init(a, plan, ctx->starts.as<int32_t>(), compact ? nullptr : d_mask, st);
        CUDA_TRY(cudaGetLastError());
        ctx->state_plan = plan;
        TRY(timer.start(st));
        {
            const cudaError_t le = launch_tc_dseq(a, plan, tq, te, st);
            if (le != cudaSuccess) {
                cudaGetLastError();
                ctx->has_state = false;
                return fail(DSEQ_ELAUNCH,
                            "cooperative launch of the persistent kernel (%d CTAs%s) refused: %s",
                            plan.grid, pair ? " in clusters of two" : "", cudaGetErrorString(le));
            }
        }
        TRY(timer.stop(st));
        g_stats.units = plan.units();
        g_stats.tile_n = plan.tile_n;
        g_stats.tile_n2 = plan.tile_n2;
        g_stats.n_wide = plan.n_wide;
        g_stats.grid = plan.grid;
        g_stats.launches = 2;
    } else {
        // ---- FP32 FFMA path, one launch pair per iteration ----
        if (ctx->opt.criterion != 0) return fail(DSEQ_EINVAL, "the FFMA engine runs the max-min criterion only");
        if (Bp / 128 > 65535) return fail(DSEQ_EINVAL, "the FFMA engine takes at most %d sequences", 65535 * 128);
        FfmaDseqArgs a;
        a.Nf = round_up(N, 128);
        a.Bp = (int)Bp;
        CUDA_TRY(ffma_configure());
        TRY(ctx->m.ensure((size_t)Bp * a.Nf * sizeof(float)));
        TRY(ctx->q.ensure((size_t)Bp * ctx->Dp * sizeof(float)));
        a.e_unit = ctx->e_unit.as<float>();
        a.q = ctx->q.as<float>();
        a.m = ctx->m.as<float>();
        a.keys = ctx->keys.as<unsigned long long>();
        a.picks = d_picks;
        a.trace_slot = d_slot;
        a.trace = trace_mindist;
        a.status = ctx->status.as<int>();
        a.N = N;
        a.B = B;
        a.L = L;
        a.Dp = ctx->Dp;
        if (!resume) launch_ffma_dseq_init(a, ctx->starts.as<int32_t>(), d_mask, st);
        CUDA_TRY(cudaGetLastError());
        TRY(timer.start(st));
        for (int t = 0; t < L; ++t) launch_ffma_dseq_iteration(a, t, st);
        CUDA_TRY(cudaGetLastError());
        TRY(timer.stop(st));
        g_stats.units = (Bp / 128) * (a.Nf / 128);
        g_stats.tile_n = 128;
        g_stats.grid = (int64_t)g_stats.units;
        g_stats.launches = 1 + 2 * (int64_t)L;
    }
    {
        const int rs = read_status(ctx->status.as<int>(), st);
        if (rs != DSEQ_OK) {
            ctx->has_state = false;
            return rs;
        }
    }
    // an epilogue-isolated run leaves meaningless state: nothing to resume
    ctx->has_state = ctx->opt.isolate_epilogue == 0;
    ctx->state_gram = use_gram;
    ctx->state_picks = done_before + L;
    ctx->state_sig = sig;
    ctx->state_starts = h_starts;
    ctx->state_mask = h_mask;
    g_stats.kernel_ns = timer.ns();
    if (!picks_on_dev) {
        CUDA_TRY(cudaMemcpyAsync(picks, d_picks, (size_t)B * L * sizeof(int32_t), cudaMemcpyDeviceToHost, st));
        CUDA_TRY(cudaStreamSynchronize(st));
    }
    return DSEQ_OK;
}

int dseq_run(dseq_ctx *ctx, const int32_t *starts, int32_t B, int32_t L, const uint8_t *mask,
             int32_t *picks, void *cuda_stream) {
    return run_impl(ctx, starts, B, L, mask, picks, nullptr, 0, nullptr, cuda_stream);
}

int dseq_run_trace(dseq_ctx *ctx, const int32_t *starts, int32_t B, int32_t L,
                   const uint8_t *mask, int32_t *picks, const int32_t *trace_seqs,
                   int32_t n_trace, float *trace_mindist, void *cuda_stream) {
    if (n_trace < 1) return fail(DSEQ_EINVAL, "n_trace must be >= 1");
    return run_impl(ctx, starts, B, L, mask, picks, trace_seqs, n_trace, trace_mindist,
                    cuda_stream);
}

// ----------------------------------------------------------------------------
// BMU: stateless entry point; its workspace is kept per device between calls.
namespace {
struct BmuWorkspace {
    std::mutex mu;
    DevBuf x_split, w_split, xn, wn, x_inv, w_inv, keys, status, x_stage, w_stage, idx_out, dist_out;
};
std::mutex g_bmu_mu;
BmuWorkspace *g_bmu[64] = {};
}  // namespace

}  // extern "C"

namespace {

int bmu_validate(int64_t n, int64_t M, int32_t D) {
    if (n < 1 || n >= (int64_t(1) << 31)) return fail(DSEQ_EINVAL, "n=%lld out of range", (long long)n);
    if (M < 1 || M >= (int64_t(1) << 31)) return fail(DSEQ_EINVAL, "M=%lld out of range", (long long)M);
    if (D < 1 || D > 16384) return fail(DSEQ_EINVAL, "D=%d out of range", D);
    return DSEQ_OK;
}

int current_device(int &dev) {
    CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(DSEQ_ECUDA, "device ordinal out of range");
    return DSEQ_OK;
}

Options default_options() {
    std::lock_guard<std::mutex> lk(g_opt_mu);
    return g_defaults;
}

BmuWorkspace *bmu_workspace(int dev) {
    std::lock_guard<std::mutex> lk(g_bmu_mu);
    if (!g_bmu[dev]) g_bmu[dev] = new BmuWorkspace();
    return g_bmu[dev];
}

// The BMU search on device operands; results into the device arrays d_idx,
// d_dist.  Leaves the stream running (status already read).
int bmu_core(const float *dX, int64_t n, const float *dW, int64_t M, int32_t D, int32_t *d_idx,
             float *d_dist, const Options &opt, const DeviceInfo &info, BmuWorkspace *ws,
             cudaStream_t st) {
    const int Dp = (int)round_up(D, kKBlock);
    TRY(ws->xn.ensure((size_t)n * sizeof(float)));
    TRY(ws->wn.ensure((size_t)M * sizeof(float)));
    TRY(ws->keys.ensure((size_t)n * sizeof(unsigned long long)));
    TRY(ws->status.ensure(sizeof(int)));
    CUDA_TRY(cudaMemsetAsync(ws->status.p, 0, sizeof(int), st));
    BmuArgs a;
    std::memset(&a, 0, sizeof a);
    a.X = dX;
    a.W = dW;
    a.xn = ws->xn.as<float>();
    a.wn = ws->wn.as<float>();
    a.keys = ws->keys.as<unsigned long long>();
    a.idx = d_idx;
    a.dist = d_dist;
    a.status = ws->status.as<int>();
    a.n = n;
    a.M = M;
    a.D = D;
    a.Dp = Dp;
    a.timeout_ns = (uint64_t)opt.timeout_ms * 1000000ull;
    a.fault_skip_copy = (int)opt.fault_skip_copy;
    EventTimer timer;
    launch_bmu_keys_init(a.keys, n, st);
    if (opt.engine == 0) {
        TRY(ws->x_split.ensure((size_t)n * kBmuPartsX * Dp * sizeof(__half)));
        TRY(ws->w_split.ensure((size_t)M * kBmuPartsW * Dp * sizeof(__half)));
        TRY(ws->x_inv.ensure((size_t)n * sizeof(float)));
        TRY(ws->w_inv.ensure((size_t)M * sizeof(float)));
        a.x_split = ws->x_split.as<__half>();
        a.w_split = ws->w_split.as<__half>();
        a.x_inv_scale = ws->x_inv.as<float>();
        a.w_inv_scale = ws->w_inv.as<float>();
        launch_bmu_prepare(dX, n, D, Dp, 0, ws->x_split.as<__half>(), ws->xn.as<float>(),
                           ws->x_inv.as<float>(), a.status, st);
        launch_bmu_prepare(dW, M, D, Dp, 1, ws->w_split.as<__half>(), ws->wn.as<float>(),
                           ws->w_inv.as<float>(), a.status, st);
        CUDA_TRY(cudaGetLastError());
        TcPlan plan{};
        plan.pair = opt.pair ? 1 : 0;
        plan.n_beta = (int)((n + kUnitRows - 1) / kUnitRows);
        if (plan.pair) plan.n_beta += plan.n_beta & 1;  // whole pairs of sample blocks
        int grid_cap = opt.grid > 0 ? (int)std::min<int64_t>(opt.grid, info.sms) : info.sms;
        plan.set_uniform(opt.tile_n > 0 ? (int)opt.tile_n : 256, M);
        if (plan.pair) {
            grid_cap = std::max(2, grid_cap / 2 * 2);
            plan.grid = 2 * (int)std::min<int64_t>(grid_cap / 2, plan.units() / 2);
        } else {
            plan.grid = (int)std::min<int64_t>(grid_cap, plan.units());
        }
        CUtensorMap tx, tw;
        TRY(encode_f16_map(tx, a.x_split, kBmuPartsX * Dp, n, kUnitRows));
        TRY(encode_f16_map(tw, a.w_split, kBmuPartsW * Dp, M, plan.pair ? plan.tile_n / 2 : plan.tile_n));
        TRY(timer.start(st));
        CUDA_TRY(launch_tc_bmu(a, plan, tx, tw, (int)opt.slice, st));
        TRY(timer.stop(st));
        g_stats.units = plan.units();
        g_stats.tile_n = plan.tile_n;
        g_stats.grid = plan.grid;
        g_stats.launches = 5;
    } else {
        if (((n + 127) / 128) * ((M + 127) / 128) > INT32_MAX)
            return fail(DSEQ_EINVAL, "the FFMA engine takes at most 2^31 - 1 tiles of 128 x 128");
        launch_row_sqnorm(dX, n, D, ws->xn.as<float>(), a.status, st);
        launch_row_sqnorm(dW, M, D, ws->wn.as<float>(), a.status, st);
        CUDA_TRY(cudaGetLastError());
        CUDA_TRY(ffma_configure());
        TRY(timer.start(st));
        launch_ffma_bmu(a, st);
        CUDA_TRY(cudaGetLastError());
        TRY(timer.stop(st));
        g_stats.units = ((n + 127) / 128) * ((M + 127) / 128);
        g_stats.tile_n = 128;
        g_stats.grid = g_stats.units;
        g_stats.launches = 5;
    }
    launch_bmu_finalize(a, st);
    CUDA_TRY(cudaGetLastError());
    TRY(read_status(a.status, st));
    g_stats.kernel_ns = timer.ns();
    return DSEQ_OK;
}

// ---- SOM neighbourhood update ------------------------------------------------
struct SomWorkspace {
    std::mutex mu;
    DevBuf S, cnt, off, tiles, order, T, Tc, status, x_stage, w_stage, bmu_stage, idx, dist;
};
std::mutex g_som_mu;
SomWorkspace *g_som[64] = {};

SomWorkspace *som_workspace(int dev) {
    std::lock_guard<std::mutex> lk(g_som_mu);
    if (!g_som[dev]) g_som[dev] = new SomWorkspace();
    return g_som[dev];
}

// Checks the map arguments and fills the window weights.
int som_validate(int64_t n, int32_t side_x, int32_t side_y, int32_t D, double sigma,
                 int32_t radius, SomArgs &a) {
    if (n < 0 || n >= (int64_t(1) << 31)) return fail(DSEQ_EINVAL, "n=%lld out of range", (long long)n);
    if (side_x < 1 || side_y < 1) return fail(DSEQ_EINVAL, "map sides must be >= 1");
    const int64_t M = (int64_t)side_x * side_y;
    if (M >= (int64_t(1) << 31)) return fail(DSEQ_EINVAL, "map of %lld neurons too large", (long long)M);
    if (D < 1 || D > 16384) return fail(DSEQ_EINVAL, "D=%d out of range", D);
    if (!(sigma >= 0.0) || !std::isfinite(sigma)) return fail(DSEQ_EINVAL, "sigma must be finite and >= 0");
    if (radius < 0 || radius > kSomMaxRadius)
        return fail(DSEQ_EINVAL, "radius=%d out of range [0, %d]", radius, kSomMaxRadius);
    // the corner weight g(R)^2 = exp(-R^2 / sigma^2) must stay a normal fp32
    if (sigma > 0.0 && (double)radius > 9.0 * sigma)
        return fail(DSEQ_EINVAL, "radius=%d exceeds 9 * sigma (window weights would underflow fp32)", radius);
    // one CTA per (32 dimensions, 128 neurons of a row) and per (32 dimensions,
    // 64 neurons of a column): both grids must fit one launch
    const int64_t nch = (D + 31) / 32;
    if (nch * ((side_x + 127) / 128) * side_y >= (int64_t(1) << 31) ||
        nch * side_x * ((side_y + 63) / 64) >= (int64_t(1) << 31))
        return fail(DSEQ_EINVAL, "map of %d x %d neurons with D=%d too large for one update", side_x, side_y, D);
    std::memset(&a, 0, sizeof a);
    a.n = n;
    a.M = M;
    a.D = D;
    a.side_x = side_x;
    a.side_y = side_y;
    a.R = sigma > 0.0 ? radius : 0;
    for (int k = 0; k <= a.R; ++k)
        a.g[k] = sigma > 0.0 ? (float)std::exp(-(double)k * k / (2.0 * sigma * sigma)) : 1.0f;
    return DSEQ_OK;
}

// The update on device operands (W updated in place).
int som_core(SomArgs &a, const DeviceInfo &info, SomWorkspace *ws, cudaStream_t st) {
    const size_t MD = (size_t)a.M * a.D;
    const size_t n_tiles = (size_t)((a.M + kSomScanTile - 1) / kSomScanTile);
    TRY(ws->S.ensure(MD * sizeof(long long)));
    TRY(ws->cnt.ensure(2 * (size_t)a.M * sizeof(unsigned)));  // counts, then cursors
    TRY(ws->off.ensure((size_t)a.M * sizeof(unsigned)));
    TRY(ws->tiles.ensure(2 * n_tiles * sizeof(unsigned)));    // totals, then offsets
    TRY(ws->order.ensure((size_t)std::max<int64_t>(1, a.n) * sizeof(int32_t)));
    TRY(ws->T.ensure(MD * sizeof(float)));
    TRY(ws->Tc.ensure((size_t)a.M * sizeof(float)));
    TRY(ws->status.ensure(2 * sizeof(int)));  // status word, then max |x| bits
    CUDA_TRY(cudaMemsetAsync(ws->status.p, 0, 2 * sizeof(int), st));
    a.S = ws->S.as<long long>();
    a.cnt = ws->cnt.as<unsigned>();
    a.cursor = a.cnt + a.M;
    a.off = ws->off.as<unsigned>();
    a.tile_sum = ws->tiles.as<unsigned>();
    a.tile_off = a.tile_sum + n_tiles;
    a.order = ws->order.as<int32_t>();
    a.T = ws->T.as<float>();
    a.Tc = ws->Tc.as<float>();
    a.status = ws->status.as<int>();
    a.maxbits = reinterpret_cast<unsigned *>(ws->status.as<int>() + 1);
    EventTimer timer;
    TRY(timer.start(st));
    CUDA_TRY(cudaMemsetAsync(a.cnt, 0, 2 * (size_t)a.M * sizeof(unsigned), st));
    CUDA_TRY(launch_som_update(a, info.sms, st));
    TRY(timer.stop(st));
    TRY(read_status(a.status, st));
    g_stats.update_ns = timer.ns();
    return DSEQ_OK;
}

// W as a device array: the pointer itself, or a staged copy of host data.
int stage_mutable(float *W, size_t count, DevBuf &buf, float *&dev, bool &on_host, cudaStream_t st) {
    bool on_device;
    TRY(locate(W, "W", on_device));
    on_host = !on_device;
    if (!on_host) {
        dev = W;
        return DSEQ_OK;
    }
    TRY(buf.ensure(count * sizeof(float)));
    CUDA_TRY(cudaMemcpyAsync(buf.p, W, count * sizeof(float), cudaMemcpyHostToDevice, st));
    dev = buf.as<float>();
    return DSEQ_OK;
}

}  // namespace

extern "C" {

int bmu_search(const float *X, int64_t n, const float *W, int64_t M, int32_t D, int32_t *idx,
               float *dist, void *cuda_stream) {
    g_err.clear();
    g_stats = Stats();
    if (!X || !W || !idx || !dist) return fail(DSEQ_EINVAL, "NULL pointer argument");
    TRY(bmu_validate(n, M, D));
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    int dev = 0;
    TRY(current_device(dev));
    const Options opt = default_options();
    BmuWorkspace *ws = bmu_workspace(dev);
    std::lock_guard<std::mutex> lk(ws->mu);
    DeviceInfo info;
    TRY(device_info(dev, info));
    const float *dX, *dW;
    TRY(stage_in(X, (size_t)n * D, ws->x_stage, dX, st, "X"));
    TRY(stage_in(W, (size_t)M * D, ws->w_stage, dW, st, "W"));
    bool idx_dev, dist_dev;
    TRY(locate(idx, "idx", idx_dev));
    TRY(locate(dist, "dist", dist_dev));
    int32_t *d_idx = idx;
    float *d_dist = dist;
    if (!idx_dev) {
        TRY(ws->idx_out.ensure((size_t)n * sizeof(int32_t)));
        d_idx = ws->idx_out.as<int32_t>();
    }
    if (!dist_dev) {
        TRY(ws->dist_out.ensure((size_t)n * sizeof(float)));
        d_dist = ws->dist_out.as<float>();
    }
    TRY(bmu_core(dX, n, dW, M, D, d_idx, d_dist, opt, info, ws, st));
    if (!idx_dev) CUDA_TRY(cudaMemcpyAsync(idx, d_idx, (size_t)n * sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    if (!dist_dev) CUDA_TRY(cudaMemcpyAsync(dist, d_dist, (size_t)n * sizeof(float), cudaMemcpyDeviceToHost, st));
    CUDA_TRY(cudaStreamSynchronize(st));
    return DSEQ_OK;
}

int som_update(const float *X, int64_t n, float *W, int32_t side_x, int32_t side_y, int32_t D,
               const int32_t *bmu, double sigma, int32_t radius, void *cuda_stream) {
    g_err.clear();
    g_stats = Stats();
    SomArgs a;
    TRY(som_validate(n, side_x, side_y, D, sigma, radius, a));
    if (!W || (n > 0 && (!X || !bmu))) return fail(DSEQ_EINVAL, "NULL pointer argument");
    if (n == 0) return DSEQ_OK;  // no sample reaches any neuron: W is unchanged
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    int dev = 0;
    TRY(current_device(dev));
    SomWorkspace *ws = som_workspace(dev);
    std::lock_guard<std::mutex> lk(ws->mu);
    DeviceInfo info;
    TRY(device_info(dev, info));
    const float *dX;
    const int32_t *dB;
    float *dW;
    bool w_host;
    TRY(stage_in(X, (size_t)n * D, ws->x_stage, dX, st, "X"));
    TRY(stage_in(bmu, (size_t)n, ws->bmu_stage, dB, st, "bmu"));
    TRY(stage_mutable(W, (size_t)a.M * D, ws->w_stage, dW, w_host, st));
    a.X = dX;
    a.bmu = dB;
    a.W = dW;
    TRY(som_core(a, info, ws, st));
    g_stats.units = a.M;
    g_stats.launches = 7;
    if (w_host) CUDA_TRY(cudaMemcpyAsync(W, dW, (size_t)a.M * D * sizeof(float), cudaMemcpyDeviceToHost, st));
    CUDA_TRY(cudaStreamSynchronize(st));
    return DSEQ_OK;
}

int som_epoch(const float *X, int64_t n, float *W, int32_t side_x, int32_t side_y, int32_t D,
              double sigma, int32_t radius, int32_t *bmu_out, float *dist_out, void *cuda_stream) {
    g_err.clear();
    g_stats = Stats();
    SomArgs a;
    TRY(som_validate(n, side_x, side_y, D, sigma, radius, a));
    if (!X || !W) return fail(DSEQ_EINVAL, "NULL pointer argument");
    TRY(bmu_validate(n, a.M, D));
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    int dev = 0;
    TRY(current_device(dev));
    const Options opt = default_options();
    BmuWorkspace *bws = bmu_workspace(dev);
    SomWorkspace *ws = som_workspace(dev);
    std::lock_guard<std::mutex> lk_bmu(bws->mu);  // always BMU first, then SOM
    std::lock_guard<std::mutex> lk(ws->mu);
    DeviceInfo info;
    TRY(device_info(dev, info));
    const float *dX;
    float *dW;
    bool w_host;
    TRY(stage_in(X, (size_t)n * D, ws->x_stage, dX, st, "X"));
    TRY(stage_mutable(W, (size_t)a.M * D, ws->w_stage, dW, w_host, st));
    bool idx_dev = false, dist_dev = false;
    if (bmu_out) TRY(locate(bmu_out, "bmu_out", idx_dev));
    if (dist_out) TRY(locate(dist_out, "dist_out", dist_dev));
    int32_t *d_idx = bmu_out;
    float *d_dist = dist_out;
    if (!idx_dev) {
        TRY(ws->idx.ensure((size_t)n * sizeof(int32_t)));
        d_idx = ws->idx.as<int32_t>();
    }
    if (!dist_dev) {
        TRY(ws->dist.ensure((size_t)n * sizeof(float)));
        d_dist = ws->dist.as<float>();
    }
    TRY(bmu_core(dX, n, dW, a.M, D, d_idx, d_dist, opt, info, bws, st));
    a.X = dX;
    a.bmu = d_idx;
    a.W = dW;
    TRY(som_core(a, info, ws, st));
    g_stats.launches += 7;
    if (bmu_out && !idx_dev)
        CUDA_TRY(cudaMemcpyAsync(bmu_out, d_idx, (size_t)n * sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    if (dist_out && !dist_dev)
        CUDA_TRY(cudaMemcpyAsync(dist_out, d_dist, (size_t)n * sizeof(float), cudaMemcpyDeviceToHost, st));
    if (w_host) CUDA_TRY(cudaMemcpyAsync(W, dW, (size_t)a.M * D * sizeof(float), cudaMemcpyDeviceToHost, st));
    CUDA_TRY(cudaStreamSynchronize(st));
    return DSEQ_OK;
}

}  // extern "C"
