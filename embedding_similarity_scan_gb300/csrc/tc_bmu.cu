// tc_bmu.cu — best-matching-unit search as a persistent, warp-specialised
// tcgen05 kernel for sm_103a.
//
// The method ("From 80x to 385x: A Best-Matching-Unit Search at the L2
// Roof", section 3 Background and section 4): for every sample x_i the
// neuron j minimising |x_i - w_j|^2 = |x_i|^2 + (|w_j|^2 - 2 <x_i, w_j>),
// with the argmin fused into the product so the sample x neuron score block
// is never materialised, and the neuron axis split into chunks whose partial
// (min, index) results are merged (section 4.2, neuron-axis chunking).
//
// Here a work unit is 128 samples (the TMEM lanes of one accumulator) times
// a chunk of tile_n neurons.  Units are ordered neuron-slice-major, then by
// sample block, then by chunk inside the slice, where a slice is as many
// chunks as fit a fraction of L2: all CTAs sweep one L2-resident slice of the
// codebook against every sample block before moving to the next slice, so
// the codebook is read from HBM once and the samples once per slice.
//
// Two kernels.  tc_bmu_kernel streams both operands through its stage ring.
// tc_bmu_resident_kernel (CTA pairs, D <= 256) keeps a CTA's 128 split
// sample rows in shared memory for a whole segment of a slice's chunks and
// streams only the codebook, which removes the sample tiles' share of the
// L2 -> SM operand traffic; both issue the same MMAs on the same data, so
// their results are bitwise equal.
//
// Operands are pre-scaled per row by a power of two (max |.| in [0.5, 1))
// and split into fp16 (prep.cu): samples [hi | lo * 2^12], codebook
// [hi * 2^12 | hi | lo * 2^12].  Three kind::f16 MMAs per 16-wide k step,
// x_hi . (2^12 w_hi) + x_hi . (2^12 w_lo) + (2^12 x_lo) . w_hi, accumulate
// 2^12 <x~, w~> in fp32 TMEM (the dropped lo . lo term is 2^-22 relative).
// The epilogue forms
// score_j = |w_j|^2 + acc * (1 / s_w[j]) * (-2^-11 / s_x[i]), keeps the
// running (min score, lowest j) per row and folds it into the row's 64-bit
// key with one atomicMin per unit; a finalize pass turns keys into
// (idx, max(0, |x|^2 + score)).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dseq {

namespace {

constexpr uint32_t kSubA = kUnitRows * kKBlock * 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
// column groups of 32 in the widest unit (256 neurons)
constexpr int kMaxGroups = 8;

// Stage geometry.  One CTA: B sub-tiles of up to 256 neuron rows, 3 stages.
// CTA pair: each CTA
// stages half of the neuron chunk (<= 128 rows), 5 stages.
template <bool kPair>
struct BmuCfg {
    static constexpr int kStagesT = kPair ? 5 : 3;
    static constexpr uint32_t kSubB = (kPair ? 128u : 256u) * kKBlock * 2;
    static constexpr uint32_t kStage = kBmuPartsX * kSubA + kBmuPartsW * kSubB;
    static constexpr size_t kSmemBytes =
        (size_t)kStagesT * kStage + 1024 + 256 + kEpiWarps * 32 * sizeof(float2);
};

// Resident-sample kernel (CTA pairs): the sample rows of up to kResKBlocks
// K blocks (D <= 256) stay in shared memory; 4 stages of codebook rows; each
// epilogue warp stages one 32-neuron group's constants at a time.  The
// layout fills 231,680 of the 232,448 bytes a CTA may have, so it leaves no
// room to align the base: the kernel requires (and checks) that the dynamic
// shared memory starts on a 1024-byte boundary.
struct BmuResCfg {
    static constexpr int kResKBlocks = 8;
    static constexpr uint32_t kSubB = 128u * kKBlock * 2;
    static constexpr uint32_t kABytes = kBmuPartsX * kResKBlocks * kSubA;  // 128 KB
    static constexpr int kStages = 4;
    static constexpr uint32_t kStage = kBmuPartsW * kSubB;                 // 24 KB
    static constexpr size_t kSmemBytes =
        (size_t)kABytes + (size_t)kStages * kStage + 256 + kEpiWarps * 32 * sizeof(float2);
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
}

// The three MMAs of one 16-wide k step: sample parts at a, a + a_step
// ([hi | lo]), codebook parts at b, b + b_step, b + 2 b_step
// ([hi * 2^12 | hi | lo]); accumulate = 0 starts a new sum.
template <bool kPair>
__device__ __forceinline__ void bmu_mma_k16(uint32_t d_tmem, uint32_t a, uint32_t a_step, uint32_t b,
                                            uint32_t b_step, uint32_t idesc, bool accumulate) {
    const uint64_t x_hi = smem_desc_sw64(a), x_lo = smem_desc_sw64(a + a_step);
    const uint64_t w_hi12 = smem_desc_sw64(b), w_hi = smem_desc_sw64(b + b_step),
                   w_lo = smem_desc_sw64(b + 2 * b_step);
    if (kPair) {
        umma_f16_pair(d_tmem, x_hi, w_hi12, idesc, accumulate ? 1u : 0u);
        umma_f16_pair(d_tmem, x_hi, w_lo, idesc, 1u);
        umma_f16_pair(d_tmem, x_lo, w_hi, idesc, 1u);
    } else {
        umma_f16(d_tmem, x_hi, w_hi12, idesc, accumulate ? 1u : 0u);
        umma_f16(d_tmem, x_hi, w_lo, idesc, 1u);
        umma_f16(d_tmem, x_lo, w_hi, idesc, 1u);
    }
}

// Epilogue of one unit (128 samples x tile_n neurons of chunk j) by one
// epilogue warp: the warp's lane quadrant q of the accumulator, every other
// 32-neuron group from h; score = |w|^2 + acc / s_w * (-2^-11 / s_x), the
// running (min score, lowest neuron) folded into the row's key.  The
// neuron constants are fetched before the accumulator wait and staged one
// group at a time in the warp's 256 bytes of shared memory (my_colc).
// Returns false if the wait gave up.
template <bool kPair>
__device__ __forceinline__ bool bmu_epilogue_unit(const BmuArgs &a, int beta, int j, uint32_t tile_n,
                                                  int groups, uint32_t tmem_base, uint32_t &acc_uses,
                                                  uint64_t *acc_full, uint64_t *acc_empty,
                                                  uint32_t acc_empty_leader0, float2 *my_colc,
                                                  volatile int *abort_flag, int warp, int lane) {
    const int e = warp - 2, q = warp & 3, h = e >> 2;
    const int64_t row = (int64_t)beta * kUnitRows + 32 * q + lane;
    const float cx = row < a.n ? -a.x_inv_scale[row] * (1.0f / 2048.0f) : 0.0f;
    float2 cv[kMaxGroups / 2];
#pragma unroll
    for (int k = 0; k < kMaxGroups / 2; ++k) {
        const int64_t col = (int64_t)j * tile_n + 32 * (h + 2 * k) + lane;
        cv[k] = (h + 2 * k < groups && col < a.M)
                    ? make_float2(__ldg(a.wn + col), __ldg(a.w_inv_scale + col))
                    : make_float2(INFINITY, 0.0f);
    }
    const uint32_t buf = acc_uses & 1u, apar = (acc_uses >> 1) & 1u;
    // every lane waits; the warp proceeds only if all of them saw the phase
    const bool ready = mbar_wait_bounded(&acc_full[buf], apar, abort_flag, a.status, a.timeout_ns,
                                         kStatusPipeTimeout);
    if (!__all_sync(0xffffffffu, ready)) return false;
    tc_fence_after();
    float best = INFINITY;
    uint32_t best_j = 0xffffffffu;
    const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + buf * kAccCols;
#pragma unroll
    for (int k = 0; k < kMaxGroups / 2; ++k) {
        const int g = h + 2 * k;
        if (g >= groups) break;
        __syncwarp();
        my_colc[lane] = cv[k];
        __syncwarp();
        float acc[32];
        tmem_ld_32cols(tbase + (uint32_t)(32 * g), acc);
        tmem_wait_ld();
        const uint32_t cbase = (uint32_t)j * tile_n + 32u * (uint32_t)g;
#pragma unroll
        for (int z = 0; z < 32; ++z) {
            const float2 cc = my_colc[z];
            const float sc = fmaf(acc[z] * cc.y, cx, cc.x);
            if (sc < best) {
                best = sc;
                best_j = cbase + z;
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
        if (kPair)
            mbar_arrive_cluster(acc_empty_leader0 + buf * (uint32_t)sizeof(uint64_t));
        else
            mbar_arrive(&acc_empty[buf]);
    }
    ++acc_uses;
    if (row < a.n && best_j != 0xffffffffu) atomicMin(a.keys + row, min_key(best, best_j));
    return true;
}

// Store epilogue of the Gram product (a.gram != nullptr): the same operands
// hold the rows of one table on both sides (X = [hi | lo * 2^12], W =
// [hi * 2^12 | hi | lo * 2^12], each row scaled by its power of two), so the
// accumulator of row i (sample side) and column c (codebook side) is
// 2^12 <x~_i, w~_c>; scaled back exactly to <e_i, e_c>, the distance
// 1 - <e_i, e_c> is stored at
// gram[c * gram_ld + i]: for each column the 32 lanes of a warp write 32
// consecutive rows, one 128-byte line.  G is symmetric, so only the items
// on and above the diagonal of 256 x 256 tiles are computed; with mirror
// set (an item off the diagonal) the same values are also stored at
// gram[i * gram_ld + c].  There a lane holds one row's 32 columns, so a
// direct store would touch 32 lines per instruction; instead the warp passes
// each half (16 rows) of its 32 x 32 block through a 2 KB shared-memory
// tile (16-byte chunks swizzled by row, so both the row-wise writes and the
// column-wise reads are free of bank conflicts) and every store instruction
// then writes 4 whole rows of the block, 4 full 128-byte lines (the number
// of requests, not of bytes, is what the L1-to-L2 path limits).  G is then
// exactly symmetric.  Returns false if the wait gave up.
constexpr uint32_t kGramStageBytes = kEpiWarps * 16 * 32 * sizeof(float);
template <bool kPair>
__device__ __forceinline__ bool gram_epilogue_unit(const BmuArgs &a, int beta, int j, uint32_t tile_n,
                                                   int groups, uint32_t tmem_base, uint32_t &acc_uses,
                                                   uint64_t *acc_full, uint64_t *acc_empty,
                                                   uint32_t acc_empty_leader0,
                                                   volatile int *abort_flag, int warp, int lane,
                                                   bool mirror, float4 *stage) {
    const int e = warp - 2, q = warp & 3, h = e >> 2;
    const int64_t row = (int64_t)beta * kUnitRows + 32 * q + lane;
    const bool row_ok = row < a.n;
    const float rx = row_ok ? a.x_inv_scale[row] * (1.0f / 4096.0f) : 0.0f;
    float cw[kMaxGroups / 2];
#pragma unroll
    for (int k = 0; k < kMaxGroups / 2; ++k) {
        const int64_t col = (int64_t)j * tile_n + 32 * (h + 2 * k) + lane;
        cw[k] = (h + 2 * k < groups && col < a.M) ? __ldg(a.w_inv_scale + col) : 0.0f;
    }
    const uint32_t buf = acc_uses & 1u, apar = (acc_uses >> 1) & 1u;
    const bool ready = mbar_wait_bounded(&acc_full[buf], apar, abort_flag, a.status, a.timeout_ns,
                                         kStatusPipeTimeout);
    if (!__all_sync(0xffffffffu, ready)) return false;
    tc_fence_after();
    const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + buf * kAccCols;
#pragma unroll
    for (int k = 0; k < kMaxGroups / 2; ++k) {
        const int g = h + 2 * k;
        if (g >= groups) break;
        float acc[32];
        tmem_ld_32cols(tbase + (uint32_t)(32 * g), acc);
        tmem_wait_ld();
        const int64_t cbase = (int64_t)j * tile_n + 32 * g;
#pragma unroll
        for (int z = 0; z < 32; ++z) {
            const float wz = __shfl_sync(0xffffffffu, cw[k], z);
            // the cosine distance 1 - <e_i, e_c>, rounded once from the fp32
            // inner product (the value the walk folds)
            acc[z] = fmaf(acc[z] * (rx * wz), -1.0f, 1.0f);
            if (row_ok && cbase + z < a.M) a.gram[(cbase + z) * a.gram_ld + row] = acc[z];
        }
        // columns past M are row padding of G (never read as values); the
        // group lies inside a row of G when it starts inside one (gram_ld is
        // a multiple of 32)
        if (mirror && cbase + 32 <= a.gram_ld) {
            const int64_t row0 = (int64_t)beta * kUnitRows + 32 * q;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                // lanes 16 half .. 16 half + 15 put their rows' 8 chunks at
                // chunk v ^ (r & 7) of tile row r = lane & 15
                if ((lane >> 4) == half) {
                    const int r = lane & 15;
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        stage[r * 8 + (v ^ (r & 7))] =
                            make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
                }
                __syncwarp();
                // 4 rows per instruction, 8 lanes per row (one 128-byte line)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 4 * k + (lane >> 3), c = lane & 7;
                    const float4 w = stage[r * 8 + (c ^ (r & 7))];
                    const int64_t grow = row0 + 16 * half + r;
                    if (grow < a.n)
                        *reinterpret_cast<float4 *>(a.gram + grow * a.gram_ld + cbase + 4 * c) = w;
                }
                __syncwarp();
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
        if (kPair)
            mbar_arrive_cluster(acc_empty_leader0 + buf * (uint32_t)sizeof(uint64_t));
        else
            mbar_arrive(&acc_empty[buf]);
    }
    ++acc_uses;
    return true;
}

// Work items of the Gram product: only the 256 x 256 tiles (row block pair
// blk, column chunk j) with j >= blk, in slices of chunks (the codebook side
// L2-resident for a slice); within a slice, by row block, then by chunk, so
// consecutive items (dealt round-robin to the CTA pairs) share their row
// block.  Enumerating only these tiles keeps the pairs' shares even.
struct GramSchedule {
    int n_chunk, slice_chunks;
    __device__ __forceinline__ int64_t slice_items(int s0, int s1) const {
        const int64_t w = s1 - s0;
        return (int64_t)s0 * w + w * (w + 1) / 2;
    }
    __device__ __forceinline__ int64_t total() const {
        int64_t t = 0;
        for (int s0 = 0; s0 < n_chunk; s0 += slice_chunks) t += slice_items(s0, min(n_chunk, s0 + slice_chunks));
        return t;
    }
    __device__ __forceinline__ void decode(int64_t u, int &blk, int &j) const {
        int s0 = 0, s1 = min(n_chunk, slice_chunks);
        while (s1 < n_chunk && u >= slice_items(s0, s1)) {
            u -= slice_items(s0, s1);
            s0 = s1;
            s1 = min(n_chunk, s0 + slice_chunks);
        }
        const int w = s1 - s0;
        if (u < (int64_t)s0 * w) {  // row blocks before the slice: every chunk of it
            blk = (int)(u / w);
            j = s0 + (int)(u - (int64_t)blk * w);
            return;
        }
        u -= (int64_t)s0 * w;  // row blocks inside the slice: chunks from the diagonal on
        int r = 0;
        while (u >= w - r) {
            u -= w - r;
            ++r;
        }
        blk = s0 + r;
        j = blk + (int)u;
    }
};

struct BmuSchedule {
    int n_blocks, n_chunk, tile_n, slice_chunks;
    // work item u -> (sample block, or sample block pair, "beta"; neuron chunk j)
    __device__ __forceinline__ void decode(int64_t u, int &beta, int &j) const {
        const int64_t per_slice = (int64_t)n_blocks * slice_chunks;
        const int64_t sl = u / per_slice;
        const int64_t rem = u - sl * per_slice;
        const int first = (int)(sl * slice_chunks);
        const int width = min(slice_chunks, n_chunk - first);
        beta = (int)(rem / width);
        j = first + (int)(rem - (int64_t)beta * width);
    }
};

// kGram: the store epilogue of the Gram product instead of the argmin.
template <bool kPair, bool kGram = false>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_bmu_kernel(const __grid_constant__ CUtensorMap tmap_x,
                  const __grid_constant__ CUtensorMap tmap_w, const BmuArgs a, const TcPlan p,
                  const int slice_chunks) {
    using Cfg = BmuCfg<kPair>;
    constexpr int kBmuStages = Cfg::kStagesT;
    constexpr uint32_t kSubB = Cfg::kSubB;
    constexpr uint32_t kStageBytes = Cfg::kStage;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kBmuStages * kStageBytes);
    uint64_t *empty = full + kBmuStages;
    uint64_t *acc_full = empty + kBmuStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *final_bar = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(final_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float2 *colc = reinterpret_cast<float2 *>(smem + kBmuStages * kStageBytes + 256);
    // the Gram store epilogue's per-warp transposition tiles (kGram only)
    float4 *gstage = reinterpret_cast<float4 *>(colc + kEpiWarps * 32);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t tmo = a.timeout_ns;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    // the launch must have the shape the kernel is written for (a pair kernel
    // addresses its peer's shared memory and TMEM): otherwise report and leave,
    // uniformly across the grid, before touching anything
    if (blockDim.x != kTcThreads || (kPair && (cluster_nctarank() != 2u || (gridDim.x & 1u)))) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, kStatusInternal);
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kBmuStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], kEpiWarps * (kPair ? 2 : 1));
        }
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        if (kPair) {
            tmem_alloc_pair(tmem_slot, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (kPair) cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // pair mode: work items are (sample block pair, chunk); this CTA takes
    // sample block 2 * pair + rank and rows [rank * tile_n / 2, ...) of the chunk
    const BmuSchedule sched{kPair ? p.n_beta / 2 : p.n_beta, p.n_chunk, p.tile_n, slice_chunks};
    const GramSchedule gsched{p.n_chunk, slice_chunks};
    const int64_t units = kGram ? gsched.total() : (int64_t)sched.n_blocks * p.n_chunk;
    auto decode_item = [&](int64_t u, int &blk, int &j) {
        if (kGram)
            gsched.decode(u, blk, j);
        else
            sched.decode(u, blk, j);
    };
    const int64_t first_item = kPair ? (blockIdx.x >> 1) : blockIdx.x;
    const int64_t item_stride = kPair ? (gridDim.x >> 1) : gridDim.x;
    const uint32_t tile_n = (uint32_t)p.tile_n;
    const uint32_t b_rows = kPair ? tile_n / 2 : tile_n;
    const uint32_t sub_b = b_rows * kKBlock * 2;
    const uint32_t tx_bytes = (kPair ? 2u : 1u) * (kBmuPartsX * kSubA + kBmuPartsW * sub_b);
    const int kblocks = a.Dp / kKBlock;
    const uint32_t idesc = idesc_f16_f32(kPair ? 2 * kUnitRows : kUnitRows, tile_n);
    const int groups = (int)(tile_n / 32);

    if (warp == 0) {
        if (lane == 0) {
            // the codebook slice is reused by every sample block: keep it in L2.
            // A sample block is read by every cluster working on it at about
            // the same time; evict-first would drop it between those reads.
            const uint64_t keep = l2_policy_evict_last(), once = l2_policy_evict_normal();
            uint32_t fills = 0;
            bool skip_copy = a.fault_skip_copy && blockIdx.x == 0;
            for (int64_t u = first_item; u < units && !*abort_flag; u += item_stride) {
                int blk, j;
                decode_item(u, blk, j);
                const int beta = kPair ? 2 * blk + (int)rank : blk;
                const int yx = beta * kUnitRows, yw = j * (int)tile_n + (int)(rank * b_rows);
                for (int kb = 0; kb < kblocks; ++kb) {
                    const uint32_t s = fills % kBmuStages, par = (fills / kBmuStages) & 1u;
                    if (!mbar_wait_bounded(&empty[s], par ^ 1u, abort_flag, a.status, tmo,
                                           kStatusPipeTimeout))
                        break;
                    uint8_t *sa = smem + s * kStageBytes;
                    uint8_t *sb = sa + kBmuPartsX * kSubA;
                    if (leader) mbar_arrive_expect_tx(&full[s], tx_bytes);
                    const int x = kb * kKBlock;
                    if (kPair) {
                        const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
#pragma unroll
                        for (int part = 0; part < kBmuPartsX; ++part)
                            tma_load_2d_pair(sa + part * kSubA, &tmap_x, fb, part * a.Dp + x, yx, once);
                        for (int part = 0; part < kBmuPartsW - (skip_copy ? 1 : 0); ++part)
                            tma_load_2d_pair(sb + part * kSubB, &tmap_w, fb, part * a.Dp + x, yw, keep);
                    } else {
#pragma unroll
                        for (int part = 0; part < kBmuPartsX; ++part)
                            tma_load_2d_hint(sa + part * kSubA, &tmap_x, &full[s], part * a.Dp + x, yx, once);
                        for (int part = 0; part < kBmuPartsW - (skip_copy ? 1 : 0); ++part)
                            tma_load_2d_hint(sb + part * kSubB, &tmap_w, &full[s], part * a.Dp + x, yw, keep);
                    }
                    skip_copy = false;
                    ++fills;
                }
            }
            if (*abort_flag && kPair) {
                // the pair's copies complete on the leader's barriers: give the
                // ones still in flight time to land
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
            if (*abort_flag && leader) {
                volatile int never = 0;
                for (uint32_t s = 0; s < kBmuStages && s < fills; ++s) {
                    const uint32_t n_s = fills / kBmuStages + (s < fills % kBmuStages ? 1u : 0u);
                    mbar_wait_bounded(&full[s], (n_s - 1) & 1u, &never, a.status,
                                      tmo < 1000000000ull ? tmo : 1000000000ull,
                                      kStatusPipeTimeout);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            uint32_t consumed = 0, acc_uses = 0;
            for (int64_t u = first_item; u < units && !*abort_flag; u += item_stride) {
                const uint32_t buf = acc_uses & 1u, apar = (acc_uses >> 1) & 1u;
                if (!mbar_wait_bounded(&acc_empty[buf], apar ^ 1u, abort_flag, a.status, tmo,
                                       kStatusPipeTimeout))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * kAccCols;
                bool ok = true;
                for (int kb = 0; kb < kblocks; ++kb) {
                    const uint32_t s = consumed % kBmuStages, par = (consumed / kBmuStages) & 1u;
                    if (!mbar_wait_bounded(&full[s], par, abort_flag, a.status, tmo,
                                           kStatusPipeTimeout)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + s * kStageBytes);
                    const uint32_t sb = sa + kBmuPartsX * kSubA;
#pragma unroll
                    for (int k16 = 0; k16 < kKBlock / 16; ++k16)
                        bmu_mma_k16<kPair>(d_tmem, sa + k16 * 32, kSubA, sb + k16 * 32, kSubB, idesc,
                                           (kb | k16) != 0);
                    if (kPair)
                        umma_commit_pair_multicast(&empty[s], 0x3);
                    else
                        umma_commit(&empty[s]);
                    ++consumed;
                }
                if (!ok) break;
                if (kPair)
                    umma_commit_pair_multicast(&acc_full[buf], 0x3);
                else
                    umma_commit(&acc_full[buf]);
                ++acc_uses;
            }
            volatile int never = 0;
            if (kPair)
                umma_commit_pair(final_bar);
            else
                umma_commit(final_bar);
            mbar_wait_bounded(final_bar, 0, &never, a.status,
                              tmo < 1000000000ull ? tmo : 1000000000ull, kStatusPipeTimeout);
        }
        __syncwarp();
    } else {
        float2 *my_colc = colc + (warp - 2) * 32;
        uint32_t acc_uses = 0;
        const uint32_t acc_empty_leader0 = kPair ? mapa_shared(smem_u32(&acc_empty[0]), 0) : 0u;
        for (int64_t u = first_item; u < units; u += item_stride) {
            int blk, j;
            decode_item(u, blk, j);
            const int beta = kPair ? 2 * blk + (int)rank : blk;
            if (kGram) {
                // off the diagonal the tile also fills its mirror image
                if (!gram_epilogue_unit<kPair>(a, beta, j, tile_n, groups, tmem_base, acc_uses,
                                               acc_full, acc_empty, acc_empty_leader0, abort_flag,
                                               warp, lane, j > blk, gstage + (warp - 2) * 128))
                    break;
            } else if (!bmu_epilogue_unit<kPair>(a, beta, j, tile_n, groups, tmem_base, acc_uses,
                                                 acc_full, acc_empty, acc_empty_leader0, my_colc,
                                                 abort_flag, warp, lane)) {
                break;
            }
        }
    }

    __syncthreads();
    // the leader's MMAs into both CTAs' TMEM are done before either frees it
    if (kPair) cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        if (kPair)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Work items of the resident-sample kernel.  A whole item is (sample block
// pair pb, one codebook slice): the pair loads its sample rows once and runs
// them against every chunk of the slice.  Whole items run slice-major, then
// by sample block pair, and are dealt round-robin to the CTA pairs, so all
// pairs sweep one L2-resident slice together and each sample block is read
// once per slice.  The last, partial round of whole items would leave pairs
// idle, so those items (the tail) are split into `tail_segs` segments of
// their slice's chunks, dealt the same way.  A segment may be empty when a
// narrow slice has fewer chunks than segments.
struct BmuResSchedule {
    int n_pb, n_chunk, slice_chunks, tail_segs;
    int64_t head;  // whole items before the tail
    __device__ __forceinline__ void decode(int64_t u, int &pb, int &c0, int &c1) const {
        int64_t w = u;
        int sg = 0, segs = 1;
        if (u >= head) {
            w = head + (u - head) / tail_segs;
            sg = (int)((u - head) % tail_segs);
            segs = tail_segs;
        }
        const int sl = (int)(w / n_pb);
        pb = (int)(w - (int64_t)sl * n_pb);
        const int first = sl * slice_chunks;
        const int width = min(slice_chunks, n_chunk - first);
        const int len = (width + segs - 1) / segs;
        c0 = first + min(width, sg * len);
        c1 = first + min(width, (sg + 1) * len);
    }
};

// CTA-pair BMU kernel with the samples resident in shared memory.  Per item
// each CTA loads its 128 sample rows (both parts, all K blocks) once, on the
// a_full barrier; the MMA issuer releases them on a_empty after the item's
// last MMA; the stage ring carries only codebook rows.
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_bmu_resident_kernel(const __grid_constant__ CUtensorMap tmap_x,
                           const __grid_constant__ CUtensorMap tmap_w, const BmuArgs a,
                           const TcPlan p, const int slice_chunks, const int tail_segs) {
    using Cfg = BmuResCfg;
    constexpr int kSt = Cfg::kStages;
    constexpr uint32_t kSubB = Cfg::kSubB;
    extern __shared__ __align__(1024) uint8_t smem_res[];
    uint8_t *smem = smem_res;
    uint8_t *s_x = smem;                          // [part][kblock] sample sub-tiles
    uint8_t *s_w = smem + Cfg::kABytes;           // stage ring of codebook rows
    uint64_t *full = reinterpret_cast<uint64_t *>(s_w + kSt * Cfg::kStage);
    uint64_t *empty = full + kSt;
    uint64_t *acc_full = empty + kSt;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *a_full = acc_empty + 2;
    uint64_t *a_empty = a_full + 1;
    uint64_t *final_bar = a_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(final_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float2 *colc = reinterpret_cast<float2 *>(s_w + kSt * Cfg::kStage + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t tmo = a.timeout_ns;
    const int kblocks = a.Dp / kKBlock;
    // launch shape and operand geometry this kernel is written for; otherwise
    // report and leave, uniformly across the grid, before touching anything
    if (blockDim.x != kTcThreads || cluster_nctarank() != 2u || (gridDim.x & 1u) ||
        kblocks > Cfg::kResKBlocks || p.tile_n > 256 || (p.n_beta & 1) || (smem_u32(smem) & 1023u)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, kStatusInternal);
        return;
    }
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSt; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], kEpiWarps * 2);
        }
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int64_t first_item = blockIdx.x >> 1, item_stride = gridDim.x >> 1;
    const int64_t n_slices = (p.n_chunk + slice_chunks - 1) / slice_chunks;
    const int64_t whole = n_slices * (p.n_beta / 2);
    const int64_t tail = whole % item_stride;
    const BmuResSchedule sched{p.n_beta / 2, p.n_chunk, slice_chunks, tail_segs, whole - tail};
    const int64_t items = (whole - tail) + tail * tail_segs;
    const uint32_t tile_n = (uint32_t)p.tile_n;
    const uint32_t b_rows = tile_n / 2;
    const uint32_t sub_b = b_rows * kKBlock * 2;
    const uint32_t tx_w = 2u * kBmuPartsW * sub_b;
    const uint32_t tx_x = 2u * kBmuPartsX * (uint32_t)kblocks * kSubA;
    const uint32_t idesc = idesc_f16_f32(2 * kUnitRows, tile_n);
    const int groups = (int)(tile_n / 32);

    if (warp == 0) {
        if (lane == 0) {
            // the codebook slice is reused by every sample block: keep it in
            // L2.  A (sample block pair, slice) item is loaded by one CTA pair
            // only (tail segments aside), so its sample rows are streamed
            // with evict-first and do not displace the slice; the prefetch
            // of the next item's rows uses the normal policy, to survive
            // until that item loads them.
            const uint64_t keep = l2_policy_evict_last(), once = l2_policy_evict_normal(),
                           stream = l2_policy_evict_first();
            uint32_t fills = 0, x_loads = 0;
            bool skip_copy = a.fault_skip_copy && blockIdx.x == 0;
            for (int64_t u = first_item; u < items && !*abort_flag; u += item_stride) {
                int pb, c0, c1;
                sched.decode(u, pb, c0, c1);
                if (c0 >= c1) continue;
                const int yx = (2 * pb + (int)rank) * kUnitRows;
                // the previous item's MMAs have finished reading the samples
                if (x_loads > 0 && !mbar_wait_bounded(a_empty, (x_loads - 1) & 1u, abort_flag,
                                                       a.status, tmo, kStatusPipeTimeout))
                    break;
                if (leader) mbar_arrive_expect_tx(a_full, tx_x);
                const uint32_t fa = mapa_shared(smem_u32(a_full), 0);
                for (int part = 0; part < kBmuPartsX; ++part)
                    for (int kb = 0; kb < kblocks; ++kb)
                        tma_load_2d_pair(s_x + (part * kblocks + kb) * kSubA, &tmap_x, fa,
                                         part * a.Dp + kb * kKBlock, yx, stream);
                ++x_loads;
                // bring the next item's sample rows (one contiguous block of
                // the split samples) into L2 while this item runs, so its
                // reload at the item boundary is an L2 hit
                if (u + item_stride < items) {
                    int pb2, d0, d1;
                    sched.decode(u + item_stride, pb2, d0, d1);
                    const int64_t row2 = (int64_t)(2 * pb2 + (int)rank) * kUnitRows;
                    if (pb2 != pb && row2 < a.n) {
                        const int64_t rows = min((int64_t)kUnitRows, a.n - row2);
                        prefetch_l2_hint(a.x_split + row2 * kBmuPartsX * a.Dp,
                                         (uint32_t)(rows * kBmuPartsX * a.Dp * (int64_t)sizeof(__half)), once);
                    }
                }
                bool ok = true;
                for (int j = c0; j < c1 && ok; ++j) {
                    const int yw = j * (int)tile_n + (int)(rank * b_rows);
                    for (int kb = 0; kb < kblocks; ++kb) {
                        const uint32_t s = fills % kSt, par = (fills / kSt) & 1u;
                        if (!mbar_wait_bounded(&empty[s], par ^ 1u, abort_flag, a.status, tmo,
                                               kStatusPipeTimeout)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sb = s_w + s * Cfg::kStage;
                        if (leader) mbar_arrive_expect_tx(&full[s], tx_w);
                        const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
                        for (int part = 0; part < kBmuPartsW - (skip_copy ? 1 : 0); ++part)
                            tma_load_2d_pair(sb + part * kSubB, &tmap_w, fb, part * a.Dp + kb * kKBlock,
                                             yw, keep);
                        skip_copy = false;
                        ++fills;
                    }
                }
                if (!ok) break;
            }
            if (*abort_flag) {
                // the pair's copies complete on the leader's barriers: give the
                // ones still in flight time to land
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
            if (*abort_flag && leader) {
                volatile int never = 0;
                const uint64_t lim = tmo < 1000000000ull ? tmo : 1000000000ull;
                for (uint32_t s = 0; s < kSt && s < fills; ++s) {
                    const uint32_t n_s = fills / kSt + (s < fills % kSt ? 1u : 0u);
                    mbar_wait_bounded(&full[s], (n_s - 1) & 1u, &never, a.status, lim, kStatusPipeTimeout);
                }
                if (x_loads > 0)
                    mbar_wait_bounded(a_full, (x_loads - 1) & 1u, &never, a.status, lim, kStatusPipeTimeout);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            uint32_t consumed = 0, acc_uses = 0, x_uses = 0;
            bool ok = true;
            for (int64_t u = first_item; u < items && ok && !*abort_flag; u += item_stride) {
                int pb, c0, c1;
                sched.decode(u, pb, c0, c1);
                if (c0 >= c1) continue;
                if (!mbar_wait_bounded(a_full, x_uses & 1u, abort_flag, a.status, tmo, kStatusPipeTimeout))
                    break;
                tc_fence_after();
                const uint32_t sx = smem_u32(s_x);
                for (int j = c0; j < c1 && ok; ++j) {
                    const uint32_t buf = acc_uses & 1u, apar = (acc_uses >> 1) & 1u;
                    if (!mbar_wait_bounded(&acc_empty[buf], apar ^ 1u, abort_flag, a.status, tmo,
                                           kStatusPipeTimeout)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * kAccCols;
                    for (int kb = 0; kb < kblocks; ++kb) {
                        const uint32_t s = consumed % kSt, par = (consumed / kSt) & 1u;
                        if (!mbar_wait_bounded(&full[s], par, abort_flag, a.status, tmo,
                                               kStatusPipeTimeout)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sb = smem_u32(s_w + s * Cfg::kStage);
                        const uint32_t sa = sx + (uint32_t)kb * kSubA;
#pragma unroll
                        for (int k16 = 0; k16 < kKBlock / 16; ++k16)
                            bmu_mma_k16<true>(d_tmem, sa + k16 * 32, (uint32_t)kblocks * kSubA,
                                              sb + k16 * 32, kSubB, idesc, (kb | k16) != 0);
                        umma_commit_pair_multicast(&empty[s], 0x3);
                        ++consumed;
                    }
                    if (!ok) break;
                    umma_commit_pair_multicast(&acc_full[buf], 0x3);
                    ++acc_uses;
                }
                if (!ok) break;
                // the samples are free once this item's MMAs have completed
                umma_commit_pair_multicast(a_empty, 0x3);
                ++x_uses;
            }
            volatile int never = 0;
            umma_commit_pair(final_bar);
            mbar_wait_bounded(final_bar, 0, &never, a.status,
                              tmo < 1000000000ull ? tmo : 1000000000ull, kStatusPipeTimeout);
        }
        __syncwarp();
    } else {
        float2 *my_colc = colc + (warp - 2) * 32;
        uint32_t acc_uses = 0;
        const uint32_t acc_empty_leader0 = mapa_shared(smem_u32(&acc_empty[0]), 0);
        bool ok = true;
        for (int64_t u = first_item; u < items && ok; u += item_stride) {
            int pb, c0, c1;
            sched.decode(u, pb, c0, c1);
            for (int j = c0; j < c1 && ok; ++j)
                ok = bmu_epilogue_unit<true>(a, 2 * pb + (int)rank, j, tile_n, groups, tmem_base, acc_uses,
                                             acc_full, acc_empty, acc_empty_leader0, my_colc, abort_flag,
                                             warp, lane);
        }
    }

    __syncthreads();
    // the leader's MMAs into both CTAs' TMEM are done before either frees it
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_tc_bmu(const BmuArgs &a, const TcPlan &p, const CUtensorMap &tmap_x,
                          const CUtensorMap &tmap_w, int slice_chunks, cudaStream_t st) {
    int dev = 0, l2 = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    // neuron slice: chunks whose split rows fill about 30 % of L2.  Larger
    // slices did not stay resident on GB300 (a 0.5-of-L2 slice was re-read
    // from DRAM several times over a som256 search: 0.96 GB vs 0.66 GB of
    // DRAM reads at this size), and the search time is the same within 1 %
    // from 19 % to 35 % of L2, so the slice is the width that reads least.
    const double row_bytes = (double)kBmuPartsW * a.Dp * 2.0;
    int slice = (int)((0.3 * (double)l2) / (row_bytes * p.tile_n));
    if (slice_chunks > 0) slice = slice_chunks;
    if (slice < 1) slice = 1;
    if (slice > p.n_chunk) slice = p.n_chunk;
    BmuArgs aa = a;
    TcPlan pp = p;
    CUtensorMap mx = tmap_x, mw = tmap_w;
    int sl = slice;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.pair && a.Dp <= BmuResCfg::kResKBlocks * kKBlock) {
        // samples resident: whole (sample block pair, slice) items, and the
        // last partial round of them split into enough segments that every
        // CTA pair has one
        const int64_t n_slices = (p.n_chunk + slice - 1) / slice;
        const int64_t pairs = p.grid / 2;
        const int64_t tail = (n_slices * (p.n_beta / 2)) % pairs;
        int64_t segs = tail > 0 ? (pairs + tail - 1) / tail : 1;
        if (segs > slice) segs = slice;
        int sg = (int)segs;
        const size_t smem = BmuResCfg::kSmemBytes;
        cudaError_t err = cudaFuncSetAttribute(tc_bmu_resident_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        cfg.dynamicSmemBytes = smem;
        return cudaLaunchKernelEx(&cfg, tc_bmu_resident_kernel, mx, mw, aa, pp, sl, sg);
    }
    if (!p.pair) {
        const size_t smem = BmuCfg<false>::kSmemBytes;
        cudaError_t err = cudaFuncSetAttribute(tc_bmu_kernel<false>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        void *args[] = {&mx, &mw, &aa, &pp, &sl};
        return cudaLaunchKernel(reinterpret_cast<const void *>(tc_bmu_kernel<false>),
                                dim3((unsigned)p.grid), dim3(kTcThreads), args, smem, st);
    }
    const size_t smem = BmuCfg<true>::kSmemBytes;
    cudaError_t err = cudaFuncSetAttribute(tc_bmu_kernel<true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, tc_bmu_kernel<true>, mx, mw, aa, pp, sl);
}

cudaError_t launch_tc_gram(const BmuArgs &a, const TcPlan &p, const CUtensorMap &tmap_x,
                           const CUtensorMap &tmap_w, cudaStream_t st) {
    // slices of the codebook side as for the BMU search (30 % of L2)
    int dev = 0, l2 = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    const double row_bytes = (double)kBmuPartsW * a.Dp * 2.0;
    int slice = (int)((0.3 * (double)l2) / (row_bytes * p.tile_n));
    if (slice < 1) slice = 1;
    if (slice > p.n_chunk) slice = p.n_chunk;
    BmuArgs aa = a;
    TcPlan pp = p;
    CUtensorMap mx = tmap_x, mw = tmap_w;
    int sl = slice;
    const size_t smem = BmuCfg<true>::kSmemBytes + kGramStageBytes;
    cudaError_t err = cudaFuncSetAttribute(tc_bmu_kernel<true, true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_bmu_kernel<true, true>, mx, mw, aa, pp, sl);
}

}  // namespace dseq
