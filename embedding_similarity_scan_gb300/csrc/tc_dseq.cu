// tc_dseq.cu — the greedy max-min diversity scan as one persistent,
// warp-specialised tcgen05 kernel for sm_103a.
//
// The method ("Issue 9-014: Tile Diversity Shader Inner Loop For L2 Cache
// Locality"): every iteration, each sequence compares its newest pick with
// every candidate, folds the cosine distance into its running minimum, and
// takes the unmasked candidate with the largest running minimum (lowest index
// on ties).  The issue asks for a tiled candidate scan that every workgroup
// walks together, with a hard grid-wide sync between steps (Intended
// Behavior, one dispatch per tile); here the loop over iterations lives on the
// device, and the sync is split per half of the sequences so that it never
// idles the grid (below).
//
// Work decomposition.  One iteration is the contraction S = Q * E^T of the
// B current query rows against the N table rows.  A work unit is a block of
// 128 sequences (the 128 TMEM lanes of one accumulator; a pair of blocks for
// a CTA pair) times a chunk of candidates (two chunk widths, see TcPlan).
// The sequence blocks form two halves; each iteration's units are ordered
// [half 0][half 1], each half candidate-chunk-major, and dealt to the
// persistent CTAs round-robin, so the grid marches over the table together.
//
// Precision.  Rows are unit-norm and split into fp16 pairs hi + lo * 2^-12
// (see prep.cu).  The query side carries (hi * 2^12, hi, lo), the table side
// (hi, lo); per 32-wide K block three kind::f16 MMAs accumulate
// hi*2^12 . hi + hi . lo + lo . hi into one fp32 TMEM accumulator, which
// equals 2^12 <q, e> up to about 2^-22 relative per product.  FP16 storage
// uses one part on each side and the rows' inverse norms.
//
// CTA roles (384 threads, two commit warps; 448 for the centroid criterion,
// four commit warps):
//   warp 0      TMA producer: Q and E K-blocks into a multi-stage smem ring;
//   warp 1      TMEM owner and MMA issuer (one thread), double-buffered
//               128 x 256 fp32 accumulators (512 TMEM columns);
//   warps 2-9   epilogue: TMEM -> registers, d = 1 - S, m = min(m, d) on the
//               running-minimum tile (read once, written back only where it
//               moved, 16-byte coalesced), running (max m, lowest index) per
//               row, one 64-bit atomicMax per row and unit into its key
//               (centroid criterion: d to the centroid against one held
//               bit per candidate, no running state);
//   warps 10-   commit warps: once every CTA has published a half of an
//               iteration, decode the winners of this CTA's share of that
//               half, record them, mask them in m (and in the held bits),
//               write the next queries
//               (the winners' stored rows, or the new centroids), and
//               release the half to the producers of the next iteration.
// Every wait is bounded in time and sets the status word instead of hanging.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "numeric.cuh"

namespace dseq {

namespace {

constexpr uint32_t kSubA = kUnitRows * kKBlock * 2;  // one 128 x 32 fp16 sub-tile: 8 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
// column groups of 32 in the widest unit (256 columns)
constexpr int kMaxGroups = 8;

// Stage geometry.  Split storage (fp32-accurate): A = 3 x (128 x 32),
// B = 2 x (rows x 32) fp16; fp16 storage: one part each, except the
// centroid query, which is not an fp16 row and keeps two parts
// (hi * 2^12, lo).  One CTA stages up to 256 candidate rows, a CTA pair half
// of the chunk (<= 128 rows) per SM.  Stage counts fill 194-231 KB of shared
// memory.
// The stages start at the dynamic shared memory base, which the kernel
// requires (and checks) to be 1024-byte aligned: there is no room for slack.
template <bool kPair, bool kF16, bool kCentroid = false>
struct DseqCfg {
    static constexpr int kPartsA = kF16 ? (kCentroid ? 2 : 1) : 3;
    static constexpr int kPartsB = kF16 ? 1 : 2;
    static constexpr uint32_t kSubB = (kPair ? 128u : 256u) * kKBlock * 2;
    // one K block's operands; an fp16-storage stage holds two K blocks, so
    // that its single issuing thread waits and commits once per four MMAs
    static constexpr uint32_t kKbBytes = kPartsA * kSubA + kPartsB * kSubB;
    static constexpr int kKbPerStage = kF16 ? 2 : 1;
    static constexpr uint32_t kStage = kKbPerStage * kKbBytes;
    static constexpr int kStagesT =
        kF16 ? (kCentroid ? (kPair ? 4 : 3) : (kPair ? 7 : 4)) : (kPair ? 5 : kStages);
    static constexpr uint32_t kBarrierBytes = 512;  // barriers, TMEM slot, flags
    // + per-warp column norms of one 32-column group (fp16 storage)
    static constexpr size_t kSmemBytes =
        (size_t)kStagesT * kStage + kBarrierBytes + (kF16 ? kEpiWarps * 32 * sizeof(float) : 0);
};


__global__ void tc_dseq_init_kernel(TcDseqArgs a, TcPlan p, const int32_t *__restrict__ starts,
                                    const uint8_t *__restrict__ mask) {
    const int64_t per_col = (int64_t)p.n_beta * kUnitRows;  // floats per candidate column
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // running minima, one 16-byte vector (4 consecutive candidates of one
    // row, 16-byte aligned in the tile layout) per step
    const int64_t total4 = p.columns() * per_col / 4;
    for (int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i4 < total4; i4 += stride) {
        const int64_t i = 4 * i4;
        const int j = p.chunk_of(i / per_col);
        const int64_t tile = (int64_t)kUnitRows * p.width(j);
        const int64_t local = i - p.col0(j) * per_col;
        const int beta = (int)(local / tile);
        const int s = (int)(local - beta * tile);
        const int t = (s >> 2) & 31, v = (s >> 7) & 7, q = (s >> 10) & 3, g = s >> 12;
        const int r = 32 * q + t;
        const int b = beta * kUnitRows + r;
        const int64_t cand0 = p.col0(j) + 32 * g + 4 * v;
        // the start's column (-1 when compaction dropped it: a masked start)
        const int st0 = b < a.B ? starts[b] : -1;
        const int st = (a.comp_of && st0 >= 0) ? a.comp_of[st0] : st0;
        float out[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int64_t cand = cand0 + e;
            bool live = b < a.B && cand < a.N;
            if (live && mask && mask[cand]) live = false;
            if (live && cand == st) live = false;
            out[e] = live ? INFINITY : -INFINITY;
        }
        reinterpret_cast<float4 *>(a.m)[i4] = make_float4(out[0], out[1], out[2], out[3]);
    }
    // centroid: the held-candidate bits, one word per (row, 32 columns)
    if (a.centroid) {
        const int64_t total_w = p.columns() * per_col / 32;
        for (int64_t wi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; wi < total_w; wi += stride) {
            const int64_t i = 32 * wi;
            const int j = p.chunk_of(i / per_col);
            const int64_t tile = (int64_t)kUnitRows * p.width(j);
            const int64_t local = i - p.col0(j) * per_col;
            const int beta = (int)(local / tile);
            const int sw = (int)((local - beta * tile) / 32);  // word within the tile
            const int g = sw / kUnitRows, r = sw % kUnitRows;
            const int b = beta * kUnitRows + r;
            const int64_t cand0 = p.col0(j) + 32 * g;
            const int st0 = b < a.B ? starts[b] : -1;
            const int st = (a.comp_of && st0 >= 0) ? a.comp_of[st0] : st0;
            unsigned bits = 0u;
            for (int z = 0; z < 32; ++z) {
                const int64_t cand = cand0 + z;
                bool live = b < a.B && cand < a.N;
                if (live && mask && mask[cand]) live = false;
                if (live && cand == st) live = false;
                if (!live) bits |= 1u << z;
            }
            a.held[wi] = bits;
        }
    }
    // query rows: the start rows, zero rows for padded sequences
    const int vec = a.Dp / 8;  // 16-byte vectors per row segment
    const int64_t qtotal = (int64_t)p.n_beta * kUnitRows * vec;
    if (a.e_f16 && !a.centroid) {  // fp16 storage: the stored row and its inverse norm
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < qtotal;
             i += stride) {
            const int b = (int)(i / vec), k = (int)(i - (int64_t)b * vec);
            uint4 *dst = reinterpret_cast<uint4 *>(a.q_split + (int64_t)b * a.Dp);
            dst[k] = b < a.B ? reinterpret_cast<const uint4 *>(a.e_f16_full +
                                                               (int64_t)starts[b] * a.Dp)[k]
                             : make_uint4(0, 0, 0, 0);
            if (k == 0) a.q_rn[b] = b < a.B ? a.rn_full[starts[b]] : 0.0f;
        }
    }
    // split queries: (hi * 2^12, hi, lo) of the start's unit row; the
    // centroid on fp16 storage keeps (hi * 2^12, lo)
    const int qparts = a.e_f16 ? 2 : 3;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
         i < qtotal && (!a.e_f16 || a.centroid); i += stride) {
        const int b = (int)(i / vec), k = (int)(i - (int64_t)b * vec);
        uint4 *dst = reinterpret_cast<uint4 *>(a.q_split + (int64_t)b * qparts * a.Dp);
        if (b < a.B) {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.e_split_full +
                                                               (int64_t)starts[b] * 2 * a.Dp);
            const uint4 hi = src[k], lo = src[vec + k];
            uint4 hi12 = hi;
            __half2 *h2 = reinterpret_cast<__half2 *>(&hi12);
            const __half2 scale = __float2half2_rn(4096.0f);
#pragma unroll
            for (int z = 0; z < 4; ++z) h2[z] = __hmul2(h2[z], scale);
            dst[k] = hi12;
            if (qparts == 3) dst[vec + k] = hi;
            dst[(qparts - 1) * vec + k] = lo;
        } else {
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int part = 0; part < qparts; ++part) dst[part * vec + k] = z;
        }
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
         i < (int64_t)p.n_beta * kUnitRows; i += stride)
        a.keys[i] = 0ull;
    if (a.centroid) {  // centroid sums start at the start rows
        // the first query is the start's unit row (factor 2^-12); the
        // centroid scale starts at the start row's norm exponent
        for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
             b < (int64_t)p.n_beta * kUnitRows; b += stride) {
            a.q_rn[b] = 1.0f / 4096.0f;
            a.c_exp[b] = b < a.B ? scale_exponent(a.nrm[starts[b]]) : 0;
        }
        const int64_t ctotal = (int64_t)p.n_beta * kUnitRows * a.Dp;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < ctotal;
             i += stride) {
            const int b = (int)(i / a.Dp), k = (int)(i - (int64_t)b * a.Dp);
            a.csum[i] = b < a.B ? to_fixed(a.e_unit[(int64_t)starts[b] * a.Dp + k] *
                                               a.nrm[starts[b]],
                                           a.csum_shift)
                                : 0ll;
        }
    }
}

__device__ __forceinline__ void stamp(const TcDseqArgs &a, int t, int slot) {
    if (a.timeline)
        a.timeline[((size_t)t * gridDim.x + blockIdx.x) * kTimelineSlots + slot] = globaltimer_ns();
}
__device__ __forceinline__ void record(const TcDseqArgs &a, int t, int slot, uint64_t value) {
    if (a.timeline) a.timeline[((size_t)t * gridDim.x + blockIdx.x) * kTimelineSlots + slot] = value;
}
// with the timeline on, adds the time a bounded wait took to *acc
__device__ __forceinline__ bool timed_wait(const TcDseqArgs &a, uint64_t *bar, uint32_t parity,
                                           volatile int *abort_flag, uint64_t tmo,
                                           uint64_t &acc) {
    if (!a.timeline)
        return mbar_wait_bounded(bar, parity, abort_flag, a.status, tmo, kStatusPipeTimeout);
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait_bounded(bar, parity, abort_flag, a.status, tmo, kStatusPipeTimeout);
    acc += globaltimer_ns() - t0;
    return ok;
}

// Commit warps per CTA: two share the copying of the winners' stored rows
// (one left the next iteration's producers waiting on the commit); the
// centroid commit (exact fixed-point centroid update of every sequence) is
// heavier and takes four.
template <bool kCentroid>
__host__ __device__ constexpr int dseq_commit_warps() {
    return kCentroid ? 4 : 2;
}
template <bool kCentroid>
__host__ __device__ constexpr int dseq_threads() {
    return kTcThreads + 32 * dseq_commit_warps<kCentroid>();
}

// kIsolate (max-min only; never chosen by the product path): the operand
// loads and the MMAs are compiled out and the accumulator is replaced by a
// distance that falls with every iteration, so that every running minimum
// is read and rewritten; everything else (epilogue, commit, cross-CTA
// counters) runs as in the real kernel.  It measures the fused epilogue's
// running-minimum stream against HBM on its own; its picks are meaningless.
template <bool kPair, bool kF16, bool kCentroid, bool kIsolate = false>
__global__ void __launch_bounds__(dseq_threads<kCentroid>(), 1)
    tc_dseq_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_e, const TcDseqArgs a,
                   const TcPlan p) {
    using Cfg = DseqCfg<kPair, kF16, kCentroid>;
    constexpr int kThreads = dseq_threads<kCentroid>();
    constexpr int kCommitWarps = dseq_commit_warps<kCentroid>();
    constexpr int kPartsA = Cfg::kPartsA, kPartsB = Cfg::kPartsB;
    constexpr int kSt = Cfg::kStagesT;
    constexpr uint32_t kSubB = Cfg::kSubB;
    constexpr uint32_t kStageB = Cfg::kStage;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kSt * kStageB);
    uint64_t *empty = full + kSt;
    uint64_t *acc_full = empty + kSt;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *final_bar = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(final_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // overlapped iterations: epilogue warps that finished each half, counted
    unsigned *epi_arrive = reinterpret_cast<unsigned *>(tmem_slot + 2);
    // fp16 storage: per epilogue warp, the inverse norms of its 32 columns
    float *col_rn = reinterpret_cast<float *>(smem + kSt * kStageB + Cfg::kBarrierBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t tmo = a.timeout_ns;
    // pair mode: CTA rank 0 of each cluster leads (issues the MMAs, owns the
    // full / acc_empty barriers that both CTAs feed)
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    // the launch must have the shape the kernel is written for (a pair kernel
    // addresses its peer's shared memory and TMEM): otherwise report and leave,
    // uniformly across the grid, before touching anything
    if (blockDim.x != kThreads || (kPair && (cluster_nctarank() != 2u || (gridDim.x & 1u))) ||
        (smem_u32(smem) & 1023u)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, kStatusInternal);
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSt; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], kEpiWarps * (kPair ? 2 : 1));
        }
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        epi_arrive[0] = epi_arrive[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_e);
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
    // both CTAs' barriers must be initialised before either signals the other
    if (kPair) cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const uint32_t tile_n = (uint32_t)p.tile_n;
    // rows of this CTA's B sub-tile (pair: half of the candidate chunk)
    const uint32_t b_rows = kPair ? tile_n / 2 : tile_n;
    const uint32_t sub_b = b_rows * kKBlock * 2;
    const uint32_t tx_bytes = (kPair ? 2u : 1u) * (kPartsA * kSubA + kPartsB * sub_b);
    const int kblocks = a.Dp / kKBlock;

    // work items: (sequence block, chunk) units, or (sequence block pair,
    // chunk) for a cluster.  The blocks form two halves, and each
    // iteration's items are ordered [half 0][half 1], each half
    // candidate-chunk-major.
    const int n_blocks = kPair ? p.n_beta / 2 : p.n_beta;
    const int n_h0 = (n_blocks + 1) / 2;
    const int n_h1 = n_blocks - n_h0;
    const int64_t work = (int64_t)n_blocks * p.n_chunk;
    const int64_t half_units = (int64_t)n_h0 * p.n_chunk;
    const int rows_per_block = kPair ? 2 * kUnitRows : kUnitRows;
    const int seq_half[3] = {0, n_h0 * rows_per_block, n_blocks * rows_per_block};
    const int64_t first_item = kPair ? (blockIdx.x >> 1) : blockIdx.x;
    const int64_t item_stride = kPair ? (gridDim.x >> 1) : gridDim.x;
    auto decode = [&](int64_t v, int &beta, int &j) {
        int blk;
        if (v < half_units) {
            blk = (int)(v % n_h0);
            j = (int)(v / n_h0);
        } else {
            const int64_t k = v - half_units;
            blk = n_h0 + (int)(k % n_h1);
            j = (int)(k / n_h1);
        }
        beta = kPair ? 2 * blk + (int)rank : blk;
    };

    uint32_t fills = 0;     // producer: stages filled so far
    // epilogue-isolated kernel: this iteration's stand-in distance
    float iso_d = 0.0f;
    uint32_t consumed = 0;  // MMA: stages consumed so far
    uint32_t acc_uses = 0;  // MMA and epilogue: accumulators used so far

    // ---- per-unit work, shared by both iteration schemes ----
    // producer: the kblocks stages of unit v
    auto produce_unit = [&](int t, int64_t v, uint64_t keep, uint64_t table_pol, uint64_t m_pol,
                            uint64_t &waited, bool &first) {
        int beta, j;
        decode(v, beta, j);
        // fp16 storage, where the epilogue is the critical path: the unit's
        // running minima (one contiguous tile) are brought into L2 ahead of
        // the epilogue that reads them.  (The split-storage kernels are
        // tensor-bound; there the prefetch only added DRAM reads.)
        if (kF16 && !kCentroid)
            prefetch_l2_hint(a.m + p.tile_base(j, beta),
                             (uint32_t)p.width(j) * kUnitRows * (uint32_t)sizeof(float), m_pol);
        const int yq = beta * kUnitRows;
        // a narrow chunk still loads a full box (its tail rows unused)
        const int ye = (int)p.col0(j) + (int)rank * (p.width(j) / (kPair ? 2 : 1));
        for (int kb0 = 0; kb0 < kblocks; kb0 += Cfg::kKbPerStage) {
            const int nkb = min(Cfg::kKbPerStage, kblocks - kb0);
            const uint32_t s = fills % kSt, par = (fills / kSt) & 1u;
            if (!timed_wait(a, &empty[s], par ^ 1u, abort_flag, tmo, waited))
                break;
            if (leader) mbar_arrive_expect_tx(&full[s], tx_bytes * (uint32_t)nkb);
            if (first) {
                stamp(a, t, 1);
                first = false;
            }
            // completion goes to the pair leader's barrier for this stage
            const uint32_t fb = kPair ? mapa_shared(smem_u32(&full[s]), 0) : 0u;
#pragma unroll
            for (int i = 0; i < Cfg::kKbPerStage; ++i) {
                if (i >= nkb) break;
                uint8_t *sa = smem + s * kStageB + i * Cfg::kKbBytes;
                uint8_t *sb = sa + kPartsA * kSubA;
                const int x = (kb0 + i) * kKBlock;
#pragma unroll
                for (int part = 0; part < kPartsA; ++part) {  // (hi*2^12, hi, lo) or fp16
                    if (kPair)
                        tma_load_2d_pair(sa + part * kSubA, &tmap_q, fb,
                                         part * a.Dp + x, yq, keep);
                    else
                        tma_load_2d_hint(sa + part * kSubA, &tmap_q, &full[s],
                                         part * a.Dp + x, yq, keep);
                }
#pragma unroll
                for (int part = 0; part < kPartsB; ++part) {  // (hi, lo) or fp16
                    if (kPair)
                        tma_load_2d_pair(sb + part * kSubB, &tmap_e, fb,
                                         part * a.Dp + x, ye, table_pol);
                    else
                        tma_load_2d_hint(sb + part * kSubB, &tmap_e, &full[s],
                                         part * a.Dp + x, ye, table_pol);
                }
            }
            ++fills;
        }
    };
    // MMA issuer: the unit's kblocks stages into one accumulator; false on abort
    auto mma_unit = [&](int t, int64_t v, uint64_t &wait_full, uint64_t &wait_acc,
                        bool &first) -> bool {
        const uint32_t buf = acc_uses & 1u, apar = (acc_uses >> 1) & 1u;
        int beta_u, j_u;
        decode(v, beta_u, j_u);
        const uint32_t idesc = idesc_f16_f32(kPair ? 2 * kUnitRows : kUnitRows,
                                             (uint32_t)p.width(j_u));
        if (!timed_wait(a, &acc_empty[buf], apar ^ 1u, abort_flag, tmo, wait_acc))
            return false;
        tc_fence_after();
        if (kIsolate) {
            // no contraction: hand the (unwritten) accumulator straight to
            // the epilogue warps of this CTA (and of the peer)
            mbar_arrive(&acc_full[buf]);
            if (kPair) mbar_arrive_cluster(mapa_shared(smem_u32(&acc_full[buf]), 1));
            if (first) {
                stamp(a, t, 2);
                first = false;
            }
            ++acc_uses;
            return true;
        }
        const uint32_t d_tmem = tmem_base + buf * kAccCols;
        bool ok = true;
        for (int kb0 = 0; kb0 < kblocks; kb0 += Cfg::kKbPerStage) {
            const int nkb = min(Cfg::kKbPerStage, kblocks - kb0);
            const uint32_t s = consumed % kSt, par = (consumed / kSt) & 1u;
            if (!timed_wait(a, &full[s], par, abort_flag, tmo, wait_full)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (first) {
                stamp(a, t, 2);
                first = false;
            }
#pragma unroll
            for (int i = 0; i < Cfg::kKbPerStage; ++i) {
                if (i >= nkb) break;
                const int kb = kb0 + i;
                const uint32_t sa = smem_u32(smem + s * kStageB + i * Cfg::kKbBytes);
                const uint32_t sb = sa + kPartsA * kSubA;
#pragma unroll
                for (int k16 = 0; k16 < kKBlock / 16; ++k16) {
                    const uint32_t off = k16 * 32;  // 16 fp16 = 32 bytes along K
                    const uint64_t a0 = smem_desc_sw64(sa + off);
                    const uint64_t b0 = smem_desc_sw64(sb + off);
                    if (kF16) {  // one product: the stored fp16 rows
                        if (kPair)
                            umma_f16_pair(d_tmem, a0, b0, idesc, (kb | k16) != 0);
                        else
                            umma_f16(d_tmem, a0, b0, idesc, (kb | k16) != 0);
                        if (kCentroid) {  // the centroid's lo part
                            const uint64_t a1 = smem_desc_sw64(sa + kSubA + off);
                            if (kPair)
                                umma_f16_pair(d_tmem, a1, b0, idesc, 1u);
                            else
                                umma_f16(d_tmem, a1, b0, idesc, 1u);
                        }
                        continue;
                    }
                    const uint64_t a1 = smem_desc_sw64(sa + kSubA + off);
                    const uint64_t a2 = smem_desc_sw64(sa + 2 * kSubA + off);
                    const uint64_t b1 = smem_desc_sw64(sb + kSubB + off);
                    if (kPair) {
                        umma_f16_pair(d_tmem, a0, b0, idesc, (kb | k16) != 0);
                        umma_f16_pair(d_tmem, a1, b1, idesc, 1u);
                        umma_f16_pair(d_tmem, a2, b0, idesc, 1u);
                    } else {
                        umma_f16(d_tmem, a0, b0, idesc, (kb | k16) != 0);
                        umma_f16(d_tmem, a1, b1, idesc, 1u);
                        umma_f16(d_tmem, a2, b0, idesc, 1u);
                    }
                }
            }
            if (kPair)
                umma_commit_pair_multicast(&empty[s], 0x3);
            else
                umma_commit(&empty[s]);
            ++consumed;
        }
        if (!ok) return false;
        if (kPair)
            umma_commit_pair_multicast(&acc_full[buf], 0x3);
        else
            umma_commit(&acc_full[buf]);
        ++acc_uses;
        return true;
    };
    // epilogue warp: distances, running minima, row winners of unit v; false on abort
    auto epilogue_unit = [&](int64_t v, uint64_t stream, uint32_t acc_empty_leader0,
                             uint64_t &epi_wait) -> bool {
        // two warps per TMEM lane quadrant q, each taking every other column group
        const int e = warp - 2, q = warp & 3, h = e >> 2;
        const int r = 32 * q + lane;
        const uint32_t buf = acc_uses & 1u, apar = (acc_uses >> 1) & 1u;
        int beta, j;
        decode(v, beta, j);
        const int groups = p.width(j) / 32;
        const int64_t c0 = p.col0(j);
        float4 *mt = reinterpret_cast<float4 *>(a.m + p.tile_base(j, beta));
        // prefetch the first group's running minima (centroid: its held
        // bits, one word per row) before waiting
        float4 mcur[8], mnext[8];
        const unsigned *ht = kCentroid ? a.held + p.tile_base(j, beta) / 32 : nullptr;
        unsigned hcur = 0u, hnext = 0u;
        if (h < groups) {
            if (kCentroid) {
                hcur = __ldcg(ht + h * kUnitRows + r);
            } else {
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    mcur[v] = ld_cg_hint(&mt[((h * 4 + q) * 8 + v) * 32 + lane], stream);
            }
        }
        // fp16 storage: d = 1 - acc * rn_q * rn_c with the rows' inverse
        // norms; this warp's (at most 4) column groups' norms are
        // fetched before the wait too
        float neg_rnq = 0.0f, rnv[kMaxGroups / 2];
        if (kCentroid) neg_rnq = -a.q_rn[beta * kUnitRows + r];
        if (kF16) {
            neg_rnq = -a.q_rn[beta * kUnitRows + r];
#pragma unroll
            for (int k = 0; k < kMaxGroups / 2; ++k) {
                const int64_t col = c0 + 32 * (h + 2 * k) + lane;
                rnv[k] = (h + 2 * k < groups && col < a.N) ? __ldg(a.rn + col) : 0.0f;
            }
        }
        // every lane waits; the warp proceeds only if all of them saw the phase
        const bool ready = timed_wait(a, &acc_full[buf], apar, abort_flag, tmo, epi_wait);
        if (!__all_sync(0xffffffffu, ready)) return false;
        tc_fence_after();
        float best = -INFINITY;
        uint32_t best_c = 0;
        const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + buf * kAccCols;
        float *my_rn = col_rn + e * 32;
        for (int g = h; g < groups; g += 2) {
            if (kF16) {
                // this group's column norms, from the registers they were
                // fetched into before the wait
                float rv = rnv[0];
#pragma unroll
                for (int k = 1; k < kMaxGroups / 2; ++k)
                    if (((g - h) >> 1) == k) rv = rnv[k];
                __syncwarp();
                my_rn[lane] = rv;
                __syncwarp();
            }
            const float *rn_g = my_rn;
            const int gn = g + 2;
            if (gn < groups) {
                if (kCentroid) {
                    hnext = __ldcg(ht + gn * kUnitRows + r);
                } else {
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        mnext[v] = ld_cg_hint(&mt[((gn * 4 + q) * 8 + v) * 32 + lane], stream);
                }
            }
            float acc[32];
            tmem_ld_32cols(tbase + (uint32_t)(32 * g), acc);
            tmem_wait_ld();
            const uint32_t cbase = (uint32_t)c0 + 32u * (uint32_t)g;
            if constexpr (kCentroid) {
                // this iteration's distances to the centroid; held, masked
                // and padding columns -inf.  They are stored only for a trace.
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    float dv[4];
#pragma unroll
                    for (int z = 0; z < 4; ++z) {
                        const int c = 4 * v + z;
                        const float sc = kF16 ? acc[c] * rn_g[c] : acc[c];
                        dv[z] = ((hcur >> c) & 1u) ? -INFINITY : fmaf(sc, neg_rnq, 1.0f);
                        if (dv[z] > best) {
                            best = dv[z];
                            best_c = cbase + c;
                        }
                    }
                    if (a.trace_slot)
                        st_cg_hint(&mt[((g * 4 + q) * 8 + v) * 32 + lane],
                                   make_float4(dv[0], dv[1], dv[2], dv[3]), stream);
                }
                hcur = hnext;
                continue;
            }
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                float mv[4] = {mcur[v].x, mcur[v].y, mcur[v].z, mcur[v].w};
                bool changed = false;
                // max-min: m keeps the running minimum
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    // split storage: d = 1 - <q, e>, the accumulator holding
                    // 2^12 <q, e> of unit rows
                    const float d = kIsolate ? iso_d
                                    : kF16   ? fmaf(acc[4 * v + z] * rn_g[4 * v + z], neg_rnq, 1.0f)
                                             : fmaf(acc[4 * v + z], -1.0f / 4096.0f, 1.0f);
                    const float nv = fminf(mv[z], d);
                    changed |= nv != mv[z];
                    mv[z] = nv;
                    if (mv[z] > best) {
                        best = mv[z];
                        best_c = cbase + 4 * v + z;
                    }
                }
                // a candidate's running minimum changes with probability
                // about 1/(t+1) after t picks: write back only what moved
                if (changed)
                    st_cg_hint(&mt[((g * 4 + q) * 8 + v) * 32 + lane],
                               make_float4(mv[0], mv[1], mv[2], mv[3]), stream);
            }
            if (gn < groups) {
#pragma unroll
                for (int v = 0; v < 8; ++v) mcur[v] = mnext[v];
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
        const int b = beta * kUnitRows + r;
        if (best > -INFINITY && b < a.B) atomicMax(a.keys + b, max_key(best, best_c));
        return true;
    };
    // commit of sequences [b_lo, b_hi) of iteration t by one warp: picks, keys
    // reset, winner masked, next queries written
    auto commit_range = [&](int t, int b_lo, int b_hi) {
        const int vec = a.Dp / 8;  // 16-byte vectors per row segment
        for (int base = b_lo; base < b_hi; base += 32) {
            const int cnt = min(32, b_hi - base);
            const int b = base + lane;
            const bool mine = lane < cnt;
            const unsigned long long key = mine ? __ldcg(a.keys + b) : 0ull;
            const uint32_t w = max_key_index(key);
            if (mine) {
                if (key == 0ull) {
                    atomicOr(a.status, kStatusNoWinner);
                    a.picks[(int64_t)b * a.L + t] = -1;
                } else {
                    a.keys[b] = 0ull;
                    a.picks[(int64_t)b * a.L + t] = a.col_map ? a.col_map[w] : (int32_t)w;
                }
            }
            if (a.trace_slot) {
                // parity-check path: copy the traced rows of m before masking
                for (int i = 0; i < cnt; ++i) {
                    const int bi = base + i;
                    const int slot = a.trace_slot[bi];
                    if (slot < 0) continue;
                    const int beta = bi / kUnitRows, r = bi % kUnitRows;
                    float *dst = a.trace + ((int64_t)slot * a.L + t) * a.n_table;
                    for (int64_t row = lane; row < a.n_table; row += 32) {
                        // a row dropped by compaction is masked: -inf, as in m
                        const int64_t c = a.comp_of ? a.comp_of[row] : row;
                        if (c < 0) {
                            dst[row] = -INFINITY;
                            continue;
                        }
                        const int jj = p.chunk_of(c);
                        const int cc = (int)(c - p.col0(jj));
                        dst[row] = __ldcg(a.m + p.tile_base(jj, beta) + tc_m_inner(r, cc));
                    }
                }
                __syncwarp();
            }
            if (mine && key != 0ull) {
                const int beta = b / kUnitRows, r = b % kUnitRows;
                const int jw = p.chunk_of(w);
                const int cw = (int)(w - p.col0(jw));
                a.m[p.tile_base(jw, beta) + tc_m_inner(r, cw)] = -INFINITY;
                if (kCentroid)
                    atomicOr(a.held + p.tile_base(jw, beta) / 32 + (cw / 32) * kUnitRows + r,
                             1u << (cw % 32));
            }
            // next queries: the centroid's (per sequence), else the winners'
            // stored rows, all rows of the run by the whole warp
            const __half2 scale = __float2half2_rn(4096.0f);
            for (int i = 0; kCentroid && i < cnt; ++i) {
                const unsigned long long ki = __shfl_sync(0xffffffffu, key, i);
                const uint32_t wi = __shfl_sync(0xffffffffu, w, i);
                if (ki == 0ull) continue;
                if (kCentroid) {
                    // add the winner to the sequence's exact centroid sum and
                    // write the centroid C, scaled by a power of two 2^-sb kept
                    // per sequence, as the split query; the epilogue divides
                    // by its norm (q_rn = 2^-12 / |C 2^-sb|), so one pass over
                    // the row suffices.  When max |C 2^-sb| leaves [2^-6, 1)
                    // the split is redone with sb corrected (max in [0.5, 1)).
                    const int bq = base + i;
                    long long *cs = a.csum + (int64_t)bq * a.Dp;
                    const int64_t wr = a.col_map ? a.col_map[wi] : wi;  // table row
                    const float *eu = a.e_unit + wr * a.Dp;
                    constexpr int kQParts = kF16 ? 2 : 3;  // (hi*2^12, [hi,] lo)
                    __half *qd = a.q_split + (int64_t)bq * kQParts * a.Dp;
                    const float nw = a.nrm[wr];
                    const int F = a.csum_shift;
                    int sb = a.c_exp[bq];
                    float s1, s2;
                    fixed_unscale(F + sb, s1, s2);
                    auto put = [&](int k, float c) {
                        const __half hi = __float2half_rn(c);
                        const __half lo = __float2half_rn((c - __half2float(hi)) * 4096.0f);
                        qd[k] = __float2half_rn(__half2float(hi) * 4096.0f);
                        if (!kF16) qd[a.Dp + k] = hi;
                        qd[(kQParts - 1) * a.Dp + k] = lo;
                    };
                    constexpr int kB = 12;  // loads in flight per lane
                    KahanSum ss;
                    float mx = 0.0f;
                    for (int k0 = 0; k0 < a.Dp; k0 += 32 * kB) {
                        long long v[kB];
                        float x[kB];
#pragma unroll
                        for (int u = 0; u < kB; ++u) {
                            const int k = k0 + 32 * u + lane;
                            v[u] = k < a.Dp ? cs[k] : 0ll;
                            x[u] = k < a.Dp ? __ldg(eu + k) : 0.0f;
                        }
#pragma unroll
                        for (int u = 0; u < kB; ++u) {
                            const int k = k0 + 32 * u + lane;
                            if (k < a.Dp) {
                                v[u] += to_fixed(x[u] * nw, F);
                                cs[k] = v[u];
                                const float c = from_fixed(v[u], s1, s2);
                                mx = fmaxf(mx, fabsf(c));
                                ss.add(c * c);
                                put(k, c);
                            }
                        }
                    }
                    mx = warp_max_f(mx);
                    if (mx >= 1.0f || (mx > 0.0f && mx < 1.0f / 64.0f)) {
                        sb += scale_exponent(mx);
                        fixed_unscale(F + sb, s1, s2);
                        ss = KahanSum();
                        __syncwarp();
                        for (int k0 = 0; k0 < a.Dp; k0 += 32 * kB) {
                            long long v[kB];
#pragma unroll
                            for (int u = 0; u < kB; ++u) {
                                const int k = k0 + 32 * u + lane;
                                v[u] = k < a.Dp ? cs[k] : 0ll;
                            }
#pragma unroll
                            for (int u = 0; u < kB; ++u) {
                                const int k = k0 + 32 * u + lane;
                                if (k < a.Dp) {
                                    const float c = from_fixed(v[u], s1, s2);
                                    ss.add(c * c);
                                    put(k, c);
                                }
                            }
                        }
                    }
                    const float sum = warp_sum_f(ss.total());
                    if (lane == 0) {
                        // a zero centroid gives a zero factor: every distance is 1
                        a.q_rn[bq] = sum > 0.0f ? (1.0f / 4096.0f) / sqrtf(sum) : 0.0f;
                        a.c_exp[bq] = sb;
                    }
                    continue;
                }
            }
            if (!kCentroid) {
                // the winners' rows, flattened over (sequence, 16-byte vector)
                // so that each lane has kCopyBatch rows' loads in flight
                constexpr int kCopyBatch = 4;
                const int total = cnt * vec;
                for (int f0 = 0; f0 < total; f0 += 32 * kCopyBatch) {
                    uint4 hv[kCopyBatch], lv[kCopyBatch];
                    int ii[kCopyBatch];
                    uint32_t wv[kCopyBatch];
                    bool ok[kCopyBatch];
#pragma unroll
                    for (int u = 0; u < kCopyBatch; ++u) {
                        const int f = f0 + 32 * u + lane;
                        ii[u] = min(f / vec, cnt - 1);
                        wv[u] = __shfl_sync(0xffffffffu, w, ii[u]);
                        const unsigned long long ku = __shfl_sync(0xffffffffu, key, ii[u]);
                        ok[u] = f < total && ku != 0ull;
                        const int k = f - ii[u] * vec;
                        if (kF16) {
                            const uint4 *src = reinterpret_cast<const uint4 *>(a.e_f16 + (int64_t)wv[u] * a.Dp);
                            hv[u] = ok[u] ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
                        } else {
                            const uint4 *src =
                                reinterpret_cast<const uint4 *>(a.e_split + (int64_t)wv[u] * 2 * a.Dp);
                            hv[u] = ok[u] ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
                            lv[u] = ok[u] ? __ldg(src + vec + k) : make_uint4(0, 0, 0, 0);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kCopyBatch; ++u) {
                        if (!ok[u]) continue;
                        const int f = f0 + 32 * u + lane;
                        const int k = f - ii[u] * vec;
                        const int bq = base + ii[u];
                        if (kF16) {
                            reinterpret_cast<uint4 *>(a.q_split + (int64_t)bq * a.Dp)[k] = hv[u];
                            if (k == 0) a.q_rn[bq] = a.rn[wv[u]];
                        } else {
                            uint4 *dst = reinterpret_cast<uint4 *>(a.q_split + (int64_t)bq * 3 * a.Dp);
                            uint4 hi12 = hv[u];
                            __half2 *h2 = reinterpret_cast<__half2 *>(&hi12);
#pragma unroll
                            for (int z = 0; z < 4; ++z) h2[z] = __hmul2(h2[z], scale);
                            dst[k] = hi12;
                            dst[vec + k] = hv[u];
                            dst[2 * vec + k] = lv[u];
                        }
                    }
                }
            }
        }
    };
    // this CTA's first work item at or after index lo
    auto first_from = [&](int64_t lo) -> int64_t {
        if (lo <= first_item) return first_item;
        return first_item + (lo - first_item + item_stride - 1) / item_stride * item_stride;
    };

    {
        // ---- two halves of the sequence blocks, overlapped ----
        // Each iteration's units are ordered [half 0][half 1].  Counters in
        // global memory synchronise the grid: done[h] counts CTAs whose
        // epilogue finished half h of an iteration (every partial winner in
        // the keys), committed[h] counts commit warps that committed it.  The
        // commit warps commit half h of iteration t once done[h] reaches
        // G (t + 1) while the other warps already compute the other half; the
        // producer loads half h of iteration t + 1 once committed[h] reaches
        // GC (t + 1).  No CTA ever waits for the whole grid to go idle.
        unsigned *done = a.barrier + 1, *committed = a.barrier + 3;
        const unsigned G = gridDim.x;
        const unsigned GC = G * kCommitWarps;  // commit warps in the grid
        const int64_t hb[3] = {0, half_units, work};
        if (warp == 0) {
            // ---------------- TMA producer ----------------
            if (lane == 0 && !kIsolate) {
                const uint64_t keep = l2_policy_evict_last();
                const uint64_t table_pol = a.keep_table ? keep : l2_policy_evict_normal();
                const uint64_t m_pol = l2_policy_evict_normal();
                for (int t = 0; t < a.L && !*abort_flag; ++t) {
                    stamp(a, t, 0);
                    bool first = true;
                    uint64_t waited = 0, gate = 0;
                    for (int h = 0; h < 2 && !*abort_flag; ++h) {
                        if (t > 0) {
                            // the queries of half h were committed for iteration t
                            if (!wait_counter(committed + h, GC * (unsigned)t, a.status, abort_flag,
                                              tmo, kStatusBarrierTimeout, &gate))
                                break;
                            fence_proxy_async_global();
                        }
                        for (int64_t v = first_from(hb[h]); v < hb[h + 1] && !*abort_flag;
                             v += item_stride)
                            produce_unit(t, v, keep, table_pol, m_pol, waited, first);
                    }
                    record(a, t, 7, gate);
                    record(a, t, 10, waited);
                }
            }
            __syncwarp();
        } else if (warp == 1) {
            // ---------------- MMA issuer (pair: the leader only) ----------------
            if (lane == 0 && leader) {
                for (int t = 0; t < a.L && !*abort_flag; ++t) {
                    bool first = true, ok = true;
                    uint64_t wait_full = 0, wait_acc = 0;
                    for (int64_t v = first_item; v < work && ok && !*abort_flag; v += item_stride)
                        ok = mma_unit(t, v, wait_full, wait_acc, first);
                    stamp(a, t, 3);
                    record(a, t, 8, wait_full);
                    record(a, t, 9, wait_acc);
                    if (!ok) break;
                }
            }
            __syncwarp();
        } else if (warp < 2 + kEpiWarps) {
            // ---------------- epilogue ----------------
            const uint64_t stream = l2_policy_evict_first();
            const uint32_t acc_empty_leader0 = mapa_shared(smem_u32(&acc_empty[0]), 0);
            bool skip_arrive = a.fault_skip_arrive && blockIdx.x == 0;
            bool ok = true;
            for (int t = 0; t < a.L && ok; ++t) {
                uint64_t epi_wait = 0;
                // falls with every iteration: every running minimum moves
                if (kIsolate) iso_d = 1.0f - (float)(t + 1) * (1.0f / 512.0f);
                for (int h = 0; h < 2 && ok; ++h) {
                    if (t > 0) {
                        // keys reset and winners masked for half h (the running
                        // minima this warp reads next)
                        int pass = 1;
                        if (lane == 0)
                            pass = wait_counter(committed + h, GC * (unsigned)t, a.status,
                                                abort_flag, tmo, kStatusBarrierTimeout, nullptr);
                        if (!__shfl_sync(0xffffffffu, pass, 0)) {
                            ok = false;
                            break;
                        }
                    }
                    for (int64_t v = first_from(hb[h]); v < hb[h + 1] && ok; v += item_stride)
                        ok = epilogue_unit(v, stream, acc_empty_leader0, epi_wait);
                    if (!ok) break;
                    // the last of this CTA's epilogue warps to finish half h
                    // publishes it (every key atomic of the CTA before it)
                    __syncwarp();
                    if (lane == 0) {
                        __threadfence();
                        const unsigned old = atomicAdd(&epi_arrive[h], 1u);
                        if (old % kEpiWarps == kEpiWarps - 1) {
                            __threadfence();
                            if (!skip_arrive) red_release_gpu_add(done + h, 1u);
                            skip_arrive = false;
                        }
                    }
                    __syncwarp();
                }
                if (warp == 2 && lane == 0) {
                    stamp(a, t, 4);
                    record(a, t, 11, epi_wait);
                }
            }
        } else {
            // ---------------- commit warp ----------------
            for (int t = 0; t < a.L; ++t) {
                bool ok = true;
                uint64_t wait_done = 0, busy = 0;
                for (int h = 0; h < 2; ++h) {
                    int pass = 1;
                    if (lane == 0)
                        pass = wait_counter(done + h, G * (unsigned)(t + 1), a.status, abort_flag,
                                            tmo, kStatusBarrierTimeout, &wait_done);
                    const uint64_t t_start = a.timeline ? globaltimer_ns() : 0;
                    if (!__shfl_sync(0xffffffffu, pass, 0)) {
                        ok = false;
                        break;
                    }
                    // this commit warp's share of the sequences of half h
                    const int s_lo = min(a.B, seq_half[h]);
                    const int s_hi = min(a.B, seq_half[h + 1]);
                    const int per = (s_hi - s_lo + (int)GC - 1) / (int)GC;
                    const int cw = (int)blockIdx.x * kCommitWarps + (warp - 2 - kEpiWarps);
                    const int b_lo = min(s_hi, s_lo + cw * per);
                    commit_range(t, b_lo, min(s_hi, b_lo + per));
                    fence_proxy_async_global();
                    __syncwarp();
                    if (lane == 0) {
                        __threadfence();
                        red_release_gpu_add(committed + h, 1u);
                        if (a.timeline) busy += globaltimer_ns() - t_start;
                    }
                    __syncwarp();
                }
                if (lane == 0 && warp == 2 + kEpiWarps) {
                    record(a, t, 5, busy);
                    record(a, t, 6, wait_done);
                }
                if (!ok) break;
            }
        }
    }

    // ---- teardown: drain what this CTA still has in flight, free TMEM ----
    __syncthreads();
    if (warp == 0 && lane == 0 && !*abort_flag) {
        // every stage this CTA filled has been consumed by the issuer; wait
        // (bounded) for the commits that say so, so that no tensor-core
        // arrival is still on its way to this CTA's barriers when it exits.
        // A failure reported anywhere in the grid ends the wait at once.
        const uint64_t lim = tmo < 1000000000ull ? tmo : 1000000000ull;
        for (uint32_t s = 0; s < (uint32_t)kSt && s < fills; ++s) {
            const uint32_t n_s = fills / kSt + (s < fills % kSt ? 1u : 0u);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&empty[s], (n_s - 1) & 1u)) {
                if (ld_volatile(a.status) != 0 || globaltimer_ns() - t0 > lim) break;
            }
        }
    }
    if (warp == 0 && lane == 0 && *abort_flag) {
        volatile int never = 0;
        if (kPair) {
            // the pair's copies complete on the leader's barriers: give the
            // ones still in flight time to land
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 200000ull) {
            }
        }
        if (!kPair || leader) {
            // wait (bounded) for the last fill of every stage that was ever filled
            for (uint32_t s = 0; s < (uint32_t)kSt && s < fills; ++s) {
                const uint32_t n_s = fills / kSt + (s < fills % kSt ? 1u : 0u);
                mbar_wait_bounded(&full[s], (n_s - 1) & 1u, &never, a.status,
                                  tmo < 1000000000ull ? tmo : 1000000000ull, kStatusPipeTimeout);
            }
        }
    }
    if (warp == 1 && lane == 0 && leader) {
        volatile int never = 0;
        if (kPair)
            umma_commit_pair(final_bar);
        else
            umma_commit(final_bar);
        mbar_wait_bounded(final_bar, 0, &never, a.status,
                          tmo < 1000000000ull ? tmo : 1000000000ull, kStatusPipeTimeout);
    }
    __syncthreads();
    // the leader's MMAs into both CTAs' TMEM are done before either frees it
    if (kPair) cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (kPair)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

void launch_tc_dseq_init_impl(const TcDseqArgs &a, const TcPlan &p, const int32_t *starts,
                         const uint8_t *mask, cudaStream_t st) {
    tc_dseq_init_kernel<<<2048, 256, 0, st>>>(a, p, starts, mask);
}

// Launch configuration of one instantiation: its thread count, its shared
// memory, clusters of two for the pair kernels.
template <bool kPair, bool kF16, bool kCentroid, bool kIsolate = false>
cudaError_t configure_variant(cudaLaunchConfig_t &cfg, cudaLaunchAttribute (&attr)[2],
                              unsigned grid, cudaStream_t st) {
    const size_t smem = DseqCfg<kPair, kF16, kCentroid>::kSmemBytes;
    cudaError_t err = cudaFuncSetAttribute(tc_dseq_kernel<kPair, kF16, kCentroid, kIsolate>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(dseq_threads<kCentroid>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    int n = 0;
    if (kPair) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaSuccess;
}

// The persistent kernel waits on counters that every CTA of the grid feeds,
// so the grid must be co-resident: it is launched cooperatively (with
// clusters of two for the pair kernels), and a launch the runtime refuses is
// returned as an error, never retried in another form.
template <bool kPair, bool kF16, bool kCentroid, bool kIsolate = false>
cudaError_t launch_variant(const TcDseqArgs &a, const TcPlan &p, const CUtensorMap &tmap_q,
                           const CUtensorMap &tmap_e, cudaStream_t st) {
    TcDseqArgs aa = a;
    TcPlan pp = p;
    CUtensorMap mq = tmap_q, me = tmap_e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    cudaError_t err =
        configure_variant<kPair, kF16, kCentroid, kIsolate>(cfg, attr, (unsigned)p.grid, st);
    if (err != cudaSuccess) return err;
    attr[cfg.numAttrs].id = cudaLaunchAttributeCooperative;
    attr[cfg.numAttrs].val.cooperative = 1;
    ++cfg.numAttrs;
    return cudaLaunchKernelEx(&cfg, tc_dseq_kernel<kPair, kF16, kCentroid, kIsolate>, mq, me, aa,
                              pp);
}

// CTAs of this instantiation that can be resident at once on the current
// device (pair kernels: whole clusters of two), from its own occupancy.
template <bool kPair, bool kF16, bool kCentroid>
int max_grid_variant() {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    if (configure_variant<kPair, kF16, kCentroid>(cfg, attr, kPair ? 2u : 1u, nullptr) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    auto kernel = tc_dseq_kernel<kPair, kF16, kCentroid>;
    if (kPair) {
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return 2 * clusters;
    }
    int per_sm = 0, dev = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, (int)cfg.blockDim.x,
                                                      cfg.dynamicSmemBytes) != cudaSuccess ||
        cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return per_sm * sms;
}

}  // namespace

void launch_tc_dseq_init(const TcDseqArgs &a, const TcPlan &p, const int32_t *starts,
                         const uint8_t *mask, cudaStream_t st) {
    launch_tc_dseq_init_impl(a, p, starts, mask, st);
}

cudaError_t launch_tc_dseq(const TcDseqArgs &a, const TcPlan &p, const CUtensorMap &tmap_q,
                           const CUtensorMap &tmap_e, cudaStream_t st) {
    const bool f16 = a.e_f16 != nullptr;
    if (a.isolate_epilogue) {
        if (a.centroid) return cudaErrorInvalidValue;
        if (p.pair)
            return f16 ? launch_variant<true, true, false, true>(a, p, tmap_q, tmap_e, st)
                       : launch_variant<true, false, false, true>(a, p, tmap_q, tmap_e, st);
        return f16 ? launch_variant<false, true, false, true>(a, p, tmap_q, tmap_e, st)
                   : launch_variant<false, false, false, true>(a, p, tmap_q, tmap_e, st);
    }
    if (a.centroid) {
        if (p.pair)
            return f16 ? launch_variant<true, true, true>(a, p, tmap_q, tmap_e, st)
                       : launch_variant<true, false, true>(a, p, tmap_q, tmap_e, st);
        return f16 ? launch_variant<false, true, true>(a, p, tmap_q, tmap_e, st)
                   : launch_variant<false, false, true>(a, p, tmap_q, tmap_e, st);
    }
    if (p.pair)
        return f16 ? launch_variant<true, true, false>(a, p, tmap_q, tmap_e, st)
                   : launch_variant<true, false, false>(a, p, tmap_q, tmap_e, st);
    return f16 ? launch_variant<false, true, false>(a, p, tmap_q, tmap_e, st)
               : launch_variant<false, false, false>(a, p, tmap_q, tmap_e, st);
}

int tc_dseq_max_grid(bool pair, bool f16, bool centroid) {
    if (centroid) {
        if (pair) return f16 ? max_grid_variant<true, true, true>() : max_grid_variant<true, false, true>();
        return f16 ? max_grid_variant<false, true, true>() : max_grid_variant<false, false, true>();
    }
    if (pair) return f16 ? max_grid_variant<true, true, false>() : max_grid_variant<true, false, false>();
    return f16 ? max_grid_variant<false, true, false>() : max_grid_variant<false, false, false>();
}

}  // namespace dseq
