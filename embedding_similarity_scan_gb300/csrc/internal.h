// internal.h — launchers and layouts shared between the host API (api.cu)
// and the kernel translation units of libdseq.so.  Plain pointers only.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dseq {

// device status word bits (OR-ed by any thread that gives up)
enum : int {
    kStatusBarrierTimeout = 1,
    kStatusPipeTimeout = 2,
    kStatusNoWinner = 4,
    kStatusNonFinite = 8,
    kStatusInternal = 16,
    kStatusBadIndex = 32,
};


// Rows of the query side (sequences / samples) per work unit: the 128 TMEM
// lanes of one tensor-core accumulator.
constexpr int kUnitRows = 128;
// K extent of one pipeline stage (fp16 elements = 64 bytes per row).
constexpr int kKBlock = 32;
// Pipeline stages of the tensor-core kernels.
constexpr int kStages = 4;
// Epilogue warps of the tensor-core kernels (two per TMEM lane quadrant).
constexpr int kEpiWarps = 8;
// Threads per CTA of the BMU kernel: TMA producer warp, MMA warp, epilogue
// warps (the diversity kernel adds its commit warps).
constexpr int kTcThreads = 32 * (2 + kEpiWarps);
// Bytes of one pipeline stage for a unit of tile_n candidate columns:
// A = 3 x (128 x 32) fp16 (hi*2^12, hi, lo*2^12), B = 2 x (tile_n x 32) fp16.
__host__ __device__ constexpr uint32_t tc_stage_bytes_a() { return 3u * kUnitRows * kKBlock * 2u; }
__host__ __device__ constexpr uint32_t tc_stage_bytes_b_max() { return 2u * 256u * kKBlock * 2u; }
__host__ __device__ constexpr uint32_t tc_smem_bytes() {
    return kStages * (tc_stage_bytes_a() + tc_stage_bytes_b_max()) + 1024u /*align*/ + 256u;
}

// Layout of the running-minimum array of the tensor-core path.  Candidate
// chunk j covers columns [col0(j), col0(j) + width(j)) (see TcPlan); the
// tiles of one chunk are contiguous, sequence block after sequence block, and
// work unit (beta, j) owns a tile of 128 x width(j) floats.  Inside a tile,
// element (row r, column c) with r = 32 q + t (TMEM lane quadrant q, lane t)
// and c = 32 g + 4 v + e sits at ((((g * 4 + q) * 8 + v) * 32 + t) * 4 + e),
// so each warp's 16-byte accesses of one column group are 512 contiguous bytes.
__host__ __device__ __forceinline__ int64_t tc_m_inner(int r, int c) {
    const int q = r >> 5, t = r & 31, g = c >> 5, v = (c >> 2) & 7, e = c & 3;
    return ((((g * 4 + q) * 8 + v) * 32 + t) * 4 + e);
}

// Phase stamps per CTA and iteration of the persistent diversity kernel:
// 0 producer starts the iteration, 1 first copy issued, 2 first MMA issued,
// 3 last MMA committed, 4 epilogue done (first epilogue warp); then
// nanoseconds spent in the iteration: 5 committing and 6 waiting for done
// halves (first commit warp), 7 producer waiting for committed queries,
// 8 MMA issuer waiting for filled stages, 9 for a free accumulator,
// 10 producer waiting for a free stage, 11 first epilogue warp waiting for a
// finished accumulator.
constexpr int kTimelineSlots = 12;

struct TcPlan {
    int n_beta;    // sequence blocks (ceil(B / 128))
    int n_chunk;   // candidate chunks
    int tile_n;    // candidate columns of the wide chunks (the TMA box)
    int grid;      // persistent CTAs (pair mode: even, two CTAs per cluster)
    int pair;      // 1: CTA pairs share each MMA (cta_group::2), n_beta even
    // chunks j < n_wide are tile_n columns wide, the others tile_n2 <= tile_n
    // (a uniform plan has n_wide = n_chunk, tile_n2 = tile_n)
    int n_wide;
    int tile_n2;
    __host__ __device__ int64_t units() const { return (int64_t)n_beta * n_chunk; }
    __host__ __device__ int width(int j) const { return j < n_wide ? tile_n : tile_n2; }
    __host__ __device__ int64_t col0(int j) const {
        return j <= n_wide ? (int64_t)j * tile_n
                           : (int64_t)n_wide * tile_n + (int64_t)(j - n_wide) * tile_n2;
    }
    __host__ __device__ int64_t columns() const { return col0(n_chunk); }
    __host__ __device__ int chunk_of(int64_t c) const {
        const int64_t wide = (int64_t)n_wide * tile_n;
        return c < wide ? (int)(c / tile_n) : n_wide + (int)((c - wide) / tile_n2);
    }
    // float offset of the running-minimum tile of unit (beta, j)
    __host__ __device__ int64_t tile_base(int j, int beta) const {
        return (col0(j) * n_beta + (int64_t)beta * width(j)) * kUnitRows;
    }
    __host__ __device__ void set_uniform(int tn, int64_t ncols) {
        tile_n = tile_n2 = tn;
        n_chunk = n_wide = (int)((ncols + tn - 1) / tn);
    }
};

// ---- table preparation (api.cu calls; prep.cu defines) ---------------------
// One warp per row: checks finiteness and a non-zero norm, writes the unit
// row (float, zero-padded to Dp), its split (hi | lo * 2^12) in fp16 and the
// row's norm.
void launch_table_prepare(const float *E, int64_t N, int D, int Dp, float *e_unit,
                          __half *e_split, float *nrm, int *status, cudaStream_t st);

// dst row i = src row map[i] for i < rows; rows of row_bytes bytes (a
// multiple of 4; of 16 for 16-byte copies, with both arrays 16-byte aligned).
void launch_gather_rows(const void *src, void *dst, const int32_t *map, int64_t rows,
                        int64_t row_bytes, cudaStream_t st);

// fp16 storage of the candidate table: row * 2^-e (max |.| in [0.5, 1)) rounded
// to fp16, zero-padded to Dp; rn[r] = 1 / |stored row| (compensated fp32 sum).
void launch_table_prepare_f16(const float *E, int64_t N, int D, int Dp, __half *e_f16,
                              float *rn, int *status, cudaStream_t st);
// out[r][k] = e_f16[r][k] as fp32 (exact)
void launch_f16_rows(const __half *e_f16, int64_t N, int Dp, float *out, cudaStream_t st);
// a[r] *= rn[r], b[r] *= rn[r]
void launch_scale_rows(float *a, float *b, const float *rn, int64_t N, cudaStream_t st);

// Rows of a BMU operand scaled by a per-row power of two (max |.| in [0.5, 1))
// and split into fp16.  triple = 1: [hi*2^12 | hi | lo*2^12] (the codebook,
// kBmuPartsW parts); triple = 0: [hi | lo*2^12] (the samples, kBmuPartsX
// parts).  norm2[r] = |row|^2 (compensated fp32 sum), inv_scale[r] = 1 / scale.
constexpr int kBmuPartsX = 2;
constexpr int kBmuPartsW = 3;
void launch_bmu_prepare(const float *A, int64_t rows, int D, int Dp, int triple, __half *split,
                        float *norm2, float *inv_scale, int *status, cudaStream_t st);

// ---- diversity, tensor-core path (tc_dseq.cu) -------------------------------
struct TcDseqArgs {
    const __half *e_split;   // N x 2Dp: [hi | lo * 2^12] of the unit rows (split storage)
    __half *q_split;         // Bp x 3Dp (split) or Bp x Dp (fp16 storage)
    // fp16 storage (nullptr = split storage): rows scaled by a power of two
    // and rounded to fp16, N x Dp; inverse norms of those stored rows
    const __half *e_f16;
    const float *rn;
    float *q_rn;             // Bp: inverse norm of each current query row
    // centroid criterion (centroid = 1): the query is the unit centroid of the
    // rows a sequence holds; csum (Bp x Dp) keeps their exact sum in fixed
    // point (2^-csum_shift units), rebuilt from the unit rows e_unit (N x Dp)
    // times the row norms nrm (N)
    int centroid;
    long long *csum;
    int csum_shift;
    int *c_exp;              // Bp: exponent sb of each query's scale 2^-sb (centroid)
    // centroid: one bit per (sequence, candidate), set for held, masked and
    // padding candidates; word (g, r) of tile (j, beta) at
    // tile_base(j, beta) / 32 + g * 128 + r covers columns 32 g .. 32 g + 31
    // of that tile for row r
    unsigned *held;
    const float *e_unit;
    const float *nrm;
    float *m;                // units x 128 x tile_n
    unsigned long long *keys;  // Bp
    int32_t *picks;          // B x L
    const int32_t *trace_slot;  // Bp (-1 = not traced) or nullptr
    float *trace;            // n_trace x L x N
    int *status;
    unsigned *barrier;
    int64_t N;               // candidate columns the kernel scans
    int B, L, Dp;
    uint64_t timeout_ns;
    int fault_skip_arrive;
    // global-mask compaction (col_map == nullptr: none).  The kernel then
    // scans only the unmasked rows: e_split / e_f16 / rn hold them in table
    // order, col_map[c] (N) is the table row of column c and comp_of[r]
    // (n_table) the column of table row r, or -1 for a masked row.  The
    // *_full pointers always address the whole table (the first queries are
    // the start rows, which may be masked); n_table is its row count, the
    // width of a trace row.
    const int32_t *col_map;
    const int32_t *comp_of;
    const __half *e_split_full;
    const __half *e_f16_full;
    const float *rn_full;
    int64_t n_table;
    int keep_table;  // 1: load table tiles with the evict-last L2 policy (table fits L2)
    // optional [L][grid][kTimelineSlots] globaltimer stamps (nullptr = off)
    unsigned long long *timeline;
    // measurement only (max-min): run the epilogue-isolated kernel, whose
    // contraction is compiled out (picks meaningless)
    int isolate_epilogue;
};
void launch_tc_dseq_init(const TcDseqArgs &a, const TcPlan &p, const int32_t *starts,
                         const uint8_t *mask, cudaStream_t st);
cudaError_t launch_tc_dseq(const TcDseqArgs &a, const TcPlan &p, const CUtensorMap &tmap_q,
                           const CUtensorMap &tmap_e, cudaStream_t st);
// CTAs of the persistent kernel variant (pair, fp16 storage, centroid) that
// can be co-resident on the current device, from that instantiation's own
// thread count and shared memory (pair: twice its co-resident clusters of
// two); 0 on error
int tc_dseq_max_grid(bool pair, bool f16, bool centroid);

// ---- diversity, Gram engine (gram.cu; the Gram product in tc_bmu.cu) --------
struct GramWalkArgs {
    const float *G;          // N x Np: distances 1 - <e_p, e_c> of the unit rows
    float *m;                // B x Np running minima, row-major (in and out)
    int32_t *cur;            // B: the newest row of each sequence (in and out)
    int32_t *picks;          // B x L
    const int32_t *trace_slot;  // B (-1 = not traced) or nullptr
    float *trace;            // n_trace x L x N
    int *status;
    int64_t N, Np;           // table rows; row stride of G and m (a multiple of 32)
    int B, L;
    // a fresh run with the running minima on chip (registers or shared
    // memory): the walk sets them up itself from the starts and the mask
    // (nullptr: read m and cur, as left by gram_walk_init or an earlier run)
    const int32_t *starts;
    const uint8_t *mask;
    // where the running minima live during the walk: 1 one CTA's registers
    // or shared memory, 2 a cluster's shared memory, 3 global memory
    // (gram_walk_place)
    int place;
    uint64_t timeout_ns;     // limit of the cluster walk's wait for its peers
};
// The default place of a walk's running minima for rows of Np floats.
int gram_walk_place(int64_t Np);
// Largest running-minimum row (bytes) one CTA takes when that place is asked
// for (the default place keeps one CTA to 64 KB: gram_walk_place); rows up
// to kGramWalkClusterMax are spread over the shared memory of a cluster of
// 8 CTAs; longer still, they stay in global memory.
constexpr size_t kGramWalkSmemMax = 96 * 1024;
constexpr size_t kGramWalkClusterMax = 8 * 96 * 1024;
// m <- +inf, or -inf for masked rows, the start and the row padding; cur <- starts.
void launch_gram_walk_init(const GramWalkArgs &a, const int32_t *starts, const uint8_t *mask,
                           cudaStream_t st);
// All L iterations of every sequence in one launch: one CTA or one cluster
// of 8 CTAs per sequence, as a.place says.
cudaError_t launch_gram_walk(const GramWalkArgs &a, cudaStream_t st);

// ---- diversity, FFMA path (ffma.cu) -----------------------------------------
struct FfmaDseqArgs {
    const float *e_unit;   // N x Dp
    float *q;              // Bp x Dp
    float *m;              // Bp x Nf (Nf: N rounded up to 128)
    unsigned long long *keys;
    int32_t *picks;
    const int32_t *trace_slot;
    float *trace;
    int *status;
    int64_t N, Nf;
    int B, Bp, L, Dp;
};
// Sets the FFMA kernels' shared-memory limit; call before their launches.
cudaError_t ffma_configure();
void launch_ffma_dseq_init(const FfmaDseqArgs &a, const int32_t *starts, const uint8_t *mask,
                           cudaStream_t st);
void launch_ffma_dseq_iteration(const FfmaDseqArgs &a, int t, cudaStream_t st);

// ---- BMU ----------------------------------------------------------------------
struct BmuArgs {
    const float *X, *W;          // fp32 inputs (FFMA path)
    const __half *x_split;       // n x kBmuPartsX*Dp (tensor path)
    const __half *w_split;       // M x kBmuPartsW*Dp (tensor path)
    const float *xn, *wn;        // squared norms
    const float *x_inv_scale, *w_inv_scale;
    unsigned long long *keys;    // n
    int32_t *idx;
    float *dist;
    int *status;
    int64_t n, M;
    int D, Dp;
    uint64_t timeout_ns;
    // test only: CTA 0 leaves out one copy of its first codebook stage, so
    // that stage never fills and the waits on it run out
    int fault_skip_copy;
    // Gram product (launch_tc_gram): 1 - <e_i, e_c> stored at gram[c * gram_ld + i]
    float *gram;
    int64_t gram_ld;
};
void launch_bmu_keys_init(unsigned long long *keys, int64_t n, cudaStream_t st);
void launch_ffma_bmu(const BmuArgs &a, cudaStream_t st);
// slice_chunks: neuron chunks per L2 slice, 0 = about 30 % of L2.
cudaError_t launch_tc_bmu(const BmuArgs &a, const TcPlan &p, const CUtensorMap &tmap_x,
                          const CUtensorMap &tmap_w, int slice_chunks, cudaStream_t st);
void launch_bmu_finalize(const BmuArgs &a, cudaStream_t st);
// The Gram product of one table, G = E E^T, on the BMU kernel's tensor-core
// pipeline (CTA pairs, the streaming operand ring) with a store epilogue: the
// sample side (x_split, x_inv_scale, n rows) and the codebook side (w_split,
// w_inv_scale, M = n rows) are the same table's rows split twice; a.gram
// receives G (row stride gram_ld >= n).  p: n_beta (even) sample blocks,
// uniform 256-wide chunks of the table, an even grid.
cudaError_t launch_tc_gram(const BmuArgs &a, const TcPlan &p, const CUtensorMap &tmap_x,
                           const CUtensorMap &tmap_w, cudaStream_t st);
void launch_row_sqnorm(const float *A, int64_t rows, int D, float *out, int *status,
                       cudaStream_t st);

// ---- SOM neighbourhood update -------------------------------------------------
// Largest neighbourhood window half-width (grid steps).
constexpr int kSomMaxRadius = 255;
constexpr int kSomScanTile = 4096;  // neurons per tile of the offsets' scan
constexpr int kSomChunk = 32;       // grouped samples per accumulating warp
struct SomArgs {
    const float *X;        // n x D samples
    const int32_t *bmu;    // n
    float *W;              // M x D codebook, updated in place
    long long *S;          // M x D per-neuron sample sums, fixed point (rows of
                           // neurons without samples are neither written nor read)
    unsigned *cnt;         // M per-neuron sample counts (cleared by the host)
    unsigned *cursor;      // M samples placed per neuron so far (cleared by the host)
    unsigned *off;         // M offsets of each neuron's samples within its scan tile
    unsigned *tile_sum;    // samples per tile of kSomScanTile neurons
    unsigned *tile_off;    // exclusive prefix of tile_sum
    int32_t *order;        // n sample indices grouped by BMU
    float *T;              // M x D row-smoothed sums
    float *Tc;             // M row-smoothed counts
    int *status;
    unsigned *maxbits;     // bits of max |x| (cleared by the host)
    int64_t n, M;
    int D, side_x, side_y, R;
    float g[kSomMaxRadius + 1];  // g[k] = exp(-k^2 / (2 sigma^2)), k = 0..R
};
cudaError_t launch_som_update(const SomArgs &a, int sms, cudaStream_t st);

// ---- host helpers of api.cu used by noalloc.cu --------------------------------
namespace host {
int fail_msg(int code, const char *msg);
void clear_error();
// on_device: p is device (or managed) memory of the current device; device
// memory of another device is an error (DSEQ_EINVAL with a message)
int locate_ptr(const void *p, const char *what, bool &on_device);
int sm_count(int dev, int *sms);
int encode_map(CUtensorMap &map, const void *base, int64_t cols, int64_t rows, int box_rows);
int read_device_status(int *status_dev, cudaStream_t st);
}  // namespace host

}  // namespace dseq
