/*
 * dseq.h — C ABI of the embedding similarity scan library (libdseq.so).
 *
 * One data-parallel hot path serves two uses:
 *
 *  - Greedy diversity sequences ("Issue 9-014: Tile Diversity Shader Inner
 *    Loop For L2 Cache Locality", Current Behavior and Intended Behavior).
 *    Each of B independent sequences holds its newest pick; every iteration
 *    computes the cosine distance of that pick to all N candidate rows,
 *    folds it into the sequence's running minimum distance, and picks the
 *    unmasked candidate whose running minimum is largest, lowest index on
 *    ties (the max-min, farthest-first reading of the criterion of "Issue
 *    9-014: Tile Diversity Shader Inner Loop For L2 Cache Locality").  The
 *    candidate scan is tiled and the running (max, index) carried across
 *    tiles, which by associativity of max gives the one-pass winner (same
 *    issue, Intended Behavior).
 *
 *  - Best-matching-unit search ("From 80x to 385x: A Best-Matching-Unit
 *    Search at the L2 Roof", section 3 Background, and section 4.2, neuron-
 *    axis chunking): for every sample, the codebook row at the smallest
 *    squared Euclidean distance, lowest index on ties, with the argmin fused
 *    into the product so the sample x neuron score block is never stored.
 *
 * Conventions shared by every call:
 *  - Return value: DSEQ_OK (0) on success, a negative DSEQ_E* code on error;
 *    dseq_last_error() then returns a message for the calling thread.
 *    Outputs are unspecified after an error.
 *  - Array arguments may be host or device pointers (the library inspects
 *    each with cudaPointerGetAttributes); host arrays are staged through
 *    library-owned device buffers on the given stream.  Pinned host memory
 *    makes those copies asynchronous.  Device arrays must be memory of the
 *    current device: a pointer into another GPU's memory is rejected with
 *    DSEQ_EINVAL before any work is enqueued.
 *  - cuda_stream is a cudaStream_t (NULL = the legacy default stream) on the
 *    current device.  Every call is synchronous at return: it enqueues its
 *    work on the stream, synchronizes the stream and reads back the device
 *    status word.
 *  - All tables are row-major float32, rows contiguous.  The caller owns
 *    every array it passes; the library never frees or retains them past
 *    the call (dseq_create copies the table).
 *  - Calls on one dseq_ctx must not overlap; bmu_search and distinct
 *    contexts may be used from different threads.
 */
#ifndef DSEQ_H
#define DSEQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    DSEQ_OK = 0,
    DSEQ_EINVAL = -1,     /* NULL pointer, bad size, start out of range or repeated, L too large */
    DSEQ_ENONFINITE = -2, /* NaN / Inf in an input table, or an all-zero table row */
    DSEQ_ENOMEM = -3,     /* device allocation failed */
    DSEQ_ELAUNCH = -4,    /* the runtime refused the persistent grid's cooperative launch */
    DSEQ_ETIMEOUT = -5,   /* a device-side wait gave up (the kernel returned cleanly) */
    DSEQ_ECUDA = -6,      /* any other CUDA runtime / driver error */
    DSEQ_EINTERNAL = -7   /* an internal consistency check failed on the device */
};

/* Opaque context: owns the device copy of one candidate table (unit-norm
 * rows, float32 and the split half-precision pair used by the tensor-core
 * path) and the workspace of its runs (running minimum distances, current
 * query rows, per-sequence argmax keys, barrier counters, status word). */
typedef struct dseq_ctx dseq_ctx;

/* Upload a candidate table of N rows x D float32 columns and prepare it.
 *   table            N*D floats, row-major; host or device memory.
 *   N                number of candidates, 1 <= N < 2^31.
 *   D                embedding dimension, 1 <= D <= 16384.
 *   table_on_device  ignored (kept for source compatibility: the pointer
 *                    kind is detected); pass 0 or 1.
 *   cuda_stream      stream for the upload and preparation kernels.
 *   out              receives the new context (NULL on error).
 * Errors: DSEQ_EINVAL (NULL pointer, N or D out of range), DSEQ_ENONFINITE
 * (a NaN/Inf element or a row whose norm is zero: cosine distance is
 * undefined there), DSEQ_ENOMEM, DSEQ_ECUDA.  The table is copied; the
 * caller may free it when the call returns. */
int dseq_create(const float *table, int64_t N, int32_t D, int table_on_device,
                void *cuda_stream, dseq_ctx **out);

/* Run B greedy max-min diversity sequences of L picks each.
 *   starts   int32[B]: the start row of each sequence; distinct, in [0, N).
 *   B        number of sequences, >= 1.
 *   L        picks per sequence after its start, >= 0.
 *   mask     uint8[N] or NULL: mask[c] != 0 excludes row c from every
 *            sequence (a start may itself be masked).
 *   picks    int32[B*L], out: picks[b*L + t] is the t-th pick of sequence b
 *            after its start (the start itself is not included); may be
 *            NULL when L = 0.
 * Semantics (one iteration t, every sequence b, p = the newest row of b):
 *   m_b[c] <- min(m_b[c], 1 - <e_p, e_c> / (|e_p| |e_c|)) for every c,
 *   pick = argmax over unmasked c of m_b[c], ties to the lowest c,
 *   with m_b initialised to +inf and the start masked.
 * Errors: DSEQ_EINVAL (NULL pointers, B < 1, L < 0, a start out of range or
 * repeated, or L larger than the candidates some sequence has left:
 * N - |mask U {start_b}|), DSEQ_ENOMEM, DSEQ_ELAUNCH, DSEQ_ETIMEOUT,
 * DSEQ_ECUDA, DSEQ_EINTERNAL. */
int dseq_run(dseq_ctx *ctx, const int32_t *starts, int32_t B, int32_t L, const uint8_t *mask,
             int32_t *picks, void *cuda_stream);

/* dseq_run that also records the running minimum distances of selected
 * sequences after every fold (for parity checks).
 *   trace_seqs      int32[n_trace]: distinct sequence indices in [0, B).
 *   trace_mindist   float[n_trace * L * N], out, DEVICE memory only:
 *                   trace_mindist[(k*L + t)*N + c] = m_{trace_seqs[k]}[c]
 *                   after the fold of iteration t, before pick t is masked.
 *                   Masked candidates (the global mask, the start and the
 *                   picks before t) hold -inf.
 * Errors: as dseq_run, plus DSEQ_EINVAL for a host trace buffer or bad
 * trace indices. */
int dseq_run_trace(dseq_ctx *ctx, const int32_t *starts, int32_t B, int32_t L,
                   const uint8_t *mask, int32_t *picks, const int32_t *trace_seqs,
                   int32_t n_trace, float *trace_mindist, void *cuda_stream);

/* Phase timestamps of the last dseq_run on ctx made with the "timeline"
 * option on (tensor-core path).  out receives iters x grid x 12 int64
 * values per iteration and CTA: nanosecond stamps (%globaltimer) 0 the
 * producer starts the iteration, 1 its first copy issued, 2 first MMA
 * issued, 3 last MMA committed, 4 epilogue done; then nanoseconds spent in
 * the iteration: 5 by the CTA's first commit warp committing, 6 by it
 * waiting for the halves to be done, 7 by the producer waiting for
 * committed queries, 8 by the MMA issuer waiting for filled stages, 9 by it
 * waiting for a free accumulator, 10 by the producer waiting for a free
 * stage, 11 by the first epilogue warp waiting for a finished accumulator
 * (slots 2, 3, 8 and 9 only on CTAs that issue MMAs).  *iters and *grid
 * receive the dimensions (0 when no timeline was recorded); capacity is the
 * length of out in elements; out = NULL only queries the dimensions.
 * Errors: DSEQ_EINVAL (NULL ctx/iters/grid, capacity too small), DSEQ_ECUDA. */
int dseq_get_timeline(dseq_ctx *ctx, int64_t *out, int64_t capacity, int32_t *iters,
                      int32_t *grid);

/* Free the context and everything it owns.  NULL is accepted. */
void dseq_destroy(dseq_ctx *ctx);

/* Best-matching-unit search of n samples against an M-neuron codebook.
 *   X     float[n*D] samples, row-major; host or device.
 *   W     float[M*D] codebook, row-major (neuron j = row j); host or device.
 *   idx   int32[n], out: argmin_j |X_i - W_j|^2, ties to the lowest j.
 *   dist  float[n], out: that squared distance, clamped at 0 (computed as
 *         |x|^2 + (|w_j|^2 - 2<x, w_j>) with both norms precomputed).
 * Sizes: 1 <= n, M < 2^31, 1 <= D <= 16384.
 * Errors: DSEQ_EINVAL, DSEQ_ENONFINITE (NaN/Inf in X or W), DSEQ_ENOMEM,
 * DSEQ_ETIMEOUT, DSEQ_ECUDA. */
int bmu_search(const float *X, int64_t n, const float *W, int64_t M, int32_t D, int32_t *idx,
               float *dist, void *cuda_stream);

/* Neighbourhood update of a self-organising map from every sample's BMU,
 * the step that follows the BMU search in an epoch ("From 80x to 385x: A
 * Best-Matching-Unit Search at the L2 Roof", section 3 Background: each
 * sample's closest neuron is found, then that neuron and its neighbours are
 * updated).  The batch map:
 *   W_j <- sum_i h(j, bmu_i) X_i / sum_i h(j, bmu_i)   (W_j kept if the sum is 0)
 * on a planar side_x x side_y grid, neuron j at column j % side_x and row
 * j / side_x, with h = exp(-(dx^2 + dy^2) / (2 sigma^2)) for |dx|, |dy| <=
 * radius and 0 outside that square window (sigma = 0: a neuron takes the
 * mean of its own samples).
 *   X       float[n*D] samples, row-major; host or device.
 *   W       float[M*D], M = side_x * side_y, updated in place; host or device.
 *   bmu     int32[n], every sample's neuron in [0, M); host or device.
 *   sigma   >= 0; radius in [0, 255] and, for sigma > 0, radius <= 9 sigma
 *           (wider windows would take weights below fp32's normal range).
 * Sums over samples are exact: each sample is converted to 64-bit integer
 * fixed point (a scale set by the largest |x|) and the sums are integer
 * additions, so the result does not depend on the order in which samples
 * are added; the smoothing and the division are fp32.  n = 0 leaves W
 * unchanged.  On any error W is left unchanged.
 * Errors: DSEQ_EINVAL (sizes, sigma, radius, a BMU out of range),
 * DSEQ_ENONFINITE (NaN/Inf in X), DSEQ_ENOMEM, DSEQ_ECUDA. */
int som_update(const float *X, int64_t n, float *W, int32_t side_x, int32_t side_y, int32_t D,
               const int32_t *bmu, double sigma, int32_t radius, void *cuda_stream);

/* One SOM epoch: bmu_search of every sample against W, then som_update of W
 * with those BMUs, on the stream.  bmu_out (int32[n]) and dist_out
 * (float[n]) receive the search's results and may each be NULL; host or
 * device.  The search follows the process-wide options as bmu_search does.
 * dseq_last_stat("kernel_ns") is the search kernel's time and
 * dseq_last_stat("update_ns") the update's.
 * Sizes: n >= 1, otherwise as som_update.  Errors: those of bmu_search and
 * som_update; on an error W is left unchanged. */
int som_epoch(const float *X, int64_t n, float *W, int32_t side_x, int32_t side_y, int32_t D,
              double sigma, int32_t radius, int32_t *bmu_out, float *dist_out,
              void *cuda_stream);

/* bmu_search for callers that cannot allocate device memory: code inside a
 * framework whose pooling allocator already holds nearly all of the GPU's
 * memory (a cudaMalloc there fails, or takes memory the pool counts on), or
 * a latency-critical loop that cannot absorb the device-wide synchronisation
 * cudaMalloc / cudaFree may imply.  The method pages have no counterpart of
 * this entry point; it exists for such callers only.
 * Same arguments, semantics and results as bmu_search, except:
 *  - X, W, idx and dist must all be device memory of the current device
 *    (nothing is staged; memory of another device is rejected);
 *  - no call allocates: the scratch (split operands, norms, scales, keys,
 *    status) lives in one fixed 64 MiB array inside the library, which every
 *    GPU that loads the library holds until the process exits.  A request
 *    needing more (about n*(4*Dp + 16) + M*(6*Dp + 8) bytes, Dp = D rounded
 *    up to 32) fails with DSEQ_EINVAL and says how much it needed;
 *  - every call shares that one array, so calls whose GPU work overlaps
 *    (other threads, other streams) race and give wrong results: serialise
 *    them.  Each call resets the parts that must start from a known value;
 *  - set-up: the first call on a device looks up the array's device address
 *    (once per device, with that device current) and keeps it for the rest
 *    of the process; make that first call before any stream capture.  The
 *    kept address is not valid after cudaDeviceReset on that device: do not
 *    call this entry point on a device after resetting it;
 *  - every call enqueues its kernels on cuda_stream, synchronises that
 *    stream and reads the device status word back to the host before it
 *    returns;
 *  - the process-wide "engine", "tile_n", "grid" and "timeout_ms" options do
 *    not apply: the tensor-core path always runs on CTA pairs, 256 neurons
 *    per unit, one CTA per SM, 10 s wait limit.
 * Errors: DSEQ_EINVAL (as bmu_search, host pointers or memory of another
 * device, scratch too small), DSEQ_ENONFINITE, DSEQ_ETIMEOUT, DSEQ_ECUDA. */
int bmu_search_noalloc(const float *X, int64_t n, const float *W, int64_t M, int32_t D,
                       int32_t *idx, float *dist, void *cuda_stream);

/* Tuning and test knobs.  ctx = NULL sets the process-wide default used by
 * bmu_search and by contexts created afterwards; otherwise the setting
 * applies to that context only.  Names:
 *   "engine"      0 = tensor-core path (default), 1 = FP32 FFMA path.
 *   "gram"        diversity path: how dseq_run finds the distances.
 *                 0 = per iteration, the newest picks against the whole
 *                 table on the tensor cores, fused with the fold and the
 *                 argmax (the scan); 1 = the table's Gram matrix G = E E^T
 *                 of the unit rows once per run on the tensor cores, stored
 *                 as the distances 1 - G (N x Np float32, Np = N rounded up
 *                 to 32; the tiles on and above the diagonal are computed
 *                 and every entry is stored at (i, c) and (c, i), so the
 *                 matrix is exactly symmetric), then one CTA (or cluster)
 *                 per sequence reads the row of its newest pick p every
 *                 iteration, distance 1 - G[p][c]; 2 = 1 where
 *                 a cost model (the product plus B * L row reads against B *
 *                 L table scans) says it is cheaper and G fits in 80 % of
 *                 the free device memory, else 0 (default).  Both give the
 *                 same picks up to fp32 rounding of the distances, with the
 *                 same tie-break.  With storage 1, G holds the inner
 *                 products of the stored fp16 rows' unit vectors (the
 *                 distances of that storage).  Only the max-min criterion
 *                 with the tensor-core engine (and neither timeline nor
 *                 isolate_epilogue) uses G; other settings run the scan.
 *                 A resumed run stays on the engine of the run it resumes.
 *   "walk"        Gram engine: where each sequence keeps its running minima
 *                 while it reads G.  0 = chosen from N (default): one CTA
 *                 per sequence up to 64 KB of minima (N <= 16384; in its
 *                 registers for N <= 8704, else in its shared memory),
 *                 spread over the shared memory of a cluster of 8 CTAs up
 *                 to 768 KB (N <= 196608), global memory beyond; 1, 2, 3
 *                 force one CTA (up to 96 KB, N <= 24576), cluster,
 *                 global memory (DSEQ_EINVAL from dseq_run when the row
 *                 does not fit the place asked for).
 *                 Every place gives identical picks.
 *   "tile_n"      candidate (or neuron) columns per work unit, a multiple of
 *                 32 in [32, 256]; 0 = chosen from the shape (default).
 *                 Alone it fixes every diversity chunk to that width.
 *   "tile_n2"     diversity path: width of the narrower chunks that follow
 *                 the tile_n-wide ones (a multiple of 32, <= tile_n); 0 =
 *                 chosen with tile_n (default).  Mixing two widths balances
 *                 the work units over the SMs without narrowing every MMA.
 *   "grid"        persistent CTAs; 0 = as many as can be co-resident for the
 *                 kernel variant that runs (its own occupancy; one per SM
 *                 for the tensor-core kernels) (default).  A diversity grid
 *                 larger than can be co-resident is refused by the
 *                 cooperative launch: dseq_run returns DSEQ_ELAUNCH.
 *   "timeout_ms"  limit of every device-side wait (default 10000).
 *   "cache_mb"    process-wide only (ctx must be NULL): device memory, per
 *                 device, that the library keeps for reuse after a context
 *                 is destroyed or a call's staging buffers are no longer
 *                 needed, instead of freeing it; later contexts and calls
 *                 take buffers of a similar size from it, so a create /
 *                 run / destroy cycle maps no new device memory once warm.
 *                 Default -1: half of each device's memory (a Gram
 *                 matrix of N = 131072 is 68.7 GB; freeing and mapping it
 *                 again costs a create / run / destroy cycle about 60 ms);
 *                 0 keeps nothing; -1 restores the default.  Lowering it
 *                 frees kept buffers down to the new limit at once; a
 *                 failed allocation frees the device's kept buffers and
 *                 retries.  That memory is not available to other
 *                 allocators in the process (torch's among them) while it
 *                 is kept; the engine choice counts it as free.
 *   "resume"      1 = dseq_run continues the last successful run on this
 *                 context from the state it left on the device (running
 *                 minima, current queries): the same starts, mask and
 *                 engine / pair / storage / criterion settings are required,
 *                 picks[b*L + t] then holds pick (earlier picks + t) of
 *                 sequence b, and L may use the candidates left after the
 *                 earlier picks.  A long ordering (L up to N - 1) can so be
 *                 made in chunks, with results identical to one long call.
 *                 Default 0 (every call starts its sequences afresh).
 *   "criterion"   0 = max-min (default): a candidate's score is its smallest
 *                 cosine distance to any row the sequence holds; 1 = centroid:
 *                 its cosine distance to the centroid (plain mean) of those
 *                 rows, a zero centroid giving distance 1 (the ranking by
 *                 distance from the centroid in "Issue 9-014: Tile
 *                 Diversity Shader Inner Loop For L2 Cache Locality",
 *                 section FP16 storage (compounding optimization)).  With 1,
 *                 dseq_run_trace records these centroid distances instead
 *                 of running minima.  Tensor-core engine only (DSEQ_EINVAL
 *                 with engine 1); with storage 1 the table is held as fp16
 *                 rows and the centroid query keeps fp32-level precision
 *                 (two fp16 parts), so the distance is the cosine between
 *                 the exact centroid and the stored row.
 *   "storage"     how the diversity kernel holds the table: 0 = fp16 hi/lo
 *                 split of the unit rows, three tensor-core products per
 *                 step, fp32-level distances (default); 1 = fp16 rows (each
 *                 row scaled by a power of two, then rounded once to fp16),
 *                 one product per step, distances exact for the stored rows
 *                 up to fp32 accumulation (fp16 in memory, fp32 arithmetic).
 *   "pair"        1 = the tensor-core kernels run on CTA pairs (clusters of
 *                 two SMs) that share each MMA (each SM stages half of the
 *                 candidate or neuron tile; default); 0 = one CTA per MMA.
 *   "compact"     1 = when dseq_run's mask removes at least 1/16 of the
 *                 table, the tensor-core kernel scans only the unmasked rows
 *                 (gathered once per call; picks are mapped back to table
 *                 rows, ties still go to the lowest row; results identical to
 *                 the full scan); default.  0 = always scan the whole table.
 *   "slice"       bmu_search: neuron chunks per codebook slice, the part of
 *                 the codebook every CTA sweeps against all samples before
 *                 moving on; 0 = as many as fill about 30 % of L2 (default).
 *                 Any value gives the same results.
 *   "timeline"    1 = dseq_run records, per CTA and iteration of the
 *                 tensor-core kernel, device timestamps of its phases (read
 *                 them back with dseq_get_timeline); default 0.
 *   "fault_skip_arrive"  test only: 1 makes CTA 0 skip its first arrival on
 *                 the cross-CTA "half done" counter, so the other CTAs'
 *                 waits run out (the kernel then returns DSEQ_ETIMEOUT
 *                 without hanging).
 *   "fault_skip_copy"    test only: 1 makes CTA 0 of the tensor-core BMU
 *                 kernels leave out one copy of its first codebook stage, so
 *                 that stage never fills and the waits on it run out
 *                 (bmu_search then returns DSEQ_ETIMEOUT without hanging).
 *   "isolate_epilogue"   measurement only: 1 makes dseq_run launch the
 *                 max-min tensor-core kernel with its contraction compiled
 *                 out (no operand copies, no MMAs) and a stand-in distance
 *                 that falls every iteration, so that the fused epilogue's
 *                 running-minimum stream, the commit and the cross-CTA
 *                 synchronisation run alone; its picks are meaningless.
 *   The three test options accept a non-zero value only when the
 *   environment variable DSEQ_ENABLE_TEST_OPTIONS is "1" (DSEQ_EINVAL
 *   otherwise); 0 is always accepted.
 * Errors: DSEQ_EINVAL for an unknown name or a value out of range. */
int dseq_set_option(dseq_ctx *ctx, const char *name, int64_t value);

/* Read back a knob (the value in effect; -1 for an unknown name). */
int64_t dseq_get_option(dseq_ctx *ctx, const char *name);

/* Statistics of the last successful dseq_run / bmu_search / som_update /
 * som_epoch on this thread:
 *   "units"        work units (sequence block x candidate chunk) per iteration;
 *                  neurons for som_update,
 *   "tile_n"       candidate columns per (wide) unit, "tile_n2" of the narrow
 *                  units, "n_wide" the number of wide chunks (diversity path),
 *   "grid"         CTAs launched,
 *   "launches"     kernels launched by the call,
 *   "kernel_ns"    device time of the main kernel (CUDA events; 0 if unknown),
 *   "update_ns"    device time of the SOM update's kernels (0 if none ran),
 *   "gram"         1 if the last dseq_run used the Gram engine, else 0,
 *   "gram_ns"      its Gram product's device time (operand split included),
 *   "walk_ns"      its walk's device time,
 *   "walk"         where that walk kept its running minima (1 one CTA's
 *                  registers or shared memory, 2 cluster, 3 global
 *                  memory). */
int64_t dseq_last_stat(const char *name);

/* Message of the last error on the calling thread ("" if none). */
const char *dseq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DSEQ_H */
