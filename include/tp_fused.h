/*
 * tp_fused.h -- tensor-parallel sharded Linear on one GB300 (sm_103a).
 *
 * All p "ranks" of a tensor-parallel Linear live in one GPU's memory; rank
 * r's shards are plain device pointers.  Each entry point runs the per-rank
 * partial GEMMs fused with their cross-shard reduction (or gather): the p
 * partials of an output tile are accumulated in one fp32 tensor-memory
 * accumulator in rank order r = 0..p-1 and the tile is written once.  (On
 * contractions of 8192 and deeper, the CTA-pair kernel runs the tiles of
 * every other wave in the reverse order, p-1..0 and last k-block first, so
 * that a wave re-reads from L2 what the previous one read last; the order
 * of each tile is fixed by the shapes and the GPU's SM count, so results
 * are reproducible.)  Rows
 * are processed chunk by chunk along M (chunk-major tile order), and a
 * tile's write-out overlaps the next tile's MMAs.
 *
 * Sources (web pages, cited by title and section):
 *   [M027] ai-infra-kb M027 "compute-communication fusion":
 *          §01 row-parallel Linear, AllReduce vs ReduceScatter layouts,
 *          AllGather then MatMul; §02-§03 the chunked pipeline and its
 *          timeline; §05 small (decode) matrices.
 *   [TP]   cnblogs zuoyang/p/22340322 "PyTorch 2.x tensor parallelism":
 *          §2.3 column parallel, §2.4 row parallel, §2.5-2.7 collectives,
 *          §三/§四/§六 forward and backward, §7.1 MLP block, §11.3 SP pair.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Matrices are row-major.  Weights are [in, out] (Y = X . A, [TP] §2.3).
 *  - Tensor pointers are DEVICE pointers owned by the caller.  Pointer
 *    arrays (x, w, y, ...) are HOST arrays of length p (or n_out); they are
 *    read during the call only.  The library never allocates or frees
 *    device memory on a call; all work is enqueued on `stream`.
 *  - Inputs are bfloat16.  Outputs are bfloat16 (rounded to nearest even,
 *    once) or float32, chosen by `out_dtype`.  Accumulation is fp32.
 *  - 1 <= p <= 8.  Every base pointer is 16-byte aligned; every row pitch is
 *    a multiple of 16 bytes, i.e. K and N are multiples of 8.
 *  - `chunk_m`: rows per pipeline chunk.  0 lets the scheduler choose
 *    (tp_choose_chunk_m); a value above M is clamped to M; the last chunk
 *    may be short.  Chunks of 128 rows or more run on 128-row tiles; chunks
 *    below 128 rows run the operand-swapped kernel whose token tile is the
 *    chunk (rounded up to a multiple of 16).
 *  - Outputs must not overlap inputs (checked; TP_ERR_INVALID_ARG).
 *  - `ws` is a device workspace of at least tp_workspace_size(...) bytes,
 *    16-byte aligned, zero-filled before its first use.  It holds the
 *    device status word (which stays zero unless a device wait times out)
 *    and, when a launch needs them, fp32 partials: split-K partials, or the
 *    k-slices of the last partial wave of a CTA-pair launch together with
 *    their counters (tagged with a per-launch number, so a counter left
 *    by any earlier launch, finished or stopped, reads as zero).
 *    tp_workspace_size() is the size of the fastest plan; a smaller
 *    workspace that still holds the plan without last-wave slices is
 *    accepted, and the call then runs without them.
 *    Calls that share a workspace must be ordered on the same stream.
 *    The GEMM kernels use programmatic dependent launch: a kernel's set-up
 *    (barriers, tensor memory) may overlap the end of the previous kernel in
 *    the stream, but it reads and writes global memory only after that
 *    kernel has completed, so stream order is kept as for plain launches.
 *  - Any host thread may call; a call runs on that thread's current CUDA
 *    device (the library makes the device's primary context current).
 *  - Calls may be captured into a CUDA graph once the same call has run
 *    eagerly on the device (that first call sets each kernel's attributes).
 *    A replay re-enqueues the captured launches with the captured pointers
 *    and shapes and reads the buffers' current contents; the workspace must
 *    not be shared with work that runs concurrently with the replay.
 *  - Biases (forward) and bias gradients (backward) are optional bf16 /
 *    out_dtype vectors over the output columns; NULL leaves them out.
 *  - Errors: argument checks run on the host before anything is enqueued
 *    and return a tp_status; on error nothing is launched.  A device-side
 *    wait that runs out of time latches TP_ERR_DEVICE_TIMEOUT into the
 *    workspace status word; tp_get_device_status() reads (and clears) it.
 *  - Determinism: identical inputs give bitwise-identical outputs.
 *  - Degenerate sizes: M == 0 or N == 0 is a no-op; K == 0 writes the
 *    epilogue of a zero product (zeros, or the bias and its activation).
 */
#ifndef TP_FUSED_H_
#define TP_FUSED_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TP_OK = 0,
  TP_ERR_INVALID_ARG = 1,        /* bad p, size, null pointer, aliasing, enum */
  TP_ERR_ALIGNMENT = 2,          /* base pointer or row pitch not 16-byte aligned */
  TP_ERR_UNSUPPORTED_SHAPE = 3,  /* e.g. M % p != 0 for ReduceScatter / AllGather */
  TP_ERR_WORKSPACE_TOO_SMALL = 4,
  TP_ERR_ARCH = 5,               /* device is not sm_103 / sm_100 family */
  TP_ERR_CUDA = 6,               /* a CUDA runtime or driver call failed */
  TP_ERR_DEVICE_TIMEOUT = 7      /* a device wait ran out of time (latched) */
} tp_status;

typedef enum { TP_BF16 = 0, TP_FP32 = 1 } tp_dtype;

typedef enum {
  TP_EPI_NONE = 0,   /* write the GEMM result */
  TP_EPI_GELU = 1,   /* write GeLU(H) (exact erf form) and optionally H */
  TP_EPI_DGELU = 2   /* write G * GeLU'(H), H read from `preact` */
} tp_epilogue;

typedef enum {
  TP_OP_ROW_AR = 0,  /* tp_row_linear_fwd_allreduce */
  TP_OP_ROW_RS = 1,  /* tp_row_linear_fwd_reducescatter */
  TP_OP_COL_FWD = 2, /* tp_col_linear_fwd */
  TP_OP_COL_BWD = 3, /* tp_col_linear_bwd */
  TP_OP_ROW_BWD = 4, /* tp_row_linear_bwd */
  TP_OP_AG_MM = 5,   /* tp_ag_matmul */
  TP_OP_ROW_AR_UNFUSED = 6, /* tp_row_linear_fwd_unfused */
  TP_OP_AG_MM_BWD = 7,      /* tp_ag_matmul_bwd */
  TP_OP_ROW_RS_BWD = 8      /* tp_row_linear_bwd_reducescatter */
} tp_op;

/* Bytes of device workspace the call (op, p, M, N, K, chunk_m, out_dtype)
 * needs, with M, N, K meant as in that call.  Always >= 256 (the status
 * word).  out_dtype matters: with TP_FP32 outputs no tensor-core
 * accumulator takes more than 2048 of the contraction (all ranks' K laid
 * end to end), so a longer contraction is split and its fp32 partials,
 * ceil(sum K / 2048) copies of the outputs, live in the workspace.  This
 * keeps fp32 outputs within 1e-5 of max|Y| of the exact sum at any K. */
size_t tp_workspace_size(tp_op op, int p, int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                         tp_dtype out_dtype);

/* Row-parallel forward, MatMul+AllReduce layout.  [M027 §01; TP §2.4, §四]
 *   Y = sum_{r=0}^{p-1} X_r . W_r (+ b), accumulated in one accumulator, written once.
 *   x[r]: X_r [M, K] (rank r's column block of the layer input)
 *   w[r]: W_r [K, N] (rank r's row block of the weight)
 *   bias: b [N] bf16 or NULL, added once after the reduction (in fp32,
 *         before the output rounding).  [TP §四: Y = AllReduce(X_k A_k) + b]
 *   y[i]: Y [M, N] for i < n_out.  n_out == 1 writes the full Y once;
 *         n_out == p writes p bit-identical replicas (one per rank).    */
tp_status tp_row_linear_fwd_allreduce(const void* const* x, const void* const* w, const void* bias,
                                      void* const* y, int n_out, int p,
                                      int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                                      tp_dtype out_dtype, void* ws, size_t ws_bytes,
                                      cudaStream_t stream);

/* Row-parallel forward, MatMul+ReduceScatter layout.  [M027 §01; TP §2.7]
 *   Same reduction (and bias); rank j receives rows [j*M/p, (j+1)*M/p) of Y.
 *   y[j]: [M/p, N].  Requires M % p == 0.                                */
tp_status tp_row_linear_fwd_reducescatter(const void* const* x, const void* const* w,
                                          const void* bias, void* const* y, int p,
                                          int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                                          tp_dtype out_dtype, void* ws, size_t ws_bytes,
                                          cudaStream_t stream);

/* Column-parallel forward.  [TP §2.3, §三, §7.1]
 *   H_k = X . A_k (+ b_k) for k = 0..p-1 (one grouped launch, no reduction).
 *   x: X [M, K] (replicated input); w[k]: A_k [K, N]; y[k]: [M, N].
 *   bias: NULL, or bias[k] = b_k [N] bf16, rank k's block of the bias,
 *         added before the activation.  [TP §三: Y_k = X A_k + b_k]
 *   epi == TP_EPI_NONE: y[k] = H_k.
 *   epi == TP_EPI_GELU: y[k] = GeLU(H_k); if preact != NULL, preact[k]
 *   ([M, N], same dtype as y) receives H_k for the backward pass.         */
tp_status tp_col_linear_fwd(const void* x, const void* const* w, const void* const* bias,
                            void* const* y, void* const* preact, tp_epilogue epi, int p,
                            int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                            tp_dtype out_dtype, void* ws, size_t ws_bytes,
                            cudaStream_t stream);

/* Column-parallel backward.  [TP §三, §六]
 *   dX = sum_{k=0}^{p-1} dY_k . A_k^T  (the backward AllReduce, fused,
 *        accumulated in one accumulator, written once) -> dx [M, K] if dx != NULL
 *   dA_k = X^T . dY_k (local)                     -> dw[k] [K, N] if dw != NULL
 *   db_k = sum over the M rows of dY_k (the gradient of b_k; summed in a
 *          fixed order, so deterministic)         -> db[k] [N] if db != NULL
 *   x: X [M, K] (only read when dw != NULL); w[k]: A_k [K, N] (only read
 *   when dx != NULL); dy[k]: dY_k [M, N].  At least one of dx, dw, db is
 *   given; all outputs have dtype out_dtype.                             */
tp_status tp_col_linear_bwd(const void* x, const void* const* w, const void* const* dy,
                            void* dx, void* const* dw, void* const* db, int p,
                            int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                            tp_dtype out_dtype, void* ws, size_t ws_bytes,
                            cudaStream_t stream);

/* Row-parallel backward (no reduction).  [TP §四, §六, §7.1]
 *   dX_k = dY . A_k^T, times GeLU'(H_k) when preact != NULL -> dx[k] [M, K]
 *   dA_k = X_k^T . dY                                        -> dw[k] [K, N]
 *   db   = sum over the M rows of dY (the bias' gradient)    -> db [N]
 *   x[k]: X_k [M, K] (only read when dw != NULL); w[k]: A_k [K, N];
 *   dy: dY [M, N]; preact[k]: H_k [M, K] bf16 or NULL.  Each of dx, dw,
 *   db may be NULL, not all three.                                       */
tp_status tp_row_linear_bwd(const void* const* x, const void* const* w, const void* dy,
                            void* const* dx, void* const* dw, void* db, const void* const* preact,
                            int p, int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                            tp_dtype out_dtype, void* ws, size_t ws_bytes,
                            cudaStream_t stream);

/* AllGather+MatMul.  [M027 §01-§02; TP §2.6, §11.3]
 *   Y_k = [X_0; X_1; ...; X_{p-1}] . A_k (+ b_k).  The M-tiles of rank s's
 *   rows read X_s directly, in shard order; the gathered X is written to
 *   x_gathered ([M, K]) only when that pointer is non-NULL.
 *   x[s]: X_s [M/p, K]; w[k]: A_k [K, N]; y[k]: [M, N];
 *   bias / epi / preact as in tp_col_linear_fwd.  Requires M % p == 0.    */
tp_status tp_ag_matmul(const void* const* x, const void* const* w, const void* const* bias,
                       void* const* y, void* x_gathered, tp_epilogue epi, void* const* preact, int p,
                       int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                       tp_dtype out_dtype, void* ws, size_t ws_bytes,
                       cudaStream_t stream);

/* Sequence-parallel backward of AllGather+MatMul (the dual collectives of
 * tp_ag_matmul).  [TP §2.6-2.7, §11.3]
 *   dX_s = rows [s*M/p, (s+1)*M/p) of sum_k dY_k . A_k^T   (ReduceScatter of
 *          the input gradient; the sum runs k = 0..p-1 in one accumulator)
 *          -> dx[s] [M/p, K] if dx != NULL
 *   dA_k = [X_0; ...; X_{p-1}]^T . dY_k  (contraction over all M tokens; the
 *          row shards X_s are read in place, in shard order)
 *          -> dw[k] [K, N] if dw != NULL
 *   db_k = sum over the M rows of dY_k -> db[k] [N] if db != NULL
 *   x[s]: X_s [M/p, K] (read when dw != NULL); w[k]: A_k [K, N];
 *   dy[k]: dY_k [M, N].  Requires M % p == 0.                              */
tp_status tp_ag_matmul_bwd(const void* const* x, const void* const* w, const void* const* dy,
                           void* const* dx, void* const* dw, void* const* db, int p, int64_t M,
                           int64_t N, int64_t K,
                           int64_t chunk_m, tp_dtype out_dtype, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/* Sequence-parallel backward of MatMul+ReduceScatter (the dual collectives
 * of tp_row_linear_fwd_reducescatter).  [TP §2.6-2.7, §11.3]
 *   dX_r = [dY_0; ...; dY_{p-1}] . A_r^T, times GeLU'(H_r) when preact is
 *          given (AllGather of the output gradient; the M-tiles of shard s
 *          read dY_s in place) -> dx[r] [M, K] if dx != NULL
 *   dA_r = X_r^T . [dY_0; ...; dY_{p-1}] -> dw[r] [K, N] if dw != NULL
 *   db   = sum over all rows of dY_0, ..., dY_{p-1}, shard by shard
 *          -> db [N] if db != NULL
 *   x[r]: X_r [M, K] (read when dw != NULL); w[r]: A_r [K, N];
 *   dy[s]: dY_s [M/p, N]; preact[r]: H_r [M, K] bf16 or NULL.
 *   Requires M % p == 0.                                                    */
tp_status tp_row_linear_bwd_reducescatter(const void* const* x, const void* const* w,
                                          const void* const* dy, void* const* dx, void* const* dw,
                                          void* db, const void* const* preact, int p, int64_t M,
                                          int64_t N,
                                          int64_t K, int64_t chunk_m, tp_dtype out_dtype, void* ws,
                                          size_t ws_bytes, cudaStream_t stream);

/* Unfused baseline of the row-parallel MatMul+AllReduce, for measurement
 * and for the output-error comparison against it.
 * [M027 §04: time the MatMul and the collective separately, compare the
 *  whole layer's output error; §06: record the separate baseline and the
 *  output error]
 *   phase bit 0: every rank's partial P_r = X_r . W_r into its own fp32
 *                buffer in the workspace (one launch over all ranks);
 *   phase bit 1: Y = P_0 + P_1 + ... + P_{p-1} in rank order, cast, -> y.
 *   phases = 3 runs both.  Arguments as in tp_row_linear_fwd_allreduce with
 *   n_out = 1; the workspace holds p fp32 copies of Y
 *   (tp_workspace_size(TP_OP_ROW_AR_UNFUSED, ...)).  Phase 1 without a
 *   later phase 2 leaves y untouched.
 *   flags: 0, or TP_UNFUSED_BF16_COLLECTIVE to make phase 2 sum the way an
 *   unfused AllReduce of bf16 tensors does: each rank's partial is first
 *   rounded to bf16 (the tensor it would hand to the collective), and the
 *   running sum is rounded to bf16 after every addition, in rank order:
 *   acc = bf16(P_0); acc = bf16(acc + bf16(P_r)) for r = 1..p-1.  Any
 *   other bit is TP_ERR_INVALID_ARG.                                     */
#define TP_UNFUSED_BF16_COLLECTIVE 1
tp_status tp_row_linear_fwd_unfused(const void* const* x, const void* const* w, void* y, int p,
                                    int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                                    tp_dtype out_dtype, int phases, int flags, void* ws,
                                    size_t ws_bytes, cudaStream_t stream);

/* Two-engine chunk timeline: c + (n-1) * max(c, m) + m for n >= 1, 0 for
 * n <= 0; c = per-chunk compute time, m = per-chunk reduce time.  [M027 §03] */
double tp_pipeline_time(double c, double m, int64_t n_chunks);

/* Number of chunks ceil(M / min(chunk_m, M)) (0 when M <= 0).  [M027 §03] */
int64_t tp_num_chunks(int64_t M, int64_t chunk_m);

/* The scheduler's chunk size for a call: the candidate with the smallest
 * modelled tp_pipeline_time, where a chunk's compute time is the larger of
 * its tensor-core time (with the MMA-width efficiency of its tile) and its
 * operand-streaming time, and its reduce time is the write-out of its
 * reduced rows.  Host only; never fails (returns >= 1, or 0 when M <= 0). */
int64_t tp_choose_chunk_m(tp_op op, int p, int64_t M, int64_t N, int64_t K);

/* The chunk size to use given MEASURED per-chunk times.  [M027 §03-§04:
 * try candidate chunkings, measure the small-chunk compute and
 * communication, pick the shortest timeline]
 *   chunk[i], c[i], m[i] for i < n: a candidate chunk_m and the measured
 *   compute and communication time of one of its chunks (any time unit).
 *   Returns the candidate whose tp_pipeline_time(c, m, ceil(M / chunk))
 *   is smallest (the first one on ties), or 0 when n <= 0, M <= 0, or a
 *   pointer is NULL.  Host only.                                         */
int64_t tp_choose_chunk_m_measured(int64_t M, const int64_t* chunk, const double* c, const double* m,
                                   int n);

/* Synchronises `stream`, returns the latched device status of `ws`
 * (TP_OK or TP_ERR_DEVICE_TIMEOUT) and clears it.                         */
tp_status tp_get_device_status(void* ws, cudaStream_t stream);

/* Row-parallel MatMul+AllReduce for callers that cannot allocate device
 * memory.  The paper has no counterpart: this is a library convenience.
 *
 * Some callers have no way to hand the library a workspace: a host plugin
 * interface that passes only input and output buffers, or an engine that
 * has reserved all of device memory up front for its own pool, so a
 * cudaMalloc from inside a call would fail or stall every stream (it
 * synchronises the device).  This entry point computes exactly what
 * tp_row_linear_fwd_allreduce computes, with the same arguments minus the
 * workspace, and allocates nothing.  Its scratch (the status word and the
 * split-K fp32 partials) lives in one static device array of
 * TP_NOALLOC_SCRATCH_BYTES bytes that every GPU loading this library holds
 * until the process exits.
 *
 *  - A call that needs more scratch than TP_NOALLOC_SCRATCH_BYTES, even
 *    without last-wave slices (see `ws` above), is rejected with
 *    TP_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls on a device share the one array.  Calls that may overlap on
 *    the GPU (different streams without ordering between them) race on it;
 *    order them on one stream.  Nothing in the array has to start at zero:
 *    every partial a call reads was written earlier by that same call, and
 *    slice counters carry the number of the launch that wrote them, so
 *    stale ones read as zero.
 *  - A device-side wait that runs out of time latches
 *    TP_ERR_DEVICE_TIMEOUT into the array's status word, as it would into a
 *    workspace; tp_noalloc_device_status() reads and clears it.
 *  - The array's address is looked up again when the device's context has
 *    changed (for instance after cudaDeviceReset), so a reset does not
 *    leave a stale address behind; the first call after it then repeats
 *    the look-up and must also come before any stream capture.           */
#define TP_NOALLOC_SCRATCH_BYTES (16u << 20)
tp_status tp_row_linear_fwd_allreduce_noalloc(const void* const* x, const void* const* w,
                                              void* const* y, int n_out, int p,
                                              int64_t M, int64_t N, int64_t K, int64_t chunk_m,
                                              tp_dtype out_dtype, cudaStream_t stream);

/* Status word of the allocation-free entry point's static scratch on the
 * calling thread's current device (no counterpart in the paper either).
 * Synchronises `stream`, then returns TP_ERR_DEVICE_TIMEOUT (and clears the
 * word) if a device wait of an earlier tp_row_linear_fwd_allreduce_noalloc
 * call ran out of time, TP_OK if none did, TP_ERR_CUDA if the CUDA calls
 * fail.  Like the entry point itself it allocates nothing.                */
tp_status tp_noalloc_device_status(cudaStream_t stream);

/* Test hooks of the failure-detection path (process-wide, read when a call
 * is planned).  Not for production use.
 *   TP_DEBUG_TIMEOUT_MS: limit of every device-side wait, in ms; 0 restores
 *     the default (TP_DEVICE_TIMEOUT_MS from the environment, else 2000).
 *   TP_DEBUG_DROP_LOAD: n >= 0 makes CTA 0 of every following launch skip
 *     arming its n-th k-block load, so the MMA issuer's wait on it runs out:
 *     the kernel latches TP_ERR_DEVICE_TIMEOUT, stops its other roles, waits
 *     (bounded) for its own copies and MMAs in flight, frees its tensor
 *     memory and returns; -1 turns the hook off.  No fault or trap is used.
 *   TP_DEBUG_TILE_MODE: 0 (default) lets the planner choose 128x256 tiles on
 *     one CTA or 256x256 tiles on a CTA pair; 1 forces single-CTA tiles; 2
 *     uses CTA pairs for every non-swapped launch (parity testing of both
 *     tile paths at small, ragged sizes).
 *   TP_DEBUG_NO_TAIL_SLICES: 1 runs the last partial wave of a CTA-pair
 *     launch as whole tiles instead of k-slices; 0 (default) lets the
 *     planner slice it.
 *   TP_DEBUG_SPLIT_K: 0 (default) lets the planner choose the split-K
 *     factor of single-CTA launches with fewer tiles than SMs; n in 1..16
 *     splits their contraction n ways instead (clamped to one k-block per
 *     split; fp32 outputs still split further where they need it).  Changes
 *     the workspace size of those calls; for parity testing of the split-K
 *     path on shapes the planner would not split.
 *   TP_DEBUG_L2_HINTS: 1 (default) loads an operand that every output group
 *     of a launch re-reads (and that fits in half the L2) with an
 *     evict_last policy and writes final outputs evict_first; 0 leaves
 *     every access at the normal policy.  Results are identical either way.
 *   TP_DEBUG_TMA_STORE: 1 (default) lets the staged epilogue leave shared
 *     memory by TMA tensor stores wherever the outputs allow it; 0 forces
 *     plain 16-byte stores (bit-identical results; for testing both paths).
 *   TP_DEBUG_NO_BWD_FUSION: 0 (default) lets a backward call run its dX and
 *     dW products as one CTA-pair launch where that is planned to finish
 *     sooner; 1 always runs them as two launches (bit-identical results).
 *   TP_DEBUG_K_ALTERNATE: 1 (default) lets CTA-pair launches whose
 *     contraction is 8192 or deeper run the whole tiles of every other wave
 *     last k-block first (rank p-1's segment first), which re-reads from L2
 *     what the previous wave read last; 0 runs every tile first to last.
 *     The order changes the fp32 rounding of non-integer sums (both orders
 *     are deterministic), not exact ones.
 * Returns TP_ERR_INVALID_ARG for an unknown key or a bad value.            */
typedef enum {
  TP_DEBUG_TIMEOUT_MS = 0,
  TP_DEBUG_DROP_LOAD = 1,
  TP_DEBUG_TILE_MODE = 2,
  TP_DEBUG_NO_TAIL_SLICES = 3,
  TP_DEBUG_SPLIT_K = 4,
  TP_DEBUG_L2_HINTS = 5,
  TP_DEBUG_TMA_STORE = 6,
  TP_DEBUG_NO_BWD_FUSION = 7,
  TP_DEBUG_K_ALTERNATE = 8
} tp_debug_key;
tp_status tp_debug_set(tp_debug_key key, int64_t value);

/* Timeline trace of the GEMM launches that follow (process-wide, for
 * measuring the chunk pipeline: [M027 §03, the two-engine timeline]).
 *   buf: device buffer of cap_units x 4 uint64, zero-filled by the caller
 *        before each traced launch; NULL (with cap_units 0) stops tracing.
 *   Unit t of a launch (t < cap_units; units are the launch's tiles, or
 *   split-K / last-wave slices, in the launch's chunk-major order) records
 *     [0] %globaltimer (ns) when its first MMA was issued,
 *     [1] when the epilogue saw its accumulator complete,
 *     [2] when the last epilogue warp finished writing it out,
 *     [3] (chunk index << 32) | CTA (single-CTA tiles) or cluster index.
 *   Every traced launch writes from unit 0, so trace one launch at a time.
 * Returns TP_ERR_INVALID_ARG for a negative size or a NULL/size mismatch,
 * TP_ERR_ALIGNMENT for a buffer not 16-byte aligned.                      */
tp_status tp_trace_set(void* buf, int64_t cap_units);

/* Static description of a status code. */
const char* tp_status_string(tp_status s);

#ifdef __cplusplus
}
#endif

#endif /* TP_FUSED_H_ */
