/*
 * hytopk.h -- exact per-query top-k selection over DeepSeek-style indexer
 * scores without a score table (HyTopK, also called FlashTopK), selection
 * replay, and the conventional two-pass materialise-then-top-k path, for one
 * NVIDIA GB300 (sm_103a).
 *
 * Sources, cited by page title and paragraph:
 *   [Summary]   "HyScale: Scaling Long-Context Training for Learned Sparse
 *               Attention" (neuraltrendhub), "What the paper found" and
 *               "Original abstract".
 *   [Explainer] "HyScale sparse-attention training -- Selection without a
 *               score table -- What does it mean?" (learnaivisually): the
 *               score-table, HyTopK, selection-replay and worked-example
 *               paragraphs.
 *
 * The operation. For query t at position pos[t] (it sees keys s <= pos[t]:
 * each query scores all tokens before it, Summary) the indexer score is
 *
 *     I[t,s] = sum_h w[t,h] * ReLU( q[t,h,:] . k[s,:] )
 *
 * with one shared key head. hytopk_select returns, per query, the exact top-k
 * key positions of I[t, 0..pos[t]] ordered by score descending, ties by lower
 * position first (Explainer, HyTopK paragraph: ties at the k-th score are
 * resolved by position and the k kept entries are radix sorted, so the output
 * is bitwise reproducible), without writing the n x L score table to memory.
 * hytopk_replay rescores only stored (query, index) pairs (Explainer,
 * selection-replay paragraph). hytopk_select_twopass is the conventional
 * method (Explainer, score-table paragraph): a kernel writes every score, a
 * second kernel reads them back and selects.
 *
 * Conventions shared by every call:
 *   - Every array pointer is DEVICE memory owned by the caller. The library
 *     allocates nothing and keeps no state between calls; scratch memory is
 *     the caller's `workspace` (hytopk_select_noalloc, for callers that
 *     cannot provide one, uses a fixed array the library holds instead).
 *   - Calls are asynchronous on `stream` (0 = legacy default stream). The
 *     return code covers host-side argument checks and launch errors only;
 *     conditions found on the device are reported through the device status
 *     word (HYTOPK_DEV_* bits) of hytopk_stats or of the replay call.
 *   - Layouts are row-major and contiguous:
 *       q        [n, H, d] elements of `dt`
 *       q_scale  [n, H]    fp32, one scale per (query, head) row of d elements;
 *                          required when q is e4m3 (HYTOPK_E4M3 and
 *                          HYTOPK_E4M3_BF16), must be NULL for bf16 q
 *       k        [L, d]    elements of `dt`
 *       k_scale  [L]       fp32 per key row; required for e4m3 k (HYTOPK_E4M3),
 *                          NULL for bf16 k (HYTOPK_BF16 and HYTOPK_E4M3_BF16)
 *       w        [n, H]    fp32 head weights (any sign)
 *       positions[n]       int32, 0 <= pos < L, any order
 *     e4m3 is OCP FP8 E4M3 ("fn"); an element's value is code * scale. Scales
 *     must be finite and > 0 (then ReLU(a*x) = a*ReLU(x) and scales may be
 *     applied after the dot); a non-positive scale sets HYTOPK_DEV_BAD_SCALE.
 *     Inputs must be finite.
 *     HYTOPK_E4M3_BF16 converts q to bf16 exactly (every e4m3 value is a bf16
 *     value) and runs the bf16 path; q_scale is folded into w as for e4m3.
 *   - Supported shapes: H in {1,2,4,8,16,32,64,128}; key rows of 64, 128 or
 *     256 bytes, i.e. d in {32, 64, 128} for bf16 and d in {64, 128, 256} for
 *     e4m3; 1 <= k_top <= 16384; n >= 0; L >= 1 (hytopk_replay_backward:
 *     H in {1, 2, ..., 64}, d in {64, 128}). Other shapes return
 *     HYTOPK_UNSUPPORTED.
 *   - q and k (and dq, dk of hytopk_replay_backward) must be 16-byte
 *     aligned, every other array 4-byte aligned, so that an array offset by
 *     whole rows stays a valid argument.
 *   - Scores are fp32. A selected score agrees with the definition above to
 *     within 1e-3 relative (exact for integer-valued data that fits fp32).
 */
#ifndef HYTOPK_H
#define HYTOPK_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

/* Only the functions below are exported from the shared library; every
 * other symbol is hidden (the library is built with hidden visibility). */
#if defined(__GNUC__)
#define HYTOPK_API __attribute__((visibility("default")))
#else
#define HYTOPK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HYTOPK_OK = 0,
  HYTOPK_INVALID_ARG = 1,          /* null pointer, negative size, bad enum, k_top > capacity */
  HYTOPK_UNSUPPORTED = 2,          /* H, d or k_top outside the supported set */
  HYTOPK_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below the *_workspace_size value */
  HYTOPK_CUDA_ERROR = 4,           /* a CUDA runtime call or launch failed */
  HYTOPK_MISALIGNED = 5            /* a device pointer breaks the alignment rules above */
} hytopk_status;

/* Element types of q and k: both bf16, both e4m3 (with q_scale and k_scale),
 * or e4m3 q (with q_scale) and bf16 k (no k_scale). */
typedef enum { HYTOPK_BF16 = 0, HYTOPK_E4M3 = 1, HYTOPK_E4M3_BF16 = 2 } hytopk_dtype;

/* Device status bits (written with atomicOr on the device). */
#define HYTOPK_DEV_REPLAY_BAD_INDEX 0x1u /* replay index not -1 and outside [0, L): entry is NaN */
#define HYTOPK_DEV_BAD_SCALE 0x2u        /* a q_scale or k_scale <= 0 (results undefined) */
#define HYTOPK_DEV_BAD_POSITION 0x4u     /* a position outside [0, L): that query is all -1 */
/* A bounded wait inside a tensor-core kernel gave up (after 2 s): the kernel
 * stopped its loops, freed its tensor memory and returned, so every output of
 * that call is undefined. It signals a stalled GPU or a library bug. */
#define HYTOPK_DEV_WAIT_TIMEOUT 0x80000000u

/* Per-call statistics of hytopk_select (device memory, written at the end of
 * the call's stream work). The check kernel flags a query with ctx > k whose
 * candidate count is below k (under-k) or above the capacity (overflow)
 * (Explainer, HyTopK paragraph); when more than 64 queries fail, every query
 * is rescored over its whole context (fallback_used = 1). */
typedef struct {
  int32_t n_failed;
  int32_t n_overflow;
  int32_t n_under_k;
  int32_t fallback_used;
  int64_t total_candidates; /* sum over queries of the filter's candidate count */
  uint32_t device_status;   /* HYTOPK_DEV_* bits */
  int32_t n_queries;
} hytopk_stats;

/* Largest number of failed queries repaired one by one; above it the whole
 * selection is rescored (Explainer, HyTopK paragraph: the fallback starts
 * past 64 failed queries). */
#define HYTOPK_MAX_RECOVERY_ROWS 64

/* Phase boundaries of hytopk_select that hytopk_select_ex can time. */
enum {
  HYTOPK_PHASE_PREP = 0,      /* order queries by position, pack q, fold scales */
  HYTOPK_PHASE_THRESHOLD = 1, /* score the evenly spaced samples, take the r-th best */
  HYTOPK_PHASE_FILTER = 2,    /* score every causal key, keep those >= threshold */
  HYTOPK_PHASE_CHECK = 3,     /* flag under-k and overflowed queries */
  HYTOPK_PHASE_SELECT = 4,    /* exact radix select + sort of the candidates */
  HYTOPK_PHASE_RECOVER = 5,   /* rescore failed queries over their whole context */
  HYTOPK_NUM_PHASES = 6
};

/* Options of hytopk_select_ex. Zero-initialise for the defaults. */
typedef struct {
  /* Device fp32 [n] or NULL. Replaces the sampled threshold of each query
   * (a testing hook: -inf forces overflow, +inf forces under-k). The result
   * is the exact top-k whatever the thresholds are. */
  const float* threshold_override;
  /* NULL or HYTOPK_NUM_PHASES + 1 events recorded on `stream` before the
   * first phase and after each phase (CUDA events, caller-created). */
  cudaEvent_t* phase_events;
  /* Nonzero: the filter walks its work list in reverse (determinism tests). */
  int reverse_schedule;
  int reserved;
} hytopk_select_options;

/* The evenly spaced samples of a query with ctx = pos + 1 visible keys
 * (Explainer, HyTopK paragraph and worked example): returns the sample count
 *     M = min(ctx, max(4096, floor(ctx / 128)), 8192)
 * and, when the pointers are not NULL, writes the sample positions
 * p_j = floor(j * ctx / M), j = 0 .. M-1, to positions_out (HOST memory, room
 * for M <= 8192 entries) and the threshold rank r = min(M, ceil(3 k M / ctx))
 * to *rank_out (host). The threshold of the query is the r-th best score
 * among its samples. A query with ctx <= k_top keeps all its keys and uses no
 * samples. Host-only: no CUDA call. Returns 0 (writing nothing) when ctx < 1
 * or k_top < 1. These are the same integer formulas the kernels use. */
HYTOPK_API int32_t hytopk_sample_plan(int64_t ctx, int32_t k_top, int32_t* positions_out,
                                      int32_t* rank_out);

/* Bytes of workspace hytopk_select needs. capacity = candidate buffer slots
 * per query (0 selects the default 8 * k_top). Returns 0 for invalid or
 * unsupported arguments. */
HYTOPK_API size_t hytopk_select_workspace_size(int n, int L, int H, int d, int k_top, int capacity,
                                    hytopk_dtype dt);

/* Score-table chunks of hytopk_select's fallback (HyScale explainer, HyTopK
 * paragraph: past 64 failed queries every query is rescored). The fallback
 * writes whole rows of L scores into the candidate and recovery-row buffers
 * of the workspace and reads them back chunk by chunk; since only the device
 * knows whether it is needed, every call launches one table writer and one
 * read-back per chunk, which return at once when no fallback is needed.
 * Arguments as for hytopk_select_workspace_size. Returns the chunk count (0
 * for n = 0), or -1 for invalid or unsupported arguments. Host-only: no CUDA
 * call. */
HYTOPK_API int32_t hytopk_select_fallback_chunks(int n, int L, int H, int d, int k_top,
                                                 int capacity, hytopk_dtype dt);

/* Exact top-k selection without a score table (HyTopK).
 *   idx_out    [n, k_top] int32: key positions, score descending then position
 *              ascending; a query with ctx = pos+1 < k_top has its ctx keys
 *              followed by -1.
 *   scores_out [n, k_top] fp32 or NULL: the scores of idx_out, -inf padding.
 *   capacity   candidate slots per query, >= k_top (0: 8 * k_top).
 *   workspace  device memory of at least hytopk_select_workspace_size(...)
 *              bytes, 256-byte aligned; contents need not be initialised.
 *   stats_out  device hytopk_stats or NULL.
 * The steps: per query, M = min(ctx, max(4096, floor(ctx/128)), 8192) evenly
 * spaced keys p_j = floor(j*ctx/M) are scored and the threshold T is the r-th
 * best of them, r = min(M, ceil(3*k*M/ctx)) (Explainer, HyTopK paragraph and
 * worked example); every causal key is scored on chip and keys with score >= T
 * are appended to the query's candidate buffer; queries with ctx > k and fewer
 * than k or more than `capacity` candidates are rescored over their whole
 * context (up to 64 of them one by one; past 64, every query, through
 * score-table rows written into the workspace chunk by chunk); the candidates
 * are radix-selected (score, then position) and radix-sorted. */
HYTOPK_API hytopk_status hytopk_select(const void* q, const float* q_scale, const void* k,
                            const float* k_scale, const float* w, const int32_t* positions, int n,
                            int L, int H, int d, int k_top, hytopk_dtype dt, int32_t* idx_out,
                            float* scores_out, int capacity, void* workspace,
                            size_t workspace_bytes, hytopk_stats* stats_out, cudaStream_t stream);

/* hytopk_select with options (opts may be NULL). */
HYTOPK_API hytopk_status hytopk_select_ex(const void* q, const float* q_scale, const void* k,
                               const float* k_scale, const float* w, const int32_t* positions,
                               int n, int L, int H, int d, int k_top, hytopk_dtype dt,
                               int32_t* idx_out, float* scores_out, int capacity,
                               void* workspace, size_t workspace_bytes, hytopk_stats* stats_out,
                               const hytopk_select_options* opts, cudaStream_t stream);

/* Selection replay (Explainer, selection-replay paragraph): scores_out[t,j] =
 * I[t, idx[t,j]] for idx [n, k_top] int32, with the same arithmetic as
 * hytopk_select (so replayed scores equal the selected scores bit for bit).
 * idx = -1 gives -inf. Any other index outside [0, L) gives NaN and sets
 * HYTOPK_DEV_REPLAY_BAD_INDEX in *dev_status (device uint32, may be NULL).
 * Replay does not check causality. Needs no workspace. */
HYTOPK_API hytopk_status hytopk_replay(const void* q, const float* q_scale, const void* k,
                            const float* k_scale, const float* w, const int32_t* idx, int n,
                            int L, int H, int d, int k_top, hytopk_dtype dt, float* scores_out,
                            uint32_t* dev_status, cudaStream_t stream);

/* Replay with adjacent queries grouped (HyScale summary, "What the paper
 * found", and Explainer, limits paragraph: neighbouring tokens select mostly
 * the same keys). group = 1 is hytopk_replay. group = 2 replays queries 2i
 * and 2i+1 together: the union of their two index lists is gathered once and
 * scored for both, so a key both select is read once. Results, -inf / NaN
 * entries and status bits are those of hytopk_replay, bit for bit. Grouping
 * applies when H <= 64 and k_top <= 2048; other shapes run hytopk_replay.
 * Any other group returns HYTOPK_INVALID_ARG.
 * Use group = 1. Measured on one GB300 at L = 2^20, n = 8192, k = 2048, e4m3:
 * group = 2 is SLOWER than hytopk_replay (about 0.55 against 0.40 ms) even
 * when neighbouring queries share 71% of their keys, because hytopk_replay
 * already serves a shared key's second read from L2 (queries 2i and 2i+1 run
 * at the same time) and building the union costs more than the L2 traffic it
 * saves. It is kept as the measured counterexample. */
HYTOPK_API hytopk_status hytopk_replay_grouped(const void* q, const float* q_scale, const void* k,
                                               const float* k_scale, const float* w,
                                               const int32_t* idx, int n, int L, int H, int d,
                                               int k_top, hytopk_dtype dt, int group,
                                               float* scores_out, uint32_t* dev_status,
                                               cudaStream_t stream);

/* Gradients of the indexer score at the selected entries, with the replay
 * rescoring fused in (Explainer, key-observation paragraph: the indexer's own
 * loss reads only the scores at those entries; selection-replay paragraph:
 * only those entries are rescored during recomputation). The loss is not on
 * the pages; its gradient at the entries is the input:
 *   grad  [n, k_top] fp32: dLoss/dI[t, idx[t,j]] (ignored where idx is -1)
 * With qd = q * q_scale (per row of d), kd = k * k_scale and
 * x = qd[t,h] . kd[idx[t,j]], the outputs are
 *   dw [n, H]     fp32, written:  sum_j grad * max(0, x)
 *   dq [n, H, d]  fp32, written:  sum_j grad * w[t,h] * [x > 0] * kd[idx[t,j]]
 *   dk [L, d]     fp32, ADDED TO (the caller zeroes it, or accumulates over
 *                 calls): grad * sum_h w[t,h] * [x > 0] * qd[t,h] for every
 *                 entry, at row idx[t,j]
 * i.e. gradients with respect to the dequantised q and k. The derivative of
 * max(0, x) at x = 0 is 0. The tensor cores take bf16 operands: e4m3 codes
 * convert exactly, and every product that carries a weight, gradient or
 * scale is split into a bf16 high part and a bf16 remainder (about 16
 * significant bits); accumulation is fp32. dk takes floating-point atomic
 * additions, so its low bits depend on the order of arrival.
 *   Supported: H in {1, 2, 4, 8, 16, 32, 64}, d in {64, 128}, every dtype (others:
 *   HYTOPK_UNSUPPORTED). dq and dk must be 16-byte aligned.
 *   An index that is not -1 and outside [0, L) contributes nothing and sets
 *   HYTOPK_DEV_REPLAY_BAD_INDEX in *dev_status (device uint32, may be NULL).
 *   No workspace; asynchronous on `stream`. */
HYTOPK_API hytopk_status hytopk_replay_backward(const void* q, const float* q_scale, const void* k,
                                     const float* k_scale, const float* w, const int32_t* idx,
                                     const float* grad, int n, int L, int H, int d, int k_top,
                                     hytopk_dtype dt, float* dq, float* dk, float* dw,
                                     uint32_t* dev_status, cudaStream_t stream);

/* Bytes of workspace the two-pass path needs to hold `rows_per_chunk` rows of
 * the score table at once (rows_per_chunk <= 0: all n rows). */
HYTOPK_API size_t hytopk_twopass_workspace_size(int n, int L, int H, int d, int k_top, hytopk_dtype dt,
                                     int rows_per_chunk);

/* The conventional two-pass path (Explainer, score-table paragraph): for each
 * chunk of queries, one kernel writes the fp32 score rows [chunk, L] (-inf
 * beyond each query's position) to the workspace and a second kernel reads
 * them back and selects the exact top-k with the same tie rule and order as
 * hytopk_select. The chunk size is the largest the workspace holds. Same
 * outputs as hytopk_select, bit for bit. When the whole table is small (a few
 * hundred MiB: short contexts) this path is the faster of the two, since
 * writing and reading the table costs less than hytopk_select's sampled
 * threshold and candidate select; at long contexts hytopk_select is faster
 * and needs no table. */
HYTOPK_API hytopk_status hytopk_select_twopass(const void* q, const float* q_scale, const void* k,
                                    const float* k_scale, const float* w,
                                    const int32_t* positions, int n, int L, int H, int d,
                                    int k_top, hytopk_dtype dt, int32_t* idx_out,
                                    float* scores_out, void* workspace, size_t workspace_bytes,
                                    uint32_t* dev_status, cudaStream_t stream);

/* hytopk_select without a caller workspace, for callers that cannot allocate
 * device memory: code inside a host framework that owns the whole device
 * memory budget through its own pool and forbids other allocations, or
 * latency-critical paths where an allocation (and the device synchronisation
 * that cudaMalloc/cudaFree can imply) is not acceptable. The HyScale pages
 * have no counterpart to this entry point; it only changes where the scratch
 * memory comes from.
 *   The scratch is one fixed array of HYTOPK_NOALLOC_SCRATCH_BYTES in device
 *   memory, held by the library on every GPU that loads it until the process
 *   exits. The entry point allocates nothing (no cudaMalloc, cudaFree or
 *   allocating library call).
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.
 *   Argument errors are reported as by hytopk_select (shape, then pointers
 *   and alignment); only then does a problem whose
 *   hytopk_select_workspace_size exceeds the array return
 *   HYTOPK_WORKSPACE_TOO_SMALL, launching nothing.
 *   All calls share the one array and each call overwrites it (the call
 *   itself clears what must start at zero), so calls whose GPU work overlaps
 *   in time -- on different streams or host threads -- race; the caller must
 *   order them.
 * Arguments and outputs are those of hytopk_select. */
#define HYTOPK_NOALLOC_SCRATCH_BYTES (32u << 20)

HYTOPK_API hytopk_status hytopk_select_noalloc(const void* q, const float* q_scale, const void* k,
                                    const float* k_scale, const float* w,
                                    const int32_t* positions, int n, int L, int H, int d,
                                    int k_top, hytopk_dtype dt, int32_t* idx_out,
                                    float* scores_out, int capacity, hytopk_stats* stats_out,
                                    cudaStream_t stream);

/* Key-sharded exact selection: the single-GPU stand-in for selection under
 * context parallelism, where each GPU holds one range of the keys (Summary,
 * "What the paper found", and Explainer, limits paragraph: context-parallel
 * communication overlapped with selection; the pages do not describe how a
 * sharded selection is combined).
 *   The keys [0, L) are split into ranges of S = ceil(L / num_shards) keys
 *   rounded up to a multiple of 128; range p is [p*S, min(L, (p+1)*S)).
 *   For each range, in turn, hytopk_select runs over that range alone (its
 *   own sampled threshold, filter, check and recovery), giving each query the
 *   exact top-k of its causal keys inside the range (none if its position is
 *   below the range). Then one merge per query keeps the exact top-k of the
 *   union of those lists, with the same order and tie rule (score
 *   descending, then lower global position). The result equals hytopk_select
 *   bit for bit: under one total order the k best of a union are among the k
 *   best of each part.
 *   num_shards: 1 .. 64. Ranges that start at or after L are skipped.
 *   workspace: hytopk_select_sharded_workspace_size bytes, 256-byte aligned.
 *   stats_out: device hytopk_stats or NULL; counts are summed over the
 *   ranges (a query can fail in several), fallback_used is set if any range
 *   fell back, device_status ORs the ranges' bits, n_queries = n.
 * Other arguments, outputs and errors are those of hytopk_select. */
HYTOPK_API size_t hytopk_select_sharded_workspace_size(int n, int L, int H, int d, int k_top, int capacity,
                                            hytopk_dtype dt, int num_shards);

HYTOPK_API hytopk_status hytopk_select_sharded(const void* q, const float* q_scale, const void* k,
                                    const float* k_scale, const float* w,
                                    const int32_t* positions, int n, int L, int H, int d,
                                    int k_top, hytopk_dtype dt, int num_shards, int32_t* idx_out,
                                    float* scores_out, int capacity, void* workspace,
                                    size_t workspace_bytes, hytopk_stats* stats_out,
                                    cudaStream_t stream);

/* Packed variable-length batches: B independent sequences whose queries and
 * keys are concatenated, as in long-context training that packs several
 * documents into one step. Sequence b owns the query rows
 * [cu_q[b], cu_q[b+1]) and the key rows [cu_k[b], cu_k[b+1]); its queries'
 * positions are relative to the sequence (0 <= pos < cu_k[b+1] - cu_k[b]) and
 * select within it only, and the returned indices are relative to it too.
 *   cu_q, cu_k: HOST arrays of B + 1 int32, non-decreasing, cu_q[0] = cu_k[0]
 *   = 0, cu_q[B] = n, cu_k[B] = L. Every other argument is that of
 *   hytopk_select over the whole packed arrays (idx_out, scores_out [n,
 *   k_top]).
 *   Each sequence runs the whole selection on its own rows, one after another
 *   on `stream`, in one workspace of hytopk_select_varlen_workspace_size
 *   bytes (the largest sequence's need). stats_out sums the sequences'
 *   counts and ORs their status bits; n_queries = n.
 *   Errors: as hytopk_select, plus HYTOPK_INVALID_ARG for inconsistent
 *   cu_q / cu_k. */
HYTOPK_API size_t hytopk_select_varlen_workspace_size(const int32_t* cu_q, const int32_t* cu_k,
                                                      int B, int H, int d, int k_top,
                                                      int capacity, hytopk_dtype dt);

HYTOPK_API hytopk_status hytopk_select_varlen(const void* q, const float* q_scale, const void* k,
                                              const float* k_scale, const float* w,
                                              const int32_t* positions, const int32_t* cu_q,
                                              const int32_t* cu_k, int B, int H, int d, int k_top,
                                              hytopk_dtype dt, int32_t* idx_out,
                                              float* scores_out, int capacity, void* workspace,
                                              size_t workspace_bytes, hytopk_stats* stats_out,
                                              cudaStream_t stream);

/* Replay of a packed batch: idx [n, k_top] relative to each query's sequence
 * (as hytopk_select_varlen returns them); otherwise as hytopk_replay. */
HYTOPK_API hytopk_status hytopk_replay_varlen(const void* q, const float* q_scale, const void* k,
                                              const float* k_scale, const float* w,
                                              const int32_t* idx, const int32_t* cu_q,
                                              const int32_t* cu_k, int B, int H, int d, int k_top,
                                              hytopk_dtype dt, float* scores_out,
                                              uint32_t* dev_status, cudaStream_t stream);

/* Backward of a packed batch: as hytopk_replay_backward per sequence, with
 * idx relative to each query's sequence; dq [n, H, d] and dw [n, H] are
 * written, dk [L, d] (all sequences' keys, concatenated) is added to. */
HYTOPK_API hytopk_status hytopk_replay_backward_varlen(
    const void* q, const float* q_scale, const void* k, const float* k_scale, const float* w,
    const int32_t* idx, const float* grad, const int32_t* cu_q, const int32_t* cu_k, int B, int H,
    int d, int k_top, hytopk_dtype dt, float* dq, float* dk, float* dw, uint32_t* dev_status,
    cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
HYTOPK_API const char* hytopk_status_string(hytopk_status status);

/* Library version as 10000*major + 100*minor + patch. */
HYTOPK_API int hytopk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HYTOPK_H */
