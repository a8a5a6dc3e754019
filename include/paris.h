/*
 * paris.h -- C ABI of the ParisKV decode-time KV-cache retrieval library
 * (GB300, sm_103a).
 *
 * Method: "ParisKV: Fast and Drift-Robust KV-Cache Retrieval for Long-Context
 * LLMs" (gist.science summary of arXiv 2602.07721).  Keys and queries are
 * l2-normalised and share a random orthogonal rotation realised as an SRHT;
 * the rotated vector is split into B subspaces; each subspace direction is
 * assigned to its nearest analytic sign-pattern centroid (+-1/sqrt(m))
 * (Methodology 1).  A query's top-rho centroids per subspace give collision
 * votes that cut the Retrieval zone to a small candidate set; candidates are
 * reranked with the 4-bit RSQ-IP estimator ||q|| sum_b w_{i,b} <v_{i,b}, q~_b>
 * and the top-k attend together with the Sink, Local and Update-Buffer zones
 * (Methodology 2; system level: UVA offload and the sliding-window update).
 *
 * Conventions for every call:
 *  - Device pointers are plain CUDA device addresses (or addresses the device
 *    can dereference, e.g. mapped host memory); host pointers are ordinary
 *    process memory.  Each argument says which it is.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Device work is enqueued on it and the call returns without
 *    waiting, unless the call says it synchronises.
 *  - Arguments are checked before any work is enqueued; a rejected call
 *    changes no state and returns PARIS_EINVAL / PARIS_ESTATE /
 *    PARIS_ECAPACITY.  A failing CUDA call returns PARIS_ECUDA.  The text of
 *    the last error is available from paris_last_error().
 *  - Faults detected on the device (an out-of-range token index handed to
 *    paris_sparse_attend) never trap: the offending read is skipped and a
 *    status word in the context is set; paris_check_device() reports it.
 *  - A context is not thread-safe; use one per layer and per thread.
 *  - No call allocates device memory after paris_create.
 */
#ifndef PARIS_H_
#define PARIS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct paris_ctx paris_ctx;

typedef enum {
  PARIS_OK = 0,
  PARIS_EINVAL = -1,    /* bad argument or unsupported configuration        */
  PARIS_ENOMEM = -2,    /* device or pinned-host allocation failed          */
  PARIS_ECUDA = -3,     /* a CUDA runtime call failed                       */
  PARIS_ESTATE = -4,    /* call not valid in the context's current state    */
  PARIS_ECAPACITY = -6, /* the sequence would exceed max_ctx tokens         */
  PARIS_EDEVICE = -7    /* a kernel reported a fault through the status word */
} paris_status;

typedef enum { PARIS_F32 = 0, PARIS_BF16 = 1 } paris_dtype;

typedef enum {
  PARIS_VOTE_RANK = 0, /* rank r of the query's top-rho centroids gives rho - r votes */
  PARIS_VOTE_FLAT = 1  /* every selected centroid gives 1 vote                     */
} paris_vote_weighting;

typedef enum {
  PARIS_TOPK_BY_SCORE = 0,   /* best estimate first, equal estimates by ascending
                                position (each block writes its entries at
                                their rank; past 16384 candidates one block per
                                list sorts it at the end of the kernel)       */
  PARIS_TOPK_BY_POSITION = 1 /* the same set in ascending position (no sort)   */
} paris_topk_order;

/* Shape and policy of one layer's cache.  Supported: head_dim = 128,
 * n_sub = 16 (m = 8), 1 <= rho <= 15 with rank weights or <= 256 with flat
 * weights, n_q_heads a multiple of n_kv_heads, update_buf >= 1,
 * 0 < cand_bp <= 10000, topk >= 1 (at most 16384 with PARIS_TOPK_BY_SCORE),
 * max_ctx <= 2^31 - 1.                                                       */
typedef struct {
  int batch;             /* sequences decoded in lock step                     */
  int n_kv_heads;        /* Hkv                                                */
  int n_q_heads;         /* Hq; G = Hq / Hkv query heads share a KV head       */
  int head_dim;          /* d                                                  */
  int n_sub;             /* B subspaces of m = d / B coordinates               */
  int rho;               /* top-rho centroids per subspace vote                */
  int sink;              /* S: first tokens always attended                    */
  int local;             /* L: most recent tokens always attended              */
  int update_buf;        /* U: appended tokens buffered before a flush         */
  int topk;              /* k retrieved tokens per query head                  */
  int cand_bp;           /* candidate fraction p in basis points (500 = 5%)    */
  int max_ctx;           /* capacity in tokens per sequence                    */
  int retrieval_on_host; /* 1: Retrieval-zone K/V in mapped pinned host memory */
  int vote_weighting;    /* paris_vote_weighting                               */
  int topk_order;        /* paris_topk_order of the top-k lists                */
} paris_config;

/* Zone bookkeeping, identical for every sequence of the batch.
 * Sink = [0, min(S, T)), Retrieval = [S, S + N), Local = [S + N, S + N + n_local),
 * Update Buffer = [S + N + n_local, T)  (token positions).                    */
typedef struct {
  int64_t T;       /* tokens in the cache                                      */
  int64_t N;       /* Retrieval-zone size                                      */
  int64_t n_local; /* Local-zone size                                          */
  int64_t n_buf;   /* tokens waiting in the Update Buffer                      */
  int64_t C;       /* candidates per query head for the current N              */
  int64_t k_eff;   /* min(topk, C): retrieved tokens per query head            */
  int64_t n_flushes; /* Update-Buffer flushes so far                           */
} paris_state;

/* Create a context for one layer.  srht_signs: host, head_dim entries, each
 * +1 or -1: the diagonal D of the shared rotation R = H D / sqrt(d) (ParisKV,
 * Methodology 1, "Normalization and Rotation"; the random draw is the
 * caller's).  Allocates every buffer the context will ever use (device
 * memory, and pinned mapped host memory for the Retrieval K/V when
 * retrieval_on_host = 1) and computes the RSQ-IP levels.  *out receives the
 * context; it is NULL on failure.                                            */
paris_status paris_create(const paris_config* cfg, const int8_t* srht_signs, paris_ctx** out);

/* Release everything the context owns.  Synchronises the device first.
 * NULL is ignored.                                                           */
void paris_destroy(paris_ctx* ctx);

/* Prefill: take T prompt tokens (ParisKV, system level, "Sliding-window
 * update mechanism": Sink = first S tokens, Local = last L tokens, the rest
 * is the Retrieval zone; w_{i,b} is precomputed here, Methodology 2,
 * "Calibration").  K, V: device, dtype elements, layout [batch][Hkv][T][d],
 * contiguous, owned by the caller and only read.  K/V are stored as bf16
 * (round to nearest even); keys are encoded from the given precision.
 * Valid only on an empty context; 0 <= T <= max_ctx.                         */
paris_status paris_encode_prefill(paris_ctx* ctx, const void* K, const void* V, paris_dtype dtype,
                                  int64_t T, void* stream);

/* Append one decode token per (sequence, KV head).  k, v: device, dtype
 * elements, [batch][Hkv][d].  The token enters the Update Buffer (or the
 * Sink while T < S); when the buffer holds U tokens they join Local and the
 * oldest Local tokens beyond L move to the Retrieval zone, whose search
 * index is then rebuilt for the affected chunks (ParisKV, system level,
 * "Sliding-window update mechanism").  Returns PARIS_ECAPACITY at max_ctx. */
paris_status paris_append_decode(paris_ctx* ctx, const void* k, const void* v, paris_dtype dtype,
                                 void* stream);

/* Retrieve the top-k Retrieval-zone tokens for each query head (ParisKV,
 * Methodology 2: collision votes over the top-rho centroids per subspace,
 * the top C = max(ceil(p N), min(k, N)) keys by (votes desc, position asc)
 * as candidates, RSQ-IP rerank, top min(k, C) by (estimate desc, position
 * asc)).  q: device, dtype, [batch][Hq][d].  topk_idx: device int32
 * [batch][Hq][topk] receives absolute token positions, listed by (estimate
 * desc, position asc) with topk_order = PARIS_TOPK_BY_SCORE, in ascending
 * position with PARIS_TOPK_BY_POSITION; topk_score: device float32, same
 * layout, the RSQ-IP estimates of <k, q> of those positions; entries past
 * k_eff are -1 and -inf.  topk_score may be NULL.  k_eff: host, receives
 * min(topk, C) (0 while the Retrieval zone is empty).  One launch (with
 * PARIS_TOPK_BY_SCORE its blocks write position order to context scratch
 * and, where every key of the query head is in their shared memory, each
 * entry at its best-first rank in topk_idx/score; otherwise one block per
 * query head sorts the scratch into them).                                */
paris_status paris_retrieve(paris_ctx* ctx, const void* q, paris_dtype dtype, int32_t* topk_idx,
                            float* topk_score, int64_t* k_eff, void* stream);

/* Sparse attention over Sink U Local U Update Buffer U the retrieved tokens
 * (ParisKV: attention restricted to the selected KV; the Retrieval-zone rows
 * are read in place, from mapped host memory when retrieval_on_host = 1 --
 * system level, "UVA offloading").  o = softmax(K_S q / sqrt(d)) V_S with
 * float32 accumulation.  q: device, dtype, [batch][Hq][d]; topk_idx: device
 * int32 [batch][Hq][topk] as produced by paris_retrieve (entries < 0 are
 * skipped; an entry outside the Retrieval zone is skipped and flagged in the
 * status word); out: device bf16 [batch][Hq][d].                            */
paris_status paris_sparse_attend(paris_ctx* ctx, const void* q, paris_dtype dtype,
                                 const int32_t* topk_idx, void* out_bf16, void* stream);

/* The same sparse attention as paris_sparse_attend (same arguments, same
 * result), for callers that must not allocate device memory: code running
 * while another component owns the device allocator, or a serving loop whose
 * device memory budget is fixed up front.  Its per-call scratch (the split
 * partials and merge counters) lives in one fixed area compiled into the
 * library (about 545 KB, held by every GPU that loads the library until the
 * process exits) instead of in the context, and the call allocates nothing.
 * The pages have no counterpart; this is a property of this library.
 * Limit: batch x n_q_heads x splits <= 1024, with splits =
 * ceil((tokens in Sink, Local and Update Buffer + k_eff) / 64), and
 * batch x n_q_heads <= 1024; larger calls return PARIS_EINVAL.  The first call
 * on a device looks up the area's device address once (cudaGetSymbolAddress
 * with that device current); make that first call before any stream capture.
 * Every call on a device shares the one area, which keeps the last call's
 * contents: calls that may overlap on the GPU (different streams, or
 * different host threads) race and must be serialised by the caller.      */
paris_status paris_sparse_attend_noalloc(paris_ctx* ctx, const void* q, paris_dtype dtype,
                                         const int32_t* topk_idx, void* out_bf16, void* stream);

/* Learned-centroid baseline (ParisKV, "Problem definition": learned
 * codebooks such as k-means centroids fitted on the prefill keys, against
 * which the analytic centroids are compared under drift): centroids
 * replaces the 2^m sign-pattern centroids of every subspace by a table,
 * device float32 [Hkv][B][2^m][m] (m = 8), for this context's bucket ids
 * and query scores.  A key's id in subspace b is the centroid c with the
 * largest float32 score ((0 + z_0 c_0) + z_1 c_1) + ... + z_7 c_7 over the
 * rotated subvector z (lowest id on ties); a query's centroid scores are
 * the same sums, its top-rho chosen as with the analytic centroids.
 * Everything else (codes, w, votes, rerank) is unchanged.  The table is
 * copied into the context.  centroids = NULL restores the analytic
 * centroids.  Only while the cache is empty (else PARIS_ESTATE).           */
paris_status paris_set_centroids(paris_ctx* ctx, const float* centroids, void* stream);

/* GQA-shared sparse attention: every query head of a KV head attends over
 * Sink U Local U Update Buffer U the union of the retrieved tokens of all G
 * query heads of that KV head, so each K/V row is read once per KV head
 * instead of once per query head that retrieved it (the GQA-shared
 * retrieval variant: K/V gather bytes fall by up to G when the heads'
 * top-k sets overlap).  Each head's set is a superset of its own
 * paris_sparse_attend set; with G = 1 the two calls attend over the same
 * rows.  topk_idx: device int32 [batch][Hq][topk] as produced by
 * paris_retrieve (in either order; entries < 0 are skipped, entries
 * outside the Retrieval zone skipped and flagged).  q and out as in
 * paris_sparse_attend.  Same arithmetic as paris_dense_attend.  Limit: at
 * most 16 query heads per KV head, else PARIS_EINVAL.  One launch: each
 * block builds the union over its own slice of the Retrieval zone and
 * attends over it and its share of the window; scratch from paris_create. */
paris_status paris_sparse_attend_gqa(paris_ctx* ctx, const void* q, paris_dtype dtype, const int32_t* topk_idx,
                                     void* out_bf16, void* stream);

/* Dense decode attention over every cached token -- Sink, Retrieval zone,
 * Local and Update Buffer -- for each query head: the full-attention
 * baseline ParisKV's decode throughput is compared against (ParisKV,
 * Experiments, "Efficiency": throughput over full attention).  Same
 * arithmetic as paris_sparse_attend (o = softmax(K q / sqrt(d)) V, float32
 * accumulation, bf16 output) over all T rows instead of the selected ones;
 * Retrieval-zone rows are read in place (mapped host memory when
 * retrieval_on_host = 1).  q: device, dtype, [batch][Hq][d]; out: device
 * bf16 [batch][Hq][d] (zeros while the cache is empty).  Streams every K/V
 * row once per call for all query heads of its KV head (at most 16 query
 * heads per KV head, else PARIS_EINVAL), split over about one block per SM;
 * the query enters the products as two bf16 parts, the softmax weights
 * rounded to bf16.
 * Its scratch is allocated by paris_create.                                 */
paris_status paris_dense_attend(paris_ctx* ctx, const void* q, paris_dtype dtype, void* out_bf16, void* stream);

/* One decode step: paris_append_decode(k, v), then paris_retrieve(q, ...),
 * then paris_sparse_attend(q, topk_idx, out), with the same arguments.  The
 * top-k positions, their estimates and k_eff are bit for bit those of the
 * three calls; the attention output is the same sum in another float32
 * order (here it runs inside the retrieval kernel, its rows split over the
 * blocks that serve each query head).  One kernel launch when the append
 * does not fill the Update Buffer: the step's own token is read from k/v
 * where the attention needs it and written to the cache at the end of the
 * kernel.
 * When it does, the append, flush and index rebuild run first.
 * k, v: device, kv_dtype, [batch][Hkv][d]; q: device, q_dtype,
 * [batch][Hq][d]; outputs as in the three calls.                           */
paris_status paris_decode_step(paris_ctx* ctx, const void* k, const void* v, paris_dtype kv_dtype, const void* q,
                               paris_dtype q_dtype, int32_t* topk_idx, float* topk_score, void* out_bf16,
                               int64_t* k_eff, void* stream);

/* Copy the zone bookkeeping to *out (host).  No device work.               */
paris_status paris_get_state(const paris_ctx* ctx, paris_state* out);

/* Synchronise the device and report the status word: PARIS_OK, or
 * PARIS_EDEVICE (then cleared) if a kernel flagged a fault since the last
 * check.                                                                    */
paris_status paris_check_device(paris_ctx* ctx);

/* Debug and test access.  Synchronises the device, then copies one table
 * to host memory `dst` of `bytes` bytes (PARIS_EINVAL if too small):
 *  PARIS_DUMP_IDS      seq, head = KV head: uint8  [N][B] bucket ids
 *  PARIS_DUMP_CODES    seq, KV head:        uint8  [N][d/2] packed 4-bit codes
 *                      (coordinate c in byte c/2, even c in the low nibble)
 *  PARIS_DUMP_W        seq, KV head:        float  [N][B] calibration w
 *  PARIS_DUMP_VOTES    seq, head = q head:  uint8  [N] votes of the last retrieve
 *  PARIS_DUMP_CANDS    seq, q head:         int32  [C] candidate positions, ascending
 *  PARIS_DUMP_CAND_EST seq, q head:         float  [C] their estimates
 *  PARIS_DUMP_QT       seq, q head:         float  [d] rotated unit query q~
 *  PARIS_DUMP_QNORM    seq, q head:         float  [1] ||q||
 *  PARIS_DUMP_HOT      seq, q head:         uint32 [B][rho] centroid id | weight << 16
 *  PARIS_DUMP_LEVELS   (seq, head ignored): float  [15] 8 levels, 7 thresholds
 *  PARIS_DUMP_KV       seq, KV head:        uint16 [2][T][d] bf16 K then V by position
 *  PARIS_DUMP_TRACE    (seq, head ignored): uint64 phase timestamps (ns, GPU
 *                      global timer) of the last kernels, recorded only when the
 *                      environment had PARIS_TRACE=1 at paris_create: 64 phase
 *                      slots, then (start, after wait, -, end) of each of up to
 *                      4096 blocks of 8 kernels; copies min(bytes, size) */
enum {
  PARIS_DUMP_IDS = 0, PARIS_DUMP_CODES = 1, PARIS_DUMP_W = 2, PARIS_DUMP_VOTES = 3,
  PARIS_DUMP_CANDS = 4, PARIS_DUMP_CAND_EST = 5, PARIS_DUMP_QT = 6, PARIS_DUMP_QNORM = 7,
  PARIS_DUMP_HOT = 8, PARIS_DUMP_LEVELS = 9, PARIS_DUMP_KV = 10, PARIS_DUMP_TRACE = 11
};
paris_status paris_debug_dump(paris_ctx* ctx, int what, int seq, int head, void* dst, size_t bytes);

/* Text of the last error on this context ("" if none).  ctx may be NULL:
 * then the last error of a failed paris_create is returned.                */
const char* paris_last_error(const paris_ctx* ctx);

/* Kernels of the library, for per-kernel accounting. */
typedef enum {
  PARIS_KERNEL_PLACE_KV = 0,    /* prefill: K/V into Sink, store and Local ring          */
  PARIS_KERNEL_ENCODE = 1,      /* prefill: SRHT, bucket ids, codes, w                   */
  PARIS_KERNEL_BUILD_INDEX = 2, /* per-chunk inverted bucket index                       */
  PARIS_KERNEL_APPEND = 3,      /* standalone decode append (store + encode one token)   */
  PARIS_KERNEL_DECODE = 4,      /* fused retrieval: query preparation, votes, candidates,
                                   rerank, top-k; in a decode step also the sparse
                                   attention and the append of the step's token      */
  PARIS_KERNEL_ATTEND = 5,      /* standalone sparse attention and the merge of its splits */
  PARIS_KERNEL_FILL = 6,        /* empty-result fill                                     */
  PARIS_KERNEL_DENSE = 7,       /* attention streaming rows once per KV head: the dense
                                   comparator, and the GQA-shared sparse attention      */
  PARIS_KERNEL_UNION = 8,       /* not launched: the GQA-shared attention builds its union
                                   inside its PARIS_KERNEL_DENSE launch                 */
  PARIS_KERNEL_COUNT = 9
} paris_kernel;

/* Cumulative kernel launches of this context since paris_create, per
 * paris_kernel.  counts: host, PARIS_KERNEL_COUNT entries.  No device work. */
paris_status paris_launch_counts(const paris_ctx* ctx, int64_t* counts);

/* Per-kernel timing.  After paris_profile_begin, every kernel the context
 * launches (up to max_launches of them) is bracketed by two CUDA events
 * recorded on its launch stream.  paris_profile_end synchronises, writes the
 * summed event time in milliseconds and the number of timed launches per
 * paris_kernel to total_ms / launches (host, PARIS_KERNEL_COUNT entries each,
 * either may be NULL), and releases the events.  Launches past max_launches
 * run untimed.                                                             */
paris_status paris_profile_begin(paris_ctx* ctx, int max_launches);
paris_status paris_profile_end(paris_ctx* ctx, double* total_ms, int64_t* launches);

/* Host only, no device work: the RSQ-IP magnitude levels for subspace width
 * m, computed by float64 Lloyd-Max on the density of |x_j| for x uniform on
 * the unit sphere S^{m-1} (x_j^2 ~ Beta(1/2, (m-1)/2); ParisKV,
 * Methodology 2, "Quantization": levels from the rotation-induced Beta
 * prior).  levels: host, 8 doubles ascending; thresholds: host, 7 doubles,
 * the midpoints.  2 <= m <= 64.                                              */
paris_status paris_rsq_levels(int m, double* levels, double* thresholds);

#ifdef __cplusplus
}
#endif

#endif /* PARIS_H_ */
