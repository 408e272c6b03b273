/*
 * qrita.h - exact, deterministic top-k / top-p candidate-set selection over
 * large-vocabulary logits, on one NVIDIA GB300 (sm_103a).
 *
 * Method: Qrita technical summary (gist.science, paper 2602.01518).
 *  - "Problem statement": the result is the full candidate set with the exact
 *    semantics of sort-based top-k / top-p (deterministic, not one sample).
 *  - "Methodology", part 1 (Gaussian sigma-truncation): mu and sigma from a
 *    sample block, threshold t = mu + delta*sigma with delta from tables built
 *    from the normal quantile function for the target k or p; one pass keeps
 *    Z_t = {x >= t}; the search runs on Z_t on a truncation hit and on the
 *    full row otherwise.
 *  - "Methodology", part 2 (quaternary pivot search with duplicate handling):
 *    three pivots at 25/50/75 % of the current range per iteration, tracking
 *    z_mn (smallest logit above the pivot) and N_zmn (its count) to know how
 *    many boundary duplicates to keep.
 *  - "Implementation details", pipeline: rows in parallel; truncation, then
 *    quaternary search, then the duplicate-handling mask.
 *
 * Result contract (every entry point below): for row r with logits
 * x[0..V), the kept set is what a stable descending sort gives (equal logits:
 * lower token id first; -0 == +0; -inf last): top-k first (k_r in [1, V)),
 * then, over the top-k set renormalised, the smallest prefix whose softmax
 * mass reaches p_r (p_r < 1). k_r <= 0 or k_r >= V disables top-k; p_r >= 1
 * or NaN disables top-p; p_r <= 0 keeps exactly one token. A row holding NaN
 * or +inf gets an all-zero mask and a non-zero row status. At least one token
 * is kept in every valid row.
 *
 * Top-k masks are bit-exact. Top-p masks are bit-exact except on rows whose
 * cumulative mass at the boundary lies within 1e-6 * p of p. On such a row
 * the kept set is still a prefix of the stable descending order of S_k, of
 * n tokens, where n is the definition's count, one more or one fewer, or any
 * count the band cannot tell from it: c(n) >= p - 1e-6 p and
 * c(n - 1) < p + 1e-6 p, c(n) being the renormalised mass of the first n
 * tokens. On short rows that is one token either way; on rows of millions of
 * logits, where one token carries far less than 1e-6 of the mass, it can be
 * several. Arithmetic: every softmax weight is fp32 exp(x - m) rounded to an
 * unsigned 64-bit fixed-point integer, and all masses are exact integer sums
 * of those weights (so every decision is deterministic and independent of
 * summation order); the definition is fp64.
 *
 * Threading: every entry point is reentrant and thread-safe, keeps no state
 * between calls and allocates no memory. Launches are stream-ordered; the
 * device entry points never synchronise.
 */
#ifndef QRITA_H_
#define QRITA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* qrita_stream_t;

/* Logit element types. */
enum {
  QRITA_DTYPE_F32 = 0,  /* IEEE binary32 */
  QRITA_DTYPE_BF16 = 1  /* bfloat16, widened exactly to binary32 */
};

/* Return codes of every entry point. */
enum {
  QRITA_OK = 0,
  QRITA_EINVAL = 1,       /* bad argument: null pointer, B < 0, V < 1, V > 2^31-1,
                             unknown dtype, misaligned element pointer, bad flags */
  QRITA_EUNSUPPORTED = 2, /* valid but outside this build: B*C CTAs above 2^31-1,
                             or no launch shape fits the device */
  QRITA_ECUDA = 3         /* a CUDA runtime call or the launch failed */
};

/* Per-row status written to row_status[r] (qrita_select_ex). */
enum {
  QRITA_ROW_OK = 0,
  QRITA_ROW_NONFINITE = 1,  /* NaN or +inf in the row: mask all zero */
  QRITA_ROW_SEARCH_CAP = 2, /* pivot search exceeded its round cap: mask all zero
                               (cannot happen by construction; kept as a guard) */
  QRITA_ROW_TIMEOUT = 3     /* a bounded wait for a bulk copy of the row's logits
                               gave up (not expected on a healthy device): mask
                               all zero */
};

/* Flags of qrita_select_ex (path forcing for tests and ablations). */
#define QRITA_FLAG_NO_TRUNCATION 0x1u  /* skip sigma-truncation: search the full row */
#define QRITA_FLAG_FORCE_FALLBACK 0x2u /* treat every truncation as a miss and search
                                          the full row (no second truncation) */
#define QRITA_FLAG_KEY_PIVOTS 0x4u     /* pivots at quartiles of the 32-bit key range
                                          only (no value-space quartiles) */
#define QRITA_FLAG_FORCE_RETRY 0x8u    /* top-k rows: treat the first truncation as a
                                          miss, so the second truncation runs */
#define QRITA_FLAG_HIST_MISS 0x10u     /* top-p rows binned by the streaming pass: after
                                          the pass that lists the boundary's bin, treat
                                          its bracket as missed, so the narrowing passes
                                          run (and the mask is written again) */
#define QRITA_FLAG_CLUSTER_SHIFT 8     /* bits 8..10: force 2^n CTAs per row (n in 0..4);
                                          0 in these bits and bit 11 clear = automatic */
#define QRITA_FLAG_CLUSTER_SET 0x800u  /* bit 11: the cluster-size bits are set */
#define QRITA_FLAG_TEST_GIVE_UP 0x1000u /* tests only: the first bounded wait for a bulk
                                           copy in the first CTA of row 0 reports that it
                                           gave up (without waiting), so that row takes the
                                           QRITA_ROW_TIMEOUT path; the copy still lands and is
                                           waited for before the CTA exits */
#define QRITA_FLAG_NO_KEY_HIST 0x2000u /* bf16 rows: search with pivot rounds even where the
                                           survivors span few enough 16-bit keys for the
                                           key histogram */
#define QRITA_FLAG_SEARCH_QUATERNARY 0x4000u /* ablation: the pages' literal search form, three
                                                 pivots (25/50/75 %) a round or narrowing pass,
                                                 four bins per tail split, no 256-bin first pass */
#define QRITA_FLAG_SEARCH_BINARY 0x8000u     /* ablation: one pivot (the middle) a round or pass,
                                                 two bins per tail split, no 256-bin first pass
                                                 (wins over QRITA_FLAG_SEARCH_QUATERNARY) */
#define QRITA_FLAG_KNOWN_MASK 0xFFFFu

/* Bits of qrita_row_info_t.path. */
#define QRITA_PATH_TOPK 0x1u      /* top-k active for the row */
#define QRITA_PATH_TOPP 0x2u      /* top-p active for the row */
#define QRITA_PATH_TRUNC 0x4u     /* sigma-truncation pass ran */
#define QRITA_PATH_HIT 0x8u       /* truncation hit: the search ran on Z_t */
#define QRITA_PATH_FALLBACK 0x10u /* the search ran on the full row */
#define QRITA_PATH_OVERFLOW 0x20u /* Z_t did not fit a CTA's shared-memory list */
#define QRITA_PATH_KEEP_ALL 0x40u /* both filters off: every token kept */
#define QRITA_PATH_RETRY 0x80u    /* top-k: a second truncation at an order statistic
                                     of a 4096-logit sample ran (the search ran on
                                     its survivors unless FALLBACK is also set) */
#define QRITA_PATH_SAMPLE_T 0x200u /* top-k: the sample contradicted the Gaussian
                                     threshold; an order statistic of the sample
                                     was the threshold */
#define QRITA_PATH_HIST 0x100u    /* top-p alone: value bins counted by the streaming
                                     pass placed the boundary, and one more pass
                                     extracted those bins for the search */
#define QRITA_PATH_KEYHIST 0x400u /* bf16 truncation hit: one histogram of the survivors'
                                     16-bit keys placed the top-k boundary (and the
                                     top-p boundary over S_k) */

/* Diagnostics of one row (qrita_select_ex, optional). Device memory. */
typedef struct qrita_row_info {
  float mu;            /* sample-block mean of the finite logits */
  float sigma;         /* sample-block standard deviation */
  float threshold;     /* t = mu + delta*sigma; -inf when truncation did not run */
  float row_max;       /* largest logit m (softmax shift) */
  uint32_t survivors;  /* |Z_t| = #{x >= t} (0 when truncation did not run) */
  uint32_t path;       /* QRITA_PATH_* bits */
  uint32_t rounds_k;   /* quaternary rounds of the top-k search */
  uint32_t rounds_p;   /* quaternary rounds of the top-p search */
  float boundary;      /* logit of the last kept token in sort order */
  uint32_t n_boundary; /* kept tokens whose logit equals boundary */
  uint32_t kept;       /* kept tokens */
  uint32_t status;     /* QRITA_ROW_* (same as row_status[r]) */
  double z;            /* softmax denominator top-p normalised by (0 if top-p off) */
  uint32_t passes;     /* distributed narrowing passes (fallback searches) */
  uint32_t reserved;
} qrita_row_info_t;

/*
 * qrita_select: the whole pipeline for B rows on one stream.
 *
 *   logits   device, [B, V] row-major, leading dimension V, dtype elements;
 *            aligned to the element size (any 16-byte misalignment is fine).
 *   dtype    QRITA_DTYPE_F32 or QRITA_DTYPE_BF16.
 *   B, V     rows and vocabulary size; B == 0 returns QRITA_OK and launches
 *            nothing; 1 <= V <= 2^31-1.
 *   k        device int32[B], or NULL (top-k off for every row).
 *   p        device float[B], or NULL (top-p off for every row).
 *   out_mask device uint8[B, V]: 1 = kept, 0 = dropped (torch.bool layout).
 *   stream   CUDA stream the kernel is enqueued on.
 *
 * Ownership: all pointers belong to the caller; nothing is retained after
 * the call returns; inputs must stay unchanged until the stream reaches the
 * kernel. Errors are returned synchronously for arguments and launches only
 * (QRITA_EINVAL, QRITA_EUNSUPPORTED, QRITA_ECUDA); data problems go to the
 * per-row status of qrita_select_ex and never abort the call.
 */
int qrita_select(const void* logits, int dtype, int64_t B, int64_t V, const int32_t* k,
                 const float* p, uint8_t* out_mask, qrita_stream_t stream);

/*
 * qrita_select_ex: qrita_select plus path flags and optional outputs.
 *
 *   flags      QRITA_FLAG_* (0 = same as qrita_select); unknown bits: EINVAL.
 *   row_status device int32[B] or NULL: QRITA_ROW_* per row.
 *   row_info   device qrita_row_info_t[B] or NULL: per-row diagnostics.
 *
 * Same ownership and error behaviour as qrita_select.
 */
int qrita_select_ex(const void* logits, int dtype, int64_t B, int64_t V, const int32_t* k,
                    const float* p, uint8_t* out_mask, qrita_stream_t stream, uint32_t flags,
                    int32_t* row_status, qrita_row_info_t* row_info);

/*
 * qrita_host_staging_bytes: device bytes qrita_select_host needs as staging
 * for B rows of V dtype logits (inputs, k, p and the mask, 256-byte aligned
 * sections). Returns 0 for invalid arguments.
 */
size_t qrita_host_staging_bytes(int dtype, int64_t B, int64_t V);

/*
 * qrita_select_host: the same selection for HOST buffers, end to end.
 *
 *   h_logits, h_k, h_p   host inputs (h_k / h_p may be NULL as above); pinned
 *                        memory gives full-speed copies, pageable works too.
 *   h_mask               host uint8[B, V] output.
 *   d_staging            device buffer of at least qrita_host_staging_bytes
 *                        bytes, owned by the caller (the call allocates none).
 *
 * Enqueues the host-to-device copies, the kernel and the device-to-host copy
 * on stream, then waits for the stream; the mask is in h_mask on return.
 * Errors as qrita_select (QRITA_EINVAL also when staging_bytes is short).
 */
int qrita_select_host(const void* h_logits, int dtype, int64_t B, int64_t V, const int32_t* h_k,
                      const float* h_p, uint8_t* h_mask, void* d_staging, size_t staging_bytes,
                      qrita_stream_t stream);

/*
 * qrita_topk_ids: the top-k token ids of every row in stable order (logit
 * descending, equal logits by lower id), as a drafter keeps them (Qrita
 * technical summary, "Problem statement": the full candidate set with the
 * exact sort-based semantics, here in rank order).
 *
 *   logits, dtype, B, V   as qrita_select.
 *   k        device int32[B] (required): row r gets the first k_r ids of its
 *            stable descending order when 1 <= k_r <= kmax (and min(k_r, V)
 *            when k_r >= V); other rows get none.
 *   kmax     1 .. 8192: the length of each row of out_ids.
 *   out_mask device uint8[B, V]: the top-k keep-mask (also an output; the
 *            ids are read back from it).
 *   out_ids  device int32[B, kmax]: the ids in rank order, then -1.
 *
 * Two kernels on stream (the selection, then the ids); allocates nothing.
 * Errors as qrita_select; QRITA_EINVAL also for k == NULL, out_ids == NULL
 * or kmax outside 1 .. 8192.
 */
int qrita_topk_ids(const void* logits, int dtype, int64_t B, int64_t V, const int32_t* k, int32_t kmax,
                   uint8_t* out_mask, int32_t* out_ids, qrita_stream_t stream);

/*
 * qrita_candidates: the candidate lists a verifier or a sampler consumes
 * after the mask, and one token drawn from each (Qrita technical summary,
 * "Problem statement": the complete candidate set, beside the single sampled
 * token stochastic samplers return).
 *
 *   logits, dtype, B, V   as qrita_select.
 *   mask       device uint8[B, V], e.g. qrita_select's output (nonzero = kept).
 *   cap        >= 1: the length of each row of out_ids / out_probs.
 *   out_ids    device int32[B, cap]: the kept ids in increasing id order; a
 *              row keeping more than cap writes its first cap.
 *   out_probs  device float[B, cap]: their probabilities renormalised over
 *              the row's kept set, p_i = exp(x_i - m) / sum over kept of
 *              exp(x_j - m), m the largest kept logit (fp32, from 64-bit
 *              fixed-point weights; within a few 1e-7 relative of fp64).
 *   out_count  device int32[B]: the row's kept count (may exceed cap).
 *   u          device float[B] or NULL: one uniform in [0, 1) per row.
 *   out_sample device int32[B] or NULL (NULL exactly when u is): the first
 *              kept id, in id order, whose cumulative probability exceeds
 *              u_r; -1 for a row that keeps nothing.
 *
 * Entries past a row's count are left as they were. Two kernels at most on
 * stream; allocates nothing. Errors as qrita_select; QRITA_EINVAL also for
 * cap < 1, a NULL output, or exactly one of u / out_sample NULL.
 */
int qrita_candidates(const void* logits, int dtype, int64_t B, int64_t V, const uint8_t* mask, int32_t cap,
                     int32_t* out_ids, float* out_probs, int32_t* out_count, const float* u, int32_t* out_sample,
                     qrita_stream_t stream);

/*
 * qrita_delta_table: copy one of the host-built truncation tables the kernel
 * receives (Qrita technical summary, "Methodology", part 1: delta comes from
 * precomputed tables of the normal quantile function keyed on k or p).
 *
 *   which  0: the top-k table, entry i = Phi^-1(1 - 2^(-i/4));
 *          1: the top-p table, entry i = Phi^-1(2^(-i/4)).
 *   out    host float[n] or NULL; receives min(n, length) entries.
 *
 * Returns the table's length (entries), or -1 when `which` is unknown.
 * Touches no device; for tests and diagnostics.
 */
int qrita_delta_table(int which, float* out, int n);

/* Static, human-readable text for a QRITA_* return code. */
const char* qrita_strerror(int code);

/* Library version: major*10000 + minor*100 + patch. */
int qrita_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QRITA_H_ */
