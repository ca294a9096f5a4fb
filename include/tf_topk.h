/*
 * tf_topk.h -- exact per-row top-k over wide bf16 logit rows, on GB300 (sm_103a).
 *
 * The operation: TensorFold PR #713, "perf(qwen27): a drafted round overlaps
 * its cache commit with the next draft, and the drafter's attention and top-k
 * use more of the GPU".
 *   - Change 3 of the PR's list: each row of a bf16 draft-head logit matrix
 *     (15 rows x 98592 columns there) yields its best k entries, ordered by
 *     score descending and, between equal scores, by the lower token index.
 *     Wide rows are scanned in column spans and the span results merged in the
 *     same order; a compile-time check ties the kernel constants (lanes, spans,
 *     max_k) to the host side.
 *   - The "Exactness" table: each row reports its entries, a count and a
 *     non-finite mask; the cases cover widths 4096 to 248320, ties, both
 *     zeros, NaN, infinities and padded row strides, and a "Row ABI and guards"
 *     check validates the call's arguments.
 *
 * Conventions the pages leave open (the same readings as the CPU oracle):
 *   - a NaN (any sign or payload) is never selected;
 *   - +0 and -0 are equal scores (they tie, the lower column wins); every
 *     reported value keeps the original bits of its column;
 *   - +inf and -inf are ordinary extreme scores; subnormals are exact;
 *   - count = min(k, number of non-NaN columns of the row);
 *   - mask = (row has NaN ? 1 : 0) | (has +inf ? 2 : 0) | (has -inf ? 4 : 0),
 *     over columns [0, cols) only;
 *   - slots count..k-1 hold index -1 and value bits 0x7FC0.
 * The result is unique (ties are broken by column), so two correct
 * implementations agree bit for bit.
 *
 * Every call is asynchronous on the given stream and returns after the launch;
 * device faults, if any, surface at the caller's next synchronisation.  The
 * library allocates no output.  The allocating entry points keep no per-call
 * state beyond their per-stream scratch, so their calls on different streams
 * and host threads may overlap.  The exception is tf_topk_bf16_noalloc, whose
 * calls all share one static scratch array and must not overlap on the GPU
 * (see its section).  On an error return nothing has been launched and no
 * output has been written.
 */
#ifndef TF_TOPK_H
#define TF_TOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest k a call accepts (the pages' max_k constant; its value is not given
 * there -- 64 is the largest k of the workloads this library targets). */
#define TF_TOPK_MAX_K 64
/* Most column spans (cooperating CTAs) one row may be split over, and most
 * pieces a row is cut into by the stream plan. */
#define TF_TOPK_MAX_SPANS 16

/* Status codes. */
#define TF_TOPK_OK 0
#define TF_TOPK_ERR_NULL 1   /* a required pointer is NULL (rows > 0) */
#define TF_TOPK_ERR_SHAPE 2  /* rows < 0, cols < 1, row_stride < cols, cols >= 2^31,
                                or rows * row_stride overflows */
#define TF_TOPK_ERR_K 3      /* k < 1 or k > TF_TOPK_MAX_K */
#define TF_TOPK_ERR_ALIGN 4  /* logits/out_val not 2-byte, out_idx/out_count/mask not
                                4-byte aligned */
#define TF_TOPK_ERR_PLAN 5   /* tf_topk_bf16_with_plan: unknown plan code */
#define TF_TOPK_ERR_DEVICE 6 /* current device is not compute capability 10.3 */
#define TF_TOPK_ERR_CUDA 7   /* a CUDA runtime call or the launch failed; see
                                tf_topk_last_cuda_error() */

/*
 * Exact top-k of every row of a bf16 matrix.
 *
 *   logits             device pointer, bf16 bit patterns, row r at
 *                      logits + r * row_stride (elements); columns
 *                      [cols, row_stride) are padding and are never read.
 *                      Any 2-byte-aligned address and any row_stride >= cols
 *                      are accepted.
 *   rows, cols         matrix shape; rows == 0 is a no-op returning TF_TOPK_OK.
 *   row_stride         elements between row starts.
 *   k                  1..TF_TOPK_MAX_K; k > cols is allowed (empty slots).
 *   out_idx            device, int32 [rows][k]: selected column indices.
 *   out_val            device, uint16 [rows][k]: bf16 bits of those columns.
 *   out_count          device, int32 [rows].
 *   out_nonfinite_mask device, uint32 [rows].
 *   stream             cudaStream_t to launch on (NULL = the legacy default
 *                      stream).
 * All buffers are owned by the caller; outputs must not overlap the input.
 * The call runs on the current CUDA device.  Returns a TF_TOPK_* status.
 *
 * Scratch: the plans this call picks need none.  The stream plan
 * (TF_TOPK_PLAN_STREAM, only through tf_topk_bf16_with_plan) keeps a small
 * per-(device, stream) area (two k-entry lists and a ticket per CTA, under
 * 1 MB) that the library allocates on its first call on that stream and keeps
 * until exit; that first call therefore allocates (cudaMalloc) and should not
 * be made during stream capture.  Each stream-plan launch first clears the
 * tickets it uses with an asynchronous memset on `stream`.  Outputs are never
 * allocated by the library.
 */
int tf_topk_bf16(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                 int32_t *out_idx, uint16_t *out_val, int32_t *out_count,
                 uint32_t *out_nonfinite_mask, void *stream);

/* Launch plans (tf_topk_bf16_with_plan).  Every plan gives identical results. */
#define TF_TOPK_PLAN_AUTO 0      /* what tf_topk_bf16 picks for the shape (measured on
                                    GB300): with at least one row per SM, SINGLE when a
                                    row is at most one chunk (16384 columns) or when two
                                    spans a row would take three waves or more, else
                                    CLUSTER2; with fewer rows, the span count whose grid
                                    reaches about two CTAs per SM without spans narrower
                                    than half a chunk (SINGLE when even two would be) */
#define TF_TOPK_PLAN_SINGLE 1    /* one CTA per whole row (the pages' single-group
                                    kernel): the cluster kernel without a split */
#define TF_TOPK_PLAN_CLUSTER2 2  /* each row split into 2/4/8/16 column spans, one */
#define TF_TOPK_PLAN_CLUSTER4 4  /*   CTA each, inside one thread-block cluster; */
#define TF_TOPK_PLAN_CLUSTER8 8  /*   the span lists are merged through distributed */
#define TF_TOPK_PLAN_CLUSTER16 16/*   shared memory */
#define TF_TOPK_PLAN_STREAM 32   /* persistent CTAs stream equal contiguous ranges
                                    of the matrix through a TMA ring; rows cut by a
                                    range boundary are merged by the last CTA to
                                    finish one of their pieces */

/*
 * The same operation with the launch plan named by the caller (for
 * cross-path tests and A/B timing).  `plan` is one of TF_TOPK_PLAN_*;
 * anything else returns TF_TOPK_ERR_PLAN.
 */
int tf_topk_bf16_with_plan(const void *logits, int64_t rows, int64_t cols, int64_t row_stride,
                           int32_t k, int32_t *out_idx, uint16_t *out_val, int32_t *out_count,
                           uint32_t *out_nonfinite_mask, int32_t plan, void *stream);

/* The plan tf_topk_bf16 picks for this shape on the current device (a
 * TF_TOPK_PLAN_* code), or a negative TF_TOPK_* status if the shape is
 * invalid. */
int32_t tf_topk_bf16_plan(int64_t rows, int64_t cols, int32_t k);

/*
 * Device-side fault check.  Every wait inside the kernels is bounded; a wait
 * that runs out records a nonzero code in a per-device word and the kernel
 * returns early (its rows' outputs are then not valid).  This call waits for
 * the current device to finish its work, returns 0 when no kernel recorded a
 * fault since the last check, else the fault code (1 = a bulk-copy wait ran
 * out), and clears it.  A negative value is -TF_TOPK_ERR_CUDA.
 */
int tf_topk_device_fault(void);

/* Compile-time constants of the kernels, exported so a host-side check can
 * compare them with the header (the pages' constant tie between kernel and
 * host). */
int32_t tf_topk_bf16_max_k(void);         /* == TF_TOPK_MAX_K */
int32_t tf_topk_bf16_max_spans(void);     /* == TF_TOPK_MAX_SPANS */
int32_t tf_topk_bf16_cta_threads(void);   /* threads per CTA */
int32_t tf_topk_bf16_chunk_columns(void); /* columns one CTA holds in registers per pass */

/* Most shard lists tf_topk_merge_bf16 merges per row. */
#define TF_TOPK_MAX_SHARDS 64

/*
 * Merge of per-shard top lists into each row's top k: the pages' merge stage
 * on its own (PR #713, change 3: span results merged in the same score /
 * lower-index order), for rows whose columns were split over shards (a
 * vocab-sharded head, or rows spread over several calls or devices).
 *
 *   in_idx, in_val, in_count, in_nonfinite_mask
 *                      device; shard s, row r: in_idx[(s * rows + r) * k_in ..
 *                      + k_in), likewise in_val, and in_count[s * rows + r],
 *                      in_nonfinite_mask[s * rows + r] -- exactly what
 *                      tf_topk_bf16 writes for one shard's column block
 *                      (indices local to the block, best first).  Only the
 *                      first min(k, k_in, in_count) entries of a list are read
 *                      (no entry past them can reach the top k); a list ends
 *                      early at an entry with a negative index or a NaN
 *                      value.
 *   rows, shards       1 <= shards <= TF_TOPK_MAX_SHARDS.
 *   k_in               entries per input list, 1..TF_TOPK_MAX_K.
 *   shard_offset       HOST array [shards]: the column of shard s's first
 *                      column in the full row (0 <= offset < 2^31); global
 *                      index = offset + local index.  Shards are meant to be
 *                      disjoint column blocks.
 *   k                  1..TF_TOPK_MAX_K; outputs as for tf_topk_bf16.
 * The result is the top k of the union of the input entries under (score
 * descending, lower global index first); its count is min(k, entries read);
 * its mask is the OR of the shards' masks.  When every shard list holds its
 * block's top k_in >= k, the result equals tf_topk_bf16 on the whole row.
 * Asynchronous on `stream`; allocates nothing.  Returns a TF_TOPK_* status
 * (ERR_SHAPE for a bad row/shard count or offset, ERR_K for k or k_in out of
 * range, ERR_NULL, ERR_ALIGN as for tf_topk_bf16).
 */
int tf_topk_merge_bf16(const int32_t *in_idx, const uint16_t *in_val, const int32_t *in_count,
                       const uint32_t *in_nonfinite_mask, int64_t rows, int32_t shards, int32_t k_in,
                       const int64_t *shard_offset, int32_t k, int32_t *out_idx, uint16_t *out_val,
                       int32_t *out_count, uint32_t *out_nonfinite_mask, void *stream);

/*
 * Allocation-free variant of the stream plan.
 *
 * The paper has no counterpart: this entry point exists for callers that must
 * not allocate device memory once they are running -- serving engines that
 * reserve nearly all of HBM for their caches up front (a late cudaMalloc can
 * fail there), and hosts of custom operators that hand a kernel only the
 * buffers they own.  The stream plan of tf_topk_bf16_with_plan allocates its
 * per-stream scratch on the first call on each stream (and frees and regrows
 * it if a later call needs more); this call never allocates or frees anything.
 *
 * Same arguments, same results as tf_topk_bf16 (always the stream plan).  Its
 * scratch is one static device array built into the library: room for
 * TF_TOPK_NOALLOC_MAX_CTAS CTAs, two k-entry lists and a ticket each
 * (534,528 bytes), held by every GPU that loads the library until the process
 * exits.  A call needs one slot per CTA of its launch, at most twice the SM
 * count of the device (304 on a 152-SM GB300); a call that would need more
 * returns TF_TOPK_ERR_SCRATCH and launches nothing.
 *
 * The first call on each device looks up that device's address of the array
 * (a host-side lookup, no allocation); make that first call before any stream
 * capture begins.  Every call clears the tickets it uses (an asynchronous
 * memset on `stream`) before its launch.  All calls share the one array:
 * calls whose work overlaps on the GPU -- on different streams, or from
 * different host threads without ordering -- race and give wrong results.
 * Order them on one stream, or use tf_topk_bf16_with_plan, whose stream-plan
 * scratch is per stream.
 */
#define TF_TOPK_NOALLOC_MAX_CTAS 512
#define TF_TOPK_ERR_SCRATCH 8 /* tf_topk_bf16_noalloc: the launch would need more
                                 than TF_TOPK_NOALLOC_MAX_CTAS scratch slots */
int tf_topk_bf16_noalloc(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                         int32_t *out_idx, uint16_t *out_val, int32_t *out_count,
                         uint32_t *out_nonfinite_mask, void *stream);

/*
 * Sampling probabilities over each row's top-k list (nucleus / top-p).
 *
 * The speculative decoding receipts of the TensorFold PR #3069 page
 * ("Receipt") sample draft streams at temperature 0.7 with top-k 20 and top-p
 * 0.95.  The page names those settings, not the procedure; this call takes
 * the usual one, top-k first and then top-p:
 *   - the entries of row r are the first min(k, count[r]) of its list, cut
 *     before the first NaN value (the top-k ranks NaN below every number);
 *   - with T > 0 their probabilities are the softmax of value / T over those
 *     entries alone (computed in fp32, relative to the best value); T == 0
 *     is greedy (the first entry alone); an infinite best value gives the
 *     entries equal to it equal shares;
 *   - keep[r] is the length of the shortest best-first prefix whose mass
 *     reaches top_p (every entry when top_p == 1), and out_prob holds that
 *     prefix renormalised to sum 1, then zeros.
 *
 *   val, count         device: val[r * k + i] bf16 bits and count[r], exactly
 *                      as tf_topk_bf16 (or tf_topk_merge_bf16) writes them.
 *   rows, k            rows >= 0; k 1..TF_TOPK_MAX_K (the lists' length).
 *   temperature        finite, >= 0.
 *   top_p              0 < top_p <= 1.
 *   out_prob           device float [rows][k], row-major.
 *   out_keep           device int32 [rows]; 0 for a row with no number.
 * Asynchronous on `stream`; allocates nothing; launched as a programmatic
 * dependent of the call before it on the stream, so queued right after
 * tf_topk_bf16 it starts as that call's last CTAs finish.  Returns a
 * TF_TOPK_* status (ERR_ARG for temperature or top_p, ERR_K, ERR_SHAPE for
 * rows < 0, ERR_NULL, ERR_ALIGN: val 2-byte, the others 4-byte aligned).
 */
#define TF_TOPK_ERR_ARG 9 /* tf_topk_nucleus_bf16: temperature or top_p out of range */
int tf_topk_nucleus_bf16(const uint16_t *val, const int32_t *count, int64_t rows, int32_t k, float temperature,
                         float top_p, float *out_prob, int32_t *out_keep, void *stream);

/*
 * Top-k of bf16, fp16 or fp32 rows, k up to TF_TOPK_MAX_K_WIDE.
 *
 * The operation of tf_topk_bf16 (TensorFold PR #713, change 3: score
 * descending, the lower column first; the "Exactness" table's count and
 * non-finite mask) on two more logit formats and for larger k.  The pages
 * state it for bf16 with a max_k constant; the same order and readings hold
 * here: NaN is never selected, +0 and -0 tie, infinities are ordinary
 * extreme scores, subnormals are exact, and empty slots hold index -1 and the
 * format's quiet NaN (bf16 0x7FC0, fp16 0x7E00, fp32 0x7FC00000).
 *
 *   logits       device, rows x row_stride elements of `dtype`
 *                (TF_TOPK_DTYPE_*), aligned to the element size; columns
 *                [cols, row_stride) are never read.
 *   k            1..TF_TOPK_MAX_K_WIDE; k > cols is allowed.
 *   out_idx      device int32 [rows][k]; out_val device [rows][k] elements of
 *                `dtype` (the original bits); out_count int32 [rows];
 *                out_nonfinite_mask uint32 [rows] (1 NaN, 2 +inf, 4 -inf).
 * bf16 with k <= TF_TOPK_MAX_K runs the plans of tf_topk_bf16 (the same
 * results, byte for byte).  fp16 with k <= TF_TOPK_MAX_K runs the cluster
 * kernel's plans, SINGLE and CLUSTER2..16 (it shares bf16's order-preserving
 * key map; only its special values differ).  fp32 with k <=
 * TF_TOPK_MAX_K on AUTO runs the fp32 cluster kernel: each row's column spans
 * over a thread-block cluster, read once against a running bound, on 32-bit
 * keys.  Everything else (and TF_TOPK_PLAN_WIDE) runs the wide kernel: one
 * CTA per row, two passes over the row (a bound from each thread's largest
 * vector maxima, then every element reaching it, read back through a table of
 * the maxima and ranked or sorted), with an exact counting search when ties
 * crowd the bound.  Asynchronous on `stream`; allocates nothing.
 * Returns a TF_TOPK_* status: ERR_DTYPE for an unknown format, ERR_K,
 * ERR_SHAPE, ERR_NULL, ERR_ALIGN as for tf_topk_bf16.
 */
#define TF_TOPK_MAX_K_WIDE 1024
#define TF_TOPK_DTYPE_BF16 0
#define TF_TOPK_DTYPE_F16 1
#define TF_TOPK_DTYPE_F32 2
#define TF_TOPK_PLAN_WIDE 64 /* tf_topk_select_with_plan: the wide kernel for any format and k */
#define TF_TOPK_ERR_DTYPE 10 /* tf_topk_select: unknown logit format */
int tf_topk_select(const void *logits, int32_t dtype, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                   int32_t *out_idx, void *out_val, int32_t *out_count, uint32_t *out_nonfinite_mask, void *stream);

/* tf_topk_select with a plan: TF_TOPK_PLAN_AUTO, TF_TOPK_PLAN_WIDE, or, with
 * k <= TF_TOPK_MAX_K, a plan of tf_topk_bf16_with_plan (bf16) or SINGLE and
 * the cluster plans CLUSTER2..16 (fp16); anything else returns
 * TF_TOPK_ERR_PLAN. */
int tf_topk_select_with_plan(const void *logits, int32_t dtype, int64_t rows, int64_t cols, int64_t row_stride,
                             int32_t k, int32_t *out_idx, void *out_val, int32_t *out_count,
                             uint32_t *out_nonfinite_mask, int32_t plan, void *stream);
int32_t tf_topk_select_max_k(void); /* == TF_TOPK_MAX_K_WIDE */

/*
 * tf_topk_nucleus_bf16 for lists of any format tf_topk_select writes: `val`
 * holds [rows][k] elements of `dtype` (TF_TOPK_DTYPE_*; bf16 and fp16 2-byte
 * aligned, fp32 4-byte aligned), decoded exactly to float.  Everything else as
 * tf_topk_nucleus_bf16 (k <= TF_TOPK_MAX_K).  Returns TF_TOPK_ERR_DTYPE for an
 * unknown format, otherwise the statuses of tf_topk_nucleus_bf16.
 */
int tf_topk_nucleus(const void *val, int32_t dtype, const int32_t *count, int64_t rows, int32_t k, float temperature,
                    float top_p, float *out_prob, int32_t *out_keep, void *stream);

/*
 * Draft head with the top-k in its epilogue (producer fusion).
 *
 * The operation is the one the top-k of TensorFold PR #713, change 3, is fed
 * by: the drafter's head turns each draft position's hidden state into a row
 * of bf16 logits (15 rows x 98592 columns there), and the top-k takes the
 * best entries of each row.  The pages give the logits' shape and format
 * only; the head is read here as the usual LM head, a matrix product with a
 * [vocab][dim] weight, accumulated in fp32 and rounded to bf16 (round to
 * nearest even).  This call computes that product and selects each row's
 * top k from the rounded logits in the same kernel, so the logits never
 * reach device memory:
 *   logit[r][v] = bf16_rne( sum over d of hidden[r][d] * weight[v][d] )   (fp32 sum)
 * and then exactly what tf_topk_bf16 gives for a [rows][vocab] logit matrix
 * (same order, count, mask and empty slots).  The fp32 sum runs in the
 * tensor cores' order: the result is bit-exact against any other
 * implementation of the formula whenever that sum is exact in fp32 (as for
 * small-integer products); otherwise the selection is exact over this
 * kernel's own rounded logits.
 *
 *   hidden      device, bf16 [rows][dim], row stride dim; 16-byte aligned.
 *   weight      device, bf16 [vocab][dim], row stride dim; 16-byte aligned.
 *   rows        1..TF_TOPK_HEAD_MAX_ROWS (the draft window).
 *   dim         >= 8, a multiple of 8 (16-byte rows).
 *   vocab       1..2^31 - 64 columns of the logit rows.
 *   k           1..TF_TOPK_MAX_K.
 *   workspace   device, at least tf_topk_head_bf16_workspace(rows, k) bytes,
 *               8-byte aligned, owned by the caller; its contents on entry do
 *               not matter.  Calls that overlap on the GPU must not share it.
 *               A call leaves its ticket words cleared, so a call captured in
 *               a CUDA graph may be replayed on the same workspace.
 *   outputs     as for tf_topk_bf16 with cols = vocab.
 * Asynchronous on `stream`; allocates nothing.  Returns a TF_TOPK_* status:
 * ERR_SHAPE, ERR_K, ERR_NULL, ERR_ALIGN, ERR_SCRATCH (workspace too small),
 * ERR_DEVICE or ERR_CUDA.
 */
#define TF_TOPK_HEAD_MAX_ROWS 16
int tf_topk_head_bf16(const void *hidden, const void *weight, int32_t rows, int32_t dim, int64_t vocab, int32_t k,
                      void *workspace, size_t workspace_bytes, int32_t *out_idx, uint16_t *out_val,
                      int32_t *out_count, uint32_t *out_nonfinite_mask, void *stream);

/* Workspace bytes tf_topk_head_bf16 needs for (rows, k) on the current device
 * (per CTA of its grid: for each row a k-entry list with a header word, a
 * split ticket, and the fp32 partial sums of two tiles that a CTA may share
 * with a neighbour); 0 for invalid arguments. */
size_t tf_topk_head_bf16_workspace(int32_t rows, int32_t k);

/* Human-readable text for a TF_TOPK_* status (static storage). */
const char *tf_topk_strerror(int status);

/* cudaError_t value behind the calling thread's last TF_TOPK_ERR_CUDA (0 if none). */
int tf_topk_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TF_TOPK_H */
