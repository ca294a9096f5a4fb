// Exact per-row top-k over wide bf16 logit rows for GB300 (sm_103a).
//
// What is computed: TensorFold PR #713, "perf(qwen27): a drafted round overlaps
// its cache commit with the next draft, and the drafter's attention and top-k
// use more of the GPU" -- change 3 (every row's best k entries, score
// descending, lower token index first; wide rows scanned in column spans whose
// results are merged in the same order) and the "Exactness" table (entries,
// count and non-finite mask per row; ties, both zeros, NaN, infinities, padded
// strides).  The conventions the pages leave open are stated in
// include/tf_topk.h.
//
// Common machinery of the two bf16 / fp16 kernels (for k <= 64):
//   * A CTA processes a row a chunk at a time: kThreads x kVecPerThread
//     16-byte vectors (16384 columns), held in registers as order-preserving
//     16-bit keys, two per register: positive bits b -> b | 0x8000, negative
//     bits b -> ~b.  -0 and +0 land on the neighbouring keys 0x7FFF / 0x8000 and
//     are treated as one score wherever a threshold or a comparison is taken.
//     The key map is the same for fp16; only the special values differ
//     (Fmt16<format>).
//   * Prefilter: every thread keeps the max key of its elements; each warp finds
//     the j-th largest of its 32 thread maxima (j = ceil(k / warps)); the
//     minimum T over warps is reached by at least k elements, so the chunk's
//     top-k lies in {key >= T}.  Once a running list holds k entries, its k-th
//     key is the bound instead.  Only candidates touch shared memory.
//   * Candidates are ranked exactly with a unique 32-bit composite
//     (key << 16 | ~chunk-local column).  Chunks with heavy ties (e.g. an
//     all-zero row) overflow the candidate buffer and take an exact path: a
//     binary search for the k-th key, then the lowest columns among the ties at
//     that key, ranked by a block scan in column order.
//   * A running list (<= k entries, 64-bit: key | ~column | original bits)
//     absorbs the chunks of a row piece; pieces are merged (the pages'
//     tournament) in the same order.
//
// topk_cluster_kernel<S, format> (the plans tf_topk_bf16 picks): S CTAs of a
// thread-block cluster split one row into S spans, load with 16-byte register
// loads, and merge through distributed shared memory in the leader CTA.  Each
// chunk's loads are issued as soon as the previous chunk's candidates are
// spilled, and candidates are ranked and merged into the running list in one
// phase.
//
// topk_stream_kernel (plans SINGLE and STREAM): a persistent grid of
// kStreamCtasPerSm CTAs per SM.  The rows x vectors space is cut into equal
// contiguous ranges, one per CTA.  Each CTA streams its range through a
// kStages-deep shared-memory ring filled by TMA bulk copies (cp.async.bulk +
// mbarrier).  A row cut by a range boundary leaves one partial list per piece
// in a small scratch area; the last CTA to finish a piece of that row (an
// atomic ticket) merges them and writes the row.  With one range per row the
// same kernel is the single-CTA control path.
//
// Also here: topk_merge_kernel (per-shard lists into each row's top k),
// topk_nucleus_kernel (top-p probabilities over the lists) and
// topk_wide_kernel (bf16 / fp16 / fp32 rows, k up to 1024: a bound from each
// thread's best keys, then every element reaching it, ranked).
//
// No wait is unbounded: mbarrier waits give up after kWaitLimit polls, record
// a fault code in a device word, drain their own copies (again bounded) and
// return.  Nothing waits on another CTA: cross-CTA hand-off is the hardware
// cluster barrier or the last-arriver ticket.

#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cmath>

#include <map>
#include <mutex>
#include <thread>

#include <type_traits>
#include <utility>

#include "tf_topk.h"

// Scratch of tf_topk_bf16_noalloc, for callers that may not allocate: per CTA
// slot two partial lists of (TF_TOPK_MAX_K + 1) 64-bit words, then one 32-bit
// ticket per slot.  Host code reaches it only through the address
// cudaGetSymbolAddress returns for the current device.
constexpr size_t kNoAllocListWords = (size_t)TF_TOPK_NOALLOC_MAX_CTAS * 2 * (TF_TOPK_MAX_K + 1);
constexpr size_t kNoAllocWords = kNoAllocListWords + TF_TOPK_NOALLOC_MAX_CTAS / 2;
static_assert(TF_TOPK_NOALLOC_MAX_CTAS % 2 == 0, "tickets fill whole 64-bit words");
static_assert(kNoAllocListWords * 8 % 256 == 0, "the ticket block starts 256-byte aligned");
static __device__ __align__(256) uint64_t g_noalloc_scratch[kNoAllocWords];

namespace cg = cooperative_groups;

// fp32 rows with k <= TF_TOPK_MAX_K on the fp32 cluster kernel (tf_topk_f32.cu).
int tf_topk_internal_select_f32(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                                int32_t *out_idx, void *out_val, int32_t *out_count, uint32_t *out_mask,
                                int sm_count, void *stream);

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerThread = 8;                     // 16-byte vectors per thread per chunk
constexpr int kChunkVecs = kThreads * kVecPerThread; // 2048 vectors
constexpr int kChunkCols = kChunkVecs * 8;           // 16384 columns
constexpr int kMaxK = TF_TOPK_MAX_K;
constexpr int kMaxSpans = TF_TOPK_MAX_SPANS;
constexpr int kCandCap = 256;        // candidates ranked directly (one per thread)
constexpr int kStages = 3;           // TMA ring depth of the stream kernel
constexpr int kStreamCtasPerSm = 2;  // resident stream CTAs per SM
constexpr int kClusterCtasPerSm = 4; // resident cluster-kernel CTAs per SM (its launch bounds)
constexpr int kMinVecsPerCta = 1024; // smallest range a stream CTA is given
constexpr int kMaxPieces = kMaxSpans;// most pieces a stream row is cut into
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kPendCap = 512;        // stream kernel: candidates waiting for a merge
constexpr int kMergeAt = 64;         // merge the waiting candidates once this many

// The constant ties the pages ask for: a change to one of these fails the build.
static_assert(kThreads % 32 == 0 && kThreads >= 64, "whole warps");
static_assert(kChunkCols <= 65536, "chunk-local column must fit the 16-bit composite field");
static_assert(kCandCap <= kThreads, "rank pass gives each candidate its own thread");
static_assert(kMaxK <= kCandCap, "exact path writes k candidates");
static_assert((kMaxK + kWarps - 1) / kWarps <= 32, "per-warp order statistic needs j <= 32");
static_assert(kMaxSpans == 16 && (kMaxSpans & (kMaxSpans - 1)) == 0, "merge tree over 2^n lists");
static_assert(kMaxK == 64, "header and kernels agree on max_k");
static_assert(kStages >= 2, "a ring needs two stages");
static_assert(kMinVecsPerCta >= 4 * kThreads, "moved range starts stay strictly increasing");
static_assert(kVecPerThread * 4 == 32, "the candidate scan maps a lane to one word of a thread's slice");

// What the fast kernels need to know of a 16-bit format; the order-preserving
// key map (sign-magnitude flip) is the same for every IEEE 16-bit format.
// Keys above the +inf key or below the -inf key are NaN; empty output slots
// hold the format's quiet NaN.
template <int kFmt>
struct Fmt16;
template <>
struct Fmt16<TF_TOPK_DTYPE_BF16> {
    static constexpr uint32_t kKeyPosInf = 0xFF80, kKeyNegInf = 0x007F;
    static constexpr uint32_t kRawPosInf = 0x7F80, kRawNegInf = 0xFF80, kEmpty = 0x7FC0;
};
template <>
struct Fmt16<TF_TOPK_DTYPE_F16> {
    static constexpr uint32_t kKeyPosInf = 0xFC00, kKeyNegInf = 0x03FF;
    static constexpr uint32_t kRawPosInf = 0x7C00, kRawNegInf = 0xFC00, kEmpty = 0x7E00;
};
constexpr int kBf16 = TF_TOPK_DTYPE_BF16;

constexpr uint32_t kEmptyVal = Fmt16<kBf16>::kEmpty;
constexpr uint32_t kKeyNegZero = 0x7FFF;
constexpr uint32_t kKeyPosZero = 0x8000;

// Device fault word: 0, or the first fault code a kernel recorded.
constexpr uint32_t kFaultWaitTimeout = 1;
__device__ uint32_t g_fault;

struct __align__(16) SmemCore {
    uint32_t cand[kCandCap + 4];            // chunk candidates, 32-bit composites (+ zero pad)
    uint16_t cand_raw[kCandCap];            // their original bf16 bits
    uint64_t list[3][kMaxK];                // running list, chunk list, merge output
    uint32_t warp_t[kWarps];
    uint32_t red[2][kWarps];
    uint32_t scan[kWarps][4];
    uint64_t mbar[kStages];
    uint32_t n_cand;
    uint32_t npend;                         // stream kernel: entries waiting in pend
    uint32_t flags;
    uint32_t kmax;
    uint32_t ticket[2];                     // stream kernel: tickets of the split pieces
};

// The cluster leader's gather area: every span CTA pushes its list here.
struct __align__(16) SmemGather {
    uint64_t gather[kMaxSpans][kMaxK];      // lists being merged
    uint64_t gather2[kMaxSpans / 2][kMaxK]; // merge-tree ping-pong
    int32_t glen[kMaxSpans];
    int32_t glen2[kMaxSpans / 2];
    uint32_t gflags[kMaxSpans];
};

// ---------------------------------------------------------------- bit helpers

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t max_s16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t min_u16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two bf16 bit patterns -> two order-preserving keys: each 16-bit half is
// XORed with 0xFFFF when its sign bit is set, else with 0x8000.  The prmt
// selector 0xBB99 replicates the sign bit of bytes 1 and 3 over their halves.
__device__ __forceinline__ uint32_t keys_from_raw2(uint32_t x)
{
    uint32_t s;
    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(s) : "r"(x));
    return x ^ (s | 0x80008000u);
}

__device__ __forceinline__ uint32_t raw_from_key(uint32_t key)
{
    return key ^ ((key & 0x8000u) ? 0x8000u : 0xFFFFu);
}

// -0 and +0 are one score.
__device__ __forceinline__ uint32_t canon(uint32_t key)
{
    return key == kKeyNegZero ? kKeyPosZero : key;
}

// Smallest key a candidate may have so that every element whose score is >=
// the score of key t is kept: the -0 key sits just below +0.
__device__ __forceinline__ uint32_t key_floor(uint32_t t)
{
    return t == kKeyPosZero ? kKeyNegZero : t;
}

__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 64-bit list entry: canonical key (16) | ~column (32) | original bits (16).
// Ordering the integers orders (score desc, column asc); the low 16 bits never
// decide because (key, column) is unique.
__device__ __forceinline__ uint64_t entry_from_cand(uint32_t c32, uint32_t raw, int32_t col_base)
{
    const uint32_t key = c32 >> 16;
    const int32_t col = col_base + (int32_t)(0xFFFFu - (c32 & 0xFFFFu));
    return ((uint64_t)key << 48) | ((uint64_t)(~(uint32_t)col) << 16) | (uint64_t)raw;
}

__device__ __forceinline__ int32_t entry_col(uint64_t e)
{
    return (int32_t)(~(uint32_t)(e >> 16));
}

// The list entry of key `key` (order-preserving, not 0) at row column `col`.
__device__ __forceinline__ uint64_t list_entry(uint32_t key, int32_t col)
{
    return ((uint64_t)canon(key) << 48) | ((uint64_t)(~(uint32_t)col) << 16) | (uint64_t)raw_from_key(key);
}

// Number of entries of a descending list of distinct values that exceed x.
__device__ __forceinline__ int count_greater(const uint64_t *list, int len, uint64_t x)
{
    int lo = 0, hi = len;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (list[mid] > x)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

__device__ __forceinline__ uint32_t block_sum(uint32_t v, SmemCore &sm, int parity)
{
    v = __reduce_add_sync(0xFFFFFFFFu, v);
    if ((threadIdx.x & 31) == 0) sm.red[parity][threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += sm.red[parity][w];
    return s;
}

// A candidate at a given slot (chunk-relative); slots past the buffer are
// not written.
__device__ __forceinline__ void put_candidate(SmemCore &sm, uint32_t key, int local, uint32_t slot)
{
    if (slot < (uint32_t)kCandCap) {
        sm.cand[slot] = (canon(key) << 16) | (0xFFFFu - (uint32_t)local);
        sm.cand_raw[slot] = (uint16_t)raw_from_key(key);
    }
}

// The candidate counter only grows within a chunk loop: a chunk's slots count
// from `base`, the counter's value when the chunk began.  Returns the slot.
__device__ __forceinline__ uint32_t push_candidate(SmemCore &sm, uint32_t key, int local, uint32_t base)
{
    const uint32_t slot = atomicAdd(&sm.n_cand, 1u) - base;
    put_candidate(sm, key, local, slot);
    return slot;
}

// Keys of the staged chunk whose score is >= the score of key t (t >= 1), this
// thread's share.
__device__ __forceinline__ uint32_t count_at_least(const uint32_t *keys, uint32_t t)
{
    const uint32_t f = key_floor(t);
    uint32_t c = 0;
    for (int w = threadIdx.x; w < kChunkCols / 2; w += kThreads) {
        const uint32_t k2 = keys[w];
        c += (k2 & 0xFFFFu) >= f;
        c += (k2 >> 16) >= f;
    }
    return c;
}

// Exact selection for a chunk whose candidate set {key >= t_floor} is larger
// than the candidate buffer (heavy ties, e.g. an all-zero row).  The chunk's
// keys have been staged in `keys` in column order (0 = not a candidate).
// Writes the chunk's top-k within that set -- k candidates, or all of them
// when fewer reach t_floor -- into sm.cand, and their number into sm.n_cand.
// Block-uniform; every thread calls it.
template <int kFmt = kBf16>
__device__ __noinline__ void exact_select(const uint32_t *keys, uint32_t t_floor, int k, SmemCore &sm)
{
    const int tid = threadIdx.x;
    // 1. K* = the largest canonical key that at least k elements reach.
    uint32_t my_max = 0;
    for (int w = tid; w < kChunkCols / 2; w += kThreads)
        my_max = max(my_max, max(canon(keys[w] & 0xFFFFu), canon(keys[w] >> 16)));
    my_max = __reduce_max_sync(0xFFFFFFFFu, my_max);
    if (tid == 0) sm.kmax = 0;
    __syncthreads();
    if ((tid & 31) == 0) atomicMax(&sm.kmax, my_max);
    __syncthreads();
    uint32_t lo = canon(t_floor); // count(lo) > kCandCap >= k
    uint32_t hi = sm.kmax + 1;    // count(hi) == 0
    int parity = 0;
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        const uint32_t c = block_sum(count_at_least(keys, mid), sm, parity);
        parity ^= 1;
        if (c >= (uint32_t)k)
            lo = mid;
        else
            hi = mid;
    }
    const uint32_t kstar = lo;

    // 2. Each thread owns a contiguous run of columns (kWordsPerThread words,
    //    a word per lane per step: lane L starts L words into its run, so a
    //    step's 32 reads fall in 32 banks).  One exclusive scan of the
    //    per-thread counts -- keys above K* in the high half, ties at K* in
    //    the low half (at most a chunk of them: no carry into the high half)
    //    -- gives every entry its slot: the entries above K* first, then the
    //    lowest columns among the ties, as many as the k places left.
    constexpr int kWordsPerThread = kChunkCols / 2 / kThreads;
    static_assert(kWordsPerThread == 32, "one rotation step per lane");
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t *tk = keys + tid * kWordsPerThread;
    uint32_t mine = 0, pre = 0; // pre: ties in the run's first `lane` words
    for (int i = 0; i < kWordsPerThread; ++i) {
        const int w = (i + lane) & (kWordsPerThread - 1);
        const uint32_t k2 = tk[w];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t c = canon(h ? (k2 >> 16) : (k2 & 0xFFFFu)); // key 0 is never >= K* >= 1
            mine += c > kstar ? 0x10000u : (c == kstar ? 1u : 0u);
            pre += (c == kstar && w < lane) ? 1u : 0u;
        }
    }
    uint32_t incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += u;
    }
    if (lane == 31) sm.scan[warp][0] = incl;
    __syncthreads();
    uint32_t excl = incl - mine, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = sm.scan[w][0];
        excl += w < warp ? t : 0u;
        total += t;
    }
    const uint32_t above = total >> 16;                     // < k: K* is the k-th largest key
    const uint32_t need = (uint32_t)k - above;              // ties to take, lowest columns first
    const uint32_t taken = min(need, total & 0xFFFFu);      // fewer when fewer than k keys reach t_floor
    if (tid == 0) sm.n_cand = above + taken;

    // 3. Place them, in the same rotated order: the run's words from `lane`
    //    on hold the ties after its first `pre`, the words before it the
    //    first ones.
    uint32_t a_ord = excl >> 16, t_ord = (excl & 0xFFFFu) + pre;
    const bool places = (mine >> 16) != 0 || (excl & 0xFFFFu) < need; // else nothing of this run is taken
    for (int i = 0; i < (places ? kWordsPerThread : 0); ++i) {
        const int w = (i + lane) & (kWordsPerThread - 1);
        if (w == 0) t_ord = excl & 0xFFFFu;
        const uint32_t k2 = tk[w];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t key = h ? (k2 >> 16) : (k2 & 0xFFFFu);
            const uint32_t c = canon(key);
            if (c > kstar) {
                put_candidate(sm, key, 2 * (tid * kWordsPerThread + w) + h, a_ord++);
            } else if (c == kstar) {
                if (t_ord < need) put_candidate(sm, key, 2 * (tid * kWordsPerThread + w) + h, above + t_ord);
                ++t_ord;
            }
        }
    }
    __syncthreads();
}

// Where a chunk sits in its row.  Vector v covers row columns [8v - m, 8v - m + 8);
// vectors [vfull0, vfull1) lie wholly inside [0, cols).
struct ChunkGeom {
    const uint16_t *rowp;
    int32_t cols, m, vfull0, vfull1;
};

__device__ __forceinline__ ChunkGeom row_geometry(const uint16_t *rowp, int32_t cols)
{
    ChunkGeom g;
    g.rowp = rowp;
    g.cols = cols;
    g.m = (int32_t)((reinterpret_cast<uintptr_t>(rowp) >> 1) & 7);
    g.vfull0 = g.m ? 1 : 0;
    g.vfull1 = (cols + g.m) >> 3;
    return g;
}


// Element-wise load of an edge vector (a vector that straddles a row end):
// columns outside [0, cols) read as 0xFFFF, whose key is 0 (never selected).
__device__ __noinline__ uint4 load_edge_vector(const uint16_t *rowp, int32_t cols, int32_t m, int32_t v)
{
    uint32_t w4[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const int32_t c0 = v * 8 + 2 * w - m;
        const uint32_t lo = (c0 >= 0 && c0 < cols) ? rowp[c0] : 0xFFFFu;
        const uint32_t hi = (c0 + 1 >= 0 && c0 + 1 < cols) ? rowp[c0 + 1] : 0xFFFFu;
        w4[w] = lo | (hi << 16);
    }
    return make_uint4(w4[0], w4[1], w4[2], w4[3]);
}

// The exact key pass for one thread whose chunk slice holds a column outside
// the row (its keys may also hold non-finite values).  Its keys sit in its own stage slots
// (vector i at stage[i * kThreads + tid]); columns outside the row and NaNs
// become key 0 and the row's non-finite flags are recorded.  Returns the
// thread's max key over what remains.
template <int kFmt = kBf16>
__device__ __noinline__ uint32_t fix_keys(uint4 *stage, int32_t col_base, int32_t cols, int nvalid,
                                          SmemCore &sm)
{
    const int tid = threadIdx.x;
    uint32_t tmax = 0, flags = 0;
    for (int i = 0; i < kVecPerThread; ++i) {
        const int lv = i * kThreads + tid;
        if (lv >= nvalid) continue;
        uint4 q = stage[lv];
        uint32_t qw[4] = {q.x, q.y, q.z, q.w};
        for (int w = 0; w < 4; ++w) {
            uint32_t out = 0;
            for (int h = 0; h < 2; ++h) {
                const int32_t c = col_base + lv * 8 + 2 * w + h;
                uint32_t key = (qw[w] >> (16 * h)) & 0xFFFFu;
                if (c < 0 || c >= cols) {
                    key = 0;
                } else if (key > Fmt16<kFmt>::kKeyPosInf || key < Fmt16<kFmt>::kKeyNegInf) {
                    flags |= 1u; // NaN
                    key = 0;
                } else if (key == Fmt16<kFmt>::kKeyPosInf) {
                    flags |= 2u;
                } else if (key == Fmt16<kFmt>::kKeyNegInf) {
                    flags |= 4u;
                }
                tmax = max(tmax, key);
                out |= key << (16 * h);
            }
            qw[w] = out;
        }
        stage[lv] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    }
    if (flags) atomicOr(&sm.flags, flags);
    return tmax;
}

// Keys of one chunk.  kv holds the raw words of this thread's vectors (vector
// i is chunk vector cbeg + i * kThreads + tid; vectors past the chunk end are
// 0); on return it holds their keys (0 where no score may be selected), and
// the thread's max key is returned.  kFull: every vector of the chunk lies
// wholly inside the row (no predicates).
//
// A thread whose keys pass an infinity's (above +inf's, below -inf's) holds a
// NaN or a column outside the row.  Without the latter, its keys are fixed two at
// a time in registers: a half is a NaN when its magnitude bits exceed the
// infinity's (one add into the half's top bit: the sum stays below 2^16, so
// nothing carries into the other half), and an infinity when its key XOR the
// infinity's key is zero (the borrow test for a zero half; a borrow into the
// high half only happens when the low half is itself zero, so "some half is
// zero" stays exact).  A thread holding an edge vector -- columns outside the
// row, read as 0xFFFF -- takes the exact per-element pass through its own
// `stage` slots instead (at most the two vectors at a row's ends).
template <bool kFull, int kFmt = kBf16>
__device__ __forceinline__ uint32_t chunk_keys(uint32_t (&kv)[kVecPerThread][4], const ChunkGeom &geo, int32_t cbeg,
                                               int nvalid, uint4 *stage, SmemCore &sm)
{
    using F = Fmt16<kFmt>;
    const int tid = threadIdx.x;
    uint32_t mx = 0, mn = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
        if (kFull || i * kThreads + tid < nvalid) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t key = keys_from_raw2(kv[i][w]);
                kv[i][w] = key;
                mx = max_u16x2(mx, key);
                mn = min_u16x2(mn, key);
            }
        }
    }
    uint32_t tmax = max(mx & 0xFFFFu, mx >> 16);
    const uint32_t tmin = min(mn & 0xFFFFu, mn >> 16);
    // infinities without a NaN (a -inf mask, say): their keys are valid as
    // they are, only the flags are needed
    if (tmax <= F::kKeyPosInf && tmin >= F::kKeyNegInf) {
        const uint32_t f = (tmax == F::kKeyPosInf ? 2u : 0u) | (tmin == F::kKeyNegInf ? 4u : 0u);
        if (f) atomicOr(&sm.flags, f);
        return tmax;
    }

    bool edge = false;
    if (!kFull) {
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
            const int lv = i * kThreads + tid;
            const int32_t v = cbeg + lv;
            edge |= lv < nvalid && (v < geo.vfull0 || v >= geo.vfull1);
        }
    }
    if (!edge) {
        constexpr uint32_t kNanAdd = (0x8000u - (F::kRawPosInf + 1u)) * 0x00010001u;
        constexpr uint32_t kPosInf2 = F::kKeyPosInf * 0x00010001u, kNegInf2 = F::kKeyNegInf * 0x00010001u;
        uint32_t nan = 0, pinf = 0, ninf = 0;
        mx = 0;
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
            if (kFull || i * kThreads + tid < nvalid) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t key = kv[i][w];
                    uint32_t s;
                    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(s) : "r"(key)); // each half's top bit, spread
                    const uint32_t mag = (key ^ ~s) & 0x7FFF7FFFu;            // magnitude bits of the value
                    const uint32_t nb = (mag + kNanAdd) & 0x80008000u;         // a NaN half's top bit
                    const uint32_t xp = key ^ kPosInf2, xn = key ^ kNegInf2;
                    nan |= nb;
                    pinf |= (xp - 0x00010001u) & ~xp;
                    ninf |= (xn - 0x00010001u) & ~xn;
                    const uint32_t fixed = key & ~((nb >> 15) * 0xFFFFu);     // NaN -> key 0
                    kv[i][w] = fixed;
                    mx = max_u16x2(mx, fixed);
                }
            }
        }
        const uint32_t flags = (nan ? 1u : 0u) | ((pinf & 0x80008000u) ? 2u : 0u) | ((ninf & 0x80008000u) ? 4u : 0u);
        if (flags) atomicOr(&sm.flags, flags);
        return max(mx & 0xFFFFu, mx >> 16);
    }

    // ---- a row edge in this thread's vectors: the exact pass through shared memory
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i)
        stage[i * kThreads + tid] = make_uint4(kv[i][0], kv[i][1], kv[i][2], kv[i][3]);
    tmax = fix_keys<kFmt>(stage, cbeg * 8 - geo.m, geo.cols, nvalid, sm);
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
        const uint4 q = stage[i * kThreads + tid];
        kv[i][0] = q.x;
        kv[i][1] = q.y;
        kv[i][2] = q.z;
        kv[i][3] = q.w;
    }
    return tmax;
}

// Selection for one chunk whose keys are in kv (see chunk_keys) with this
// thread's max key tmax: the row piece's running list (run_i, run_len)
// absorbs the chunk's top-k.  Block-uniform: every thread calls it.
// Max key of this thread's raw bf16 words without turning them into keys.
// Signed 16-bit order is score order among non-negative values, so the signed
// max gives the best non-negative score (key = raw + 0x8000); the signed max
// also shows a +inf/+NaN (>= 0x7F80) and the unsigned max a -inf/-NaN
// (>= 0xFF80).  Returns false -- the keys are needed -- when the thread holds
// any of those or no non-negative value at all.
template <int kFmt = kBf16>
__device__ __forceinline__ bool raw_tmax(const uint32_t (&kv)[kVecPerThread][4], uint32_t &tmax)
{
    uint32_t smx = 0x80008000u, umx = 0;
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            smx = max_s16x2(smx, kv[i][w]);
            umx = max_u16x2(umx, kv[i][w]);
        }
    const int32_t smax = max((int32_t)(int16_t)(smx & 0xFFFFu), (int32_t)(int16_t)(smx >> 16));
    const uint32_t umax = max(umx & 0xFFFFu, umx >> 16);
    if (smax < 0 || smax >= (int32_t)Fmt16<kFmt>::kRawPosInf || umax >= Fmt16<kFmt>::kRawNegInf) return false;
    tmax = (uint32_t)smax + 0x8000u;
    return true;
}

__device__ __forceinline__ void keys_in_place(uint32_t (&kv)[kVecPerThread][4])
{
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i)
#pragma unroll
        for (int w = 0; w < 4; ++w) kv[i][w] = keys_from_raw2(kv[i][w]);
}

// Prefilter bound of one chunk (block-uniform, one barrier).  The fw warps
// whose 32 lanes all hold data each find the j-th largest of their lanes'
// maxima, j = ceil(k / fw); the minimum t0 over them is reached by at least
// fw * j >= k elements of the chunk, so no element below t0 can be in the
// top k of anything that contains the chunk.  With no such bound (a tiny
// chunk, or a warp without j positive maxima) the result is 0.
__device__ __forceinline__ uint32_t prefilter_bound(uint32_t tmax, int nvalid, int k, SmemCore &sm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int fw = min(nvalid, kThreads) / 32;
    const int j = fw ? (k + fw - 1) / fw : 33;
    uint32_t tw = 0xFFFFu; // warps without a full set of lanes do not bound
    if (warp < fw) {
        tw = 0;
        if (j <= 32) {
            uint32_t v = tmax, cnt = 0;
            for (int it = 0; it < j; ++it) {
                const uint32_t mval = __reduce_max_sync(0xFFFFFFFFu, v);
                if (mval == 0) break;
                cnt += __popc(__ballot_sync(0xFFFFFFFFu, v == mval));
                if (cnt >= (uint32_t)j) {
                    tw = mval;
                    break;
                }
                if (v == mval) v = 0;
            }
        }
    }
    if (lane == 0) sm.warp_t[warp] = tw;
    __syncthreads();
    uint32_t t0 = (fw == 0 || j > 32) ? 0u : 0xFFFFu;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t0 = min(t0, sm.warp_t[w]);
    return t0;
}

__device__ __forceinline__ uint32_t chunk_floor(uint32_t tmax, int nvalid, int k, SmemCore &sm, int run_i,
                                                int run_len)
{
    if (run_len == k) {
        // steady state: a new entry must beat the running k-th strictly (every
        // column of this chunk is higher), and that bound needs no barrier
        return (uint32_t)(sm.list[run_i][k - 1] >> 48) + 1u;
    }
    return max(key_floor(prefilter_bound(tmax, nvalid, k, sm)), 1u);
}

// Threads whose max reaches t_floor hold the chunk's candidates: each such
// thread spills its keys into its own slots of `stage` (vector i at
// stage[i * kThreads + tid]).  After this the chunk's registers are not read.
__device__ __forceinline__ bool spill_hits(uint32_t (&kv)[kVecPerThread][4], uint32_t tmax, bool raw,
                                           uint32_t t_floor, uint4 *stage)
{
    const bool hit = tmax >= t_floor;
    if (hit) {
        if (raw) keys_in_place(kv);
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i)
            stage[i * kThreads + threadIdx.x] = make_uint4(kv[i][0], kv[i][1], kv[i][2], kv[i][3]);
    }
    return hit;
}

// The chunk's candidates (keys >= t_floor) into sm.cand from the spilled
// slots of the hit threads: each hit thread's warp scans its keys one word
// per lane.  Returns their number n once every thread has pushed (a barrier);
// above kCandCap (heavy ties) the chunk is selected exactly from the spilled
// keys, and n = k.  `base` (block-uniform) is the candidate counter's value before the
// chunk and after it.  Block-uniform.
template <int kFmt = kBf16>
__device__ __forceinline__ uint32_t push_candidates(bool hit, uint32_t t_floor, int k, SmemCore &sm, uint4 *stage,
                                                    uint32_t &base)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __syncwarp();
    const uint32_t hits0 = __ballot_sync(0xFFFFFFFFu, hit);
    const bool crowded = __popc(hits0) >= 8; // only then can this warp alone fill the buffer
    for (uint32_t hits = hits0; hits; hits &= hits - 1) {
        const int src = warp * 32 + __ffs(hits) - 1;
        const int lv = (lane >> 2) * kThreads + src;
        const uint32_t key2 = reinterpret_cast<const uint32_t *>(stage)[lv * 4 + (lane & 3)];
        const int local = lv * 8 + 2 * (lane & 3);
        uint32_t top = 0;
        if ((key2 & 0xFFFFu) >= t_floor) top = push_candidate(sm, key2 & 0xFFFFu, local, base) + 1u;
        if ((key2 >> 16) >= t_floor) top = push_candidate(sm, key2 >> 16, local + 1, base) + 1u;
        // past the buffer the chunk is selected exactly from the spilled keys:
        // pushing the rest (up to a whole chunk of ties) would only cost atomics
        if (crowded && __any_sync(0xFFFFFFFFu, top > (uint32_t)kCandCap)) break;
    }
    __syncthreads();
    const uint32_t total = sm.n_cand;
    uint32_t n = total - base;
    base = total;
    if (n > (uint32_t)kCandCap) {
        // every key that can matter (>= t_floor) was spilled by its thread, in
        // column order and exact (NaN, out-of-row and past-the-end columns are
        // key 0); the other threads' slots still hold an earlier chunk
        if (!hit) {
#pragma unroll
            for (int i = 0; i < kVecPerThread; ++i) stage[i * kThreads + tid] = make_uint4(0, 0, 0, 0);
        }
        __syncthreads();
        exact_select<kFmt>(reinterpret_cast<const uint32_t *>(stage), t_floor, k, sm); // counts from 0
        n = sm.n_cand; // == k
        base = n;
    }
    return n;
}

// Second half of a chunk's selection, once its n > 0 candidates are in
// sm.cand (the chunk's registers are no longer read): every candidate and
// every running entry finds its place in the merged list at once.  A
// candidate's place is its rank among the candidates plus the running entries
// above it; a running entry's is its index plus the candidates above it.  The
// merged list goes to list[free_i], which becomes the running list.  No
// barrier: the caller's next one orders this before the list is read.
__device__ __forceinline__ void merge_candidates(uint32_t n, int32_t col_base, int k, SmemCore &sm, int &run_i,
                                                 int &free_i, int &run_len)
{
    const int tid = threadIdx.x;
    const uint64_t *run = sm.list[run_i];
    uint64_t *out = sm.list[free_i];
    const int rl = run_len;
    if (tid < (int)n) {
        // rank = number of larger composites
        const uint32_t e = sm.cand[tid];
        uint32_t rank = 0;
        const uint4 *c4 = reinterpret_cast<const uint4 *>(sm.cand);
        const uint32_t nq = n >> 2;
        for (uint32_t u = 0; u < nq; ++u) {
            const uint4 q = c4[u];
            rank += (q.x > e) + (q.y > e) + (q.z > e) + (q.w > e);
        }
        for (uint32_t u = nq * 4; u < n; ++u) rank += sm.cand[u] > e;
        if (rank < (uint32_t)k) {
            const uint64_t x = entry_from_cand(e, sm.cand_raw[tid], col_base);
            const int pos = (int)rank + count_greater(run, rl, x);
            if (pos < k) out[pos] = x;
        }
    }
    const int j = kThreads - 1 - tid; // running entries on the highest threads
    if (j < rl) {
        const uint64_t x = run[j];
        const uint64_t xs = x >> 16; // (key, ~column): the original bits never decide
        int above = 0;
        for (uint32_t u = 0; u < n; ++u) {
            const uint32_t c = sm.cand[u];
            const uint32_t col = (uint32_t)(col_base + (int32_t)(0xFFFFu - (c & 0xFFFFu)));
            above += ((((uint64_t)(c >> 16)) << 32) | (uint64_t)(~col)) > xs;
        }
        if (j + above < k) out[j + above] = x;
    }
    const int t = run_i;
    run_i = free_i;
    free_i = t;
    run_len = min(k, rl + (int)min(n, (uint32_t)k));
}


// Stream kernel, steady state: the running list (list[run_i], run_len
// entries, descending) absorbs the np pending entries pend[0..np) (distinct,
// any order) into list[out_i]; the indices swap and the pending count is
// cleared.  A rank merge: an entry's place is the number of larger pending
// entries plus the number of larger running entries.  Block-uniform.
// Push this chunk's keys that reach t_floor into the pending buffer as list
// entries.  Threads whose max reaches t_floor spill their keys into their own
// slots of `stage` (vector i at stage[i * kThreads + tid]); their warp scans
// them one word per lane, two spilled threads per step, and one atomic per
// step reserves the step's slots.  Entries past kPendCap are dropped (the
// count still grows, so the caller sees the overflow).  No block barrier.
__device__ __forceinline__ void push_pending(const uint32_t (&kv)[kVecPerThread][4], uint32_t tmax,
                                             uint32_t t_floor, int32_t col_base, uint4 *stage,
                                             SmemCore &sm, uint64_t *pend)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool hit = tmax >= t_floor;
    if (hit) {
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i)
            stage[i * kThreads + tid] = make_uint4(kv[i][0], kv[i][1], kv[i][2], kv[i][3]);
    }
    __syncwarp();
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t *words = reinterpret_cast<const uint32_t *>(stage);
    for (uint32_t hits = __ballot_sync(0xFFFFFFFFu, hit); hits;) {
        const int sa = __ffs(hits) - 1;
        hits &= hits - 1;
        const int sb = hits ? __ffs(hits) - 1 : -1;
        if (hits) hits &= hits - 1;
        const int lva = (lane >> 2) * kThreads + warp * 32 + sa;
        const int lvb = (lane >> 2) * kThreads + warp * 32 + (sb < 0 ? sa : sb);
        const uint32_t ka = words[lva * 4 + (lane & 3)];
        const uint32_t kb = sb < 0 ? 0u : words[lvb * 4 + (lane & 3)];
        const uint32_t e[4] = {ka & 0xFFFFu, ka >> 16, kb & 0xFFFFu, kb >> 16};
        uint32_t m[4], n = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            m[q] = __ballot_sync(0xFFFFFFFFu, e[q] >= t_floor);
            n += __popc(m[q]);
        }
        uint32_t base = 0;
        if (lane == 0 && n) base = atomicAdd(&sm.npend, n);
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (e[q] >= t_floor) {
                const uint32_t slot = base + __popc(m[q] & lt);
                const int32_t col = col_base + (q < 2 ? lva : lvb) * 8 + 2 * (lane & 3) + (q & 1);
                if (slot < (uint32_t)kPendCap) pend[slot] = list_entry(e[q], col);
            }
            base += __popc(m[q]);
        }
    }
}

__device__ __noinline__ void merge_pending(SmemCore &sm, const uint64_t *pend, int np, int k, int &run_i,
                                           int &out_i, int &run_len)
{
    const int tid = threadIdx.x;
    const uint64_t *run = sm.list[run_i];
    uint64_t *out = sm.list[out_i];
    const int total = np + run_len;
    // 2^sh threads (adjacent lanes) count for one entry, each over every 2^sh-th
    // element; a butterfly adds their counts
    const int sh = total <= kThreads / 4 ? 2 : (total <= kThreads / 2 ? 1 : 0);
    const int sub = tid & ((1 << sh) - 1);
    for (int t0 = 0; t0 < total; t0 += kThreads >> sh) {
        const int t = t0 + (tid >> sh);
        const bool valid = t < total;
        uint64_t x = 0;
        uint32_t g = 0;
        if (valid) {
            x = t < np ? pend[t] : run[t - np];
            const int step = 1 << sh;
            uint32_t g1 = 0, g2 = 0, g3 = 0;
            int u = sub;
            for (; u + 3 * step < np; u += 4 * step) {
                g += pend[u] > x;
                g1 += pend[u + step] > x;
                g2 += pend[u + 2 * step] > x;
                g3 += pend[u + 3 * step] > x;
            }
            for (; u < np; u += step) g += pend[u] > x;
            if (t < np) {
                for (u = sub; u + step < run_len; u += 2 * step) {
                    g1 += run[u] > x;
                    g2 += run[u + step] > x;
                }
                if (u < run_len) g3 += run[u] > x;
            }
            g += g1 + g2 + g3;
        }
        if (sh >= 1) g += __shfl_xor_sync(0xFFFFFFFFu, g, 1);
        if (sh >= 2) g += __shfl_xor_sync(0xFFFFFFFFu, g, 2);
        if (valid && sub == 0) {
            const int pos = (int)g + (t < np ? 0 : t - np);
            if (pos < k) out[pos] = x;
        }
    }
    __syncthreads();
    if (tid == 0) sm.npend = 0;
    const int t = run_i;
    run_i = out_i;
    out_i = t;
    run_len = min(k, run_len + np);
    __syncthreads();
}

// Stream kernel: a chunk whose candidates overflowed the pending buffer.  Its
// stage is not refilled yet, but only partly holds keys, so the chunk is read
// again from global memory (rare: heavy ties) and its keys staged in column
// order, 0 where nothing may be selected; then its best k over the keys that
// reach t_floor are selected exactly and put into pend[np_before ..
// np_before + k).  Returns the new pending count.  Block-uniform.
__device__ __noinline__ int lazy_overflow(SmemCore &sm, uint64_t *pend, uint4 *stage, uint32_t t_floor,
                                          ChunkGeom geo, int32_t cb, int nvalid, int np_before, int k)
{
    const int tid = threadIdx.x;
    const int32_t col_base = cb * 8 - geo.m;
    const uint4 *rowv = reinterpret_cast<const uint4 *>(geo.rowp - geo.m);
    uint32_t kv[kVecPerThread][4];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
        const int lv = i * kThreads + tid;
        uint4 q = make_uint4(0, 0, 0, 0);
        if (lv < nvalid) {
            const int32_t v = cb + lv;
            q = (v >= geo.vfull0 && v < geo.vfull1) ? ld_stream(rowv + v)
                                                   : load_edge_vector(geo.rowp, geo.cols, geo.m, v);
        }
        kv[i][0] = q.x;
        kv[i][1] = q.y;
        kv[i][2] = q.z;
        kv[i][3] = q.w;
    }
    chunk_keys<false>(kv, geo, cb, nvalid, stage, sm);
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = kv[i][j] & 0xFFFFu, hi = kv[i][j] >> 16;
            w[j] = (lo >= t_floor ? lo : 0u) | ((hi >= t_floor ? hi : 0u) << 16);
        }
        stage[i * kThreads + tid] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    exact_select(reinterpret_cast<const uint32_t *>(stage), t_floor, k, sm);
    const int n = (int)sm.n_cand; // == k
    for (int t = tid; t < n; t += kThreads)
        pend[np_before + t] = entry_from_cand(sm.cand[t], sm.cand_raw[t], col_base);
    __syncthreads();
    return np_before + n;
}

// Merge sm.gather[0..nl) (nl a power of two, lengths in sm.glen) pairwise into
// one list; returns it (in sm.gather or sm.gather2) and its length.
__device__ __forceinline__ const uint64_t *merge_tree(SmemGather &sm, int nl, int k, int &out_len)
{
    const int tid = threadIdx.x;
    uint64_t(*src)[kMaxK] = sm.gather;
    uint64_t(*dst)[kMaxK] = sm.gather2;
    int32_t *src_len = sm.glen;
    int32_t *dst_len = sm.glen2;
    for (; nl > 1; nl >>= 1) {
        for (int t = tid; t < nl * kMaxK; t += kThreads) {
            const int l = t / kMaxK, pos = t % kMaxK;
            if (pos >= src_len[l]) continue;
            const uint64_t x = src[l][pos];
            const int p = l ^ 1;
            const int out = pos + count_greater(src[p], src_len[p], x);
            if (out < k) dst[l >> 1][out] = x;
        }
        if (tid < nl / 2) dst_len[tid] = min(k, src_len[2 * tid] + src_len[2 * tid + 1]);
        __syncthreads();
        uint64_t(*tl)[kMaxK] = src;
        src = dst;
        dst = tl;
        int32_t *tlen = src_len;
        src_len = dst_len;
        dst_len = tlen;
    }
    out_len = src_len[0];
    return src[0];
}

template <int kFmt = kBf16>
__device__ __forceinline__ void write_row(int64_t row, const uint64_t *list, int len, uint32_t flags,
                                          int k, int32_t *out_idx, uint16_t *out_val,
                                          int32_t *out_count, uint32_t *out_mask)
{
    for (int t = threadIdx.x; t < k; t += kThreads) {
        const int64_t o = row * k + t;
        if (t < len) {
            const uint64_t e = list[t];
            out_idx[o] = entry_col(e);
            out_val[o] = (uint16_t)(e & 0xFFFFu);
        } else {
            out_idx[o] = -1;
            out_val[o] = (uint16_t)Fmt16<kFmt>::kEmpty;
        }
    }
    if (threadIdx.x == 0) {
        out_count[row] = len;
        out_mask[row] = flags;
    }
}

// ---------------------------------------------------------------- mbarrier / TMA

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_addr(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Bounded wait: true once the phase with this parity has completed, false
// after `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit = kWaitLimit)
{
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
                     "r"(smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// ---------------------------------------------------------------- stream kernel

// Programmatic dependent launch: the kernels are launched so that they may be
// scheduled while the previous kernel on the stream is still finishing.  Each
// waits here, before its first access to global memory, until that kernel has
// completed and its writes are visible (a no-op when there is nothing to wait
// for), then lets the next kernel on the stream be scheduled likewise.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The wait alone; a kernel using it lets its dependents be scheduled only
// once each of its CTAs reaches grid_dependents_go, near its end.
__device__ __forceinline__ void grid_dependency_wait_only()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dependents_go()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Stream-plan ranges.  CTA b nominally starts at vector b * per of the
// rows x vectors space; the start is moved to the nearest multiple of kThreads
// vectors from its row's start, or to the row's end when less than kThreads
// vectors would be left there.  So every piece of a row holds at least
// kThreads vectors (unless the whole row is shorter) and its first chunk
// always yields a prefilter bound.  Starts move by at most kThreads/2 back or
// 3*kThreads/2 forward, and per >= 4*kThreads, so they strictly increase up
// to `total`.
__device__ __forceinline__ int64_t range_start(int64_t b, int64_t per, int64_t total, int32_t nvr)
{
    const int64_t x = b * per;
    if (x >= total) return total;
    const int64_t r = x / nvr;
    const int32_t off = (int32_t)(x - r * nvr);
    int32_t cut = (off + kThreads / 2) / kThreads * kThreads;
    if (cut != 0 && nvr - cut < kThreads) cut = nvr;
    return min(total, r * nvr + cut);
}

// Take a ticket: an atomic increment with release semantics for the piece
// lists this CTA published before it (other threads' stores are ordered
// before it by the preceding barrier) and acquire semantics for the lists of
// the CTAs that took earlier tickets (the caller's barrier then hands them
// to the whole CTA).  Returns the old count.
__device__ __forceinline__ uint32_t ticket_add(uint32_t *t)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
    return old;
}

// The CTA whose range holds vector y (the last CTA whose start is <= y).
__device__ __forceinline__ int64_t range_of(int64_t y, int64_t per, int64_t total, int32_t nvr, int64_t ctas)
{
    int64_t b = min(ctas - 1, y / per + 1);
    while (b > 0 && range_start(b, per, total, nvr) > y) --b;
    return b;
}

// The last CTA to finish a piece of row r: load the np published piece lists
// (CTAs first..first+np-1, each list at most k entries, descending) into
// `buf` in one pass, then place every entry at its rank in the union (its
// position in its own list plus the entries of the other lists above it) and
// write the row.  Block-uniform; `buf` holds np * (kMaxK + 1) entries.
__device__ __noinline__ void fold_pieces(int64_t r, int64_t first, int np, int64_t per, int64_t total,
                                         int32_t nvr, int k, const uint64_t *partials, uint64_t *buf,
                                         int32_t *out_idx, uint16_t *out_val, int32_t *out_count,
                                         uint32_t *out_mask)
{
    const int tid = threadIdx.x;
    constexpr int kW = kMaxK + 1;
    for (int t = tid; t < np * (k + 1); t += kThreads) {
        const int j = t / (k + 1), e = t - j * (k + 1);
        const int64_t cta = first + j;
        const int sl = range_start(cta, per, total, nvr) / nvr == r ? 0 : 1;
        buf[j * kW + e] = __ldcg(partials + (size_t)(cta * 2 + sl) * kW + e);
    }
    __syncthreads();
    int entries = 0;
    uint32_t flags = 0;
    for (int j = 0; j < np; ++j) {
        const uint64_t h = buf[j * kW];
        entries += (int)(uint32_t)h;
        flags |= (uint32_t)(h >> 32);
    }
    for (int t = tid; t < np * kMaxK; t += kThreads) {
        const int j = t / kMaxK, p = t - j * kMaxK;
        const uint64_t *lj = buf + j * kW + 1;
        if (p >= (int)(uint32_t)buf[j * kW]) continue;
        const uint64_t x = lj[p];
        int pos = p;
        for (int i = 0; i < np && pos < k; ++i)
            if (i != j) pos += count_greater(buf + i * kW + 1, (int)(uint32_t)buf[i * kW], x);
        if (pos < k) {
            out_idx[r * k + pos] = entry_col(x);
            out_val[r * k + pos] = (uint16_t)(x & 0xFFFFu);
        }
    }
    const int cnt = min(k, entries);
    for (int t = cnt + tid; t < k; t += kThreads) {
        out_idx[r * k + t] = -1;
        out_val[r * k + t] = (uint16_t)kEmptyVal;
    }
    if (tid == 0) {
        out_count[r] = cnt;
        out_mask[r] = flags;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, kStreamCtasPerSm)
topk_stream_kernel(const uint16_t *__restrict__ logits, int32_t cols, int64_t row_stride, int32_t k,
                   int32_t nvr, int64_t total, int64_t per, int32_t *__restrict__ out_idx,
                   uint16_t *__restrict__ out_val, int32_t *__restrict__ out_count,
                   uint32_t *__restrict__ out_mask, uint64_t *__restrict__ partials,
                   uint32_t *__restrict__ tickets)
{
    grid_dependency_wait();
    extern __shared__ __align__(128) uint8_t dsmem[];
    uint4 *stages = reinterpret_cast<uint4 *>(dsmem);
    SmemCore &sm = *reinterpret_cast<SmemCore *>(dsmem + (size_t)kStages * kChunkVecs * 16);
    const int tid = threadIdx.x;
    const int64_t b = blockIdx.x;
    const int64_t ctas = gridDim.x;
    const int64_t g0 = range_start(b, per, total, nvr);
    const int64_t g1 = range_start(b + 1, per, total, nvr);

#ifdef TF_TOPK_TEST_WAIT_TIMEOUT
    // test build only: a barrier nothing completes, waited on after the first
    // chunk has landed, so that the wait runs out and the abort path runs
    __shared__ uint64_t never_bar;
#endif
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&sm.mbar[s], 1);
#ifdef TF_TOPK_TEST_WAIT_TIMEOUT
        mbar_init(&never_bar, 1);
#endif
        sm.n_cand = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // producer (thread 0): the bulk copies of chunk number `issued`, walking the
    // range [g0, g1) row by row without divisions
    const int64_t row0 = g0 / nvr;
    int64_t pg = g0, prow = row0;
    int32_t pcb = (int32_t)(g0 - row0 * nvr);
    int issued = 0;
    auto issue_next = [&]() {
        if (pg >= g1) return;
        int32_t pce = pcb + kChunkVecs;
        if (pce > nvr) pce = nvr;
        if ((int64_t)(pce - pcb) > g1 - pg) pce = pcb + (int32_t)(g1 - pg);
        const uint16_t *rowp = logits + prow * row_stride;
        const int32_t m = (int32_t)((reinterpret_cast<uintptr_t>(rowp) >> 1) & 7);
        const int32_t f0 = max(pcb, m ? 1 : 0);
        const int32_t f1 = min(pce, (cols + m) >> 3);
        const int s = issued % kStages;
        const uint32_t bytes = f1 > f0 ? (uint32_t)(f1 - f0) * 16u : 0u;
        mbar_expect_tx(&sm.mbar[s], bytes);
        if (bytes)
            bulk_load(stages + (size_t)s * kChunkVecs + (f0 - pcb),
                      reinterpret_cast<const uint4 *>(rowp - m) + f0, bytes, &sm.mbar[s]);
        pg += pce - pcb;
        if (pce == nvr) {
            ++prow;
            pcb = 0;
        } else {
            pcb = pce;
        }
        ++issued;
    };
    if (tid == 0)
        for (int s = 0; s < kStages - 1; ++s) issue_next();

    uint64_t *pend = reinterpret_cast<uint64_t *>(dsmem + (size_t)kStages * kChunkVecs * 16 + sizeof(SmemCore));
    int c = 0; // chunks consumed
    bool aborted = false;
    int64_t g = g0;
    int64_t row = row0; // the consumer's own cursor (thread 0's producer cursor runs ahead)
    int32_t vb = (int32_t)(g0 - row0 * nvr);
    int run_i = 0, free_i = 1, run_len = 0;
    int64_t split0 = -1, split1 = -1; // rows this range holds only a piece of (first, last)
    while (g < g1 && !aborted) {
        const int32_t ve = (int32_t)min((int64_t)nvr, (int64_t)vb + (g1 - g));
        const ChunkGeom geo = row_geometry(logits + row * row_stride, cols);
        if (tid == 0) {
            sm.flags = 0;
            sm.npend = 0;
        }
        run_i = 0;
        free_i = 1;
        run_len = 0;
        // the previous chunk, whose candidates wait in the pending buffer
        bool prev_lazy = false;
        uint4 *prev_st = nullptr;
        uint32_t prev_t = 0;
        int32_t prev_cb = 0;
        int prev_nvalid = 0;
        int prev_np0 = 0;
        // a bound valid for the rest of the piece: at least k of its columns
        // seen so far score at least this (0: none yet)
        uint32_t t_piece = 0;

        // Pending candidates of the previous chunk: an overflow is re-selected
        // exactly and merged; a full enough buffer is merged.  `at_end`: merge
        // whatever waits.  Returns the pending count afterwards (the same in
        // every thread).
        auto settle = [&](bool at_end) -> int {
            int np = (int)sm.npend;
            bool force = at_end;
            if (np > kPendCap) {
                np = lazy_overflow(sm, pend, prev_st, prev_t, geo, prev_cb, prev_nvalid, prev_np0, k);
                force = true;
            }
            if (np >= kMergeAt || (force && np > 0)) {
                merge_pending(sm, pend, np, k, run_i, free_i, run_len);
                np = 0;
            }
            return np;
        };
        int np_now = 0; // pending entries, as every thread knows them

        for (int32_t cb = vb; cb < ve; cb += kChunkVecs) {
            const int32_t ce = min(ve, cb + kChunkVecs);
            const int s = c % kStages;
            // one thread waits for the chunk's bulk copy; the barrier hands it on
            // (and makes the previous chunk's pushes visible)
            bool ok = true;
            if (tid == 0) ok = mbar_wait(&sm.mbar[s], (uint32_t)((c / kStages) & 1));
#ifdef TF_TOPK_TEST_WAIT_TIMEOUT
            if (tid == 0 && c == 0) ok = ok && mbar_wait(&never_bar, 0, 64);
#endif
            if (__syncthreads_or(!ok)) {
                aborted = true;
                break;
            }
            if (prev_lazy) np_now = settle(false);
            if (tid == 0) {
                // every thread is past the previous chunk: refill its stage
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_next();
            }
            uint4 *st = stages + (size_t)s * kChunkVecs;
            const int nvalid = ce - cb;
            const int32_t col_base = cb * 8 - geo.m;
            uint32_t kv[kVecPerThread][4];
            uint32_t tmax;
            if (nvalid == kChunkVecs && cb >= geo.vfull0 && ce <= geo.vfull1) {
#pragma unroll
                for (int i = 0; i < kVecPerThread; ++i) {
                    const uint4 q = st[i * kThreads + tid];
                    kv[i][0] = q.x;
                    kv[i][1] = q.y;
                    kv[i][2] = q.z;
                    kv[i][3] = q.w;
                }
                tmax = chunk_keys<true>(kv, geo, cb, nvalid, st, sm);
            } else {
#pragma unroll
                for (int i = 0; i < kVecPerThread; ++i) {
                    const int lv = i * kThreads + tid;
                    uint4 q = make_uint4(0, 0, 0, 0);
                    if (lv < nvalid) {
                        const int32_t v = cb + lv;
                        q = (v >= geo.vfull0 && v < geo.vfull1) ? st[lv]
                                                               : load_edge_vector(geo.rowp, cols, geo.m, v);
                    }
                    kv[i][0] = q.x;
                    kv[i][1] = q.y;
                    kv[i][2] = q.z;
                    kv[i][3] = q.w;
                }
                tmax = chunk_keys<false>(kv, geo, cb, nvalid, st, sm);
            }
            // A new entry must beat the running k-th strictly once the piece has
            // k entries (every column of this chunk is higher); before that, a
            // prefilter bound of the first chunk that has one.  Candidates go to
            // the pending buffer as list entries, with no barrier: only threads
            // whose max reaches the bound spill their keys, and their warp scans
            // them one word per lane.
            uint32_t t_floor;
            if (run_len == k) {
                t_floor = (uint32_t)(sm.list[run_i][k - 1] >> 48) + 1u;
            } else if (t_piece != 0) {
                t_floor = t_piece;
            } else {
                const uint32_t t0 = prefilter_bound(tmax, nvalid, k, sm);
                t_floor = max(key_floor(t0), 1u);
                if (t0 != 0) t_piece = t_floor;
            }
            push_pending(kv, tmax, t_floor, col_base, st, sm, pend);
            // the stage is next written by a bulk copy (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            prev_lazy = true;
            prev_st = st;
            prev_t = t_floor;
            prev_cb = cb;
            prev_nvalid = nvalid;
            prev_np0 = np_now;
            ++c;
        }
        if (aborted) break;
        __syncthreads(); // the running list, or the last chunk's pushes, are complete
        if (prev_lazy) settle(true);
        prev_lazy = false;

        // ---- end of a row piece
        const int len = run_len;
        if (vb == 0 && ve == nvr) {
            write_row(row, sm.list[run_i], len, sm.flags, k, out_idx, out_val, out_count, out_mask);
        } else {
            // publish this piece's list (plain stores); its ticket is taken once
            // the whole range is done, so the stream of chunks never stalls here
            const int slot = row == row0 ? 0 : 1;
            uint64_t *mine = partials + (size_t)(b * 2 + slot) * (kMaxK + 1);
            for (int t = tid; t < len; t += kThreads) mine[1 + t] = sm.list[run_i][t];
            if (tid == 0) mine[0] = (uint64_t)(uint32_t)len | ((uint64_t)sm.flags << 32);
            if (slot == 0)
                split0 = row;
            else
                split1 = row;
        }
        g += ve - vb;
        if (ve == nvr) {
            ++row;
            vb = 0;
        } else {
            vb = ve;
        }
    }

    if (!aborted && (split0 >= 0 || split1 >= 0)) {
        // every piece is published: one fence, then a ticket per split row; the
        // last piece in for a row folds all of its pieces
        __syncthreads();
        if (tid == 0) {
            uint32_t t0 = 0, t1 = 0;
            if (split0 >= 0) t0 = ticket_add(&tickets[range_of(split0 * nvr, per, total, nvr, ctas)]);
            if (split1 >= 0) t1 = ticket_add(&tickets[range_of(split1 * nvr, per, total, nvr, ctas)]);
            sm.ticket[0] = t0;
            sm.ticket[1] = t1;
        }
        __syncthreads();
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int64_t r = s == 0 ? split0 : split1;
            if (r < 0) continue;
            const int64_t first = range_of(r * nvr, per, total, nvr, ctas);
            const int64_t last = range_of((r + 1) * nvr - 1, per, total, nvr, ctas);
            const int np = (int)(last - first + 1);
            if (sm.ticket[s] != (uint32_t)(np - 1)) continue;
            fold_pieces(r, first, np, per, total, nvr, k, partials, reinterpret_cast<uint64_t *>(stages),
                        out_idx, out_val, out_count, out_mask);
            if (tid == 0) tickets[first] = 0; // ready for the next call
        }
    }

    if (aborted) {
        if (tid == 0) {
            atomicCAS(&g_fault, 0u, kFaultWaitTimeout);
            // drain this CTA's copies still in flight, each with a bounded wait
            for (int q = c; q < issued; ++q) mbar_wait(&sm.mbar[q % kStages], (uint32_t)((q / kStages) & 1));
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- cluster kernel

__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Loads the chunk of vectors [cbeg, min(v_end, cbeg + kChunkVecs)) of a row
// into this thread's registers: vector i * kThreads + tid in kv[i]; vectors
// past the chunk read as zero.  Inside the row's 16-byte-aligned body the
// loads are plain; the row's ragged head and tail go through the edge path.
__device__ __forceinline__ void load_chunk(uint32_t (&kv)[kVecPerThread][4], const uint4 *vbase,
                                           const ChunkGeom &geo, int32_t cbeg, int32_t v_end, int32_t cols)
{
    const int tid = threadIdx.x;
    const int32_t cend = min(v_end, cbeg + kChunkVecs);
    const int nvalid = cend - cbeg;
    if (nvalid == kChunkVecs && cbeg >= geo.vfull0 && cend <= geo.vfull1) {
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
            const uint4 q = ld_stream(vbase + cbeg + i * kThreads + tid);
            kv[i][0] = q.x;
            kv[i][1] = q.y;
            kv[i][2] = q.z;
            kv[i][3] = q.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
            const int lv = i * kThreads + tid;
            uint4 q = make_uint4(0, 0, 0, 0);
            if (lv < nvalid) {
                const int32_t v = cbeg + lv;
                q = (v >= geo.vfull0 && v < geo.vfull1) ? ld_stream(vbase + v)
                                                       : load_edge_vector(geo.rowp, cols, geo.m, v);
            }
            kv[i][0] = q.x;
            kv[i][1] = q.y;
            kv[i][2] = q.z;
            kv[i][3] = q.w;
        }
    }
}

// n 16-byte vectors from p toward L2 (n <= 0: none); p and the vectors lie
// inside the caller's rows.
__device__ __forceinline__ void l2_prefetch_vecs(const uint4 *p, int32_t n)
{
    if (n > 0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"((uint32_t)n * 16u) : "memory");
}

// grid.x = rows * S; the launch groups each row's S CTAs into one cluster
// (cluster rank == span).  kPf: chunks sent toward L2 before the dependency
// wait (2 for two-span grids of one wave, where the second chunk's prefetch
// gained; it cost the other span counts and grids of more waves).
template <int S, int kFmt = kBf16, int kPf = 1>
__global__ void __launch_bounds__(kThreads, kClusterCtasPerSm)
topk_cluster_kernel(const uint16_t *__restrict__ logits, int32_t cols, int64_t row_stride, int32_t k,
                    int32_t *__restrict__ out_idx, uint16_t *__restrict__ out_val,
                    int32_t *__restrict__ out_count, uint32_t *__restrict__ out_mask)
{
    __shared__ SmemCore sm;
    __shared__ SmemGather sg;
    __shared__ uint4 keys[kChunkVecs];
    const int tid = threadIdx.x;
    const int span = (int)(blockIdx.x % S);
    const int64_t row = (int64_t)(blockIdx.x / S);

    ChunkGeom geo = row_geometry(logits + row * row_stride, cols);
    const uint4 *vbase = reinterpret_cast<const uint4 *>(geo.rowp - geo.m);
    const int32_t nvec = (cols + geo.m + 7) >> 3;
    const int32_t per_span = (nvec + S - 1) / S;
    const int32_t v_begin = min(nvec, span * per_span);
    const int32_t v_end = min(nvec, v_begin + per_span);
    // while the previous kernel on the stream ends: the first kPf chunks'
    // whole vectors toward L2 (a hint only: L2 is where device memory is
    // coherent, so values that kernel writes are still read after the wait)
    if (tid == 0) {
        const int32_t a = max(v_begin, geo.vfull0), e = min(min(v_end, v_begin + kPf * kChunkVecs), geo.vfull1);
        l2_prefetch_vecs(vbase + a, e - a);
    }
    grid_dependency_wait();
    cluster_arrive_relaxed(); // paired with the wait before DSMEM use

    if (tid == 0) {
        sm.flags = 0;
        sm.n_cand = 0;
    }
    __syncthreads();
    int run_i = 0, free_i = 1, run_len = 0;
    uint32_t cand_base = 0; // the candidate counter before this chunk (block-uniform)

    uint32_t kv[kVecPerThread][4];
    if (v_begin < v_end) load_chunk(kv, vbase, geo, v_begin, v_end, cols);
    for (int32_t cbeg = v_begin; cbeg < v_end; cbeg += kChunkVecs) {
        const int32_t cend = min(v_end, cbeg + kChunkVecs);
        const int nvalid = cend - cbeg;
        const int32_t col_base = cbeg * 8 - geo.m;
        const bool full = nvalid == kChunkVecs && cbeg >= geo.vfull0 && cend <= geo.vfull1;
        // a full chunk inside the row: the max from the raw bits where it can be
        uint32_t tmax = 0;
        const bool raw = full && raw_tmax<kFmt>(kv, tmax);
        if (!raw) tmax = chunk_keys<false, kFmt>(kv, geo, cbeg, nvalid, keys, sm);
        const uint32_t t_floor = chunk_floor(tmax, nvalid, k, sm, run_i, run_len);
        const bool hit = spill_hits(kv, tmax, raw, t_floor, keys);
        // the chunk's registers are free: the next chunk's loads fly during
        // the candidate scan, the rank and the merge
        const bool more = cend < v_end;
        if (more) load_chunk(kv, vbase, geo, cend, v_end, cols);
        const uint32_t n =
            push_candidates<kFmt>(hit, t_floor, k, sm, keys, cand_base);
        if (n) merge_candidates(n, col_base, k, sm, run_i, free_i, run_len);
        __syncthreads(); // the merge is complete before the next chunk reads its bound
    }

    // ---- push this span's list into the leader's shared memory
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); // every CTA has started
    cg::cluster_group cluster = cg::this_cluster();
    uint64_t *gl = cluster.map_shared_rank(&sg.gather[span][0], 0);
    const int len = run_len;
    for (int t = tid; t < len; t += kThreads) gl[t] = sm.list[run_i][t];
    if (tid == 0) {
        *cluster.map_shared_rank(&sg.glen[span], 0) = len;
        *cluster.map_shared_rank(&sg.gflags[span], 0) = sm.flags;
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    if (span != 0) return;

    // ---- leader: pairwise merge tree over the S lists, then the row
    uint32_t flags = 0;
#pragma unroll
    for (int s = 0; s < S; ++s) flags |= sg.gflags[s];
    int flen = 0;
    const uint64_t *fin = merge_tree(sg, S, k, flen);
    write_row<kFmt>(row, fin, flen, flags, k, out_idx, out_val, out_count, out_mask);
}

// ---------------------------------------------------------------- shard-list merge kernel
//
// The merge stage on its own (TensorFold PR #713, change 3: span results are
// merged "with the same tournament", i.e. in the same (score, lower index)
// order).  Each of `shards` column blocks of a row has its own top list (as
// tf_topk_bf16 writes it for that block: entries best first, a count, a
// non-finite mask); the row's result is the top k of the union of those
// entries, with every index moved by its shard's column offset.  One CTA per
// row: each list's first min(k, count) entries become 64-bit entries (score,
// ~global index, original bits), and an entry's rank is its position in its
// own list plus, for every other list, the entries there that beat it (a
// binary search, since every list is sorted the same way).

constexpr int kMergeThreads = 128;

// Order-preserving key of one bf16 value (0 for a NaN, which is never selected).
__device__ __forceinline__ uint32_t merge_key(uint32_t raw)
{
    if ((raw & 0x7FFFu) > 0x7F80u) return 0;
    return raw ^ ((raw & 0x8000u) ? 0xFFFFu : 0x8000u);
}

struct MergeShards {
    int64_t offset[TF_TOPK_MAX_SHARDS];
};

__global__ void __launch_bounds__(kMergeThreads)
topk_merge_kernel(const int32_t *__restrict__ in_idx, const uint16_t *__restrict__ in_val,
                  const int32_t *__restrict__ in_count, const uint32_t *__restrict__ in_mask, int64_t rows,
                  int32_t shards, int32_t k_in, MergeShards off, int32_t k, int32_t *__restrict__ out_idx,
                  uint16_t *__restrict__ out_val, int32_t *__restrict__ out_count, uint32_t *__restrict__ out_mask)
{
    grid_dependency_wait();
    __shared__ uint64_t lists[TF_TOPK_MAX_SHARDS][kMaxK];
    __shared__ int32_t lens[TF_TOPK_MAX_SHARDS];
    __shared__ uint32_t flags_all;
    __shared__ int32_t total_all;
    const int tid = threadIdx.x;
    const int64_t r = blockIdx.x;
    if (tid == 0) {
        flags_all = 0;
        total_all = 0;
    }
    __syncthreads();
    // only an entry in a list's top min(k, k_in) can reach the row's top k
    const int width = min(k, k_in);
    for (int s = tid; s < shards; s += kMergeThreads) {
        const int64_t cell = (int64_t)s * rows + r;
        lens[s] = max(0, min(width, in_count[cell]));
        atomicOr(&flags_all, in_mask[cell]);
    }
    __syncthreads();
    // gather; an entry with no column or a NaN value ends its list
    for (int t = tid; t < shards * width; t += kMergeThreads) {
        const int s = t / width, p = t - s * width;
        if (p >= lens[s]) continue;
        const int64_t at = ((int64_t)s * rows + r) * k_in + p;
        const int32_t li = in_idx[at];
        const uint32_t key = merge_key(in_val[at]);
        const int64_t gi = off.offset[s] + li;
        if (li < 0 || key == 0 || gi > (int64_t)INT32_MAX) {
            atomicMin(&lens[s], p);
            continue;
        }
        lists[s][p] = list_entry(key, (int32_t)gi);
    }
    __syncthreads();
    if (tid == 0) {
        int sum = 0;
        for (int s = 0; s < shards; ++s) sum += lens[s];
        total_all = sum;
    }
    __syncthreads();
    for (int t = tid; t < shards * width; t += kMergeThreads) {
        const int s = t / width, p = t - s * width;
        if (p >= lens[s]) continue;
        const uint64_t x = lists[s][p];
        int rank = 0;
        for (int j = 0; j < shards && rank < k; ++j) rank += count_greater(lists[j], lens[j], x);
        if (rank < k) {
            out_idx[r * k + rank] = entry_col(x);
            out_val[r * k + rank] = (uint16_t)(x & 0xFFFFu);
        }
    }
    const int cnt = min(k, total_all);
    for (int t = cnt + tid; t < k; t += kMergeThreads) {
        out_idx[r * k + t] = -1;
        out_val[r * k + t] = (uint16_t)kEmptyVal;
    }
    if (tid == 0) {
        out_count[r] = cnt;
        out_mask[r] = flags_all;
    }
}

// ------------------------------------------------ nucleus (top-p) after the top-k
//
// Sampling probabilities over each row's top-k list, as the speculative
// decoding receipts of the TensorFold PR #3069 page ("Receipt": temperature
// 0.7, top-k 20, top-p 0.95) use them: the softmax of value / T over the
// row's entries, the shortest best-first prefix whose mass reaches top_p, that
// prefix renormalised.  One warp per row (k <= 64: two entries a lane); the
// prefix mass is a warp scan, the cut a ballot.

constexpr int kNucleusWarps = 8;

__device__ __forceinline__ float warp_inclusive_scan(float x, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, x, d);
        if (lane >= d) x += y;
    }
    return x;
}

// A list value as float (exact for every format): bf16 is the top half of a
// binary32, fp16 widens exactly, fp32 is itself.
template <int kFmt>
__device__ __forceinline__ float list_value(uint32_t bits)
{
    if constexpr (kFmt == TF_TOPK_DTYPE_F16) return __half2float(__ushort_as_half((unsigned short)bits));
    else if constexpr (kFmt == TF_TOPK_DTYPE_F32) return __uint_as_float(bits);
    else return __uint_as_float(bits << 16);
}

template <typename T, int kFmt>
__global__ void __launch_bounds__(kNucleusWarps * 32)
topk_nucleus_kernel(const T *__restrict__ val, const int32_t *__restrict__ count, int64_t rows, int32_t k,
                    float temperature, float top_p, float *__restrict__ out_prob, int32_t *__restrict__ out_keep)
{
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kNucleusWarps + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int n_in = max(0, min((int)k, count[r]));
    float v[2];
    bool nan[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = lane + 32 * j;
        v[j] = i < n_in ? list_value<kFmt>((uint32_t)val[r * k + i]) : 0.f;
        nan[j] = i < n_in && isnan(v[j]);
    }
    // the top-k ranks NaN below every number: the numbers are the prefix before the first NaN
    const unsigned nan_lo = __ballot_sync(0xFFFFFFFFu, nan[0]);
    const unsigned nan_hi = __ballot_sync(0xFFFFFFFFu, nan[1]);
    const int n = nan_lo ? __ffs(nan_lo) - 1 : (nan_hi ? 31 + __ffs(nan_hi) : n_in);
    const float best = __shfl_sync(0xFFFFFFFFu, v[0], 0);
    float e[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = lane + 32 * j;
        if (i >= n)
            e[j] = 0.f;
        else if (temperature == 0.f)
            e[j] = i == 0 ? 1.f : 0.f;            // greedy
        else if (isinf(best))
            e[j] = v[j] == best ? 1.f : 0.f;      // equal shares among the infinite best
        else
            e[j] = expf((v[j] - best) / temperature);
    }
    // running mass, best first: positions 0..31 then 32..63
    const float c_lo = warp_inclusive_scan(e[0], lane);
    const float c_hi = warp_inclusive_scan(e[1], lane) + __shfl_sync(0xFFFFFFFFu, c_lo, 31);
    const float total = __shfl_sync(0xFFFFFFFFu, c_hi, 31);
    int keep = n;
    if (top_p < 1.f && n > 0) {
        // mass c reaches top_p of the total when c - top_p * total >= 0; one
        // fused multiply-add rounds that difference once, which keeps its
        // sign, so the comparison is exact (equal shares cut exactly)
        const unsigned hit_lo = __ballot_sync(0xFFFFFFFFu, lane < n && fmaf(-top_p, total, c_lo) >= 0.f);
        const unsigned hit_hi = __ballot_sync(0xFFFFFFFFu, lane + 32 < n && fmaf(-top_p, total, c_hi) >= 0.f);
        keep = hit_lo ? __ffs(hit_lo) : (hit_hi ? 32 + __ffs(hit_hi) : n);
    }
    // mass of the kept prefix (position keep - 1 of the scan)
    const int last = max(keep, 1) - 1;
    const float kept_lo = __shfl_sync(0xFFFFFFFFu, c_lo, last & 31);
    const float kept_hi = __shfl_sync(0xFFFFFFFFu, c_hi, last & 31);
    const float kept = last < 32 ? kept_lo : kept_hi;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = lane + 32 * j;
        if (i < k) out_prob[r * k + i] = i < keep ? e[j] / kept : 0.f;
    }
    if (lane == 0) out_keep[r] = keep;
}

// ------------------------------------------------ wide select: any format, k <= 1024
//
// The same order (score descending, lower column first; NaN never selected,
// +0 == -0) for bf16, fp16 and fp32 rows and k up to TF_TOPK_MAX_K_WIDE.  One
// CTA per row, in two passes over the row:
//   1. each thread keeps the keys of its Q = 4 best elements (distinct
//      elements), and the CTA takes the row's non-finite mask
//      and its count of numbers.  Each warp finds the j-th largest of its
//      lanes' kept keys, j = ceil(k / warps), so B = the smallest of those is
//      reached by at least k elements of the row;
//   2. every element with key >= B -- a superset of the row's top k, ties at
//      B included -- goes into shared memory as a 64-bit entry (key << 32 |
//      ~column); ranking them (by count, or a bitonic sort when many) gives
//      the order (equal keys: the higher ~column, i.e. the lower column,
//      first), of which the first k are the result.
// When more than kWideCap elements reach B (heavy ties), the k-th key K* is
// found exactly by a 16-ary search over counting passes, the entries above it
// are collected, and the ties at K* are taken in column order from
// contiguous per-thread column ranges.

constexpr int kWideThreads = 512;
constexpr int kWideWarps = kWideThreads / 32;
constexpr int kWideUnroll = 8;                  // 16-byte loads in flight per thread
constexpr int kWideCap = 4096;                  // entries pass 2 may collect
constexpr int kWideMaxK = TF_TOPK_MAX_K_WIDE;
constexpr int kWideKeep = 4;                    // keys a thread keeps in the first pass
// a warp's 32 lanes keep at least the j = ceil(k / warps) keys its bound
// counts, for every k (more kept keys made the bound tighter but the first
// pass slower: 16 for k = 1024 cost 239k cycles a row against about 100k)
static_assert(32 * kWideKeep >= (TF_TOPK_MAX_K_WIDE + kWideWarps - 1) / kWideWarps, "a warp keeps j keys");
static_assert(32 * 16 >= (kWideMaxK + kWideWarps - 1) / kWideWarps, "a warp keeps j keys (large k)");
static_assert(kWideCap >= kWideMaxK, "a short row's numbers all fit");
// The first pass writes each 8 elements' largest key (its upper 16 bits) to a
// table in shared memory, so the second reads back only the vectors whose
// largest key reaches the bound; rows too wide for the table (or whose table
// has more than kWideList such entries) read the whole row again.
constexpr int kWideTbl = 32768;                 // entries: rows up to 262144 columns
constexpr int kWideList = 2048;                 // table entries the second pass may take
static_assert(kWideTbl % (8 * kWideThreads) == 0 && kWideList % kWideThreads == 0, "whole rounds");
static_assert(kWideTbl * 2 >= kWideCap * 8 && kWideCap == 4096 && kWideThreads == 512, "the sort's buffers");

// Order-preserving key of one element (0 for NaN, +0 and -0 one key), and
// its non-finite flag (1 NaN, 2 +inf, 4 -inf).
template <typename T, int kFmt>
struct WideFormat;

template <>
struct WideFormat<uint16_t, TF_TOPK_DTYPE_BF16> {
    static constexpr uint32_t kNanFloor = 0x7F80u, kPosInf = 0x7F80u, kNegInf = 0xFF80u, kEmpty = 0x7FC0u;
    static constexpr uint32_t kSign = 0x8000u, kOnes = 0xFFFFu;
};
template <>
struct WideFormat<uint16_t, TF_TOPK_DTYPE_F16> {
    static constexpr uint32_t kNanFloor = 0x7C00u, kPosInf = 0x7C00u, kNegInf = 0xFC00u, kEmpty = 0x7E00u;
    static constexpr uint32_t kSign = 0x8000u, kOnes = 0xFFFFu;
};
template <>
struct WideFormat<uint32_t, TF_TOPK_DTYPE_F32> {
    static constexpr uint32_t kNanFloor = 0x7F800000u, kPosInf = 0x7F800000u, kNegInf = 0xFF800000u,
                              kEmpty = 0x7FC00000u;
    static constexpr uint32_t kSign = 0x80000000u, kOnes = 0xFFFFFFFFu;
};

// Keys of the infinities: a raw key (sign-flipped bits, NaN not yet zeroed)
// above the +inf key or below the -inf key is a NaN.
template <typename T, int kFmt>
struct WideKeys {
    using F = WideFormat<T, kFmt>;
    static constexpr uint32_t kPosInfKey = F::kPosInf ^ F::kSign;
    static constexpr uint32_t kNegInfKey = F::kNegInf ^ F::kOnes;
};

// Raw keys of a 16-byte vector, one 32-bit word at a time: two 16-bit keys
// per word (packed), or one 32-bit key.
__device__ __forceinline__ uint32_t raw_key_word(uint32_t w, std::integral_constant<int, 2>)
{
    return keys_from_raw2(w);
}
__device__ __forceinline__ uint32_t raw_key_word(uint32_t w, std::integral_constant<int, 4>)
{
    return w ^ ((uint32_t)((int32_t)w >> 31) | 0x80000000u);
}

template <typename T, int kFmt>
__device__ __forceinline__ uint32_t wide_key(uint32_t raw)
{
    using F = WideFormat<T, kFmt>;
    if ((raw & ~F::kSign) > F::kNanFloor) return 0u;             // NaN
    const uint32_t key = raw ^ ((raw & F::kSign) ? F::kOnes : F::kSign);
    return key == F::kSign - 1u ? F::kSign : key;                  // -0 -> +0
}

template <typename T, int kFmt>
__device__ __forceinline__ uint32_t wide_flag(uint32_t raw)
{
    using F = WideFormat<T, kFmt>;
    if ((raw & ~F::kSign) > F::kNanFloor) return 1u;
    if (raw == F::kPosInf) return 2u;
    if (raw == F::kNegInf) return 4u;
    return 0u;
}

// Elements before the row's first 16-byte boundary (all of a short row).
template <typename T>
__device__ __forceinline__ int32_t wide_head(const T *row, int32_t cols)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(row);
    const int32_t head = (int32_t)(((16u - (uint32_t)(a & 15u)) & 15u) / sizeof(T));
    return head < cols ? head : cols;
}

// Every column of the row, each thread a strided share: the row's unaligned
// head and tail through f(column, raw bits), the 16-byte-aligned body
// through g(vector, its first column), kWideUnroll vectors a thread in flight
// before any is used.  With kEdges false only the body is visited.
template <typename T, bool kEdges, typename Fe, typename Fv>
__device__ __forceinline__ void wide_scan2(const T *row, int32_t cols, Fe &&f, Fv &&g)
{
    constexpr int kPer = 16 / (int)sizeof(T);
    const int tid = threadIdx.x;
    const int32_t head = wide_head(row, cols);
    if constexpr (kEdges)
        for (int32_t c = tid; c < head; c += kWideThreads) f(c, (uint32_t)row[c]);
    const int32_t nvec = (cols - head) / kPer;
    const uint4 *v = reinterpret_cast<const uint4 *>(row + head);
    // whole batches of kWideUnroll loads, then the rest one by one (a guarded
    // last batch here cost the exact paths' counting scans spills)
    int32_t i = tid;
    for (; i + (kWideUnroll - 1) * kWideThreads < nvec; i += kWideUnroll * kWideThreads) {
        uint4 q[kWideUnroll];
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u) q[u] = v[i + u * kWideThreads];
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u) g(q[u], head + (i + u * kWideThreads) * kPer);
    }
    for (; i < nvec; i += kWideThreads) g(v[i], head + i * kPer);
    if constexpr (kEdges)
        for (int32_t c = head + nvec * kPer + tid; c < cols; c += kWideThreads) f(c, (uint32_t)row[c]);
}

// The elements of a vector, in column order: f(column, raw bits).
template <typename T, typename Fe>
__device__ __forceinline__ void vector_elems(const uint4 &q, int32_t c0, Fe &&f)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (sizeof(T) == 2) {
            f(c0 + 2 * j, w[j] & 0xFFFFu);
            f(c0 + 2 * j + 1, w[j] >> 16);
        } else {
            f(c0 + j, w[j]);
        }
    }
}

// f(column, raw bits) for every column of the row.
template <typename T, typename Fe>
__device__ __forceinline__ void wide_scan(const T *row, int32_t cols, Fe &&f)
{
    wide_scan2<T, true>(row, cols, f, [&](const uint4 &q, int32_t c0) { vector_elems<T>(q, c0, f); });
}

// Max and min raw key of a vector (16-bit keys packed in pairs).
template <typename T>
__device__ __forceinline__ void vector_key_range(const uint4 &q, uint32_t &vmx, uint32_t &vmn)
{
    constexpr std::integral_constant<int, (int)sizeof(T)> width{};
    const uint32_t a = raw_key_word(q.x, width), b = raw_key_word(q.y, width);
    const uint32_t c = raw_key_word(q.z, width), d = raw_key_word(q.w, width);
    if constexpr (sizeof(T) == 2) {
        vmx = max_u16x2(max_u16x2(a, b), max_u16x2(c, d));
        vmn = min_u16x2(min_u16x2(a, b), min_u16x2(c, d));
    } else {
        vmx = max(max(a, b), max(c, d));
        vmn = min(min(a, b), min(c, d));
    }
}

template <typename T>
__device__ __forceinline__ uint32_t hi_key(uint32_t packed)
{
    if constexpr (sizeof(T) == 2) return max(packed & 0xFFFFu, packed >> 16);
    else return packed;
}

template <typename T>
__device__ __forceinline__ uint32_t lo_key(uint32_t packed)
{
    if constexpr (sizeof(T) == 2) return min(packed & 0xFFFFu, packed >> 16);
    else return packed;
}

// Descending bitonic sort of s[0..n) (n a power of two), every thread of the
// CTA taking part; ends with a barrier.
template <typename K>
__device__ __forceinline__ void bitonic_desc(K *s, int n)
{
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const int sh = __ffs(stride) - 1; // stride is a power of two
            for (int i = threadIdx.x; i < (n >> 1); i += kWideThreads) {
                const int lo = ((i >> sh) << (sh + 1)) | (i & (stride - 1)), hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const K x = s[lo], y = s[hi];
                if ((x < y) == desc) {
                    s[lo] = y;
                    s[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

__device__ __forceinline__ uint32_t wide_block_sum(uint32_t v, uint32_t *red)
{
    v = __reduce_add_sync(0xFFFFFFFFu, v);
    __syncthreads(); // red is free (an earlier sum has been read)
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t s = 0;
#pragma unroll
    for (int w = 0; w < kWideThreads / 32; ++w) s += red[w];
    return s;
}

struct __align__(16) WideSmem {
    uint64_t ent[kWideCap];
    uint64_t sorted[kWideThreads];           // ranked entries when few
    uint16_t tbl[kWideTbl];                  // the upper 16 bits of each 8 elements' largest key
                                             // (then the sort's second buffer)
    uint32_t list[kWideList];                // table entries that reach the bound
    uint32_t red[kWideWarps];
    uint32_t warp_b[kWideWarps];
    uint32_t n_ent, flags, nnz, kmax, n_list;
};

// Keep the Q largest keys seen (t[0] >= ... >= t[Q-1]; 0 = empty).
template <int Q>
__device__ __forceinline__ void keep_insert(uint32_t (&t)[Q], uint32_t key)
{
    if (key > t[Q - 1]) {
        t[Q - 1] = key;
#pragma unroll
        for (int i = Q - 1; i > 0; --i) {
            const uint32_t a = t[i - 1], b = t[i];
            t[i - 1] = max(a, b);
            t[i] = min(a, b);
        }
    }
}

// The j-th largest of the warp's kept keys (counted with repeats), or 0 when
// the warp holds fewer than j nonzero keys: the largest x with at least j
// keys >= x, built bit by bit from the top of a kBits-bit key.  Warp-uniform.
template <int Q, int kBits>
__device__ __forceinline__ uint32_t warp_jth(const uint32_t (&t)[Q], uint32_t j)
{
    uint32_t x = 0;
#pragma unroll 1
    for (int b = kBits - 1; b >= 0; --b) {
        const uint32_t c = x | (1u << b);
        uint32_t n = 0;
#pragma unroll
        for (int i = 0; i < Q; ++i) n += t[i] >= c;
        if (__reduce_add_sync(0xFFFFFFFFu, n) >= j) x = c;
    }
    return x;
}

// Slots for c items of every lane of the warp (all 32 lanes call): the
// lane's first slot, one atomic on the counter for the whole warp.
__device__ __forceinline__ uint32_t warp_reserve(uint32_t c, uint32_t *counter)
{
    const int lane = threadIdx.x & 31;
    uint32_t incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += u;
    }
    uint32_t base = 0;
    if (lane == 31 && incl != 0) base = atomicAdd(counter, incl);
    return __shfl_sync(0xFFFFFFFFu, base, 31) + incl - c;
}

// Descending sort of s[0..16 * 32 R) into s or u (the one returned), every
// thread of the CTA taking part.  Each warp sorts a run of 32 R entries in
// registers (a bitonic network: element r * 32 + lane in e[r], partners a
// lane apart exchanged by shuffles, the others within the thread), then four
// rounds merge pairs of runs through shared memory, each thread placing R
// consecutive outputs found by a merge-path search (the final round only
// those below `need`).  Entries equal only when they are padding.
template <int R>
__device__ uint64_t *wide_sort(uint64_t *s, uint64_t *u, int need)
{
    constexpr int L0 = 32 * R, N = 16 * L0;
    static_assert(kWideWarps == 16, "16 runs");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t e[R];
#pragma unroll
    for (int r = 0; r < R; ++r) e[r] = s[warp * L0 + r * 32 + lane];
#pragma unroll
    for (int size = 2; size <= L0; size <<= 1) {
#pragma unroll
        for (int d = size >> 1; d > 0; d >>= 1) {
            if (d >= 32) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int pr = r ^ (d >> 5);
                    if (pr > r) {
                        const bool desc = ((r * 32 + lane) & size) == 0;
                        const uint64_t hi = max(e[r], e[pr]), lo = min(e[r], e[pr]);
                        e[r] = desc ? hi : lo;
                        e[pr] = desc ? lo : hi;
                    }
                }
            } else {
                const bool lower = (lane & d) == 0;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const bool desc = ((r * 32 + lane) & size) == 0;
                    const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, e[r], d);
                    e[r] = (lower == desc) ? max(e[r], o) : min(e[r], o);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) s[warp * L0 + r * 32 + lane] = e[r];
    __syncthreads();
    uint64_t *src = s, *dst = u;
#pragma unroll 1
    for (int L = L0; L < N; L <<= 1) {
        const int o0 = threadIdx.x * R;
        if (2 * L < N || o0 < need) {
            const int base = o0 & ~(2 * L - 1), d = o0 - base;
            const uint64_t *A = src + base, *B = A + L;
            // a: how many of the first d outputs come from A (A first only when larger)
            int lo = max(0, d - L), hi = min(d, L);
            while (lo < hi) {
                const int m = (lo + hi) >> 1;
                if (A[m] > B[d - 1 - m]) lo = m + 1;
                else hi = m;
            }
            int a = lo, b = d - lo;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const bool takeA = b >= L || (a < L && A[a] > B[b]);
                dst[o0 + r] = takeA ? A[a++] : B[b++];
            }
        }
        __syncthreads();
        uint64_t *x = src;
        src = dst;
        dst = x;
    }
    return src;
}

// The k largest of the n distinct entries in sm.ent (k < n), into dst[0..k)
// in no order: the k-th largest key K by a radix select on the key, 8 bits
// a pass from the top (a 256-bin count of the entries that match the digits
// found so far, then the digit where the count from the top reaches the
// places left); the entries above K; and of the ties at K those with the
// largest entries (lowest columns), each tie placed at its count of larger
// ties.  Returns false, with nothing selected, when more ties meet at K than
// one per thread (the caller sorts all n then).  Block-uniform.
template <typename T>
__device__ __noinline__ bool wide_select_top(WideSmem &sm, uint32_t n, int k, uint64_t *dst)
{
    constexpr int kKeyBits = 8 * (int)sizeof(T); // 16-bit keys for 2-byte formats
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t *hist = sm.list; // free after the second pass
    uint32_t prefix = 0, need = (uint32_t)k;
#pragma unroll 1
    for (int shift = kKeyBits - 8; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += kWideThreads) hist[b] = 0;
        __syncthreads();
        const uint32_t hmask = shift + 8 >= 32 ? 0u : ~0u << (shift + 8); // the digits found so far
        for (uint32_t i = tid; i < n; i += kWideThreads) {
            const uint32_t key = (uint32_t)(sm.ent[i] >> 32);
            if ((key & hmask) == (prefix & hmask)) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            // lane L: bins 255 - 8L down to 248 - 8L; the lane whose bins hold
            // the need-th entry from the top names the digit
            uint32_t c[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hist[255 - 8 * lane - j];
                sum += c[j];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += u;
            }
            uint32_t acc = incl - sum;
            if (acc < need && need <= incl) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (acc < need && need <= acc + c[j]) {
                        sm.red[0] = (uint32_t)(255 - 8 * lane - j);
                        sm.red[1] = acc; // entries above this digit
                    }
                    acc += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= sm.red[0] << shift;
        need -= sm.red[1];
        __syncthreads(); // the next pass rewrites hist and red
    }
    // K = prefix: k - need entries above it, `need` of its ties to take
    if (tid == 0) {
        sm.warp_b[0] = 0;
        sm.warp_b[1] = 0;
    }
    __syncthreads();
    for (uint32_t i0 = 0; i0 < n; i0 += kWideThreads) {
        const uint32_t i = i0 + (uint32_t)tid;
        const uint64_t e = i < n ? sm.ent[i] : 0;
        const uint32_t key = (uint32_t)(e >> 32);
        const bool up = i < n && key > prefix, tie = i < n && key == prefix;
        const uint32_t a = warp_reserve(up ? 1u : 0u, &sm.warp_b[0]);
        const uint32_t t = warp_reserve(tie ? 1u : 0u, &sm.warp_b[1]);
        if (up) dst[a] = e;
        if (tie && t < (uint32_t)kWideThreads) sm.sorted[t] = e;
    }
    __syncthreads();
    const uint32_t above = sm.warp_b[0], ties = sm.warp_b[1];
    if (ties > (uint32_t)kWideThreads) return false;
    if ((uint32_t)tid < ties) {
        const uint64_t x = sm.sorted[tid];
        uint32_t r = 0;
        for (uint32_t u = 0; u < ties; ++u) r += sm.sorted[u] > x;
        if (r < need) dst[above + r] = x;
    }
    __syncthreads();
    return true;
}

template <typename T, int kFmt, int Q>
__global__ void __launch_bounds__(kWideThreads, 2)
topk_wide_kernel(const T *__restrict__ logits, int32_t cols, int64_t row_stride, int32_t k,
                 int32_t *__restrict__ out_idx, T *__restrict__ out_val, int32_t *__restrict__ out_count,
                 uint32_t *__restrict__ out_mask)
{
    using F = WideFormat<T, kFmt>;
    extern __shared__ __align__(16) unsigned char wide_dsmem[];
    WideSmem &sm = *reinterpret_cast<WideSmem *>(wide_dsmem);
    const int tid = threadIdx.x;
    const int64_t r = blockIdx.x;
    const T *row = logits + r * row_stride;
    // while the previous kernel on the stream ends: the row's first batch of
    // whole vectors toward L2 (a hint only: L2 is where device memory is
    // coherent, so values that kernel writes are still read after the wait)
    if (tid == 0) {
        const int32_t h0 = wide_head(row, cols);
        const int32_t n = min((cols - h0) / (16 / (int)sizeof(T)), kWideUnroll * kWideThreads);
        l2_prefetch_vecs(reinterpret_cast<const uint4 *>(row + h0), n);
    }
    // one CTA per row: the next launch is placed as this one's CTAs finish
    // (scheduled early, its CTAs would crowd the SMs still running rows)
    grid_dependency_wait_only();
    if (tid == 0) {
        sm.n_ent = 0;
        sm.flags = 0;
        sm.nnz = 0;
        sm.kmax = 0;
        sm.n_list = 0;
    }

    // ---- pass 1: each thread's Q largest vector maxima (a vector's largest
    // key: distinct vectors, distinct elements, so a warp's j-th largest kept
    // maximum still has j elements at or above it), the mask, the count of
    // numbers, and the table of maxima.
    using FK = WideKeys<T, kFmt>;
    constexpr int kPer = 16 / (int)sizeof(T);
    constexpr int G = 8 / kPer; // vectors a table entry covers (the thread's consecutive ones)
    uint32_t t[Q];
#pragma unroll
    for (int i = 0; i < Q; ++i) t[i] = 0;
    uint32_t flags = 0, nnz = 0, smx = 0, smn = 0xFFFFFFFFu;
    auto elem1 = [&](int32_t, uint32_t raw) {
        const uint32_t key = wide_key<T, kFmt>(raw);
        flags |= wide_flag<T, kFmt>(raw);
        nnz += key != 0u;
        keep_insert<Q>(t, key);
    };
    // a vector's largest key: its largest raw key, unless that is a NaN's
    // (a positive NaN: the elements are looked at one by one; only negative
    // NaNs: no number) or -0's
    auto vec1 = [&](const uint4 &q) -> uint32_t {
        uint32_t vmx, vmn;
        vector_key_range<T>(q, vmx, vmn);
        if constexpr (sizeof(T) == 2) {
            smx = max_u16x2(smx, vmx);
            smn = min_u16x2(smn, vmn);
        } else {
            smx = max(smx, vmx);
            smn = min(smn, vmn);
        }
        uint32_t vk = hi_key<T>(vmx);
        if (vk > FK::kPosInfKey) {
            vk = 0;
            vector_elems<T>(q, 0, [&](int32_t, uint32_t raw) { vk = max(vk, wide_key<T, kFmt>(raw)); });
        } else if (vk < FK::kNegInfKey) {
            vk = 0;
        } else if (vk == F::kSign - 1u) {
            vk = F::kSign; // -0: +0's key
        }
        keep_insert<Q>(t, vk);
        return vk;
    };
    const int32_t head = wide_head(row, cols);
    for (int32_t c = tid; c < head; c += kWideThreads) elem1(c, (uint32_t)row[c]);
    const int32_t nvec = (cols - head) / kPer;
    const uint4 *v = reinterpret_cast<const uint4 *>(row + head);
    // this thread's vectors: tid + s * threads for positions s < P; table
    // entry tid + w * threads covers positions G w .. G w + G - 1
    const int32_t P = tid < nvec ? (nvec - 1 - tid) / kWideThreads + 1 : 0;
    const int32_t W0 = ((nvec + kWideThreads - 1) / kWideThreads + G - 1) / G;
    const int32_t nent = W0 * kWideThreads;
    const bool use_tbl = nent <= kWideTbl;
    uint32_t pend = 0; // G = 2: the first vector's maximum of an entry
    for (int32_t i = tid, s0 = 0; i < nvec; i += kWideUnroll * kWideThreads, s0 += kWideUnroll) {
        uint4 q[kWideUnroll];
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u)
            if (i + u * kWideThreads < nvec) q[u] = v[i + u * kWideThreads];
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u) {
            if (i + u * kWideThreads < nvec) {
                const uint32_t vk = vec1(q[u]);
                if constexpr (G == 1) {
                    if (use_tbl) sm.tbl[i + u * kWideThreads] = (uint16_t)vk;
                } else if (u & 1) {
                    if (use_tbl) sm.tbl[tid + ((s0 + u) >> 1) * kWideThreads] = (uint16_t)(max(pend, vk) >> 16);
                } else {
                    pend = vk;
                }
            }
        }
    }
    if (use_tbl) {
        if constexpr (G == 2)
            if (P & 1) sm.tbl[tid + (P >> 1) * kWideThreads] = (uint16_t)(pend >> 16);
        for (int32_t w = (P + G - 1) / G; w < W0; ++w) sm.tbl[tid + w * kWideThreads] = 0;
    }
    for (int32_t c = head + nvec * kPer + tid; c < cols; c += kWideThreads) elem1(c, (uint32_t)row[c]);
    const uint32_t nv = (uint32_t)P;
    // infinities show in the extreme keys; only a possible NaN (a key past
    // theirs) needs the thread's vectors again, for the flag and the count
    const uint32_t hk = hi_key<T>(smx), lk = lo_key<T>(smn);
    flags |= (hk == FK::kPosInfKey ? 2u : 0u) | (lk == FK::kNegInfKey ? 4u : 0u);
    uint32_t nan = 0;
    if (hk > FK::kPosInfKey || lk < FK::kNegInfKey) {
        wide_scan2<T, false>(row, cols, elem1, [&](const uint4 &q, int32_t) {
            vector_elems<T>(q, 0, [&](int32_t, uint32_t raw) {
                flags |= wide_flag<T, kFmt>(raw);
                nan += wide_key<T, kFmt>(raw) == 0u;
            });
        });
    }
    nnz += nv * (16u / (uint32_t)sizeof(T)) - nan;
    flags = __reduce_or_sync(0xFFFFFFFFu, flags);
    nnz = __reduce_add_sync(0xFFFFFFFFu, nnz);
    const uint32_t tmax = t[0]; // this thread's largest key
    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, tmax);
    const uint32_t jth = warp_jth<Q, 8 * (int)sizeof(T)>(t, (uint32_t)((k + kWideWarps - 1) / kWideWarps));
    __syncthreads(); // the initialisation above is visible
    if ((tid & 31) == 0) {
        atomicOr(&sm.flags, flags);
        atomicAdd(&sm.nnz, nnz);
        atomicMax(&sm.kmax, wmax);
        sm.warp_b[tid >> 5] = jth;
    }
    __syncthreads();
    const uint32_t total = sm.nnz;
    const int cnt = (int)min((uint32_t)k, total);
    // each warp holds j elements at or above its j-th key, and warps * j >= k:
    // k elements reach the smallest (every number does, when a warp ran out)
    uint32_t bound = 0xFFFFFFFFu;
#pragma unroll
    for (int w = 0; w < kWideWarps; ++w) bound = min(bound, sm.warp_b[w]);
    bound = max(bound, 1u);
    const uint32_t kmax = sm.kmax;

    // ---- pass 2: every element reaching the bound (vectors below it skipped
    // whole; -0's raw key sits just below +0's)
    const uint32_t vfloor = bound == F::kSign ? bound - 1u : bound;
    auto elem2 = [&](int32_t c, uint32_t raw) {
        const uint32_t key = wide_key<T, kFmt>(raw);
        if (key >= bound) {
            const uint32_t slot = atomicAdd(&sm.n_ent, 1u);
            if (slot < (uint32_t)kWideCap) sm.ent[slot] = ((uint64_t)key << 32) | (uint64_t)(~(uint32_t)c);
        }
    };
    bool full = !use_tbl;
    if (use_tbl) {
        // the table's entries that reach the bound, listed (nent / 8 is a
        // multiple of 32: every warp takes whole rounds)
        const uint32_t vf16 = sizeof(T) == 2 ? vfloor : vfloor >> 16;
        const uint32_t vf2 = vf16 | (vf16 << 16);
        const uint4 *tb = reinterpret_cast<const uint4 *>(sm.tbl);
        for (int32_t m = tid; m < nent / 8; m += kWideThreads) {
            const uint4 c = tb[m];
            const uint32_t ge[4] = {__vcmpgeu2(c.x, vf2), __vcmpgeu2(c.y, vf2), __vcmpgeu2(c.z, vf2),
                                    __vcmpgeu2(c.w, vf2)};
            uint32_t hits = 0; // bit i: entry 8 m + i
#pragma unroll
            for (int j = 0; j < 4; ++j) hits |= ((ge[j] & 1u) | ((ge[j] >> 15) & 2u)) << (2 * j);
            if (__any_sync(0xFFFFFFFFu, hits != 0)) {
                uint32_t slot = warp_reserve(__popc(hits), &sm.n_list);
                for (uint32_t h = hits; h != 0; h &= h - 1, ++slot)
                    if (slot < (uint32_t)kWideList) sm.list[slot] = (uint32_t)(8 * m + __ffs(h) - 1);
            }
        }
        __syncthreads();
        const uint32_t nl = sm.n_list;
        full = nl > (uint32_t)kWideList;
        if (!full) {
            // their vectors, four loads of a thread issued before any is used;
            // a warp reserves the slots of its entries at once
            constexpr int X = 4 / G;
            for (int32_t j0 = 0; j0 < (int32_t)nl; j0 += X * kWideThreads) {
                uint4 q[X * G];
                int32_t vi[X * G];
#pragma unroll
                for (int x = 0; x < X; ++x) {
                    const int32_t j = j0 + tid + x * kWideThreads;
                    const uint32_t e = j < (int32_t)nl ? sm.list[j] : 0xFFFFFFFFu;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        int32_t idx = -1;
                        if (e != 0xFFFFFFFFu) {
                            idx = (int32_t)(e % kWideThreads) + ((int32_t)(e / kWideThreads) * G + g) * kWideThreads;
                            if (idx >= nvec) idx = -1;
                        }
                        vi[x * G + g] = idx;
                        if (idx >= 0) q[x * G + g] = v[idx];
                    }
                }
#pragma unroll
                for (int x = 0; x < X * G; ++x) {
                    uint32_t keys[kPer];
                    uint32_t c = 0;
                    if (vi[x] >= 0) {
                        int32_t at = 0;
                        vector_elems<T>(q[x], 0, [&](int32_t, uint32_t raw) {
                            keys[at] = wide_key<T, kFmt>(raw);
                            c += keys[at] >= bound;
                            ++at;
                        });
                    }
                    if (__any_sync(0xFFFFFFFFu, c != 0)) {
                        uint32_t slot = warp_reserve(c, &sm.n_ent);
                        if (c != 0) {
                            const int32_t c0 = head + vi[x] * kPer;
#pragma unroll
                            for (int i = 0; i < kPer; ++i) {
                                if (keys[i] >= bound) {
                                    if (slot < (uint32_t)kWideCap)
                                        sm.ent[slot] = ((uint64_t)keys[i] << 32) | (uint64_t)(~(uint32_t)(c0 + i));
                                    ++slot;
                                }
                            }
                        }
                    }
                }
            }
            for (int32_t c = tid; c < head; c += kWideThreads) elem2(c, (uint32_t)row[c]);
            for (int32_t c = head + nvec * kPer + tid; c < cols; c += kWideThreads) elem2(c, (uint32_t)row[c]);
        }
    }
    // otherwise the whole row again: only a thread whose largest key reaches
    // the bound holds an element that does; the others skip the second read
    if (full && tmax >= bound) {
        wide_scan2<T, true>(row, cols, elem2, [&](const uint4 &q, int32_t c0) {
            uint32_t vmx, vmn;
            vector_key_range<T>(q, vmx, vmn);
            if (hi_key<T>(vmx) >= vfloor) vector_elems<T>(q, c0, elem2);
        });
    }
    __syncthreads();
    const uint32_t n = sm.n_ent;
    const uint64_t *res = sm.ent;
    if (n <= (uint32_t)kWideThreads) {
        // few: an entry's place is the number of larger entries (all distinct)
        if (tid < (int)n) {
            const uint64_t x = sm.ent[tid];
            uint32_t rank = 0;
            for (uint32_t u = 0; u < n; ++u) rank += sm.ent[u] > x;
            sm.sorted[rank] = x;
        }
        __syncthreads();
        res = sm.sorted;
    } else if (n > 1024u && n <= (uint32_t)kWideCap &&
               wide_select_top<T>(sm, n, k, reinterpret_cast<uint64_t *>(sm.tbl))) {
        // the k largest of more than 1024 entries selected first (k <= 1024):
        // ranked directly, or one 1024-entry sort instead of one of n padded
        uint64_t *sel = reinterpret_cast<uint64_t *>(sm.tbl);
        if (k <= kWideThreads) {
            if (tid < k) {
                const uint64_t x = sel[tid];
                uint32_t rank = 0;
                for (int u = 0; u < k; ++u) rank += sel[u] > x;
                sm.sorted[rank] = x;
            }
            __syncthreads();
            res = sm.sorted;
        } else {
            for (int i = k + tid; i < 1024; i += kWideThreads) sel[i] = 0; // pads sort last
            __syncthreads();
            res = wide_sort<2>(sel, sm.ent, k);
        }
    } else if (n <= (uint32_t)kWideCap) {
        int pn = 1024;
        while (pn < (int)n) pn <<= 1;
        for (int i = (int)n + tid; i < pn; i += kWideThreads) sm.ent[i] = 0; // pads sort last
        __syncthreads();
        // the table is free now: the merges' second buffer
        uint64_t *u = reinterpret_cast<uint64_t *>(sm.tbl);
        if (pn == 1024) res = wide_sort<2>(sm.ent, u, k);
        else if (pn == 2048) res = wide_sort<4>(sm.ent, u, k);
        else res = wide_sort<8>(sm.ent, u, k);
    } else {
        __syncthreads(); // every thread has read n before n_ent is reused below
        // ---- heavy ties: K* by a 16-ary search on counts, kmax + 1 counts 0
        uint64_t lo = bound, hi = (uint64_t)kmax + 1u; // count(>= lo) >= k > count(>= hi)
        while (hi - lo > 1) {
            const uint64_t step = (hi - lo + 15) / 16;
            uint32_t c[15];
#pragma unroll
            for (int j = 0; j < 15; ++j) c[j] = 0;
            wide_scan(row, cols, [&](int32_t, uint32_t raw) {
                const uint64_t key = wide_key<T, kFmt>(raw);
#pragma unroll
                for (int j = 0; j < 15; ++j) c[j] += key >= lo + (uint64_t)(j + 1) * step;
            });
            uint64_t nlo = lo, nhi = hi;
            for (int j = 0; j < 15; ++j) {
                const uint64_t t = lo + (uint64_t)(j + 1) * step;
                const uint32_t cj = wide_block_sum(c[j], sm.red); // every thread, every j
                if (t < hi) {
                    if (cj >= (uint32_t)k) nlo = t;
                    else if (t < nhi) nhi = t;
                }
            }
            lo = nlo;
            hi = nhi;
        }
        const uint32_t kstar = (uint32_t)lo;
        // entries above K*: fewer than k, any order
        if (tid == 0) sm.n_ent = 0;
        __syncthreads();
        wide_scan(row, cols, [&](int32_t c, uint32_t raw) {
            const uint32_t key = wide_key<T, kFmt>(raw);
            if (key > kstar) {
                const uint32_t slot = atomicAdd(&sm.n_ent, 1u);
                sm.ent[slot] = ((uint64_t)key << 32) | (uint64_t)(~(uint32_t)c);
            }
        });
        __syncthreads();
        const uint32_t above = sm.n_ent;
        const uint32_t need = (uint32_t)k - above;
        // ties at K* in column order: each thread a contiguous column range
        const int32_t span = (cols + kWideThreads - 1) / kWideThreads;
        const int32_t c0 = min(cols, tid * span), c1 = min(cols, c0 + span);
        uint32_t ties = 0;
        for (int32_t c = c0; c < c1; ++c) ties += wide_key<T, kFmt>((uint32_t)row[c]) == kstar;
        // exclusive scan of ties over threads (thread order = column order)
        const int lane = tid & 31, warp = tid >> 5;
        uint32_t incl = ties;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += u;
        }
        __syncthreads();
        if (lane == 31) sm.red[warp] = incl;
        __syncthreads();
        uint32_t rank = incl - ties;
        for (int w = 0; w < warp; ++w) rank += sm.red[w];
        for (int32_t c = c0; c < c1 && rank < need; ++c) {
            if (wide_key<T, kFmt>((uint32_t)row[c]) == kstar) {
                sm.ent[above + rank] = ((uint64_t)kstar << 32) | (uint64_t)(~(uint32_t)c);
                ++rank;
            }
        }
        __syncthreads();
        int pn = 1;
        while (pn < k) pn <<= 1;
        for (int i = k + tid; i < pn; i += kWideThreads) sm.ent[i] = 0;
        __syncthreads();
        bitonic_desc(sm.ent, pn);
    }

    // ---- the row: the first cnt entries, original bits re-read by column
    grid_dependents_go();
    for (int i = tid; i < k; i += kWideThreads) {
        if (i < cnt) {
            const int32_t c = (int32_t)(~(uint32_t)res[i]);
            out_idx[r * k + i] = c;
            out_val[r * k + i] = row[c];
        } else {
            out_idx[r * k + i] = -1;
            out_val[r * k + i] = (T)F::kEmpty;
        }
    }
    if (tid == 0) {
        out_count[r] = cnt;
        out_mask[r] = sm.flags;
    }
}

// ---------------------------------------------------------------- host side

constexpr size_t kStreamSmemBytes =
    (size_t)kStages * kChunkVecs * 16 + sizeof(SmemCore) + (size_t)kPendCap * sizeof(uint64_t);

struct DeviceInfo {
    bool ready = false;
    int status = TF_TOPK_OK;
    int sm_count = 0;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_device_mutex;
thread_local int t_last_cuda_error = 0;

int fail_cuda(cudaError_t e)
{
    t_last_cuda_error = (int)e;
    return TF_TOPK_ERR_CUDA;
}

// Per-device set-up, once: check the architecture, allow the 16-CTA cluster and
// the stream kernel's shared-memory ring.
int device_setup(int *dev_out, int *sm_count)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return TF_TOPK_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_device_mutex);
    DeviceInfo &d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail_cuda(e);
        if (major != 10 || minor != 3) {
            d.status = TF_TOPK_ERR_DEVICE;
        } else {
            e = cudaFuncSetAttribute(topk_cluster_kernel<16, kBf16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(topk_cluster_kernel<16, TF_TOPK_DTYPE_F16>,
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(topk_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kStreamSmemBytes);
            if (e != cudaSuccess) return fail_cuda(e);
            d.status = TF_TOPK_OK;
        }
        d.sm_count = sms;
        d.ready = true;
    }
    *dev_out = dev;
    *sm_count = d.sm_count;
    return d.status;
}

// Scratch of the stream kernel: two partial lists and one ticket per CTA.
// One area per (device, stream) so that calls on different streams never share
// it; calls on one stream are ordered by the stream.  Every launch clears the
// tickets it uses first (stream-ordered), so a launch cut short by a wait that
// ran out cannot leave a later one with half-counted tickets.
struct Scratch {
    uint64_t *partials = nullptr;
    uint32_t *tickets = nullptr;
    int64_t ctas = 0;
};

struct ScratchKey {
    int dev;
    cudaStream_t stream;
    std::thread::id thread; // only set for the per-thread default stream
    bool operator<(const ScratchKey &o) const
    {
        if (dev != o.dev) return dev < o.dev;
        if (stream != o.stream) return stream < o.stream;
        return thread < o.thread;
    }
};

std::mutex g_scratch_mutex;
std::map<ScratchKey, Scratch> g_scratch;

size_t partial_bytes(int64_t ctas) { return (size_t)ctas * 2 * (kMaxK + 1) * sizeof(uint64_t); }

int get_scratch(int dev, cudaStream_t stream, int64_t ctas, Scratch **out)
{
    ScratchKey key{dev, stream, std::thread::id()};
    if (stream == cudaStreamPerThread) key.thread = std::this_thread::get_id();
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    Scratch &s = g_scratch[key];
    if (s.ctas < ctas) {
        if (s.partials) {
            // the old area may still be in use by work queued on this stream
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return fail_cuda(e);
            cudaFree(s.partials);
            cudaFree(s.tickets);
            s = Scratch();
        }
        cudaError_t e = cudaMalloc(&s.partials, partial_bytes(ctas));
        if (e == cudaSuccess) e = cudaMalloc(&s.tickets, (size_t)ctas * sizeof(uint32_t));
        if (e == cudaSuccess) e = cudaMemsetAsync(s.tickets, 0, (size_t)ctas * sizeof(uint32_t), stream);
        if (e != cudaSuccess) {
            cudaFree(s.partials);
            cudaFree(s.tickets);
            s = Scratch();
            return fail_cuda(e);
        }
        s.ctas = ctas;
    }
    *out = &s;
    return TF_TOPK_OK;
}

int validate(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
             const int32_t *out_idx, const uint16_t *out_val, const int32_t *out_count,
             const uint32_t *out_mask)
{
    if (k < 1 || k > kMaxK) return TF_TOPK_ERR_K;
    if (rows < 0 || cols < 1 || row_stride < cols || cols > (int64_t)INT32_MAX - 64)
        return TF_TOPK_ERR_SHAPE;
    if (rows > 0 && row_stride > INT64_MAX / rows) return TF_TOPK_ERR_SHAPE;
    if (rows == 0) return TF_TOPK_OK;
    if (!logits || !out_idx || !out_val || !out_count || !out_mask) return TF_TOPK_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(logits) & 1) || (reinterpret_cast<uintptr_t>(out_val) & 1) ||
        (reinterpret_cast<uintptr_t>(out_idx) & 3) || (reinterpret_cast<uintptr_t>(out_count) & 3) ||
        (reinterpret_cast<uintptr_t>(out_mask) & 3))
        return TF_TOPK_ERR_ALIGN;
    return TF_TOPK_OK;
}

// Vectors per row in the stream kernel's rows x vectors space: enough for any
// alignment of the row start.
int32_t vectors_per_row(int64_t cols) { return (int32_t)((cols + 14) >> 3); }

// Stream-plan geometry: the range each CTA gets, and the CTA count.
void stream_geometry(int64_t rows, int64_t cols, int sm_count, int64_t *per_out, int64_t *ctas_out)
{
    const int64_t nvr = vectors_per_row(cols);
    const int64_t total = rows * nvr;
    const int64_t slots = (int64_t)sm_count * kStreamCtasPerSm;
    int64_t per = (total + slots - 1) / slots;
    per = per < kMinVecsPerCta ? kMinVecsPerCta : per;
    // a row meets <= kMaxPieces CTAs, after range starts move by up to 2 * kThreads
    const int64_t min_piece = (nvr + kMaxPieces - 2) / (kMaxPieces - 1) + 2 * kThreads;
    per = per < min_piece ? min_piece : per;
    *per_out = per;
    *ctas_out = (total + per - 1) / per;
}

// The plan tf_topk_bf16 uses.  Measured on GB300 over widths 4096..248320
// and rows 1..2048: the cluster kernel is the fastest everywhere.  With at
// least one row per SM, one CTA per row (SINGLE) when a row is at most one
// chunk, or when two spans a row would take three waves or more of the
// kernel's four CTAs an SM (1024 x 248320: 88.0 -> 83.1 us; 1024 x 4096:
// 25.6 -> 13.8 us); else two spans a row.  With fewer rows, the span count
// that brings the grid to about two CTAs per SM, but no span narrower than
// half a chunk (a whole chunk for k > 32, whose merges cost more), down to
// one span.
int32_t pick_plan(int64_t rows, int64_t cols, int32_t k, int sm_count)
{
    if (rows >= sm_count) {
        const int64_t slots = (int64_t)kClusterCtasPerSm * sm_count;
        if (cols <= kChunkCols || 2 * rows >= 3 * slots) return TF_TOPK_PLAN_SINGLE;
        return TF_TOPK_PLAN_CLUSTER2;
    }
    const int64_t min_span = k > 32 ? kChunkCols : kChunkCols / 2;
    int s = 2;
    while (s < kMaxSpans && rows * s < 2 * (int64_t)sm_count) s *= 2;
    while (s > 1 && cols / s < min_span) s /= 2;
    return s == 1 ? TF_TOPK_PLAN_SINGLE : s;
}

template <int S, int kFmt = kBf16>
cudaError_t launch_cluster(const uint16_t *logits, int64_t rows, int32_t cols, int64_t row_stride, int32_t k,
                           int32_t *out_idx, uint16_t *out_val, int32_t *out_count, uint32_t *out_mask,
                           cudaStream_t stream, int sm_count)
{
    const int64_t max_rows = (int64_t)INT32_MAX / S;
    for (int64_t r0 = 0; r0 < rows; r0 += max_rows) {
        const int64_t nr = rows - r0 < max_rows ? rows - r0 : max_rows;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(nr * S), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        auto kernel = topk_cluster_kernel<S, kFmt, 1>;
        if constexpr (S == 2)
            if (nr * S <= (int64_t)kClusterCtasPerSm * sm_count) kernel = topk_cluster_kernel<S, kFmt, 2>;
        cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, logits + r0 * row_stride, cols,
                                           row_stride, k, out_idx + r0 * k, out_val + r0 * k,
                                           out_count + r0, out_mask + r0);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int launch_stream(int dev, int sm_count, const uint16_t *logits, int64_t rows, int64_t cols,
                  int64_t row_stride, int32_t k, int32_t *out_idx, uint16_t *out_val, int32_t *out_count,
                  uint32_t *out_mask, cudaStream_t stream)
{
    const int32_t nvr = vectors_per_row(cols);
    {
        const int64_t r0 = 0, nr = rows;
        int64_t per = 0, ctas = 0;
        stream_geometry(nr, cols, sm_count, &per, &ctas);
        Scratch *sc = nullptr;
        const int st = get_scratch(dev, stream, ctas, &sc);
        if (st != TF_TOPK_OK) return st;
        uint64_t *partials = sc->partials;
        uint32_t *tickets = sc->tickets;
        // a launch whose wait ran out leaves its split rows' tickets half
        // counted: start every launch from zero
        const cudaError_t em = cudaMemsetAsync(tickets, 0, (size_t)ctas * sizeof(uint32_t), stream);
        if (em != cudaSuccess) return fail_cuda(em);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ctas, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kStreamSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, topk_stream_kernel, logits + r0 * row_stride, (int32_t)cols,
                                           row_stride, k, nvr, nr * nvr, per, out_idx + r0 * k, out_val + r0 * k,
                                           out_count + r0, out_mask + r0, partials, tickets);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return fail_cuda(e);
    }
    return TF_TOPK_OK;
}

int run(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k, int32_t *out_idx,
        uint16_t *out_val, int32_t *out_count, uint32_t *out_mask, int32_t plan, void *stream)
{
    int st = validate(logits, rows, cols, row_stride, k, out_idx, out_val, out_count, out_mask);
    if (st != TF_TOPK_OK) return st;
    if (plan != TF_TOPK_PLAN_AUTO && plan != TF_TOPK_PLAN_SINGLE && plan != TF_TOPK_PLAN_CLUSTER2 &&
        plan != TF_TOPK_PLAN_CLUSTER4 && plan != TF_TOPK_PLAN_CLUSTER8 && plan != TF_TOPK_PLAN_CLUSTER16 &&
        plan != TF_TOPK_PLAN_STREAM)
        return TF_TOPK_ERR_PLAN;
    if (rows == 0) return TF_TOPK_OK;
    int dev = 0, sm_count = 0;
    st = device_setup(&dev, &sm_count);
    if (st != TF_TOPK_OK) return st;
    if (plan == TF_TOPK_PLAN_AUTO) plan = pick_plan(rows, cols, k, sm_count);
    const uint16_t *x = static_cast<const uint16_t *>(logits);
    const int32_t c = (int32_t)cols;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    switch (plan) {
    case TF_TOPK_PLAN_SINGLE:
        e = launch_cluster<1>(x, rows, c, row_stride, k, out_idx, out_val, out_count, out_mask, s, sm_count);
        break;
    case TF_TOPK_PLAN_STREAM:
        return launch_stream(dev, sm_count, x, rows, cols, row_stride, k, out_idx, out_val, out_count, out_mask, s);
    case TF_TOPK_PLAN_CLUSTER2:
        e = launch_cluster<2>(x, rows, c, row_stride, k, out_idx, out_val, out_count, out_mask, s, sm_count);
        break;
    case TF_TOPK_PLAN_CLUSTER4:
        e = launch_cluster<4>(x, rows, c, row_stride, k, out_idx, out_val, out_count, out_mask, s, sm_count);
        break;
    case TF_TOPK_PLAN_CLUSTER8:
        e = launch_cluster<8>(x, rows, c, row_stride, k, out_idx, out_val, out_count, out_mask, s, sm_count);
        break;
    default:
        e = launch_cluster<16>(x, rows, c, row_stride, k, out_idx, out_val, out_count, out_mask, s, sm_count);
        break;
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e);
    return TF_TOPK_OK;
}

// tf_topk_bf16_noalloc: the device address of g_noalloc_scratch, looked up
// once per device (with that device current) and kept.
std::mutex g_noalloc_mutex;
uint64_t *g_noalloc_addr[kMaxDevices];

int noalloc_scratch(int dev, uint64_t **out)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return fail_cuda(e);
        g_noalloc_addr[dev] = static_cast<uint64_t *>(p);
    }
    *out = g_noalloc_addr[dev];
    return TF_TOPK_OK;
}

// The stream plan with its scratch in the static array: no allocation, no free.
int run_noalloc(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                int32_t *out_idx, uint16_t *out_val, int32_t *out_count, uint32_t *out_mask, void *stream)
{
    int st = validate(logits, rows, cols, row_stride, k, out_idx, out_val, out_count, out_mask);
    if (st != TF_TOPK_OK) return st;
    if (rows == 0) return TF_TOPK_OK;
    int dev = 0, sm_count = 0;
    st = device_setup(&dev, &sm_count);
    if (st != TF_TOPK_OK) return st;
    int64_t per = 0, ctas = 0;
    stream_geometry(rows, cols, sm_count, &per, &ctas);
    if (ctas > TF_TOPK_NOALLOC_MAX_CTAS) return TF_TOPK_ERR_SCRATCH;
    uint64_t *base = nullptr;
    st = noalloc_scratch(dev, &base);
    if (st != TF_TOPK_OK) return st;
    uint64_t *partials = base;
    uint32_t *tickets = reinterpret_cast<uint32_t *>(base + kNoAllocListWords);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the previous call may have been cut short with tickets half counted
    cudaError_t e = cudaMemsetAsync(tickets, 0, (size_t)ctas * sizeof(uint32_t), s);
    if (e != cudaSuccess) return fail_cuda(e);
    const int32_t nvr = vectors_per_row(cols);
    topk_stream_kernel<<<(unsigned)ctas, kThreads, kStreamSmemBytes, s>>>(
        static_cast<const uint16_t *>(logits), (int32_t)cols, row_stride, k, nvr, rows * nvr, per, out_idx,
        out_val, out_count, out_mask, partials, tickets);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e);
    return TF_TOPK_OK;
}

// tf_topk_merge_bf16: argument checks, then one CTA per row (in blocks of at
// most 2^31 - 1 rows per launch).
int run_merge(const int32_t *in_idx, const uint16_t *in_val, const int32_t *in_count, const uint32_t *in_mask,
              int64_t rows, int32_t shards, int32_t k_in, const int64_t *shard_offset, int32_t k, int32_t *out_idx,
              uint16_t *out_val, int32_t *out_count, uint32_t *out_mask, void *stream)
{
    if (k < 1 || k > kMaxK || k_in < 1 || k_in > kMaxK) return TF_TOPK_ERR_K;
    if (rows < 0 || shards < 1 || shards > TF_TOPK_MAX_SHARDS) return TF_TOPK_ERR_SHAPE;
    if (rows == 0) return TF_TOPK_OK;
    if (!in_idx || !in_val || !in_count || !in_mask || !shard_offset || !out_idx || !out_val || !out_count ||
        !out_mask)
        return TF_TOPK_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(in_idx) & 3) || (reinterpret_cast<uintptr_t>(in_val) & 1) ||
        (reinterpret_cast<uintptr_t>(in_count) & 3) || (reinterpret_cast<uintptr_t>(in_mask) & 3) ||
        (reinterpret_cast<uintptr_t>(out_idx) & 3) || (reinterpret_cast<uintptr_t>(out_val) & 1) ||
        (reinterpret_cast<uintptr_t>(out_count) & 3) || (reinterpret_cast<uintptr_t>(out_mask) & 3))
        return TF_TOPK_ERR_ALIGN;
    MergeShards off;
    for (int s = 0; s < shards; ++s) {
        if (shard_offset[s] < 0 || shard_offset[s] > (int64_t)INT32_MAX) return TF_TOPK_ERR_SHAPE;
        off.offset[s] = shard_offset[s];
    }
    int dev = 0, sm_count = 0;
    int st = device_setup(&dev, &sm_count);
    if (st != TF_TOPK_OK) return st;
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    const int64_t max_rows = (int64_t)INT32_MAX;
    for (int64_t r0 = 0; r0 < rows; r0 += max_rows) {
        const int64_t nr = rows - r0 < max_rows ? rows - r0 : max_rows;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)nr, 1, 1);
        cfg.blockDim = dim3(kMergeThreads, 1, 1);
        cfg.stream = strm;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // the row block's cells: shard s, row r at s * rows + r (k_in entries each)
        cudaError_t e = cudaLaunchKernelEx(&cfg, topk_merge_kernel, in_idx + r0 * k_in, in_val + r0 * k_in,
                                           in_count + r0, in_mask + r0, rows, shards, k_in, off, k,
                                           out_idx + r0 * k, out_val + r0 * k, out_count + r0, out_mask + r0);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return fail_cuda(e);
    }
    return TF_TOPK_OK;
}

// tf_topk_nucleus / tf_topk_nucleus_bf16: argument checks, then one warp per row.
template <typename T, int kFmt>
cudaError_t launch_nucleus(const T *val, const int32_t *count, int64_t r0, int64_t nr, int32_t k, float temperature,
                           float top_p, float *out_prob, int32_t *out_keep, cudaStream_t strm)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((nr + kNucleusWarps - 1) / kNucleusWarps), 1, 1);
    cfg.blockDim = dim3(kNucleusWarps * 32, 1, 1);
    cfg.stream = strm;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_nucleus_kernel<T, kFmt>, val + r0 * k, count + r0, nr, k, temperature,
                              top_p, out_prob + r0 * k, out_keep + r0);
}

int run_nucleus(const void *val, int32_t dtype, const int32_t *count, int64_t rows, int32_t k, float temperature,
                float top_p, float *out_prob, int32_t *out_keep, void *stream)
{
    if (dtype != TF_TOPK_DTYPE_BF16 && dtype != TF_TOPK_DTYPE_F16 && dtype != TF_TOPK_DTYPE_F32)
        return TF_TOPK_ERR_DTYPE;
    if (k < 1 || k > kMaxK) return TF_TOPK_ERR_K;
    if (rows < 0) return TF_TOPK_ERR_SHAPE;
    if (!(temperature >= 0.f) || std::isinf(temperature) || !(top_p > 0.f && top_p <= 1.f)) return TF_TOPK_ERR_ARG;
    if (rows == 0) return TF_TOPK_OK;
    if (!val || !count || !out_prob || !out_keep) return TF_TOPK_ERR_NULL;
    const uintptr_t esz = dtype == TF_TOPK_DTYPE_F32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(val) & (esz - 1)) || (reinterpret_cast<uintptr_t>(count) & 3) ||
        (reinterpret_cast<uintptr_t>(out_prob) & 3) || (reinterpret_cast<uintptr_t>(out_keep) & 3))
        return TF_TOPK_ERR_ALIGN;
    int dev = 0, sm_count = 0;
    int st = device_setup(&dev, &sm_count);
    if (st != TF_TOPK_OK) return st;
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    const int64_t max_rows = (int64_t)INT32_MAX * kNucleusWarps;
    for (int64_t r0 = 0; r0 < rows; r0 += max_rows) {
        const int64_t nr = rows - r0 < max_rows ? rows - r0 : max_rows;
        cudaError_t e;
        if (dtype == TF_TOPK_DTYPE_F32)
            e = launch_nucleus<uint32_t, TF_TOPK_DTYPE_F32>(static_cast<const uint32_t *>(val), count, r0, nr, k,
                                                            temperature, top_p, out_prob, out_keep, strm);
        else if (dtype == TF_TOPK_DTYPE_F16)
            e = launch_nucleus<uint16_t, TF_TOPK_DTYPE_F16>(static_cast<const uint16_t *>(val), count, r0, nr, k,
                                                            temperature, top_p, out_prob, out_keep, strm);
        else
            e = launch_nucleus<uint16_t, TF_TOPK_DTYPE_BF16>(static_cast<const uint16_t *>(val), count, r0, nr, k,
                                                             temperature, top_p, out_prob, out_keep, strm);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return fail_cuda(e);
    }
    return TF_TOPK_OK;
}

// tf_topk_select with the wide kernel: one CTA per row, in blocks of at most
// 2^31 - 1 rows per launch.
template <typename T, int kFmt, int Q>
int launch_wide(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k, int32_t *out_idx,
                void *out_val, int32_t *out_count, uint32_t *out_mask, cudaStream_t strm)
{
    // per device, once (setting the attribute twice from racing threads is harmless)
    static std::atomic<bool> attr_done[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return TF_TOPK_ERR_DEVICE;
    if (!attr_done[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(topk_wide_kernel<T, kFmt, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(WideSmem));
        if (e != cudaSuccess) return fail_cuda(e);
        attr_done[dev].store(true, std::memory_order_release);
    }
    const T *x = static_cast<const T *>(logits);
    T *ov = static_cast<T *>(out_val);
    const int64_t max_rows = (int64_t)INT32_MAX;
    for (int64_t r0 = 0; r0 < rows; r0 += max_rows) {
        const int64_t nr = rows - r0 < max_rows ? rows - r0 : max_rows;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)nr, 1, 1);
        cfg.blockDim = dim3(kWideThreads, 1, 1);
        cfg.dynamicSmemBytes = sizeof(WideSmem);
        cfg.stream = strm;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, topk_wide_kernel<T, kFmt, Q>, x + r0 * row_stride, (int32_t)cols, row_stride, k,
                               out_idx + r0 * k, ov + r0 * k, out_count + r0, out_mask + r0);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return fail_cuda(e);
    }
    return TF_TOPK_OK;
}

// tf_topk_select / tf_topk_select_with_plan: guards, then bf16 with k <= 64 on
// the fast plans (AUTO unless a plan is named), everything else on the wide
// kernel.
int run_select(const void *logits, int32_t dtype, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
               int32_t *out_idx, void *out_val, int32_t *out_count, uint32_t *out_mask, int32_t plan, void *stream)
{
    if (dtype != TF_TOPK_DTYPE_BF16 && dtype != TF_TOPK_DTYPE_F16 && dtype != TF_TOPK_DTYPE_F32)
        return TF_TOPK_ERR_DTYPE;
    if (k < 1 || k > kWideMaxK) return TF_TOPK_ERR_K;
    if (rows < 0 || cols < 1 || row_stride < cols || cols > (int64_t)INT32_MAX - 64) return TF_TOPK_ERR_SHAPE;
    if (rows > 0 && row_stride > INT64_MAX / rows) return TF_TOPK_ERR_SHAPE;
    const bool cluster_plan = plan == TF_TOPK_PLAN_SINGLE || plan == TF_TOPK_PLAN_CLUSTER2 ||
                              plan == TF_TOPK_PLAN_CLUSTER4 || plan == TF_TOPK_PLAN_CLUSTER8 ||
                              plan == TF_TOPK_PLAN_CLUSTER16;
    if (plan != TF_TOPK_PLAN_AUTO && plan != TF_TOPK_PLAN_WIDE &&
        !(k <= kMaxK && (dtype == TF_TOPK_DTYPE_BF16 || (dtype == TF_TOPK_DTYPE_F16 && cluster_plan))))
        return TF_TOPK_ERR_PLAN; // bf16: every plan; fp16: SINGLE and the cluster plans; both with k <= 64
    if (rows == 0) return TF_TOPK_OK;
    if (!logits || !out_idx || !out_val || !out_count || !out_mask) return TF_TOPK_ERR_NULL;
    const uintptr_t esz = dtype == TF_TOPK_DTYPE_F32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(logits) & (esz - 1)) || (reinterpret_cast<uintptr_t>(out_val) & (esz - 1)) ||
        (reinterpret_cast<uintptr_t>(out_idx) & 3) || (reinterpret_cast<uintptr_t>(out_count) & 3) ||
        (reinterpret_cast<uintptr_t>(out_mask) & 3))
        return TF_TOPK_ERR_ALIGN;
    if (dtype == TF_TOPK_DTYPE_BF16 && k <= kMaxK && plan != TF_TOPK_PLAN_WIDE)
        return run(logits, rows, cols, row_stride, k, out_idx, static_cast<uint16_t *>(out_val), out_count,
                   out_mask, plan, stream);
    int dev = 0, sm_count = 0;
    const int st = device_setup(&dev, &sm_count);
    if (st != TF_TOPK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == TF_TOPK_DTYPE_F32 && k <= kMaxK && plan == TF_TOPK_PLAN_AUTO)
        return tf_topk_internal_select_f32(logits, rows, cols, row_stride, k, out_idx, out_val, out_count, out_mask,
                                           sm_count, stream);
    if (dtype == TF_TOPK_DTYPE_F16 && k <= kMaxK && plan != TF_TOPK_PLAN_WIDE) {
        // fp16 shares bf16's key map: the cluster plans, with fp16's special values
        int p = plan == TF_TOPK_PLAN_AUTO ? pick_plan(rows, cols, k, sm_count) : plan;
        const uint16_t *x = static_cast<const uint16_t *>(logits);
        uint16_t *ov = static_cast<uint16_t *>(out_val);
        const int32_t c = (int32_t)cols;
        cudaError_t e = cudaSuccess;
        switch (p) {
        case TF_TOPK_PLAN_SINGLE:
            e = launch_cluster<1, TF_TOPK_DTYPE_F16>(x, rows, c, row_stride, k, out_idx, ov, out_count, out_mask, s, sm_count);
            break;
        case TF_TOPK_PLAN_CLUSTER2:
            e = launch_cluster<2, TF_TOPK_DTYPE_F16>(x, rows, c, row_stride, k, out_idx, ov, out_count, out_mask, s, sm_count);
            break;
        case TF_TOPK_PLAN_CLUSTER4:
            e = launch_cluster<4, TF_TOPK_DTYPE_F16>(x, rows, c, row_stride, k, out_idx, ov, out_count, out_mask, s, sm_count);
            break;
        case TF_TOPK_PLAN_CLUSTER8:
            e = launch_cluster<8, TF_TOPK_DTYPE_F16>(x, rows, c, row_stride, k, out_idx, ov, out_count, out_mask, s, sm_count);
            break;
        case TF_TOPK_PLAN_CLUSTER16:
            e = launch_cluster<16, TF_TOPK_DTYPE_F16>(x, rows, c, row_stride, k, out_idx, ov, out_count, out_mask,
                                                      s, sm_count);
            break;
        default: // not reached (AUTO and the accepted plans are above): the wide kernel
            p = TF_TOPK_PLAN_WIDE;
            break;
        }
        if (p != TF_TOPK_PLAN_WIDE) {
            if (e == cudaSuccess) e = cudaGetLastError();
            if (e != cudaSuccess) return fail_cuda(e);
            return TF_TOPK_OK;
        }
    }
    switch (dtype) {
    case TF_TOPK_DTYPE_BF16:
        return launch_wide<uint16_t, TF_TOPK_DTYPE_BF16, kWideKeep>(logits, rows, cols, row_stride, k, out_idx,
                                                                    out_val, out_count, out_mask, s);
    case TF_TOPK_DTYPE_F16:
        return launch_wide<uint16_t, TF_TOPK_DTYPE_F16, kWideKeep>(logits, rows, cols, row_stride, k, out_idx,
                                                                   out_val, out_count, out_mask, s);
    default:
        return launch_wide<uint32_t, TF_TOPK_DTYPE_F32, kWideKeep>(logits, rows, cols, row_stride, k, out_idx,
                                                                   out_val, out_count, out_mask, s);
    }
}

} // namespace

// Shared with the head entry points (a separate translation unit).
int tf_topk_internal_fail_cuda(int cuda_error) { return fail_cuda(static_cast<cudaError_t>(cuda_error)); }
uint32_t tf_topk_internal_head_fault_take();

extern "C" {

int tf_topk_bf16(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                 int32_t *out_idx, uint16_t *out_val, int32_t *out_count, uint32_t *out_nonfinite_mask,
                 void *stream)
{
    return run(logits, rows, cols, row_stride, k, out_idx, out_val, out_count, out_nonfinite_mask,
               TF_TOPK_PLAN_AUTO, stream);
}

int tf_topk_bf16_with_plan(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                           int32_t *out_idx, uint16_t *out_val, int32_t *out_count,
                           uint32_t *out_nonfinite_mask, int32_t plan, void *stream)
{
    return run(logits, rows, cols, row_stride, k, out_idx, out_val, out_count, out_nonfinite_mask, plan,
               stream);
}

int tf_topk_bf16_noalloc(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                         int32_t *out_idx, uint16_t *out_val, int32_t *out_count, uint32_t *out_nonfinite_mask,
                         void *stream)
{
    return run_noalloc(logits, rows, cols, row_stride, k, out_idx, out_val, out_count, out_nonfinite_mask,
                       stream);
}

int tf_topk_merge_bf16(const int32_t *in_idx, const uint16_t *in_val, const int32_t *in_count,
                       const uint32_t *in_nonfinite_mask, int64_t rows, int32_t shards, int32_t k_in,
                       const int64_t *shard_offset, int32_t k, int32_t *out_idx, uint16_t *out_val,
                       int32_t *out_count, uint32_t *out_nonfinite_mask, void *stream)
{
    return run_merge(in_idx, in_val, in_count, in_nonfinite_mask, rows, shards, k_in, shard_offset, k, out_idx,
                     out_val, out_count, out_nonfinite_mask, stream);
}

int tf_topk_nucleus_bf16(const uint16_t *val, const int32_t *count, int64_t rows, int32_t k, float temperature,
                         float top_p, float *out_prob, int32_t *out_keep, void *stream)
{
    return run_nucleus(val, TF_TOPK_DTYPE_BF16, count, rows, k, temperature, top_p, out_prob, out_keep, stream);
}

int tf_topk_nucleus(const void *val, int32_t dtype, const int32_t *count, int64_t rows, int32_t k, float temperature,
                    float top_p, float *out_prob, int32_t *out_keep, void *stream)
{
    return run_nucleus(val, dtype, count, rows, k, temperature, top_p, out_prob, out_keep, stream);
}

int tf_topk_select(const void *logits, int32_t dtype, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                   int32_t *out_idx, void *out_val, int32_t *out_count, uint32_t *out_nonfinite_mask, void *stream)
{
    return run_select(logits, dtype, rows, cols, row_stride, k, out_idx, out_val, out_count, out_nonfinite_mask,
                      TF_TOPK_PLAN_AUTO, stream);
}

int tf_topk_select_with_plan(const void *logits, int32_t dtype, int64_t rows, int64_t cols, int64_t row_stride,
                             int32_t k, int32_t *out_idx, void *out_val, int32_t *out_count,
                             uint32_t *out_nonfinite_mask, int32_t plan, void *stream)
{
    return run_select(logits, dtype, rows, cols, row_stride, k, out_idx, out_val, out_count, out_nonfinite_mask,
                      plan, stream);
}

int32_t tf_topk_bf16_plan(int64_t rows, int64_t cols, int32_t k)
{
    if (k < 1 || k > kMaxK) return -TF_TOPK_ERR_K;
    if (rows < 0 || cols < 1 || cols > (int64_t)INT32_MAX - 64) return -TF_TOPK_ERR_SHAPE;
    int dev = 0, sm_count = 0;
    const int st = device_setup(&dev, &sm_count);
    if (st != TF_TOPK_OK) return -st;
    return pick_plan(rows, cols, k, sm_count);
}

int tf_topk_device_fault(void)
{
    uint32_t f = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&f, g_fault, sizeof f);
    if (e != cudaSuccess) return -fail_cuda(e);
    const uint32_t fh = tf_topk_internal_head_fault_take();
    if (f == 0) f = fh;
    if (f != 0) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_fault, &zero, sizeof zero);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        // a CTA that gave up may have left a ticket half-counted: reset them all
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        int dev = 0;
        if (e == cudaSuccess) e = cudaGetDevice(&dev);
        for (auto &kv : g_scratch)
            if (e == cudaSuccess && kv.first.dev == dev && kv.second.tickets)
                e = cudaMemset(kv.second.tickets, 0, (size_t)kv.second.ctas * sizeof(uint32_t));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return -fail_cuda(e);
    }
    return (int)f;
}

int32_t tf_topk_bf16_max_k(void) { return kMaxK; }
int32_t tf_topk_select_max_k(void) { return kWideMaxK; }
int32_t tf_topk_bf16_max_spans(void) { return kMaxSpans; }
int32_t tf_topk_bf16_cta_threads(void) { return kThreads; }
int32_t tf_topk_bf16_chunk_columns(void) { return kChunkCols; }

const char *tf_topk_strerror(int status)
{
    switch (status) {
    case TF_TOPK_OK: return "ok";
    case TF_TOPK_ERR_NULL: return "a required pointer is NULL";
    case TF_TOPK_ERR_SHAPE: return "invalid shape (rows, cols or row_stride)";
    case TF_TOPK_ERR_K: return "k out of range (1..TF_TOPK_MAX_K)";
    case TF_TOPK_ERR_ALIGN: return "misaligned pointer";
    case TF_TOPK_ERR_PLAN: return "unknown plan code";
    case TF_TOPK_ERR_DEVICE: return "current device is not compute capability 10.3 (sm_103a)";
    case TF_TOPK_ERR_CUDA: return "CUDA runtime error (see tf_topk_last_cuda_error)";
    case TF_TOPK_ERR_ARG: return "temperature or top_p out of range";
    case TF_TOPK_ERR_DTYPE: return "unknown logit format (TF_TOPK_DTYPE_*)";
    case TF_TOPK_ERR_SCRATCH: return "the launch needs more scratch slots than the static area of "
                                     "tf_topk_bf16_noalloc holds (TF_TOPK_NOALLOC_MAX_CTAS)";
    default: return "unknown status";
    }
}

int tf_topk_last_cuda_error(void) { return t_last_cuda_error; }

} // extern "C"
