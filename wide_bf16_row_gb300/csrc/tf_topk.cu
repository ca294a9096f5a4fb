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
// Design (one kernel template, one launch per call):
//   * A CTA owns one column span of one row.  It streams the span through
//     registers a chunk at a time (kThreads x kVecPerThread 16-byte vectors,
//     coalesced, read once from HBM).
//   * Each bf16 becomes an order-preserving 16-bit key in place (two keys per
//     32-bit register): positive bits b -> b | 0x8000, negative bits b -> ~b.
//     -0 and +0 land on the neighbouring keys 0x7FFF / 0x8000 and are treated
//     as one score wherever a threshold or a comparison is taken.
//   * Prefilter: every thread keeps the max key of its elements; each warp finds
//     the j-th largest of its 32 thread maxima (j = ceil(k / warps)); the
//     minimum T over warps is a value that at least k elements reach, so the
//     chunk's top-k lies in {key >= T}.  Only those candidates (typically a few
//     times k out of 16384) touch shared memory.
//   * The candidates are ranked exactly with a 32-bit composite
//     (key << 16 | ~local column), which is unique, so every rank is distinct.
//     Rows with heavy ties (e.g. all zeros) overflow the candidate buffer and
//     take an exact radix path instead: a binary search for the k-th key, then
//     the lowest columns among the threshold ties, found by a block scan in
//     column order.
//   * A CTA's running list (<= k entries, 64-bit composites holding key,
//     column and the original bits) is merged chunk by chunk.
//   * spans > 1: the CTAs of one row form a thread-block cluster; each pushes
//     its sorted list into the leader CTA's shared memory (distributed shared
//     memory) and the leader merges the lists pairwise (a tournament tree) and
//     writes the row.  spans == 1 is the single-CTA control path.
// There is no global scratch, no atomic on global memory and no spin-wait: the
// only cross-CTA synchronisation is the hardware cluster barrier.

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "tf_topk.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerThread = 8;                     // 16-byte vectors per thread per chunk
constexpr int kChunkVecs = kThreads * kVecPerThread; // 2048 vectors
constexpr int kChunkCols = kChunkVecs * 8;           // 16384 columns
constexpr int kMaxK = TF_TOPK_MAX_K;
constexpr int kMaxSpans = TF_TOPK_MAX_SPANS;
constexpr int kCandCap = 256; // candidates ranked directly (one per thread)

// The constant ties the pages ask for: a change to one of these fails the build.
static_assert(kThreads % 32 == 0 && kThreads >= 64, "whole warps");
static_assert(kChunkCols <= 65536, "chunk-local column must fit the 16-bit composite field");
static_assert(kCandCap <= kThreads, "rank pass gives each candidate its own thread");
static_assert(kMaxK <= kCandCap, "exact path writes k candidates");
static_assert((kMaxK + kWarps - 1) / kWarps <= 32, "per-warp order statistic needs j <= 32");
static_assert(kMaxSpans == 16 && (kMaxSpans & (kMaxSpans - 1)) == 0, "merge tree over 2^n spans");
static_assert(kMaxK == 64, "header and kernels agree on max_k");

constexpr uint32_t kEmptyVal = 0x7FC0;
constexpr uint32_t kKeyPosInf = 0xFF80;
constexpr uint32_t kKeyNegInf = 0x007F;
constexpr uint32_t kKeyNegZero = 0x7FFF;
constexpr uint32_t kKeyPosZero = 0x8000;

struct __align__(16) Smem {
    uint32_t cand[kCandCap + 4];      // chunk candidates, 32-bit composites (+ zero pad)
    uint16_t cand_raw[kCandCap];      // their original bf16 bits
    uint64_t list[3][kMaxK];          // running list, chunk list, merge output
    uint64_t gather[kMaxSpans][kMaxK];     // leader: the spans' lists
    uint64_t gather2[kMaxSpans / 2][kMaxK];// leader: merge-tree ping-pong
    int32_t glen[kMaxSpans];
    int32_t glen2[kMaxSpans / 2];
    uint32_t gflags[kMaxSpans];
    uint32_t warp_t[kWarps];
    uint32_t red[2][kWarps];
    uint32_t scan[kWarps][4];
    uint32_t keys[kChunkCols / 2];    // exact path: the chunk's keys, two per word, column order
    uint32_t n_cand;
    uint32_t flags;
    uint32_t kmax;
    int32_t run_len;
};

// ---------------------------------------------------------------- bit helpers

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
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

__device__ __forceinline__ uint32_t key_from_raw(uint32_t b)
{
    return b ^ ((b & 0x8000u) ? 0xFFFFu : 0x8000u);
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

// out = top-k of the union of two disjoint descending lists (rank by merge).
__device__ __forceinline__ void merge_lists(const uint64_t *a, int la, const uint64_t *b, int lb,
                                            uint64_t *out, int k)
{
    for (int t = threadIdx.x; t < la + lb; t += kThreads) {
        uint64_t x;
        int pos;
        if (t < la) {
            x = a[t];
            pos = t + count_greater(b, lb, x);
        } else {
            x = b[t - la];
            pos = (t - la) + count_greater(a, la, x);
        }
        if (pos < k) out[pos] = x;
    }
}

__device__ __forceinline__ uint32_t block_sum(uint32_t v, Smem &sm, int parity)
{
    v = __reduce_add_sync(0xFFFFFFFFu, v);
    if ((threadIdx.x & 31) == 0) sm.red[parity][threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += sm.red[parity][w];
    return s;
}

__device__ __forceinline__ void push_candidate(Smem &sm, uint32_t key, int local)
{
    const uint32_t slot = atomicAdd(&sm.n_cand, 1u);
    if (slot < (uint32_t)kCandCap) {
        sm.cand[slot] = (canon(key) << 16) | (0xFFFFu - (uint32_t)local);
        sm.cand_raw[slot] = (uint16_t)raw_from_key(key);
    }
}

// Keys of sm.keys whose score is >= the score of key t (t >= 1), this thread's share.
__device__ __forceinline__ uint32_t count_at_least(const Smem &sm, uint32_t t)
{
    const uint32_t f = key_floor(t);
    uint32_t c = 0;
    for (int w = threadIdx.x; w < kChunkCols / 2; w += kThreads) {
        const uint32_t k2 = sm.keys[w];
        c += (k2 & 0xFFFFu) >= f;
        c += (k2 >> 16) >= f;
    }
    return c;
}

// Exact selection for a chunk whose candidate set {key >= t_floor} is larger
// than the candidate buffer (heavy ties, e.g. an all-zero row).  The chunk's
// keys have been staged in sm.keys in column order (0 = not a candidate).
// Writes exactly k candidates -- the chunk's top-k within that set -- into
// sm.cand.  Block-uniform; every thread calls it.
__device__ __noinline__ void exact_select(uint32_t t_floor, int k, Smem &sm)
{
    const int tid = threadIdx.x;
    // 1. K* = the largest canonical key that at least k elements reach.
    uint32_t my_max = 0;
    for (int w = tid; w < kChunkCols / 2; w += kThreads)
        my_max = max(my_max, max(sm.keys[w] & 0xFFFFu, sm.keys[w] >> 16));
    if (tid == 0) sm.kmax = 0;
    __syncthreads();
    atomicMax(&sm.kmax, canon(my_max));
    __syncthreads();
    uint32_t lo = canon(t_floor); // count(lo) > kCandCap >= k
    uint32_t hi = sm.kmax + 1;    // count(hi) == 0
    int parity = 0;
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        const uint32_t c = block_sum(count_at_least(sm, mid), sm, parity);
        parity ^= 1;
        if (c >= (uint32_t)k)
            lo = mid;
        else
            hi = mid;
    }
    const uint32_t kstar = lo;
    const uint32_t above =
        (kstar >= kKeyPosInf) ? 0u : block_sum(count_at_least(sm, kstar + 1), sm, parity);
    const uint32_t need = (uint32_t)k - above; // ties at K* to take, lowest columns first

    // 2. Each thread owns a contiguous run of columns; an exclusive scan of the
    //    per-thread tie counts gives every tie its rank in column order.
    constexpr int kWordsPerThread = kChunkCols / 2 / kThreads;
    const int w0 = tid * kWordsPerThread;
    uint32_t ties = 0;
    for (int w = w0; w < w0 + kWordsPerThread; ++w) {
        ties += canon(sm.keys[w] & 0xFFFFu) == kstar;
        ties += canon(sm.keys[w] >> 16) == kstar;
    }
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t incl = ties;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += u;
    }
    if (lane == 31) sm.scan[warp][0] = incl;
    if (tid == 0) sm.n_cand = 0;
    __syncthreads();
    uint32_t ord = incl - ties;
    for (int w = 0; w < warp; ++w) ord += sm.scan[w][0];

    // 3. Collect everything above K* and the first `need` ties.
    for (int w = w0; w < w0 + kWordsPerThread; ++w) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t key = h ? (sm.keys[w] >> 16) : (sm.keys[w] & 0xFFFFu);
            if (key == 0) continue;
            const uint32_t c = canon(key);
            if (c > kstar) {
                push_candidate(sm, key, 2 * w + h);
            } else if (c == kstar) {
                if (ord < need) push_candidate(sm, key, 2 * w + h);
                ++ord;
            }
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- cluster barrier

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

// ---------------------------------------------------------------- the kernel

// grid.x = rows * S; with S > 1 the launch groups each row's S CTAs into one
// cluster (cluster rank == span).
template <int S>
__global__ void __launch_bounds__(kThreads, 4)
topk_rows_kernel(const uint16_t *__restrict__ logits, int32_t cols, int64_t row_stride, int32_t k,
                 int32_t *__restrict__ out_idx, uint16_t *__restrict__ out_val,
                 int32_t *__restrict__ out_count, uint32_t *__restrict__ out_mask)
{
    __shared__ Smem sm;
    const int tid = threadIdx.x;
    const int span = (S > 1) ? (int)(blockIdx.x % S) : 0;
    const int64_t row = (int64_t)(blockIdx.x / S);

    if constexpr (S > 1) cluster_arrive_relaxed(); // paired with the wait before DSMEM use

    const uint16_t *rowp = logits + row * row_stride;
    const int32_t m = (int32_t)((reinterpret_cast<uintptr_t>(rowp) >> 1) & 7); // elements before the 16-B boundary
    const uint4 *vbase = reinterpret_cast<const uint4 *>(rowp - m);
    const int32_t nvec = (cols + m + 7) >> 3;   // vectors touching [0, cols)
    const int32_t vfull0 = m ? 1 : 0;           // vectors wholly inside [0, cols)
    const int32_t vfull1 = (cols + m) >> 3;     //   are [vfull0, vfull1)
    const int32_t per_span = (nvec + S - 1) / S;
    const int32_t v_begin = min(nvec, span * per_span);
    const int32_t v_end = min(nvec, v_begin + per_span);

    if (tid == 0) {
        sm.flags = 0;
        sm.run_len = 0;
    }
    __syncthreads();
    int run_i = 0, chunk_i = 1, free_i = 2;
    const int j = (k + kWarps - 1) / kWarps;

    for (int32_t cbeg = v_begin; cbeg < v_end; cbeg += kChunkVecs) {
        const int32_t cend = min(v_end, cbeg + kChunkVecs);
        const int32_t col_base = cbeg * 8 - m;

        // ---- load: full vectors by 16-byte loads, edge vectors element-wise
        uint32_t kv[kVecPerThread][4];
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
            const int32_t v = cbeg + i * kThreads + tid;
            if (v < cend && v >= vfull0 && v < vfull1) {
                const uint4 q = ld_stream(vbase + v);
                kv[i][0] = q.x;
                kv[i][1] = q.y;
                kv[i][2] = q.z;
                kv[i][3] = q.w;
            } else if (v < cend) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int32_t c0 = v * 8 + 2 * w - m;
                    const uint32_t lo = (c0 >= 0 && c0 < cols) ? rowp[c0] : 0xFFFFu;
                    const uint32_t hi = (c0 + 1 >= 0 && c0 + 1 < cols) ? rowp[c0 + 1] : 0xFFFFu;
                    kv[i][w] = lo | (hi << 16);
                }
            } else {
#pragma unroll
                for (int w = 0; w < 4; ++w) kv[i][w] = 0;
            }
        }

        // ---- keys, thread max/min over the full vectors
        uint32_t mx = 0, mn = 0xFFFFFFFFu;
        bool edge = false;
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
            const int32_t v = cbeg + i * kThreads + tid;
            if (v < cend && v >= vfull0 && v < vfull1) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t key = keys_from_raw2(kv[i][w]);
                    kv[i][w] = key;
                    mx = max_u16x2(mx, key);
                    mn = min_u16x2(mn, key);
                }
            } else if (v < cend) {
                edge = true;
            }
        }
        uint32_t tmax = max(mx & 0xFFFFu, mx >> 16);
        const uint32_t tmin = min(mn & 0xFFFFu, mn >> 16);

        // ---- exact path for threads holding an edge vector or a non-finite key
        if (edge || tmax >= kKeyPosInf || tmin <= kKeyNegInf) {
            uint32_t tflags = 0;
            tmax = 0;
#pragma unroll
            for (int i = 0; i < kVecPerThread; ++i) {
                const int32_t v = cbeg + i * kThreads + tid;
                if (v >= cend) continue;
                const bool full = v >= vfull0 && v < vfull1;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t out = 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int32_t c = v * 8 + 2 * w + h - m;
                        uint32_t key;
                        if (full) {
                            key = h ? (kv[i][w] >> 16) : (kv[i][w] & 0xFFFFu);
                        } else if (c >= 0 && c < cols) {
                            key = key_from_raw(h ? (kv[i][w] >> 16) : (kv[i][w] & 0xFFFFu));
                        } else {
                            continue; // outside the row: key 0, never a candidate, no flag
                        }
                        if (key > kKeyPosInf || key < kKeyNegInf) {
                            tflags |= 1u; // NaN
                            key = 0;
                        } else if (key == kKeyPosInf) {
                            tflags |= 2u;
                        } else if (key == kKeyNegInf) {
                            tflags |= 4u;
                        }
                        tmax = max(tmax, key);
                        out |= key << (16 * h);
                    }
                    kv[i][w] = out;
                }
            }
            if (tflags) atomicOr(&sm.flags, tflags);
        }

        // ---- prefilter threshold: min over warps of the warp's j-th largest thread max
        {
            uint32_t v = tmax, cnt = 0, tw = 0;
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
            if ((tid & 31) == 0) sm.warp_t[tid >> 5] = tw;
        }
        if (tid == 0) sm.n_cand = 0;
        __syncthreads();
        uint32_t t0 = 0xFFFFu;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t0 = min(t0, sm.warp_t[w]);
        uint32_t t_floor = max(key_floor(t0), 1u);
        const int run_len = sm.run_len;
        if (run_len == k) {
            // a new entry must beat the running k-th strictly (it has a higher column)
            const uint32_t kth = (uint32_t)(sm.list[run_i][k - 1] >> 48);
            t_floor = max(t_floor, kth + 1);
        }

        // ---- candidates
        if (t_floor <= 0xFFFFu) {
            const uint32_t tm1 = (t_floor - 1) * 0x10001u;
#pragma unroll
            for (int i = 0; i < kVecPerThread; ++i)
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t key2 = kv[i][w];
                    if (max_u16x2(key2, tm1) != tm1) {
                        const int local = (i * kThreads + tid) * 8 + 2 * w;
                        if ((key2 & 0xFFFFu) >= t_floor) push_candidate(sm, key2 & 0xFFFFu, local);
                        if ((key2 >> 16) >= t_floor) push_candidate(sm, key2 >> 16, local + 1);
                    }
                }
        }
        __syncthreads();
        uint32_t n = sm.n_cand;
        if (n > (uint32_t)kCandCap) {
            // stage the chunk's keys in column order; what is below t_floor is
            // not a candidate and becomes 0
            const uint32_t f = t_floor;
#pragma unroll
            for (int i = 0; i < kVecPerThread; ++i) {
                uint4 q;
                uint32_t *qw = &q.x;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t lo = kv[i][w] & 0xFFFFu, hi = kv[i][w] >> 16;
                    qw[w] = (lo >= f ? lo : 0u) | ((hi >= f ? hi : 0u) << 16);
                }
                reinterpret_cast<uint4 *>(sm.keys)[i * kThreads + tid] = q;
            }
            __syncthreads();
            exact_select(t_floor, k, sm);
            n = sm.n_cand; // == k
        }
        if (tid >= (int)n && tid < (int)((n + 3) & ~3u)) sm.cand[tid] = 0;
        __syncthreads();

        // ---- rank the candidates: rank = number of larger composites
        if (tid < (int)n) {
            const uint32_t e = sm.cand[tid];
            uint32_t rank = 0;
            const uint4 *c4 = reinterpret_cast<const uint4 *>(sm.cand);
            for (uint32_t u = 0; u < (n + 3) >> 2; ++u) {
                const uint4 q = c4[u];
                rank += (q.x > e) + (q.y > e) + (q.z > e) + (q.w > e);
            }
            if (rank < (uint32_t)k) sm.list[chunk_i][rank] = entry_from_cand(e, sm.cand_raw[tid], col_base);
        }
        __syncthreads();
        const int chunk_len = min((int)n, k);
        if (run_len == 0) {
            const int t = run_i;
            run_i = chunk_i;
            chunk_i = t;
        } else if (chunk_len > 0) {
            merge_lists(sm.list[run_i], run_len, sm.list[chunk_i], chunk_len, sm.list[free_i], k);
            const int t = run_i;
            run_i = free_i;
            free_i = t;
        }
        __syncthreads();
        if (tid == 0) sm.run_len = min(k, run_len + chunk_len);
        __syncthreads();
    }

    const uint64_t *final_list;
    int final_len;
    uint32_t flags;
    if constexpr (S == 1) {
        final_list = sm.list[run_i];
        final_len = sm.run_len;
        flags = sm.flags;
    } else {
        // ---- push this span's list into the leader's shared memory
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); // every CTA has started
        cg::cluster_group cluster = cg::this_cluster();
        uint64_t *g = cluster.map_shared_rank(&sm.gather[span][0], 0);
        const int len = sm.run_len;
        for (int t = tid; t < len; t += kThreads) g[t] = sm.list[run_i][t];
        if (tid == 0) {
            *cluster.map_shared_rank(&sm.glen[span], 0) = len;
            *cluster.map_shared_rank(&sm.gflags[span], 0) = sm.flags;
        }
        cluster_arrive_release();
        cluster_wait_acquire();
        if (span != 0) return;

        // ---- leader: pairwise merge tree over the S lists
        uint64_t(*src)[kMaxK] = sm.gather;
        uint64_t(*dst)[kMaxK] = sm.gather2;
        int32_t *src_len = sm.glen;
        int32_t *dst_len = sm.glen2;
        flags = 0;
#pragma unroll
        for (int s = 0; s < S; ++s) flags |= sm.gflags[s];
        for (int nl = S; nl > 1; nl >>= 1) {
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
            // swap roles: the next level reads what this one wrote
            uint64_t(*tl)[kMaxK] = src;
            src = dst;
            dst = tl;
            int32_t *tlen = src_len;
            src_len = dst_len;
            dst_len = tlen;
        }
        final_list = src[0];
        final_len = src_len[0];
    }

    // ---- write the row
    for (int t = tid; t < k; t += kThreads) {
        const int64_t o = row * k + t;
        if (t < final_len) {
            const uint64_t e = final_list[t];
            out_idx[o] = entry_col(e);
            out_val[o] = (uint16_t)(e & 0xFFFFu);
        } else {
            out_idx[o] = -1;
            out_val[o] = (uint16_t)kEmptyVal;
        }
    }
    if (tid == 0) {
        out_count[row] = final_len;
        out_mask[row] = flags;
    }
}

// ---------------------------------------------------------------- host side

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

// Per-device set-up, once: check the architecture, allow the 16-CTA cluster.
int device_setup(int *sm_count)
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
            e = cudaFuncSetAttribute(topk_rows_kernel<16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return fail_cuda(e);
            d.status = TF_TOPK_OK;
        }
        d.sm_count = sms;
        d.ready = true;
    }
    *sm_count = d.sm_count;
    return d.status;
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

// Span count for a shape: rows below 4096 columns stay on one CTA (the pages'
// threshold); wider rows use enough spans that each CTA holds at most one
// chunk, and more while the grid is small next to the SM count.
int32_t pick_spans(int64_t rows, int64_t cols, int sm_count)
{
    if (cols < 4096) return 1;
    const int64_t nvec = (cols + 7) / 8 + 1;
    int32_t s = 1;
    while (s < kMaxSpans && (nvec + s - 1) / s > kChunkVecs) s <<= 1;
    while (s < kMaxSpans && rows * s < 2LL * sm_count && (nvec + 2 * s - 1) / (2 * s) >= 2 * kThreads)
        s <<= 1;
    return s;
}

template <int S>
cudaError_t launch(const uint16_t *logits, int64_t rows, int32_t cols, int64_t row_stride, int32_t k,
                   int32_t *out_idx, uint16_t *out_val, int32_t *out_count, uint32_t *out_mask,
                   cudaStream_t stream)
{
    const int64_t max_rows = (int64_t)INT32_MAX / S;
    for (int64_t r0 = 0; r0 < rows; r0 += max_rows) {
        const int64_t nr = rows - r0 < max_rows ? rows - r0 : max_rows;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(nr * S), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        if (S > 1) {
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = S;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        cudaError_t e = cudaLaunchKernelEx(&cfg, topk_rows_kernel<S>, logits + r0 * row_stride, cols,
                                           row_stride, k, out_idx + r0 * k, out_val + r0 * k,
                                           out_count + r0, out_mask + r0);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int run(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k, int32_t *out_idx,
        uint16_t *out_val, int32_t *out_count, uint32_t *out_mask, int32_t spans, void *stream)
{
    int st = validate(logits, rows, cols, row_stride, k, out_idx, out_val, out_count, out_mask);
    if (st != TF_TOPK_OK) return st;
    if (spans != 0 && spans != 1 && spans != 2 && spans != 4 && spans != 8 && spans != 16)
        return TF_TOPK_ERR_SPANS;
    if (rows == 0) return TF_TOPK_OK;
    int sm_count = 0;
    st = device_setup(&sm_count);
    if (st != TF_TOPK_OK) return st;
    if (spans == 0) spans = pick_spans(rows, cols, sm_count);
    const uint16_t *x = static_cast<const uint16_t *>(logits);
    const int32_t c = (int32_t)cols;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (spans) {
    case 1: e = launch<1>(x, rows, c, row_stride, k, out_idx, out_val, out_count, out_mask, s); break;
    case 2: e = launch<2>(x, rows, c, row_stride, k, out_idx, out_val, out_count, out_mask, s); break;
    case 4: e = launch<4>(x, rows, c, row_stride, k, out_idx, out_val, out_count, out_mask, s); break;
    case 8: e = launch<8>(x, rows, c, row_stride, k, out_idx, out_val, out_count, out_mask, s); break;
    default: e = launch<16>(x, rows, c, row_stride, k, out_idx, out_val, out_count, out_mask, s); break;
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e);
    return TF_TOPK_OK;
}

} // namespace

extern "C" {

int tf_topk_bf16(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                 int32_t *out_idx, uint16_t *out_val, int32_t *out_count, uint32_t *out_nonfinite_mask,
                 void *stream)
{
    return run(logits, rows, cols, row_stride, k, out_idx, out_val, out_count, out_nonfinite_mask, 0,
               stream);
}

int tf_topk_bf16_spans(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                       int32_t *out_idx, uint16_t *out_val, int32_t *out_count,
                       uint32_t *out_nonfinite_mask, int32_t spans, void *stream)
{
    return run(logits, rows, cols, row_stride, k, out_idx, out_val, out_count, out_nonfinite_mask, spans,
               stream);
}

int32_t tf_topk_bf16_plan(int64_t rows, int64_t cols, int32_t k)
{
    if (k < 1 || k > kMaxK) return -TF_TOPK_ERR_K;
    if (rows < 0 || cols < 1 || cols > (int64_t)INT32_MAX - 64) return -TF_TOPK_ERR_SHAPE;
    int sm_count = 0;
    const int st = device_setup(&sm_count);
    if (st != TF_TOPK_OK) return -st;
    return pick_spans(rows, cols, sm_count);
}

int32_t tf_topk_bf16_max_k(void) { return kMaxK; }
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
    case TF_TOPK_ERR_SPANS: return "spans must be 0, 1, 2, 4, 8 or 16";
    case TF_TOPK_ERR_DEVICE: return "current device is not compute capability 10.3 (sm_103a)";
    case TF_TOPK_ERR_CUDA: return "CUDA runtime error (see tf_topk_last_cuda_error)";
    default: return "unknown status";
    }
}

int tf_topk_last_cuda_error(void) { return t_last_cuda_error; }

} // extern "C"
