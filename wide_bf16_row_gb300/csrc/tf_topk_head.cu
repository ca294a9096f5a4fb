// Draft head with the top-k in its epilogue, for GB300 (sm_103a).
//
// What is computed: the drafter's head turns each draft position's hidden
// state into a row of bf16 logits, and the top-k of TensorFold PR #713
// ("perf(qwen27): a drafted round overlaps its cache commit with the next
// draft, and the drafter's attention and top-k use more of the GPU"),
// change 3, takes each row's best entries (score descending, lower token
// index first; count and non-finite mask per row, as in the page's
// "Exactness" table).  The head is read as the usual LM head:
//   logit[r][v] = bf16_rne( sum_d hidden[r][d] * weight[v][d] ),  fp32 sum,
// and the selection is the one tf_topk_bf16 makes over those logits.  Here
// the logits never leave the chip: the selection runs on the accumulators.
//
// topk_head_kernel: persistent, one CTA per SM; the work -- (vocabulary tile
// of kTileM columns, K stage) units -- is cut into equal contiguous ranges,
// one per CTA, and a tile cut between two CTAs is finished by whichever of
// the two arrives second, with the other's partial sum.  Warp roles:
//   warp 0     TMA producer: per ring stage, the weight tile (kTileM rows x
//              kChunkK dims) and the hidden tile (kRowsN rows x kChunkK dims),
//              each as boxes of kBoxK dims with the 128-byte swizzle the MMA
//              descriptors expect;
//   warp 1     MMA issuer: tcgen05.mma kind::f16 (M = kTileM vocabulary rows,
//              N = kRowsN draft rows, K = 16 per instruction, bf16 in, fp32
//              out) into one of two TMEM accumulators, so that the epilogue of
//              a tile overlaps the products of the next; the warp also
//              allocates and frees the TMEM;
//   warps 2-9  epilogue: tcgen05.ld of a finished accumulator (thread =
//              vocabulary column; two warps per 32 accumulator lanes, each
//              taking half of the draft rows), round to bf16, and a running
//              top-k per row: a value becomes a
//              candidate only when it beats the row's running k-th entry in
//              the row's order (score, then the lower column), and each
//              row's candidates are merged into its list by one warp after
//              every tile.
// At the end each CTA leaves one list per row in the caller's workspace.
// topk_head_merge_kernel: one CTA per row merges those lists (the same order)
// and writes the row.
//
// No wait is unbounded and no CTA waits for another: every mbarrier wait gives
// up after kHeadWaitLimit polls, records a fault code, and the CTA winds down
// (waiting, again with a bound, for its own copies and products in flight)
// and frees its TMEM.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "tf_topk.h"

// Defined with the other entry points: records a CUDA error for
// tf_topk_last_cuda_error and returns TF_TOPK_ERR_CUDA.
int tf_topk_internal_fail_cuda(int cuda_error);

namespace {

constexpr int kTileM = 128;                   // vocabulary rows per tile (MMA M)
constexpr int kRowsN = 16;                    // draft rows, padded (MMA N)
constexpr int kBoxK = 64;                     // dims per TMA box: one 128-byte swizzle row of bf16
constexpr int kChunkK = 128;                  // dims per ring stage: two boxes side by side
constexpr int kStages = 5;                    // TMA ring depth (180 KB in flight)
constexpr int kPrefetchStages = 2 * kStages;  // weight stages a CTA sends toward L2 before its inputs are ready
constexpr int kHeadThreads = 352;             // producer warp, MMA warp, eight epilogue warps, helper warp
constexpr int kEpiThreads = 256;
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr int kHalfRows = kRowsN / 2;          // an epilogue warp's rows: one half of the draft rows
constexpr int kMaxK = TF_TOPK_MAX_K;
constexpr int kCandCap = kTileM;              // a tile adds at most kTileM candidates to a row
constexpr uint32_t kBoxA = kTileM * kBoxK * 2;     // 16 KB: one swizzle atom column of the weight tile
constexpr uint32_t kBoxB = kRowsN * kBoxK * 2;     // 2 KB
constexpr uint32_t kStageA = kBoxA * (kChunkK / kBoxK);  // 32 KB
constexpr uint32_t kStageB = kBoxB * (kChunkK / kBoxK);  // 4 KB
constexpr int kTmemCols = 2 * kRowsN;         // two fp32 accumulators of kRowsN columns
constexpr uint32_t kHeadWaitLimit = 1u << 20;
constexpr uint32_t kFaultWait = 1;
constexpr uint64_t kAnyKey = 1ull << 32;      // (key << 32 | ~column) below every non-NaN key
constexpr int kRankMerge = 16;                // candidates a row merges by ranks; more are sorted first
constexpr int kMaxGrid = 160;                 // lists per row the merge kernel takes (GB300: 152 SMs)

static_assert(TF_TOPK_HEAD_MAX_ROWS == kRowsN, "header and kernel agree on the draft rows");
static_assert(kTmemCols >= 32 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocations are powers of two >= 32");
static_assert(kBoxA % 1024 == 0 && kBoxB % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
static_assert(kChunkK % kBoxK == 0 && kBoxK % 16 == 0, "whole boxes per stage, whole MMA steps per box");
static_assert(kEpiThreads == 2 * kTileM, "two epilogue threads per accumulator lane, one per half of the rows");

__device__ uint32_t g_head_fault;

struct __align__(16) HeadSmem {
    uint64_t run[kRowsN][kMaxK];              // running list per row (descending)
    uint64_t cand[kRowsN][kCandCap];          // this tile's candidates per row
    uint64_t tmp[kEpiWarps][kMaxK];           // per epilogue warp: merge output
    uint64_t full[kStages], empty[kStages];   // ring barriers
    uint64_t acc_full[2], acc_empty[2];       // accumulator barriers
    uint64_t drain;                           // the MMA warp's last products are done
    int32_t run_len[kRowsN];
    uint32_t cand_n[kRowsN];
    uint64_t bound[kRowsN];                   // a candidate's (key << 32 | ~column) must reach this
    uint32_t flags[kRowsN];
    alignas(16) float cut_other[2][kTileM][kRowsN]; // the other part's partial sums of a cut tile this CTA finishes
    uint64_t cut_ready[2];                    // epilogue -> helper: this part's partial sums are written
    uint64_t cut_done[2];                     // helper -> epilogue: ticket taken (other part staged if last)
    uint32_t cut_last[2];                     // this CTA arrived second at the cut tile's ticket
    uint32_t tmem_base;
    uint32_t abort;
};

static_assert(offsetof(HeadSmem, cut_other) % 16 == 0, "the helper stages the other part's sums as float4");

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes) : "memory");
}

// Bounded wait for the phase with this parity: false after kHeadWaitLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    for (uint32_t i = 0; i < kHeadWaitLimit; ++i) {
        uint32_t ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(ok)
                     : "r"(saddr(bar)), "r"(parity)
                     : "memory");
        if (ok) return true;
    }
    return false;
}

// Whether the phase with this parity has completed (no wait).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(saddr(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// As mbar_wait, but also gives up once another warp has set *abort.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort)
{
    for (uint32_t i = 0; i < kHeadWaitLimit; ++i) {
        uint32_t ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(ok)
                     : "r"(saddr(bar)), "r"(parity)
                     : "memory");
        if (ok) return true;
        if (*abort) return false;
    }
    atomicCAS(&g_head_fault, 0u, kFaultWait);
    *abort = 1;
    return false;
}

__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int32_t x, int32_t y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int32_t x, int32_t y, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(saddr(dst)), "l"(map), "r"(x), "r"(y), "r"(saddr(bar))
                 : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: start address >> 4 (bits 0-13), leading byte offset 16
// (not used by a swizzled K-major tile), stride byte offset 1024 (eight
// 128-byte rows; bits 32-45), descriptor version 1 (bits 46-47), swizzle mode
// 128 bytes (bits 61-63 = 2).  Moving along K inside the 128-byte row is a
// plain add to the start address.
__device__ __forceinline__ uint64_t sw128_desc(const void *smem)
{
    const uint64_t a = (saddr(smem) & 0x3FFFFu) >> 4;
    return a | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bit 4),
// bf16 A and B (bits 7 and 10), both K-major, N / 8 at bit 17, M / 16 at bit 24.
constexpr uint32_t kIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kRowsN >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, bool accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"((uint32_t)accumulate)
                 : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// This warp's 32 accumulator lanes (lane = thread), 8 consecutive columns.
__device__ __forceinline__ void tmem_load8(uint32_t taddr, uint32_t (&r)[kHalfRows])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_go() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- keys and lists

// Order-preserving key of bf16 bits, -0 and +0 merged, NaN -> 0 (never selected).
__device__ __forceinline__ uint32_t canon_key(uint32_t b)
{
    if ((b & 0x7FFFu) > 0x7F80u) return 0;
    const uint32_t key = (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
    return key == 0x7FFFu ? 0x8000u : key;
}

__device__ __forceinline__ uint32_t nonfinite_flag(uint32_t b)
{
    if ((b & 0x7FFFu) > 0x7F80u) return 1u;
    if (b == 0x7F80u) return 2u;
    if (b == 0xFF80u) return 4u;
    return 0u;
}

// List entry: canonical key (16) | ~column (32) | original bits (16).  The
// integers order as (score desc, column asc); (key, column) is unique.
__device__ __forceinline__ uint64_t head_entry(uint32_t key, uint32_t col, uint32_t bits)
{
    return ((uint64_t)key << 48) | ((uint64_t)(~col) << 16) | (uint64_t)bits;
}

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m)
{
    const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, (uint32_t)v, m);
    const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), m);
    return ((uint64_t)hi << 32) | lo;
}

__device__ __forceinline__ uint64_t shfl_idx64(uint64_t v, int src)
{
    const uint32_t lo = __shfl_sync(0xFFFFFFFFu, (uint32_t)v, src);
    const uint32_t hi = __shfl_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), src);
    return ((uint64_t)hi << 32) | lo;
}

__device__ __forceinline__ uint64_t max64(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t min64(uint64_t a, uint64_t b) { return a > b ? b : a; }

// Entries of a non-increasing list that exceed x (a binary search).
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

// A full bitonic sort into descending order of the 32 R entries a warp holds
// (entry i in lane i % 32, register i / 32): merges of sorted runs of size 2,
// 4, .., 32 R, each run ordered descending or ascending by its position, the
// last one descending.
// Compare-exchange: a gets the larger when desc, else the smaller.
__device__ __forceinline__ void cx64(uint64_t &a, uint64_t &b, bool desc)
{
    const uint64_t hi = max64(a, b), lo = min64(a, b);
    a = desc ? hi : lo;
    b = desc ? lo : hi;
}

// A full bitonic sort into descending order of the 32 R entries a warp holds
// (entry i in lane i % 32, register i / 32; R = 1, 2 or 4): merges of sorted
// runs of size 2, 4, .., 32 R, each run ordered descending or ascending by
// its position, the last one descending.  Stage loops stay rolled (the
// epilogue's code must stay small: an instruction fetch that misses waits
// behind the weight stream).
template <int R>
__device__ __forceinline__ void bitonic_full_sort(uint64_t (&x)[R], int lane)
{
    static_assert(R == 1 || R == 2 || R == 4, "one, two or four registers");
#pragma unroll 1
    for (int size = 2; size <= 32 * R; size <<= 1) {
#pragma unroll 1
        for (int d = size >> 1; d >= 1; d >>= 1) {
            if (d == 64) { // registers e and e + 2, same lane
                if constexpr (R == 4) {
                    cx64(x[0], x[2], (0 & size) == 0);
                    cx64(x[1], x[3], (32 & size) == 0);
                }
            } else if (d == 32) { // registers e and e + 1, same lane
                if constexpr (R >= 2) {
                    cx64(x[0], x[1], (0 & size) == 0);
                    if constexpr (R == 4) cx64(x[2], x[3], (64 & size) == 0);
                }
            } else {
                const bool lower = (lane & d) == 0;
#pragma unroll
                for (int e = 0; e < R; ++e) {
                    const uint64_t y = shfl_xor64(x[e], d);
                    const bool desc = ((e * 32 + lane) & size) == 0;
                    x[e] = lower == desc ? max64(x[e], y) : min64(x[e], y);
                }
            }
        }
    }
}

// One row's candidates of this tile (n > a few) into its running list, by
// one warp: the candidates sorted in registers, then the top P of them and
// of the running list -- max(A[i], B[P - 1 - i]) over the sorted candidates
// A and the running list B is bitonic and holds the top P of both (Batcher's
// bitonic merge) -- sorted by half-cleaners.
template <int R>
__device__ __forceinline__ void merge_row_sorted(HeadSmem &sm, int r, int k, int P, int n, int rl)
{
    const int lane = threadIdx.x & 31;
    uint64_t x[R];
#pragma unroll
    for (int e = 0; e < R; ++e) {
        const int i = e * 32 + lane;
        x[e] = i < n ? sm.cand[r][i] : 0ull;
    }
    bitonic_full_sort<R>(x, lane);
    uint64_t y[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int i = e * 32 + lane, j = P - 1 - i;
        const uint64_t a = e < R ? x[e < R ? e : 0] : 0ull;
        const uint64_t bb = i < P && j < rl ? sm.run[r][j] : 0ull;
        y[e] = i < P ? max64(a, bb) : 0ull;
    }
    if (P == 64) {
        const uint64_t hi = max64(y[0], y[1]), lo = min64(y[0], y[1]);
        y[0] = hi;
        y[1] = lo;
    }
#pragma unroll 1
    for (int d = (P < 32 ? P : 32) >> 1; d >= 1; d >>= 1) {
        const bool lower = (lane & d) == 0;
        const uint64_t z0 = shfl_xor64(y[0], d);
        y[0] = lower ? max64(y[0], z0) : min64(y[0], z0);
        if (P == 64) {
            const uint64_t z1 = shfl_xor64(y[1], d);
            y[1] = lower ? max64(y[1], z1) : min64(y[1], z1);
        }
    }
    __syncwarp(); // every lane has read the old running list
    const int len = min(k, rl + n);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int i = e * 32 + lane;
        if (i < len) sm.run[r][i] = y[e];
    }
    __syncwarp();
}

// One row's candidates of this tile into its running list, by one warp.  A
// few candidates: a candidate's place is the candidates above it plus the
// running entries above it; a running entry's, its index plus the candidates
// above it.  More: merge_row_sorted.  Then the new bound: once k entries are
// in, a candidate must beat the k-th in the row's order.
__device__ __forceinline__ void merge_row(HeadSmem &sm, int r, int k, int P, uint64_t *tmp)
{
    const int lane = threadIdx.x & 31;
    const int n = (int)sm.cand_n[r];
    if (n == 0) return;
    const int rl = sm.run_len[r];
    if (n <= kRankMerge) {
        const uint64_t *c = sm.cand[r];
        const uint64_t *run = sm.run[r];
        for (int i = lane; i < n; i += 32) {
            const uint64_t x = c[i];
            int pos = count_greater(run, rl, x);
            for (int j = 0; j < n; ++j) pos += c[j] > x;
            if (pos < k) tmp[pos] = x;
        }
        for (int j = lane; j < rl; j += 32) {
            const uint64_t x = run[j];
            int pos = j;
            for (int i = 0; i < n; ++i) pos += c[i] > x;
            if (pos < k) tmp[pos] = x;
        }
        __syncwarp();
        const int len = min(k, rl + n);
        for (int j = lane; j < len; j += 32) sm.run[r][j] = tmp[j];
        __syncwarp();
    } else if (n <= 32) {
        merge_row_sorted<1>(sm, r, k, P, n, rl);
    } else if (n <= 64) {
        merge_row_sorted<2>(sm, r, k, P, n, rl);
    } else {
        merge_row_sorted<4>(sm, r, k, P, n, rl);
    }
    if (lane == 0) {
        const int len = min(k, rl + n);
        sm.run_len[r] = len;
        sm.cand_n[r] = 0;
        sm.bound[r] = len == k ? (sm.run[r][k - 1] >> 16) + 1u : kAnyKey;
    }
    __syncwarp();
}

// True in every epilogue thread when `p` holds in any of them (a reduction on
// the epilogue's named barrier).
__device__ __forceinline__ bool epilogue_any(bool p)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred q, o;\n\tsetp.ne.u32 q, %1, 0;\n\t"
                 "bar.red.or.pred o, 1, %2, q;\n\tselp.u32 %0, 1, 0, o;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)p), "n"(kEpiThreads)
                 : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- the fused kernel

// Workspace of one call.  Lists: [rows][grid][k + 1] (a row's lists
// contiguous for the merge).  Per boundary i between CTAs i - 1 and i that
// cuts a tile: a ticket and the two fp32 partial sums of that tile.
// Entries a list slot of the workspace holds: k rounded up to a power of
// two, at least 2 (16-byte list blocks).
__host__ __device__ __forceinline__ int list_stride(int k)
{
    int p = 2;
    while (p < k) p <<= 1;
    return p;
}

struct HeadWorkspace {
    uint64_t *lists;    // [rows][grid][list_stride(k)], zero after a list's last entry
    uint64_t *heads;    // [rows][grid]: length | flags << 32
    uint64_t *tickets;  // [grid]
    float *partials;    // [grid][2][kTileM][kRowsN]; part 0 from CTA i - 1, part 1 from CTA i
};

// Arrive at a cut tile's ticket for this call: true for the part that
// arrives second.  Both parts exchange the call's tag into the word; the
// second finds the tag already there (a word an earlier call left holds
// another tag).  Release and acquire at GPU scope: this CTA's partial sums,
// written before (and ordered before this thread by the barrier it waited
// on), are visible to the part that arrives second, and the other part's to
// this thread when it arrives second.
__device__ __forceinline__ bool take_split_ticket(uint64_t *t, uint64_t epoch)
{
    const uint64_t tag = (epoch << 2) | 1ull;
    uint64_t old;
    asm volatile("atom.acq_rel.gpu.global.exch.b64 %0, [%1], %2;" : "=l"(old) : "l"(t), "l"(tag) : "memory");
    return old == tag;
}

// The work of a call is the units (tile, K stage) in tile-major order, cut
// into equal contiguous ranges, one per CTA (each at least a tile long, so a
// tile falls in at most two CTAs).  A CTA's segments are its tiles, the first
// and last possibly partial.  The two parts of a tile cut between CTAs i - 1
// and i (the head, in i - 1, and the tail, in i) each write their partial sum
// and take the tile's ticket; the second to arrive adds the other's partial
// to its own and selects the tile.  No part waits for the other.  A CTA
// takes its cut segments first (the tail, then the head) and its full tiles
// after them in column order.  The epilogue only writes a cut segment's
// partial sums and keeps its own in registers; the CTA's helper warp takes
// the ticket and, when this CTA is second, stages the other part's sums in
// shared memory; the epilogue finishes such a tile after its first full
// tile, by when the exchange has long completed.  Tiles thus reach the
// selection out of column order; the running bound compares (score,
// column), not the score alone.
struct Segment {
    int64_t tile;
    int kc0, kc1;     // K stages [kc0, kc1) of the tile in this CTA
    bool tail, head;  // the tail (first segment) / head (last segment) of a cut tile
};

// The tile of a CTA's si-th segment in the order above.
__device__ __forceinline__ int64_t segment_tile(int si, int64_t u0, int64_t u1, int nk)
{
    const int64_t t_first = u0 / nk, t_last = (u1 - 1) / nk;
    const bool tail_cut = (u0 % nk) != 0, head_cut = (u1 % nk) != 0;
    const int nc = (int)tail_cut + (int)head_cut;
    if (si < nc) return tail_cut && si == 0 ? t_first : t_last;
    return t_first + (tail_cut ? 1 : 0) + (si - nc);
}

__device__ __forceinline__ Segment segment_of(int64_t t, int64_t u0, int64_t u1, int nk)
{
    Segment g;
    g.tile = t;
    g.kc0 = t == u0 / nk ? (int)(u0 % nk) : 0;
    g.kc1 = t == (u1 - 1) / nk ? (int)((u1 - 1) % nk) + 1 : nk;
    g.tail = g.kc0 != 0;
    g.head = g.kc1 != nk;
    return g;
}

__global__ void __launch_bounds__(kHeadThreads, 1)
topk_head_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_h,
                 int32_t rows, int32_t dim, int64_t vocab, int32_t k, int64_t ntiles, HeadWorkspace ws,
                 uint64_t epoch)
{
    extern __shared__ __align__(1024) uint8_t head_dsmem[];
    // 1024-byte aligned (the swizzled tiles); offset from the shared array
    // itself, so that every access below stays a shared-memory access
    uint8_t *base = head_dsmem + ((1024u - (saddr(head_dsmem) & 1023u)) & 1023u);
    uint8_t *ring_a = base;                                 // kStages x kStageA
    uint8_t *ring_b = base + (size_t)kStages * kStageA;     // kStages x kStageB
    HeadSmem &sm = *reinterpret_cast<HeadSmem *>(ring_b + (size_t)kStages * kStageB);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t b = blockIdx.x, grid = gridDim.x;
    const int nk = (dim + kChunkK - 1) / kChunkK;
    const int64_t units = ntiles * nk;
    const int64_t u0 = b * units / grid, u1 = (b + 1) * units / grid;
    const int nseg = (int)((u1 - 1) / nk - u0 / nk + 1); // segments of this CTA

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.acc_full[i], 1);
            mbar_init(&sm.acc_empty[i], kEpiThreads);
        }
        mbar_init(&sm.drain, 1);
        for (int c = 0; c < 2; ++c) {
            mbar_init(&sm.cut_ready[c], kEpiThreads);
            mbar_init(&sm.cut_done[c], 32);
        }
        sm.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < kRowsN) {
        sm.run_len[tid] = 0;
        sm.cand_n[tid] = 0;
        sm.bound[tid] = kAnyKey;
        sm.flags[tid] = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&sm.tmem_base)),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    if (tid == 0) {
        // while the previous kernel on the stream ends: the weight's first
        // stages toward L2 (a hint only; L2 is where device memory is
        // coherent, so a weight that kernel writes is still read after the wait)
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_w) : "memory");
        int n = 0;
        for (int si = 0; si < nseg && n < kPrefetchStages; ++si) {
            const Segment g = segment_of(segment_tile(si, u0, u1, nk), u0, u1, nk);
            for (int kc = g.kc0; kc < g.kc1 && n < kPrefetchStages; ++kc, ++n)
#pragma unroll
                for (int bx = 0; bx < kChunkK / kBoxK; ++bx)
                    tma_prefetch_2d(&tmap_w, kc * kChunkK + bx * kBoxK, (int32_t)(g.tile * kTileM));
        }
    }
    grid_dependency_wait(); // the inputs may come from the previous kernel on the stream

    volatile uint32_t *abort = &sm.abort;
    if (warp == 0) {
        // ---- TMA producer: the units of each segment, segments in order
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int si = 0; si < nseg && ok; ++si) {
                const Segment g = segment_of(segment_tile(si, u0, u1, nk), u0, u1, nk);
                for (int kc = g.kc0; kc < g.kc1; ++kc, ++it) {
                    const uint32_t s = it % kStages, ph = it / kStages;
                    if (*abort || (ph > 0 && !mbar_wait(&sm.empty[s], (ph - 1) & 1))) {
                        if (!*abort) atomicCAS(&g_head_fault, 0u, kFaultWait);
                        *abort = 1;
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&sm.full[s], kStageA + kStageB);
#pragma unroll
                    for (int bx = 0; bx < kChunkK / kBoxK; ++bx) {
                        const int32_t x = kc * kChunkK + bx * kBoxK;
                        tma_load_2d(ring_a + (size_t)s * kStageA + bx * kBoxA, &tmap_w, x,
                                    (int32_t)(g.tile * kTileM), &sm.full[s]);
                        tma_load_2d(ring_b + (size_t)s * kStageB + bx * kBoxB, &tmap_h, x, 0, &sm.full[s]);
                    }
                }
            }
            // the copies issued land before the CTA leaves: each stage's last
            // fill completes (earlier fills were waited for by the MMA warp
            // before the stage could be refilled); bounded
            const uint32_t issued = it;
            for (uint32_t j = issued > (uint32_t)kStages ? issued - kStages : 0u; j < issued; ++j)
                mbar_wait(&sm.full[j % kStages], (j / kStages) & 1);
        }
    } else if (warp == 1) {
        // ---- MMA issuer: one accumulator per segment, alternating
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int si = 0; si < nseg && ok && !*abort; ++si) {
                const Segment g = segment_of(segment_tile(si, u0, u1, nk), u0, u1, nk);
                const uint32_t buf = si & 1, uu = si >> 1;
                if (uu > 0 && !mbar_wait(&sm.acc_empty[buf], (uu - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * kRowsN;
                for (int kc = g.kc0; kc < g.kc1; ++kc, ++it) {
                    const uint32_t s = it % kStages, ph = it / kStages;
                    if (!mbar_wait(&sm.full[s], ph & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int bx = 0; bx < kChunkK / kBoxK; ++bx) {
                        const uint64_t ad = sw128_desc(ring_a + (size_t)s * kStageA + bx * kBoxA);
                        const uint64_t bd = sw128_desc(ring_b + (size_t)s * kStageB + bx * kBoxB);
#pragma unroll
                        for (int kk = 0; kk < kBoxK / 16; ++kk) // 16 dims = 32 bytes = 2 in the address field
                            mma_bf16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2),
                                     (kc != g.kc0) || bx != 0 || kk != 0);
                    }
                    mma_commit(&sm.empty[s]); // the stage is free once these products are done
                }
                if (!ok) break;
                mma_commit(&sm.acc_full[buf]);
            }
            if (!ok) {
                atomicCAS(&g_head_fault, 0u, kFaultWait);
                *abort = 1;
            }
            // every product this thread issued is done before the TMEM is freed
            mma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0);
        }
    } else if (warp < 2 + kEpiWarps) {
        // ---- epilogue: warps 2..9.  Warp w reads accumulator lanes 32 * (w % 4) ..
        // (the tile rows = vocabulary columns of its threads) and one half of
        // the draft rows: rows 8 h .. 8 h + 7, h = (w - 2) / 4.
        const int ew = warp - 2;
        const int q = warp & 3;
        const int h = ew >> 2;
        const int r0 = h * kHalfRows;
        const int trow = 32 * q + lane; // this thread's row of the tile
        const int P = list_stride(k);   // the running lists' merge width
        uint32_t fl = 0;                // non-finite flags, 3 bits per row of the half
        // the selection of one tile's sums (fp32 bits, rows r0 .. r0 + 7 of
        // this thread's column); block-uniform (epilogue barriers inside)
        auto select_tile = [&](const uint32_t (&acc)[kHalfRows], int64_t t) {
            const int64_t v = t * kTileM + trow;
            const bool in_vocab = v < vocab;
            uint32_t keys[kHalfRows], bits16[kHalfRows];
#pragma unroll
            for (int i = 0; i < kHalfRows; ++i) {
                const bool live = in_vocab && r0 + i < rows;
                bits16[i] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(acc[i])));
                keys[i] = live ? canon_key(bits16[i]) : 0u;
                if (live) fl |= nonfinite_flag(bits16[i]) << (3 * i);
            }
            // a value becomes a candidate when it beats the row's bound; a
            // warp takes its slots in a row's candidates with one atomic.
            // Three passes over the rows, so that their loads, ballots and
            // atomics overlap.
            bool want[kHalfRows];
            uint32_t m[kHalfRows], base[kHalfRows];
#pragma unroll
            for (int i = 0; i < kHalfRows; ++i) {
                const int r = r0 + i;
                want[i] = r < rows && keys[i] != 0 &&
                          ((((uint64_t)keys[i] << 32) | (uint32_t)~(uint32_t)v) >= sm.bound[r < rows ? r : 0]);
                m[i] = __ballot_sync(0xFFFFFFFFu, want[i]);
            }
#pragma unroll
            for (int i = 0; i < kHalfRows; ++i) {
                base[i] = 0;
                if (m[i] != 0 && lane == __ffs(m[i]) - 1) base[i] = atomicAdd(&sm.cand_n[r0 + i], (uint32_t)__popc(m[i]));
            }
            bool pushed = false;
            const uint32_t below = (1u << lane) - 1u;
#pragma unroll
            for (int i = 0; i < kHalfRows; ++i) {
                if (m[i] == 0) continue; // warp-uniform
                const uint32_t at = __shfl_sync(0xFFFFFFFFu, base[i], __ffs(m[i]) - 1) + __popc(m[i] & below);
                if (want[i]) sm.cand[r0 + i][at] = head_entry(keys[i], (uint32_t)v, bits16[i]);
                pushed = true;
            }
            if (epilogue_any(pushed)) { // a barrier too: the candidates are in
#pragma unroll 1
                for (int r = ew; r < rows; r += kEpiWarps) merge_row(sm, r, k, P, sm.tmp[ew]);
                epilogue_sync();
            }
        };
        // The CTA's cut segments are its first nc; their own sums wait in
        // registers until the helper has taken the tickets.  After each full
        // tile the epilogue selects the cut tiles whose exchange is done (the
        // test does not wait: a global round trip under the weight stream
        // takes microseconds) and it finishes as first part; at the end it
        // waits for the rest.  One loop, one selection site.
        const int nc = (int)((u0 % nk) != 0) + (int)((u1 % nk) != 0);
        uint32_t cut_acc0[kHalfRows], cut_acc1[kHalfRows];
        int cuts_next = 0; // cut segments [0, cuts_next) are done with
        int si = 0;        // next segment to read from TMEM
        while (true) {
            uint32_t acc[kHalfRows];
            int64_t t = -1;
            if (cuts_next < nc && si >= nc &&
                (si >= nseg || epilogue_any(mbar_test(&sm.cut_done[cuts_next], 0)))) {
                const int c = cuts_next++;
                const bool ok = mbar_wait(&sm.cut_done[c], 0);
                if (epilogue_any(!ok || *abort)) {
                    if (!ok) atomicCAS(&g_head_fault, 0u, kFaultWait);
                    *abort = 1;
                    break;
                }
                if (!sm.cut_last[c]) continue; // the other part finishes the tile
#pragma unroll
                for (int i = 0; i < kHalfRows; ++i)
                    acc[i] = __float_as_uint(__uint_as_float(c == 0 ? cut_acc0[i] : cut_acc1[i]) +
                                             sm.cut_other[c][trow][r0 + i]);
                t = segment_tile(c, u0, u1, nk);
            } else {
                if (si >= nseg) break;
                const Segment g = segment_of(segment_tile(si, u0, u1, nk), u0, u1, nk);
                const uint32_t buf = si & 1, uu = si >> 1;
                const bool ok = mbar_wait(&sm.acc_full[buf], uu & 1);
                if (epilogue_any(!ok || *abort)) {
                    if (!ok) atomicCAS(&g_head_fault, 0u, kFaultWait);
                    *abort = 1;
                    break;
                }
                tc_fence_after();
                tmem_load8(tmem + buf * kRowsN + r0 + ((uint32_t)(32 * q) << 16), acc);
                tc_fence_before();
                mbar_arrive(&sm.acc_empty[buf]); // the accumulator may take the next segment's products
                if (g.tail || g.head) {
                    // a cut tile (si < nc): this part's sums to the workspace
                    // for the other part, and kept for finishing it here
                    const int64_t bnd = g.tail ? b : b + 1;
                    float4 *mine = reinterpret_cast<float4 *>(
                        ws.partials + (((size_t)bnd * 2 + (g.tail ? 1 : 0)) * kTileM + trow) * kRowsN + r0);
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        mine[j] = make_float4(__uint_as_float(acc[4 * j]), __uint_as_float(acc[4 * j + 1]),
                                              __uint_as_float(acc[4 * j + 2]), __uint_as_float(acc[4 * j + 3]));
#pragma unroll
                    for (int i = 0; i < kHalfRows; ++i) {
                        if (si == 0) cut_acc0[i] = acc[i];
                        else cut_acc1[i] = acc[i];
                    }
                    mbar_arrive(&sm.cut_ready[si]);
                    ++si;
                    continue;
                }
                t = g.tile;
                ++si;
            }
            select_tile(acc, t);
        }
        // this CTA's list per row into the workspace: the entries, zero
        // after the last, and a header (length | flags << 32)
#pragma unroll
        for (int i = 0; i < kHalfRows; ++i) {
            const uint32_t f = __reduce_or_sync(0xFFFFFFFFu, (fl >> (3 * i)) & 7u);
            if (lane == 0 && f && r0 + i < rows) atomicOr(&sm.flags[r0 + i], f);
        }
        epilogue_sync();
        for (int r = ew; r < rows; r += kEpiWarps) {
            uint64_t *out = ws.lists + ((size_t)r * grid + b) * (size_t)P;
            const int len = sm.run_len[r];
            for (int j = lane; j < P; j += 32) out[j] = j < len ? sm.run[r][j] : 0ull;
            if (lane == 0) ws.heads[(size_t)r * grid + b] = (uint64_t)(uint32_t)len | ((uint64_t)sm.flags[r] << 32);
        }
    } else {
        // ---- helper (warp 2 + kEpiWarps): the tickets of the cut tiles, in
        // the epilogue's order; when this CTA arrives second it stages the
        // other part's partial sums for the epilogue
        const int nc = (int)((u0 % nk) != 0) + (int)((u1 % nk) != 0);
        for (int c = 0; c < nc; ++c) {
            const Segment g = segment_of(segment_tile(c, u0, u1, nk), u0, u1, nk);
            const int64_t bnd = g.tail ? b : b + 1;
            if (!mbar_wait_or_abort(&sm.cut_ready[c], 0, abort)) break;
            uint32_t last = 0;
            if (lane == 0) last = take_split_ticket(&ws.tickets[bnd], epoch) ? 1u : 0u;
            __syncwarp(); // the other lanes' reads below come after lane 0's acquire
            last = __shfl_sync(0xFFFFFFFFu, last, 0);
            if (last) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    ws.partials + ((size_t)bnd * 2 + (g.tail ? 0 : 1)) * kTileM * kRowsN);
                float4 *dst = reinterpret_cast<float4 *>(&sm.cut_other[c][0][0]);
                for (int i = lane; i < kTileM * kRowsN / 4; i += 32) dst[i] = __ldcg(src + i);
            }
            if (lane == 0) sm.cut_last[c] = last;
            mbar_arrive(&sm.cut_done[c]);
        }
    }
    grid_dependents_go(); // the merge may be scheduled; it still waits for this grid to finish
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------- the merge of the per-CTA lists

constexpr int kMergeThreads = 512;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kLeadCap = 512; // entries at or above the k-th lead the merge ranks directly
// The row's lists in shared memory; more than half of an SM's, so that merge
// CTAs scheduled early (while the head kernel still runs) take an SM each.
constexpr uint32_t kMergeSmemBytes = 120 * 1024;
static_assert((size_t)kMaxGrid * kMaxK * sizeof(uint64_t) <= kMergeSmemBytes, "a row's lists fit");

// One CTA per row merges the row's `lists` per-CTA lists.  A list holds its
// CTA's best entries in descending order, then zeros, P entries in all (P =
// k rounded up to a power of two, at least 2).  Entries are distinct (each
// holds its column) and the entry order is the row order (score descending,
// lower column first), so the row's top k are the k largest entries of the
// union, and a zero (an empty slot) sorts below every entry.  A CTA never
// contributes more than k entries to the row and its list keeps its best k,
// so nothing the row needs was left out.  Usually the k-th largest list head
// bounds the row's top k from below, and the few entries at or above it are
// ranked directly.  Otherwise the union's top P comes from pairwise merges:
// for sorted A and B, max(A[i], B[P-1-i]) holds the top P of both and is
// bitonic, so half-cleaners sort it (Batcher's bitonic merge).
//
// A warp holds P-entry lists in registers: for P <= 32 a group of P lanes
// holds one (entry i in lane i of the group, 32 / P groups side by side); for
// P = 64 entry i sits in lane i % 32, register i / 32.

template <int P> struct MergeShape {
    static constexpr int E = P > 32 ? 2 : 1;  // registers a lane holds per list
    static constexpr int G = P > 32 ? 1 : 32 / P; // lists side by side in a warp
};

// N bitonic sequences of P entries each into descending order: half-cleaners
// at distances P/2, .., 1; of each pair the lower index keeps the larger.
template <int P, int N>
__device__ __forceinline__ void bitonic_sort_desc(uint64_t (&x)[N][MergeShape<P>::E], int lane)
{
    constexpr int E = MergeShape<P>::E;
    if constexpr (P == 64) {
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const uint64_t hi = max64(x[n][0], x[n][1]), lo = min64(x[n][0], x[n][1]);
            x[n][0] = hi;
            x[n][1] = lo;
        }
    }
#pragma unroll
    for (int d = (P > 32 ? 32 : P) / 2; d >= 1; d >>= 1) {
        const bool upper = (lane & d) != 0;
#pragma unroll
        for (int n = 0; n < N; ++n)
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const uint64_t y = shfl_xor64(x[n][e], d);
                x[n][e] = upper ? min64(x[n][e], y) : max64(x[n][e], y);
            }
    }
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(saddr(dst)), "l"(src), "r"(bytes), "r"(saddr(bar))
                 : "memory");
}

template <int P>
__global__ void __launch_bounds__(kMergeThreads, 1)
topk_head_merge_kernel(const uint64_t *__restrict__ ws_entries, const uint64_t *__restrict__ ws_heads, int32_t lists,
                       int32_t k, int32_t *__restrict__ out_idx, uint16_t *__restrict__ out_val,
                       int32_t *__restrict__ out_count, uint32_t *__restrict__ out_mask, uint64_t *__restrict__ tickets)
{
    constexpr int E = MergeShape<P>::E, G = MergeShape<P>::G;
    extern __shared__ __align__(16) uint64_t merge_dsmem[]; // the row's lists: [lists][P]
    __shared__ uint64_t part[2][kMergeWarps][P];
    __shared__ uint64_t lead[kMaxGrid];             // each list's first entry
    __shared__ uint64_t cand[kLeadCap];             // the entries at or above the k-th lead
    __shared__ uint64_t kth_lead;
    __shared__ uint32_t wsum[kMergeWarps];
    __shared__ uint64_t bar;
    __shared__ uint32_t flags;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x;
    const int g = P > 32 ? 0 : lane / P, i = P > 32 ? lane : lane % P; // lane group, entry
    if (tid == 0) {
        mbar_init(&bar, 1);
        flags = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    grid_dependency_wait();
    // the next call's head kernel may be scheduled now: its CTAs set up on the
    // SMs the head kernel left, and wait for this grid before touching memory
    grid_dependents_go();
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)lists * P * (uint32_t)sizeof(uint64_t);
        mbar_expect_tx(&bar, bytes);
        bulk_load(merge_dsmem, ws_entries + (size_t)r * lists * P, bytes, &bar);
    }
    // The head kernel has finished, and with it every use of the split-tile
    // tickets: clear them, so that the next call on this workspace -- also a
    // replay of a captured call, which repeats its tag -- starts from empty.
    if (r == 0)
        for (int j = tid; j < lists; j += kMergeThreads) tickets[j] = 0;
    uint32_t f = tid < lists ? (uint32_t)(__ldcg(ws_heads + (size_t)r * lists + tid) >> 32) : 0u;
    if (__syncthreads_or(!mbar_wait(&bar, 0))) {
        // the copy did not land in time: report, and wait (bounded) for it
        // before the CTA's shared memory goes away
        if (tid == 0) atomicCAS(&g_head_fault, 0u, kFaultWait);
        mbar_wait(&bar, 0);
        return;
    }
    f = __reduce_or_sync(0xFFFFFFFFu, f);
    if (lane == 0 && f) atomicOr(&flags, f);

    // The usual case: b, the k-th largest of the lists' first entries, has k
    // entries at or above it, so only entries >= b can be in the row's top k.
    // They are few (about k): each list gives its leading ones, and each
    // takes its place by rank among them.
    const uint64_t m = tid < lists ? merge_dsmem[(size_t)tid * P] : 0ull;
    if (tid < lists) lead[tid] = m;
    if (tid == 0) kth_lead = 0;
    __syncthreads();
    if (m != 0) {
        uint32_t above = 0;
        for (int u = 0; u < lists; ++u) above += lead[u] > m;
        if (above == (uint32_t)(k - 1)) kth_lead = m; // leads are distinct: one thread
    }
    __syncthreads();
    const uint64_t bnd = kth_lead;
    if (bnd != 0) { // else fewer than k lists hold an entry
        uint32_t c = 0;
        if (tid < lists)
            while (c < (uint32_t)P && merge_dsmem[(size_t)tid * P + c] >= bnd) ++c;
        uint32_t incl = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += u;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        uint32_t off = incl - c, total = 0;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
            off += w < warp ? wsum[w] : 0u;
            total += wsum[w];
        }
        if (total <= (uint32_t)kLeadCap) { // at least k: the k largest leads
            for (uint32_t j = 0; j < c; ++j) cand[off + j] = merge_dsmem[(size_t)tid * P + j];
            __syncthreads();
            uint64_t *row = &part[0][0][0];
            for (uint32_t q = tid; q < total; q += kMergeThreads) {
                const uint64_t x = cand[q];
                uint32_t rank = 0;
                for (uint32_t u = 0; u < total; ++u) rank += cand[u] > x;
                if (rank < (uint32_t)k) row[rank] = x;
            }
            __syncthreads();
            if (tid < k) {
                const uint64_t x = row[tid];
                out_idx[(int64_t)r * k + tid] = (int32_t)(~(uint32_t)(x >> 16));
                out_val[(int64_t)r * k + tid] = (uint16_t)(x & 0xFFFFu);
            }
            if (tid == 0) {
                out_count[r] = k;
                out_mask[r] = flags;
            }
            return;
        }
    }

    // Otherwise every entry: per lane group two running lists (two
    // independent chains), starting empty; list j enters as max with its
    // reverse, then a sort
    uint64_t x[2][E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[0][e] = x[1][e] = 0;
    const int nslots = kMergeWarps * G;
#pragma unroll 1
    for (int j0 = warp * G; j0 < lists; j0 += 2 * nslots) {
        const int ja = j0 + g, jb = ja + nslots;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int ie = i + 32 * e;
            const uint64_t ya = ja < lists ? merge_dsmem[(size_t)ja * P + (P - 1 - ie)] : 0ull;
            const uint64_t yb = jb < lists ? merge_dsmem[(size_t)jb * P + (P - 1 - ie)] : 0ull;
            x[0][e] = max64(x[0][e], ya);
            x[1][e] = max64(x[1][e], yb);
        }
        bitonic_sort_desc<P, 2>(x, lane);
    }
    // the second chain reversed into the first, then the lane groups together
    uint64_t a[1][E];
    {
        uint64_t c[E];
        if constexpr (P == 64) {
            c[0] = shfl_idx64(x[1][1], 31 - lane);
            c[1] = shfl_idx64(x[1][0], 31 - lane);
        } else {
            c[0] = shfl_idx64(x[1][0], g * P + (P - 1 - i));
        }
#pragma unroll
        for (int e = 0; e < E; ++e) a[0][e] = max64(x[0][e], c[e]);
        bitonic_sort_desc<P, 1>(a, lane);
    }
#pragma unroll
    for (int h = 1; h < G; h <<= 1) {
        const uint64_t c = shfl_idx64(a[0][0], (g ^ h) * P + (P - 1 - i));
        a[0][0] = max64(a[0][0], c);
        bitonic_sort_desc<P, 1>(a, lane);
    }
    if (g == 0) {
#pragma unroll
        for (int e = 0; e < E; ++e) part[0][warp][i + 32 * e] = a[0][e];
    }
    // a tree over the warps' lists: warp w merges lists 2w and 2w + 1
    int src = 0;
#pragma unroll 1
    for (int n = kMergeWarps; n > 1; n >>= 1, src ^= 1) {
        __syncthreads();
        if (warp < n / 2) {
            const uint64_t *A = part[src][2 * warp], *B = part[src][2 * warp + 1];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int ie = i + 32 * e;
                a[0][e] = g == 0 ? max64(A[ie], B[P - 1 - ie]) : 0ull;
            }
            bitonic_sort_desc<P, 1>(a, lane);
            if (n > 2 && g == 0) {
#pragma unroll
                for (int e = 0; e < E; ++e) part[src ^ 1][warp][i + 32 * e] = a[0][e];
            }
        }
    }
    if (warp == 0) {
        // the row: the first k entries; the empty ones (zero) come last
        int len = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int t = i + 32 * e;
            const bool mine = g == 0 && t < k;
            const bool full = mine && a[0][e] != 0;
            len += __popc(__ballot_sync(0xFFFFFFFFu, full));
            if (mine) {
                const int64_t o = (int64_t)r * k + t;
                out_idx[o] = full ? (int32_t)(~(uint32_t)(a[0][e] >> 16)) : -1;
                out_val[o] = full ? (uint16_t)(a[0][e] & 0xFFFFu) : (uint16_t)0x7FC0;
            }
        }
        if (lane == 0) {
            out_count[r] = len;
            out_mask[r] = flags;
        }
    }
}

// ---------------------------------------------------------------- host side

constexpr size_t kHeadSmemBytes = 1024 + (size_t)kStages * (kStageA + kStageB) + sizeof(HeadSmem);
static_assert(kHeadSmemBytes <= 227 * 1024, "the head kernel's shared memory fits one CTA");



// The merge kernel for each list stride P = 2, 4, .., 64.
using MergeKernel = void (*)(const uint64_t *, const uint64_t *, int32_t, int32_t, int32_t *, uint16_t *, int32_t *,
                             uint32_t *, uint64_t *);
constexpr int kMergeKernels = 6;
const MergeKernel kMergeKernel[kMergeKernels] = {topk_head_merge_kernel<2>,  topk_head_merge_kernel<4>,
                                                 topk_head_merge_kernel<8>,  topk_head_merge_kernel<16>,
                                                 topk_head_merge_kernel<32>, topk_head_merge_kernel<64>};
static_assert(kMaxK <= 64, "the largest list stride has a merge kernel");
MergeKernel merge_kernel_for(int P)
{
    int i = 0;
    while ((2 << i) < P) ++i;
    return kMergeKernel[i];
}

struct HeadDevice {
    std::atomic<bool> ready{false};
    int status = TF_TOPK_OK;
    int sm_count = 0;
};
constexpr int kMaxDevices = 64;
HeadDevice g_head_dev[kMaxDevices];
std::mutex g_head_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per device, once: the architecture, the SM count, the kernels' shared
// memory limits, and the driver's tensor-map encoder.
int head_setup(int *sm_count)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tf_topk_internal_fail_cuda((int)e);
    if (dev < 0 || dev >= kMaxDevices) return TF_TOPK_ERR_DEVICE;
    HeadDevice &d = g_head_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_head_mutex);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int major = 0, minor = 0, sms = 0;
            if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
                return tf_topk_internal_fail_cuda((int)e);
            if (major != 10 || minor != 3) {
                d.status = TF_TOPK_ERR_DEVICE;
            } else {
                e = cudaFuncSetAttribute(topk_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kHeadSmemBytes);
                for (int i = 0; i < kMergeKernels && e == cudaSuccess; ++i)
                    e = cudaFuncSetAttribute(kMergeKernel[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kMergeSmemBytes);
                if (e != cudaSuccess) return tf_topk_internal_fail_cuda((int)e);
                if (!g_encode) {
                    void *fn = nullptr;
                    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
                    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                                         &q);
                    if (e != cudaSuccess) return tf_topk_internal_fail_cuda((int)e);
                    if (q != cudaDriverEntryPointSuccess || !fn) return TF_TOPK_ERR_DEVICE;
                    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
                }
                d.status = TF_TOPK_OK;
            }
            d.sm_count = sms;
            d.ready.store(true, std::memory_order_release);
        }
    }
    *sm_count = d.sm_count;
    return d.status;
}

// A 2-D bf16 tensor map with the 128-byte swizzle: `outer` rows of `inner`
// elements (row stride `inner`), boxes of kBoxK x box_rows.  Coordinates
// past either extent read as zero.
bool encode_map(CUtensorMap *map, const void *p, uint64_t inner, uint64_t outer, uint32_t box_rows)
{
    cuuint64_t gdim[2] = {inner, outer};
    cuuint64_t gstride[1] = {inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBoxK, box_rows};
    cuuint32_t estride[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bytes of a call's workspace: the list entries and the partial sums, each
// on a 256-byte boundary (vector loads and stores; hence the slack), the
// list headers and the tickets.
size_t workspace_bytes_for(int grid, int rows, int k)
{
    return (size_t)grid * ((size_t)rows * (size_t)(list_stride(k) + 1) * sizeof(uint64_t) + sizeof(uint64_t) +
                           2 * (size_t)kTileM * kRowsN * sizeof(float)) +
           512;
}

// A call's epoch tags the tickets it takes, so a ticket an earlier call left
// in the same workspace never counts for this call.  Starts from a value no
// fresh buffer is likely to hold.
std::atomic<uint64_t> g_epoch{0x9E3779B97F4A7C15ull};

int head_grid(int sm_count, int64_t ntiles)
{
    int64_t g = sm_count < kMaxGrid ? sm_count : kMaxGrid;
    if (ntiles < g) g = ntiles;
    return (int)(g < 1 ? 1 : g);
}

int run_head(const void *hidden, const void *weight, int32_t rows, int32_t dim, int64_t vocab, int32_t k,
             void *workspace, size_t workspace_bytes, int32_t *out_idx, uint16_t *out_val, int32_t *out_count,
             uint32_t *out_mask, void *stream)
{
    if (k < 1 || k > kMaxK) return TF_TOPK_ERR_K;
    if (rows < 1 || rows > kRowsN || dim < 8 || (dim % 8) != 0 || vocab < 1 || vocab > (int64_t)INT32_MAX - 64)
        return TF_TOPK_ERR_SHAPE;
    if (!hidden || !weight || !workspace || !out_idx || !out_val || !out_count || !out_mask) return TF_TOPK_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15) || (reinterpret_cast<uintptr_t>(weight) & 15) ||
        (reinterpret_cast<uintptr_t>(workspace) & 7) || (reinterpret_cast<uintptr_t>(out_idx) & 3) ||
        (reinterpret_cast<uintptr_t>(out_val) & 1) || (reinterpret_cast<uintptr_t>(out_count) & 3) ||
        (reinterpret_cast<uintptr_t>(out_mask) & 3))
        return TF_TOPK_ERR_ALIGN;
    int sm_count = 0;
    int st = head_setup(&sm_count);
    if (st != TF_TOPK_OK) return st;
    const int64_t ntiles = (vocab + kTileM - 1) / kTileM;
    const int grid = head_grid(sm_count, ntiles);
    if (workspace_bytes_for(grid, rows, k) > workspace_bytes) return TF_TOPK_ERR_SCRATCH;
    CUtensorMap tw, th;
    if (!encode_map(&tw, weight, (uint64_t)dim, (uint64_t)vocab, kTileM) ||
        !encode_map(&th, hidden, (uint64_t)dim, (uint64_t)rows, kRowsN))
        return tf_topk_internal_fail_cuda((int)cudaErrorInvalidValue);
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kHeadThreads, 1, 1);
    cfg.dynamicSmemBytes = kHeadSmemBytes;
    cfg.stream = strm;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const auto align256 = [](const void *p) {
        return reinterpret_cast<void *>((reinterpret_cast<uintptr_t>(p) + 255) & ~(uintptr_t)255);
    };
    HeadWorkspace ws;
    ws.lists = static_cast<uint64_t *>(align256(workspace));
    ws.heads = ws.lists + (size_t)rows * grid * list_stride(k);
    ws.tickets = ws.heads + (size_t)rows * grid;
    ws.partials = static_cast<float *>(align256(ws.tickets + grid));

    const uint64_t epoch = g_epoch.fetch_add(1, std::memory_order_relaxed) & (~0ull >> 2);
    cudaError_t e = cudaLaunchKernelEx(&cfg, topk_head_kernel, tw, th, rows, dim, vocab, k, ntiles, ws, epoch);
    if (e == cudaSuccess) {
        cudaLaunchConfig_t mcfg = cfg;
        mcfg.gridDim = dim3((unsigned)rows, 1, 1);
        mcfg.blockDim = dim3(kMergeThreads, 1, 1);
        mcfg.dynamicSmemBytes = kMergeSmemBytes;
        e = cudaLaunchKernelEx(&mcfg, merge_kernel_for(list_stride(k)), (const uint64_t *)ws.lists,
                               (const uint64_t *)ws.heads, (int32_t)grid, k, out_idx, out_val, out_count, out_mask,
                               ws.tickets);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return tf_topk_internal_fail_cuda((int)e);
    return TF_TOPK_OK;
}

} // namespace

// The head kernel's fault word, read and cleared (tf_topk_device_fault reports it).
uint32_t tf_topk_internal_head_fault_take()
{
    uint32_t f = 0;
    if (cudaMemcpyFromSymbol(&f, g_head_fault, sizeof f) != cudaSuccess) return 0;
    if (f) {
        const uint32_t zero = 0;
        cudaMemcpyToSymbol(g_head_fault, &zero, sizeof zero);
    }
    return f;
}

extern "C" {

int tf_topk_head_bf16(const void *hidden, const void *weight, int32_t rows, int32_t dim, int64_t vocab, int32_t k,
                      void *workspace, size_t workspace_bytes, int32_t *out_idx, uint16_t *out_val,
                      int32_t *out_count, uint32_t *out_nonfinite_mask, void *stream)
{
    return run_head(hidden, weight, rows, dim, vocab, k, workspace, workspace_bytes, out_idx, out_val, out_count,
                    out_nonfinite_mask, stream);
}

size_t tf_topk_head_bf16_workspace(int32_t rows, int32_t k)
{
    if (rows < 1 || rows > kRowsN || k < 1 || k > kMaxK) return 0;
    int sm_count = 0;
    if (head_setup(&sm_count) != TF_TOPK_OK) return 0;
    const int g = sm_count < kMaxGrid ? sm_count : kMaxGrid;
    return workspace_bytes_for(g, rows, k);
}

} // extern "C"
