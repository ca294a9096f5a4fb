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
//              candidate only when it beats the row's running k-th (strictly:
//              this CTA's tiles come in column order, so an equal value has
//              the higher column and loses), and each row's candidates are
//              merged into its list by one warp after every tile.
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
constexpr int kHeadThreads = 320;             // producer warp, MMA warp, eight epilogue warps
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
    uint32_t warp_bound[4][kRowsN];           // per lane group and row: a prefilter bound
    uint64_t full[kStages], empty[kStages];   // ring barriers
    uint64_t acc_full[2], acc_empty[2];       // accumulator barriers
    uint64_t drain;                           // the MMA warp's last products are done
    int32_t run_len[kRowsN];
    uint32_t cand_n[kRowsN];
    uint32_t bound[kRowsN];                   // a candidate's canonical key must reach this
    uint32_t flags[kRowsN];
    uint32_t tmem_base;
    uint32_t abort;
    uint32_t last;                            // the epilogue's view of a split tile's ticket
};

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

// Entries of a descending list of distinct values that exceed x.
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

// One row's candidates of this tile into its running list, by one warp: a
// candidate's place is the candidates above it plus the running entries above
// it; a running entry's, its index plus the candidates above it.
__device__ __forceinline__ void merge_row(HeadSmem &sm, int r, int k, uint64_t *tmp)
{
    const int lane = threadIdx.x & 31;
    const int n = (int)sm.cand_n[r];
    if (n == 0) return;
    const int rl = sm.run_len[r];
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
    if (lane == 0) {
        sm.run_len[r] = len;
        sm.cand_n[r] = 0;
        // once k entries are in, a later column must beat the k-th strictly
        sm.bound[r] = len == k ? (uint32_t)(sm.run[r][k - 1] >> 48) + 1u : 1u;
    }
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
struct HeadWorkspace {
    uint64_t *lists;
    uint64_t *tickets;  // [grid]
    float *partials;    // [grid][2][kTileM][kRowsN]; part 0 from CTA i - 1, part 1 from CTA i
};

// Take the ticket of a split tile for this call: true for the second of its
// two parts to arrive.  The word holds (call epoch << 2) | arrivals, so a word
// an earlier call left counts as empty.  Release before, acquire after (the
// partial sums written before the ticket are seen by the other part).
__device__ __forceinline__ bool split_ticket_is_last(uint64_t *t, uint64_t epoch)
{
    const uint64_t tag = epoch << 2;
    __threadfence();
    uint64_t cur = *reinterpret_cast<volatile uint64_t *>(t);
    bool last = false;
    for (int i = 0; i < 64; ++i) { // two arrivals per word: a few rounds at most
        const uint64_t next = (cur & ~3ull) == tag ? cur + 1 : tag | 1ull;
        const uint64_t seen = atomicCAS(reinterpret_cast<unsigned long long *>(t), cur, next);
        if (seen == cur) {
            last = (next & 3ull) == 2ull;
            break;
        }
        cur = seen;
    }
    __threadfence();
    return last;
}

// The work of a call is the units (tile, K stage) in tile-major order, cut
// into equal contiguous ranges, one per CTA (each at least a tile long, so a
// tile falls in at most two CTAs).  A CTA's segments are its tiles, the first
// and last possibly partial.  The two parts of a tile cut between CTAs i - 1
// and i (the head at the end of i - 1, the tail at the start of i) each write
// their partial sum and take the tile's ticket; the second to arrive adds the
// other's partial to its own and selects the tile.  Nothing waits: usually
// CTA i - 1 finishes the tile at its end; if CTA i arrives second it does so
// at its start, before its own tiles.  Tiles reach the selection in column
// order within a CTA either way.
struct Segment {
    int64_t tile;
    int kc0, kc1;     // K stages [kc0, kc1) of the tile in this CTA
    bool tail, head;  // the tail (first segment) / head (last segment) of a cut tile
};

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
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(head_dsmem) + 1023) & ~(uintptr_t)1023);
    uint8_t *ring_a = base;                                 // kStages x kStageA
    uint8_t *ring_b = base + (size_t)kStages * kStageA;     // kStages x kStageB
    HeadSmem &sm = *reinterpret_cast<HeadSmem *>(ring_b + (size_t)kStages * kStageB);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t b = blockIdx.x, grid = gridDim.x;
    const int nk = (dim + kChunkK - 1) / kChunkK;
    const int64_t units = ntiles * nk;
    const int64_t u0 = b * units / grid, u1 = (b + 1) * units / grid;
    const int64_t t_first = u0 / nk, t_last = (u1 - 1) / nk;

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
        sm.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < kRowsN) {
        sm.run_len[tid] = 0;
        sm.cand_n[tid] = 0;
        sm.bound[tid] = 1;
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
    grid_dependency_wait(); // the inputs may come from the previous kernel on the stream

    volatile uint32_t *abort = &sm.abort;
    if (warp == 0) {
        // ---- TMA producer: the units [u0, u1) in order
        if (lane == 0) {
            uint32_t it = 0;
            for (int64_t u = u0; u < u1 && !*abort; ++u, ++it) {
                const int64_t t = u / nk;
                const int kc = (int)(u - t * nk);
                const uint32_t s = it % kStages, ph = it / kStages;
                if (ph > 0 && !mbar_wait(&sm.empty[s], (ph - 1) & 1)) {
                    atomicCAS(&g_head_fault, 0u, kFaultWait);
                    *abort = 1;
                    break;
                }
                mbar_expect_tx(&sm.full[s], kStageA + kStageB);
#pragma unroll
                for (int bx = 0; bx < kChunkK / kBoxK; ++bx) {
                    const int32_t x = kc * kChunkK + bx * kBoxK;
                    tma_load_2d(ring_a + (size_t)s * kStageA + bx * kBoxA, &tmap_w, x, (int32_t)(t * kTileM),
                                &sm.full[s]);
                    tma_load_2d(ring_b + (size_t)s * kStageB + bx * kBoxB, &tmap_h, x, 0, &sm.full[s]);
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
            int si = 0;
            for (int64_t t = t_first; t <= t_last && ok && !*abort; ++t, ++si) {
                const Segment g = segment_of(t, u0, u1, nk);
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
    } else {
        // ---- epilogue: warps 2..9.  Warp w reads accumulator lanes 32 * (w % 4) ..
        // (the tile rows = vocabulary columns of its threads) and one half of
        // the draft rows: rows 8 h .. 8 h + 7, h = (w - 2) / 4.
        const int ew = warp - 2;
        const int q = warp & 3;
        const int h = ew >> 2;
        const int r0 = h * kHalfRows;
        const int trow = 32 * q + lane; // this thread's row of the tile
        uint32_t fl = 0;                // non-finite flags, 3 bits per row of the half
        int si = 0;
        for (int64_t t = t_first; t <= t_last; ++t, ++si) {
            const Segment g = segment_of(t, u0, u1, nk);
            const uint32_t buf = si & 1, uu = si >> 1;
            const bool ok = mbar_wait(&sm.acc_full[buf], uu & 1);
            if (epilogue_any(!ok || *abort)) {
                if (!ok) atomicCAS(&g_head_fault, 0u, kFaultWait);
                *abort = 1;
                break;
            }
            tc_fence_after();
            uint32_t acc[kHalfRows];
            tmem_load8(tmem + buf * kRowsN + r0 + ((uint32_t)(32 * q) << 16), acc);
            tc_fence_before();
            mbar_arrive(&sm.acc_empty[buf]); // the accumulator may take the next segment's products
            if (g.tail || g.head) {
                // a cut tile: hand this part's sum over; the second part in finishes it
                const int64_t bnd = g.tail ? b : b + 1;
                float4 *mine = reinterpret_cast<float4 *>(
                    ws.partials + (((size_t)bnd * 2 + (g.tail ? 1 : 0)) * kTileM + trow) * kRowsN + r0);
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    mine[j] = make_float4(__uint_as_float(acc[4 * j]), __uint_as_float(acc[4 * j + 1]),
                                          __uint_as_float(acc[4 * j + 2]), __uint_as_float(acc[4 * j + 3]));
                __threadfence();
                epilogue_sync();
                if (ew == 0 && lane == 0) sm.last = split_ticket_is_last(&ws.tickets[bnd], epoch) ? 1u : 0u;
                epilogue_sync();
                if (!sm.last) continue;
                const float4 *other = reinterpret_cast<const float4 *>(
                    ws.partials + (((size_t)bnd * 2 + (g.tail ? 0 : 1)) * kTileM + trow) * kRowsN + r0);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float4 p = __ldcg(other + j);
                    acc[4 * j] = __float_as_uint(__uint_as_float(acc[4 * j]) + p.x);
                    acc[4 * j + 1] = __float_as_uint(__uint_as_float(acc[4 * j + 1]) + p.y);
                    acc[4 * j + 2] = __float_as_uint(__uint_as_float(acc[4 * j + 2]) + p.z);
                    acc[4 * j + 3] = __float_as_uint(__uint_as_float(acc[4 * j + 3]) + p.w);
                }
            }
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
            // rows whose list is not full yet (a CTA's first tile): a prefilter
            // bound for the tile -- each lane group's j-th largest key, j =
            // ceil(k / 4); the smallest of the four is reached by at least k
            // keys of the tile
            bool prefilter = false;
#pragma unroll
            for (int r = 0; r < kRowsN; ++r) prefilter |= r < rows && sm.run_len[r] < k;
            if (prefilter) { // block-uniform: run_len changes only between barriers
                const int j = (k + 3) / 4;
#pragma unroll
                for (int i = 0; i < kHalfRows; ++i) {
                    const int r = r0 + i;
                    if (r < rows && sm.run_len[r] < k) {
                        uint32_t x = keys[i], cnt = 0, tw = 0;
                        for (int it = 0; it < j; ++it) {
                            const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, x);
                            if (m == 0) break;
                            cnt += __popc(__ballot_sync(0xFFFFFFFFu, x == m));
                            if (cnt >= (uint32_t)j) {
                                tw = m;
                                break;
                            }
                            if (x == m) x = 0;
                        }
                        if (lane == 0) sm.warp_bound[q][r] = tw;
                    }
                }
                epilogue_sync();
            }
            bool pushed = false;
#pragma unroll
            for (int i = 0; i < kHalfRows; ++i) {
                const int r = r0 + i;
                if (r < rows && keys[i] != 0) {
                    uint32_t bound = sm.bound[r];
                    if (sm.run_len[r] < k)
                        bound = max(bound, min(min(sm.warp_bound[0][r], sm.warp_bound[1][r]),
                                               min(sm.warp_bound[2][r], sm.warp_bound[3][r])));
                    if (keys[i] >= bound) {
                        const uint32_t slot = atomicAdd(&sm.cand_n[r], 1u);
                        sm.cand[r][slot] = head_entry(keys[i], (uint32_t)v, bits16[i]);
                        pushed = true;
                    }
                }
            }
            if (epilogue_any(pushed)) { // a barrier too: the candidates are in
                for (int r = ew; r < rows; r += kEpiWarps) merge_row(sm, r, k, sm.tmp[ew]);
                epilogue_sync();
            }
        }
        // this CTA's list per row into the workspace: [rows][grid][k + 1],
        // a header (length | flags << 32) and the entries
#pragma unroll
        for (int i = 0; i < kHalfRows; ++i) {
            const uint32_t f = __reduce_or_sync(0xFFFFFFFFu, (fl >> (3 * i)) & 7u);
            if (lane == 0 && f && r0 + i < rows) atomicOr(&sm.flags[r0 + i], f);
        }
        epilogue_sync();
        for (int r = ew; r < rows; r += kEpiWarps) {
            uint64_t *out = ws.lists + ((size_t)r * grid + b) * (size_t)(k + 1);
            const int len = sm.run_len[r];
            for (int j = lane; j < len; j += 32) out[1 + j] = sm.run[r][j];
            if (lane == 0) out[0] = (uint64_t)(uint32_t)len | ((uint64_t)sm.flags[r] << 32);
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

// One CTA per row merges the row's `lists` per-CTA lists: each holds its
// CTA's best entries (descending, at most k), and the CTAs cover increasing
// column ranges, so list order is column order.  The row's k-th key K* (the
// k-th largest score, counted with multiplicity) comes from a radix select
// over the keys, eight bits a pass.  The row is then every entry above K*
// (fewer than k) and, of the entries at K*, the lowest columns: those of the
// earliest lists first, each list's own in column order -- a scan over the
// lists.  A CTA's list holds at most k entries, and a CTA never contributes
// more than k to the row, so nothing the row needs was left out of a list.
// One radix pass over the row's keys: a histogram of the digit (key >> shift)
// & 0xFF over every entry (match: only entries whose high byte is match_hi).
// Warp w takes lists w, w + warps, ...; a list's entries are sorted, so lanes
// holding the same digit sit side by side: each run of equal digits adds its
// length once, into the warp's own sub-histogram (hist_w: [warps][256]);
// then the sub-histograms are summed into hist.  Block-uniform.
__device__ __forceinline__ void merge_hist(const uint64_t *buf, int lists, int w, int k, int shift, uint32_t match_hi,
                                           bool match, uint32_t *hist_w, uint32_t *hist)
{
    constexpr int kWarps = kMergeThreads / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t *mine = hist_w + warp * 256;
    for (int i = lane; i < 256; i += 32) mine[i] = 0;
    __syncwarp();
    for (int j = warp; j < lists; j += kWarps) {
        const uint64_t *lj = buf + (size_t)j * w;
        const int n = (int)(uint32_t)lj[0];
        for (int e0 = 0; e0 < n; e0 += 32) {
            const int e = e0 + lane;
            uint32_t digit = 0xFFFFFFFFu;
            if (e < n) {
                const uint32_t key = (uint32_t)(lj[1 + e] >> 48);
                if (!match || (key >> 8) == match_hi) digit = (key >> shift) & 0xFFu;
            }
            const uint32_t prev = __shfl_up_sync(0xFFFFFFFFu, digit, 1);
            const bool start = digit != 0xFFFFFFFFu && (lane == 0 || prev != digit);
            const uint32_t starts = __ballot_sync(0xFFFFFFFFu, start);
            const uint32_t valid = __ballot_sync(0xFFFFFFFFu, digit != 0xFFFFFFFFu);
            if (start) {
                // the run ends where the next run starts, or where the valid lanes end
                const uint32_t later = starts & ~((2u << lane) - 1u);
                const int end = later ? __ffs(later) - 1 : 32 - __clz(valid);
                mine[digit] += (uint32_t)(end - lane);
            }
            __syncwarp();
        }
    }
    (void)k;
    __syncthreads();
    for (int i = tid; i < 256; i += kMergeThreads) {
        uint32_t sum = 0;
#pragma unroll
        for (int x = 0; x < kWarps; ++x) sum += hist_w[x * 256 + i];
        hist[i] = sum;
    }
}

// In one warp: the digit holding the need-th largest count of `hist`, and how
// many lie in the digits above it.
__device__ __forceinline__ void merge_pick(const uint32_t *hist, uint32_t need, uint32_t *digit, uint32_t *above)
{
    const int lane = threadIdx.x & 31;
    uint32_t c8 = 0; // this lane's eight bins, from the top: 255 - 8 * lane ...
#pragma unroll
    for (int i = 0; i < 8; ++i) c8 += hist[255 - 8 * lane - i];
    uint32_t incl = c8;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += u;
    }
    const uint32_t excl = incl - c8;
    if (excl < need && need <= incl) {
        uint32_t a = excl;
        for (int i = 0; i < 8; ++i) {
            const uint32_t bin = 255 - 8 * lane - i, h = hist[bin];
            if (a + h >= need) {
                *digit = bin;
                *above = a;
                break;
            }
            a += h;
        }
    }
}

__global__ void __launch_bounds__(kMergeThreads)
topk_head_merge_kernel(const uint64_t *__restrict__ ws_lists, int32_t lists, int32_t k,
                       int32_t *__restrict__ out_idx, uint16_t *__restrict__ out_val,
                       int32_t *__restrict__ out_count, uint32_t *__restrict__ out_mask)
{
    grid_dependency_wait();
    extern __shared__ __align__(16) uint64_t merge_dsmem[];
    __shared__ uint32_t flags, entries, hist[256], digit_s, above_s;
    __shared__ uint32_t hist_w[(kMergeThreads / 32) * 256];
    __shared__ int32_t wsum[kMergeThreads / 32];
    __shared__ uint64_t pick[kMaxK], fin[kMaxK];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x;
    const int w = k + 1;
    uint64_t *buf = merge_dsmem; // the row's lists, contiguous: [lists][k + 1] (header, entries)
    if (tid == 0) {
        flags = 0;
        entries = 0;
    }
    const uint64_t *src = ws_lists + (size_t)r * lists * w;
    for (int i = tid; i < lists * w; i += kMergeThreads) buf[i] = __ldcg(src + i);
    __syncthreads();
    uint32_t my_flags = 0, my_n = 0;
    for (int j = tid; j < lists; j += kMergeThreads) {
        const uint64_t h = buf[(size_t)j * w];
        my_flags |= (uint32_t)(h >> 32);
        my_n += (uint32_t)h;
    }
    my_flags = __reduce_or_sync(0xFFFFFFFFu, my_flags);
    my_n = __reduce_add_sync(0xFFFFFFFFu, my_n);
    if (lane == 0) {
        atomicOr(&flags, my_flags);
        atomicAdd(&entries, my_n);
    }
    __syncthreads();
    const int total = (int)entries;
    const int len = min(k, total);
    // K*: with k or fewer entries every key is in; else two radix passes
    uint32_t kstar = 0;
    if (total > k) {
        uint32_t need = (uint32_t)k, hi = 0;
        for (int pass = 0; pass < 2; ++pass) {
            merge_hist(buf, lists, w, k, pass == 0 ? 8 : 0, hi, pass == 1, hist_w, hist);
            __syncthreads();
            if (warp == 0) merge_pick(hist, need, &digit_s, &above_s);
            __syncthreads();
            if (pass == 0) hi = digit_s;
            need -= above_s;
        }
        kstar = (hi << 8) | digit_s;
    }
    // per list: entries above K* (a prefix), then entries at K* (next); one
    // scan over the lists (packed: above << 16 | ties) gives each its places
    static_assert(kMaxGrid <= kMergeThreads, "one list per scanning thread");
    uint32_t a = 0, tie = 0;
    if (tid < lists) {
        const uint64_t *lj = buf + (size_t)tid * w + 1;
        const int n = (int)(uint32_t)buf[(size_t)tid * w];
        if (total <= k) {
            a = (uint32_t)n;
        } else {
            a = (uint32_t)count_greater(lj, n, ((uint64_t)(kstar + 1) << 48) - 1);
            tie = (uint32_t)count_greater(lj, n, ((uint64_t)kstar << 48) - 1) - a;
        }
    }
    const uint32_t mine = (a << 16) | tie;
    uint32_t incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += u;
    }
    if (lane == 31) wsum[warp] = (int32_t)incl;
    __syncthreads();
    uint32_t excl = incl - mine, all = 0;
    for (int x = 0; x < kMergeThreads / 32; ++x) {
        excl += x < warp ? (uint32_t)wsum[x] : 0u;
        all += (uint32_t)wsum[x];
    }
    const uint32_t above_all = all >> 16;        // entries above K*: fewer than k
    const uint32_t need = (uint32_t)len - above_all;
    if (tid < lists) {
        const uint64_t *lj = buf + (size_t)tid * w + 1;
        const uint32_t a0 = excl >> 16, t0 = excl & 0xFFFFu;
        for (uint32_t i = 0; i < a; ++i) pick[a0 + i] = lj[i];
        for (uint32_t i = 0; i < tie && t0 + i < need; ++i) pick[above_all + t0 + i] = lj[a + i];
    }
    __syncthreads();
    // the len chosen entries in order: a place is the number of larger ones
    for (int t = tid; t < len; t += kMergeThreads) {
        const uint64_t x = pick[t];
        int rank = 0;
        for (int u = 0; u < len; ++u) rank += pick[u] > x;
        fin[rank] = x;
    }
    __syncthreads();
    for (int t = tid; t < k; t += kMergeThreads) {
        const int64_t o = (int64_t)r * k + t;
        if (t < len) {
            const uint64_t e = fin[t];
            out_idx[o] = (int32_t)(~(uint32_t)(e >> 16));
            out_val[o] = (uint16_t)(e & 0xFFFFu);
        } else {
            out_idx[o] = -1;
            out_val[o] = 0x7FC0;
        }
    }
    if (tid == 0) {
        out_count[r] = len;
        out_mask[r] = flags;
    }
}

// ---------------------------------------------------------------- host side

constexpr size_t kHeadSmemBytes = 1024 + (size_t)kStages * (kStageA + kStageB) + sizeof(HeadSmem);

// The merge kernel's dynamic shared memory: the row's lists.
size_t merge_smem_bytes(int lists, int k)
{
    return (size_t)lists * (size_t)(k + 1) * sizeof(uint64_t); // the row's lists
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
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(topk_head_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)merge_smem_bytes(kMaxGrid, kMaxK));
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

// Bytes of a call's workspace: the lists, the tickets, the partial sums (on a
// 256-byte boundary, hence the slack).
size_t workspace_bytes_for(int grid, int rows, int k)
{
    return (size_t)grid * ((size_t)rows * (size_t)(k + 1) * sizeof(uint64_t) + sizeof(uint64_t) +
                           2 * (size_t)kTileM * kRowsN * sizeof(float)) +
           256;
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
    uint64_t *lists = static_cast<uint64_t *>(workspace);
    HeadWorkspace ws;
    ws.lists = lists;
    ws.tickets = lists + (size_t)grid * rows * (k + 1);
    // the partial sums start on a 256-byte boundary (vector stores)
    ws.partials = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(ws.tickets + grid) + 255) & ~(uintptr_t)255);

    const uint64_t epoch = g_epoch.fetch_add(1, std::memory_order_relaxed) & (~0ull >> 2);
    cudaError_t e = cudaLaunchKernelEx(&cfg, topk_head_kernel, tw, th, rows, dim, vocab, k, ntiles, ws, epoch);
    if (e == cudaSuccess) {
        cudaLaunchConfig_t mcfg = cfg;
        mcfg.gridDim = dim3((unsigned)rows, 1, 1);
        mcfg.blockDim = dim3(kMergeThreads, 1, 1);
        mcfg.dynamicSmemBytes = merge_smem_bytes(grid, k);
        e = cudaLaunchKernelEx(&mcfg, topk_head_merge_kernel, (const uint64_t *)lists, (int32_t)grid, k, out_idx,
                               out_val, out_count, out_mask);
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
