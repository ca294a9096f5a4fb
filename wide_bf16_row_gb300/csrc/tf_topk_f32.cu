// Exact per-row top-k of fp32 rows (k <= 64) for GB300 (sm_103a): the
// TensorFold PR #713, change 3 selection (score descending, the lower column
// first on ties; NaN never selected; +0 and -0 one score; a count and a
// non-finite mask per row) on 32-bit keys.
//
// topk_f32_cluster_kernel<S>: one thread-block cluster of S CTAs per row, one
// column span per CTA (the span's columns ascending), chunks of 8192 values
// held in registers (eight 16-byte vectors a thread):
//   - each thread's largest key; the chunk's bound is the prefilter bound
//     (each warp's j-th largest lane maximum, the smallest over the warps)
//     until the span's running list holds k entries, then the running k-th
//     (strictly: every column of a later chunk is higher);
//   - threads whose largest key reaches the bound spill their keys to shared
//     memory, which frees the registers: the next chunk's loads are issued
//     at once and fly during the rest of the chunk;
//   - each such thread counts its keys that reach the bound; a warp scan and
//     one atomic give their slots; entries (canonical key << 32 | ~column)
//     go to the candidate buffer; a chunk with no candidate ends there;
//   - candidates and running entries find their places by rank (entries are
//     distinct): a candidate's is its rank among the candidates plus the
//     running entries above it;
//   - more candidates than the buffer holds (heavy ties) are selected exactly
//     from the spilled keys: the k-th key by a binary search on block
//     counts, then the entries above it and the lowest columns among its
//     ties.
// The spans' lists meet in the leader CTA's shared memory (distributed
// shared memory) and are merged pairwise; the leader writes the row, the
// values re-read by column (their original bits).
//
// Keys: a value's order-preserving key is its bits with the sign bit set
// (>= +0) or all bits flipped (< 0); -0 is folded onto +0 wherever a key is
// compared or stored, and NaN becomes key 0 (never selected).

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tf_topk.h"

namespace cg = cooperative_groups;

// Defined with the other entry points: records a CUDA error for
// tf_topk_last_cuda_error and returns TF_TOPK_ERR_CUDA.
int tf_topk_internal_fail_cuda(int cuda_error);

namespace {

constexpr int kF32Threads = 256;
constexpr int kF32Warps = kF32Threads / 32;
constexpr int kF32Vec = 8;                              // 16-byte vectors a thread holds of a chunk
constexpr int kF32ChunkVecs = kF32Threads * kF32Vec;   // 2048 vectors = 8192 values = 32 KB
constexpr int kF32MaxK = TF_TOPK_MAX_K;
constexpr int kF32Cap = 256;                           // candidates a chunk may push
constexpr int kF32MaxSpans = 8;
constexpr uint32_t kKeyPos0 = 0x80000000u;             // the key of +0 (and of -0)
constexpr uint32_t kKeyNeg0 = 0x7FFFFFFFu;             // -0's key before folding
constexpr uint32_t kEdgeRaw = 0xFFFFFFFFu;             // a column outside the row: a NaN's bits, key 0

static_assert(kF32MaxK <= kF32Threads && kF32Cap <= kF32Threads, "one entry per thread in the rank merge");

struct F32Smem {
    uint4 stage[kF32ChunkVecs];                        // spilled keys: vector lv at stage[lv]
    uint64_t list[2][kF32MaxK];                        // the span's running list and the merge target
    uint64_t cand[kF32Cap];
    uint64_t gather[kF32MaxSpans][kF32MaxK];           // the leader's: every span's list
    uint64_t gather2[kF32MaxSpans / 2][kF32MaxK];
    int32_t glen[kF32MaxSpans], glen2[kF32MaxSpans / 2];
    uint32_t gflags[kF32MaxSpans], gnnz[kF32MaxSpans];
    uint32_t warp_t[kF32Warps];
    uint32_t red[2][kF32Warps];
    uint32_t n_cand, flags, nnz, kmax;
};

// ------------------------------------------------------------------ keys

__device__ __forceinline__ uint32_t f32_key_raw(uint32_t raw)
{
    return raw ^ ((uint32_t)((int32_t)raw >> 31) | kKeyPos0); // sign set: flip all; else set the sign
}

__device__ __forceinline__ uint32_t fold0(uint32_t key) { return key == kKeyNeg0 ? kKeyPos0 : key; }

// A floor on folded keys, as a floor on unfolded ones: -0's unfolded key sits
// just below +0's.
__device__ __forceinline__ uint32_t unfolded_floor(uint32_t f) { return f == kKeyPos0 ? kKeyNeg0 : f; }

__device__ __forceinline__ uint64_t f32_entry(uint32_t folded_key, int32_t col)
{
    return ((uint64_t)folded_key << 32) | (uint64_t)(~(uint32_t)col);
}

__device__ __forceinline__ int32_t f32_entry_col(uint64_t e) { return (int32_t)(~(uint32_t)e); }

__device__ __forceinline__ uint4 ld_stream4(const uint4 *p)
{
    uint4 q;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w)
                 : "l"(p));
    return q;
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_go() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Entries of a non-increasing list that exceed x (a binary search).
__device__ __forceinline__ int f32_count_greater(const uint64_t *list, int len, uint64_t x)
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

// Sum over the block (two alternating reduction rows: no barrier is needed
// before a row is reused).  Block-uniform.
__device__ __forceinline__ uint32_t f32_block_sum(uint32_t v, F32Smem &sm, int &parity)
{
    v = __reduce_add_sync(0xFFFFFFFFu, v);
    if ((threadIdx.x & 31) == 0) sm.red[parity][threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t s = 0;
#pragma unroll
    for (int w = 0; w < kF32Warps; ++w) s += sm.red[parity][w];
    parity ^= 1;
    return s;
}

// Row geometry: the row seen as 16-byte vectors from the 16-byte boundary at
// or below its start (m = the values before the row in the first vector).
struct F32Geom {
    const uint32_t *rowp;
    int32_t cols;
    int32_t m;              // 0..3
    int32_t nvec;           // vectors covering [-m, cols)
    int32_t vfull0, vfull1; // vectors [vfull0, vfull1) lie inside the row
};

__device__ __forceinline__ F32Geom f32_geometry(const uint32_t *rowp, int32_t cols)
{
    F32Geom g;
    g.rowp = rowp;
    g.cols = cols;
    g.m = (int32_t)((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3);
    g.nvec = (cols + g.m + 3) >> 2;
    g.vfull0 = g.m ? 1 : 0;
    g.vfull1 = (cols + g.m) >> 2;
    if (g.vfull1 < g.vfull0) g.vfull1 = g.vfull0;
    return g;
}

// A vector with a column outside the row: its values one by one, the outside
// ones as kEdgeRaw.
__device__ __noinline__ uint4 f32_edge_vector(const F32Geom &g, int32_t v)
{
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int32_t c = v * 4 + j - g.m;
        w[j] = (c >= 0 && c < g.cols) ? g.rowp[c] : kEdgeRaw;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The chunk's vectors [v0, v1) of the span: vector v0 + lv in thread
// lv % threads, register lv / threads; past v1: kEdgeRaw.
__device__ __forceinline__ void f32_load_chunk(uint32_t (&kv)[kF32Vec][4], const F32Geom &g, int32_t v0, int32_t v1)
{
    const uint4 *base = reinterpret_cast<const uint4 *>(g.rowp - g.m);
#pragma unroll
    for (int i = 0; i < kF32Vec; ++i) {
        const int32_t v = v0 + i * kF32Threads + (int32_t)threadIdx.x;
        uint4 q = make_uint4(kEdgeRaw, kEdgeRaw, kEdgeRaw, kEdgeRaw);
        if (v < v1) q = (v >= g.vfull0 && v < g.vfull1) ? ld_stream4(base + v) : f32_edge_vector(g, v);
        kv[i][0] = q.x;
        kv[i][1] = q.y;
        kv[i][2] = q.z;
        kv[i][3] = q.w;
    }
}

} // namespace

namespace {

// ------------------------------------------------------------------ the chunk

// The thread's largest key over the chunk.  With every value finite and in
// the span and the largest >= +0, it comes from the raw bits alone (the
// largest signed raw value) and kv stays raw (raw = true: the caller makes
// keys only if it needs them).  Otherwise kv becomes keys in place
// (unfolded: -0 stays just below +0; an infinity's key is valid as it is,
// with the row's flag recorded; exact where the thread saw a NaN or a column
// outside the span: NaN and outside columns become 0, and the row's flags
// are recorded).  The span's vectors are [.., v1).  Adds
// the thread's numbers to nnz.
__device__ __forceinline__ uint32_t f32_chunk_keys(uint32_t (&kv)[kF32Vec][4], const F32Geom &g, int32_t v0,
                                                   int32_t v1, uint32_t &nnz, F32Smem &sm, bool &raw)
{
    raw = false;
    int32_t smax = INT32_MIN;
    uint32_t umax = 0;
#pragma unroll
    for (int i = 0; i < kF32Vec; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            smax = max(smax, (int32_t)kv[i][j]);
            umax = max(umax, kv[i][j]);
        }
    uint32_t tmax = 0;
    if (smax < 0x7F800000 && umax < 0xFF800000u && smax >= 0) {
        // every value finite and inside the span, the largest >= +0
        raw = true;
        nnz += kF32Vec * 4;
        return (uint32_t)smax | kKeyPos0;
    }
    if (smax <= 0x7F800000 && umax <= 0xFF800000u) {
        // every value a number inside the span (all negative, or infinities
        // among them: a -inf mask, say); the infinities' keys are valid
#pragma unroll
        for (int i = 0; i < kF32Vec; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                kv[i][j] = f32_key_raw(kv[i][j]);
                tmax = max(tmax, kv[i][j]);
            }
        const uint32_t f = (smax == 0x7F800000 ? 2u : 0u) | (umax == 0xFF800000u ? 4u : 0u);
        if (f) atomicOr(&sm.flags, f);
        nnz += kF32Vec * 4;
        return tmax;
    }
    // the exact pass: outside columns (kEdgeRaw) are no value; NaN is a value
    // the count leaves out
    uint32_t flags = 0, cnt = 0;
#pragma unroll
    for (int i = 0; i < kF32Vec; ++i) {
        const int32_t v = v0 + i * kF32Threads + (int32_t)threadIdx.x;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int32_t c = v * 4 + j - g.m;
            const uint32_t raw = kv[i][j];
            uint32_t key = 0;
            if (c >= 0 && c < g.cols && v < v1) { // a column of the span (kEdgeRaw there is a NaN)
                if ((raw & 0x7FFFFFFFu) > 0x7F800000u) {
                    flags |= 1u;
                } else {
                    key = f32_key_raw(raw);
                    flags |= raw == 0x7F800000u ? 2u : (raw == 0xFF800000u ? 4u : 0u);
                    ++cnt;
                }
            }
            kv[i][j] = key;
            tmax = max(tmax, key);
        }
    }
    if (flags) atomicOr(&sm.flags, flags);
    nnz += cnt;
    return tmax;
}

// Prefilter bound of one chunk (block-uniform, one barrier).  The fw warps
// whose 32 lanes all hold data each find the j-th largest of their lanes'
// maxima, j = ceil(k / fw); the minimum t0 over them is reached by at least
// fw * j >= k values of the chunk, so no value below t0 can be in the top k
// of anything that contains the chunk.  With no such bound, 0.
__device__ __forceinline__ uint32_t f32_prefilter(uint32_t tmax, int nvalid_vecs, int k, F32Smem &sm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int fw = min(nvalid_vecs, kF32Threads) / 32;
    const int j = fw ? (k + fw - 1) / fw : 33;
    uint32_t tw = 0xFFFFFFFFu; // warps without a full set of lanes do not bound
    if (warp < fw) {
        tw = 0;
        if (j <= 32) {
            uint32_t v = fold0(tmax), cnt = 0;
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
    uint32_t t0 = (fw == 0 || j > 32) ? 0u : 0xFFFFFFFFu;
#pragma unroll
    for (int w = 0; w < kF32Warps; ++w) t0 = min(t0, sm.warp_t[w]);
    return t0;
}

// Exact selection for a chunk whose values reaching `floor` (a folded key)
// outnumber the candidate buffer: every key that can matter was spilled into
// `sm.stage` in column order (the other slots hold 0).  Writes the chunk's
// top k among them -- k entries, or all when fewer reach the floor -- to
// sm.cand and their number to sm.n_cand.  Block-uniform.
__device__ __noinline__ void f32_exact_select(int32_t col0, uint32_t floor, int k, F32Smem &sm)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t *keys = reinterpret_cast<const uint32_t *>(sm.stage);
    constexpr int kPer = kF32ChunkVecs * 4 / kF32Threads; // 32 contiguous keys a thread
    const int w0 = tid * kPer;
    uint32_t my_max = 0;
    for (int w = w0; w < w0 + kPer; ++w) my_max = max(my_max, fold0(keys[w]));
    my_max = __reduce_max_sync(0xFFFFFFFFu, my_max);
    if (tid == 0) sm.kmax = 0;
    __syncthreads();
    if (lane == 0) atomicMax(&sm.kmax, my_max);
    __syncthreads();
    // K* = the largest folded key at least k values reach
    uint64_t lo = floor, hi = (uint64_t)sm.kmax + 1u; // count(lo) > cap >= k, count(hi) = 0
    int parity = 0;
    while (hi - lo > 1) {
        const uint64_t mid = (lo + hi) >> 1;
        uint32_t c = 0;
        for (int w = w0; w < w0 + kPer; ++w) c += fold0(keys[w]) >= mid;
        if (f32_block_sum(c, sm, parity) >= (uint32_t)k)
            lo = mid;
        else
            hi = mid;
    }
    const uint32_t kstar = (uint32_t)lo;
    // one exclusive scan of (above << 16 | ties) over the threads' contiguous
    // column ranges places the entries above K* first, then the lowest
    // columns among the ties
    uint32_t mine = 0;
    for (int w = w0; w < w0 + kPer; ++w) {
        const uint32_t c = fold0(keys[w]);
        mine += c > kstar ? 0x10000u : (c == kstar ? 1u : 0u);
    }
    uint32_t incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += u;
    }
    if (lane == 31) sm.red[parity][warp] = incl;
    __syncthreads();
    uint32_t excl = incl - mine, total = 0;
#pragma unroll
    for (int w = 0; w < kF32Warps; ++w) {
        const uint32_t t = sm.red[parity][w];
        excl += w < warp ? t : 0u;
        total += t;
    }
    const uint32_t above = total >> 16;
    const uint32_t need = (uint32_t)k - above;
    const uint32_t taken = min(need, total & 0xFFFFu);
    uint32_t a_ord = excl >> 16, t_ord = excl & 0xFFFFu;
    for (int w = w0; w < w0 + kPer; ++w) {
        const uint32_t c = fold0(keys[w]);
        if (c > kstar) {
            sm.cand[a_ord++] = f32_entry(c, col0 + w);
        } else if (c == kstar) {
            if (t_ord < need) sm.cand[above + t_ord] = f32_entry(c, col0 + w);
            ++t_ord;
        }
    }
    __syncthreads();
    if (tid == 0) sm.n_cand = above + taken;
    __syncthreads();
}

} // namespace

namespace {

// ------------------------------------------------------------------ the kernel

// grid.x = rows * S; each row's S CTAs form one cluster (cluster rank = span).
template <int S>
__global__ void __launch_bounds__(kF32Threads, 4)
topk_f32_cluster_kernel(const uint32_t *__restrict__ logits, int32_t cols, int64_t row_stride, int32_t k,
                        int32_t *__restrict__ out_idx, uint32_t *__restrict__ out_val,
                        int32_t *__restrict__ out_count, uint32_t *__restrict__ out_mask)
{
    __shared__ F32Smem sm;
    const int tid = threadIdx.x, lane = tid & 31;
    const int span = (int)(blockIdx.x % S);
    const int64_t row = (int64_t)(blockIdx.x / S);
    const F32Geom g = f32_geometry(logits + row * row_stride, cols);
    const int32_t per = (g.nvec + S - 1) / S;
    const int32_t vb = min(g.nvec, span * per), ve = min(g.nvec, vb + per);
    // while the previous kernel on the stream ends: the first chunk's whole
    // vectors toward L2 (a hint only: L2 is where device memory is coherent)
    if (tid == 0) {
        const int32_t a = max(vb, g.vfull0), e = min(min(ve, vb + kF32ChunkVecs), g.vfull1);
        if (e > a)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<const uint4 *>(g.rowp - g.m) + a),
                         "r"((uint32_t)(e - a) * 16u)
                         : "memory");
    }
    grid_dependency_wait();
    if constexpr (S > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    if (tid == 0) {
        sm.flags = 0;
        sm.n_cand = 0;
        sm.nnz = 0;
    }
    __syncthreads();
    int run_i = 0, run_len = 0;
    uint32_t cand_base = 0, nnz = 0;
    uint32_t kv[kF32Vec][4];
    if (vb < ve) f32_load_chunk(kv, g, vb, ve);
    for (int32_t cb = vb; cb < ve; cb += kF32ChunkVecs) {
        const int32_t ce = min(ve, cb + kF32ChunkVecs);
        bool raw;
        const uint32_t tmax = f32_chunk_keys(kv, g, cb, ve, nnz, sm, raw);
        // the bound, a folded key: the running k-th (strictly) once the span's
        // list holds k entries, else the chunk's prefilter bound
        const uint32_t floor = run_len == k ? (uint32_t)(sm.list[run_i][k - 1] >> 32) + 1u
                                            : max(f32_prefilter(tmax, ce - cb, k, sm), 1u);
        const uint32_t uf = unfolded_floor(floor);
        // threads holding a key that reaches it spill their keys and count them
        const bool hit = tmax >= uf;
        uint32_t c = 0;
        if (hit) {
            if (raw) {
#pragma unroll
                for (int i = 0; i < kF32Vec; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) kv[i][j] = f32_key_raw(kv[i][j]);
            }
#pragma unroll
            for (int i = 0; i < kF32Vec; ++i) {
                sm.stage[i * kF32Threads + tid] = make_uint4(kv[i][0], kv[i][1], kv[i][2], kv[i][3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) c += kv[i][j] >= uf;
            }
        }
        // the registers are free: the next chunk's loads fly from here on
        if (ce < ve) f32_load_chunk(kv, g, ce, ve);
        // slots: a warp scan of the counts and one atomic a warp (warps
        // without a candidate skip it)
        if (__any_sync(0xFFFFFFFFu, c != 0)) {
            uint32_t incl = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += u;
            }
            uint32_t wbase = 0;
            if (lane == 31) wbase = atomicAdd(&sm.n_cand, incl);
            uint32_t slot = __shfl_sync(0xFFFFFFFFu, wbase, 31) + incl - c - cand_base;
            if (c != 0) {
                for (int i = 0; i < kF32Vec; ++i) {
                    const uint4 q = sm.stage[i * kF32Threads + tid];
                    const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
                    const int32_t col = (cb + i * kF32Threads + tid) * 4 - g.m;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (w4[j] >= uf) {
                            if (slot < (uint32_t)kF32Cap) sm.cand[slot] = f32_entry(fold0(w4[j]), col + j);
                            ++slot;
                        }
                    }
                }
            }
        }
        // no candidate anywhere (the steady state): the list, its bound and
        // the counter are unchanged and nothing of this chunk is read again
        if (!__syncthreads_or(c != 0)) continue;
        const uint32_t total = sm.n_cand;
        uint32_t n = total - cand_base;
        cand_base = total;
        if (n > (uint32_t)kF32Cap) {
            // heavy ties: exactly, from the spilled keys (the other threads'
            // slots hold an earlier chunk: zeroed)
            if (!hit) {
#pragma unroll
                for (int i = 0; i < kF32Vec; ++i) sm.stage[i * kF32Threads + tid] = make_uint4(0, 0, 0, 0);
            }
            __syncthreads();
            f32_exact_select(cb * 4 - g.m, floor, k, sm);
            n = sm.n_cand;
            cand_base = n;
        }
        // the candidates into the running list: a candidate's place is its
        // rank among the candidates plus the running entries above it; a
        // running entry's, its index plus the candidates above it
        {
            const uint64_t *run = sm.list[run_i];
            uint64_t *out = sm.list[run_i ^ 1];
            const int rl = run_len;
            if (tid < (int)n) {
                const uint64_t e = sm.cand[tid];
                int pos = f32_count_greater(run, rl, e);
                for (uint32_t u = 0; u < n; ++u) pos += sm.cand[u] > e;
                if (pos < k) out[pos] = e;
            }
            if (tid < rl) {
                const uint64_t e = run[tid];
                int pos = tid;
                for (uint32_t u = 0; u < n; ++u) pos += sm.cand[u] > e;
                if (pos < k) out[pos] = e;
            }
            run_len = min(k, rl + (int)n);
            run_i ^= 1;
        }
        __syncthreads();
    }
    {
        const uint32_t s = __reduce_add_sync(0xFFFFFFFFu, nnz);
        if (lane == 0 && s) atomicAdd(&sm.nnz, s);
    }
    __syncthreads();
    grid_dependents_go();

    const uint64_t *fin = sm.list[run_i];
    int flen = run_len;
    uint32_t flags = sm.flags, total = sm.nnz;
    if constexpr (S > 1) {
        // ---- the span's list into the leader's shared memory, then the merge
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); // every CTA has started
        cg::cluster_group cluster = cg::this_cluster();
        uint64_t *gl = cluster.map_shared_rank(&sm.gather[span][0], 0);
        for (int t = tid; t < run_len; t += kF32Threads) gl[t] = sm.list[run_i][t];
        if (tid == 0) {
            *cluster.map_shared_rank(&sm.glen[span], 0) = run_len;
            *cluster.map_shared_rank(&sm.gflags[span], 0) = sm.flags;
            *cluster.map_shared_rank(&sm.gnnz[span], 0) = sm.nnz;
        }
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        if (span != 0) return;
        flags = 0;
        total = 0;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            flags |= sm.gflags[s];
            total += sm.gnnz[s];
        }
        // pairwise merge tree over the S lists
        uint64_t(*src)[kF32MaxK] = sm.gather;
        uint64_t(*dst)[kF32MaxK] = sm.gather2;
        int32_t *src_len = sm.glen, *dst_len = sm.glen2;
        for (int nl = S; nl > 1; nl >>= 1) {
            for (int t = tid; t < nl * kF32MaxK; t += kF32Threads) {
                const int l = t / kF32MaxK, pos = t % kF32MaxK;
                if (pos >= src_len[l]) continue;
                const uint64_t x = src[l][pos];
                const int p = l ^ 1;
                const int o = pos + f32_count_greater(src[p], src_len[p], x);
                if (o < k) dst[l >> 1][o] = x;
            }
            if (tid < nl / 2) dst_len[tid] = min(k, src_len[2 * tid] + src_len[2 * tid + 1]);
            __syncthreads(); // the next level writes into the rows this one read
            uint64_t(*tl)[kF32MaxK] = src;
            src = dst;
            dst = tl;
            int32_t *tlen = src_len;
            src_len = dst_len;
            dst_len = tlen;
        }
        fin = src[0];
        flen = src_len[0];
    }
    // ---- the row: the first count entries, original bits re-read by column
    const int cnt = min((int)min((uint32_t)k, total), flen);
    for (int t = tid; t < k; t += kF32Threads) {
        const int64_t o = row * k + t;
        if (t < cnt) {
            const int32_t col = f32_entry_col(fin[t]);
            out_idx[o] = col;
            out_val[o] = g.rowp[col];
        } else {
            out_idx[o] = -1;
            out_val[o] = 0x7FC00000u;
        }
    }
    if (tid == 0) {
        out_count[row] = cnt;
        out_mask[row] = flags;
    }
}

} // namespace

namespace {

// ------------------------------------------------------------------ host side

template <int S>
cudaError_t launch_f32(const uint32_t *x, int64_t rows, int32_t cols, int64_t stride, int32_t k, int32_t *oi,
                       uint32_t *ov, int32_t *oc, uint32_t *om, cudaStream_t st)
{
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (S > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = S;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * S), 1, 1);
    cfg.blockDim = dim3(kF32Threads, 1, 1);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, topk_f32_cluster_kernel<S>, x, cols, stride, k, oi, ov, oc, om);
}

// Spans a row: with at least one row per SM, two; with fewer rows, the count
// that brings the grid to about two CTAs an SM, no span shorter than a chunk.
int f32_spans(int64_t rows, int64_t cols, int sm_count)
{
    // with a row per SM or more: one CTA per row when a row is at most one
    // chunk, or when two spans a row would take three waves or more of the
    // kernel's four CTAs an SM (1024 x 248320: 161.4 -> 148.7 us;
    // 1024 x 8192: 33.4 -> 13.5 us); else two spans
    if (rows >= sm_count)
        return (cols <= (int64_t)kF32ChunkVecs * 4 || 2 * rows >= 3 * 4 * (int64_t)sm_count) ? 1 : 2;
    int s = 1;
    while (s < kF32MaxSpans && rows * s * 2 < 2 * (int64_t)sm_count && cols / (2 * s) >= kF32ChunkVecs * 4) s <<= 1;
    return s;
}

} // namespace

// fp32 rows, k <= TF_TOPK_MAX_K, arguments already checked by the caller.
int tf_topk_internal_select_f32(const void *logits, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                                int32_t *out_idx, void *out_val, int32_t *out_count, uint32_t *out_mask,
                                int sm_count, void *stream)
{
    const uint32_t *x = static_cast<const uint32_t *>(logits);
    uint32_t *ov = static_cast<uint32_t *>(out_val);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int S = f32_spans(rows, cols, sm_count);
    const int64_t max_rows = (int64_t)INT32_MAX / kF32MaxSpans;
    for (int64_t r0 = 0; r0 < rows; r0 += max_rows) {
        const int64_t nr = rows - r0 < max_rows ? rows - r0 : max_rows;
        const uint32_t *xr = x + r0 * row_stride;
        int32_t *oi = out_idx + r0 * k, *oc = out_count + r0;
        uint32_t *ovr = ov + r0 * k, *om = out_mask + r0;
        cudaError_t e;
        switch (S) {
        case 1: e = launch_f32<1>(xr, nr, (int32_t)cols, row_stride, k, oi, ovr, oc, om, st); break;
        case 2: e = launch_f32<2>(xr, nr, (int32_t)cols, row_stride, k, oi, ovr, oc, om, st); break;
        case 4: e = launch_f32<4>(xr, nr, (int32_t)cols, row_stride, k, oi, ovr, oc, om, st); break;
        default: e = launch_f32<8>(xr, nr, (int32_t)cols, row_stride, k, oi, ovr, oc, om, st); break;
        }
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return tf_topk_internal_fail_cuda((int)e);
    }
    return TF_TOPK_OK;
}
