// sv_fast.cu -- one-pass row kernel for greedy rows and rows with top-k <= 32.
//
// Target-distribution build of jianc99/sglang PR #8 ("build_speculative_verify_
// target_probs"): the top-k is selected on the raw logits (a positive
// temperature keeps their order) and only the k kept values are divided by the
// temperature.  Here the selection streams each [rows, vocab] row from HBM
// exactly once and keeps at most a few dozen (logit, index) candidates:
//
//  * The (row, 4 KB chunk) units of all rows are split into one contiguous,
//    balanced range per warp of a persistent grid.  A range covers the tail of
//    one row, whole rows and the head of another; each of its row parts gives
//    one partial list.  Warps never wait for one another while streaming.
//  * Lane 0 of each warp keeps a private ring of 3 shared-memory stages filled
//    with bulk asynchronous copies (cp.async.bulk, completion on mbarriers,
//    bounded waits).
//  * Each lane takes a NaN-propagating packed max (max.NaN.bf16x2) of its
//    8 x 16 B of a chunk.  In a part's first chunk theta = the k-th largest of
//    the 32 lane maxima (bisection on the key bits with warp votes): at least
//    k elements reach it.  The warp keeps the part's best k composite keys
//    (logit, inverted index) as a sorted list across its lanes.  Lanes whose
//    vectors reach theta re-read them from the stage and append the elements
//    that do to a 32-key buffer of the warp; a full buffer is sorted (bitonic
//    network) and merged into the list.  theta moves only between chunks: to
//    the exact k-th best so far after a part's first chunk and whenever a
//    chunk ends with the buffer half full.  Once k entries exist an element
//    must beat theta strictly (its index is higher than those of the entries,
//    so a tie cannot win).  A chunk with no lane maximum above theta costs one
//    vote.
//  * The k-th entry of a full part list is a lower bound on the row's k-th
//    largest logit.  Parts publish it (atomicMax on the row's order key) and
//    read the others' one chunk ahead; an element below the best bound
//    cannot be kept (one equal to it can: it may have a lower index).  The
//    row's parts run at different times (a range starts with the tail of one
//    row and ends with the head of the next), so a part that starts late
//    starts with a near-final threshold.
//  * At a part's end the warp writes its top k, ordered by (logit desc, index
//    asc), and counts the part in the row's counter.  The warp that finishes a
//    row's last part merges the row's lists (bitonic merges of sorted lists of
//    32) and builds the row's distribution in fp64 from the <= 32 kept values:
//    temperature, top-p over the top-k mass, normaliser, the probability of
//    the row's token, and the kept list in index order for the resample.
//    Greedy rows are the k = 1 case (argmax, lowest index wins ties).
//  * In a verify call the warp that finalises a request's last row then runs
//    the request's chain walk (acceptance, residual or bonus draw; see
//    sv_walk.cuh), so no separate chain launch waits for the whole grid.
#include <math.h>

#include "sv_internal.cuh"
#include "sv_walk.cuh"

namespace sv {
namespace {

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
// Larger of the two bf16 halves of a word, as fp32 (NaN-propagating).
__device__ __forceinline__ float bf16x2_hmax(uint32_t w)
{
    return fmax_nan(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// ---- per-warp shared-memory ring fed by bulk async copies (cp.async.bulk) ----
constexpr int kCtaWarps = kFastThreads / 32;
constexpr int kStages = 3;                                  // chunks in flight per warp
constexpr int kWarpChunkBytes = 32 * kFastVecs * 16;        // 4 KB: one warp chunk of either dtype
constexpr int kBufCap = 32;                                 // buffered candidates per warp
constexpr int kMergeAt = 16;                                // a chunk's end merges a buffer this full

// Ragged edge of a row (or a misaligned row): element loads, -inf past the end.
template <int DT>
__device__ __forceinline__ uint4 load_edge(const char* row, int e0, int vocab)
{
    uint32_t w[4];
    if (DT == 0) {
        const uint16_t* r16 = (const uint16_t*)row;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i0 = e0 + 2 * q, i1 = i0 + 1;
            const uint32_t lo = i0 < vocab ? (uint32_t)r16[i0] : 0xFF80u;
            const uint32_t hi = i1 < vocab ? (uint32_t)r16[i1] : 0xFF80u;
            w[q] = lo | (hi << 16);
        }
    } else {
        const uint32_t* r32 = (const uint32_t*)row;
#pragma unroll
        for (int q = 0; q < 4; ++q) w[q] = (e0 + q) < vocab ? r32[e0 + q] : 0xFF800000u;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Vector vi (16 bytes) of a chunk whose first `bytes` bytes sit in the stage:
// from the stage when it is all there, else from the row.
template <int DT>
__device__ __forceinline__ uint4 stage_or_edge(const unsigned char* stg, uint32_t bytes, const char* row, int c0, int vi,
                                               int vocab)
{
    constexpr int EPV = DT == 0 ? 8 : 4;
    if ((uint32_t)(vi * 16 + 16) <= bytes) return ld_shared_v4(stg + vi * 16);
    return load_edge<DT>(row, c0 + vi * EPV, vocab);
}
// Element q (0 .. EPV-1) of a 16-byte vector as fp32, for a q known at compile time.
template <int DT>
__device__ __forceinline__ float vec_elem(const uint4& v, int q)
{
    const uint32_t w = (DT == 0 ? (q >> 1) : q) == 0 ? v.x
                     : (DT == 0 ? (q >> 1) : q) == 1 ? v.y
                     : (DT == 0 ? (q >> 1) : q) == 2 ? v.z : v.w;
    if (DT == 0) return __uint_as_float((q & 1) ? (w & 0xFFFF0000u) : (w << 16));
    return __uint_as_float(w);
}
// The same for a run-time q, by selects rather than an indexed register array.
template <int DT>
__device__ __forceinline__ float vec_elem_dyn(const uint4& v, int q)
{
    const int j = DT == 0 ? (q >> 1) : q;
    const uint32_t lo = (j & 1) ? v.y : v.x, hi = (j & 1) ? v.w : v.z;
    const uint32_t w = (j & 2) ? hi : lo;
    if (DT == 0) return __uint_as_float((q & 1) ? (w & 0xFFFF0000u) : (w << 16));
    return __uint_as_float(w);
}

// Byte offset of a row and the bulk-copied bytes of one warp chunk of it.
template <int DT>
__device__ __forceinline__ const char* task_row(const RowsArgs& a, const RowTask& t)
{
    constexpr int ESZ = DT == 0 ? 2 : 4;
    const int64_t stride = t.is_draft ? a.stride_d : a.stride_t;
    return (const char*)(t.is_draft ? a.drf : a.tgt) + (size_t)t.row * (size_t)stride * ESZ;
}
template <int DT>
__device__ __forceinline__ uint32_t chunk_bytes(const char* row, int c0, int vocab)
{
    constexpr int ESZ = DT == 0 ? 2 : 4;
    constexpr int CHUNK = kWarpChunkBytes / ESZ;
    const int n_here = min(CHUNK, vocab - c0);
    const char* src = row + (size_t)c0 * ESZ;
    return ((uintptr_t)src & 15u) ? 0u : ((uint32_t)(n_here * ESZ) & ~15u);
}

// Balanced split of U = tasks x chunks units over W warps: warp w takes
// [w U / W, (w + 1) U / W).  With W <= U every warp has at least one unit,
// and a warp's range touches at most Pw = ceil(ceil(U / W) / nc) + 1 rows, so
// W * Pw <= tasks + 3 W part slots suffice.
struct Split {
    long long U, W;
    int nc, Pw;
};
__device__ __forceinline__ long long split_lo(const Split& s, long long w) { return w * s.U / s.W; }
// The warp whose range holds unit g: the largest w with split_lo(w) <= g.
__device__ __forceinline__ long long split_owner(const Split& s, long long g) { return ((g + 1) * s.W + s.U - 1) / s.U - 1; }
__device__ __forceinline__ size_t part_slot(const Split& s, long long w, int t)
{
    return (size_t)(w * s.Pw + (t - split_lo(s, w) / s.nc));
}

// k-th largest (1 <= k <= 32) of one NB-bit key per lane: bisection on the
// key bits, one warp vote per bit.
template <int NB>
__device__ __forceinline__ uint32_t warp_kth_key(uint32_t key, int k)
{
    uint32_t pre = 0u;
#pragma unroll
    for (int b = NB - 1; b >= 0; --b) {
        const uint32_t tv = pre | (1u << b);
        if (__popc(__ballot_sync(0xFFFFFFFFu, key >= tv)) >= k) pre = tv;
    }
    return pre;
}

// Top 32 of two descending lists of 32 (lane i holds element i of each), as a
// descending list: the elementwise max against the reversed second list is
// bitonic and holds the top 32; five compare-exchange stages sort it.
__device__ __forceinline__ unsigned long long merge_desc(unsigned long long acc, unsigned long long b)
{
    const int lane = threadIdx.x & 31;
    const unsigned long long rb = __shfl_sync(0xFFFFFFFFu, b, 31 - lane);
    unsigned long long c = acc > rb ? acc : rb;
#pragma unroll
    for (int j = 16; j; j >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xFFFFFFFFu, c, j);
        c = (lane & j) ? (x < c ? x : c) : (x > c ? x : c);
    }
    return c;
}

// Descending bitonic sort of one key per lane over the first P lanes, P the
// power of two >= n (lanes >= n hold 0 and stay below every key).
__device__ __forceinline__ unsigned long long sort_desc(unsigned long long v, int n)
{
    const int lane = threadIdx.x & 31;
    int P = 1;
    while (P < n) P <<= 1;
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride; stride >>= 1) {
            const unsigned long long x = __shfl_xor_sync(0xFFFFFFFFu, v, stride);
            const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
            v = keep_max ? (x > v ? x : v) : (x < v ? x : v);
        }
    }
    return v;
}

// Merges the n (<= 32) buffered keys of a warp into its descending list.
__device__ __noinline__ unsigned long long merge_buffer(unsigned long long list, const unsigned long long* buf, int n)
{
    const int lane = threadIdx.x & 31;
    __syncwarp();
    const unsigned long long b = lane < n ? buf[lane] : 0ull;
    __syncwarp();   // the buffer may be refilled after this
    return merge_desc(list, sort_desc(b, n));
}

__device__ __forceinline__ void finalize_list(const RowTask& task, RowInfo* info, unsigned long long acc, uint32_t st);

// Fast task t's parts' lists merged (one warp).  Out of line: it runs once
// per row.  Its distribution goes to the task's RowInfo, or, for a vocabulary
// shard (shard_out set), the merged list goes to the task's record with the
// indices of the whole vocabulary (the shard starts at element v0).
__device__ __noinline__ void finalize_row(TaskList tasks, RowInfo* infos, const Partial* parts, int t, Split sp,
                                         Partial* shard_out, uint32_t v0)
{
    const int lane = threadIdx.x & 31;
    const RowTask task = tasks.get(t);
    const long long g0 = (long long)t * sp.nc;
    const long long w0 = split_owner(sp, g0), w1 = split_owner(sp, g0 + sp.nc - 1);
    unsigned long long acc = 0ull;
    uint32_t st = 0u;
    for (long long wb = w0; wb <= w1; wb += 4) {   // four parts' loads in flight at once
        unsigned long long key[4];
        uint32_t cnt[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            cnt[j] = 0u;
            key[j] = 0ull;
            if (wb + j <= w1) {
                const Partial* P = parts + part_slot(sp, wb + j, t);
                cnt[j] = __ldcg(&P->count);
                st |= __ldcg(&P->status);
                key[j] = __ldcg(&P->keys[lane]);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (wb + j <= w1) acc = merge_desc(acc, lane < (int)cnt[j] ? key[j] : 0ull);
    }
    if (shard_out) {   // a shard's record: its top k with whole-vocabulary indices
        const int k = task.k_eff < kFastK ? task.k_eff : kFastK;
        const unsigned long long ck = lane < k ? acc : 0ull;
        const int n = __popc(__ballot_sync(0xFFFFFFFFu, ck != 0ull));
        Partial* R = shard_out + task.slot;
        if (lane < n) R->keys[lane] = ck - (unsigned long long)v0;   // the inverted index drops by v0
        if (lane == 0) {
            R->status = st & (uint32_t)kNonfinite;
            R->count = (uint32_t)n;
        }
        return;
    }
    finalize_list(task, infos + task.slot, acc, st);
}

// The distribution of a fast row from its top-k composite keys (acc, lane i
// the i-th best) and status bits (one warp): argmax, temperature, top-p over
// the top-k mass, normaliser, p of the row's token, the kept list.
__device__ __forceinline__ void finalize_list(const RowTask& task, RowInfo* info, unsigned long long acc, uint32_t st)
{
    const int lane = threadIdx.x & 31;
    const int k = task.k_eff < kFastK ? task.k_eff : kFastK;
    const unsigned long long ck = lane < k ? acc : 0ull;
    const int n_top = __popc(__ballot_sync(0xFFFFFFFFu, ck != 0ull));
    const float lv = ckey_value(ck);
    const int li = ckey_index(ck);
    const float m = __shfl_sync(0xFFFFFFFFu, lv, 0);
    const int amax = __shfl_sync(0xFFFFFFFFu, li, 0);
    const float T = task.temp;
    int status = (int)st & kNonfinite;
    if (status == 0 && T > 0.0f && m == -INFINITY) status = kEmpty;
    if (lane == 0) {
        info->desc.max_logit = m;
        info->desc.argmax = amax;
        info->desc.status = status;
        info->desc.temperature = T;
        info->cut_count = -1;
    }
    if (status != 0) {
        if (lane == 0) {
            info->desc.log_norm = 0.0f;
            info->desc.cutoff_logit = m;
            info->desc.cutoff_ties = 0;
            info->desc.kept = 0;
            info->p_token = nan("");
            info->z = 0.0;
            info->n_list = -1;
        }
        return;
    }
    if (T == 0.0f) {
        if (lane == 0) {
            info->desc.log_norm = 0.0f;
            info->desc.cutoff_logit = m;
            info->desc.cutoff_ties = 1;
            info->desc.kept = 1;
            info->p_token = task.token >= 0 ? (task.token == amax ? 1.0 : 0.0) : nan("");
            info->z = 1.0;
            info->z_rest = 0.0;
            info->n_list = 1;
            info->list_idx[0] = amax;
            info->list_p[0] = 1.0;
        }
        return;
    }
    // Sampling row: masses of the kept values in fp64, in sorted order, and
    // their running sums (a warp scan): the top-p prefix is the first one
    // whose running sum reaches top_p times the top-k mass.
    const double inv_t = 1.0 / (double)T;
    const double e = lane < n_top ? exp(((double)lv - (double)m) * inv_t) : 0.0;
    double cum = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, cum, o);
        if (lane >= o) cum += y;
    }
    int kept = n_top;
    if (task.top_p < 1.0f) {
        const double target = (double)task.top_p * __shfl_sync(0xFFFFFFFFu, cum, 31);
        const unsigned reach = __ballot_sync(0xFFFFFFFFu, lane < n_top && cum >= target);
        if (reach) kept = __ffs(reach);
    }
    const double z = __shfl_sync(0xFFFFFFFFu, cum, kept - 1);
    const bool in = lane < kept;
    double z_rest = (in && lane > 0) ? e : 0.0;   // kept mass after the top token
#pragma unroll
    for (int o = 16; o; o >>= 1) z_rest += __shfl_xor_sync(0xFFFFFFFFu, z_rest, o);
    const double p = in ? e * (1.0 / z) : 0.0;
    const float cut = __shfl_sync(0xFFFFFFFFu, lv, kept - 1);
    const int ties = __popc(__ballot_sync(0xFFFFFFFFu, in && lv == cut));
    int rank = 0;
    for (int j = 0; j < kept; ++j) rank += (__shfl_sync(0xFFFFFFFFu, li, j) < li) ? 1 : 0;
    if (in) {
        info->list_idx[rank] = li;
        info->list_p[rank] = p;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, in && li == task.token);
    const double ptok = hit ? __shfl_sync(0xFFFFFFFFu, p, __ffs(hit) - 1) : 0.0;
    if (lane == 0) {
        info->desc.log_norm = logf((float)z);   // z is in [1, 32]: fp32 is exact enough for a float output
        info->desc.cutoff_logit = cut;
        info->desc.cutoff_ties = ties;
        info->desc.kept = kept;
        info->p_token = task.token >= 0 ? ptok : nan("");
        info->z = z;
        info->z_rest = z_rest;
        info->n_list = kept;
    }
}

template <int DT>
__global__ void __launch_bounds__(kFastThreads, 1) fast_rows_kernel(const __grid_constant__ RowsArgs a)
{
    constexpr int EPV = DT == 0 ? 8 : 4;
    constexpr int ESZ = DT == 0 ? 2 : 4;
    constexpr int CHUNK = 32 * kFastVecs * EPV;   // elements of a warp chunk
    static_assert(CHUNK * ESZ == kWarpChunkBytes, "one warp chunk fills one ring stage");
    constexpr unsigned FULL = 0xFFFFFFFFu;
    extern __shared__ __align__(128) unsigned char ring[];   // warps x kStages x 4 KB
    __shared__ __align__(8) unsigned long long s_bar[kCtaWarps][kStages];
    __shared__ unsigned long long s_buf[kCtaWarps][kBufCap]; // candidate buffer of each warp
    __shared__ double s_qp[kCtaWarps][kFastK];               // chain walk: the draft row's kept list
    __shared__ int s_qi[kCtaWarps][kFastK];

    pdl_enter();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_tasks = a.counters->n_fast;
    Split sp;
    sp.nc = (a.vocab + CHUNK - 1) / CHUNK;
    sp.U = (long long)n_tasks * sp.nc;
    sp.W = min((long long)gridDim.x * kCtaWarps, sp.U);
    const long long w = (long long)blockIdx.x * kCtaWarps + warp;
    if (w >= sp.W) return;   // whole warps leave: nothing below waits on the block
    sp.Pw = (int)(((sp.U + sp.W - 1) / sp.W + sp.nc - 1) / sp.nc) + 1;
    const long long lo = split_lo(sp, w), hi = split_lo(sp, w + 1);
    unsigned long long* bar = s_bar[warp];
    unsigned char* wring = ring + (size_t)warp * (kStages * kWarpChunkBytes);
    unsigned long long* buf = s_buf[warp];

    // The range's parts: part j is row t_lo + j, chunks [part_c0(j),
    // part_c1(j)).  Odd warps take their parts last to first (chunks still in
    // order within a part): a row split between an even warp and the odd one
    // after it is then the first part of both or the last part of both, so
    // only every other split row finishes at the end of the ranges.
    const int t_lo = (int)(lo / sp.nc);
    const int np = (int)((hi - 1) / sp.nc) - t_lo + 1;
    const bool rev = (w & 1) != 0;
    auto part_c0 = [&](int j) { return (int)(max(lo, (long long)(t_lo + j) * sp.nc) - (long long)(t_lo + j) * sp.nc); };
    auto part_c1 = [&](int j) {
        return (int)(min(hi, (long long)(t_lo + j + 1) * sp.nc) - (long long)(t_lo + j) * sp.nc);
    };

    // Producer (lane 0): the part and chunk to copy next, the row, the stage.
    int p_i = 0, p_j = rev ? np - 1 : 0;
    int p_c = part_c0(p_j), p_c1 = part_c1(p_j);
    int p_slot = 0, p_n = 0;   // p_n: copies issued
    const char* p_row = nullptr;
    auto produce = [&]() {
        if (p_i >= np) return;
        const int c0 = p_c * CHUNK;
        const uint32_t bytes = chunk_bytes<DT>(p_row, c0, a.vocab);
        unsigned long long* b = &bar[p_slot];
        if (bytes) {
            mbar_expect_tx(b, bytes);
            bulk_g2s(wring + p_slot * kWarpChunkBytes, p_row + (size_t)c0 * ESZ, bytes, b);
        } else {
            mbar_arrive(b);
        }
        if (++p_slot == kStages) p_slot = 0;
        ++p_n;
        if (++p_c == p_c1 && ++p_i < np) {
            p_j = rev ? np - 1 - p_i : p_i;
            p_c = part_c0(p_j);
            p_c1 = part_c1(p_j);
            p_row = task_row<DT>(a, a.fast_tasks.get(t_lo + p_j));
        }
    };
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1u);
        mbar_fence_init();
        p_row = task_row<DT>(a, a.fast_tasks.get(t_lo + p_j));
        for (int s = 0; s < kStages; ++s) produce();
    }
    __syncwarp();

    int c_slot = 0, c_n = 0;   // c_n: chunks consumed
    uint32_t c_phase = 0u;
    for (int i = 0; i < np; ++i) {
        // One row part: chunks [c, c_end) of task t.  The part's top k live in
        // `list` (lane i: i-th best composite key, 0 = empty).
        const int j = rev ? np - 1 - i : i;
        const int t = t_lo + j;
        const int c = part_c0(j), c_end = part_c1(j);
        const RowTask task = a.fast_tasks.get(t);
        const char* row = task_row<DT>(a, task);
        const int k = task.k_eff < kFastK ? task.k_eff : kFastK;
        unsigned long long list = 0ull;
        int nb = 0;   // keys in the warp's buffer
        int strict = 0, bad = 0;
        float theta = -INFINITY;
        // Lower bound on the row's k-th largest logit published by the row's
        // other parts (the k-th entry of a full part list is one): elements
        // below it cannot be kept, ties with it can (they may have lower
        // indices).  Read one chunk ahead so its latency stays hidden.
        uint32_t* bound_at = &a.row_sync[t].bound;
        uint32_t bkey = 0u, bnext = __ldcg(bound_at);
        float bval = -INFINITY;
        for (int cc = c; cc < c_end; ++cc) {
            const int c0 = cc * CHUNK;
            const uint32_t bytes = chunk_bytes<DT>(row, c0, a.vocab);
            if (!__all_sync(FULL, mbar_wait(&bar[c_slot], c_phase))) {
                // A bulk copy never arrived: flag it, let this warp's copies in
                // flight land (bounded), fail the requests of the rows this
                // warp has not finished (those rows will never be complete),
                // and leave.
                if (lane == 0) {
                    atomicOr(&a.counters->timeout, 1);
                    int s = c_slot;
                    uint32_t ph = c_phase;
                    for (int q = c_n; q < p_n; ++q) {
                        mbar_wait(&bar[s], ph);
                        if (++s == kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                }
                __syncwarp();
                if (a.chain.fuse)
                    for (int ii = i; ii < np; ++ii)
                        chain_fail(a.chain, a.fast_tasks.get(t_lo + (rev ? np - 1 - ii : ii)).req);
                return;
            }
            const unsigned char* stg = wring + c_slot * kWarpChunkBytes;
            const bool full = bytes == (uint32_t)kWarpChunkBytes;   // the chunk is all in the stage
            uint4 v[kFastVecs];
            if (full) {
#pragma unroll
                for (int i = 0; i < kFastVecs; ++i) v[i] = ld_shared_v4(stg + (i * 32 + lane) * 16);
            } else {
#pragma unroll
                for (int i = 0; i < kFastVecs; ++i) v[i] = stage_or_edge<DT>(stg, bytes, row, c0, i * 32 + lane, a.vocab);
            }
            // Per-vector NaN-propagating maxima, then the lane maximum.
            uint32_t m2[kFastVecs];
            float vmx[kFastVecs];
            float tmax;
            if constexpr (DT == 0) {
#pragma unroll
                for (int i = 0; i < kFastVecs; ++i)
                    m2[i] = bmax2_nan(bmax2_nan(v[i].x, v[i].y), bmax2_nan(v[i].z, v[i].w));
                const uint32_t mm = bmax2_nan(bmax2_nan(bmax2_nan(m2[0], m2[1]), bmax2_nan(m2[2], m2[3])),
                                              bmax2_nan(bmax2_nan(m2[4], m2[5]), bmax2_nan(m2[6], m2[7])));
                tmax = bf16x2_hmax(mm);
            } else {
#pragma unroll
                for (int i = 0; i < kFastVecs; ++i)
                    vmx[i] = fmax_nan(fmax_nan(__uint_as_float(v[i].x), __uint_as_float(v[i].y)),
                                      fmax_nan(__uint_as_float(v[i].z), __uint_as_float(v[i].w)));
                tmax = fmax_nan(fmax_nan(fmax_nan(vmx[0], vmx[1]), fmax_nan(vmx[2], vmx[3])),
                                fmax_nan(fmax_nan(vmx[4], vmx[5]), fmax_nan(vmx[6], vmx[7])));
            }
            bad |= (isnan(tmax) || tmax == INFINITY) ? 1 : 0;
            if (cc == c) {   // first chunk of the part: k-th largest lane maximum
                if constexpr (DT == 0)
                    theta = f32_of_key16(warp_kth_key<16>(key16_of_bf16(__float_as_uint(tmax) >> 16), k));
                else
                    theta = f32_of_key(warp_kth_key<32>(key_of_f32_bits(__float_as_uint(tmax)), k));
            }
            // The chunk's filter: the part's own threshold, or the published
            // bound when that is higher.
            float th = theta;
            int sf = strict;
            if (bval > th) {
                th = bval;
                sf = 0;
            }
            if (__ballot_sync(FULL, sf ? tmax > th : tmax >= th)) {
                // Each lane re-reads its vectors that reach theta from the
                // stage and marks their elements that do; the marked elements
                // of the warp are merged into the list.  Every element of this
                // chunk has a higher index than the entries kept from earlier
                // chunks, so the order of the merges does not matter and, once
                // the list was full at the chunk's start, a tie with theta
                // cannot enter.
                uint32_t pend = 0u;
#pragma unroll
                for (int i = 0; i < kFastVecs; ++i) {
                    float vm;
                    if constexpr (DT == 0)
                        vm = bf16x2_hmax(m2[i]);
                    else
                        vm = vmx[i];
                    pend |= ((sf ? vm > th : vm >= th) ? 1u : 0u) << i;
                }
                while (__any_sync(FULL, pend != 0u)) {
                    uint4 vv = make_uint4(0u, 0u, 0u, 0u);
                    int e0 = 0;
                    uint32_t cm = 0u;   // elements of vv to insert
                    if (pend) {
                        const int i = __ffs(pend) - 1;
                        pend &= pend - 1u;
                        vv = full ? ld_shared_v4(stg + (i * 32 + lane) * 16)
                                  : stage_or_edge<DT>(stg, bytes, row, c0, i * 32 + lane, a.vocab);
                        e0 = c0 + (i * 32 + lane) * EPV;
#pragma unroll
                        for (int q = 0; q < EPV; ++q) {
                            const float x = vec_elem<DT>(vv, q);
                            cm |= ((sf ? x > th : x >= th) && e0 + q < a.vocab ? 1u : 0u) << q;
                        }
                    }
                    // One marked element per lane at a time goes to the
                    // warp's buffer (merged into the list when it is full).
                    while (__any_sync(FULL, cm != 0u)) {
                        unsigned long long key = 0ull;
                        if (cm) {
                            const int q = __ffs(cm) - 1;
                            cm &= cm - 1u;
                            key = ckey(vec_elem_dyn<DT>(vv, q), (uint32_t)(e0 + q));
                        }
                        const unsigned own = __ballot_sync(FULL, key != 0ull);
                        const int add = __popc(own);
                        if (nb + add > kBufCap) {
                            list = merge_buffer(list, buf, nb);
                            nb = 0;
                        }
                        if (key) buf[nb + __popc(own & ((1u << lane) - 1u))] = key;
                        nb += add;
                    }
                }
            }
            // theta moves only between chunks: after a part's first chunk, or
            // when the buffer holds enough to be worth a merge.
            if (cc == c || nb >= kMergeAt) {
                if (nb) {
                    list = merge_buffer(list, buf, nb);
                    nb = 0;
                }
                const unsigned long long kth = __shfl_sync(FULL, list, k - 1);
                if (kth != 0ull) {   // k entries: theta is the exact k-th best so far
                    const float nt = ckey_value(kth);
                    if (lane == 0 && (!strict || nt > theta) && nt > bval)
                        atomicMax(bound_at, key_of_f32_bits(__float_as_uint(nt)));
                    theta = nt;
                    strict = 1;
                }
            }
            if (bnext > bkey) {
                bkey = bnext;
                bval = f32_of_key(bkey);
            }
            bnext = __ldcg(bound_at);
            __syncwarp();   // every lane is done with the stage: refill it
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                produce();
            }
            if (++c_slot == kStages) {
                c_slot = 0;
                c_phase ^= 1u;
            }
            ++c_n;
        }

        // The part's list (and its bound), then the row's counter; the last
        // part finalises.
        if (nb) list = merge_buffer(list, buf, nb);
        {
            const unsigned long long kth = __shfl_sync(FULL, list, k - 1);
            if (lane == 0 && kth != 0ull && ckey_value(kth) > bval)
                atomicMax(bound_at, key_of_f32_bits(__float_as_uint(ckey_value(kth))));
        }
        const int m = __popc(__ballot_sync(FULL, lane < k && list != 0ull));
        const int any_bad = __any_sync(FULL, bad);
        Partial* P = a.partials + part_slot(sp, w, t);
        if (!any_bad && lane < m) P->keys[lane] = list;
        if (lane == 0) {
            P->status = any_bad ? (uint32_t)kNonfinite : 0u;
            P->count = any_bad ? 0u : (uint32_t)m;
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            const long long g0 = (long long)t * sp.nc;
            const int parts = (int)(split_owner(sp, g0 + sp.nc - 1) - split_owner(sp, g0) + 1);
            last = atomicAdd(&a.row_sync[t].done, 1) == parts - 1;
        }
        if (__shfl_sync(FULL, last, 0)) {
            __threadfence();
            finalize_row(a.fast_tasks, a.info, a.partials, t, sp, a.shard_out, a.shard_v0);
            if (a.chain.fuse) {   // the request's last row: its chain walk
                __threadfence();
                __syncwarp();
                int chain = 0;
                if (lane == 0) chain = atomicAdd(&a.chain.req_done[task.req], 1) == task.req_rows - 1;
                if (__shfl_sync(FULL, chain, 0)) {
                    __threadfence();
                    chain_walk(a.chain, task.req, s_qp[warp], s_qi[warp], false);
                }
            }
        }
    }
}

// Vocabulary-sharded verify, the merge: the records of the row's slot from
// every shard (each the shard's top k with whole-vocabulary indices) merged
// into the row's top k, then the same finalisation as an unsharded row.  One
// warp per fast task, records of shard s at records + s * slots.
__global__ void __launch_bounds__(256) shard_merge_kernel(const __grid_constant__ RowsArgs a, const Partial* records,
                                                          int n_shards, int slots)
{
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int n_tasks = a.counters->n_fast;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < n_tasks; t += (gridDim.x * blockDim.x) >> 5) {
        const RowTask task = a.fast_tasks.get(t);
        unsigned long long acc = 0ull;
        uint32_t st = 0u;
        for (int s0 = 0; s0 < n_shards; s0 += 4) {   // four records' loads in flight at once
            unsigned long long key[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                key[j] = 0ull;
                if (s0 + j < n_shards) {
                    const Partial* R = records + (size_t)(s0 + j) * (size_t)slots + (size_t)task.slot;
                    const uint32_t cnt = R->count;
                    st |= R->status;
                    key[j] = lane < (int)cnt ? R->keys[lane] : 0ull;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (s0 + j < n_shards) acc = merge_desc(acc, key[j]);
        }
        finalize_list(task, a.info + task.slot, acc, st);
    }
}

}  // namespace

template <int DT>
cudaError_t launch_fast_rows_t(const RowsArgs& a, cudaStream_t s)
{
    // Persistent grid: the CTAs that fit at once (at most kMaxRowWarps warps),
    // each warp with its own ring.
    const size_t smem = (size_t)kCtaWarps * kStages * kWarpChunkBytes;
    static int blocks_per_sm[128] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& nb = blocks_per_sm[(dev >= 0 && dev < 128) ? dev : 0];
    if (nb == 0) {
        cudaError_t e = cudaFuncSetAttribute(fast_rows_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fast_rows_kernel<DT>, kFastThreads, smem);
        if (e != cudaSuccess) return e;
        if (nb < 1) nb = 1;
    }
    int grid = a.num_sms * nb;
    if (grid > kMaxRowWarps / kCtaWarps) grid = kMaxRowWarps / kCtaWarps;
    return launch_pdl(fast_rows_kernel<DT>, dim3(grid), dim3(kFastThreads), smem, s, a);
}

cudaError_t launch_fast_rows(const RowsArgs& a, cudaStream_t s)
{
    return a.dtype == 0 ? launch_fast_rows_t<0>(a, s) : launch_fast_rows_t<1>(a, s);
}

}  // namespace sv

namespace sv {
cudaError_t launch_shard_merge(const RowsArgs& a, const void* records, int n_shards, int slots, cudaStream_t s)
{
    int grid = (a.max_tasks + 7) / 8;
    if (grid > 4 * a.num_sms) grid = 4 * a.num_sms;
    if (grid < 1) grid = 1;
    return launch_pdl(shard_merge_kernel, dim3(grid), dim3(256), 0, s, a, static_cast<const Partial*>(records),
                      n_shards, slots);
}
}  // namespace sv
