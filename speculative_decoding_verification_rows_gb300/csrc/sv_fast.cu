// sv_fast.cu -- one-pass row kernel for greedy rows and rows with top-k <= 32.
//
// Target-distribution build of jianc99/sglang PR #8 ("build_speculative_verify_
// target_probs"): the top-k is selected on the raw logits (a positive
// temperature keeps their order) and only the k kept values are divided by the
// temperature.  Here the selection streams each [rows, vocab] row from HBM
// exactly once and keeps at most a few hundred (logit, index) candidates:
//
//  * A persistent CTA owns segments of rows (4 chunks of 32 KB).  Thread 0
//    keeps a ring of 3 shared-memory stages filled with bulk asynchronous
//    copies (cp.async.bulk, completion on mbarriers, bounded waits), so loads
//    stay in flight while the CTA selects.
//  * Each thread takes a NaN-propagating packed max (max.NaN.bf16x2) of its
//    8 x 16 B of a chunk.  In a segment's first chunk theta = the k-th largest
//    of the 256 thread maxima (a radix select with warp-aggregated shared
//    atomics): at least k elements are >= theta, and few more.
//  * Only threads whose maximum reaches theta push composite keys (logit,
//    inverted index) into shared memory.  Once the candidates hold k entries,
//    theta becomes the exact k-th best so far, and later elements must beat
//    it strictly (their indices are higher, so a tie cannot win).
//  * At the segment's end a rank-by-counting pass writes its top-k, ordered by
//    (logit desc, index asc), to the workspace.
// A warp per row then merges the segment lists (a k-round tournament) and
// builds the row's distribution in fp64 from the <= 32 kept values:
// temperature, top-p over the top-k mass, normaliser, the probability of the
// row's token, and the kept list in index order for the resample.  Greedy rows
// are the k = 1 case (argmax, lowest index wins ties).
#include <math.h>

#include "sv_internal.cuh"

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

// ---- shared-memory ring fed by bulk async copies (TMA, cp.async.bulk) ----
constexpr int kStages = 3;                                  // chunks in flight per CTA
constexpr int kChunkBytes = kFastThreads * kFastVecs * 16;  // 32 KB: one chunk of either dtype
constexpr int kSegChunks = 8;                               // chunks per segment (one partial list)
constexpr long long kWaitPolls = 1ll << 20;                 // try_wait polls before a wait gives up
constexpr int kWarpCap = 64;                                // candidate slots per warp
constexpr int kCandCapS = kWarpCap * (kFastThreads / 32);   // candidate buffer of a segment

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0u;
}
// Bounded wait: false when the phase did not complete within kWaitPolls polls.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity)
{
    for (long long i = 0; i < kWaitPolls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// Global -> shared bulk copy of `bytes` (multiple of 16, both ends 16-byte
// aligned) completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, unsigned long long* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(const void* p)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_u32(p)));
    return r;
}

// Element s (0..EPV-1) of a 16-byte vector, as fp32.
template <int DT>
__device__ __forceinline__ float vec_elem(const uint4& v, int s)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (DT == 0) {
        const uint32_t word = w[s >> 1];
        return __uint_as_float((s & 1) ? (word & 0xFFFF0000u) : (word << 16));
    }
    return __uint_as_float(w[s]);
}

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

// Byte offset of a row and the bulk-copied bytes of one chunk of it.
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
    constexpr int CHUNK = kChunkBytes / ESZ;
    const int n_here = min(CHUNK, vocab - c0);
    const char* src = row + (size_t)c0 * ESZ;
    return ((uintptr_t)src & 15u) ? 0u : ((uint32_t)(n_here * ESZ) & ~15u);
}

// k-th largest of one 32-bit key per thread (k <= blockDim) by a byte-wise
// radix select over the top `rounds` bytes.  Lanes of a warp that share a
// digit add their count through one leader (__match_any_sync), so the many
// equal digits of similar keys do not serialise on one shared counter.  Keys
// whose low bytes are not examined are equal below a given top (bf16-derived
// keys: 0x0000 under a positive value, 0xFFFF under a negative one).
__device__ __noinline__ uint32_t block_kth_largest(uint32_t key, int k, int rounds, uint32_t* hist, uint32_t* s_digit,
                                                    int* s_kk)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0u, mask = 0u;
    int kk = k;
    for (int r = 0; r < rounds; ++r) {
        const int shift = 24 - 8 * r;
        for (int b = tid; b < 256; b += blockDim.x) hist[b] = 0u;
        __syncthreads();
        const uint32_t d = ((key & mask) == prefix) ? ((key >> shift) & 255u) : 0x100u;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, d);
        if (d != 0x100u && lane == __ffs(peers) - 1) atomicAdd(&hist[d], (uint32_t)__popc(peers));
        __syncthreads();
        if (warp == 0) {
            uint32_t c[8], sum = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = hist[255 - 8 * lane - i];
                sum += c[i];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            uint32_t excl = incl - sum;
            if (excl < (uint32_t)kk && (uint32_t)kk <= incl) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (excl + c[i] >= (uint32_t)kk) {
                        *s_digit = (uint32_t)(255 - 8 * lane - i);
                        *s_kk = kk - (int)excl;
                        break;
                    }
                    excl += c[i];
                }
            }
        }
        __syncthreads();
        prefix |= (*s_digit) << shift;
        mask |= 0xFFu << shift;
        kk = *s_kk;
    }
    if (rounds == 2) prefix |= (prefix & 0x80000000u) ? 0u : 0xFFFFu;
    return prefix;
}

// Keep the top k of the candidates (rank by counting; composite keys are
// distinct).  The candidates sit in per-warp regions of kWarpCap slots with
// their counts in wcnt[]; they are gathered into `all`, ranked, and the top k
// go back to warp 0's region (the other regions become empty).  Raises theta
// to the k-th best once k candidates exist.
__device__ __noinline__ void compact_candidates(unsigned long long* cand, int* wcnt, unsigned long long* all,
                                                float* s_theta, int* s_strict, int* s_n, int k)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __syncthreads();
    int off = 0, n = 0;
    for (int w = 0; w < kFastThreads / 32; ++w) {
        const int c = min(wcnt[w], kWarpCap);
        if (w < warp) off += c;
        n += c;
    }
    const int mine = min(wcnt[warp], kWarpCap);
    for (int i = lane; i < mine; i += 32) all[off + i] = cand[warp * kWarpCap + i];
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
        const unsigned long long ck = all[i];
        int r8[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // eight independent chains
        int j = 0;
        for (; j + 8 <= n; j += 8) {
#pragma unroll
            for (int q = 0; q < 8; ++q) r8[q] += (all[j + q] > ck) ? 1 : 0;
        }
        for (; j < n; ++j) r8[0] += (all[j] > ck) ? 1 : 0;
        const int rank = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
        if (rank < k) cand[rank] = ck;   // warp 0's region, ordered
    }
    const int m = min(n, k);
    __syncthreads();
    if (tid < kFastThreads / 32) wcnt[tid] = tid == 0 ? m : 0;
    if (tid == 0) {
        *s_n = m;
        if (m == k) {
            *s_theta = ckey_value(cand[k - 1]);
            *s_strict = 1;
        }
    }
    __syncthreads();
}

// Exact top-k of a segment by k rounds of a block max over keys below the last
// (used when too many elements tie at theta).  Out of line: it is cold.
template <int DT>
__device__ __noinline__ int exact_segment_topk(const char* row, int seg0, int seg_end, int k,
                                               unsigned long long* out_keys, unsigned long long* s_red64)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long last = ~0ull;
    int n_out = 0;
    for (int r = 0; r < k; ++r) {
        unsigned long long best = 0ull;
        for (int e = seg0 + tid; e < seg_end; e += kFastThreads) {
            const float val = DT == 0 ? __uint_as_float((uint32_t)((const uint16_t*)row)[e] << 16)
                                      : ((const float*)row)[e];
            const unsigned long long ck = ckey(val, (uint32_t)e);
            if (ck < last && ck > best) best = ck;
        }
        best = warp_max_u64(best);
        if (lane == 0) s_red64[warp] = best;
        __syncthreads();
        best = s_red64[0];
        for (int w = 1; w < kFastThreads / 32; ++w) best = s_red64[w] > best ? s_red64[w] : best;
        __syncthreads();
        if (best == 0ull) break;
        if (tid == 0) out_keys[r] = best;
        last = best;
        ++n_out;
    }
    return n_out;
}

template <int DT>
__global__ void __launch_bounds__(kFastThreads, 2) fast_rows_kernel(RowsArgs a)
{
    constexpr int EPV = DT == 0 ? 8 : 4;
    constexpr int ESZ = DT == 0 ? 2 : 4;
    constexpr int CHUNK = kFastThreads * kFastVecs * EPV;
    static_assert(CHUNK * ESZ == kChunkBytes, "one chunk fills one ring stage");
    extern __shared__ __align__(128) unsigned char ring[];   // kStages x 32 KB
    __shared__ __align__(8) unsigned long long full_bar[kStages];
    __shared__ unsigned long long s_cand[kCandCapS];      // per-warp candidate regions
    __shared__ unsigned long long s_all[kCandCapS];       // gathered candidates (compaction)
    __shared__ int s_wcnt[kFastThreads / 32];
    __shared__ unsigned long long s_red64[kFastThreads / 32];
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_digit;
    __shared__ int s_kk;
    __shared__ float s_theta;
    __shared__ int s_strict, s_n, s_overflow;
    __shared__ int s_compact[2];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_tasks = a.counters->n_fast;
    const int nchunks = (a.vocab + CHUNK - 1) / CHUNK;
    const int nseg = (nchunks + kSegChunks - 1) / kSegChunks;
    const int n_units = n_tasks * nseg;   // the host keeps this below 2^31
    const int G = gridDim.x;
    if ((int)blockIdx.x >= n_units) return;

    // Consumer tasks: the current unit's and the next one's (prefetched).
    int u = blockIdx.x;
    int cur_t = u / nseg;
    RowTask task = a.fast_tasks[cur_t];
    int next_t = (u + G < n_units) ? (u + G) / nseg : -1;
    RowTask next_task = next_t >= 0 ? a.fast_tasks[next_t] : task;

    // Producer state (thread 0): the next (unit, chunk) to copy, where it goes
    // in the ring, and the row it reads.  It runs up to kStages chunks ahead,
    // which can be more than one unit when segments are short; it reuses the
    // consumer's tasks when it can and reads the task list otherwise.
    int p_u = u, p_t = cur_t, p_chunk = (u - cur_t * nseg) * kSegChunks;
    int p_end = min(nchunks, p_chunk + kSegChunks);
    int p_slot = 0;
    const char* p_row = task_row<DT>(a, task);
    auto produce = [&]() {
        if (p_u >= n_units) return;
        const int c0 = p_chunk * CHUNK;
        const uint32_t bytes = chunk_bytes<DT>(p_row, c0, a.vocab);
        unsigned long long* bar = &full_bar[p_slot];
        if (bytes) {
            mbar_expect_tx(bar, bytes);
            bulk_g2s(ring + p_slot * kChunkBytes, p_row + (size_t)c0 * ESZ, bytes, bar);
        } else {
            mbar_arrive(bar);
        }
        if (++p_slot == kStages) p_slot = 0;
        if (++p_chunk == p_end) {
            p_u += G;
            if (p_u < n_units) {
                const int t = p_u / nseg;
                if (t != p_t) {
                    p_row = (t == cur_t) ? task_row<DT>(a, task)
                                         : (t == next_t ? task_row<DT>(a, next_task) : task_row<DT>(a, a.fast_tasks[t]));
                    p_t = t;
                }
                p_chunk = (p_u - t * nseg) * kSegChunks;
                p_end = min(nchunks, p_chunk + kSegChunks);
            }
        }
    };
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full_bar[s], 1u);
        mbar_fence_init();
        s_compact[0] = s_compact[1] = 0;
    }
    __syncthreads();
    if (tid == 0)
        for (int i = 0; i < kStages; ++i) produce();

    int c_slot = 0;
    uint32_t c_phase = 0u;
    for (; u < n_units; u += G) {
        if (u != (int)blockIdx.x) {
            cur_t = next_t;
            task = next_task;
            next_t = (u + G < n_units) ? (u + G) / nseg : -1;
            if (next_t >= 0) next_task = (next_t == cur_t) ? task : a.fast_tasks[next_t];
        }
        const char* row = task_row<DT>(a, task);
        const int k = task.k_eff < kFastK ? task.k_eff : kFastK;
        const int compact_at = max(2 * k, 40);
        const int chunk0 = (u - cur_t * nseg) * kSegChunks;
        const int ns = min(kSegChunks, nchunks - chunk0);
        __syncthreads();   // the previous segment's buffers are free
        if (tid == 0) {
            s_overflow = 0;
            s_strict = 0;
        }
        int wcnt = 0;   // this warp's candidates (same value in every lane)
        int bad = 0;
        for (int j = 0; j < ns; ++j) {
            const int c0 = (chunk0 + j) * CHUNK;
            const uint32_t bytes = chunk_bytes<DT>(row, c0, a.vocab);
            const bool arrived = mbar_wait(&full_bar[c_slot], c_phase);
            const unsigned char* st = ring + c_slot * kChunkBytes;
            uint4 v[kFastVecs];
#pragma unroll
            for (int i = 0; i < kFastVecs; ++i) {
                const int off = (i * kFastThreads + tid) * 16;
                if ((uint32_t)(off + 16) <= bytes)
                    v[i] = ld_shared_v4(st + off);
                else
                    v[i] = load_edge<DT>(row, c0 + (i * kFastThreads + tid) * EPV, a.vocab);
            }
            if (++c_slot == kStages) {
                c_slot = 0;
                c_phase ^= 1u;
            }
            // Per-vector NaN-propagating maxima, then their tree max: the same
            // operation count as one running max, with independent chains.
            float vmax[kFastVecs];
            if (DT == 0) {
                uint32_t m2[kFastVecs];
#pragma unroll
                for (int i = 0; i < kFastVecs; ++i) {
                    m2[i] = bmax2_nan(bmax2_nan(v[i].x, v[i].y), bmax2_nan(v[i].z, v[i].w));
                    vmax[i] = fmax_nan(__uint_as_float(m2[i] << 16), __uint_as_float(m2[i] & 0xFFFF0000u));
                }
            } else {
#pragma unroll
                for (int i = 0; i < kFastVecs; ++i)
                    vmax[i] = fmax_nan(fmax_nan(__uint_as_float(v[i].x), __uint_as_float(v[i].y)),
                                       fmax_nan(__uint_as_float(v[i].z), __uint_as_float(v[i].w)));
            }
            const float tmax = fmax_nan(fmax_nan(fmax_nan(vmax[0], vmax[1]), fmax_nan(vmax[2], vmax[3])),
                                        fmax_nan(fmax_nan(vmax[4], vmax[5]), fmax_nan(vmax[6], vmax[7])));
            bad |= (isnan(tmax) || tmax == INFINITY) ? 1 : 0;
            // Thread 0 decides whether to compact before this chunk's pushes (a
            // slightly stale count is fine; the flag is double-buffered so the
            // previous chunk's readers are not overtaken).
            if (lane == 0) s_wcnt[warp] = wcnt;
            if (tid == 0) {
                int tot = 0;   // possibly a little stale: the decision only needs to be shared
                for (int w = 0; w < kFastThreads / 32; ++w) tot += s_wcnt[w];
                s_compact[j & 1] = (j > 0 && s_strict == 0 && tot > compact_at) ? 1 : 0;
            }
            // One barrier per chunk: every thread holds its data (the stage can
            // be refilled), the compaction decision is published, and a bulk
            // copy that never arrived stops the whole CTA.
            if (__syncthreads_or(!arrived)) {
                if (tid == 0) {
                    atomicOr(&a.counters->timeout, 1);
                    // let the copies already issued land (bounded), then leave
                    for (int q = 0; q < kStages; ++q) mbar_wait(&full_bar[q], c_phase ^ (q < c_slot ? 1u : 0u));
                }
                __syncthreads();
                return;
            }
            if (tid == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                produce();
            }
            float theta;
            int strict;
            if (j == 0) {   // exact k-th largest of the 256 thread maxima
                const uint32_t key = key_of_f32_bits(__float_as_uint(tmax));
                theta = f32_of_key(block_kth_largest(key, k, DT == 0 ? 2 : 4, s_hist, &s_digit, &s_kk));
                strict = 0;
                if (tid == 0) s_theta = theta;
            } else {
                if (s_compact[j & 1]) {
                    compact_candidates(s_cand, s_wcnt, s_all, &s_theta, &s_strict, &s_n, k);
                    wcnt = s_wcnt[warp];
                }
                theta = s_theta;
                strict = s_strict;
            }
            // Warp-cooperative push: one ballot per vector slot; for each lane
            // whose vector maximum reaches theta, the warp takes that vector
            // (broadcast), EPV lanes test one element each, and one atomic
            // reserves the slots.  Uniform control flow, no calls.
#pragma unroll
            for (int i = 0; i < kFastVecs; ++i) {
                unsigned bal = __ballot_sync(0xFFFFFFFFu, strict ? (vmax[i] > theta) : (vmax[i] >= theta));
                while (bal) {
                    const int src = __ffs(bal) - 1;
                    bal &= bal - 1u;
                    const uint32_t w0 = __shfl_sync(0xFFFFFFFFu, v[i].x, src);
                    const uint32_t w1 = __shfl_sync(0xFFFFFFFFu, v[i].y, src);
                    const uint32_t w2 = __shfl_sync(0xFFFFFFFFu, v[i].z, src);
                    const uint32_t w3 = __shfl_sync(0xFFFFFFFFu, v[i].w, src);
                    const int q = DT == 0 ? (lane >> 1) : lane;
                    const uint32_t word = q == 0 ? w0 : (q == 1 ? w1 : (q == 2 ? w2 : w3));
                    const float val = DT == 0 ? __uint_as_float((lane & 1) ? (word & 0xFFFF0000u) : (word << 16))
                                              : __uint_as_float(word);
                    const int e = c0 + (i * kFastThreads + warp * 32 + src) * EPV + lane;
                    const bool take = lane < EPV && e < a.vocab && (strict ? val > theta : val >= theta);
                    const unsigned tb = __ballot_sync(0xFFFFFFFFu, take);
                    if (take) {
                        const int pos = wcnt + __popc(tb & ((1u << lane) - 1u));
                        if (pos < kWarpCap)
                            s_cand[warp * kWarpCap + pos] = ckey(val, (uint32_t)e);
                        else
                            s_overflow = 1;
                    }
                    wcnt += __popc(tb);
                }
            }
        }
        Partial* out = a.partials + u;
        const int any_bad = __syncthreads_or(bad);
        if (any_bad) {
            if (tid == 0) {
                out->status = kNonfinite;
                out->count = 0u;
            }
            continue;
        }
        if (lane == 0) s_wcnt[warp] = wcnt;
        if (!s_overflow) {
            compact_candidates(s_cand, s_wcnt, s_all, &s_theta, &s_strict, &s_n, k);
            const int m = s_n;
            if (tid < m) out->keys[tid] = s_cand[tid];
            if (tid == 0) {
                out->status = 0u;
                out->count = (uint32_t)m;
            }
            continue;
        }
        // Too many elements reached theta (heavy ties): exact k rounds of a
        // block max over the segment, re-read from the row.
        const int seg0 = chunk0 * CHUNK;
        const int n_out = exact_segment_topk<DT>(row, seg0, min(a.vocab, seg0 + ns * CHUNK), k, out->keys, s_red64);
        if (tid == 0) {
            out->status = 0u;
            out->count = (uint32_t)n_out;
        }
    }
}

constexpr int kFinalizeWarps = 8;
constexpr int kMaxChunkSlots = 4;   // segment lists per lane in the merge: up to 128 per row
constexpr int kStagedLists = 8;     // rows with at most this many lists merge in shared memory

template <int DT>
__global__ void __launch_bounds__(kFinalizeWarps * 32) fast_finalize_kernel(RowsArgs a)
{
    constexpr int EPV = DT == 0 ? 8 : 4;
    constexpr int CHUNK = kFastThreads * kFastVecs * EPV;
    __shared__ unsigned long long s_top[kFinalizeWarps][kFastK];
    __shared__ unsigned long long s_lists[kFinalizeWarps][kStagedLists][kFastK];
    __shared__ double s_e[kFinalizeWarps][kFastK];
    __shared__ int s_kept[kFinalizeWarps];
    __shared__ double s_z[kFinalizeWarps];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_tasks = a.counters->n_fast;
    const int nchunks = ((a.vocab + CHUNK - 1) / CHUNK + kSegChunks - 1) / kSegChunks;   // segment lists per row
    for (int t = blockIdx.x * kFinalizeWarps + warp; t < n_tasks; t += gridDim.x * kFinalizeWarps) {
        const RowTask task = a.fast_tasks[t];
        const Partial* P = a.partials + (size_t)t * nchunks;
        RowInfo* info = a.info + task.slot;
        uint32_t st = 0u;
        for (int c = lane; c < nchunks; c += 32) st |= P[c].status;
        st = __reduce_or_sync(0xFFFFFFFFu, st);

        const int k = task.k_eff < kFastK ? task.k_eff : kFastK;
        int n_top = 0;
        if (!(st & kNonfinite)) {
            if (nchunks <= kStagedLists) {
                // Stage the lists in shared memory with independent loads, then
                // merge: lane c holds the head of list c.
                for (int c = 0; c < nchunks; ++c) s_lists[warp][c][lane] = P[c].keys[lane];
                const int cnt = lane < nchunks ? (int)P[lane].count : 0;
                __syncwarp();
                int head = 0;
                for (int r = 0; r < k; ++r) {
                    const unsigned long long key = head < cnt ? s_lists[warp][lane][head] : 0ull;
                    const unsigned long long wbest = warp_max_u64(key);
                    if (wbest == 0ull) break;
                    if (key == wbest) ++head;
                    if (lane == 0) s_top[warp][r] = wbest;
                    n_top = r + 1;
                }
            } else {
                int head[kMaxChunkSlots];
#pragma unroll
                for (int j = 0; j < kMaxChunkSlots; ++j) head[j] = 0;
                for (int r = 0; r < k; ++r) {
                    unsigned long long best = 0ull;
                    int bj = -1;
#pragma unroll
                    for (int j = 0; j < kMaxChunkSlots; ++j) {
                        const int c = lane + 32 * j;
                        if (c < nchunks && head[j] < (int)P[c].count) {
                            const unsigned long long key = P[c].keys[head[j]];
                            if (key > best) {
                                best = key;
                                bj = j;
                            }
                        }
                    }
                    const unsigned long long wbest = warp_max_u64(best);
                    if (wbest == 0ull) break;
#pragma unroll
                    for (int j = 0; j < kMaxChunkSlots; ++j)
                        if (best == wbest && bj == j) head[j] += 1;
                    if (lane == 0) s_top[warp][r] = wbest;
                    n_top = r + 1;
                }
            }
        }
        __syncwarp();

        const unsigned long long ck = lane < n_top ? s_top[warp][lane] : 0ull;
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
            continue;
        }
        if (T == 0.0f) {
            if (lane == 0) {
                info->desc.log_norm = 0.0f;
                info->desc.cutoff_logit = m;
                info->desc.cutoff_ties = 1;
                info->desc.kept = 1;
                info->p_token = task.token >= 0 ? (task.token == amax ? 1.0 : 0.0) : nan("");
                info->z = 1.0;
                info->n_list = 1;
                info->list_idx[0] = amax;
                info->list_p[0] = 1.0;
            }
            continue;
        }
        // Sampling row: masses of the kept values in fp64, in sorted order.
        const double e = lane < n_top ? exp(((double)lv - (double)m) / (double)T) : 0.0;
        s_e[warp][lane] = e;
        __syncwarp();
        if (lane == 0) {
            double z1 = 0.0;
            for (int i = 0; i < n_top; ++i) z1 += s_e[warp][i];
            int kept = n_top;
            if (task.top_p < 1.0f) {
                const double target = (double)task.top_p * z1;
                double cum = 0.0;
                for (int i = 0; i < n_top; ++i) {
                    cum += s_e[warp][i];
                    if (cum >= target) {
                        kept = i + 1;
                        break;
                    }
                }
            }
            double z = 0.0;
            for (int i = 0; i < kept; ++i) z += s_e[warp][i];
            s_kept[warp] = kept;
            s_z[warp] = z;
        }
        __syncwarp();
        const int kept = s_kept[warp];
        const double z = s_z[warp];
        const bool in = lane < kept;
        const double p = in ? e / z : 0.0;
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
            info->desc.log_norm = (float)log(z);
            info->desc.cutoff_logit = cut;
            info->desc.cutoff_ties = ties;
            info->desc.kept = kept;
            info->p_token = task.token >= 0 ? ptok : nan("");
            info->z = z;
            info->n_list = kept;
        }
    }
}

}  // namespace

template <int DT>
cudaError_t launch_fast_rows_t(const RowsArgs& a, cudaStream_t s)
{
    // Persistent grid: exactly the CTAs that fit at once, each with its ring.
    const size_t smem = (size_t)kStages * kChunkBytes;
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
    fast_rows_kernel<DT><<<a.num_sms * nb, kFastThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fast_rows(const RowsArgs& a, cudaStream_t s)
{
    return a.dtype == 0 ? launch_fast_rows_t<0>(a, s) : launch_fast_rows_t<1>(a, s);
}

cudaError_t launch_fast_finalize(const RowsArgs& a, cudaStream_t s)
{
    int grid = (a.max_tasks + kFinalizeWarps - 1) / kFinalizeWarps;
    if (grid > a.num_sms * 8) grid = a.num_sms * 8;
    if (grid < 1) grid = 1;
    if (a.dtype == 0)
        fast_finalize_kernel<0><<<grid, kFinalizeWarps * 32, 0, s>>>(a);
    else
        fast_finalize_kernel<1><<<grid, kFinalizeWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace sv
