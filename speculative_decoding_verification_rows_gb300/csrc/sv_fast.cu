// sv_fast.cu -- one-pass row kernel for greedy rows and rows with top-k <= 32.
//
// Target-distribution build of jianc99/sglang PR #8 ("build_speculative_verify_
// target_probs"): the top-k is selected on the raw logits (a positive
// temperature keeps their order) and only the k kept values are divided by the
// temperature.  Here the selection streams each [rows, vocab] row from HBM
// exactly once, in chunks of 16 K bf16 (8 K fp32) elements:
//
//   1. each thread loads 8 x 16 B with streaming (L1 no-allocate) loads and
//      takes a NaN-propagating packed max (max.NaN.bf16x2);
//   2. the CTA finds theta = the k-th largest of its 256 thread maxima by a
//      byte-wise radix select -- at least k elements are >= theta;
//   3. only threads whose maximum reaches theta rescan their registers and
//      push (logit, index) composite keys >= theta into shared memory;
//   4. a rank-by-counting pass writes the chunk's top-k, ordered by (logit
//      desc, index asc), to the workspace.
// A warp per row then merges the chunk lists (a k-round tournament) and builds
// the row's distribution in fp64 from the <= 32 kept values: temperature,
// top-p over the top-k mass, normaliser, the probability of the row's token,
// and the kept list in index order for the resample.  Greedy rows are the
// k = 1 case (argmax, lowest index wins ties).
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
__device__ __forceinline__ uint4 ld_stream(const void* p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// ---- shared-memory ring fed by bulk async copies (TMA, cp.async.bulk) ----
constexpr int kStages = 3;                                  // chunks in flight per CTA
constexpr int kChunkBytes = kFastThreads * kFastVecs * 16;  // 32 KB: one chunk of either dtype
constexpr long long kWaitPolls = 1ll << 26;                 // try_wait polls before a wait gives up

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
// Global -> shared bulk copy of `bytes` (multiple of 16, both ends 16-byte aligned)
// completing on `bar`.
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

__device__ __forceinline__ float warp_max_f(float x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
}

// k-th largest of one 32-bit key per thread (k <= blockDim), by a radix select
// over the top `rounds` bytes.  Keys whose low bytes are not examined are
// assumed equal (bf16-derived keys: 0x0000 below a positive value, 0xFFFF
// below a negative one).
__device__ uint32_t block_kth_largest(uint32_t key, int k, int rounds, uint32_t* hist, uint32_t* s_digit, int* s_kk)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0u, mask = 0u;
    int kk = k;
    for (int r = 0; r < rounds; ++r) {
        const int shift = 24 - 8 * r;
        for (int b = tid; b < 256; b += blockDim.x) hist[b] = 0u;
        __syncthreads();
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        __syncthreads();
        if (warp == 0) {
            uint32_t c[8], s = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = hist[255 - 8 * lane - i];
                s += c[i];
            }
            uint32_t incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            uint32_t excl = incl - s;
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
        __syncthreads();
    }
    if (rounds == 2) prefix |= (prefix & 0x80000000u) ? 0u : 0xFFFFu;
    return prefix;
}

// Where unit u (row task t, chunk c) starts, and how many bytes of it the bulk
// copy moves (a 16-byte-aligned multiple of 16; the rest, if any, is loaded
// element by element).
template <int DT>
__device__ __forceinline__ const char* unit_source(const RowsArgs& a, long long u, int nchunks, int& c0,
                                                   uint32_t& bytes, RowTask& task)
{
    constexpr int ESZ = DT == 0 ? 2 : 4;
    constexpr int CHUNK = kChunkBytes / ESZ;
    const int t = (int)(u / nchunks);
    const int c = (int)(u - (long long)t * nchunks);
    task = a.fast_tasks[t];
    const int64_t stride = task.is_draft ? a.stride_d : a.stride_t;
    const char* row = (const char*)(task.is_draft ? a.drf : a.tgt) + (size_t)task.row * (size_t)stride * ESZ;
    c0 = c * CHUNK;
    const int n_here = min(CHUNK, a.vocab - c0);
    const char* src = row + (size_t)c0 * ESZ;
    bytes = ((uintptr_t)src & 15u) ? 0u : (uint32_t)(n_here * ESZ) & ~15u;
    return row;
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
    __shared__ unsigned long long s_cand[kCandCap];
    __shared__ uint32_t s_hist[256];
    __shared__ float s_redf[kFastThreads / 32];
    __shared__ unsigned long long s_red64[kFastThreads / 32];
    __shared__ uint32_t s_digit;
    __shared__ int s_kk;
    __shared__ int s_cnt;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_tasks = a.counters->n_fast;
    const int nchunks = (a.vocab + CHUNK - 1) / CHUNK;
    const long long n_units = (long long)n_tasks * nchunks;
    if ((long long)blockIdx.x >= n_units) return;

    // Thread 0 feeds the ring: unit i of this CTA goes to stage i % kStages.
    auto issue = [&](long long i) {
        const long long uu = (long long)blockIdx.x + i * gridDim.x;
        if (uu >= n_units) return;
        int cc0;
        uint32_t bytes;
        RowTask tk;
        const char* row = unit_source<DT>(a, uu, nchunks, cc0, bytes, tk);
        unsigned long long* bar = &full_bar[i % kStages];
        if (bytes) {
            mbar_expect_tx(bar, bytes);
            bulk_g2s(ring + (i % kStages) * kChunkBytes, row + (size_t)cc0 * ESZ, bytes, bar);
        } else {
            mbar_arrive(bar);
        }
    };
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full_bar[s], 1u);
        mbar_fence_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int i = 0; i < kStages; ++i) issue(i);

    long long it = 0;
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
        __syncthreads();   // shared memory of the previous unit is free
        int c0;
        uint32_t bytes;
        RowTask task;
        const char* row = unit_source<DT>(a, u, nchunks, c0, bytes, task);
        const int stage = (int)(it % kStages);
        const bool arrived = mbar_wait(&full_bar[stage], (uint32_t)((it / kStages) & 1));
        if (!__syncthreads_and(arrived)) {
            // A bulk copy never completed: report it, let the copies already
            // issued land (bounded), and leave the remaining rows unprocessed.
            if (tid == 0) {
                atomicOr(&a.counters->timeout, 1);
                for (long long j = it; j < it + kStages; ++j) {
                    if ((long long)blockIdx.x + j * gridDim.x >= n_units) break;
                    mbar_wait(&full_bar[j % kStages], (uint32_t)((j / kStages) & 1));
                }
            }
            __syncthreads();
            return;
        }
        const unsigned char* st = ring + stage * kChunkBytes;

        uint4 v[kFastVecs];
#pragma unroll
        for (int i = 0; i < kFastVecs; ++i) {
            const int off = (i * kFastThreads + tid) * 16;
            const int e0 = c0 + (i * kFastThreads + tid) * EPV;
            if ((uint32_t)(off + 16) <= bytes)
                v[i] = ld_shared_v4(st + off);
            else
                v[i] = load_edge<DT>(row, e0, a.vocab);
        }

        float tmax;
        if (DT == 0) {
            uint32_t m2 = 0xFF80FF80u;
#pragma unroll
            for (int i = 0; i < kFastVecs; ++i) {
                m2 = bmax2_nan(m2, v[i].x);
                m2 = bmax2_nan(m2, v[i].y);
                m2 = bmax2_nan(m2, v[i].z);
                m2 = bmax2_nan(m2, v[i].w);
            }
            tmax = fmax_nan(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
        } else {
            tmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < kFastVecs; ++i) {
                tmax = fmax_nan(tmax, __uint_as_float(v[i].x));
                tmax = fmax_nan(tmax, __uint_as_float(v[i].y));
                tmax = fmax_nan(tmax, __uint_as_float(v[i].z));
                tmax = fmax_nan(tmax, __uint_as_float(v[i].w));
            }
        }
        Partial* out = a.partials + u;
        const int any_bad = __syncthreads_or(isnan(tmax) || tmax == INFINITY);
        // every thread holds its data in registers: refill this stage
        if (tid == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(it + kStages);
        }
        if (any_bad) {
            if (tid == 0) {
                out->status = kNonfinite;
                out->count = 0u;
            }
            continue;
        }

        const int k = task.k_eff < kFastK ? task.k_eff : kFastK;
        float theta;
        if (k == 1) {
            const float wm = warp_max_f(tmax);
            if (lane == 0) s_redf[warp] = wm;
            __syncthreads();
            theta = s_redf[0];
#pragma unroll
            for (int w = 1; w < kFastThreads / 32; ++w) theta = fmaxf(theta, s_redf[w]);
        } else {
            const uint32_t key = key_of_f32_bits(__float_as_uint(tmax));
            theta = f32_of_key(block_kth_largest(key, k, DT == 0 ? 2 : 4, s_hist, &s_digit, &s_kk));
        }

        if (tid == 0) s_cnt = 0;
        __syncthreads();
        if (tmax >= theta) {
#pragma unroll
            for (int i = 0; i < kFastVecs; ++i) {
                const int e0 = c0 + (i * kFastThreads + tid) * EPV;
#pragma unroll
                for (int s = 0; s < EPV; ++s) {
                    const float val = vec_elem<DT>(v[i], s);
                    if (e0 + s < a.vocab && val >= theta) {
                        const int pos = atomicAdd(&s_cnt, 1);
                        if (pos < kCandCap) s_cand[pos] = ckey(val, (uint32_t)(e0 + s));
                    }
                }
            }
        }
        __syncthreads();
        const int cnt = s_cnt;
        if (cnt <= kCandCap) {
            if (tid < cnt) {
                const unsigned long long ck = s_cand[tid];
                int rank = 0;
                for (int j = 0; j < cnt; ++j) rank += (s_cand[j] > ck) ? 1 : 0;
                if (rank < k) out->keys[rank] = ck;
            }
            if (tid == 0) {
                out->status = 0u;
                out->count = (uint32_t)(cnt < k ? cnt : k);
            }
        } else {
            // Many elements tie at theta (or one thread holds most of the
            // top): exact k rounds of a block max over keys below the last.
            // The values are re-read from the row (L2) so that the registers
            // of the common path stay free.
            unsigned long long last = ~0ull;
            int n_out = 0;
            for (int r = 0; r < k; ++r) {
                unsigned long long best = 0ull;
                for (int i = 0; i < kFastVecs; ++i) {
                    const int e0 = c0 + (i * kFastThreads + tid) * EPV;
                    const uint4 w = load_edge<DT>(row, e0, a.vocab);
#pragma unroll
                    for (int s = 0; s < EPV; ++s) {
                        if (e0 + s < a.vocab) {
                            const unsigned long long ck = ckey(vec_elem<DT>(w, s), (uint32_t)(e0 + s));
                            if (ck < last && ck > best) best = ck;
                        }
                    }
                }
                best = warp_max_u64(best);
                if (lane == 0) s_red64[warp] = best;
                __syncthreads();
                best = s_red64[0];
#pragma unroll
                for (int w = 1; w < kFastThreads / 32; ++w) best = s_red64[w] > best ? s_red64[w] : best;
                __syncthreads();
                if (best == 0ull) break;
                if (tid == 0) out->keys[r] = best;
                last = best;
                ++n_out;
            }
            if (tid == 0) {
                out->status = 0u;
                out->count = (uint32_t)n_out;
            }
        }
    }
}

constexpr int kFinalizeWarps = 8;
constexpr int kMaxChunkSlots = 4;   // chunks per lane in the merge: up to 128 chunks per row

template <int DT>
__global__ void __launch_bounds__(kFinalizeWarps * 32) fast_finalize_kernel(RowsArgs a)
{
    constexpr int EPV = DT == 0 ? 8 : 4;
    constexpr int CHUNK = kFastThreads * kFastVecs * EPV;
    __shared__ unsigned long long s_top[kFinalizeWarps][kFastK];
    __shared__ double s_e[kFinalizeWarps][kFastK];
    __shared__ int s_kept[kFinalizeWarps];
    __shared__ double s_z[kFinalizeWarps];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_tasks = a.counters->n_fast;
    const int nchunks = (a.vocab + CHUNK - 1) / CHUNK;
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
