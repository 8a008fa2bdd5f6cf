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

template <int DT>
__global__ void __launch_bounds__(kFastThreads) fast_rows_kernel(RowsArgs a)
{
    constexpr int EPV = DT == 0 ? 8 : 4;
    constexpr int ESZ = DT == 0 ? 2 : 4;
    constexpr int CHUNK = kFastThreads * kFastVecs * EPV;
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
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
        __syncthreads();   // shared memory of the previous unit is free
        const int t = (int)(u / nchunks);
        const int c = (int)(u - (long long)t * nchunks);
        const RowTask task = a.fast_tasks[t];
        const int64_t stride = task.is_draft ? a.stride_d : a.stride_t;
        const char* row = (const char*)(task.is_draft ? a.drf : a.tgt) + (size_t)task.row * (size_t)stride * ESZ;
        const int c0 = c * CHUNK;
        const bool aligned = (((uintptr_t)row + (size_t)c0 * ESZ) & 15u) == 0u;

        uint4 v[kFastVecs];
#pragma unroll
        for (int i = 0; i < kFastVecs; ++i) {
            const int e0 = c0 + (i * kFastThreads + tid) * EPV;
            if (aligned && e0 + EPV <= a.vocab)
                v[i] = ld_stream(row + (size_t)e0 * ESZ);
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
        if (__syncthreads_or(isnan(tmax) || tmax == INFINITY)) {
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
            unsigned long long last = ~0ull;
            int n_out = 0;
            for (int r = 0; r < k; ++r) {
                unsigned long long best = 0ull;
#pragma unroll
                for (int i = 0; i < kFastVecs; ++i) {
                    const int e0 = c0 + (i * kFastThreads + tid) * EPV;
#pragma unroll
                    for (int s = 0; s < EPV; ++s) {
                        if (e0 + s < a.vocab) {
                            const unsigned long long ck = ckey(vec_elem<DT>(v[i], s), (uint32_t)(e0 + s));
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

cudaError_t launch_fast_rows(const RowsArgs& a, cudaStream_t s)
{
    // Persistent grid: a few resident CTAs per SM walk the (row, chunk) units.
    const int grid = a.num_sms * 6;
    if (a.dtype == 0)
        fast_rows_kernel<0><<<grid, kFastThreads, 0, s>>>(a);
    else
        fast_rows_kernel<1><<<grid, kFastThreads, 0, s>>>(a);
    return cudaGetLastError();
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
