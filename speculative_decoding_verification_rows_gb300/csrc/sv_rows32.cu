// sv_rows32.cu -- fp32 rows whose kept set is too large to list (top-k above
// 32 or off, with or without top-p over the vocabulary), and the full-row
// resample of their requests.
//
// The row transform follows jianc99/sglang PR #8, "build_speculative_verify_
// target_probs" (temperature, top-k, top-p over the [rows, vocab] logits):
// tokens in the order (logit descending, index ascending); top-k keeps the
// first k, top-p the shortest prefix of those whose mass exp((l - m) / T)
// reaches top_p of theirs.  fp32 rows hold too many distinct values for the
// per-value counts of the bf16 path, so each row is resolved by a radix
// descent on its 32-bit order keys: per bin of 11 (then 11, then 10) key bits,
// the count and the exact mass of its elements (each element's mass in
// double-float arithmetic, rounded once to 58-bit fixed point, summed in 128
// bits), the bin where the top-k count or the top-p mass is crossed, and the
// next level inside it, down to one value; the number of its ties that stay
// kept follows from the exact sums.
//
// The resample follows local-inference-lab/rtx6kpro dspark-upstream-
// consolidation.md, "Identical rejection scheme": at the first rejection the
// token is drawn from the residual max(0, p - q), after full acceptance from
// p, by inverse CDF in index order over 62-bit fixed-point weights (the same
// weights and draw as the bf16 full-row resample); one CTA per job, tiles of
// consecutive elements in index order for the tie ranks at the cutoffs.
#include "sv_internal.cuh"

namespace sv {
namespace {

typedef unsigned __int128 u128;

constexpr int kR32Threads = 512;
constexpr int kR32Warps = kR32Threads / 32;
constexpr int kR32Bins = 2048;                      // bins of a level (11 key bits; the last level has 10)
constexpr int kR32Copies = 4;                       // copies of each bin's counters (lane & 3): fewer lanes per address
// An element's mass is summed in 2^-58 units (fix_split(e, 29)); the
// resample's weights are 2^-62 units (fix_split(p, 31)), as in the bf16 one.

// Canonical order key of an fp32 pattern (-0 as +0): larger value, larger key.
__device__ __forceinline__ uint32_t key32(uint32_t u)
{
    if ((u & 0x7FFFFFFFu) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float value32(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
constexpr uint32_t kKeyNegInf = 0x007FFFFFu;   // key of -inf

// floor(e 2^(2 hb)) for 0 <= e <= 1 held as a double-float, hb <= 31, with
// 32-bit conversions only: e 2^hb = a + f (a its integer part), then
// floor((f + lo 2^hb) 2^hb); about 2^-24 of a unit of 2^hb is lost in f's
// rounding, far below the margins the sums serve.
__device__ __forceinline__ unsigned long long fix_split(dfloat e, int hb)
{
    const float s = __int_as_float((127 + hb) << 23);   // 2^hb
    const float h = e.hi * s;
    const float a = truncf(h);
    const int b = __float2int_rd(((h - a) + e.lo * s) * s);   // may be slightly negative
    const long long v = ((long long)(unsigned)a << hb) + b;
    return v > 0 ? (unsigned long long)v : 0ull;
}

__device__ __forceinline__ double u128_to_double(u128 x)
{
    return (double)(unsigned long long)(x >> 64) * 18446744073709551616.0 + (double)(unsigned long long)x;
}

// ----------------------------------------------------------------------------
// The row kernel
// ----------------------------------------------------------------------------
struct R32Smem {
    dfloat tab[64];
    uint32_t cnt[kR32Copies][kR32Bins];
    unsigned long long mlo[kR32Copies][kR32Bins];   // mass per bin in 2^-58 units: low word
    uint32_t mhi[kR32Copies][kR32Bins];             // and the carries out of it
    unsigned long long red64[kR32Warps];
    uint32_t redu[kR32Warps];
    int redi[kR32Warps];
    // a level's crossing (warp 0 writes, everyone reads)
    int bin;
    uint32_t above_cnt;
    u128 above_mass;
};

__device__ __forceinline__ u128 bin_mass(const R32Smem& sm, int b)
{
    u128 t = 0;
#pragma unroll
    for (int c = 0; c < kR32Copies; ++c) t += ((u128)sm.mhi[c][b] << 64) | (u128)sm.mlo[c][b];
    return t;
}
__device__ __forceinline__ uint32_t bin_count(const R32Smem& sm, int b)
{
    uint32_t t = 0u;
#pragma unroll
    for (int c = 0; c < kR32Copies; ++c) t += sm.cnt[c][b];
    return t;
}

// f(value, index) over a row, every element once: 16-byte loads, four of
// them in flight per thread (the elements before the first 16-byte boundary
// and after the last whole vector one by one).
template <typename F>
__device__ __forceinline__ void stream_row(const float* row, int V, F f)
{
    const int tid = threadIdx.x;
    const int head = min(V, (int)(((16u - ((uint32_t)(uintptr_t)row & 15u)) & 15u) >> 2));
    if (tid < head) f(__ldg(row + tid), tid);
    const int nvec = (V - head) >> 2;
    const float4* vp = reinterpret_cast<const float4*>(row + head);
    for (int v0 = tid; v0 < nvec; v0 += kR32Threads * 4) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int vi = v0 + u * kR32Threads;
            x[u] = vi < nvec ? __ldg(vp + vi) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int vi = v0 + u * kR32Threads;
            if (vi < nvec) {
                const int i = head + 4 * vi;
                f(x[u].x, i);
                f(x[u].y, i + 1);
                f(x[u].z, i + 2);
                f(x[u].w, i + 3);
            }
        }
    }
    const int tail0 = head + 4 * nvec;
    if (tail0 + tid < V) f(__ldg(row + tail0 + tid), tail0 + tid);
}

// Histogram of one level: the elements whose key matches `pre` under
// `pre_mask` and is at least `min_key`, binned by the `nbins` key bits above
// `shift`: counts and masses.  Every thread calls it.
__device__ void level_pass(R32Smem& sm, const float* row, int V, float m, float T, uint32_t pre_mask,
                           uint32_t pre, uint32_t min_key, int shift, int nbins)
{
    for (int b = threadIdx.x; b < nbins * kR32Copies; b += kR32Threads) {
        sm.cnt[b / nbins][b % nbins] = 0u;
        sm.mlo[b / nbins][b % nbins] = 0ull;
        sm.mhi[b / nbins][b % nbins] = 0u;
    }
    __syncthreads();
    const int cp = threadIdx.x & (kR32Copies - 1);
    const float inv_t = 1.0f / T;
    stream_row(row, V, [&](float x, int) {
        const uint32_t k = key32(__float_as_uint(x));
        if ((k & pre_mask) != pre || k < min_key) return;
        const int b = (int)((k >> shift) & (uint32_t)(nbins - 1));
        const dfloat sl = scaled_logit(x, m, T, inv_t);
        // below -41 the mass is under 2^-59: it floors to 0 in 2^-58 units
        const unsigned long long v = sl.hi < -41.0f ? 0ull : fix_split(exp_df(sl, sm.tab), 29);
        atomicAdd(&sm.cnt[cp][b], 1u);
        if (v) {
            const unsigned long long old = atomicAdd(&sm.mlo[cp][b], v);
            if (old + v < old) atomicAdd(&sm.mhi[cp][b], 1u);
        }
    });
    __syncthreads();
}

// The bin of the current histogram where, going down from the top bin, the
// running count reaches `tc` (by_mass = false) or the running mass reaches
// `tm` (by_mass = true); also the count and mass of the bins above it.
// Warp 0 scans (each lane a run of nbins / 32 bins, lane 0 the top run);
// every thread calls it and reads the result from sm.
__device__ void find_crossing(R32Smem& sm, int nbins, bool by_mass, uint32_t tc, u128 tm)
{
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x, w = nbins / 32;
        const int top = nbins - 1 - lane * w;   // this lane's bins: top, top - 1, ..., top - w + 1
        uint32_t c = 0u;
        u128 ms = 0;
        for (int b = top; b > top - w; --b) {
            c += bin_count(sm, b);
            ms += bin_mass(sm, b);
        }
        // exclusive prefix over the lanes above
        uint32_t pc = c;
        unsigned long long plo = (unsigned long long)ms, phi = (unsigned long long)(ms >> 64);
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t yc = __shfl_up_sync(0xFFFFFFFFu, pc, o);
            const unsigned long long ylo = __shfl_up_sync(0xFFFFFFFFu, plo, o);
            const unsigned long long yhi = __shfl_up_sync(0xFFFFFFFFu, phi, o);
            if (lane >= o) {
                pc += yc;
                const unsigned long long nlo = plo + ylo;
                phi += yhi + (nlo < plo ? 1ull : 0ull);
                plo = nlo;
            }
        }
        uint32_t above_c = pc - c;
        u128 above_m = (((u128)phi << 64) | (u128)plo) - ms;
        int hit = -1;
        for (int b = top; b > top - w; --b) {
            const uint32_t bc = bin_count(sm, b);
            const u128 bm = bin_mass(sm, b);
            const bool cross = by_mass ? (above_m < tm && tm <= above_m + bm) : (above_c < tc && tc <= above_c + bc);
            if (cross) {
                hit = b;
                break;
            }
            above_c += bc;
            above_m += bm;
        }
        const unsigned hits = __ballot_sync(0xFFFFFFFFu, hit >= 0);
        if (hits && lane == __ffs(hits) - 1) {
            sm.bin = hit;
            sm.above_cnt = above_c;
            sm.above_mass = above_m;
        } else if (!hits && lane == 0) {   // not reached (targets never exceed the totals): the lowest bin
            sm.bin = 0;
            sm.above_cnt = above_c;
            sm.above_mass = above_m;
        }
    }
    __syncthreads();
}

// Mass of the whole current histogram (warp 0 sums, every thread gets it).
__device__ u128 hist_total(R32Smem& sm, int nbins)
{
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x, w = nbins / 32;
        u128 t = 0;
        for (int b = lane * w; b < lane * w + w; ++b) t += bin_mass(sm, b);
        unsigned long long lo = (unsigned long long)t, hi = (unsigned long long)(t >> 64);
        for (int o = 16; o; o >>= 1) {
            const unsigned long long ylo = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
            const unsigned long long yhi = __shfl_xor_sync(0xFFFFFFFFu, hi, o);
            const unsigned long long nlo = lo + ylo;
            hi += yhi + (nlo < lo ? 1ull : 0ull);
            lo = nlo;
        }
        if (lane == 0) sm.above_mass = ((u128)hi << 64) | (u128)lo;
    }
    __syncthreads();
    const u128 t = sm.above_mass;
    __syncthreads();
    return t;
}

// Sum over the CTA of an int (every thread gets it).
__device__ __forceinline__ int block_sum_int(R32Smem& sm, int x)
{
    x = __reduce_add_sync(0xFFFFFFFFu, x);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sm.redi[threadIdx.x >> 5] = x;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int w = 0; w < kR32Warps; ++w) t += sm.redi[w];
    __syncthreads();
    return t;
}

// Result of a descent to one key value.
struct Cut {
    uint32_t key;       // the value's key
    uint32_t above;     // elements above it (in the histogrammed set)
    u128 above_mass;    // their mass
    uint32_t count;     // elements at the value (in the histogrammed set)
};

// Descent from the top level down to one value: the value where the running
// count reaches tc, or the running mass reaches tm.  The histogrammed set is
// the elements at or above min_key, less `excess` ties of the value with key
// min_key (those a top-k cut left out).  Every thread calls it.
__device__ Cut descend(R32Smem& sm, const float* row, int V, float m, float T, bool by_mass, uint32_t tc, u128 tm,
                       uint32_t min_key, uint32_t excess, u128 excess_mass, bool level0_ready = false)
{
    Cut c{0u, 0u, 0, 0u};
    uint32_t pre = 0u, pre_mask = 0u;
    const int shifts[3] = {21, 10, 0}, nb[3] = {kR32Bins, kR32Bins, kR32Bins / 2};
#pragma unroll
    for (int lv = 0; lv < 3; ++lv) {
        if (lv > 0 || !level0_ready) level_pass(sm, row, V, m, T, pre_mask, pre, min_key, shifts[lv], nb[lv]);
        if (excess && (min_key & pre_mask) == pre) {   // the cut value lies in this level's range
            if (threadIdx.x == 0) {
                const int b = (int)((min_key >> shifts[lv]) & (uint32_t)(nb[lv] - 1));
                const uint32_t nc = bin_count(sm, b) - excess;
                const u128 nm = bin_mass(sm, b) - excess_mass;
                for (int c = 1; c < kR32Copies; ++c) {   // the corrected bin, held in copy 0
                    sm.cnt[c][b] = 0u;
                    sm.mlo[c][b] = 0ull;
                    sm.mhi[c][b] = 0u;
                }
                sm.cnt[0][b] = nc;
                sm.mlo[0][b] = (unsigned long long)nm;
                sm.mhi[0][b] = (uint32_t)(nm >> 64);
            }
            __syncthreads();
        }
        find_crossing(sm, nb[lv], by_mass, tc - (by_mass ? 0u : c.above), tm - (by_mass ? c.above_mass : (u128)0));
        const int b = sm.bin;
        c.above += sm.above_cnt;
        c.above_mass += sm.above_mass;
        pre |= (uint32_t)b << shifts[lv];
        pre_mask |= (uint32_t)(nb[lv] - 1) << shifts[lv];
        if (lv == 2) c.count = bin_count(sm, b);
        __syncthreads();
    }
    c.key = pre;
    return c;
}

__device__ void write_failed_row(RowInfo* info, double m, int argmax, int status, float temp)
{
    info->desc.max_logit = (float)m;
    info->desc.log_norm = 0.0f;
    info->desc.cutoff_logit = (float)m;
    info->desc.cutoff_ties = 0;
    info->desc.kept = 0;
    info->desc.argmax = argmax;
    info->desc.status = status;
    info->desc.temperature = temp;
    info->p_token = nan("");
    info->z = 0.0;
    info->z_rest = 0.0;
    info->n_list = -1;
    info->cut_count = 0;
}

__device__ void row32(R32Smem& sm, const RowsArgs& a, const RowTask& task)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int V = a.vocab;
    const int64_t stride = task.is_draft ? a.stride_d : a.stride_t;
    const float* row = (const float*)(task.is_draft ? a.drf : a.tgt) + (size_t)task.row * (size_t)stride;
    RowInfo* info = a.info + task.slot;

    // 1. maximum (lowest index first), smallest key, non-finite values
    unsigned long long best = 0ull;
    uint32_t kmin = 0xFFFFFFFFu;
    int bad = 0;
    stream_row(row, V, [&](float x, int i) {
        const uint32_t u = __float_as_uint(x);
        bad |= (u & 0x7FFFFFFFu) >= 0x7F800000u && u != 0xFF800000u;   // NaN or +inf
        const uint32_t k = key32(u);
        const unsigned long long c = ((unsigned long long)k << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)i);
        best = c > best ? c : best;
        kmin = min(kmin, k);
    });
    best = warp_max_u64(best);
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    bad = __reduce_or_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
        sm.red64[warp] = best;
        sm.redu[warp] = kmin;
        sm.redi[warp] = bad;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kR32Warps; ++w) {
        best = sm.red64[w] > best ? sm.red64[w] : best;
        kmin = min(kmin, sm.redu[w]);
        bad |= sm.redi[w];
    }
    __syncthreads();
    const uint32_t m_key = (uint32_t)(best >> 32);
    const int argmax = (int)(0xFFFFFFFFu - (uint32_t)best);
    const float m = value32(m_key);
    const float T = task.temp, inv_t = 1.0f / T;
    const int status = bad ? kNonfinite : (m_key == kKeyNegInf ? kEmpty : 0);
    if (status) {
        if (tid == 0) write_failed_row(info, m, argmax, status, task.temp);
        __syncthreads();
        return;
    }

    // 2. top-k by count, then top-p by mass inside the top-k set
    const int kk = task.k_eff;
    const bool topk_on = kk > 0 && kk < V;
    const bool topp_on = task.top_p < 1.0f;
    uint32_t cut_key = kmin, ties = 0u, kept = (uint32_t)V, cut_count = 0u;
    u128 z_fix = 0;
    uint32_t min_key = 0u, excess = 0u;
    u128 excess_mass = 0, e_cut = 0;
    if (topk_on) {
        const Cut c = descend(sm, row, V, m, T, false, (uint32_t)kk, 0, 0u, 0u, 0);
        cut_key = c.key;
        ties = (uint32_t)kk - c.above;
        cut_count = c.count;
        e_cut = (u128)fix_split(exp_df(scaled_logit(value32(c.key), m, T, inv_t), sm.tab), 29);
        kept = (uint32_t)kk;
        z_fix = c.above_mass + (u128)ties * e_cut;
        min_key = c.key;
        excess = c.count - ties;
        excess_mass = (u128)excess * e_cut;
    }
    if (!topk_on || topp_on) {
        // the whole row's mass when top-k is off (one level-0 pass), and the
        // count of the smallest value (every token kept if top-p is off too)
        if (!topk_on) {
            level_pass(sm, row, V, m, T, 0u, 0u, 0u, 21, kR32Bins);   // kept for the top-p descent's first level
            z_fix = hist_total(sm, kR32Bins);
            if (!topp_on) {
                int nmin = 0;
                stream_row(row, V, [&](float x, int) { nmin += key32(__float_as_uint(x)) == kmin ? 1 : 0; });
                cut_count = (uint32_t)block_sum_int(sm, nmin);
                ties = cut_count;
            }
        }
        if (topp_on) {
            // target = top_p * Z1 rounded up, exactly: top_p = M 2^-sh with a
            // 24-bit M (Z1 < 2^77, so the product stays below 2^101)
            int E;
            const float fr = frexpf(task.top_p, &E);          // top_p = fr 2^E, fr in [0.5, 1)
            const uint32_t M = (uint32_t)ldexpf(fr, 24);       // exact: fr has 24 significant bits
            const int sh = 24 - E;                             // >= 24 for top_p < 1
            const u128 prod = z_fix * (u128)M;
            const u128 target = sh >= 127 ? (u128)1 : (prod + ((((u128)1) << sh) - 1)) >> sh;
            const Cut c = descend(sm, row, V, m, T, true, 0u, target, min_key, excess, excess_mass, !topk_on);
            const u128 e_c = (u128)fix_split(exp_df(scaled_logit(value32(c.key), m, T, inv_t), sm.tab), 29);
            // ties of the value needed to reach the target (at least one)
            const u128 need = target > c.above_mass ? target - c.above_mass : (u128)0;
            uint32_t t = e_c ? (uint32_t)((need + e_c - 1) / e_c) : c.count;
            t = max(1u, min(t, c.count));
            cut_key = c.key;
            ties = t;
            kept = c.above + t;
            z_fix = c.above_mass + (u128)t * e_c;
            cut_count = c.count + (c.key == min_key ? excess : 0u);   // every token at the value, kept or not
        }
    }

    // 3. the record and the row's token
    const double z = u128_to_double(z_fix) * (1.0 / 288230376151711744.0);
    const int d = task.token;
    int tie_rank = 0;
    bool tok_kept = false;
    uint32_t kd = 0u;
    if (d >= 0 && d < V) {
        kd = key32(__float_as_uint(__ldg(row + d)));
        if (kd == cut_key && ties < cut_count) {   // its rank among the ties decides
            int n_before = 0;
            for (int i = tid; i < d; i += kR32Threads) n_before += key32(__float_as_uint(__ldg(row + i))) == cut_key ? 1 : 0;
            tie_rank = block_sum_int(sm, n_before);
            tok_kept = (uint32_t)tie_rank < ties;
        } else {
            tok_kept = kd >= cut_key;
        }
    }
    if (tid == 0) {
        info->desc.max_logit = m;
        info->desc.log_norm = logf((float)z);
        info->desc.cutoff_logit = value32(cut_key);
        info->desc.cutoff_ties = (int)ties;
        info->desc.kept = (int)kept;
        info->desc.argmax = argmax;
        info->desc.status = 0;
        info->desc.temperature = task.temp;
        info->z = z;
        info->z_rest = z - 1.0;   // the top token's mass is exp(0)
        info->n_list = -1;
        info->cut_count = (int)cut_count;
        if (d >= 0 && d < V) {
            const dfloat e = exp_df(scaled_logit(value32(kd), m, T, inv_t), sm.tab);
            info->p_token = tok_kept ? df_val(e) / z : 0.0;
        } else {
            info->p_token = nan("");
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kR32Threads, 1) rows32_kernel(const __grid_constant__ RowsArgs a)
{
    pdl_enter();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    R32Smem& sm = *reinterpret_cast<R32Smem*>(smem_raw);
    fill_exp_table(sm.tab);
    const int n_tasks = a.counters->n_slow;
    for (int t = blockIdx.x; t < n_tasks; t += gridDim.x) row32(sm, a, a.slow_tasks.get(t));
}

// ----------------------------------------------------------------------------
// The resample kernel: one CTA per job, each thread a run of consecutive
// elements (index order), so that one block scan gives every run its tie ranks
// and one more its starting weight; the run holding the target is then
// walked by its warp.
// ----------------------------------------------------------------------------
constexpr int kRs32Threads = 512;
constexpr int kRs32Warps = kRs32Threads / 32;

struct Dist32 {
    const float* row;
    float m, T, inv_t;
    double inv_z;
    uint32_t cut;       // key of the cutoff value
    int ties;           // its kept ties (index order)
    bool partial;       // some ties left out
};

struct Rs32Smem {
    dfloat tab[64];
    unsigned long long red[kRs32Warps][2];
    int redi[kRs32Warps][2];
    int run;            // thread whose run holds the target
    unsigned long long run_target;
    int found;
};

// Exclusive prefix (thread order) of two ints over the CTA.
__device__ __forceinline__ void block_excl_int2(Rs32Smem& sm, int a, int b, int& pa, int& pb)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ya = __shfl_up_sync(0xFFFFFFFFu, ia, o), yb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
        if (lane >= o) {
            ia += ya;
            ib += yb;
        }
    }
    __syncthreads();
    if (lane == 31) {
        sm.redi[warp][0] = ia;
        sm.redi[warp][1] = ib;
    }
    __syncthreads();
    int ba = 0, bb = 0;
    for (int k = 0; k < warp; ++k) {
        ba += sm.redi[k][0];
        bb += sm.redi[k][1];
    }
    pa = ba + ia - a;
    pb = bb + ib - b;
}

// Exclusive prefix (thread order) of two u64 over the CTA, and their totals.
__device__ __forceinline__ void block_excl_u64x2(Rs32Smem& sm, unsigned long long a, unsigned long long b,
                                                 unsigned long long& pa, unsigned long long& pb,
                                                 unsigned long long& ta, unsigned long long& tb)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long ya = __shfl_up_sync(0xFFFFFFFFu, ia, o), yb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
        if (lane >= o) {
            ia += ya;
            ib += yb;
        }
    }
    __syncthreads();
    if (lane == 31) {
        sm.red[warp][0] = ia;
        sm.red[warp][1] = ib;
    }
    __syncthreads();
    unsigned long long ba = 0ull, bb = 0ull;
    ta = tb = 0ull;
    for (int k = 0; k < kRs32Warps; ++k) {
        if (k < warp) {
            ba += sm.red[k][0];
            bb += sm.red[k][1];
        }
        ta += sm.red[k][0];
        tb += sm.red[k][1];
    }
    pa = ba + ia - a;
    pb = bb + ib - b;
}

__device__ __forceinline__ unsigned long long sat_sub64(unsigned long long x, unsigned long long y)
{
    return x > y ? x - y : 0ull;
}

// floor(p 2^62) of an element kept by D, with p = exp((x - m) / T) / Z.
__device__ __forceinline__ unsigned long long weight32(const Dist32& D, float x, const dfloat* tab)
{
    const dfloat e = exp_df(scaled_logit(x, D.m, D.T, D.inv_t), tab);
    return fix_split(df_mul(e, df_of(D.inv_z)), 31);
}

// Element x's residual weight and p weight, given the ranks of x among the
// ties of each cutoff (advanced past x when it is one).
__device__ __forceinline__ void element_weights(const Dist32& P, const Dist32& Q, bool residual,
                                                unsigned long long wfix, int x, int& rp, int& rq,
                                                const dfloat* tab, unsigned long long& w_res,
                                                unsigned long long& w_p)
{
    const float xp = __ldg(P.row + x);
    const uint32_t kp = key32(__float_as_uint(xp));
    const bool in_p = kp > P.cut || (kp == P.cut && (!P.partial || rp < P.ties));
    if (P.partial && kp == P.cut) ++rp;
    bool in_q = false;
    float xq = 0.0f;
    if (residual) {
        xq = __ldg(Q.row + x);
        const uint32_t kq = key32(__float_as_uint(xq));
        in_q = kq > Q.cut || (kq == Q.cut && (!Q.partial || rq < Q.ties));
        if (Q.partial && kq == Q.cut) ++rq;
    }
    w_res = w_p = 0ull;
    if (in_p) {
        w_p = weight32(P, xp, tab);
        const unsigned long long wpw = wfix ? __umul64hi(w_p, wfix) : w_p;   // p's weighted value in the residual
        w_res = residual ? sat_sub64(wpw, in_q ? weight32(Q, xq, tab) : 0ull) : w_p;
    }
}

__global__ void __launch_bounds__(kRs32Threads, 1) resample32_kernel(const __grid_constant__ ChainArgs a, int wave)
{
    pdl_enter();
    __shared__ Rs32Smem sm;
    fill_exp_table(sm.tab);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int V = a.vocab, K = a.K;
    const int j0 = wave ? a.counters->n_jobs : 0;
    const int n_jobs = wave ? a.counters->n_jobs2 : a.counters->n_jobs;
    // this thread's run of consecutive elements
    const int per = (V + kRs32Threads - 1) / kRs32Threads;
    const int x_lo = min(V, tid * per), x_hi = min(V, x_lo + per);
    for (int jj = blockIdx.x; jj < n_jobs; jj += gridDim.x) {
        const ResampleJob job = a.jobs[j0 + jj];
        const bool residual = job.residual != 0;
        const int r = job.req, pa = job.a;
        const RowInfo& IP = a.info[slot_target(r, K, pa)];
        const int64_t trow = a.layout == 1 ? (int64_t)a.qo_indptr[r] + pa : (int64_t)r * (K + 1) + pa;
        Dist32 P, Q;
        P.row = (const float*)a.tgt + (size_t)trow * (size_t)a.stride_t;
        P.m = IP.desc.max_logit;
        P.T = IP.desc.temperature;
        P.inv_t = 1.0f / P.T;
        P.inv_z = 1.0 / IP.z;
        P.cut = key32(__float_as_uint(IP.desc.cutoff_logit));
        P.ties = IP.desc.cutoff_ties;
        P.partial = IP.desc.cutoff_ties < IP.cut_count;
        Q = P;
        if (residual) {
            const RowInfo& IQ = draft_info(a, r, pa);
            Q.row = (const float*)a.drf + ((size_t)r * K + pa) * (size_t)a.stride_d;
            Q.m = IQ.desc.max_logit;
            Q.T = IQ.desc.temperature;
            Q.inv_t = 1.0f / Q.T;
            Q.inv_z = 1.0 / IQ.z;
            Q.cut = key32(__float_as_uint(IQ.desc.cutoff_logit));
            Q.ties = IQ.desc.cutoff_ties;
            Q.partial = IQ.desc.cutoff_ties < IQ.cut_count;
        }
        // 1. tie ranks at the start of each run (only for a partially kept cutoff)
        int rp0 = 0, rq0 = 0;
        if (P.partial || (residual && Q.partial)) {
            int tp = 0, tq = 0;
            for (int x = x_lo; x < x_hi; ++x) {
                tp += (P.partial && key32(__float_as_uint(__ldg(P.row + x))) == P.cut) ? 1 : 0;
                tq += (residual && Q.partial && key32(__float_as_uint(__ldg(Q.row + x))) == Q.cut) ? 1 : 0;
            }
            block_excl_int2(sm, tp, tq, rp0, rq0);
        }
        // 2. the run's weights: residual and p
        unsigned long long s_res = 0ull, s_p = 0ull;
        {
            int rp = rp0, rq = rq0;
            for (int x = x_lo; x < x_hi; ++x) {
                unsigned long long wr, wp;
                element_weights(P, Q, residual, job.wfix, x, rp, rq, sm.tab, wr, wp);
                s_res += wr;
                s_p += wp;
            }
        }
        unsigned long long pre_res, pre_p, W, Wp;
        block_excl_u64x2(sm, s_res, s_p, pre_res, pre_p, W, Wp);
        if (job.kind == kJobSum) {   // block verification's H_j: the exact total is all it needs
            if (tid == 0) a.blk_h[(size_t)r * (K + 1) + pa] = W;
            __syncthreads();
            continue;
        }
        const bool zero = residual && W == 0ull;
        const bool use_p = !residual || zero;
        const unsigned long long Wu = use_p ? Wp : W;
        const unsigned long long u24 = uniform24(a.seed, (uint32_t)r, (uint32_t)pa, 1u);
        const unsigned long long hi = __umul64hi(Wu, u24), lo = Wu * u24;
        const unsigned long long target = (hi << 40) | (lo >> 24);   // floor(W * u)
        // 3. the run holding the target, then the first element in it whose
        //    running sum passes the target (that run's warp, lane by lane
        //    over consecutive stretches)
        const unsigned long long mine = use_p ? s_p : s_res, before = use_p ? pre_p : pre_res;
        if (tid == 0) {
            sm.run = -1;
            sm.found = -1;
        }
        __syncthreads();
        if (before <= target && target < before + mine) {
            sm.run = tid;
            sm.run_target = target - before;
        }
        __syncthreads();
        const int run = sm.run;
        if (run >= 0 && warp == run / 32) {
            const int r_lo = min(V, run * per), r_hi = min(V, r_lo + per);
            const int sub = (per + 31) / 32;
            const int s_lo = min(r_hi, r_lo + lane * sub), s_hi = min(r_hi, s_lo + sub);
            // tie ranks at this stretch's start: the run's start plus the ties in the stretches before
            int rp = __shfl_sync(0xFFFFFFFFu, rp0, run & 31), rq = __shfl_sync(0xFFFFFFFFu, rq0, run & 31);
            int tp = 0, tq = 0;
            for (int x = s_lo; x < s_hi; ++x) {
                tp += (P.partial && key32(__float_as_uint(__ldg(P.row + x))) == P.cut) ? 1 : 0;
                tq += (residual && Q.partial && key32(__float_as_uint(__ldg(Q.row + x))) == Q.cut) ? 1 : 0;
            }
            int ip = tp, iq = tq;
            for (int o = 1; o < 32; o <<= 1) {
                const int yp = __shfl_up_sync(0xFFFFFFFFu, ip, o), yq = __shfl_up_sync(0xFFFFFFFFu, iq, o);
                if (lane >= o) {
                    ip += yp;
                    iq += yq;
                }
            }
            rp += ip - tp;
            rq += iq - tq;
            const int rp_s = rp, rq_s = rq;   // the stretch's start, for the walk below
            unsigned long long ssum = 0ull;
            for (int x = s_lo; x < s_hi; ++x) {
                unsigned long long wr, wp;
                element_weights(P, Q, residual, job.wfix, x, rp, rq, sm.tab, wr, wp);
                ssum += use_p ? wp : wr;
            }
            unsigned long long incl = ssum;
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned long long tgt = sm.run_target;
            unsigned long long c = incl - ssum;
            if (c <= tgt && tgt < c + ssum) {   // this lane's stretch: walk it again
                rp = rp_s;
                rq = rq_s;
                for (int x = s_lo; x < s_hi; ++x) {
                    unsigned long long wr, wp;
                    element_weights(P, Q, residual, job.wfix, x, rp, rq, sm.tab, wr, wp);
                    c += use_p ? wp : wr;
                    if (c > tgt) {
                        sm.found = x;
                        break;
                    }
                }
            }
        }
        __syncthreads();
        if (tid == 0) {
            int x = sm.found;
            if (x < 0) x = IP.desc.argmax;   // not reached: the sums are exact
            a.out_tokens[(size_t)r * (K + 1) + pa] = x;
            if (zero && a.row_status) a.row_status[(size_t)r * (K + 1) + pa] |= kResidZero;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_rows32(const RowsArgs& a, cudaStream_t s)
{
    static int attr_set[128] = {0};   // once per device, before any graph capture
    int dev = 0;
    cudaGetDevice(&dev);
    const int di = (dev >= 0 && dev < 128) ? dev : 0;
    if (!attr_set[di]) {
        const cudaError_t e =
            cudaFuncSetAttribute(rows32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(R32Smem));
        if (e != cudaSuccess) return e;
        attr_set[di] = 1;
    }
    return launch_pdl(rows32_kernel, dim3(a.num_sms), dim3(kR32Threads), sizeof(R32Smem), s, a);
}

cudaError_t launch_resample32(const ChainArgs& a, int wave, cudaStream_t s)
{
    return launch_pdl(resample32_kernel, dim3(a.num_sms), dim3(kRs32Threads), 0, s, a, wave);
}

}  // namespace sv
