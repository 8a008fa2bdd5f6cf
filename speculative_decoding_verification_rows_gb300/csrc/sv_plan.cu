// sv_plan.cu -- the confidence-scheduled verify-budget planner.
//
// NVIDIA/TensorRT-LLM PR #17056, description section "Scheduler": prefix
// survival is the cumulative product of per-position confidences, and the
// batch's verify budget is handed out by global survival rank with a
// value-independent tie-break, so the path needs no host synchronisation;
// section "Ragged (per-request) verification": windows packed on a flat token
// axis by qo_indptr and padded to a token bucket; review commit, "Cost model":
// a request submits verify_len + 1 tokens (its bonus row included).
//
// One CTA: survivals in fp32 left to right per request, a 64-bit rank key
// (survival bits, then position ascending, then request ascending -- every
// key distinct), a byte-wise radix select of the N_sel-th largest key, and a
// count per request.  The keys live in shared memory when they fit (12,288 of
// them), else in the workspace; the select stops at the first digit whose
// keys are all selected (every key of the chosen prefix is then >= the
// prefix with zeros below).  Survival never grows along a request and the tie-break
// prefers earlier positions, so each request's selection is a prefix and its
// count is its verify length.  No device-to-host readback anywhere.
#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanSmemKeys = 12288;   // rank keys held in shared memory (96 KB)

__device__ __forceinline__ long long warp_sum_ll(long long x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}

__device__ __forceinline__ unsigned long long rank_key(float s, int i, int r)
{
    return ((unsigned long long)__float_as_uint(s) << 32) | ((unsigned long long)(0xFFFu - (uint32_t)i) << 20) |
           (unsigned long long)(0xFFFFFu - (uint32_t)r);
}

template <bool SMEM>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const float* conf, int ld, const int32_t* draft_len, int n,
                                                             int K, int budget_arg, const int32_t* budget_dev,
                                                             int32_t* verify_lens, int32_t* qo, int32_t* total,
                                                             int32_t* status, unsigned long long* keys_ws)
{
    extern __shared__ unsigned long long s_keys[];
    unsigned long long* keys = SMEM ? s_keys : keys_ws;
    pdl_enter();
    const int budget = budget_dev ? *budget_dev : budget_arg;   // chosen on the device, or given
    __shared__ uint32_t hist[256];
    __shared__ int s_digit, s_kk, s_any_bad, s_done;
    __shared__ long long s_ncand;
    __shared__ int s_warp[33];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_any_bad = 0;
        s_ncand = 0;
    }
    __syncthreads();
    // survivals and rank keys: keys[i * n + r] (consecutive requests side by
    // side: no bank conflicts), 0 for positions past K_r
    long long local = 0;
    for (int r = tid; r < n; r += kPlanThreads) {
        int kr = draft_len ? draft_len[r] : K;
        if (kr < 0 || kr > K) {
            atomicOr(&s_any_bad, 1);
            kr = kr < 0 ? 0 : K;
        }
        // eight confidences loaded at a time (independent loads), then
        // multiplied in order
        float s = 1.0f;
        for (int i0 = 0; i0 < K; i0 += 8) {
            float cv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) cv[u] = i0 + u < kr ? conf[(size_t)r * ld + i0 + u] : 0.0f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u;
                if (i >= K) break;
                unsigned long long key = 0ull;
                if (i < kr) {
                    const float c = (cv[u] > 0.0f) ? fminf(cv[u], 1.0f) : 0.0f;   // NaN and -0 -> +0
                    s = __fmul_rn(s, c);
                    key = rank_key(s, i, r);
                }
                keys[(size_t)i * n + r] = key;
            }
        }
        local += kr;
    }
    local = warp_sum_ll(local);
    if (lane == 0 && local) atomicAdd((unsigned long long*)&s_ncand, (unsigned long long)local);
    __syncthreads();
    const long long ncand = s_ncand;
    long long nsel = (long long)budget - n;
    if (nsel > ncand) nsel = ncand;
    // N_sel-th largest key over the real candidates.  Every real key is
    // distinct and nonzero (i < 4095 keeps the position field above zero), so
    // key 0 marks an empty slot.
    unsigned long long kth = ~0ull;
    if (nsel > 0) {
        unsigned long long prefix = 0ull, mask = 0ull;
        int kk = (int)nsel;
        for (int digit = 0; digit < 8; ++digit) {   // 8-bit digits, most significant first
            if (tid == 0) s_done = 0;
            const int shift = 56 - 8 * digit;
            for (int b = tid; b < 256; b += kPlanThreads) hist[b] = 0u;
            __syncthreads();
            for (long long c = tid; c < (long long)n * K; c += kPlanThreads) {
                const unsigned long long key = keys[c];
                if (key != 0ull && (key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255ull], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                uint32_t cnt[8], sum = 0u;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    cnt[i] = hist[255 - 8 * lane - i];
                    sum += cnt[i];
                }
                uint32_t incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += y;
                }
                uint32_t excl = incl - sum;
                if (excl < (uint32_t)kk && (uint32_t)kk <= incl) {
                    for (int i = 0; i < 8; ++i) {
                        if (excl + cnt[i] >= (uint32_t)kk) {
                            s_digit = 255 - 8 * lane - i;
                            s_kk = kk - (int)excl;
                            s_done = excl + cnt[i] == (uint32_t)kk;   // every key of this digit is selected
                            break;
                        }
                        excl += cnt[i];
                    }
                }
            }
            __syncthreads();
            prefix |= (unsigned long long)s_digit << shift;
            mask |= 255ull << shift;
            kk = s_kk;
            const int done = s_done;
            __syncthreads();
            if (done) break;
        }
        kth = prefix;
    }
    // verify lengths: selected keys are >= kth; along a request they form a prefix
    int run = 0;
    for (int r0 = 0; r0 < n; r0 += kPlanThreads) {
        const int r = r0 + tid;
        int vr = 0;
        if (r < n && nsel > 0) {
            for (int i = 0; i < K; ++i) {
                const unsigned long long key = keys[(size_t)i * n + r];
                if (key == 0ull || key < kth) break;
                ++vr;
            }
        }
        const int w = r < n ? vr + 1 : 0;   // window: verified drafts + the bonus row
        int incl = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int x = s_warp[lane];
            int xi = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, xi, o);
                if (lane >= o) xi += y;
            }
            s_warp[lane] = xi - x;
            if (lane == 31) s_warp[32] = xi;
        }
        __syncthreads();
        const int excl = run + s_warp[warp] + incl - w;
        if (r < n) {
            verify_lens[r] = vr;
            qo[r] = excl;
        }
        if (r == n - 1) {
            qo[n] = excl + w;
            *total = excl + w;
        }
        run += s_warp[32];
        __syncthreads();
    }
    if (tid == 0 && status) *status = s_any_bad;
}

// ----------------------------------------------------------------------------
// Budget from a profiled step-cost table (NVIDIA/TensorRT-LLM PR #17056,
// description "What is here / Planner"; review commit, "Cost model").
//
// Theta(B) = tau(B) / (cost(B) + fixed + batch overhead), tau(B) = n + the sum
// of the B - n largest survivals, cost(B) = the cost of the first shelf whose
// token count is >= B.  Inside one shelf tau never falls and the cost is
// constant, so only each shelf's right edge (clipped to the largest budget)
// can win; ties go to the larger budget.  One CTA: survivals as the planner
// computes them, a bitonic sort of their fp32 bit patterns (non-negative, so
// the bits order like the values) in shared memory, fp64 sums per thread
// chunk and a scan of the chunk sums, Theta per shelf, an argmax.
// ----------------------------------------------------------------------------
constexpr int kBudgetThreads = 1024;

__global__ void __launch_bounds__(kBudgetThreads) budget_kernel(const float* conf, int ld, const int32_t* draft_len, int n,
                                                                 int K, int P, const int32_t* cost_tokens,
                                                                 const float* cost_ms, int n_cost, float fixed_ms,
                                                                 const int32_t* batch_sizes, const float* batch_ms,
                                                                 int n_batch, int bucket, int32_t* budget_out,
                                                                 int32_t* budget_status)
{
    pdl_enter();
    extern __shared__ uint32_t sv[];                  // P survival bit patterns, P a power of two
    __shared__ double s_chunk[kBudgetThreads];        // per-thread chunk sums, then their exclusive scan
    __shared__ double s_warp[32];
    __shared__ long long s_ncand;
    __shared__ int s_bad, s_table_bad;
    __shared__ double s_best[32];
    __shared__ long long s_best_b[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_ncand = 0;
        s_bad = 0;
        s_table_bad = 0;
    }
    for (int i = tid; i < P; i += kBudgetThreads) sv[i] = 0u;
    __syncthreads();
    long long local = 0;
    for (int r = tid; r < n; r += kBudgetThreads) {
        int kr = draft_len ? draft_len[r] : K;
        if (kr < 0 || kr > K) {
            atomicOr(&s_bad, 1);
            kr = kr < 0 ? 0 : K;
        }
        float s = 1.0f;
        for (int i0 = 0; i0 < kr; i0 += 8) {   // eight loads at a time, then the products in order
            float cv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) cv[u] = i0 + u < kr ? conf[(size_t)r * ld + i0 + u] : 0.0f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (i0 + u >= kr) break;
                const float c = (cv[u] > 0.0f) ? fminf(cv[u], 1.0f) : 0.0f;   // NaN and -0 -> +0
                s = __fmul_rn(s, c);
                sv[r * K + i0 + u] = __float_as_uint(s);
            }
        }
        local += kr;
    }
    // the table: shelves strictly ascending, costs and overheads finite and >= 0
    for (int j = tid; j < n_cost; j += kBudgetThreads) {
        const float cj = cost_ms[j];
        if (!(isfinite(cj) && cj >= 0.0f) || (j > 0 && cost_tokens[j] <= cost_tokens[j - 1])) atomicOr(&s_table_bad, 1);
    }
    for (int j = tid; j < n_batch; j += kBudgetThreads) {
        const float bj = batch_ms[j];
        if (!(isfinite(bj) && bj >= 0.0f)) atomicOr(&s_table_bad, 1);
    }
    if (tid == 0 && !(isfinite(fixed_ms) && fixed_ms >= 0.0f)) atomicOr(&s_table_bad, 1);
    local = warp_sum_ll(local);
    if (lane == 0 && local) atomicAdd((unsigned long long*)&s_ncand, (unsigned long long)local);
    __syncthreads();
    // descending bitonic sort
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < P; i += kBudgetThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const uint32_t x = sv[i], y = sv[ixj];
                    const bool desc = (i & k) == 0;
                    if (desc ? x < y : x > y) {
                        sv[i] = y;
                        sv[ixj] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
    // chunk sums (chunk = E consecutive sorted values per thread), exclusive scan
    const int E = (P + kBudgetThreads - 1) / kBudgetThreads;
    double cs = 0.0;
    for (int e = 0; e < E; ++e) {
        const int i = tid * E + e;
        if (i < P) cs += (double)__uint_as_float(sv[i]);
    }
    double incl = cs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const double x = s_warp[lane];
        double xi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, xi, o);
            if (lane >= o) xi += y;
        }
        s_warp[lane] = xi - x;
    }
    __syncthreads();
    s_chunk[tid] = s_warp[warp] + incl - cs;
    __syncthreads();

    const long long ncand = s_ncand;
    const long long m_max = ncand < (long long)(bucket - n) ? ncand : (long long)(bucket - n);
    const long long b_max = n + m_max;
    double batch_oh = 0.0;
    if (n_batch > 0) {
        int j = 0;
        while (j < n_batch - 1 && batch_sizes[j] < n) ++j;
        batch_oh = (double)batch_ms[j];
    }
    // each thread: shelves j = tid, tid + 1024, ...; candidate B = min(t_j, b_max)
    double best = -1.0;
    long long best_b = -1;
    if (!s_table_bad) {
        for (int j = tid; j < n_cost; j += kBudgetThreads) {
            const long long t = cost_tokens[j];
            if (t < n) continue;                                   // cannot hold the anchors
            if (j > 0 && (long long)cost_tokens[j - 1] >= b_max) continue;   // b_max sits on an earlier shelf
            const long long b = t < b_max ? t : b_max;
            const long long m = b - n;
            // tau = n + sum of the m largest survivals
            double tau = (double)n;
            if (m > 0) {
                const long long owner = (m - 1) / E;
                double part = s_chunk[owner];
                for (long long i = owner * E; i < m; ++i) part += (double)__uint_as_float(sv[i]);
                tau += part;
            }
            const double th = tau / ((double)cost_ms[j] + (double)fixed_ms + batch_oh);
            if (th > best || (th == best && b > best_b)) {
                best = th;
                best_b = b;
            }
        }
    }
    // block argmax, ties to the larger budget
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const double ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const long long obb = __shfl_xor_sync(0xFFFFFFFFu, best_b, o);
        if (ob > best || (ob == best && obb > best_b)) {
            best = ob;
            best_b = obb;
        }
    }
    if (lane == 0) {
        s_best[warp] = best;
        s_best_b[warp] = best_b;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kBudgetThreads / 32; ++w)
            if (s_best[w] > best || (s_best[w] == best && s_best_b[w] > best_b)) {
                best = s_best[w];
                best_b = s_best_b[w];
            }
        int st = s_bad ? 1 : 0;
        if (s_table_bad) st |= 4;
        if (best_b < 0) {
            if (!s_table_bad) st |= 2;
            best_b = b_max;
        }
        *budget_out = (int32_t)best_b;
        if (budget_status) *budget_status = st;
    }
}

// Acceptance against trimming (NVIDIA/TensorRT-LLM PR #17056, the commit that
// adds trim_regret_rate): tokens emitted, tokens submitted, requests trimmed,
// trimmed requests that accepted their whole window.  One CTA.
__global__ void __launch_bounds__(kBudgetThreads) stats_kernel(const int32_t* accept_len, const int32_t* num_emitted,
                                                                const int32_t* verify_lens, const int32_t* draft_len,
                                                                int n, int K, long long* out)
{
    pdl_enter();
    __shared__ unsigned long long s_acc[4];
    if (threadIdx.x < 4) s_acc[threadIdx.x] = 0ull;
    __syncthreads();
    unsigned long long a0 = 0, a1 = 0, a2 = 0, a3 = 0;
    for (int r = threadIdx.x; r < n; r += kBudgetThreads) {
        const int acc = accept_len[r];
        if (num_emitted[r] == 0 || acc < 0) continue;
        int kr = draft_len ? draft_len[r] : K;
        kr = kr < 0 ? 0 : (kr > K ? K : kr);
        const int v = verify_lens ? verify_lens[r] : kr;
        a0 += (unsigned long long)(acc + 1);
        a1 += (unsigned long long)(v + 1);
        if (v < kr) {
            a2 += 1;
            if (acc == v) a3 += 1;
        }
    }
    atomicAdd(&s_acc[0], a0);
    atomicAdd(&s_acc[1], a1);
    atomicAdd(&s_acc[2], a2);
    atomicAdd(&s_acc[3], a3);
    __syncthreads();
    if (threadIdx.x < 4) out[threadIdx.x] = (long long)s_acc[threadIdx.x];
}

}  // namespace

cudaError_t launch_plan(const float* conf, int ld, const int32_t* draft_len, int n, int K, int budget,
                        const int32_t* budget_dev, int32_t* verify_lens, int32_t* qo_indptr, int32_t* total,
                        int32_t* status, unsigned long long* keys, cudaStream_t s)
{
    if ((long long)n * K <= kPlanSmemKeys) {
        static int attr_set[128] = {0};   // once per device, before any graph capture
        int dev = 0;
        cudaGetDevice(&dev);
        int& done = attr_set[(dev >= 0 && dev < 128) ? dev : 0];
        if (!done) {
            const cudaError_t e = cudaFuncSetAttribute(plan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       (int)(kPlanSmemKeys * sizeof(unsigned long long)));
            if (e != cudaSuccess) return e;
            done = 1;
        }
        const size_t smem = sizeof(unsigned long long) * (size_t)(n * K > 0 ? n * K : 1);
        return launch_pdl(plan_kernel<true>, dim3(1), dim3(kPlanThreads), smem, s, conf, ld, draft_len, n, K, budget,
                          budget_dev, verify_lens, qo_indptr, total, status, keys);
    }
    return launch_pdl(plan_kernel<false>, dim3(1), dim3(kPlanThreads), 0, s, conf, ld, draft_len, n, K, budget,
                      budget_dev, verify_lens, qo_indptr, total, status, keys);
}

cudaError_t launch_budget(const float* conf, int ld, const int32_t* draft_len, int n, int K, const int32_t* cost_tokens,
                          const float* cost_ms, int n_cost, float fixed_ms, const int32_t* batch_sizes,
                          const float* batch_ms, int n_batch, int bucket, int32_t* budget_out, int32_t* budget_status,
                          cudaStream_t s)
{
    int P = 2;
    while (P < n * K) P <<= 1;
    const size_t smem = sizeof(uint32_t) * (size_t)P;
    static int attr_set[128] = {0};   // once per device, before any graph capture
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 128 || !attr_set[dev]) {
        const cudaError_t err =
            cudaFuncSetAttribute(budget_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(sizeof(uint32_t) * kBudgetMaxCand));
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < 128) attr_set[dev] = 1;
    }
    return launch_pdl(budget_kernel, dim3(1), dim3(kBudgetThreads), smem, s, conf, ld, draft_len, n, K, P, cost_tokens,
                      cost_ms, n_cost, fixed_ms, batch_sizes, batch_ms, n_batch, bucket, budget_out, budget_status);
}

cudaError_t launch_stats(const int32_t* accept_len, const int32_t* num_emitted, const int32_t* verify_lens,
                         const int32_t* draft_len, int n, int K, long long* out, cudaStream_t s)
{
    return launch_pdl(stats_kernel, dim3(1), dim3(kBudgetThreads), 0, s, accept_len, num_emitted, verify_lens, draft_len,
                      n, K, out);
}

}  // namespace sv
