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
// count per request.  Survival never grows along a request and the tie-break
// prefers earlier positions, so each request's selection is a prefix and its
// count is its verify length.  No device-to-host readback anywhere.
#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ unsigned long long rank_key(float s, int i, int r)
{
    return ((unsigned long long)__float_as_uint(s) << 32) | ((unsigned long long)(0xFFFu - (uint32_t)i) << 20) |
           (unsigned long long)(0xFFFFFu - (uint32_t)r);
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const float* conf, int ld, const int32_t* draft_len, int n,
                                                             int K, int budget, int32_t* verify_lens, int32_t* qo,
                                                             int32_t* total, int32_t* status, unsigned long long* keys)
{
    pdl_enter();
    __shared__ uint32_t hist[256];
    __shared__ int s_digit, s_kk, s_any_bad;
    __shared__ long long s_ncand;
    __shared__ int s_warp[33];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_any_bad = 0;
        s_ncand = 0;
    }
    __syncthreads();
    // survivals and rank keys: keys[r * K + i], 0 for positions past K_r
    long long local = 0;
    for (int r = tid; r < n; r += kPlanThreads) {
        int kr = draft_len ? draft_len[r] : K;
        if (kr < 0 || kr > K) {
            atomicOr(&s_any_bad, 1);
            kr = kr < 0 ? 0 : K;
        }
        float s = 1.0f;
        for (int i = 0; i < K; ++i) {
            unsigned long long key = 0ull;
            if (i < kr) {
                float c = conf[(size_t)r * ld + i];
                c = (c > 0.0f) ? fminf(c, 1.0f) : 0.0f;   // NaN and -0 -> +0
                s = __fmul_rn(s, c);
                key = rank_key(s, i, r);
            }
            keys[(size_t)r * K + i] = key;
        }
        local += kr;
    }
    atomicAdd((unsigned long long*)&s_ncand, (unsigned long long)local);
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
        for (int round = 0; round < 8; ++round) {
            const int shift = 56 - 8 * round;
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
            __syncthreads();
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
                const unsigned long long key = keys[(size_t)r * K + i];
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

}  // namespace

cudaError_t launch_plan(const float* conf, int ld, const int32_t* draft_len, int n, int K, int budget,
                        int32_t* verify_lens, int32_t* qo_indptr, int32_t* total, int32_t* status,
                        unsigned long long* keys, cudaStream_t s)
{
    return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, conf, ld, draft_len, n, K, budget, verify_lens,
                      qo_indptr, total, status, keys);
}

}  // namespace sv
