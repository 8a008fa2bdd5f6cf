// sv_est.cu -- the online acceptance estimator.
//
// jianc99/sglang PR #8, DFLASH adaptive-verification commits: a logistic model
// calibrated while serving, p_k = sigmoid(slope * x_k + bias_k), x_k =
// logit(q_max) of the draft distribution at position k (greedy requests at
// T = 1), clamped to +-40; observe() adds the accepted drafts and the first
// rejected one to Newton (IRLS) statistics, and every refit_every calls a
// damped ridge Newton step on the arrowhead system updates the coefficients in
// place (a slope step that would make the slope negative is halved up to 8
// times, then dropped; the intercepts step given the slope step taken).  The
// refit counter lives in the state, so nothing synchronises with the host.
//
// The features come from the row transform the verify step uses (the draft
// rows are processed as plain rows by the prep and row kernels); q_max = 1 / z
// because the top token's mass is exp(0), so x = -ln(z - 1) with z - 1 the
// kept mass after the top token.  observe() runs as one cluster of CTAs and
// reduces in a fixed order, so identical inputs give identical coefficients.
//
// State (doubles): [0] slope, [1..K] bias, [K+1] g_a, [K+2] H_aa, [K+3 ..]
// g_k (K), H_ak (K), H_kk (K), [4K+3] observations, [4K+4] calls.
#include <math.h>

#include <cooperative_groups.h>

#include "sv_internal.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace {

__global__ void est_init_kernel(double* st, int K)
{
    pdl_enter();
    for (int i = threadIdx.x; i < 4 * K + 5; i += blockDim.x) st[i] = (i == 0) ? 0.5 : (i <= K ? -0.2 : 0.0);
}

// One thread per draft row (request r = u / K, position k = u % K).
__global__ void est_predict_kernel(const RowInfo* info, const double* st, int n, int K, float* x_out, float* p_out,
                                   const Counters* counters)
{
    pdl_enter();
    const int rows = n * K;
    for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < rows; u += gridDim.x * blockDim.x) {
        const RowInfo& I = info[u];
        double x;
        if ((I.desc.status & kErrorMask) || counters->timeout) {
            x = nan("");
        } else {
            x = I.z_rest > 0.0 ? -log(I.z_rest) : INFINITY;
            x = x > 40.0 ? 40.0 : (x < -40.0 ? -40.0 : x);
        }
        const float xf = (float)x;
        const int k = u % K;
        x_out[u] = xf;
        p_out[u] = (float)(1.0 / (1.0 + exp(-(st[0] * (double)xf + st[1 + k]))));
    }
}

// Statistics of one call, then (every refit_every calls) the refit.  A
// cluster of kObsCTAs CTAs, one (request, position) item per thread, item
// i = r * K + k: the fp64 terms of the items spread over the cluster's SMs
// (GB300's fp64 pipe is narrow).  Each warp sums its items over all
// positions by a butterfly and per position in item order, the CTA adds its
// warps' sums in warp order, and CTA 0 adds the CTAs' sums in CTA order
// through distributed shared memory: short dependent chains, in an order
// fixed in advance, so identical inputs give identical coefficients.
constexpr int kObsCTAs = 8;
constexpr int kObsThreads = 128;

struct ObsSums {
    double pos[3][kMaxK + 1];   // per position: sum (y - p), sum w x, sum w
    double all[3];              // over all items: sum (y - p) x, sum w x^2, count
};

__global__ void __cluster_dims__(kObsCTAs, 1, 1) __launch_bounds__(kObsThreads)
    est_observe_kernel(double* st, const float* x, const int32_t* acc, const int32_t* emitted, const int32_t* vlens,
                       int n, int K, int refit_every)
{
    pdl_enter();
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ double s_t[kObsThreads][3];                    // this round's items: y - p, w x, w
    __shared__ int s_ok[kObsThreads];
    __shared__ double s_w[kObsThreads / 32][3];                 // per warp: sum (y - p) x, sum w x^2, count
    __shared__ double s_pw[kObsThreads / 32][3][kMaxK + 1];     // per warp and position: the three sums
    __shared__ ObsSums sums;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, rank = (int)cluster.block_rank();
    const double slope = st[0];
    const int items = n * K;
    // thread k < K keeps position k's sums of this CTA; thread K the totals
    double q0 = 0.0, q1 = 0.0, q2 = 0.0;
    for (int base = 0; base < items; base += kObsCTAs * kObsThreads) {
        const int i0 = base + rank * kObsThreads, i = i0 + tid;
        bool ok = false;
        double t0 = 0.0, t1 = 0.0, t2 = 0.0, t3 = 0.0, t4 = 0.0;
        if (i < items) {
            const int r = i / K, k = i - r * K;
            const int em = emitted[r], a = acc[r], vr = vlens ? vlens[r] : K;   // independent loads
            const double xv = (double)x[i], bk = st[1 + k];
            const int v = vr < 0 ? 0 : (vr > K ? K : vr);
            const int last = a < v - 1 ? a : v - 1;
            if (em != 0 && a >= 0 && k <= last && isfinite(xv)) {
                const double y = k < a ? 1.0 : 0.0;
                const double p = 1.0 / (1.0 + exp(-(slope * xv + bk)));
                const double w = p * (1.0 - p);
                t0 = (y - p) * xv;
                t1 = w * xv * xv;
                t2 = y - p;
                t3 = w * xv;
                t4 = w;
                ok = true;
            }
        }
        // the totals: a butterfly over the warp, then the warps in order
        double c0 = t0, c1 = t1, c2 = ok ? 1.0 : 0.0;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            c0 += __shfl_xor_sync(0xFFFFFFFFu, c0, o);
            c1 += __shfl_xor_sync(0xFFFFFFFFu, c1, o);
            c2 += __shfl_xor_sync(0xFFFFFFFFu, c2, o);
        }
        if (lane == 0) {
            s_w[warp][0] = c0;
            s_w[warp][1] = c1;
            s_w[warp][2] = c2;
        }
        s_t[tid][0] = t2;
        s_t[tid][1] = t3;
        s_t[tid][2] = t4;
        s_ok[tid] = ok;
        __syncthreads();
        // per position: each warp's items of that position in item order, then the warps in order
        const int n_here = min(kObsThreads, items - i0);
        for (int j = tid; j < (kObsThreads / 32) * K; j += kObsThreads) {
            const int k = j % K, w = j / K;
            double b0 = 0.0, b1 = 0.0, b2 = 0.0;
            for (int l = ((k - (i0 + 32 * w) % K) % K + K) % K; l < 32; l += K) {
                const int jj = 32 * w + l;
                if (jj < n_here && s_ok[jj]) {
                    b0 += s_t[jj][0];
                    b1 += s_t[jj][1];
                    b2 += s_t[jj][2];
                }
            }
            s_pw[w][0][k] = b0;
            s_pw[w][1][k] = b1;
            s_pw[w][2][k] = b2;
        }
        __syncthreads();
        if (tid < K) {
#pragma unroll
            for (int w = 0; w < kObsThreads / 32; ++w) {
                q0 += s_pw[w][0][tid];
                q1 += s_pw[w][1][tid];
                q2 += s_pw[w][2][tid];
            }
        } else if (tid == K) {
#pragma unroll
            for (int w = 0; w < kObsThreads / 32; ++w) {
                q0 += s_w[w][0];
                q1 += s_w[w][1];
                q2 += s_w[w][2];
            }
        }
        __syncthreads();
    }
    if (tid < K) {
        sums.pos[0][tid] = q0;
        sums.pos[1][tid] = q1;
        sums.pos[2][tid] = q2;
    } else if (tid == K) {
        sums.all[0] = q0;
        sums.all[1] = q1;
        sums.all[2] = q2;
    }
    cluster.sync();
    double* g_b = st + K + 3;
    double* h_ab = g_b + K;
    double* h_bb = h_ab + K;
    double tot[3] = {0.0, 0.0, 0.0};
    if (rank == 0 && tid <= K) {
        for (int c = 0; c < kObsCTAs; ++c) {
            const ObsSums* o = cluster.map_shared_rank(&sums, c);
#pragma unroll
            for (int f = 0; f < 3; ++f) tot[f] += tid < K ? o->pos[f][tid] : o->all[f];
        }
    }
    cluster.sync();   // the other CTAs' sums stay in place until CTA 0 has read them
    if (rank != 0) return;
    if (tid < K) {
        g_b[tid] += tot[0];
        h_ab[tid] += tot[1];
        h_bb[tid] += tot[2];
    }
    if (tid == K) {
        st[K + 1] += tot[0];
        st[K + 2] += tot[1];
        st[4 * K + 3] += tot[2];
    }
    __syncthreads();
    if (tid != 0) return;
    st[4 * K + 4] += 1.0;
    if (refit_every <= 0 || fmod(st[4 * K + 4], (double)refit_every) != 0.0) return;
    // refit: damped ridge Newton step on the arrowhead system
    const double lam = 1e-3, nobs = st[4 * K + 3];
    if (nobs > 0.0) {
        double num = st[K + 1], den = st[K + 2] + lam;
        for (int k = 0; k < K; ++k) {
            num -= h_ab[k] * g_b[k] / (h_bb[k] + lam);
            den -= h_ab[k] * h_ab[k] / (h_bb[k] + lam);
        }
        double t = num / den;
        const double d = nobs / (nobs + 50.0);
        for (int i = 0; i < 8 && st[0] + d * t < 0.0; ++i) t *= 0.5;
        if (st[0] + d * t < 0.0) t = 0.0;
        bool ok = isfinite(t);
        for (int k = 0; k < K; ++k) ok = ok && isfinite((g_b[k] - h_ab[k] * t) / (h_bb[k] + lam));
        if (ok) {
            for (int k = 0; k < K; ++k) st[1 + k] += d * (g_b[k] - h_ab[k] * t) / (h_bb[k] + lam);
            st[0] += d * t;
        }
    }
    for (int i = K + 1; i < 4 * K + 4; ++i) st[i] = 0.0;
}

}  // namespace

cudaError_t launch_est_init(double* state, int K, cudaStream_t s)
{
    return launch_pdl(est_init_kernel, dim3(1), dim3(256), 0, s, state, K);
}

cudaError_t launch_est_predict(const RowInfo* info, const double* state, int n, int K, float* x, float* p,
                               const Counters* counters, cudaStream_t s)
{
    // one warp per CTA: the fp64 log and exp of the rows spread over the SMs
    int grid = (n * K + 31) / 32;
    if (grid < 1) grid = 1;
    if (grid > 4096) grid = 4096;
    return launch_pdl(est_predict_kernel, dim3(grid), dim3(32), 0, s, info, state, n, K, x, p, counters);
}

cudaError_t launch_est_observe(double* state, const float* x, const int32_t* accept_len, const int32_t* num_emitted,
                               const int32_t* verify_lens, int n, int K, int refit_every, cudaStream_t s)
{
    return launch_pdl(est_observe_kernel, dim3(kObsCTAs), dim3(kObsThreads), 0, s, state, x, accept_len, num_emitted,
                      verify_lens, n, K, refit_every);
}

}  // namespace sv
