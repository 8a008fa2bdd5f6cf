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
// (GB300's fp64 pipe is narrow).  Each CTA sums its items per position and
// over all positions in item order; CTA 0 then adds the CTAs' sums in CTA
// order through distributed shared memory.  The order is fixed, so identical
// inputs give identical coefficients.
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
    __shared__ double s_t[kObsThreads][5];   // this round's items: (y - p) x, w x^2, y - p, w x, w
    __shared__ int s_ok[kObsThreads];
    __shared__ ObsSums sums;
    const int tid = threadIdx.x, rank = (int)cluster.block_rank();
    const double slope = st[0];
    const int items = n * K;
    // thread k < K keeps position k's sums of this CTA; thread K the totals
    double q0 = 0.0, q1 = 0.0, q2 = 0.0;
    for (int base = 0; base < items; base += kObsCTAs * kObsThreads) {
        const int i0 = base + rank * kObsThreads, i = i0 + tid;
        bool ok = false;
        double t[5] = {0.0, 0.0, 0.0, 0.0, 0.0};
        if (i < items) {
            const int r = i / K, k = i - r * K;
            if (emitted[r] != 0 && acc[r] >= 0) {
                int v = vlens ? vlens[r] : K;
                v = v < 0 ? 0 : (v > K ? K : v);
                const int a = acc[r];
                const int last = a < v - 1 ? a : v - 1;
                const double xv = (double)x[i];
                if (k <= last && isfinite(xv)) {
                    const double y = k < a ? 1.0 : 0.0;
                    const double p = 1.0 / (1.0 + exp(-(slope * xv + st[1 + k])));
                    const double w = p * (1.0 - p);
                    t[0] = (y - p) * xv;
                    t[1] = w * xv * xv;
                    t[2] = y - p;
                    t[3] = w * xv;
                    t[4] = w;
                    ok = true;
                }
            }
        }
#pragma unroll
        for (int f = 0; f < 5; ++f) s_t[tid][f] = t[f];
        s_ok[tid] = ok;
        __syncthreads();
        const int n_here = min(kObsThreads, items - i0);
        if (tid < K) {   // position tid: the round's items of that position, in item order
            for (int j = (tid - i0 % K + K) % K; j < n_here; j += K)
                if (s_ok[j]) {
                    q0 += s_t[j][2];
                    q1 += s_t[j][3];
                    q2 += s_t[j][4];
                }
        } else if (tid == K) {
            for (int j = 0; j < n_here; ++j)
                if (s_ok[j]) {
                    q0 += s_t[j][0];
                    q1 += s_t[j][1];
                    q2 += 1.0;
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
