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
// kept mass after the top token.  observe() runs in one CTA and reduces in a
// fixed order, so identical inputs give identical coefficients.
//
// State (doubles): [0] slope, [1..K] bias, [K+1] g_a, [K+2] H_aa, [K+3 ..]
// g_k (K), H_ak (K), H_kk (K), [4K+3] observations, [4K+4] calls.
#include <math.h>

#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kEstThreads = 512;
constexpr int kEstWarps = kEstThreads / 32;

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

// Statistics of one call, then (every refit_every calls) the refit.  Warp w
// takes requests w, w + kEstWarps, ...; lane l positions l and l + 32.
__global__ void __launch_bounds__(kEstThreads) est_observe_kernel(double* st, const float* x, const int32_t* acc,
                                                                    const int32_t* emitted, const int32_t* vlens, int n,
                                                                    int K, int refit_every)
{
    pdl_enter();
    __shared__ double s_gb[kEstWarps][kMaxK + 1], s_hab[kEstWarps][kMaxK + 1], s_hbb[kEstWarps][kMaxK + 1];
    __shared__ double s_ga[kEstWarps], s_haa[kEstWarps], s_n[kEstWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const double slope = st[0];
    double gb[2] = {0.0, 0.0}, hab[2] = {0.0, 0.0}, hbb[2] = {0.0, 0.0};
    double ga = 0.0, haa = 0.0, cnt = 0.0;
    for (int r = warp; r < n; r += kEstWarps) {
        if (emitted[r] == 0 || acc[r] < 0) continue;
        int v = vlens ? vlens[r] : K;
        v = v < 0 ? 0 : (v > K ? K : v);
        const int a = acc[r];
        const int last = a < v - 1 ? a : v - 1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = lane + 32 * h;
            if (k > last) continue;
            const double xv = (double)x[(size_t)r * K + k];
            if (!isfinite(xv)) continue;
            const double y = k < a ? 1.0 : 0.0;
            const double p = 1.0 / (1.0 + exp(-(slope * xv + st[1 + k])));
            const double w = p * (1.0 - p);
            ga += (y - p) * xv;
            haa += w * xv * xv;
            gb[h] += y - p;
            hab[h] += w * xv;
            hbb[h] += w;
            cnt += 1.0;
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int k = lane + 32 * h;
        if (k < K) {
            s_gb[warp][k] = gb[h];
            s_hab[warp][k] = hab[h];
            s_hbb[warp][k] = hbb[h];
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        ga += __shfl_xor_sync(0xFFFFFFFFu, ga, o);
        haa += __shfl_xor_sync(0xFFFFFFFFu, haa, o);
        cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
    }
    if (lane == 0) {
        s_ga[warp] = ga;
        s_haa[warp] = haa;
        s_n[warp] = cnt;
    }
    __syncthreads();
    double* g_b = st + K + 3;
    double* h_ab = g_b + K;
    double* h_bb = h_ab + K;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        double a0 = 0.0, a1 = 0.0, a2 = 0.0;
        for (int w = 0; w < kEstWarps; ++w) {
            a0 += s_gb[w][k];
            a1 += s_hab[w][k];
            a2 += s_hbb[w][k];
        }
        g_b[k] += a0;
        h_ab[k] += a1;
        h_bb[k] += a2;
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    double a0 = 0.0, a1 = 0.0, a2 = 0.0;
    for (int w = 0; w < kEstWarps; ++w) {
        a0 += s_ga[w];
        a1 += s_haa[w];
        a2 += s_n[w];
    }
    st[K + 1] += a0;
    st[K + 2] += a1;
    st[4 * K + 3] += a2;
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
    int grid = (n * K + 255) / 256;
    if (grid < 1) grid = 1;
    if (grid > 1024) grid = 1024;
    return launch_pdl(est_predict_kernel, dim3(grid), dim3(256), 0, s, info, state, n, K, x, p, counters);
}

cudaError_t launch_est_observe(double* state, const float* x, const int32_t* accept_len, const int32_t* num_emitted,
                               const int32_t* verify_lens, int n, int K, int refit_every, cudaStream_t s)
{
    return launch_pdl(est_observe_kernel, dim3(1), dim3(kEstThreads), 0, s, state, x, accept_len, num_emitted,
                      verify_lens, n, K, refit_every);
}

}  // namespace sv
