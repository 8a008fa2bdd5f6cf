// sv_walk.cuh -- the chain walk of one request ([P3] "Identical rejection
// scheme"; [P2] accept paths stop at the planned verify length, the bonus
// comes from the last verified row), run by the chain kernel and, for the
// requests whose rows it takes, by the one-pass row kernel in the warp that
// finishes the request's last row.  [P2] jianc99/sglang PR #8; [P3]
// local-inference-lab/rtx6kpro dspark-upstream-consolidation.md.
#pragma once

#include "sv_internal.cuh"

namespace sv {
namespace {   // each translation unit that includes this header gets its own copy

// Inclusive warp scan (fp64) in lane order.
__device__ __forceinline__ double warp_scan_f64(double x)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Request r, one warp (every lane calls it).  Every lane takes its own
// positions j (lane, lane + 32): it loads the rows' results, draws u(r, j, 0)
// and decides acceptance; a ballot gives the first rejection, which is where
// the sequential walk would stop.  The emitted token is drawn from the kept
// lists (index order), one listed token per lane: weights max(0, p_x - q_x)
// (q_x found by binary search in the draft row's list) or p_x, a warp scan of
// the running sums, and the first lane whose running sum exceeds u * W.  A
// kept set too large to list becomes a job of the full-row resample kernel.
// The rows' results are read through L2 (they may come from other SMs of the
// same launch).  q_p / q_i: 32 entries of warp-private shared scratch.
// check_timeout: a bulk-copy wait of the row kernels that gave up anywhere
// fails the request (the chain kernel, which runs after them all).
__device__ __noinline__ void chain_walk(const ChainArgs& a, int r, double* q_p, int* q_i, bool check_timeout)
{
    const int lane = threadIdx.x & 31;
    const int K = a.K, width = K + 1;
    const ReqState st = a.req[r];
    const int v = st.v;
    int32_t* out = a.out_tokens + (size_t)r * width;
    const int32_t* d = a.draft_tokens + (size_t)r * K;

    // position status (target row j, draft row j, token j) and, for j < v,
    // the acceptance decision; the rows' results are read before the
    // request's state is known (every slot j <= K exists)
    const int timed_out = (check_timeout && a.counters->timeout) ? kTimeout : 0;
    int any_err = st.err | timed_out;
    unsigned long long rejects = 0ull, qzero = 0ull;
    for (int j = lane; j <= K; j += 32) {
        const RowInfo& T = a.info[slot_target(r, K, j)];
        const int t_status = __ldcg(&T.desc.status), t_argmax = __ldcg(&T.desc.argmax);
        const double p = __ldcg(&T.p_token);
        int q_status = 0;
        double q = 0.0;
        if (j < K) {
            const RowInfo& Q = draft_info(a, r, j);
            q_status = __ldcg(&Q.desc.status);
            q = __ldcg(&Q.p_token);
        }
        const int dj = j < K ? d[j] : -1;
        int ps = 0;
        if (!st.err && j <= v) {
            ps |= t_status;
            if (j < v && ((st.tok_bad >> j) & 1)) ps |= kBadToken;
            if (j < v) {
                bool accept;
                if (st.greedy) {
                    accept = dj == t_argmax;
                } else {
                    ps |= q_status;
                    const double u = uniform_f64(a.seed, (uint32_t)r, (uint32_t)j, 0u);
                    if (q > 0.0) {
                        accept = u * q < p;   // u < p / q without the division
                    } else {
                        qzero |= 1ull << j;
                        accept = p > 0.0;
                    }
                }
                if (!accept) rejects |= 1ull << j;
            }
        }
        if (j == 0) ps |= st.err | timed_out;
        any_err |= ps & kErrorMask;
        if (a.row_status) a.row_status[(size_t)r * width + j] = ps;
        out[j] = -1;
    }
    any_err = __reduce_or_sync(0xFFFFFFFFu, any_err);
    // combine the lanes' 64-bit masks
    rejects |= ((unsigned long long)__reduce_or_sync(0xFFFFFFFFu, (unsigned)rejects)) |
               ((unsigned long long)__reduce_or_sync(0xFFFFFFFFu, (unsigned)(rejects >> 32)) << 32);
    qzero |= ((unsigned long long)__reduce_or_sync(0xFFFFFFFFu, (unsigned)qzero)) |
             ((unsigned long long)__reduce_or_sync(0xFFFFFFFFu, (unsigned)(qzero >> 32)) << 32);
    if (any_err) {
        if (lane == 0) {
            a.accept_len[r] = 0;
            a.num_emitted[r] = 0;
        }
        return;
    }
    const int acc_len = rejects ? (__ffsll((long long)rejects) - 1) : v;
    const uint64_t tested = acc_len < 63 ? ((2ull << acc_len) - 1ull) : ~0ull;   // positions 0..acc_len
    __syncwarp();
    for (int j = lane; j < acc_len; j += 32) out[j] = d[j];

    int t = -1;
    int extra_bits = 0;
    const RowInfo& P = a.info[slot_target(r, K, acc_len)];
    if (st.greedy) {
        t = __ldcg(&P.desc.argmax);
    } else {
        const bool residual = acc_len < v;
        const int np = __ldcg(&P.n_list);
        const RowInfo* Qp = residual ? &draft_info(a, r, acc_len) : nullptr;
        const int nq = residual ? __ldcg(&Qp->n_list) : 0;
        if (np >= 0 && nq >= 0) {
            const bool in = lane < np;
            const int x = in ? __ldcg(&P.list_idx[lane]) : 0;
            const double px = in ? __ldcg(&P.list_p[lane]) : 0.0;
            double w = px;
            if (residual) {
                if (lane < nq) {
                    q_i[lane] = __ldcg(&Qp->list_idx[lane]);
                    q_p[lane] = __ldcg(&Qp->list_p[lane]);
                }
                __syncwarp();
                double qx = 0.0;
                if (in) {   // first q position with index >= x
                    int lo = 0, hi = nq;
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        if (q_i[mid] < x) lo = mid + 1; else hi = mid;
                    }
                    if (lo < nq && q_i[lo] == x) qx = q_p[lo];
                }
                const double rw = px - qx;
                w = (in && rw > 0.0) ? rw : 0.0;
            }
            double cum = warp_scan_f64(w);
            double W = __shfl_sync(0xFFFFFFFFu, cum, 31);
            if (residual && !(W > 0.0)) {   // empty residual: draw from p itself
                extra_bits = kResidZero;
                w = px;
                cum = warp_scan_f64(w);
                W = __shfl_sync(0xFFFFFFFFu, cum, 31);
            }
            const double target = uniform_f64(a.seed, (uint32_t)r, (uint32_t)acc_len, 1u) * W;
            const unsigned over = __ballot_sync(0xFFFFFFFFu, in && cum > target);
            if (over) {
                t = __shfl_sync(0xFFFFFFFFu, x, __ffs(over) - 1);
            } else {   // rounding left none: the last token with positive weight
                const unsigned pos = __ballot_sync(0xFFFFFFFFu, in && w > 0.0);
                t = pos ? __shfl_sync(0xFFFFFFFFu, x, 31 - __clz(pos)) : -1;
            }
        } else if (lane == 0) {
            // kept set too large to list: the resample kernel draws the token
            const int slot = atomicAdd(&a.counters->n_jobs, 1);
            ResampleJob job;
            job.req = r;
            job.a = acc_len;
            job.residual = residual ? 1 : 0;
            job.done = 0;
            job.kind = kJobDraw;
            job.pad = 0;
            job.wfix = 0ull;
            a.jobs[slot] = job;
            t = -2;
        }
    }
    if (lane == 0) {
        if (t != -2) out[acc_len] = t;
        a.accept_len[r] = acc_len;
        a.num_emitted[r] = acc_len + 1;
        if (a.row_status) {
            const uint64_t qz = qzero & tested;
            for (int j = 0; j < v; ++j)
                if ((qz >> j) & 1) a.row_status[(size_t)r * width + j] |= kQZero;
            if (extra_bits) a.row_status[(size_t)r * width + acc_len] |= extra_bits;
        }
    }
}

// The outputs of a request whose rows will never all be processed (a
// bulk-copy wait of the row kernel gave up while it held one of them): an
// error with status SV_ROW_TIMEOUT at position 0.  Every lane calls it.
__device__ __forceinline__ void chain_fail(const ChainArgs& a, int r)
{
    const int lane = threadIdx.x & 31;
    const int width = a.K + 1;
    for (int j = lane; j < width; j += 32) {
        a.out_tokens[(size_t)r * width + j] = -1;
        if (a.row_status) a.row_status[(size_t)r * width + j] = j == 0 ? kTimeout : 0;
    }
    if (lane == 0) {
        a.accept_len[r] = 0;
        a.num_emitted[r] = 0;
    }
}

}  // namespace
}  // namespace sv
