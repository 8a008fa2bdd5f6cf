// sv_chain.cu -- task lists, the chain rejection walk and the resample.
//
//  * prep: one CTA turns (requests, sampling parameters, windows) into the
//    row task lists of the two row kernels, checks parameters, draft tokens
//    and ragged windows ([P4] `_rejection_buffers_valid`: a window that does
//    not match qo_indptr is refused, padding rows are never read).
//  * chain: one warp per request walks its window ([P3] "Identical rejection
//    scheme"): greedy accepts iff d_j == argmax_j, otherwise accepts iff
//    u(r, j, 0) < p_j(d_j) / q_j(d_j); stops at the first rejection or at the
//    planned window ([P2] accept paths stop at the planned verify length).
//    When the rows' kept sets are listed (<= 32 tokens) it also draws the
//    emitted token in fp64: inverse CDF in index order of max(0, p_a - q_a)
//    ([P3] residual-mass reweighting) or of p_a after full acceptance ([P2]
//    the bonus comes from the last verified row).
//  * resample: one CTA per request whose kept set is too large to list draws
//    the same token from the full rows with exact 62-bit fixed-point weights
//    (fp64 per distinct logit value, integer prefix sums in index order).
//  [P2] jianc99/sglang PR #8; [P3] local-inference-lab/rtx6kpro
//  dspark-upstream-consolidation.md; [P4] NVIDIA/TensorRT-LLM PR #17056.
#include <math.h>

#include "sv_internal.cuh"
#include "sv_walk.cuh"

namespace sv {
namespace {

constexpr int kPrepThreads = 1024;
// A greedy request's histogram-path rows (argmax scans, the same cost whether
// or not an earlier test rejects) are listed this many positions ahead of the
// sampling rows of their position, so that the CTAs a short scan frees early
// take them while the first sampling tests are still being decided.
constexpr int kGreedyAhead = 2;


__device__ __forceinline__ int bad_params(float T, float top_p)
{
    if (!(T >= 0.0f) || isinf(T)) return 1;
    if (T == 0.0f) return 0;
    if (!(top_p > 0.0f)) return 1;
    return 0;
}

// Block-wide exclusive scan of two counters (blockDim = kPrepThreads).
__device__ void block_scan2(int a, int b, int* ea, int* eb, int* ta, int* tb, int* sa, int* sb)
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
    if (lane == 31) {
        sa[warp] = ia;
        sb[warp] = ib;
    }
    __syncthreads();
    if (warp == 0) {
        int wa = sa[lane], wb = sb[lane];
        int xa = wa, xb = wb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ya = __shfl_up_sync(0xFFFFFFFFu, xa, o), yb = __shfl_up_sync(0xFFFFFFFFu, xb, o);
            if (lane >= o) {
                xa += ya;
                xb += yb;
            }
        }
        sa[lane] = xa - wa;
        sb[lane] = xb - wb;
        if (lane == 31) {
            *ta = xa;
            *tb = xb;
        }
    }
    __syncthreads();
    *ea = sa[warp] + ia - a;
    *eb = sb[warp] + ib - b;
    __syncthreads();
}

// Per-unit results of the prep kernel's first phase, for its second.
struct PrepUnit {
    int req, k_eff, v, start, pos, n_rows, flags;   // flags: 1 fast, 2 greedy
    float T, tp;
};

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const __grid_constant__ ChainArgs a)
{
    pdl_enter();
    __shared__ int s_wa[32], s_wb[32];
    __shared__ int s_tot_a, s_tot_b;
    __shared__ PrepUnit s_u[kPrepThreads];
    __shared__ unsigned long long s_tokbad[kPrepThreads];
    int base_fast = 0, base_slow = 0;
    const int n_units = a.n_req;   // requests, or rows for the plain row layout
    // histogram rows of chain verification: their requests, and the rows of
    // each position over all of them (counted here, listed after the loop)
    __shared__ int s_nsr;
    __shared__ int s_pos[kMaxK + 1];    // per listing bucket: the sampling rows, then (s_posg) the greedy rows
    __shared__ int s_posg[kMaxK + 1];
    const int kinds = a.q_rows ? 1 : 2;   // histogram rows per verified position (1 for greedy requests)
    if (threadIdx.x == 0) s_nsr = 0;
    for (int j = threadIdx.x; j <= kMaxK; j += kPrepThreads) s_pos[j] = s_posg[j] = 0;
    // Chain verification with bf16 rows: when any request's kept set takes
    // the histogram path, greedy requests go there too (their rows as argmax
    // scans), so that their bytes stream while the histogram passes, bound by
    // shared-memory atomics, leave the memory idle, instead of in a launch of
    // their own before them.
    __shared__ int s_hist_greedy;
    if (threadIdx.x == 0) s_hist_greedy = 0;
    __syncthreads();
    if (a.lazy && a.dtype == 0 && a.layout != 2 && !a.shard && !(a.sp.flags & SV_SAMPLING_SMALL_TOPK)) {
        int any = 0;
        for (int u = threadIdx.x; u < a.n_req && !any; u += kPrepThreads) {
            const float T = a.sp.temperature[u];
            const int tk = a.sp.top_k ? a.sp.top_k[u] : 0;
            const int ke = (tk > 0 && tk < a.vocab) ? tk : a.vocab;
            any = T > 0.0f && ke > kFastK;
        }
        if (__syncthreads_or(any) && threadIdx.x == 0) s_hist_greedy = 1;
    }
    __syncthreads();
    const bool hist_greedy = s_hist_greedy != 0;
    const int K = a.K;
    const int W2 = a.layout == 2 ? 1 : 2 * K + 1;   // row slots per unit
    for (int u0 = 0; u0 < n_units; u0 += kPrepThreads) {
        // Phase 1, one thread per unit: parameters, window, row counts.
        const int u = u0 + threadIdx.x;
        const bool active = u < n_units;
        int nf = 0, ns = 0;
        int err = 0, v = 0, greedy = 0, k_eff = 1, req = u, start = 0;
        float T = 0.0f, tp = 1.0f;
        bool fast = true;
        if (active) {
            if (a.layout == 2) req = a.row_to_req ? a.row_to_req[u] : u / a.rows_per_req;
            const bool req_ok = req >= 0 && req < a.n_params;
            T = req_ok ? a.sp.temperature[req] : 0.0f;
            if (a.est && T == 0.0f) T = 1.0f;   // estimator features: greedy requests at T = 1
            const int tk = (req_ok && a.sp.top_k) ? a.sp.top_k[req] : 0;
            tp = (req_ok && a.sp.top_p) ? a.sp.top_p[req] : 1.0f;
            if (!req_ok || bad_params(T, tp)) err |= kBadParam;
            greedy = T == 0.0f;
            k_eff = greedy ? 1 : ((tk > 0 && tk < a.vocab) ? tk : a.vocab);
            fast = (greedy && !hist_greedy) || (!greedy && k_eff <= kFastK);
            // full-vocabulary kept sets: not under the caller's promise that
            // the batch has none, nor in a vocabulary-sharded call
            if (!err && !fast && ((a.sp.flags & SV_SAMPLING_SMALL_TOPK) || a.shard)) err |= kUnsupported;
            if (a.layout == 0) {
                v = a.verify_len ? a.verify_len[u] : K;
                if (v < 0 || v > K) {
                    err |= kBadLayout;
                    v = 0;
                }
                start = u * (K + 1);
            } else if (a.layout == 1) {
                v = a.verify_len[u];
                const long long s0 = a.qo_indptr[u], e = a.qo_indptr[u + 1];
                if (v < 0 || v > K || s0 < 0 || e - s0 != (long long)v + 1 || e > (long long)a.bucket) {
                    err |= kBadLayout;
                    v = 0;
                }
                start = (int)s0;
            }
            if (a.layout != 2 && a.shard != 2 && !greedy && v > 0 && !a.drf) err |= kBadParam;   // q needs draft logits
            if (a.layout != 2) {
                // one request-level error: a bad window first, then bad parameters
                if (err & kBadLayout) err = kBadLayout;
                else if (err & kBadParam) err = kBadParam;
            }
            if (!err) {
                // target rows 0..v, and draft rows 0..v-1 of a sampling request
                // unless their results were made beforehand (q_rows)
                const int n_rows = a.layout == 2 ? 1 : (v + 1) + ((greedy || a.q_rows) ? 0 : v);
                if (fast) nf = n_rows; else ns = n_rows;
            }
        }
        int off_f, off_s;
        block_scan2(nf, ns, &off_f, &off_s, &s_tot_a, &s_tot_b, s_wa, s_wb);
        PrepUnit pu;
        pu.req = req;
        pu.k_eff = k_eff;
        pu.v = v;
        pu.start = start;
        pu.pos = nf ? base_fast + off_f : base_slow + off_s;
        pu.n_rows = nf + ns;
        pu.flags = (fast ? 1 : 0) | (greedy ? 2 : 0);
        pu.T = T;
        pu.tp = tp;
        s_u[threadIdx.x] = pu;
        s_tokbad[threadIdx.x] = 0ull;
        __syncthreads();

        // Phase 2, one thread per (unit, row slot): the row tasks, each with
        // its own draft token (checked here; bad ones are collected per unit).
        const int n_here = min(kPrepThreads, n_units - u0);
        for (int idx = threadIdx.x; idx < n_here * W2; idx += kPrepThreads) {
            const int ul = idx / W2, i = idx - ul * W2;
            const PrepUnit q = s_u[ul];
            if (i >= q.n_rows) continue;
            const int uu = u0 + ul;
            RowTask t;
            t.req = q.req;
            t.k_eff = q.k_eff;
            t.temp = q.T;
            t.top_p = q.tp;
            t.req_rows = q.n_rows;
            if (a.layout == 2) {
                t.row = uu;
                t.slot = uu;
                t.is_draft = 0;
                const int d = a.token_per_row ? a.token_per_row[uu] : -1;
                t.token = (d >= 0 && d < a.vocab) ? d : -1;
            } else {
                const bool draft_row = i > q.v;
                const int j = draft_row ? i - q.v - 1 : i;
                t.is_draft = draft_row;
                t.row = draft_row ? (int64_t)uu * K + j : (int64_t)q.start + j;
                t.slot = draft_row ? slot_draft(uu, K, j) : slot_target(uu, K, j);
                int tok = -1;
                if (j < q.v) {
                    const int d = a.draft_tokens[(size_t)uu * K + j];
                    if (d >= 0 && d < a.vocab)
                        tok = d;
                    else if (!draft_row)
                        atomicOr(&s_tokbad[ul], 1ull << j);
                }
                t.token = tok;
            }
            const bool is_fast = (q.flags & 1) != 0;
            (is_fast ? a.fast_tasks : a.slow_tasks).put(q.pos + i, t);
            if (is_fast) a.row_sync[q.pos + i] = RowSync{0, 0u};
        }
        __syncthreads();

        // Phase 3, one thread per unit: the request state (or a row's error).
        if (active) {
            if (a.layout == 2) {
                if (err) {
                    RowInfo* info = a.info + u;
                    info->desc.max_logit = 0.0f;
                    info->desc.log_norm = 0.0f;
                    info->desc.cutoff_logit = 0.0f;
                    info->desc.cutoff_ties = 0;
                    info->desc.kept = 0;
                    info->desc.argmax = -1;
                    info->desc.status = err;
                    info->desc.temperature = T;
                    info->p_token = nan("");
                    info->z = 0.0;
                    info->n_list = -1;
                    info->cut_count = 0;
                }
            } else {
                // bad draft tokens of a request that failed before its rows
                // were listed are read here (its rows were not)
                uint64_t tok_bad = s_tokbad[threadIdx.x];
                if (err)
                    for (int j = 0; j < v; ++j) {
                        const int d = a.draft_tokens[(size_t)u * K + j];
                        if (d < 0 || d >= a.vocab) tok_bad |= 1ull << j;
                    }
                ReqState st;
                st.v = v;
                st.greedy = greedy;
                st.err = err;
                st.fast = (a.fuse && fast && !err) ? 1 : 0;
                st.tok_bad = tok_bad;
                st.first_reject = v;
                const bool slow = !err && !fast;
                st.slow_base = slow ? s_u[threadIdx.x].pos : -1;
                a.req[u] = st;
                if (slow && a.lazy) {   // the histogram path takes its rows position by position
                    a.slow_req[atomicAdd(&s_nsr, 1)] = make_int2((u << 7) | (greedy << 6) | v, st.slow_base);
                    for (int j = 0; j <= v; ++j) {
                        a.pair_done[(size_t)u * (K + 1) + j] = 0;
                        if (greedy)
                            atomicAdd(&s_posg[max(0, j - kGreedyAhead)], 1);
                        else
                            atomicAdd(&s_pos[j], j < v ? kinds : 1);
                    }
                }
                a.req_done[u] = 0;
                if (err && a.accept_len) {   // no rows were listed: the outputs of a failed request
                    const int width = K + 1;
                    for (int j = 0; j < width; ++j) {
                        a.out_tokens[(size_t)u * width + j] = -1;
                        if (a.row_status) a.row_status[(size_t)u * width + j] = j == 0 ? err : 0;
                    }
                    a.accept_len[u] = 0;
                    a.num_emitted[u] = 0;
                }
            }
        }
        base_fast += s_tot_a;
        base_slow += s_tot_b;
        __syncthreads();
    }
    if (a.lazy) {
        // The histogram rows of chain verification in position order (all
        // requests' rows of position 0, then of position 1, ...), target row
        // before draft row, greedy requests' rows kGreedyAhead positions
        // early (after the sampling rows of the position they join); the
        // order among requests is immaterial.
        const int K1 = K + 1, nsr = s_nsr;
        if (threadIdx.x == 0) {
            int run = 0;
            for (int j = 0; j < K1; ++j) {
                const int cs = s_pos[j], cg = s_posg[j];
                s_pos[j] = run;
                s_posg[j] = run + cs;
                run += cs + cg;
            }
            a.counters->n_units = run;
            a.counters->n_slow_req = nsr;
        }
        __syncthreads();
        // rows that fit in one wave of the histogram kernel are taken one per
        // CTA in task order: no list
        const int n_list = a.counters->n_units > a.lazy_grid ? nsr : 0;
        for (int i = threadIdx.x; i < n_list; i += kPrepThreads) {
            const int2 e = a.slow_req[i];
            const int r = e.x >> 7, v = e.x & 63;
            const int kr = ((e.x >> 6) & 1) ? 1 : kinds;
            const bool g = ((e.x >> 6) & 1) != 0;
            for (int j = 0; j <= v; ++j) {
                const int nk = j < v ? kr : 1;
                const int at = g ? atomicAdd(&s_posg[max(0, j - kGreedyAhead)], nk) : atomicAdd(&s_pos[j], nk);
                a.slow_units[at] = make_int2((r << 7) | (j << 1), e.y + j);
                if (nk == 2) a.slow_units[at + 1] = make_int2((r << 7) | (j << 1) | 1, e.y + v + 1 + j);
            }
        }
    }
    if (threadIdx.x == 0) {
        if (!a.lazy) a.counters->n_units = 0;
        a.counters->n_fast = base_fast;
        a.counters->n_slow = base_slow;
        a.counters->n_jobs = 0;
        a.counters->timeout = 0;
        a.counters->n_ovf = 0;
        a.counters->n_jobs2 = 0;
        a.counters->next_slow = 0;
    }
}

constexpr int kChainWarps = 8;

// One warp per request (sv_walk.cuh), for the requests the row kernel did not
// chain itself (rows of the histogram path, block verification off).
__global__ void __launch_bounds__(kChainWarps * 32) chain_kernel(const __grid_constant__ ChainArgs a)
{
    pdl_enter();
    __shared__ double s_qp[kChainWarps][kFastK];
    __shared__ int s_qi[kChainWarps][kFastK];
    const int warp = threadIdx.x >> 5;
    const int r = blockIdx.x * kChainWarps + warp;
    if (r >= a.n_req) return;
    if (a.req[r].fast) return;   // chained by the one-pass row kernel
    chain_walk(a, r, s_qp[warp], s_qi[warp], true);
}

// ----------------------------------------------------------------------------
// Block verification (local-inference-lab/rtx6kpro dspark-upstream-
// consolidation.md, rejection_sample_method "block": joint block acceptance
// with residual-mass reweighting; the steps of Sun et al., "Block Verification
// Accelerates Speculative Decoding", 2024).  One warp per request, kept sets
// listed (<= 32 tokens per row):
//   w_0 = 1, w_j = min(w_{j-1} p_{j-1}(d_{j-1}) / q_{j-1}(d_{j-1}), 1)   (lane 0, in order)
//   H_j = sum over p_j's kept tokens x of max(w_j p_j(x) - q_j(x), 0)   (a warp sum)
//   h_j = H_j / (H_j + 1 - w_j) (1 if the denominator is 0), h_v = w_v
//   accept length a = the largest j in 1..v with u(r, j-1, 0) < h_j, else 0
//   next token: inverse CDF of max(w_a p_a - q_a, 0) (a < v) or p_v, u(r, a, 1).
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(kChainWarps * 32) block_kernel(const __grid_constant__ ChainArgs a)
{
    pdl_enter();
    __shared__ double s_qp[kChainWarps][kFastK];
    __shared__ int s_qi[kChainWarps][kFastK];
    __shared__ double s_wgt[kChainWarps][kMaxK + 2];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = blockIdx.x * kChainWarps + warp;
    if (r >= a.n_req) return;
    const int K = a.K, width = K + 1;
    const ReqState st = a.req[r];
    const int v = st.v;
    int32_t* out = a.out_tokens + (size_t)r * width;
    const int32_t* d = a.draft_tokens + (size_t)r * K;
    const int timed_out = a.counters->timeout ? kTimeout : 0;

    // position status; every drafted position's ratio enters the weights
    int any_err = st.err | timed_out;
    unsigned long long qzero = 0ull, rejects = 0ull;
    bool unlisted = false;
    for (int j = lane; j <= K; j += 32) {
        const RowInfo& T = a.info[slot_target(r, K, j)];
        const int t_status = T.desc.status, t_argmax = T.desc.argmax, t_list = T.n_list;
        int q_status = 0, q_list = 0;
        double q = 0.0;
        if (j < K) {
            const RowInfo& Q = draft_info(a, r, j);
            q_status = Q.desc.status;
            q = Q.p_token;
            q_list = Q.n_list;
        }
        const int dj = j < K ? d[j] : -1;
        int ps = 0;
        if (!st.err && j <= v) {
            ps |= t_status;
            if (j < v && ((st.tok_bad >> j) & 1)) ps |= kBadToken;
            if (st.greedy) {
                if (j < v && dj != t_argmax) rejects |= 1ull << j;
            } else {
                if (t_list < 0) unlisted = true;
                if (j < v) {
                    ps |= q_status;
                    if (q_list < 0) unlisted = true;
                    if (!(q > 0.0)) qzero |= 1ull << j;
                }
            }
        }
        if (j == 0) ps |= st.err | timed_out;
        any_err |= ps & kErrorMask;
        if (a.row_status) a.row_status[(size_t)r * width + j] = ps;
        out[j] = -1;
    }
    any_err = __reduce_or_sync(0xFFFFFFFFu, any_err);
    unlisted = __any_sync(0xFFFFFFFFu, unlisted);
    rejects |= ((unsigned long long)__reduce_or_sync(0xFFFFFFFFu, (unsigned)rejects)) |
               ((unsigned long long)__reduce_or_sync(0xFFFFFFFFu, (unsigned)(rejects >> 32)) << 32);
    qzero |= ((unsigned long long)__reduce_or_sync(0xFFFFFFFFu, (unsigned)qzero)) |
             ((unsigned long long)__reduce_or_sync(0xFFFFFFFFu, (unsigned)(qzero >> 32)) << 32);
    if (a.blk_h && lane == 0) a.blk_h[(size_t)r * width] = 0ull;   // not waiting for full-row sums
    if (!any_err && !st.greedy && unlisted) {
        // Kept sets too large to list: the weights here, the residual masses
        // H_j (positions 1 .. v-1) as full-row sum jobs of the resample
        // kernel, the decision in block_finish_kernel.  With v <= 1 no H_j is
        // needed: decide now and list the draw.
        if (lane == 0) {
            double w = 1.0;
            a.blk_w[(size_t)r * width] = 1.0;
            for (int j = 1; j <= v; ++j) {
                const double p = a.info[slot_target(r, K, j - 1)].p_token;
                const double q = draft_info(a, r, j - 1).p_token;
                const double ratio = q > 0.0 ? p / q : (p > 0.0 ? INFINITY : 0.0);
                const double x = w > 0.0 ? w * ratio : 0.0;
                w = x < 1.0 ? x : 1.0;
                a.blk_w[(size_t)r * width + j] = w;
            }
            if (a.row_status)
                for (int j = 0; j < v; ++j)
                    if ((qzero >> j) & 1) a.row_status[(size_t)r * width + j] |= kQZero;
        }
        __syncwarp();
        if (v >= 2) {
            for (int j = 1 + lane; j < v; j += 32) {
                ResampleJob job;
                job.req = r;
                job.a = j;
                job.residual = 1;
                job.done = 0;
                job.kind = kJobSum;
                job.pad = 0;
                job.wfix = weight_fix(a.blk_w[(size_t)r * width + j]);
                a.jobs[atomicAdd(&a.counters->n_jobs, 1)] = job;
            }
            if (lane == 0) a.blk_h[(size_t)r * width] = 1ull;   // decided by block_finish_kernel
        } else if (lane == 0) {
            const double wv = a.blk_w[(size_t)r * width + v];
            const int acc = (v == 1 && uniform_f64(a.seed, (uint32_t)r, 0u, 0u) < wv) ? 1 : 0;
            if (acc) out[0] = d[0];
            a.accept_len[r] = acc;
            a.num_emitted[r] = acc + 1;
            ResampleJob job;
            job.req = r;
            job.a = acc;
            job.residual = acc < v ? 1 : 0;
            job.done = 0;
            job.kind = kJobDraw;
            job.pad = 0;
            job.wfix = acc < v ? weight_fix(a.blk_w[(size_t)r * width + acc]) : 0ull;
            a.jobs[atomicAdd(&a.counters->n_jobs, 1)] = job;
        }
        return;
    }
    if (any_err) {
        if (lane == 0) {
            a.accept_len[r] = 0;
            a.num_emitted[r] = 0;
        }
        return;
    }

    int acc_len, t = -1, extra_bits = 0;
    if (st.greedy) {
        acc_len = rejects ? (__ffsll((long long)rejects) - 1) : v;
        t = a.info[slot_target(r, K, acc_len)].desc.argmax;
    } else {
        // weights, in order (lane 0)
        if (lane == 0) {
            double w = 1.0;
            s_wgt[warp][0] = 1.0;
            for (int j = 1; j <= v; ++j) {
                const double p = a.info[slot_target(r, K, j - 1)].p_token;
                const double q = draft_info(a, r, j - 1).p_token;
                const double ratio = q > 0.0 ? p / q : (p > 0.0 ? INFINITY : 0.0);
                const double x = w > 0.0 ? w * ratio : 0.0;
                w = x < 1.0 ? x : 1.0;
                s_wgt[warp][j] = w;
            }
        }
        __syncwarp();
        // stopping probabilities for positions 1..v: one position at a time,
        // a kept token of p_j per lane (q_j's list staged for a binary search)
        unsigned long long stop = 0ull;
        for (int j = 1; j <= v; ++j) {
            const double wj = s_wgt[warp][j];
            double h = wj;
            if (j < v) {
                const RowInfo& Pj = a.info[slot_target(r, K, j)];
                const RowInfo& Qj = draft_info(a, r, j);
                const int np = Pj.n_list, nq = Qj.n_list;
                const bool in = lane < np;
                const int x = in ? Pj.list_idx[lane] : 0;
                const double px = in ? Pj.list_p[lane] : 0.0;
                __syncwarp();
                if (lane < nq) {
                    s_qi[warp][lane] = Qj.list_idx[lane];
                    s_qp[warp][lane] = Qj.list_p[lane];
                }
                __syncwarp();
                double qx = 0.0;
                if (in) {
                    int lo = 0, hi = nq;
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        if (s_qi[warp][mid] < x) lo = mid + 1; else hi = mid;
                    }
                    if (lo < nq && s_qi[warp][lo] == x) qx = s_qp[warp][lo];
                }
                const double m = in ? wj * px - qx : 0.0;
                double H = m > 0.0 ? m : 0.0;
#pragma unroll
                for (int o = 16; o; o >>= 1) H += __shfl_xor_sync(0xFFFFFFFFu, H, o);
                const double den = H + 1.0 - wj;
                h = den > 0.0 ? H / den : 1.0;
            }
            if (uniform_f64(a.seed, (uint32_t)r, (uint32_t)(j - 1), 0u) < h) stop |= 1ull << j;
        }
        acc_len = stop ? 63 - __clzll((long long)stop) : 0;
        __syncwarp();

        // the next token, one listed token per lane
        const bool residual = acc_len < v;
        const RowInfo& P = a.info[slot_target(r, K, acc_len)];
        const int np = P.n_list;
        const bool in = lane < np;
        const int x = in ? P.list_idx[lane] : 0;
        const double px = in ? P.list_p[lane] : 0.0;
        double w = px;
        if (residual) {
            const RowInfo& Q = draft_info(a, r, acc_len);
            const int nq = Q.n_list;
            if (lane < nq) {
                s_qi[warp][lane] = Q.list_idx[lane];
                s_qp[warp][lane] = Q.list_p[lane];
            }
            __syncwarp();
            double qx = 0.0;
            if (in) {
                int lo = 0, hi = nq;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (s_qi[warp][mid] < x) lo = mid + 1; else hi = mid;
                }
                if (lo < nq && s_qi[warp][lo] == x) qx = s_qp[warp][lo];
            }
            const double rw = s_wgt[warp][acc_len] * px - qx;
            w = (in && rw > 0.0) ? rw : 0.0;
        }
        double cum = warp_scan_f64(w);
        double W = __shfl_sync(0xFFFFFFFFu, cum, 31);
        if (residual && !(W > 0.0)) {
            extra_bits = kResidZero;
            w = px;
            cum = warp_scan_f64(w);
            W = __shfl_sync(0xFFFFFFFFu, cum, 31);
        }
        const double target = uniform_f64(a.seed, (uint32_t)r, (uint32_t)acc_len, 1u) * W;
        const unsigned over = __ballot_sync(0xFFFFFFFFu, in && cum > target);
        if (over) {
            t = __shfl_sync(0xFFFFFFFFu, x, __ffs(over) - 1);
        } else {
            const unsigned pos = __ballot_sync(0xFFFFFFFFu, in && w > 0.0);
            t = pos ? __shfl_sync(0xFFFFFFFFu, x, 31 - __clz(pos)) : -1;
        }
    }
    for (int j = lane; j < acc_len; j += 32) out[j] = d[j];
    if (lane == 0) {
        out[acc_len] = t;
        a.accept_len[r] = acc_len;
        a.num_emitted[r] = acc_len + 1;
        if (a.row_status) {
            for (int j = 0; j < v; ++j)
                if ((qzero >> j) & 1) a.row_status[(size_t)r * width + j] |= kQZero;
            if (extra_bits) a.row_status[(size_t)r * width + acc_len] |= extra_bits;
        }
    }
}

// ----------------------------------------------------------------------------
// Block verification of requests whose kept sets are not listed: with the
// residual sums H_j of positions 1 .. v-1 in hand (the resample kernel's sum
// jobs), the stopping probabilities, the accepted length, and the job that
// draws the emitted token (max(w_a p_a - q_a, 0), or p_v after full
// acceptance).  One warp per request.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(kChainWarps * 32) block_finish_kernel(const __grid_constant__ ChainArgs a)
{
    pdl_enter();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = blockIdx.x * kChainWarps + warp;
    if (r >= a.n_req) return;
    const int K = a.K, width = K + 1;
    if (a.blk_h[(size_t)r * width] == 0ull) return;   // decided in block_kernel
    const int v = a.req[r].v;
    int32_t* out = a.out_tokens + (size_t)r * width;
    const int32_t* d = a.draft_tokens + (size_t)r * K;
    unsigned long long stop = 0ull;
    for (int j = 1 + lane; j <= v; j += 32) {
        const double wj = a.blk_w[(size_t)r * width + j];
        double h = wj;
        if (j < v) {
            const double H = (double)a.blk_h[(size_t)r * width + j] * 0x1p-62;
            const double den = H + 1.0 - wj;
            h = den > 0.0 ? H / den : 1.0;
        }
        if (uniform_f64(a.seed, (uint32_t)r, (uint32_t)(j - 1), 0u) < h) stop |= 1ull << j;
    }
    stop = ((unsigned long long)__reduce_or_sync(0xFFFFFFFFu, (unsigned)stop)) |
           ((unsigned long long)__reduce_or_sync(0xFFFFFFFFu, (unsigned)(stop >> 32)) << 32);
    const int acc = stop ? 63 - __clzll((long long)stop) : 0;
    for (int j = lane; j < acc; j += 32) out[j] = d[j];
    if (lane == 0) {
        a.accept_len[r] = acc;
        a.num_emitted[r] = acc + 1;
        ResampleJob job;
        job.req = r;
        job.a = acc;
        job.residual = acc < v ? 1 : 0;
        job.done = 0;
        job.kind = kJobDraw;
        job.pad = 0;
        job.wfix = acc < v ? weight_fix(a.blk_w[(size_t)r * width + acc]) : 0ull;
        a.jobs[a.counters->n_jobs + atomicAdd(&a.counters->n_jobs2, 1)] = job;
    }
}

// ----------------------------------------------------------------------------
// sv_build_target_probs outputs
// ----------------------------------------------------------------------------
__global__ void rows_out_kernel(ChainArgs a, float* prob_of_token, sv_row_desc_t* desc)
{
    pdl_enter();
    const int rows = a.n_req;
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) {
        const RowInfo& I = a.info[r];
        if (desc) {
            sv_row_desc_t d = I.desc;
            if (a.counters->timeout) d.status |= kTimeout;
            desc[r] = d;
        }
        if (prob_of_token) prob_of_token[r] = (float)I.p_token;
    }
}

// Dense p of every row, in fp64 then rounded to fp32 (a test aid): one CTA
// per row, tiles of blockDim elements in index order for the tie ranks.
__global__ void __launch_bounds__(1024) dense_kernel(ChainArgs a, float* dense)
{
    pdl_enter();
    __shared__ int s_w[32];
    const int row = blockIdx.x;
    const RowInfo& I = a.info[row];
    const int V = a.vocab;
    float* out = dense + (size_t)row * V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (I.desc.status & kErrorMask) {
        for (int x = tid; x < V; x += blockDim.x) out[x] = 0.0f;
        return;
    }
    if (I.n_list >= 0) {
        for (int x = tid; x < V; x += blockDim.x) out[x] = 0.0f;
        __syncthreads();
        if (tid < I.n_list) out[I.list_idx[tid]] = (float)I.list_p[tid];
        return;
    }
    const double m = I.desc.max_logit, T = I.desc.temperature, z = I.z;
    const float cut = I.desc.cutoff_logit;
    const int ties = I.desc.cutoff_ties;
    const char* base = (const char*)a.tgt + (size_t)row * (size_t)a.stride_t * (a.dtype == 0 ? 2 : 4);
    int run = 0;
    for (int x0 = 0; x0 < V; x0 += blockDim.x) {
        const int x = x0 + tid;
        float l = -INFINITY;
        if (x < V) l = a.dtype == 0 ? load_logit<0>(base, x) : load_logit<1>(base, x);
        const int is_tie = (x < V && l == cut) ? 1 : 0;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, is_tie);
        if (lane == 0) s_w[warp] = __popc(bal);
        __syncthreads();
        int before = run;
        for (int w = 0; w < warp; ++w) before += s_w[w];
        before += __popc(bal & ((1u << lane) - 1u));
        int tot = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_w[w];
        __syncthreads();
        run += tot;
        if (x < V) {
            const bool keep = l > cut || (is_tie && before < ties);
            out[x] = keep ? (float)(exp(((double)l - m) / T) / z) : 0.0f;
        }
    }
}

}  // namespace

cudaError_t launch_prep(const ChainArgs& a, cudaStream_t s)
{
    return launch_pdl(prep_kernel, dim3(1), dim3(kPrepThreads), 0, s, a);
}

cudaError_t launch_chain(const ChainArgs& a, cudaStream_t s)
{
    const int grid = (a.n_req + kChainWarps - 1) / kChainWarps;
    if (a.block) return launch_pdl(block_kernel, dim3(grid), dim3(kChainWarps * 32), 0, s, a);
    return launch_pdl(chain_kernel, dim3(grid), dim3(kChainWarps * 32), 0, s, a);
}

cudaError_t launch_block_finish(const ChainArgs& a, cudaStream_t s)
{
    const int grid = (a.n_req + kChainWarps - 1) / kChainWarps;
    return launch_pdl(block_finish_kernel, dim3(grid), dim3(kChainWarps * 32), 0, s, a);
}

cudaError_t launch_rows_out(const ChainArgs& a, float* prob_of_token, sv_row_desc_t* desc, float* dense,
                            cudaStream_t s)
{
    int grid = (a.n_req + 255) / 256;
    if (grid < 1) grid = 1;
    cudaError_t err = launch_pdl(rows_out_kernel, dim3(grid), dim3(256), 0, s, a, prob_of_token, desc);
    if (err != cudaSuccess || !dense) return err;
    return launch_pdl(dense_kernel, dim3(a.n_req), dim3(1024), 0, s, a, dense);
}

}  // namespace sv
