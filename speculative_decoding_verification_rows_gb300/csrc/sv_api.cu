// sv_api.cu -- the C ABI of libsv (declared in include/sv.h): argument checks,
// workspace carving and the launch sequence of each entry point.
#include <stdint.h>

#include "sv_internal.cuh"

using namespace sv;

namespace {

constexpr int kMaxVocab = kMaxCluster * kHistMaxSlice;   // 524,280: one cluster per row
constexpr int kPlanMaxK = 4094;
constexpr int kPlanMaxN = (1 << 20) - 1;

int sm_count()
{
    static int cached[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 1;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
        cached[dev] = n;
    }
    return cached[dev];
}

bool ws_ok(const void* ws, size_t bytes, size_t need)
{
    return ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0u && bytes >= need;
}

template <typename T>
T* at(void* ws, size_t off)
{
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// The three arrays of a task list carved at `off` (each 16-byte aligned).
TaskList task_list(void* ws, size_t off, int n)
{
    TaskList L;
    L.row = at<int64_t>(ws, off);
    L.meta = at<int4>(ws, off + sizeof(int64_t) * (size_t)n + (n & 1 ? 8 : 0));
    L.samp = reinterpret_cast<float4*>(L.meta + n);
    return L;
}

sv_status_t to_status(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;   // sv_set_timing_events
cudaEvent_t g_hv_start = nullptr, g_hv_stop = nullptr;   // sv_set_hist_timing_events

// Row kernels for whatever tasks the prep kernel listed (the one-pass kernel
// also finalises its rows).  `small_topk`: the caller promised that no row
// needs the histogram path (prep refuses any that would).
sv_status_t run_rows(const RowsArgs& ra, cudaStream_t s, bool small_topk)
{
    const cudaEvent_t ev0 = g_ev_start, ev1 = g_ev_stop;
    if (ev0 && ev1 && cudaEventRecord(ev0, s) != cudaSuccess) return SV_ERR_CUDA;
    cudaError_t e = launch_fast_rows(ra, s);
    if (e != cudaSuccess) return SV_ERR_CUDA;
    if (ev0 && ev1 && cudaEventRecord(ev1, s) != cudaSuccess) return SV_ERR_CUDA;
    if (!small_topk) {   // rows whose kept sets are not listed: bf16 by exact histograms, fp32 by radix descent
        const cudaEvent_t hv0 = g_hv_start, hv1 = g_hv_stop;
        if (hv0 && hv1 && cudaEventRecord(hv0, s) != cudaSuccess) return SV_ERR_CUDA;
        e = ra.dtype == 0 ? launch_hist_rows(ra, s) : launch_rows32(ra, s);
        if (e != cudaSuccess) return SV_ERR_CUDA;
        if (hv0 && hv1 && cudaEventRecord(hv1, s) != cudaSuccess) return SV_ERR_CUDA;
    }
    return SV_OK;
}

struct Carved {
    RowsArgs ra;
    ChainArgs ca;
};

Carved carve(void* ws, int n_req, int k_max, int vocab, int dtype, const void* tgt, const void* drf,
             int64_t stride_t, int64_t stride_d, int block = 0)
{
    const WsLayout L = ws_layout(n_req, k_max, vocab, block);
    Carved c{};
    RowsArgs& ra = c.ra;
    ra.tgt = tgt;
    ra.drf = drf;
    ra.stride_t = stride_t;
    ra.stride_d = stride_d;
    ra.vocab = vocab;
    ra.dtype = dtype;
    ra.fast_tasks = task_list(ws, L.fast_tasks, L.max_tasks);
    ra.slow_tasks = task_list(ws, L.slow_tasks, L.max_tasks);
    ra.counters = at<Counters>(ws, L.counters);
    ra.info = at<RowInfo>(ws, L.info);
    ra.partials = at<Partial>(ws, L.partials);
    ra.row_sync = at<RowSync>(ws, L.row_sync);
    ra.ovf_idx = at<int32_t>(ws, L.ovf);
    ra.max_tasks = L.max_tasks;
    ra.num_sms = sm_count();
    ChainArgs& ca = c.ca;
    ca.n_req = n_req;
    ca.n_params = n_req;
    ca.rows_per_req = 1;
    ca.K = k_max;
    ca.vocab = vocab;
    ca.dtype = dtype;
    ca.tgt = tgt;
    ca.drf = drf;
    ca.stride_t = stride_t;
    ca.stride_d = stride_d;
    ca.counters = ra.counters;
    ca.fast_tasks = ra.fast_tasks;
    ca.slow_tasks = ra.slow_tasks;
    ca.row_sync = ra.row_sync;
    ca.info = ra.info;
    ca.req = at<ReqState>(ws, L.req);
    ca.req_done = at<int32_t>(ws, L.req_done);
    ca.pair_done = at<int32_t>(ws, L.pair_done);
    ca.slow_req = at<int2>(ws, L.slow_req);
    ca.slow_units = at<int2>(ws, L.slow_units);
    ca.jobs = at<ResampleJob>(ws, L.jobs);
    ca.tiles = at<TileSums>(ws, L.tiles);
    ca.blk_w = block ? at<double>(ws, L.blk) : nullptr;
    ca.blk_h = block ? at<unsigned long long>(ws, L.blk + sizeof(double) * (size_t)n_req * (size_t)(k_max + 1)) : nullptr;
    ca.num_sms = ra.num_sms;
    return c;
}

bool dtype_ok(sv_dtype_t dt) { return dt == SV_DTYPE_BF16 || dt == SV_DTYPE_F32; }

sv_status_t run_verify(int layout, const void* tgt, const void* drf, sv_dtype_t dt, int n, int K, int V, int bucket,
                       const int32_t* qo, const int32_t* vl, const int32_t* toks, sv_sampling_t sp, uint64_t seed,
                       int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted, int32_t* row_status, void* ws,
                       size_t ws_bytes, cudaStream_t s, int block = 0, const RowInfo* q_rows = nullptr)
{
    if (!tgt || n < 1 || K < 0 || V < 1 || !sp.temperature || !accept_len || !out_tokens || !num_emitted)
        return SV_ERR_INVALID_ARG;
    if (K > 0 && !toks) return SV_ERR_INVALID_ARG;
    if (!dtype_ok(dt)) return SV_ERR_INVALID_ARG;
    if (layout == 1 && (!qo || !vl || bucket < 1)) return SV_ERR_INVALID_ARG;
    if (K > kMaxK || V > kMaxVocab || n > (1 << 22)) return SV_ERR_UNSUPPORTED;
    const size_t need = block ? sv_workspace_size_block(n, K, V) : sv_workspace_size(n, K, V);
    if (need == 0) return SV_ERR_UNSUPPORTED;
    if (!ws_ok(ws, ws_bytes, need)) return SV_ERR_WORKSPACE;
    Carved c = carve(ws, n, K, V, (int)dt, tgt, drf, V, V, block);
    ChainArgs& ca = c.ca;
    ca.layout = layout;
    ca.block = block;
    ca.bucket = bucket;
    ca.qo_indptr = qo;
    ca.verify_len = vl;
    ca.draft_tokens = toks;
    ca.sp = sp;
    ca.seed = seed;
    ca.accept_len = accept_len;
    ca.out_tokens = out_tokens;
    ca.num_emitted = num_emitted;
    ca.row_status = row_status;
    ca.q_rows = q_rows;
    // The one-pass row kernel runs the chain of every request whose rows it
    // takes (greedy and top-k <= 32); the chain kernel takes the others
    // (block verification: every request).  Under the small-top-k promise
    // every request is of the first kind and every kept set is listed, so
    // neither the chain kernel nor the full-row resample has work.
    const bool small_topk = (sp.flags & SV_SAMPLING_SMALL_TOPK) != 0;
    ca.fuse = block ? 0 : 1;
    ca.lazy = block ? 0 : 1;   // chain verify: rows past a known rejection need only their status
    ca.lazy_grid = ca.lazy ? hist_wide_grid(ca.num_sms) : 0;
    if (ca.lazy && ca.lazy_grid < 1) return SV_ERR_CUDA;
    c.ra.chain = ca;
    if (launch_prep(ca, s) != cudaSuccess) return SV_ERR_CUDA;
    sv_status_t st = run_rows(c.ra, s, small_topk);
    if (st != SV_OK) return st;
    if (small_topk && !block) return SV_OK;
    if (launch_chain(ca, s) != cudaSuccess) return SV_ERR_CUDA;
    if (small_topk) return SV_OK;
    auto resample = [&](int wave) {
        return dt == SV_DTYPE_BF16 ? launch_resample(ca, wave, s) : launch_resample32(ca, wave, s);
    };
    if (resample(0) != cudaSuccess) return SV_ERR_CUDA;
    if (block) {   // requests with unlisted kept sets: decide, then draw
        if (launch_block_finish(ca, s) != cudaSuccess) return SV_ERR_CUDA;
        if (resample(1) != cudaSuccess) return SV_ERR_CUDA;
    }
    return SV_OK;
}

}  // namespace

extern "C" {

size_t sv_workspace_size_block(int n_req, int k_max, int vocab)
{
    if (n_req < 1 || k_max < 0 || vocab < 1 || n_req > (1 << 22) || k_max > kMaxK || vocab > kMaxVocab) return 0;
    if ((long long)n_req * (2LL * k_max + 1) > (1LL << 30)) return 0;
    return ws_layout(n_req, k_max, vocab, 1).total;
}

size_t sv_workspace_size(int n_req, int k_max, int vocab)
{
    if (n_req < 0 || k_max < 0 || vocab < 0) return 0;
    if (vocab == 0) {   // the planner: its rank keys only
        if (n_req > kPlanMaxN || k_max > kPlanMaxK) return 0;
        return align256(sizeof(unsigned long long) * (size_t)n_req * (size_t)(k_max > 0 ? k_max : 1));
    }
    if (n_req > (1 << 22) || k_max > kMaxK || vocab > kMaxVocab) return 0;
    if ((long long)n_req * (2LL * k_max + 1) > (1LL << 30)) return 0;
    return ws_layout(n_req, k_max, vocab).total;
}

const char* sv_status_string(sv_status_t status)
{
    switch (status) {
        case SV_OK: return "SV_OK";
        case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG";
        case SV_ERR_WORKSPACE: return "SV_ERR_WORKSPACE";
        case SV_ERR_CUDA: return "SV_ERR_CUDA";
        case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED";
    }
    return "SV_ERR_UNKNOWN";
}

sv_status_t sv_plan_budget(const float* conf, int ld_conf, const int32_t* draft_len, int n_req, int K,
                           int budget_tokens, int bucket_tokens, int32_t* verify_lens, int32_t* qo_indptr,
                           int32_t* total_tokens, int32_t* status, void* ws, size_t ws_bytes, sv_stream_t stream)
{
    if (n_req < 1 || K < 0 || ld_conf < K || budget_tokens < n_req || bucket_tokens < budget_tokens)
        return SV_ERR_INVALID_ARG;
    if ((K > 0 && !conf) || !verify_lens || !qo_indptr || !total_tokens) return SV_ERR_INVALID_ARG;
    if (K > kPlanMaxK || n_req > kPlanMaxN) return SV_ERR_UNSUPPORTED;
    const size_t need = sv_workspace_size(n_req, K, 0);
    if (need == 0) return SV_ERR_UNSUPPORTED;
    if (!ws_ok(ws, ws_bytes, need)) return SV_ERR_WORKSPACE;
    return to_status(launch_plan(conf, ld_conf, draft_len, n_req, K, budget_tokens, nullptr, verify_lens, qo_indptr,
                                 total_tokens, status, static_cast<unsigned long long*>(ws), stream));
}

sv_status_t sv_plan_budget_cost(const float* conf, int ld_conf, const int32_t* draft_len, int n_req, int K,
                                const int32_t* cost_tokens, const float* cost_ms, int n_cost, float fixed_overhead_ms,
                                const int32_t* batch_sizes, const float* batch_overhead_ms, int n_batch,
                                int bucket_tokens, int32_t* budget_out, int32_t* budget_status, int32_t* verify_lens,
                                int32_t* qo_indptr, int32_t* total_tokens, int32_t* status, void* ws, size_t ws_bytes,
                                sv_stream_t stream)
{
    if (n_req < 1 || K < 0 || ld_conf < K || bucket_tokens < n_req || n_cost < 0 || n_batch < 0)
        return SV_ERR_INVALID_ARG;
    if ((K > 0 && !conf) || !verify_lens || !qo_indptr || !total_tokens || !budget_out) return SV_ERR_INVALID_ARG;
    if ((n_cost > 0 && (!cost_tokens || !cost_ms)) || (n_batch > 0 && (!batch_sizes || !batch_overhead_ms)))
        return SV_ERR_INVALID_ARG;
    if ((long long)n_req * K > kBudgetMaxCand || n_cost > kBudgetMaxShelves || n_batch > kBudgetMaxShelves)
        return SV_ERR_UNSUPPORTED;
    const size_t need = sv_workspace_size(n_req, K, 0);
    if (need == 0) return SV_ERR_UNSUPPORTED;
    if (!ws_ok(ws, ws_bytes, need)) return SV_ERR_WORKSPACE;
    cudaError_t e = launch_budget(conf, ld_conf, draft_len, n_req, K, cost_tokens, cost_ms, n_cost, fixed_overhead_ms,
                                  batch_sizes, batch_overhead_ms, n_batch, bucket_tokens, budget_out, budget_status,
                                  stream);
    if (e != cudaSuccess) return SV_ERR_CUDA;
    return to_status(launch_plan(conf, ld_conf, draft_len, n_req, K, 0, budget_out, verify_lens, qo_indptr,
                                 total_tokens, status, static_cast<unsigned long long*>(ws), stream));
}

size_t sv_estimator_state_bytes(int K)
{
    if (K < 1 || K > kMaxK) return 0;
    return sizeof(double) * (size_t)(4 * K + 5);
}

sv_status_t sv_estimator_init(double* state, int K, sv_stream_t stream)
{
    if (!state || K < 1 || K > kMaxK) return SV_ERR_INVALID_ARG;
    return to_status(launch_est_init(state, K, stream));
}

sv_status_t sv_estimator_predict(const void* draft_logits, sv_dtype_t dt, int n_req, int K, int vocab,
                                 sv_sampling_t sp, const double* state, float* x_out, float* p_out, void* ws,
                                 size_t ws_bytes, sv_stream_t stream)
{
    if (!draft_logits || n_req < 1 || K < 1 || K > kMaxK || vocab < 1 || !sp.temperature || !state || !x_out ||
        !p_out)
        return SV_ERR_INVALID_ARG;
    if (!dtype_ok(dt)) return SV_ERR_INVALID_ARG;
    if (vocab > kMaxVocab || (long long)n_req * K > (1 << 22)) return SV_ERR_UNSUPPORTED;
    const int rows = n_req * K;
    const size_t need = sv_workspace_size(rows, 0, vocab);
    if (need == 0) return SV_ERR_UNSUPPORTED;
    if (!ws_ok(ws, ws_bytes, need)) return SV_ERR_WORKSPACE;
    Carved c = carve(ws, rows, 0, vocab, (int)dt, draft_logits, nullptr, vocab, vocab);
    ChainArgs& ca = c.ca;
    ca.layout = 2;
    ca.est = 1;
    ca.rows_per_req = K;
    ca.n_params = n_req;
    ca.sp = sp;
    ca.sp.flags = 0;   // greedy requests' features are taken at T = 1 over the whole row
    c.ra.chain = ca;
    if (launch_prep(ca, stream) != cudaSuccess) return SV_ERR_CUDA;
    sv_status_t st = run_rows(c.ra, stream, false);
    if (st != SV_OK) return st;
    return to_status(launch_est_predict(c.ra.info, state, n_req, K, x_out, p_out, c.ra.counters, stream));
}

size_t sv_q_rows_bytes(int n_req, int K)
{
    if (n_req < 1 || K < 1 || K > kMaxK || (long long)n_req * K > (1 << 22)) return 0;
    return sizeof(RowInfo) * (size_t)n_req * (size_t)K;
}

sv_status_t sv_estimator_predict_q(const void* draft_logits, sv_dtype_t dt, int n_req, int K, int vocab,
                                   sv_sampling_t sp, const double* state, const int32_t* draft_tokens, float* x_out,
                                   float* p_out, void* q_rows, void* ws, size_t ws_bytes, sv_stream_t stream)
{
    if (!draft_logits || n_req < 1 || K < 1 || K > kMaxK || vocab < 1 || !sp.temperature || !state || !x_out ||
        !p_out || !draft_tokens || !q_rows)
        return SV_ERR_INVALID_ARG;
    if (!dtype_ok(dt)) return SV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q_rows) & 15u) != 0u) return SV_ERR_INVALID_ARG;
    if (vocab > kMaxVocab || (long long)n_req * K > (1 << 22)) return SV_ERR_UNSUPPORTED;
    const int rows = n_req * K;
    const size_t need = sv_workspace_size(rows, 0, vocab);
    if (need == 0) return SV_ERR_UNSUPPORTED;
    if (!ws_ok(ws, ws_bytes, need)) return SV_ERR_WORKSPACE;
    Carved c = carve(ws, rows, 0, vocab, (int)dt, draft_logits, nullptr, vocab, vocab);
    ChainArgs& ca = c.ca;
    ca.layout = 2;
    ca.est = 1;
    ca.rows_per_req = K;
    ca.n_params = n_req;
    ca.token_per_row = draft_tokens;   // row r K + j carries draft token j of request r
    ca.sp = sp;
    ca.sp.flags = 0;
    ca.info = c.ra.info = static_cast<RowInfo*>(q_rows);   // the rows' results go to the caller's buffer
    c.ra.chain = ca;
    if (launch_prep(ca, stream) != cudaSuccess) return SV_ERR_CUDA;
    sv_status_t st = run_rows(c.ra, stream, false);
    if (st != SV_OK) return st;
    return to_status(launch_est_predict(c.ra.info, state, n_req, K, x_out, p_out, c.ra.counters, stream));
}

sv_status_t sv_verify_chain_q(const void* target_logits, const void* draft_logits, sv_dtype_t dt, int n_req, int K,
                              int vocab, const int32_t* draft_tokens, const int32_t* verify_len, sv_sampling_t sp,
                              uint64_t seed, const void* q_rows, int32_t* accept_len, int32_t* out_tokens,
                              int32_t* num_emitted, int32_t* row_status, void* ws, size_t ws_bytes,
                              sv_stream_t stream)
{
    if (!q_rows || K < 1) return SV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q_rows) & 15u) != 0u) return SV_ERR_INVALID_ARG;
    return run_verify(0, target_logits, draft_logits, dt, n_req, K, vocab, 0, nullptr, verify_len, draft_tokens, sp,
                      seed, accept_len, out_tokens, num_emitted, row_status, ws, ws_bytes, stream, 0,
                      static_cast<const RowInfo*>(q_rows));
}

sv_status_t sv_estimator_observe(double* state, const float* x, const int32_t* accept_len, const int32_t* num_emitted,
                                 const int32_t* verify_lens, int n_req, int K, int refit_every, sv_stream_t stream)
{
    if (!state || !x || !accept_len || !num_emitted || n_req < 1 || K < 1 || K > kMaxK) return SV_ERR_INVALID_ARG;
    return to_status(launch_est_observe(state, x, accept_len, num_emitted, verify_lens, n_req, K, refit_every, stream));
}

sv_status_t sv_verify_stats(const int32_t* accept_len, const int32_t* num_emitted, const int32_t* verify_lens,
                            const int32_t* draft_len, int n_req, int K, int64_t* out, sv_stream_t stream)
{
    if (n_req < 1 || K < 0 || !accept_len || !num_emitted || !out) return SV_ERR_INVALID_ARG;
    return to_status(launch_stats(accept_len, num_emitted, verify_lens, draft_len, n_req, K,
                                  reinterpret_cast<long long*>(out), stream));
}

sv_status_t sv_build_target_probs(const void* logits, sv_dtype_t dt, int64_t row_stride, int rows, int vocab,
                                  const int32_t* row_to_req, int n_req, sv_sampling_t sp, const int32_t* token_per_row,
                                  float* prob_of_token, sv_row_desc_t* desc, float* dense_probs, void* ws,
                                  size_t ws_bytes, sv_stream_t stream)
{
    if (!logits || rows < 1 || vocab < 1 || row_stride < vocab || n_req < 1 || !sp.temperature)
        return SV_ERR_INVALID_ARG;
    if (!dtype_ok(dt)) return SV_ERR_INVALID_ARG;
    if (!row_to_req && n_req < rows) return SV_ERR_INVALID_ARG;
    if (vocab > kMaxVocab || rows > (1 << 22)) return SV_ERR_UNSUPPORTED;
    const size_t need = sv_workspace_size(rows, 0, vocab);
    if (need == 0) return SV_ERR_UNSUPPORTED;
    if (!ws_ok(ws, ws_bytes, need)) return SV_ERR_WORKSPACE;
    Carved c = carve(ws, rows, 0, vocab, (int)dt, logits, nullptr, row_stride, row_stride);
    ChainArgs& ca = c.ca;
    ca.layout = 2;
    ca.n_params = n_req;
    ca.row_to_req = row_to_req;
    ca.token_per_row = token_per_row;
    ca.sp = sp;
    c.ra.chain = ca;
    if (launch_prep(ca, stream) != cudaSuccess) return SV_ERR_CUDA;
    sv_status_t st = run_rows(c.ra, stream, (sp.flags & SV_SAMPLING_SMALL_TOPK) != 0);
    if (st != SV_OK) return st;
    return to_status(launch_rows_out(ca, prob_of_token, desc, dense_probs, stream));
}

sv_status_t sv_verify_chain(const void* target_logits, const void* draft_logits, sv_dtype_t dt, int n_req, int K,
                            int vocab, const int32_t* draft_tokens, const int32_t* verify_len, sv_sampling_t sp,
                            uint64_t seed, int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                            int32_t* row_status, void* ws, size_t ws_bytes, sv_stream_t stream)
{
    return run_verify(0, target_logits, draft_logits, dt, n_req, K, vocab, 0, nullptr, verify_len, draft_tokens, sp,
                      seed, accept_len, out_tokens, num_emitted, row_status, ws, ws_bytes, stream);
}

sv_status_t sv_verify_block(const void* target_logits, const void* draft_logits, sv_dtype_t dt, int n_req, int K,
                            int vocab, const int32_t* draft_tokens, const int32_t* verify_len, sv_sampling_t sp,
                            uint64_t seed, int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                            int32_t* row_status, void* ws, size_t ws_bytes, sv_stream_t stream)
{
    sp.flags = 0;   // block verification keeps its full launch sequence
    return run_verify(0, target_logits, draft_logits, dt, n_req, K, vocab, 0, nullptr, verify_len, draft_tokens, sp,
                      seed, accept_len, out_tokens, num_emitted, row_status, ws, ws_bytes, stream, 1);
}

sv_status_t sv_verify_ragged(const void* target_logits, const void* draft_logits, sv_dtype_t dt, int n_req,
                             int K_max, int vocab, int bucket_tokens, const int32_t* qo_indptr,
                             const int32_t* verify_lens, const int32_t* draft_tokens, sv_sampling_t sp,
                             uint64_t seed, int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                             int32_t* row_status, void* ws, size_t ws_bytes, sv_stream_t stream)
{
    return run_verify(1, target_logits, draft_logits, dt, n_req, K_max, vocab, bucket_tokens, qo_indptr, verify_lens,
                      draft_tokens, sp, seed, accept_len, out_tokens, num_emitted, row_status, ws, ws_bytes, stream);
}

size_t sv_shard_record_bytes(void) { return sizeof(Partial); }

sv_status_t sv_verify_chain_shard_rows(const void* target_shard, const void* draft_shard, sv_dtype_t dt, int n_req,
                                       int K, int vocab, int v0, int v1, const int32_t* draft_tokens,
                                       const int32_t* verify_len, sv_sampling_t sp, void* records, void* ws,
                                       size_t ws_bytes, sv_stream_t stream)
{
    if (!target_shard || !records || n_req < 1 || K < 0 || vocab < 1 || v0 < 0 || v1 <= v0 || v1 > vocab ||
        !sp.temperature)
        return SV_ERR_INVALID_ARG;
    if (K > 0 && !draft_tokens) return SV_ERR_INVALID_ARG;
    if (!dtype_ok(dt)) return SV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(records) & 15u) != 0u) return SV_ERR_INVALID_ARG;
    if (K > kMaxK || vocab > kMaxVocab || n_req > (1 << 22)) return SV_ERR_UNSUPPORTED;
    const int vs = v1 - v0;
    const size_t need = sv_workspace_size(n_req, K, vs);
    if (need == 0) return SV_ERR_UNSUPPORTED;
    if (!ws_ok(ws, ws_bytes, need)) return SV_ERR_WORKSPACE;
    Carved c = carve(ws, n_req, K, vs, (int)dt, target_shard, draft_shard, vs, vs);
    ChainArgs& ca = c.ca;
    ca.vocab = vocab;   // parameters and tokens refer to the whole vocabulary; the rows hold [v0, v1)
    ca.layout = 0;
    ca.shard = 1;
    ca.verify_len = verify_len;
    ca.draft_tokens = draft_tokens;
    ca.sp = sp;
    c.ra.chain = ca;
    c.ra.shard_out = static_cast<Partial*>(records);
    c.ra.shard_v0 = (uint32_t)v0;
    if (launch_prep(ca, stream) != cudaSuccess) return SV_ERR_CUDA;
    return to_status(launch_fast_rows(c.ra, stream));
}

sv_status_t sv_verify_chain_shard_merge(const void* records, int n_shards, int n_req, int K, int vocab,
                                        const int32_t* draft_tokens, const int32_t* verify_len, sv_sampling_t sp,
                                        uint64_t seed, int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                                        int32_t* row_status, void* ws, size_t ws_bytes, sv_stream_t stream)
{
    if (!records || n_shards < 1 || n_req < 1 || K < 0 || vocab < 1 || !sp.temperature || !accept_len ||
        !out_tokens || !num_emitted)
        return SV_ERR_INVALID_ARG;
    if (K > 0 && !draft_tokens) return SV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(records) & 15u) != 0u) return SV_ERR_INVALID_ARG;
    if (K > kMaxK || vocab > kMaxVocab || n_req > (1 << 22) || n_shards > 1024) return SV_ERR_UNSUPPORTED;
    const size_t need = sv_workspace_size(n_req, K, 1);
    if (need == 0) return SV_ERR_UNSUPPORTED;
    if (!ws_ok(ws, ws_bytes, need)) return SV_ERR_WORKSPACE;
    Carved c = carve(ws, n_req, K, 1, (int)SV_DTYPE_BF16, nullptr, nullptr, 1, 1);
    ChainArgs& ca = c.ca;
    ca.vocab = vocab;
    ca.layout = 0;
    ca.shard = 2;
    ca.verify_len = verify_len;
    ca.draft_tokens = draft_tokens;
    ca.sp = sp;
    ca.seed = seed;
    ca.accept_len = accept_len;
    ca.out_tokens = out_tokens;
    ca.num_emitted = num_emitted;
    ca.row_status = row_status;
    c.ra.chain = ca;
    if (launch_prep(ca, stream) != cudaSuccess) return SV_ERR_CUDA;
    if (launch_shard_merge(c.ra, records, n_shards, n_req * (2 * K + 1), stream) != cudaSuccess) return SV_ERR_CUDA;
    return to_status(launch_chain(ca, stream));
}

sv_status_t sv_set_timing_events(void* start_event, void* stop_event)
{
    g_ev_start = static_cast<cudaEvent_t>(start_event);
    g_ev_stop = static_cast<cudaEvent_t>(stop_event);
    return SV_OK;
}

sv_status_t sv_set_hist_timing_events(void* start_event, void* stop_event)
{
    g_hv_start = static_cast<cudaEvent_t>(start_event);
    g_hv_stop = static_cast<cudaEvent_t>(stop_event);
    return SV_OK;
}

}  // extern "C"
