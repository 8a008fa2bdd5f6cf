// sv_hist.cu -- exact per-value histogram kernels for sampling rows whose
// kept set can be large (top-k off or above 32, with or without top-p).
//
// The target distribution of jianc99/sglang PR #8 ("build_speculative_verify_
// target_probs") needs, for top-p, the mass-ordered cutoff over the whole
// vocabulary.  A bf16 logit takes one of 65,536 values, so the row's multiset
// of values is its histogram over the 16-bit order key, and every quantity of
// the transform follows from it exactly: the mass of a value is its count
// times exp((v - m) / T), computed once per distinct value in fp64.
//
// Two kernels share the cutoff walk:
//
// * wide_rows_kernel (every row first): one CTA per row, several rows in
//   flight per SM.  The row is streamed once with 16-byte loads; each key is
//   counted in a 32-bit shared-memory counter of its binade (the 128 keys of
//   one sign + exponent), and a binade gets its 128 counters the first time
//   one of its keys is seen.  Rows of ordinary logits occupy a few dozen
//   binades; a row that needs more than kWideSlots of them is handed on.
// * hist_rows_kernel (rows handed on): one thread-block cluster per row, each
//   CTA counting a slice of <= 65,535 elements in a full 65,536-key 16-bit
//   histogram (so a counter cannot wrap), summed through distributed shared
//   memory.
//
// Either way the occupied binades' counts become fp64 masses (two exps per
// binade and a geometric polynomial along the mantissa evaluated in
// double-float arithmetic), and one CTA walks
// binades and then keys from the top to the top-k and top-p cutoffs.  Only the
// probability of the row's own token may need one more look at the row (the
// rank of a tied token at the cutoff).
#include <climits>
#include <cooperative_groups.h>
#include <math.h>

#include "sv_internal.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace {

struct BinSum {
    double mass;
    uint32_t count;
    uint32_t pad;
};

struct CtaRes {
    unsigned long long maxc;   // (key16 << 32) | ~index of this CTA's maximum
    int bad;                   // NaN / +inf seen
    int tie_count;             // tie-rank pass: ties below the token in this slice
};

struct RowPlan {               // decided by the walking CTA, read by the others
    int skip;                  // 1: row is an error or done
    int need_tie;              // 1: run the tie-rank pass
    uint32_t cut_key;
    int token;
};

struct WalkState {             // the walk, phase to phase
    double z_all, z1, mk_bin, mass_above_bk, mass_above_bp, z;
    uint32_t cnt_above_bk, k_key, k_ties, cut_key, cut_ties, kept;
    int bk, bp, bmin, found, done, slot;
};

// Shared memory of the cutoff walk: per-binade count and mass (zero where a
// binade is empty), per-key counts and masses of up to two binades.
struct WalkSmem {
    BinSum sums[512];
    uint32_t kc[2][128];
    double ke[2][128];
    WalkState walk;
    RowPlan plan;
    double wmass[16];      // block scan: per-warp mass totals, then their exclusive prefixes
    uint32_t wcount[16];   // the same for counts
    int wlow[16];          // per-warp lowest occupied binade
    double e_tok;          // exp((v - m) / T) of the row's token (computed beside the scans)
};
constexpr int kWalkThreads = 512;   // walk_row runs on CTAs of this size: one binade per thread

struct HistSmem {
    uint32_t hist[kHistWords];
    uint32_t occ[16];
    uint32_t occ_all[16];
    int occ_list[512];
    int n_occ;
    CtaRes res;
    unsigned long long red64[kHistThreads / 32];
    int redi[kHistThreads / 32];
    uint32_t csc[kHistThreads][33];   // per-thread key counts of one binade quarter
    WalkSmem w;
};

// Counts of the 32 keys b*128 + 32 q .. + 31, summed over the cluster's
// histograms: 16 words (two counters each) read as four 16-byte vectors per
// rank.
__device__ __forceinline__ void cluster_counts32(cg::cluster_group& cluster, HistSmem& sm, int C, int b, int q,
                                                 uint32_t c[32])
{
#pragma unroll
    for (int j = 0; j < 32; ++j) c[j] = 0u;
    for (int r = 0; r < C; ++r) {
        const uint4* h4 = reinterpret_cast<const uint4*>(cluster.map_shared_rank(sm.hist, r)) + (b * 64 + q * 16) / 4;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 x = h4[v];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                c[8 * v + 2 * i] += w[i] & 0xFFFFu;
                c[8 * v + 2 * i + 1] += w[i] >> 16;
            }
        }
    }
}

// exp((v - m) / T) of the 32 keys b*128 + 32 q + j in fp64, handed to f(j, e)
// in key order: along a binade the mantissa step is constant, so while the
// step is small against T the masses follow a geometric recurrence from two
// exps; otherwise one exp per key.  Binade 0 holds -inf (mass 0).
template <typename F>
__device__ __forceinline__ void for_binade_masses32(int b, int q, double m, double T, F f)
{
    if (b == 0) {
        for (int j = 0; j < 32; ++j) f(j, 0.0);
        return;
    }
    const uint32_t kb = (uint32_t)b * 128u + 32u * (uint32_t)q;
    const double v_first = key_value(kb);
    const double step = key_value(kb + 1u) - v_first;
    if (step / T <= 1.0) {
        const double R = exp(step / T);
        double cur = exp((v_first - m) / T);
        for (int j = 0; j < 32; ++j) {
            f(j, cur);
            cur *= R;
        }
    } else {
        for (int j = 0; j < 32; ++j) f(j, exp((key_value(kb + j) - m) / T));
    }
}

// Mass of one binade, the sum over its 128 keys of c_k exp((v_k - m) / T),
// by its four quarter threads (adjacent lanes q = 0..3; c[j] is the count of
// key 128 b + 32 q + j).  Every lane of the warp calls it; a lane group with
// act false gets 0.  Along a binade the value step s is constant, so with
// r = exp(-s / T) a quarter's sum is exp((v_top - m) / T) r^(96 - 32 q) times
// the polynomial sum_j c_j r^(31 - j), evaluated by Horner's rule in
// double-float arithmetic; fp64 is left for the first lane's two exps and
// the products that join the quarters (a fixed-order 4-lane sum).  A step
// above T (keys far apart against T) takes one exp per key instead.
__device__ double binade_mass4(int b, int q, double m, double T, bool act, const uint32_t* c)
{
    const int lead = (threadIdx.x & 31) & ~3;
    const bool on = act && b > 0;
    const uint32_t kb = (uint32_t)b * 128u;
    double r64 = 0.0, etop = 0.0, r32 = 0.0;
    int geo = 0;   // the step is at most T: geometric masses
    if (on && q == 0) {
        const double x = (key_value(kb + 1u) - key_value(kb)) / T;
        geo = x <= 1.0;
        if (geo) {
            r64 = exp(-x);
            etop = exp((key_value(kb + 127u) - m) / T);
            r32 = r64;
#pragma unroll
            for (int i = 0; i < 5; ++i) r32 *= r32;
        }
    }
    geo = __shfl_sync(0xFFFFFFFFu, geo, lead);
    r64 = __shfl_sync(0xFFFFFFFFu, r64, lead);
    etop = __shfl_sync(0xFFFFFFFFu, etop, lead);
    r32 = __shfl_sync(0xFFFFFFFFu, r32, lead);
    double part = 0.0;
    if (on) {
        if (geo) {
            const dfloat r = df_of(r64);
            dfloat acc = {0.0f, 0.0f};
#pragma unroll 8
            for (int j = 0; j < 32; ++j) acc = df_add_f(df_mul(acc, r), (float)c[j]);
            double w = etop;
            for (int i = q; i < 3; ++i) w *= r32;
            part = w * df_val(acc);
        } else {
            for (int j = 0; j < 32; ++j)
                if (c[j]) part += (double)c[j] * exp((key_value(kb + 32u * (uint32_t)q + (uint32_t)j) - m) / T);
        }
    }
#pragma unroll
    for (int o = 2; o; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o, 4);
    return part;
}

// Per-key counts (summed over the cluster) and masses of binade b into slot s
// of the walk scratch.  Run by threads 0..3 of CTA 0 (32 keys each).
__device__ void load_binade_keys(cg::cluster_group& cluster, HistSmem& sm, int C, int b, int s, double m, double T)
{
    const int q = threadIdx.x;
    if (q >= 4) return;
    if (b < 0 || b > 511) {
        for (int j = 0; j < 32; ++j) {
            sm.w.kc[s][32 * q + j] = 0u;
            sm.w.ke[s][32 * q + j] = 0.0;
        }
        return;
    }
    uint32_t c[32];
    cluster_counts32(cluster, sm, C, b, q, c);
#pragma unroll
    for (int j = 0; j < 32; ++j) sm.w.kc[s][32 * q + j] = c[j];
    for_binade_masses32(b, q, m, T, [&](int j, double e) { sm.w.ke[s][32 * q + j] = e; });
}

// The cutoff walk of one row on one CTA, from the per-binade sums in sm.sums
// (filled for every occupied binade, zero elsewhere): binade scans run on
// warp 0, key walks on warp 0 and thread 0 (fp64 is scarce), and the
// decisions travel through shared memory between phases.  load_keys(b, s)
// fills sm.kc[s] / sm.ke[s] with the per-key counts and masses of binade b
// (every thread calls it; it may use threads 0..127).  sm.e_tok, the token's
// exp((v - m) / T), is computed here unless the caller set it (tok_ready).
// Writes the row's record unless status != 0, and leaves in sm.plan whether
// the token's tie rank is needed.  Every thread of the CTA must call it.
template <typename LoadKeys>
__device__ __noinline__ void walk_row(WalkSmem& sm, const RowsArgs& a, const RowTask& task, const uint16_t* row, RowInfo* info,
                         double m, int argmax, int status, bool tok_ready, LoadKeys load_keys)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const double T = (double)task.temp;
    WalkState& W = sm.walk;
    const int kk = task.k_eff;
    const bool topk_on = kk < a.vocab;
    if (tid == 0) {
        sm.plan.skip = status != 0;
        sm.plan.need_tie = 0;
        sm.plan.token = task.token;
    }
    const bool topp_on = task.top_p < 1.0f;
    const int d_tok = task.token;
    // the token's mass, on warp 1 while the scans below run on the others
    if (!tok_ready && status == 0 && tid == 32 && d_tok >= 0 && d_tok < a.vocab)
        sm.e_tok = exp((key_value(key16_of_bf16(row[d_tok])) - m) / T);
    if (!topk_on) {
        // Without top-k the top-p cut runs on the binade masses themselves:
        // one block-wide scan, binade 511 - tid on thread tid (descending),
        // gives Z1, the lowest occupied binade and the binade holding the
        // top-p crossing (its mass above and count above).
        const int b = 511 - tid;
        const uint32_t cnt = status == 0 ? sm.sums[b].count : 0u;
        const double ms = status == 0 ? sm.sums[b].mass : 0.0;
        uint32_t ci = cnt;
        double mi = ms;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, ci, o);
            const double z = __shfl_up_sync(0xFFFFFFFFu, mi, o);
            if (lane >= o) {
                ci += y;
                mi += z;
            }
        }
        const int low = __reduce_max_sync(0xFFFFFFFFu, cnt ? tid : -1);   // lowest binade = highest thread
        if (lane == 31) {
            sm.wmass[warp] = mi;
            sm.wcount[warp] = ci;
            sm.wlow[warp] = low;
        }
        __syncthreads();
        if (warp == 0) {   // exclusive prefixes of the 16 warp totals
            const double wm = lane < 16 ? sm.wmass[lane] : 0.0;
            const uint32_t wc = lane < 16 ? sm.wcount[lane] : 0u;
            double pm = wm;
            uint32_t pc = wc;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                const double z = __shfl_up_sync(0xFFFFFFFFu, pm, o);
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, pc, o);
                if (lane >= o) {
                    pm += z;
                    pc += y;
                }
            }
            const int lw = __reduce_max_sync(0xFFFFFFFFu, lane < 16 ? sm.wlow[lane] : -1);
            __syncwarp();
            if (lane < 16) {
                sm.wmass[lane] = pm - wm;
                sm.wcount[lane] = pc - wc;
            }
            if (lane == 15) {
                W.z_all = pm;
                W.z1 = pm;
            }
            if (lane == 0) {
                W.bmin = lw >= 0 ? 511 - lw : (1 << 30);
                W.bk = -1;
                W.found = 0;
            }
        }
        __syncthreads();
        if (status == 0 && topp_on) {
            const double target = (double)task.top_p * W.z1;
            const double mex = sm.wmass[warp] + (mi - ms);
            if (ms > 0.0 && mex < target && target <= mex + ms) {
                W.bp = b;
                W.mass_above_bp = mex;
                W.found = 1;
            }
        }
        __syncthreads();
    } else {
    // Phase A (warp 0): binade scan on counts and masses, descending.
    if (status == 0 && warp == 0) {
        uint32_t cs = 0u;
        double ms = 0.0;
        int lowest = 1 << 30;
        for (int i = 0; i < 16; ++i) {
            const int b = 511 - 16 * lane - i;
            cs += sm.sums[b].count;
            ms += sm.sums[b].mass;
            if (sm.sums[b].count) lowest = b;
        }
        uint32_t cin = cs;
        double min_ = ms;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, cin, o);
            const double z = __shfl_up_sync(0xFFFFFFFFu, min_, o);
            if (lane >= o) {
                cin += y;
                min_ += z;
            }
        }
        lowest = __reduce_min_sync(0xFFFFFFFFu, lowest);
        if (lane == 31) W.z_all = min_;
        if (lane == 0) {
            W.bmin = lowest;
            W.bk = -1;
        }
        __syncwarp();
        uint32_t cex = cin - cs;
        double mex = min_ - ms;
        if (topk_on && cex < (uint32_t)kk && (uint32_t)kk <= cin) {
            for (int i = 0; i < 16; ++i) {
                const int b = 511 - 16 * lane - i;
                if (cex + sm.sums[b].count >= (uint32_t)kk) {
                    W.bk = b;
                    W.cnt_above_bk = cex;
                    W.mass_above_bk = mex;
                    break;
                }
                cex += sm.sums[b].count;
                mex += sm.sums[b].mass;
            }
        }
    }
    __syncthreads();
    // Phase B: keys of the top-k boundary binade.
    if (status == 0 && topk_on) load_keys(W.bk, 0);
    __syncthreads();
    // Phase C (warp 0): top-k cutoff key, kept ties, Z1.  Lane l holds
    // keys 127 - 4l .. 124 - 4l (descending); warp scans give the counts
    // and masses above each lane's keys.
    if (status == 0 && warp == 0) {
        if (topk_on) {
            uint32_t c4 = 0u;
            double m4 = 0.0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int f = 127 - 4 * lane - i;
                c4 += sm.kc[0][f];
                m4 += (double)sm.kc[0][f] * sm.ke[0][f];
            }
            uint32_t ci = c4;
            double mi = m4;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, ci, o);
                const double z = __shfl_up_sync(0xFFFFFFFFu, mi, o);
                if (lane >= o) {
                    ci += y;
                    mi += z;
                }
            }
            uint32_t cum = W.cnt_above_bk + (ci - c4);
            double mass = W.mass_above_bk + (mi - m4);
            const bool mine = cum < (uint32_t)kk && (uint32_t)kk <= cum + c4;
            if (mine) {
                for (int i = 0; i < 4; ++i) {
                    const int f = 127 - 4 * lane - i;
                    const uint32_t c = sm.kc[0][f];
                    if (c == 0u) continue;
                    if (cum + c >= (uint32_t)kk) {
                        W.k_key = (uint32_t)W.bk * 128u + f;
                        W.k_ties = (uint32_t)kk - cum;
                        W.mk_bin = mass - W.mass_above_bk + (double)W.k_ties * sm.ke[0][f];
                        W.z1 = mass + (double)W.k_ties * sm.ke[0][f];
                        break;
                    }
                    cum += c;
                    mass += (double)c * sm.ke[0][f];
                }
            }
        } else if (lane == 0) {
            W.z1 = W.z_all;
        }
        if (lane == 0) W.found = 0;
    }
    __syncthreads();
    // Phase D (warp 0): top-p binade on masses capped at the top-k cutoff.
    if (status == 0 && topp_on && warp == 0) {
        const double target = (double)task.top_p * W.z1;
        const int bk = W.bk;
        double ms = 0.0;
        for (int i = 0; i < 16; ++i) {
            const int b = 511 - 16 * lane - i;
            ms += (!topk_on || b > bk) ? sm.sums[b].mass : (b == bk ? W.mk_bin : 0.0);
        }
        double min_ = ms;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, min_, o);
            if (lane >= o) min_ += y;
        }
        double mex = min_ - ms;
        if (mex < target && target <= min_) {
            for (int i = 0; i < 16; ++i) {
                const int b = 511 - 16 * lane - i;
                const double mb = (!topk_on || b > bk) ? sm.sums[b].mass : (b == bk ? W.mk_bin : 0.0);
                if (mb > 0.0 && mex + mb >= target) {
                    W.bp = b;
                    W.mass_above_bp = mex;
                    W.found = 1;
                    break;
                }
                mex += mb;
            }
        }
    }
    __syncthreads();
    }
    // Phase E: keys of the binade that holds the final cutoff (slot 1).
    int load_b = -1;
    if (status == 0) {
        if (W.found)
            load_b = (topk_on && W.bp == W.bk) ? -1 : W.bp;
        else if (!topk_on)
            load_b = W.bmin;
    }
    if (load_b >= 0) load_keys(load_b, 1);
    __syncthreads();
    // Phase F (warp 0): the final cutoff, by a warp walk over the keys of
    // binade bp (lane l: keys 127 - 4l .. 124 - 4l), then thread 0
    // writes the row's record.
    if (status == 0 && warp == 0) {
        if (W.found) {
            const int bp = W.bp;
            const int slot = (topk_on && bp == W.bk) ? 0 : 1;
            const double target = (double)task.top_p * W.z1;
            uint32_t above = 0u;   // elements in binades above bp
            for (int b = 511 - lane; b > bp; b -= 32) above += sm.sums[b].count;
            above = __reduce_add_sync(0xFFFFFFFFu, above);
            uint32_t ce4[4];
            double e4[4];
            uint32_t c4 = 0u;
            double m4 = 0.0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int f = 127 - 4 * lane - i;
                const uint32_t key = (uint32_t)bp * 128u + f;
                uint32_t ce = sm.kc[slot][f];
                if (topk_on && bp == W.bk) ce = key > W.k_key ? ce : (key == W.k_key ? W.k_ties : 0u);
                ce4[i] = ce;
                e4[i] = sm.ke[slot][f];
                c4 += ce;
                m4 += (double)ce * e4[i];
            }
            uint32_t ci = c4;
            double mi = m4;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, ci, o);
                const double z = __shfl_up_sync(0xFFFFFFFFu, mi, o);
                if (lane >= o) {
                    ci += y;
                    mi += z;
                }
            }
            uint32_t cnt_above = above + (ci - c4);
            double cum = W.mass_above_bp + (mi - m4);
            int hit_f = -1;
            uint32_t hit_j = 0u, hit_kept = 0u;
            double hit_z = 0.0;
            for (int i = 0; i < 4 && hit_f < 0; ++i) {
                const uint32_t ce = ce4[i];
                if (ce == 0u) continue;
                const double e = e4[i];
                if (cum + (double)ce * e >= target) {
                    const double jd = ceil((target - cum) / e);
                    uint32_t j = jd < 1.0 ? 1u : (jd > (double)ce ? ce : (uint32_t)jd);
                    while (j > 1u && cum + (double)(j - 1u) * e >= target) --j;
                    while (j < ce && cum + (double)j * e < target) ++j;
                    hit_f = 127 - 4 * lane - i;
                    hit_j = j;
                    hit_kept = cnt_above + j;
                    hit_z = cum + (double)j * e;
                    break;
                }
                cum += (double)ce * e;
                cnt_above += ce;
            }
            const unsigned hits = __ballot_sync(0xFFFFFFFFu, hit_f >= 0);
            if (hits && lane == __ffs(hits) - 1) {
                W.cut_key = (uint32_t)bp * 128u + hit_f;
                W.cut_ties = hit_j;
                W.kept = hit_kept;
                W.z = hit_z;
                W.slot = slot;
            }
            if (lane == 0) W.done = hits != 0u;
        } else if (lane == 0) {
            W.done = 0;
        }
    }
    __syncthreads();
    if (status == 0 && tid == 0) {
        uint32_t cut_key = W.cut_key, cut_ties = W.cut_ties, kept = W.kept;
        double z = W.z;
        int slot = W.slot;
        if (!W.done) {
            if (topk_on) {
                cut_key = W.k_key;
                cut_ties = W.k_ties;
                kept = (uint32_t)kk;
                z = W.z1;
                slot = 0;
            } else {
                int f = 0;
                while (f < 127 && sm.kc[1][f] == 0u) ++f;
                cut_key = (uint32_t)W.bmin * 128u + f;
                cut_ties = sm.kc[1][f];
                kept = (uint32_t)a.vocab;
                z = W.z1;
                slot = 1;
            }
        }
        const uint32_t cut_count = sm.kc[slot][cut_key & 127u];
        info->desc.max_logit = (float)m;
        info->desc.log_norm = logf((float)z);
        info->desc.cutoff_logit = f32_of_key16(cut_key);
        info->desc.cutoff_ties = (int)cut_ties;
        info->desc.kept = (int)kept;
        info->desc.argmax = argmax;
        info->desc.status = 0;
        info->desc.temperature = task.temp;
        info->z = z;
        info->z_rest = z - 1.0;   // the top token's mass is exp(0)
        info->n_list = -1;
        info->cut_count = (int)cut_count;
        sm.plan.cut_key = cut_key;
        // the row's token: kept unless it sits in a partial tie group
        const int d = task.token;
        if (d >= 0 && d < a.vocab) {
            const uint32_t kd = key16_of_bf16(row[d]);
            if (kd == cut_key && cut_ties < cut_count) {
                sm.plan.need_tie = 1;
            } else {
                info->p_token = kd >= cut_key ? sm.e_tok / z : 0.0;
            }
        } else {
            info->p_token = nan("");
        }
    }
}

// Record of a row that failed (non-finite logits, or nothing but -inf).
__device__ void write_error_row(RowInfo* info, double m, int argmax, int status, float temp)
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

// p of a token tied with the cutoff: kept when fewer than cutoff_ties of its
// ties come before it.
__device__ void finish_tied_token(RowInfo* info, uint32_t cut_key, int rank_d, double m, double T)
{
    const bool keep = rank_d < info->desc.cutoff_ties;
    info->p_token = keep ? exp((key_value(cut_key) - m) / T) / info->z : 0.0;
}

// Process one row with the whole cluster; CTA 0 writes the RowInfo.
__device__ void hist_row(cg::cluster_group& cluster, HistSmem& sm, const RowsArgs& a, const RowTask& task, int C,
                         int rank, int slice)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t stride = task.is_draft ? a.stride_d : a.stride_t;
    const uint16_t* row = (const uint16_t*)(task.is_draft ? a.drf : a.tgt) + (size_t)task.row * (size_t)stride;
    RowInfo* info = a.info + task.slot;
    const double T = (double)task.temp;

    // 1. zero the histogram and the binade sums
    {
        uint4* h4 = reinterpret_cast<uint4*>(sm.hist);
        for (int i = tid; i < kHistWords / 4; i += kHistThreads) h4[i] = make_uint4(0u, 0u, 0u, 0u);
        for (int i = tid; i < 512; i += kHistThreads) {
            sm.w.sums[i].mass = 0.0;
            sm.w.sums[i].count = 0u;
        }
    }
    cluster.sync();

    // 2. stream the slice once: counts, NaN/+inf, first maximum
    const int s0 = rank * slice;
    const int s1 = min(a.vocab, s0 + slice);
    uint32_t best_key = 0u;
    int best_idx = 0x7FFFFFFF;
    int bad = 0;
    const bool aligned = ((((uintptr_t)(row + s0)) & 15u) == 0u);
    auto count_one = [&](uint32_t h, int idx) {
        const uint32_t k = key16_of_bf16(h);
        bad |= (k >= 0xFF80u) | (k < 0x007Fu);
        atomicAdd(&sm.hist[k >> 1], (k & 1u) ? 0x10000u : 1u);
        if (k > best_key || (k == best_key && idx < best_idx)) {
            best_key = k;
            best_idx = idx;
        }
    };
    constexpr int kUnroll = 8;   // 8 x 16 B per thread in flight
    for (int base = s0 + tid * 8; base < s1; base += kHistThreads * 8 * kUnroll) {
        uint4 v[kUnroll];
        bool full[kUnroll];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const int e0 = base + q * kHistThreads * 8;
            full[q] = aligned && (e0 + 8 <= s1);
            if (full[q]) v[q] = __ldg(reinterpret_cast<const uint4*>(row + e0));
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const int e0 = base + q * kHistThreads * 8;
            if (full[q]) {
                const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    count_one(w[j] & 0xFFFFu, e0 + 2 * j);
                    count_one(w[j] >> 16, e0 + 2 * j + 1);
                }
            } else {
                for (int i = e0; i < min(e0 + 8, s1); ++i) count_one(row[i], i);
            }
        }
    }
    {
        unsigned long long c = best_idx == 0x7FFFFFFF
                                   ? 0ull
                                   : (((unsigned long long)best_key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)best_idx));
        c = warp_max_u64(c);
        const int wb = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0) {
            sm.red64[warp] = c;
            sm.redi[warp] = wb;
        }
        __syncthreads();
        if (tid == 0) {
            unsigned long long mc = 0ull;
            int bb = 0;
            for (int w = 0; w < kHistThreads / 32; ++w) {
                mc = sm.red64[w] > mc ? sm.red64[w] : mc;
                bb |= sm.redi[w];
            }
            sm.res.maxc = mc;
            sm.res.bad = bb;
        }
    }
    cluster.sync();

    // 3. row maximum, argmax and status (every CTA computes the same)
    unsigned long long maxc = 0ull;
    int any_bad = 0;
    for (int r = 0; r < C; ++r) {
        const CtaRes* o = cluster.map_shared_rank(&sm.res, r);
        maxc = o->maxc > maxc ? o->maxc : maxc;
        any_bad |= o->bad;
    }
    const uint32_t m_key = (uint32_t)(maxc >> 32);
    const int argmax = (int)(0xFFFFFFFFu - (uint32_t)maxc);
    const double m = key_value(m_key);
    int status = any_bad ? kNonfinite : (m_key == 0x007Fu ? kEmpty : 0);

    // 4. occupied binades (a binade = 128 keys = 64 histogram words)
    if (status == 0) {
        const int b = tid;   // 512 threads, one binade each
        const uint4* h4 = reinterpret_cast<const uint4*>(sm.hist) + b * 16;
        uint32_t any = 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint4 q = h4[i];
            any |= q.x | q.y | q.z | q.w;
        }
        const unsigned bits = __ballot_sync(0xFFFFFFFFu, any != 0u);
        if (lane == 0) sm.occ[warp] = bits;
    }
    cluster.sync();
    if (status == 0) {
        if (tid < 16) {
            uint32_t o = 0u;
            for (int r = 0; r < C; ++r) o |= cluster.map_shared_rank(sm.occ, r)[tid];
            sm.occ_all[tid] = o;
        }
        __syncthreads();
        if (warp == 0) {
            const uint32_t word = lane < 16 ? sm.occ_all[lane] : 0u;
            const int cnt = __popc(word);
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            int pos = incl - cnt;
            for (int bit = 0; bit < 32; ++bit)
                if (word & (1u << bit)) sm.occ_list[pos++] = lane * 32 + bit;
            if (lane == 31) sm.n_occ = incl;
        }
        __syncthreads();
        // 5. binade sums: this CTA owns occupied binades j = rank, rank + C,
        //    ...; four threads per binade, 32 keys each.  Every thread of a
        //    warp runs the same number of rounds (the loop bound is uniform
        //    per warp), so the 4-lane reductions below see all their lanes.
        const int n_occ = sm.n_occ;
        BinSum* sums0 = cluster.map_shared_rank(sm.w.sums, 0);
        const int q4 = tid & 3;
        const int n_mine = n_occ > rank ? (n_occ - rank + C - 1) / C : 0;
        for (int i0 = (tid >> 2) - (lane >> 2); i0 < n_mine; i0 += kHistThreads / 4) {
            const int i = i0 + (lane >> 2);
            const bool act = i < n_mine;
            const int b = act ? sm.occ_list[rank + C * i] : 0;
            uint32_t csum = 0u;
            uint32_t* cs = sm.csc[tid];   // counts in shared scratch, indexed freely by the mass loop
            if (act) {
                uint32_t c[32];
                cluster_counts32(cluster, sm, C, b, q4, c);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    csum += c[j];
                    cs[j] = c[j];
                }
            }
            const double mass = binade_mass4(b, q4, m, T, act, cs);
#pragma unroll
            for (int o = 2; o; o >>= 1) csum += __shfl_xor_sync(0xFFFFFFFFu, csum, o, 4);
            if (act && q4 == 0) {
                sums0[b].mass = mass;
                sums0[b].count = csum;
            }
        }
    }
    cluster.sync();

    // 6. CTA 0: the cutoff walk on the cluster's sums.
    if (rank == 0)
        walk_row(sm.w, a, task, row, info, m, argmax, status, false,
                 [&](int b, int s) { load_binade_keys(cluster, sm, C, b, s, m, T); });
    cluster.sync();

    // 7. tie rank of the row's token inside a partial tie group
    const RowPlan plan = *cluster.map_shared_rank(&sm.w.plan, 0);
    if (!plan.skip && plan.need_tie) {
        const int d = plan.token;
        const int e1 = min(s1, d);
        int cnt = 0;
        for (int i = s0 + tid; i < e1; i += kHistThreads) cnt += key16_of_bf16(row[i]) == plan.cut_key ? 1 : 0;
        cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
        if (lane == 0) sm.redi[warp] = cnt;
        __syncthreads();
        if (tid == 0) {
            int tot = 0;
            for (int w = 0; w < kHistThreads / 32; ++w) tot += sm.redi[w];
            sm.res.tie_count = tot;
        }
    }
    cluster.sync();
    if (rank == 0 && tid == 0) {
        if (status != 0) {
            write_error_row(info, m, argmax, status, task.temp);
        } else if (plan.need_tie) {
            int rank_d = 0;
            for (int r = 0; r < C; ++r) rank_d += cluster.map_shared_rank(&sm.res, r)->tie_count;
            finish_tied_token(info, plan.cut_key, rank_d, m, T);
        }
    }
    cluster.sync();   // the histograms may be cleared for the next row
}

__global__ void __launch_bounds__(kHistThreads, 1) hist_rows_kernel(const __grid_constant__ RowsArgs a, int slice)
{
    pdl_enter();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    HistSmem& sm = *reinterpret_cast<HistSmem*>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int cluster_id = blockIdx.x / C;
    const int n_clusters = gridDim.x / C;
    const int n_tasks = a.counters->n_ovf;   // rows the one-CTA kernel handed on
    for (int t = cluster_id; t < n_tasks; t += n_clusters) {
        const RowTask task = a.slow_tasks.get(a.ovf_idx[t]);
        hist_row(cluster, sm, a, task, C, rank, slice);
    }
}

// ----------------------------------------------------------------------------
// One CTA per row, counters for the binades the row occupies
// ----------------------------------------------------------------------------
constexpr int kWideThreads = 512;
constexpr int kWideBlocks = 3;          // CTAs per SM the launch bounds aim at (registers: 65,536 / 1,536)
constexpr int kWideSlots = 64;           // binades with counters per row (4 threads per slot in the mass pass)
constexpr int kWideUnroll = 4;           // 16-byte vectors per thread in flight
constexpr int kUnclaimed = INT_MIN;      // base[] of a binade not seen yet in this row
constexpr int kClaiming = INT_MIN + 1;   // base[] while a thread assigns the binade its counters
constexpr int kBaseMin = -65536;         // a claimed base is 128 * (slot - b) >= -65,408
constexpr int kClaimSpins = 1 << 14;     // polls before a thread stops waiting for a claim
constexpr int kDecideSpins = 120;        // polls (about 256 ns apart) for the previous position's test
static_assert(kWideThreads >= 4 * kWideSlots, "the mass pass takes four threads per slot");
static_assert(kWideThreads == kWalkThreads && kHistThreads == kWalkThreads, "walk_row takes one binade per thread");
static_assert(2 * kWideSlots < kWideThreads, "the last thread is idle in the exps of the mass pass");

struct WideSmem {
    uint32_t cnt[(kWideSlots + 1) * 128];   // per-key counters of the claimed binades, then 128 catch-alls
    int32_t base[512];                      // binade b: 128 * (slot - b), so base + key indexes cnt
    int32_t bin_of[kWideSlots];             // binade of each slot
    int32_t n_slots;                        // slots handed out (beyond kWideSlots: overflow)
    int32_t ovf;                            // 1: a key found no counter; the cluster kernel redoes the row
    int32_t zero_mix;                       // 1: the row holds both -0 and +0
    int32_t neg_nan;                        // 1: a key below that of -inf (a NaN with the sign bit set)
    unsigned long long red64[kWideThreads / 32];
    int32_t redi[kWideThreads / 32];
    double inv_t;                           // 1 / T of the row
    double g_r[kWideSlots];                 // per slot: r = exp(-step / T) along its binade (0: one exp per key)
    double g_r32[kWideSlots];               // r^32
    double g_etop[kWideSlots];              // exp((v - m) / T) of the binade's top key
    WalkSmem w;
};

// Counter base of binade b, giving it the next slot if it has none.  The
// first thread to see b takes a slot and publishes the base; a thread that
// sees b meanwhile polls (a bounded number of times) until it is published.
// Out of slots, or out of patience, the keys go to the catch-all counters and
// the row is marked for the cluster kernel.
__device__ __noinline__ int claim_binade(WideSmem& sm, int b)
{
    int v = atomicCAS(&sm.base[b], kUnclaimed, kClaiming);
    if (v == kUnclaimed) {
        const int n = atomicAdd(&sm.n_slots, 1);
        int nb;
        if (n < kWideSlots) {
            sm.bin_of[n] = b;
            nb = 128 * (n - b);
        } else {
            sm.ovf = 1;
            nb = 128 * (kWideSlots - b);
        }
        atomicExch(&sm.base[b], nb);
        return nb;
    }
    volatile int* vb = &sm.base[b];
    for (int i = 0; v == kClaiming && i < kClaimSpins; ++i) v = *vb;
    if (v == kClaiming) {
        sm.ovf = 1;
        return 128 * (kWideSlots - b);
    }
    return v;
}

__device__ __forceinline__ void count_key(WideSmem& sm, uint32_t key)
{
    const int b = (int)(key >> 7);
    int bs = sm.base[b];
    if (bs < kBaseMin) bs = claim_binade(sm, b);
    atomicAdd(&sm.cnt[bs + (int)key], 1u);
}

// Order key of a bf16 pattern without folding -0 into +0 (-0 gets the key
// just below that of +0; the two counters are merged after the row).
__device__ __forceinline__ uint32_t key_raw16(uint32_t h)
{
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
}

// Returns true when the row went to the cluster kernel (no record written here).
__device__ bool wide_row(WideSmem& sm, const RowsArgs& a, const RowTask& task, int t)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t stride = task.is_draft ? a.stride_d : a.stride_t;
    const uint16_t* row = (const uint16_t*)(task.is_draft ? a.drf : a.tgt) + (size_t)task.row * (size_t)stride;
    RowInfo* info = a.info + task.slot;
    const double T = (double)task.temp;
    const int V = a.vocab;

    // the token's key, loaded now so that its latency hides behind the row
    const int d_tok = task.token;
    const uint32_t tok_key = (tid == kWideThreads - 1 && d_tok >= 0 && d_tok < V) ? key16_of_bf16(row[d_tok]) : 0u;

    // 1. stream the row once: per-key counts and the first maximum.  The
    //    elements before the first 16-byte boundary and after the last whole
    //    vector are taken one by one.
    uint32_t best_key = 0u;
    int best_idx = INT_MAX;
    auto note = [&](uint32_t key, int idx) {
        if (key > best_key || (key == best_key && idx < best_idx)) {
            best_key = key;
            best_idx = idx;
        }
    };
    const int head = min(V, (int)(((16u - ((uint32_t)(uintptr_t)row & 15u)) & 15u) >> 1));
    const int nvec = (V - head) >> 3;
    const int tail0 = head + 8 * nvec;
    if (tid < head) {
        const uint32_t k = key_raw16(row[tid]);
        count_key(sm, k);
        note(k, tid);
    }
    if (tail0 + tid < V) {
        const uint32_t k = key_raw16(row[tail0 + tid]);
        count_key(sm, k);
        note(k, tail0 + tid);
    }
    const uint4* vp = reinterpret_cast<const uint4*>(row + head);
    for (int v0 = tid; v0 < nvec; v0 += kWideThreads * kWideUnroll) {
        uint4 x[kWideUnroll];
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u) {
            const int vi = v0 + u * kWideThreads;
            x[u] = vi < nvec ? __ldg(vp + vi) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u) {
            const int vi = v0 + u * kWideThreads;
            if (vi < nvec) {
                const uint32_t k0 = keys2_raw(x[u].x), k1 = keys2_raw(x[u].y), k2 = keys2_raw(x[u].z),
                               k3 = keys2_raw(x[u].w);
                count_key(sm, k0 & 0xFFFFu);
                count_key(sm, k0 >> 16);
                count_key(sm, k1 & 0xFFFFu);
                count_key(sm, k1 >> 16);
                count_key(sm, k2 & 0xFFFFu);
                count_key(sm, k2 >> 16);
                count_key(sm, k3 & 0xFFFFu);
                count_key(sm, k3 >> 16);
                const uint32_t mx = max_u16x2(max_u16x2(k0, k1), max_u16x2(k2, k3));
                const uint32_t vmax = max(mx & 0xFFFFu, mx >> 16);
                if (vmax >= best_key) {   // first element of the vector holding its maximum
                    const int j = (k0 & 0xFFFFu) == vmax ? 0
                                  : (k0 >> 16) == vmax   ? 1
                                  : (k1 & 0xFFFFu) == vmax ? 2
                                  : (k1 >> 16) == vmax   ? 3
                                  : (k2 & 0xFFFFu) == vmax ? 4
                                  : (k2 >> 16) == vmax   ? 5
                                  : (k3 & 0xFFFFu) == vmax ? 6
                                                           : 7;
                    note(vmax, head + 8 * vi + j);
                }
            }
        }
    }
    {
        unsigned long long c = best_idx == INT_MAX ? 0ull
                                                   : (((unsigned long long)best_key << 32) |
                                                      (unsigned long long)(0xFFFFFFFFu - (uint32_t)best_idx));
        c = warp_max_u64(c);
        if (lane == 0) sm.red64[warp] = c;
    }
    __syncthreads();   // every count is in

    // 2. thread 0: fold -0 into +0, look for negative NaNs
    if (tid == 0) {
        int mix = 0;
        const int bn = sm.base[255];   // binade of -0 (key 0x7FFF)
        if (bn >= kBaseMin && sm.cnt[bn + 0x7FFF] != 0u) {
            int bp = sm.base[256];     // binade of +0 (key 0x8000)
            mix = bp >= kBaseMin && sm.cnt[bp + 0x8000] != 0u;
            if (bp < kBaseMin) bp = claim_binade(sm, 256);
            sm.cnt[bp + 0x8000] += sm.cnt[bn + 0x7FFF];
            sm.cnt[bn + 0x7FFF] = 0u;
        }
        sm.zero_mix = mix;
        int nn = 0;
        const int b0 = sm.base[0];
        if (b0 >= kBaseMin)
            for (int k = 0; k < 0x7F; ++k) nn |= sm.cnt[b0 + k] != 0u ? 1 : 0;
        sm.neg_nan = nn;
    }
    __syncthreads();
    unsigned long long maxc = 0ull;
#pragma unroll
    for (int w = 0; w < kWideThreads / 32; ++w) maxc = sm.red64[w] > maxc ? sm.red64[w] : maxc;
    const uint32_t raw_key = (uint32_t)(maxc >> 32);
    const uint32_t m_key = raw_key == 0x7FFFu ? 0x8000u : raw_key;
    int argmax = (int)(0xFFFFFFFFu - (uint32_t)maxc);
    const double m = key_value(m_key);
    const int status = (m_key >= 0xFF80u || sm.neg_nan) ? kNonfinite : (m_key == 0x007Fu ? kEmpty : 0);
    const bool ovf = sm.ovf != 0;
    const int used = ovf ? kWideSlots + 1 : sm.n_slots;

    if (ovf) {
        if (tid == 0) a.ovf_idx[atomicAdd(&a.counters->n_ovf, 1)] = t;
    } else {
        // the maximum is a zero and both signs occur: the first zero of either sign
        if (sm.zero_mix && m_key == 0x8000u) {
            int first = INT_MAX;
            for (int i = tid; i < V; i += kWideThreads)
                if ((row[i] & 0x7FFFu) == 0u) {
                    first = i;
                    break;
                }
            first = __reduce_min_sync(0xFFFFFFFFu, first);
            if (lane == 0) sm.redi[warp] = first;
            __syncthreads();
#pragma unroll
            for (int w = 0; w < kWideThreads / 32; ++w) first = min(first, sm.redi[w]);
            argmax = first;
            __syncthreads();
        }

        // 3. per-binade count and mass.  Each fp64 warp instruction holds the
        //    narrow fp64 pipe for the whole warp, so the two exps of each
        //    occupied binade go one per lane (r = exp(-step / T) and the top
        //    key's exp((v - m) / T)), and the mantissa polynomials run in
        //    double-float arithmetic on four threads per slot (32 keys each).
        if (status == 0) {
            if (tid == 0) sm.inv_t = 1.0 / T;
            __syncthreads();
            const double inv_t = sm.inv_t;
            if (tid == kWideThreads - 1)   // an idle thread here: the token's mass for the walk's record
                sm.w.e_tok = tok_key ? exp((key_value(tok_key) - m) * inv_t) : 0.0;
            for (int i = tid; i < 2 * used; i += kWideThreads) {
                const int sl = i < used ? i : i - used;
                const int b = sm.bin_of[sl];
                const uint32_t kb = (uint32_t)b * 128u;
                if (i < used) {
                    const double x = (key_value(kb + 1u) - key_value(kb)) * inv_t;
                    double r = 0.0, r32 = 0.0;
                    if (b > 0 && x <= 1.0) {
                        r = exp(-x);
                        r32 = r;
#pragma unroll
                        for (int k = 0; k < 5; ++k) r32 *= r32;
                    }
                    sm.g_r[sl] = r;
                    sm.g_r32[sl] = r32;
                } else {
                    sm.g_etop[sl] = b > 0 ? exp((key_value(kb + 127u) - m) * inv_t) : 0.0;
                }
            }
            __syncthreads();
        }
        {
            const int sl = tid >> 2, q = tid & 3;
            const bool act = status == 0 && sl < used;
            const int b = act ? sm.bin_of[sl] : 0;
            const uint32_t* c = sm.cnt + (act ? sl : 0) * 128 + 32 * q;
            uint32_t csum = 0u;
            double part = 0.0;
            if (act) {
#pragma unroll
                for (int j = 0; j < 32; ++j) csum += c[j];
                if (b > 0 && csum) {
                    const double r64 = sm.g_r[sl];
                    if (r64 > 0.0) {   // sum_j c_j r^(31 - j), relative to the quarter's top key
                        const dfloat r = df_of(r64);
                        dfloat acc = {0.0f, 0.0f};
#pragma unroll 8
                        for (int j = 0; j < 32; ++j) acc = df_add_f(df_mul(acc, r), (float)c[j]);
                        double w = sm.g_etop[sl];
                        for (int i = q; i < 3; ++i) w *= sm.g_r32[sl];
                        part = w * df_val(acc);
                    } else {   // keys far apart against T: one exp per key
                        for (int j = 0; j < 32; ++j)
                            if (c[j])
                                part += (double)c[j] *
                                        exp((key_value((uint32_t)b * 128u + 32u * (uint32_t)q + (uint32_t)j) - m) * sm.inv_t);
                    }
                }
            }
#pragma unroll
            for (int o = 2; o; o >>= 1) {   // fixed-order sum over the four threads of a slot
                part += __shfl_xor_sync(0xFFFFFFFFu, part, o, 4);
                csum += __shfl_xor_sync(0xFFFFFFFFu, csum, o, 4);
            }
            if (act && q == 0) {
                sm.w.sums[b].mass = part;
                sm.w.sums[b].count = csum;
            }
        }
        __syncthreads();

        // 4. the cutoff walk, with per-key counts straight from the slots and
        //    per-key masses e_top r^(127 - k) (double-float powers), one key
        //    per thread
        walk_row(sm.w, a, task, row, info, m, argmax, status, true, [&](int b, int s) {
            const int k = threadIdx.x;
            if (k >= 128) return;
            const int bs = (b >= 0 && b < 512) ? sm.base[b] : kUnclaimed;
            if (bs < kBaseMin) {
                sm.w.kc[s][k] = 0u;
                sm.w.ke[s][k] = 0.0;
                return;
            }
            const int sl = (bs >> 7) + b;   // bs = 128 (slot - b)
            sm.w.kc[s][k] = sm.cnt[sl * 128 + k];
            double e = 0.0;
            if (b > 0) {
                const double r64 = sm.g_r[sl];
                if (r64 > 0.0) {
                    dfloat p = {1.0f, 0.0f}, base = df_of(r64);
                    for (int n = 127 - k; n; n >>= 1) {
                        if (n & 1) p = df_mul(p, base);
                        base = df_mul(base, base);
                    }
                    e = sm.g_etop[sl] * df_val(p);
                } else {
                    e = exp((key_value((uint32_t)b * 128u + (uint32_t)k) - m) * sm.inv_t);
                }
            }
            sm.w.ke[s][k] = e;
        });
        __syncthreads();

        // 5. tie rank of the row's token inside a partial tie group, or the
        //    record of a failed row
        const RowPlan plan = sm.w.plan;
        if (status == 0 && plan.need_tie) {
            int cnt = 0;
            for (int i = tid; i < plan.token; i += kWideThreads) cnt += key16_of_bf16(row[i]) == plan.cut_key ? 1 : 0;
            cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
            if (lane == 0) sm.redi[warp] = cnt;
            __syncthreads();
            if (tid == 0) {
                int tot = 0;
#pragma unroll
                for (int w = 0; w < kWideThreads / 32; ++w) tot += sm.redi[w];
                finish_tied_token(info, plan.cut_key, tot, m, T);
            }
        }
        if (status != 0 && tid == 0) write_error_row(info, m, argmax, status, task.temp);
    }

    // 6. clear what the row used
    __syncthreads();
    {
        uint4* c4 = reinterpret_cast<uint4*>(sm.cnt);
        for (int i = tid; i < used * 32; i += kWideThreads) c4[i] = make_uint4(0u, 0u, 0u, 0u);
        for (int i = tid; i < 512; i += kWideThreads) {
            sm.base[i] = kUnclaimed;
            sm.w.sums[i].mass = 0.0;
            sm.w.sums[i].count = 0u;
        }
        if (tid == 0) {
            sm.n_slots = 0;
            sm.ovf = 0;
        }
    }
    __syncthreads();
    return ovf;
}

// A row whose acceptance test can no longer matter (it lies past a position
// its request is known to reject): one streaming pass for what the row's
// status needs (largest and smallest order key: NaN, +inf, every element
// -inf), and a record with that status and no distribution (p_token NaN).
__device__ __noinline__ void scan_row(WideSmem& sm, const RowsArgs& a, const RowTask& task)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t stride = task.is_draft ? a.stride_d : a.stride_t;
    const uint16_t* row = (const uint16_t*)(task.is_draft ? a.drf : a.tgt) + (size_t)task.row * (size_t)stride;
    const int V = a.vocab;
    // both keys of a word side by side: hi = max, lo = min (each u16x2)
    uint32_t hi = 0u, lo = 0xFFFFFFFFu;
    const int head = min(V, (int)(((16u - ((uint32_t)(uintptr_t)row & 15u)) & 15u) >> 1));
    const int nvec = (V - head) >> 3;
    const int tail0 = head + 8 * nvec;
    if (tid < head) {
        const uint32_t k = key_raw16(row[tid]);
        hi = max_u16x2(hi, k);
        lo = min_u16x2(lo, k | 0xFFFF0000u);
    }
    if (tail0 + tid < V) {
        const uint32_t k = key_raw16(row[tail0 + tid]);
        hi = max_u16x2(hi, k);
        lo = min_u16x2(lo, k | 0xFFFF0000u);
    }
    const uint4* vp = reinterpret_cast<const uint4*>(row + head);
    for (int v0 = tid; v0 < nvec; v0 += kWideThreads * kWideUnroll) {
        uint4 x[kWideUnroll];
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u) {
            const int vi = v0 + u * kWideThreads;
            x[u] = vi < nvec ? __ldcs(vp + vi) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u) {
            if (v0 + u * kWideThreads < nvec) {
                const uint32_t k0 = keys2_raw(x[u].x), k1 = keys2_raw(x[u].y), k2 = keys2_raw(x[u].z),
                               k3 = keys2_raw(x[u].w);
                hi = max_u16x2(hi, max_u16x2(max_u16x2(k0, k1), max_u16x2(k2, k3)));
                lo = min_u16x2(lo, min_u16x2(min_u16x2(k0, k1), min_u16x2(k2, k3)));
            }
        }
    }
    uint32_t kmax = max(hi & 0xFFFFu, hi >> 16), kmin = min(lo & 0xFFFFu, lo >> 16);
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    if (lane == 0) {
        sm.redi[warp] = (int)kmax;
        sm.red64[warp] = kmin;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 0; w < kWideThreads / 32; ++w) {
            kmax = max(kmax, (uint32_t)sm.redi[w]);
            kmin = min(kmin, (uint32_t)sm.red64[w]);
        }
        // -0 and +0 order as one value; only the thresholds below matter
        const int status = (kmax >= 0xFF80u || kmin < 0x007Fu) ? kNonfinite : (kmax == 0x007Fu ? kEmpty : 0);
        write_error_row(a.info + task.slot, key_value(kmax == 0x7FFFu ? 0x8000u : kmax), -1, status, task.temp);
    }
    __syncthreads();
}

// Canonical order keys of both bf16 halves of a word (-0 as +0: the raw key
// 0x7FFF becomes 0x8000, no carry across the halves).
__device__ __forceinline__ uint32_t keys2_canon(uint32_t w)
{
    const uint32_t k = keys2_raw(w);
    const uint32_t t = k ^ 0x7FFF7FFFu;   // zero halves where the key is -0's
    const uint32_t z = ~(((t & 0x7FFF7FFFu) + 0x7FFF7FFFu) | t) & 0x80008000u;
    return k + (z >> 15);
}

// A greedy row of chain verification on the histogram path: one streaming
// pass for the first largest value (-0 as +0, lowest index among equals) and
// the status (NaN or +inf; a row of nothing but -inf is fine for greedy), and
// the record the one-pass kernel writes for a greedy row.  Returns the argmax
// in thread 0.
__device__ __noinline__ int argmax_row(WideSmem& sm, const RowsArgs& a, const RowTask& task)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint16_t* row = (const uint16_t*)a.tgt + (size_t)task.row * (size_t)a.stride_t;
    const int V = a.vocab;
    unsigned long long best = 0ull;   // composite: key << 32 | ~index
    uint32_t lo = 0xFFFFFFFFu;        // smallest key (both halves)
    auto one = [&](int i) {
        const uint32_t k = keys2_canon(row[i]) & 0xFFFFu;
        const unsigned long long c = ((unsigned long long)k << 32) | (0xFFFFFFFFu - (uint32_t)i);
        best = c > best ? c : best;
        lo = min_u16x2(lo, k | 0xFFFF0000u);
    };
    const int head = min(V, (int)(((16u - ((uint32_t)(uintptr_t)row & 15u)) & 15u) >> 1));
    const int nvec = (V - head) >> 3;
    const int tail0 = head + 8 * nvec;
    if (tid < head) one(tid);
    if (tail0 + tid < V) one(tail0 + tid);
    const uint4* vp = reinterpret_cast<const uint4*>(row + head);
    uint32_t best_key = 0u;   // this thread's largest key so far (its vectors come in index order)
    for (int v0 = tid; v0 < nvec; v0 += kWideThreads * kWideUnroll) {
        uint4 x[kWideUnroll];
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u) {
            const int vi = v0 + u * kWideThreads;
            x[u] = vi < nvec ? __ldcs(vp + vi) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u) {
            const int vi = v0 + u * kWideThreads;
            if (vi < nvec) {
                const uint32_t k0 = keys2_canon(x[u].x), k1 = keys2_canon(x[u].y), k2 = keys2_canon(x[u].z),
                               k3 = keys2_canon(x[u].w);
                lo = min_u16x2(lo, min_u16x2(min_u16x2(k0, k1), min_u16x2(k2, k3)));
                const uint32_t mx = max_u16x2(max_u16x2(k0, k1), max_u16x2(k2, k3));
                const uint32_t vmax = max(mx & 0xFFFFu, mx >> 16);
                if (vmax > best_key) {   // the vector's first element holding it
                    best_key = vmax;
                    const int jj = (k0 & 0xFFFFu) == vmax ? 0
                                   : (k0 >> 16) == vmax   ? 1
                                   : (k1 & 0xFFFFu) == vmax ? 2
                                   : (k1 >> 16) == vmax   ? 3
                                   : (k2 & 0xFFFFu) == vmax ? 4
                                   : (k2 >> 16) == vmax   ? 5
                                   : (k3 & 0xFFFFu) == vmax ? 6
                                                            : 7;
                    const int idx = head + 8 * vi + jj;
                    const unsigned long long c = ((unsigned long long)vmax << 32) | (0xFFFFFFFFu - (uint32_t)idx);
                    best = c > best ? c : best;
                }
            }
        }
    }
    best = warp_max_u64(best);
    uint32_t kmin = __reduce_min_sync(0xFFFFFFFFu, min(lo & 0xFFFFu, lo >> 16));
    if (lane == 0) {
        sm.red64[warp] = best;
        sm.redi[warp] = (int)kmin;
    }
    __syncthreads();
    int amax = 0;
    if (tid == 0) {
        for (int w = 0; w < kWideThreads / 32; ++w) {
            best = sm.red64[w] > best ? sm.red64[w] : best;
            kmin = min(kmin, (uint32_t)sm.redi[w]);
        }
        const uint32_t kmax = (uint32_t)(best >> 32);
        amax = (int)(0xFFFFFFFFu - (uint32_t)best);
        const float m = (float)key_value(kmax);
        const int status = (kmax >= 0xFF80u || kmin < 0x007Fu) ? kNonfinite : 0;
        RowInfo* info = a.info + task.slot;
        info->desc.max_logit = m;
        info->desc.argmax = amax;
        info->desc.status = status;
        info->desc.temperature = task.temp;
        info->desc.log_norm = 0.0f;
        info->desc.cutoff_logit = m;
        info->cut_count = -1;
        if (status) {
            info->desc.cutoff_ties = 0;
            info->desc.kept = 0;
            info->p_token = nan("");
            info->z = 0.0;
            info->n_list = -1;
        } else {
            info->desc.cutoff_ties = 1;
            info->desc.kept = 1;
            info->p_token = task.token >= 0 ? (task.token == amax ? 1.0 : 0.0) : nan("");
            info->z = 1.0;
            info->z_rest = 0.0;
            info->n_list = 1;
            info->list_idx[0] = amax;
            info->list_p[0] = 1.0;
        }
    }
    __syncthreads();
    return amax;
}

// Both rows of position j of request r are done (lazy chain verify): the
// acceptance test the chain walk will make at j, made now; a rejection
// lowers the request's known first rejection.  Thread 0 only.
__device__ __noinline__ void decide_position(const RowsArgs& a, int r, int j)
{
    const ChainArgs& c = a.chain;
    const double p = __ldcg(&a.info[slot_target(r, c.K, j)].p_token);
    const double q = __ldcg(&draft_info(c, r, j).p_token);
    const double u = uniform_f64(c.seed, (uint32_t)r, (uint32_t)j, 0u);
    const bool accept = q > 0.0 ? u * q < p : p > 0.0;
    if (!accept) atomicMin(&c.req[r].first_reject, j);
}

__global__ void __launch_bounds__(kWideThreads, kWideBlocks) wide_rows_kernel(const __grid_constant__ RowsArgs a)
{
    // the counters are cleared before the wait for the kernel before this
    // one (shared memory only: it overlaps that kernel's end)
    extern __shared__ __align__(16) unsigned char smem_raw[];
    WideSmem& sm = *reinterpret_cast<WideSmem*>(smem_raw);
    const int tid = threadIdx.x;
    for (int i = tid; i < (kWideSlots + 1) * 128; i += kWideThreads) sm.cnt[i] = 0u;
    for (int i = tid; i < 512; i += kWideThreads) {
        sm.base[i] = kUnclaimed;
        sm.w.sums[i].mass = 0.0;
        sm.w.sums[i].count = 0u;
    }
    if (tid == 0) {
        sm.n_slots = 0;
        sm.ovf = 0;
    }
    pdl_enter();
    if (a.counters->n_slow == 0) return;   // no histogram rows in this batch
    __syncthreads();
    if (!a.chain.lazy) {
        const int n_tasks = a.counters->n_slow;
        for (int t = blockIdx.x; t < n_tasks; t += gridDim.x) wide_row(sm, a, a.slow_tasks.get(t), t);
        return;
    }
    // Chain verify.  When the rows all fit in one wave, each CTA takes one (in
    // task order).  Otherwise they are listed position by position across the
    // requests (slow_units: every request's rows of position 0, then of
    // position 1, ...) and the CTAs take them in that order, so the tests of the early positions are
    // decided while the later rows still wait; a row past its request's known
    // first rejection cannot change the outcome (the walk stops at the first
    // rejection, which is never above the known one) and gets the status scan
    // only.
    __shared__ int s_unit[4];
    const ChainArgs& c = a.chain;
    const int U = a.counters->n_units, K1 = c.K + 1;
    const int kinds = c.q_rows ? 1 : 2;   // rows per position (the draft's results may exist already)
    enum { kNone = 0, kFull = 1, kScan = 2 };
    if (U <= (int)gridDim.x) {   // no test is decided early then: no CTA would wait for one
        if ((int)blockIdx.x < U) {
            const RowTask task = a.slow_tasks.get(blockIdx.x);
            if (task.temp == 0.0f)
                argmax_row(sm, a, task);
            else
                wide_row(sm, a, task, blockIdx.x);
        }
        return;
    }
    for (;;) {
        if (tid == 0) {
            int mode = kNone, t = -1, r = 0, j = 0;
            const int u = atomicAdd(&a.counters->next_slow, 1);
            if (u < U) {
                const int2 e = __ldcg(&c.slow_units[u]);
                r = e.x >> 7;
                j = (e.x >> 1) & 63;
                t = e.y;
                int fr = __ldcg(&c.req[r].first_reject);
                // Wait a little while the lowest undecided test before this
                // row is being decided (one of its rows is finished): far
                // cheaper than a full pass that a rejection there would make
                // useless.  Bounded; after it the row gets its full pass as if
                // nothing were decided.
                const int32_t* done = &c.pair_done[(size_t)r * K1];
                const bool greedy = c.req[r].greedy != 0;     // its rows get the argmax scan whatever is decided
                const int kr = greedy ? 1 : kinds;           // rows per position of this request
                for (int spin = 0; spin < kDecideSpins && j <= fr && !greedy; ++spin) {
                    int i = 0;
                    while (i < j && __ldcg(done + i) > kr) ++i;   // decided positions
                    if (i == j || __ldcg(done + i) == 0) break;      // all decided, or not started
                    __nanosleep(256);
                    fr = __ldcg(&c.req[r].first_reject);
                }
                fr = __ldcg(&c.req[r].first_reject);
                mode = j > fr ? kScan : kFull;
            }
            s_unit[0] = mode;
            s_unit[1] = t;
            s_unit[2] = r;
            s_unit[3] = j;
        }
        __syncthreads();
        const int mode = s_unit[0], t = s_unit[1], r = s_unit[2], j = s_unit[3];
        __syncthreads();   // s_unit is rewritten only after every thread has read it
        if (mode == kNone) break;
        const RowTask task = a.slow_tasks.get(t);
        if (task.temp == 0.0f) {   // a greedy row: the argmax scan, then its test (draft token == argmax)
            const int amax = argmax_row(sm, a, task);
            if (tid == 0 && j < c.req[r].v) {
                if (c.draft_tokens[(size_t)r * c.K + j] != amax) atomicMin(&c.req[r].first_reject, j);
                __threadfence();
                atomicAdd(&c.pair_done[(size_t)r * K1 + j], 2);   // above one row: decided
            }
            continue;
        }
        if (mode == kScan) {
            scan_row(sm, a, task);
            continue;
        }
        const bool ovf = wide_row(sm, a, task, t);
        if (tid == 0 && !ovf && j < c.req[r].v) {   // a handed-on row decides nothing
            __threadfence();
            if (atomicAdd(&c.pair_done[(size_t)r * K1 + j], 1) == kinds - 1) {
                __threadfence();
                decide_position(a, r, j);
                __threadfence();
                atomicAdd(&c.pair_done[(size_t)r * K1 + j], 1);   // kinds + 1: decided
            }
        } else if (tid == 0 && ovf && j < c.req[r].v) {
            // a handed-on row leaves the position's test to the chain kernel:
            // mark it so that no later row of the request waits for it here
            atomicAdd(&c.pair_done[(size_t)r * K1 + j], kinds + 1);
        }
    }
}

}  // namespace

// Every histogram row goes to the one-CTA kernel; the rows it hands on (more
// occupied binades than it has counters for) go to the cluster kernel, which
// finds their number on the device.
int hist_wide_grid(int num_sms)
{
    int dev = 0;
    cudaGetDevice(&dev);
    static int wide_blocks[128] = {0};   // CTAs per SM, once per device (before any graph capture)
    int& nb = wide_blocks[(dev >= 0 && dev < 128) ? dev : 0];
    if (nb == 0) {
        const size_t smem = sizeof(WideSmem);
        if (cudaFuncSetAttribute(wide_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return 0;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, wide_rows_kernel, kWideThreads, smem) != cudaSuccess)
            return 0;
        nb = n < 1 ? 1 : n;
    }
    return num_sms * nb;
}

cudaError_t launch_hist_rows(const RowsArgs& a, cudaStream_t s)
{
    int dev = 0;
    cudaGetDevice(&dev);
    const int di = (dev >= 0 && dev < 128) ? dev : 0;
    cudaError_t err = cudaSuccess;
    {
        const int grid = hist_wide_grid(a.num_sms);
        if (grid < 1) return cudaErrorUnknown;
        err = launch_pdl(wide_rows_kernel, dim3(grid), dim3(kWideThreads), sizeof(WideSmem), s, a);
        if (err != cudaSuccess) return err;
    }
    int C = (a.vocab + kHistMaxSlice - 1) / kHistMaxSlice;
    if (C < 1) C = 1;
    if (C > kMaxCluster) return cudaErrorInvalidValue;
    int slice = (a.vocab + C - 1) / C;
    slice = (slice + 7) & ~7;
    if (slice > kHistMaxSlice) slice = kHistMaxSlice & ~7;
    const size_t smem = sizeof(HistSmem);
    static int attr_set[128] = {0};   // once per device, before any graph capture
    if (!attr_set[di]) {
        err = cudaFuncSetAttribute(hist_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        attr_set[di] = 1;
    }
    int n_clusters = a.num_sms / C;
    if (n_clusters < 1) n_clusters = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_clusters * C), 1, 1);
    cfg.blockDim = dim3(kHistThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    pdl_attr(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, hist_rows_kernel, a, slice);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace sv
