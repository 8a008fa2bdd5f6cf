// sv_hist.cu -- exact per-value histogram kernel for sampling rows whose kept
// set can be large (top-k off or above 32, with or without top-p).
//
// The target distribution of jianc99/sglang PR #8 ("build_speculative_verify_
// target_probs") needs, for top-p, the mass-ordered cutoff over the whole
// vocabulary.  A bf16 logit takes one of 65,536 values, so the row's multiset
// of values is its histogram over the 16-bit order key, and every quantity of
// the transform follows from it exactly: the mass of a value is its count
// times exp((v - m) / T), computed once per distinct value in fp64.
//
// One thread-block cluster handles one row at a time.  Each CTA streams its
// slice (<= 65,535 elements, so a 16-bit counter cannot wrap) from HBM once
// and counts keys in a 128 KB shared-memory histogram (two 16-bit counters
// per word).  The cluster then works only on occupied binades (the 128 keys
// of one sign+exponent): the CTAs sum their counters through distributed
// shared memory, turn counts into fp64 masses (one exp per binade and a
// geometric recurrence along the mantissa), and the first CTA walks binades
// and then keys from the top to the top-k and top-p cutoffs.  Only the
// probability of the row's own token may need one more look at the row (the
// rank of a tied token at the cutoff).
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

struct RowPlan {               // decided by CTA 0, read by the others
    int skip;                  // 1: row is an error or done
    int need_tie;              // 1: run the tie-rank pass
    uint32_t cut_key;
    int token;
};

struct WalkState {             // CTA 0's walk, phase to phase
    double z_all, z1, mk_bin, mass_above_bk, mass_above_bp, z;
    uint32_t cnt_above_bk, k_key, k_ties, cut_key, cut_ties, kept;
    int bk, bp, bmin, found, done, slot;
};

struct HistSmem {
    uint32_t hist[kHistWords];
    BinSum sums[512];
    uint32_t occ[16];
    uint32_t occ_all[16];
    int occ_list[512];
    int n_occ;
    CtaRes res;
    RowPlan plan;
    unsigned long long red64[kHistThreads / 32];
    int redi[kHistThreads / 32];
    uint32_t kc[2][128];       // per-key counts of up to two binades (walk)
    uint32_t csc[kHistThreads][33];   // per-thread key counts of one binade quarter
    double ke[2][128];         // per-key masses exp((v - m) / T)
    WalkState walk;
};

// 16-bit counter of key k in a histogram.
__device__ __forceinline__ uint32_t hist_count(const uint32_t* h, uint32_t k)
{
    const uint32_t w = h[k >> 1];
    return (k & 1u) ? (w >> 16) : (w & 0xFFFFu);
}

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

// Per-key counts (summed over the cluster) and masses of binade b into slot s
// of the walk scratch.  Run by threads 0..3 of CTA 0 (32 keys each).
__device__ void load_binade_keys(cg::cluster_group& cluster, HistSmem& sm, int C, int b, int s, double m, double T)
{
    const int q = threadIdx.x;
    if (q >= 4) return;
    if (b < 0 || b > 511) {
        for (int j = 0; j < 32; ++j) {
            sm.kc[s][32 * q + j] = 0u;
            sm.ke[s][32 * q + j] = 0.0;
        }
        return;
    }
    uint32_t c[32];
    cluster_counts32(cluster, sm, C, b, q, c);
#pragma unroll
    for (int j = 0; j < 32; ++j) sm.kc[s][32 * q + j] = c[j];
    for_binade_masses32(b, q, m, T, [&](int j, double e) { sm.ke[s][32 * q + j] = e; });
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
            sm.sums[i].mass = 0.0;
            sm.sums[i].count = 0u;
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
        BinSum* sums0 = cluster.map_shared_rank(sm.sums, 0);
        const int q4 = tid & 3;
        const int n_mine = n_occ > rank ? (n_occ - rank + C - 1) / C : 0;
        for (int i0 = (tid >> 2) - (lane >> 2); i0 < n_mine; i0 += kHistThreads / 4) {
            const int i = i0 + (lane >> 2);
            const bool act = i < n_mine;
            const int b = act ? sm.occ_list[rank + C * i] : 0;
            uint32_t csum = 0u;
            double mass = 0.0;
            if (act) {
                uint32_t c[32];
                cluster_counts32(cluster, sm, C, b, q4, c);
#pragma unroll
                for (int j = 0; j < 32; ++j) csum += c[j];
                if (csum) {
                    // counts go to shared scratch so the mass loop indexes them freely
                    uint32_t* cs = sm.csc[tid];
#pragma unroll
                    for (int j = 0; j < 32; ++j) cs[j] = c[j];
                    for_binade_masses32(b, q4, m, T, [&](int j, double e) { mass += (double)cs[j] * e; });
                }
            }
            // fixed-order reduction over the 4 threads of each binade
#pragma unroll
            for (int o = 2; o; o >>= 1) {
                mass += __shfl_xor_sync(0xFFFFFFFFu, mass, o, 4);
                csum += __shfl_xor_sync(0xFFFFFFFFu, csum, o, 4);
            }
            if (act && q4 == 0) {
                sums0[b].mass = mass;
                sums0[b].count = csum;
            }
        }
    }
    cluster.sync();

    // 6. CTA 0: walk binades and keys from the top to the cutoffs.  Binade
    //    scans run on warp 0, key walks on thread 0 (fp64 is scarce), and the
    //    decisions travel through shared memory between phases.
    if (rank == 0) {
        WalkState& W = sm.walk;
        const int kk = task.k_eff;
        const bool topk_on = kk < a.vocab;
        if (tid == 0) {
            sm.plan.skip = status != 0;
            sm.plan.need_tie = 0;
            sm.plan.token = task.token;
        }
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
        if (status == 0 && topk_on) load_binade_keys(cluster, sm, C, W.bk, 0, m, T);
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
        const bool topp_on = task.top_p < 1.0f;
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
        // Phase E: keys of the binade that holds the final cutoff (slot 1).
        int load_b = -1;
        if (status == 0) {
            if (W.found)
                load_b = (topk_on && W.bp == W.bk) ? -1 : W.bp;
            else if (!topk_on)
                load_b = W.bmin;
        }
        if (load_b >= 0) load_binade_keys(cluster, sm, C, load_b, 1, m, T);
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
                    info->p_token = kd >= cut_key ? exp((key_value(kd) - m) / T) / z : 0.0;
                }
            } else {
                info->p_token = nan("");
            }
        }
    }
    cluster.sync();

    // 7. tie rank of the row's token inside a partial tie group
    const RowPlan plan = *cluster.map_shared_rank(&sm.plan, 0);
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
            info->desc.max_logit = (float)m;
            info->desc.log_norm = 0.0f;
            info->desc.cutoff_logit = (float)m;
            info->desc.cutoff_ties = 0;
            info->desc.kept = 0;
            info->desc.argmax = argmax;
            info->desc.status = status;
            info->desc.temperature = task.temp;
            info->p_token = nan("");
            info->z = 0.0;
            info->n_list = -1;
            info->cut_count = 0;
        } else if (plan.need_tie) {
            int rank_d = 0;
            for (int r = 0; r < C; ++r) rank_d += cluster.map_shared_rank(&sm.res, r)->tie_count;
            const bool keep = rank_d < info->desc.cutoff_ties;
            info->p_token = keep ? exp((key_value(plan.cut_key) - m) / T) / info->z : 0.0;
        }
    }
    cluster.sync();   // the histograms may be cleared for the next row
}

__global__ void __launch_bounds__(kHistThreads, 1) hist_rows_kernel(RowsArgs a, int slice)
{
    pdl_enter();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    HistSmem& sm = *reinterpret_cast<HistSmem*>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int cluster_id = blockIdx.x / C;
    const int n_clusters = gridDim.x / C;
    const int n_tasks = a.counters->n_slow;
    for (int t = cluster_id; t < n_tasks; t += n_clusters) {
        const RowTask task = a.slow_tasks.get(t);
        hist_row(cluster, sm, a, task, C, rank, slice);
    }
}

}  // namespace

cudaError_t launch_hist_rows(const RowsArgs& a, cudaStream_t s)
{
    int C = (a.vocab + kHistMaxSlice - 1) / kHistMaxSlice;
    if (C < 1) C = 1;
    if (C > kMaxCluster) return cudaErrorInvalidValue;
    int slice = (a.vocab + C - 1) / C;
    slice = (slice + 7) & ~7;
    if (slice > kHistMaxSlice) slice = kHistMaxSlice & ~7;
    const size_t smem = sizeof(HistSmem);
    static int attr_set[128] = {0};   // once per device, before any graph capture
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t err = cudaSuccess;
    if (dev < 0 || dev >= 128 || !attr_set[dev]) {
        err = cudaFuncSetAttribute(hist_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < 128) attr_set[dev] = 1;
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
