// sv_resample.cu -- full-row resample of the emitted token when the kept set
// is not listed (more than 32 tokens): the residual max(0, p_a - q_a) at the
// first rejection, or p at the bonus position (the "Identical rejection
// scheme" of local-inference-lab/rtx6kpro dspark-upstream-consolidation.md).
//
// Weights are exact fixed-point numbers, p and q times 2^62, floored, so
// sums of them do not depend on the order of summation.  The token is the
// first index, in index order, where the running sum passes floor(W * u) for
// the job's uniform u(r, a, 1).  Elements tied at a partially kept cutoff are
// kept in index order up to the row's cutoff_ties.
//
// The weight of a key comes from a per-binade table in shared memory (fp64
// exp((v - m) / T) / Z along the binade's mantissa, then floored), built for
// the kept binades of magnitude 2^-6 and up, where ordinary logits sit; keys
// below the one whose weight floors to 0 weigh 0; any other kept key (small
// magnitudes, or binades beyond the table) gets its own fp64 exp.
//
// Every row is cut into tiles, eight tiles (one per warp) to a chunk, and the
// chunks of all jobs are spread over a persistent grid.  A warp streams its
// tiles of p's and q's rows once, straight from global memory, and leaves
// each tile's sums, with the tied elements summed in each of their possible
// states.  The CTA that finishes a job's last chunk combines the sums,
// rescans in index order the (at most two) tiles where a tie group's kept
// part ends, and then the one tile that holds the target, to find the token.
#include <math.h>

#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr double kFix = 4611686018427387904.0;   // 2^62
constexpr float kFix62f = 4611686018427387904.0f;  // the same as a float
constexpr int kSmallLo = 135, kSmallHi = 377;      // binades of |v| < 2^-6 (both signs, and the zeros)

struct Dist {                 // one row's distribution, as the weight passes need it
    const uint16_t* row;
    double m, T, z;
    uint32_t cut_key;         // smallest kept key
    uint32_t zero_key;        // keys below it weigh 0 (p < 2^-62)
    int ties;                 // kept ties at the cutoff
    int partial;              // ties < tokens at the cutoff: ranks are needed
    int16_t* map;             // binade -> table slot, -1: weight computed per key
    unsigned long long* tab;
    unsigned long long wfix;  // p's weight in the residual (64-bit fraction; 0: none)
};

// p's weight applied to a fixed-point probability: floor(wp w).
__device__ __forceinline__ unsigned long long pweight(const Dist& P, unsigned long long wp)
{
    return P.wfix ? __umul64hi(wp, P.wfix) : wp;
}

__device__ __forceinline__ unsigned long long fix_of(double p)
{
    const unsigned long long x = __double2ull_rd(p * kFix);   // floor; 0 for p <= 0
    return x < (1ull << 62) ? x : (1ull << 62);
}

// A key outside the tables: its own fp64 exp (out of line: rare, and it keeps
// the streaming loops small).
__device__ __noinline__ unsigned long long fixp_exp(double m, double T, double z, uint32_t key)
{
    return fix_of(exp((key_value(key) - m) / T) / z);
}

// 62-bit fixed-point probability of a key under a distribution (kept test
// done by the caller).
__device__ __forceinline__ unsigned long long fixp(const Dist& D, uint32_t key)
{
    if (key < D.zero_key) return 0ull;
    const int s = D.map[key >> 7];
    if (s >= 0) return D.tab[s * 128 + (key & 127u)];
    return fixp_exp(D.m, D.T, D.z, key);
}

__device__ __forceinline__ bool kept_key(const Dist& D, uint32_t key, int tie_rank)
{
    return key > D.cut_key || (key == D.cut_key && tie_rank < D.ties);
}

// Key below which every weight floors to 0: values under m + T (ln Z - 62 ln 2),
// less two keys for the roundings of the bound.  The bound is taken in fp32,
// an error of about 1e-5 T + 1e-7 |m| (ln Z <= 22, 62 ln 2 and their
// difference each within an fp32 rounding, then the product and the sum),
// while two keys span at least |v0| / 128; the bound is 0 where that margin
// would not cover the error with room to spare.
__device__ __forceinline__ uint32_t zero_key_of(float m, float T, double z)
{
    const float v0 = m + T * (logf((float)z) - 62.0f * (float)kLn2);
    if (!(fabsf(v0) > 2e-3f * T + 1e-4f * fabsf(m)) || !(v0 > -3.0e38f)) return 0u;
    const uint32_t k = key16_of_bf16(__float_as_uint(v0) >> 16);
    return k >= 2u ? k - 2u : 0u;
}

constexpr int kResThreads = 256;
constexpr int kResWarps = kResThreads / 32;
constexpr int kResBinades = 48;    // table slots, p's and q's binades together
constexpr int kResTile = kResampleTile;
constexpr int kResStep = 512;        // elements a warp loads at a time (two 16-byte vectors per lane and row)
constexpr int kResCostJobs = 2048;   // jobs up to which the chunks are split by estimated cost
constexpr int kResCostBase = 120;    // a chunk's fixed part, in units of one candidate's gathering and weighing
constexpr int kResWarpBuf = kResStep + 64;   // candidates a warp gathers before weighing them
static_assert(kResampleTile == kResThreads * 8, "a rescanned tile is at most eight elements per thread");
static_assert((kResTile / 2) % kResStep == 0, "a tile is whole steps");

struct ResSmem {
    unsigned long long buf[kResWarps * kResWarpBuf];   // per warp: its candidates, then (rescan) their weights
    unsigned long long tab[kResBinades * 128];
    dfloat ratio[kResBinades];                      // per slot: exp(step / T) along the binade (0: one exp per key)
    dfloat exp_tab[64];                             // 2^(j / 64) for the double-float exp
    uint32_t zkey[2];                               // the loaded job's zero keys of p and q
    dfloat inv_z[2];                                // and 1 / Z of each
    int16_t map[2][512];
    int slot_bin[kResBinades];
    int slot_dist[kResBinades];
    int cur_job;      // job whose tables are loaded (-1: none)
    int last;         // this CTA finished the job's last chunk
    int found;        // token found by the target search (-1: not yet)
    int halt;         // the target search is over
    unsigned long long scan[kResThreads / 32];
    unsigned long long tacc[kResWarps][kTsTiesP - kTsTieRes];   // per warp: its tile's tied-element sums
    // the combine
    unsigned long long ex_res[2], ex_p[2];   // exact sums of the tiles where a tie group's kept part ends
    int ex_tile[2], ex_off_p[2], ex_off_q[2];
    int n_ex;
    int found_tile, tile_off_p, tile_off_q;  // the tile that holds the target
    unsigned long long tile_target;
};

// Binades of a range that may hold a table: not binade 0 (-inf and negative
// NaN) and not of small magnitude.  Count of them in [x, y).
__device__ __forceinline__ int tabled_in(int x, int y)
{
    if (y <= x) return 0;
    int n = y - x;
    const int t0 = max(x, kSmallLo), t1 = min(y, kSmallHi);
    if (t1 > t0) n -= t1 - t0;
    if (x == 0) n -= 1;
    return n;
}

// The job's p row (target logits at its position) and q row (draft logits).
__device__ __forceinline__ const uint16_t* job_p_row(const ChainArgs& a, int r, int pa)
{
    const int64_t trow = a.layout == 1 ? (int64_t)a.qo_indptr[r] + pa : (int64_t)r * (a.K + 1) + pa;
    return (const uint16_t*)a.tgt + (size_t)trow * (size_t)a.stride_t;
}
__device__ __forceinline__ const uint16_t* job_q_row(const ChainArgs& a, int r, int pa)
{
    return (const uint16_t*)a.drf + ((size_t)r * a.K + pa) * (size_t)a.stride_d;
}

// The job's p and q as the weight passes need them (tables in shared memory;
// the zero keys are those load_tables found for the loaded job).
__device__ __forceinline__ void job_dists(const ChainArgs& a, const ResampleJob& job, ResSmem& sm, Dist& P, Dist& Q)
{
    const int r = job.req, pa = job.a, K = a.K;
    const RowInfo& IP = a.info[slot_target(r, K, pa)];
    const RowInfo& IQ = draft_info(a, r, pa);
    P.row = job_p_row(a, r, pa);
    P.m = IP.desc.max_logit;
    P.T = IP.desc.temperature;
    P.z = IP.z;
    P.cut_key = key16_of_bf16(__float_as_uint(IP.desc.cutoff_logit) >> 16);
    P.zero_key = sm.zkey[0];
    P.ties = IP.desc.cutoff_ties;
    P.partial = IP.desc.cutoff_ties < IP.cut_count;
    P.map = sm.map[0];
    P.tab = sm.tab;
    P.wfix = job.wfix;
    Q = P;
    if (job.residual) {
        Q.row = job_q_row(a, r, pa);
        Q.m = IQ.desc.max_logit;
        Q.T = IQ.desc.temperature;
        Q.z = IQ.z;
        Q.cut_key = key16_of_bf16(__float_as_uint(IQ.desc.cutoff_logit) >> 16);
        Q.zero_key = sm.zkey[1];
        Q.ties = IQ.desc.cutoff_ties;
        Q.partial = IQ.desc.cutoff_ties < IQ.cut_count;
        Q.map = sm.map[1];
    }
}

// Tables of the job's kept binades that may hold one, from the top binade of
// each distribution down, p's first; q keeps at least half of the slots when
// it needs them.  Every thread calls it.
__device__ void load_tables(ResSmem& sm, Dist& P, Dist& Q, bool residual)
{
    const int tid = threadIdx.x;
    if (tid < 2) {   // once per distribution for the whole CTA (lane 0: p, lane 1: q)
        const Dist& D = tid ? Q : P;   // q is p in p's own draw
        sm.zkey[tid] = zero_key_of((float)D.m, (float)D.T, D.z);
        sm.inv_z[tid] = df_recip(D.z);
    }
    __syncthreads();
    P.zero_key = sm.zkey[0];
    Q.zero_key = sm.zkey[1];
    const int hiP = (int)(key16_of_bf16(__float_as_uint((float)P.m) >> 16) >> 7);
    const int loP = (int)(max(P.cut_key, P.zero_key) >> 7);
    const int hiQ = (int)(key16_of_bf16(__float_as_uint((float)Q.m) >> 16) >> 7);
    const int loQ = (int)(max(Q.cut_key, Q.zero_key) >> 7);
    const int nP = tabled_in(loP, hiP + 1);
    const int nQ = residual ? tabled_in(loQ, hiQ + 1) : 0;
    const int capP = min(nP, kResBinades - min(nQ, kResBinades / 2));
    const int capQ = min(nQ, kResBinades - capP);
    for (int b = tid; b < 512; b += kResThreads) {
        const bool tb = b != 0 && (b < kSmallLo || b >= kSmallHi);
        int sP = -1, sQ = -1;
        if (tb && b >= loP && b <= hiP) {
            const int above = tabled_in(b + 1, hiP + 1);
            if (above < capP) sP = above;
        }
        if (residual && tb && b >= loQ && b <= hiQ) {
            const int above = tabled_in(b + 1, hiQ + 1);
            if (above < capQ) sQ = capP + above;
        }
        sm.map[0][b] = (int16_t)sP;
        sm.map[1][b] = (int16_t)sQ;
        if (sP >= 0) {
            sm.slot_bin[sP] = b;
            sm.slot_dist[sP] = 0;
        }
        if (sQ >= 0) {
            sm.slot_bin[sQ] = b;
            sm.slot_dist[sQ] = 1;
        }
    }
    __syncthreads();
    // the step ratio of each slot's binade, then 8 keys per thread: one exp,
    // a geometric recurrence along the mantissa, a product with 1 / Z -- in
    // double-float arithmetic (about 2^-46; the fp64 pipe would make these
    // tables a large part of a job's time)
    for (int sl = tid; sl < capP + capQ; sl += kResThreads) {
        const Dist& D = sm.slot_dist[sl] ? Q : P;
        const uint32_t kb = (uint32_t)sm.slot_bin[sl] * 128u;
        const float T = (float)D.T;
        const dfloat x = scaled_logit(f32_of_key16(kb + 1u), f32_of_key16(kb), T, 1.0f / T);   // step / T >= 0
        sm.ratio[sl] = x.hi <= 1.0f ? exp_df(x, sm.exp_tab) : dfloat{0.0f, 0.0f};
    }
    __syncthreads();
    const dfloat inv_zp = sm.inv_z[0], inv_zq = sm.inv_z[1];
    for (int item = tid; item < (capP + capQ) * 16; item += kResThreads) {
        const int sl = item >> 4, g = item & 15;
        const bool isq = sm.slot_dist[sl] != 0;
        const Dist& D = isq ? Q : P;
        const uint32_t k0 = (uint32_t)sm.slot_bin[sl] * 128u + 8u * (uint32_t)g;
        const dfloat R = sm.ratio[sl], inv_z = isq ? inv_zq : inv_zp;
        const float m = (float)D.m, T = (float)D.T, inv_t = 1.0f / T;
        unsigned long long* out = sm.tab + sl * 128 + 8 * g;
        if (R.hi > 0.0f) {
            dfloat cur = exp_df(scaled_logit(f32_of_key16(k0), m, T, inv_t), sm.exp_tab);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                out[j] = fix_df(df_mul(cur, inv_z), kFix62f);
                cur = df_mul(cur, R);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                out[j] = fix_df(df_mul(exp_df(scaled_logit(f32_of_key16(k0 + j), m, T, inv_t), sm.exp_tab), inv_z),
                                kFix62f);
        }
    }
    __syncthreads();
}

// Canonical keys of eight consecutive elements of a row (x0 .. x0 + 7, those
// at or past x_end read as -inf, which no kept set holds).
__device__ __forceinline__ void load_keys8(const uint16_t* row, int x0, int x_end, bool vec_ok, uint32_t k[8])
{
    if (vec_ok && x0 + 8 <= x_end) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + x0));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            k[2 * i] = key16_of_bf16(w[i] & 0xFFFFu);
            k[2 * i + 1] = key16_of_bf16(w[i] >> 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) k[i] = x0 + i < x_end ? key16_of_bf16(row[x0 + i]) : 0x007Fu;
    }
}

// Eight consecutive elements as raw bf16 pairs (x0 .. x0 + 7, those at or
// past x_end read as -inf).
__device__ __forceinline__ uint4 load_raw8(const uint16_t* row, int x0, int x_end, bool vec_ok)
{
    if (vec_ok && x0 + 8 <= x_end) return __ldg(reinterpret_cast<const uint4*>(row + x0));
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = x0 + 2 * i < x_end ? row[x0 + 2 * i] : 0xFF80u;
        const uint32_t hi = x0 + 2 * i + 1 < x_end ? row[x0 + 2 * i + 1] : 0xFF80u;
        w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Elements among eight (four words of raw key pairs) whose canonical key is
// `cut` (a canonical key: at +0 the raw keys of -0 count too).
__device__ __forceinline__ int ties8(const uint32_t r[4], uint32_t cut)
{
    const uint32_t c2 = cut * 0x10001u;
    int n = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) n += zero_halves(r[i] ^ c2);
    if (cut == 0x8000u)
#pragma unroll
        for (int i = 0; i < 4; ++i) n += zero_halves(r[i] ^ 0x7FFF7FFFu);
    return n;
}

// Bit i set for element i among eight (four words of raw key pairs) whose
// canonical key is at least `cut` (a canonical key).  Raw keys order as the
// canonical ones do except -0, one below +0: at a cut of +0 the raw test
// starts one lower.
__device__ __forceinline__ uint32_t at_least8(const uint32_t r[4], uint32_t cut)
{
    const uint32_t c2 = (cut == 0x8000u ? 0x7FFFu : cut) * 0x10001u;
    uint32_t below = 0u;   // bits 15 + 2w and 31 + 2w: the half of word w is below the cut
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t d = max_u16x2(r[w], c2) ^ r[w];   // a half is 0 where it is at least the cut
        const uint32_t nz = (((d & 0x7FFF7FFFu) + 0x7FFF7FFFu) | d) & 0x80008000u;
        below |= nz >> (15 - 2 * w);
    }
    below |= below >> 15;   // word w's high half from bit 16 + 2w to bit 1 + 2w
    return ~below & 0xFFu;
}

// Element i's raw p key (low half) and raw q key (high half) from a word of
// each.
__device__ __forceinline__ uint32_t pair_raw(const uint32_t rp[4], const uint32_t rq[4], int i)
{
    uint32_t x;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(x) : "r"(rp[i >> 1]), "r"(rq[i >> 1]), "r"((i & 1) ? 0x7632u : 0x5410u));
    return x;
}

__device__ __forceinline__ uint32_t canon16(uint32_t k) { return k == 0x7FFFu ? 0x8000u : k; }

__device__ __forceinline__ unsigned long long sat_sub(unsigned long long x, unsigned long long y)
{
    return x > y ? x - y : 0ull;
}

// Sum of x over the CTA (every thread gets it).
__device__ __forceinline__ unsigned long long block_sum_u64(ResSmem& sm, unsigned long long x)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x = warp_sum_u64(x);
    __syncthreads();
    if (lane == 0) sm.scan[warp] = x;
    __syncthreads();
    unsigned long long t = 0ull;
#pragma unroll
    for (int w = 0; w < kResThreads / 32; ++w) t += sm.scan[w];
    return t;
}

// Exclusive prefix of x over the CTA in thread order, and the total.
__device__ __forceinline__ unsigned long long block_excl_u64(ResSmem& sm, unsigned long long x,
                                                             unsigned long long& total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) sm.scan[warp] = incl;
    __syncthreads();
    unsigned long long before = 0ull;
    total = 0ull;
#pragma unroll
    for (int w = 0; w < kResThreads / 32; ++w) {
        const unsigned long long t = sm.scan[w];
        before += w < warp ? t : 0ull;
        total += t;
    }
    return before + incl - x;
}

// A warp's candidates of one tile, packed into its part of sm.buf in lane
// order: the elements of mask `cm` (bit i: element i of the lane's eight),
// each as pack(i).  Returns the warp's count.
template <typename Pack>
__device__ __forceinline__ int compact8(unsigned long long* wb, uint32_t cm, Pack pack)
{
    const int lane = threadIdx.x & 31;
    const uint32_t nm = (uint32_t)__popc(cm), below = (1u << lane) - 1u;
    int pos = 0, total = 0;   // the lanes' counts (0 .. 8) summed bit by bit: four independent ballots
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (nm >> k) & 1u);
        pos += __popc(b & below) << k;
        total += __popc(b) << k;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if ((cm >> i) & 1u) wb[pos++] = pack(i);
    __syncwarp();
    return total;
}

// One tile in index order with the exact tie ranks (thread i: elements
// t0 + 8 i .. + 7; run_p / run_q ties before the tile): the residual and p
// sums (mode 0), or the index where the running sum of the chosen weights
// passes `target` (mode 1; -1 if it does not within the tile).  Each thread
// decides its elements' kept states from their ranks; each warp then computes
// the weights of its elements kept in p, packed densely.  Every thread calls
// it.
__device__ int rescan_tile(ResSmem& sm, const Dist& P, const Dist& Q, bool residual, int t0, int x_end, int run_p,
                           int run_q, bool vec_ok, int mode, bool use_p, unsigned long long target,
                           unsigned long long& sum_res, unsigned long long& sum_p)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long* wb = sm.buf + warp * kResWarpBuf;
    const int x0 = t0 + 8 * tid;
    uint32_t kp[8], kq[8];
    load_keys8(P.row, x0, x_end, vec_ok, kp);
    if (residual)
        load_keys8(Q.row, x0, x_end, vec_ok, kq);
    else
#pragma unroll
        for (int i = 0; i < 8; ++i) kq[i] = 0u;
    if (tid == 0) sm.found = -1;
    uint32_t cp = 0u, cq = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        cp += (P.partial && kp[i] == P.cut_key) ? 1u : 0u;
        cq += (residual && Q.partial && kq[i] == Q.cut_key) ? 1u : 0u;
    }
    unsigned long long tot;
    const unsigned long long ex = block_excl_u64(sm, ((unsigned long long)cp << 32) | cq, tot);
    int rp = run_p + (int)(ex >> 32), rq = run_q + (int)(ex & 0xFFFFFFFFu);
    uint32_t inp = 0u, inq = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (kept_key(P, kp[i], rp)) inp |= 1u << i;
        if (P.partial && kp[i] == P.cut_key) ++rp;
        if (residual) {
            if (kept_key(Q, kq[i], rq)) inq |= 1u << i;
            if (Q.partial && kq[i] == Q.cut_key) ++rq;
        }
    }
    const int total = compact8(wb, inp, [&](int i) {
        return (unsigned long long)kp[i] | ((unsigned long long)kq[i] << 16) |
               ((unsigned long long)((inq >> i) & 1u) << 32) | ((unsigned long long)(lane * 8 + i) << 33);
    });
    unsigned long long wv[8];   // this lane's entries lane, lane + 32, ... (at most 8)
    int ws[8];
    unsigned long long tr = 0ull, tpp = 0ull;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int e = lane + 32 * q;
        wv[q] = 0ull;
        ws[q] = -1;
        if (e < total) {
            const unsigned long long en = wb[e];
            const uint32_t ekp = (uint32_t)(en & 0xFFFFu), ekq = (uint32_t)((en >> 16) & 0xFFFFu);
            const unsigned long long wp = fixp(P, ekp);
            const unsigned long long wr =
                residual ? sat_sub(pweight(P, wp), ((en >> 32) & 1ull) ? fixp(Q, ekq) : 0ull) : wp;
            tr += wr;
            tpp += wp;
            wv[q] = use_p ? wp : wr;
            ws[q] = (int)(en >> 33);
        }
    }
    if (mode == 0) {
        sum_res = block_sum_u64(sm, tr);
        sum_p = block_sum_u64(sm, tpp);
        __syncthreads();
        return -1;
    }
    // back to index order: each weight in its element's slot, per-thread
    // sums, the CTA's prefix, and the walk of the thread holding the crossing
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) wb[lane * 8 + i] = 0ull;
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (ws[q] >= 0) wb[ws[q]] = wv[q];
    __syncwarp();
    unsigned long long w8[8], mine = 0ull;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        w8[i] = wb[lane * 8 + i];
        mine += w8[i];
    }
    unsigned long long tile;
    const unsigned long long before = block_excl_u64(sm, mine, tile);
    if (before <= target && target < before + mine) {
        unsigned long long c = before;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c += w8[i];
            if (c > target) {
                sm.found = x0 + i;
                break;
            }
        }
    }
    __syncthreads();
    const int found = sm.found;
    __syncthreads();
    return found;
}

// This CTA's chunks [u_lo, u_hi) when the ranges are cut at equal estimated
// cost rather than equal length: a chunk costs a fixed part plus its expected
// candidates (p's kept count over the row), which the weighing loop pays for.
// Out of line: it runs once per launch.  Every thread calls it.
__device__ __noinline__ void cost_split(ResSmem& sm, const ChainArgs& a, int j0, int n_jobs, int n_units,
                                        long long& u_lo, long long& u_hi)
{
    const int tid = threadIdx.x, K = a.K, V = a.vocab, tile_len = resample_tile_len(V);
    long long C = 0, lo = 0, hi = 0;
    for (int pass = 0; pass < 2; ++pass) {   // pass 0: the total; pass 1: this CTA's bounds
        const long long x0 = C * blockIdx.x / gridDim.x, x1 = C * (blockIdx.x + 1) / gridDim.x;
        long long before = 0;
        for (int b0 = 0; b0 < n_jobs; b0 += kResThreads) {
            const int jj = b0 + tid;
            long long cost = 0;   // per chunk of job jj
            if (jj < n_jobs) {
                const ResampleJob job = a.jobs[j0 + jj];
                const int kept = __ldcg(&a.info[slot_target(job.req, K, job.a)].desc.kept);
                cost = (job.residual ? kResCostBase : kResCostBase / 2) +
                       (long long)max(kept, 0) * tile_len / max(V, 1);
            }
            unsigned long long all;
            const long long s0 = before + (long long)block_excl_u64(sm, (unsigned long long)(cost * n_units), all);
            if (pass == 1 && jj < n_jobs) {   // this job's chunks that start below each bound
                lo += min((long long)n_units, max(0ll, (x0 - s0 + cost - 1) / cost));
                hi += min((long long)n_units, max(0ll, (x1 - s0 + cost - 1) / cost));
            }
            before += (long long)all;
        }
        C = before;
    }
    unsigned long long n_lo, n_hi;
    block_excl_u64(sm, (unsigned long long)lo, n_lo);
    block_excl_u64(sm, (unsigned long long)hi, n_hi);
    u_lo = (long long)n_lo;
    u_hi = (long long)n_hi;
}

__global__ void __launch_bounds__(kResThreads, 2) resample_kernel(const __grid_constant__ ChainArgs a, int n_units, int wave)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ResSmem& sm = *reinterpret_cast<ResSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    fill_exp_table(sm.exp_tab);   // constants into shared memory: before the wait for the kernel before this one
    pdl_enter();
    const int V = a.vocab, K = a.K;
    const int n_tiles = resample_tiles(V), tile_len = resample_tile_len(V);
    // wave 0: the jobs the chain or block kernel listed; wave 1: those the
    // block finish kernel listed after them
    const int j0 = wave ? a.counters->n_jobs : 0;
    const int n_jobs = wave ? a.counters->n_jobs2 : a.counters->n_jobs;
    const long long total = (long long)n_jobs * n_units;
    long long u_lo = total * blockIdx.x / gridDim.x, u_hi = total * (blockIdx.x + 1) / gridDim.x;
    if (n_jobs <= kResCostJobs && total >= 4ll * gridDim.x) cost_split(sm, a, j0, n_jobs, n_units, u_lo, u_hi);
    if (tid == 0) sm.cur_job = -1;
    __syncthreads();
    // this CTA's chunks, one job at a time: [u, u_end) are those of job j
    for (long long u = u_lo, u_end; u < u_hi; u = u_end) {
        const int j = j0 + (int)(u / n_units);
        u_end = min(u_hi, (long long)(j - j0 + 1) * n_units);
        const int c_lo = (int)(u - (long long)(j - j0) * n_units), c_hi = c_lo + (int)(u_end - u);
        const ResampleJob job = a.jobs[j];
        const bool residual = job.residual != 0;
        Dist P, Q;
        job_dists(a, job, sm, P, Q);
        if (sm.cur_job != j) {
            load_tables(sm, P, Q, residual);
            if (tid == 0) sm.cur_job = j;
        }
        const bool vec_ok = ((uintptr_t)P.row & 15u) == 0u && (!residual || ((uintptr_t)Q.row & 15u) == 0u);
        TileSums* recs = a.tiles + (size_t)j * n_tiles;

        // 1. each warp streams its tiles of the chunks (tile c * warps + warp
        //    of chunk c), with no barrier between them: tie counts over every
        //    element, weights over the elements at or above p's cutoff (the
        //    others have p = 0 in every state), gathered densely in the warp's
        //    buffer and weighed a batch at a time; the warp writes each tile's
        //    record.  Each lane loads 16-byte vectors straight from the rows,
        //    the next step's (of this tile or the next) while it works on this
        //    one.
        {
            unsigned long long* wb = sm.buf + warp * kResWarpBuf;
            unsigned long long* tacc = sm.tacc[warp];   // elements tied at a partial cutoff: rare, summed here
            const int tile_hi = min(n_tiles, c_hi * kResWarps);
            int tile = c_lo * kResWarps + warp;
            uint4 np[2], nq[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
            auto load_step = [&](int x_step, int x_end) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int x0 = x_step + h * 256 + 8 * lane;
                    np[h] = load_raw8(P.row, x0, x_end, vec_ok);
                    if (residual) nq[h] = load_raw8(Q.row, x0, x_end, vec_ok);
                }
            };
            if (tile < tile_hi) load_step(tile * tile_len, min(V, (tile + 1) * tile_len));
            for (; tile < tile_hi; tile += kResWarps) {
                const int t0 = tile * tile_len;
                const int t_end = min(V, t0 + tile_len);
                unsigned long long base_res = 0ull, base_p = 0ull;
                int ties_p = 0, ties_q = 0;
                if (lane < kTsTiesP - kTsTieRes) tacc[lane] = 0ull;
                int nbuf = 0;
                // the weights of the gathered candidates, into acc
                auto weigh = [&]() {
                    __syncwarp();
                    for (int e = lane; e < nbuf; e += 32) {
                        const uint32_t en = (uint32_t)wb[e];
                        const uint32_t ekp = canon16(en & 0xFFFFu), ekq = canon16(en >> 16);
                        const bool tP = P.partial && ekp == P.cut_key;
                        ties_p += tP ? 1 : 0;   // p's tied elements are all candidates
                        const bool tQ = residual && Q.partial && ekq == Q.cut_key;
                        const unsigned long long wp = fixp(P, ekp);
                        const bool qk = residual && (ekq > Q.cut_key || (ekq == Q.cut_key && !Q.partial));
                        const unsigned long long wq = qk ? fixp(Q, ekq) : 0ull;
                        const unsigned long long wpw = pweight(P, wp);   // p's weighted value in the residual
                        if (!tP && !tQ) {
                            base_p += wp;
                            base_res += residual ? sat_sub(wpw, wq) : wp;
                        } else {
                            const unsigned long long wqt = tQ ? fixp(Q, ekq) : wq;
#pragma unroll
                            for (int sp_ = 0; sp_ < 2; ++sp_) {
                                const unsigned long long p_ = (tP && !sp_) ? 0ull : wp;
                                const unsigned long long pw_ = (tP && !sp_) ? 0ull : wpw;
                                atomicAdd(&tacc[kTsTieP - kTsTieRes + sp_], p_);
#pragma unroll
                                for (int sq = 0; sq < 2; ++sq) {
                                    const unsigned long long q_ = tQ ? (sq ? wqt : 0ull) : wq;
                                    atomicAdd(&tacc[2 * sp_ + sq], residual ? sat_sub(pw_, q_) : p_);
                                }
                            }
                        }
                    }
                    __syncwarp();
                    nbuf = 0;
                };
                const int t_stop = t0 + tile_len;
                for (int s0 = t0;; s0 += kResStep) {   // one weighing site: the loop body stays small
                    const bool more = s0 < t_stop;
                    if (more) {
                        const uint4 cp[2] = {np[0], np[1]}, cq[2] = {nq[0], nq[1]};
                        if (s0 + kResStep < t_stop)
                            load_step(s0 + kResStep, t_end);
                        else if (tile + kResWarps < tile_hi)   // the first step of the warp's next tile
                            load_step(t0 + kResWarps * tile_len, min(V, t0 + (kResWarps + 1) * tile_len));
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            // raw key pairs (two elements per word); most elements are
                            // below p's cutoff and need no more than the pair-wise tie
                            // counts and one packed maximum for the lane's eight
                            const uint32_t rp[4] = {keys2_raw(cp[h].x), keys2_raw(cp[h].y), keys2_raw(cp[h].z),
                                                    keys2_raw(cp[h].w)};
                            uint32_t rq[4] = {0u, 0u, 0u, 0u};   // canonical key 0 stands for q in p's own draw
                            if (residual) {
                                rq[0] = keys2_raw(cq[h].x);
                                rq[1] = keys2_raw(cq[h].y);
                                rq[2] = keys2_raw(cq[h].z);
                                rq[3] = keys2_raw(cq[h].w);
                            }
                            if (residual && Q.partial) ties_q += ties8(rq, Q.cut_key);
                            const uint32_t cm = at_least8(rp, P.cut_key);
                            if (__any_sync(0xFFFFFFFFu, cm != 0u))   // raw pairs: the weighing makes them canonical
                                nbuf += compact8(wb + nbuf, cm, [&](int i) { return (unsigned long long)pair_raw(rp, rq, i); });
                        }
                    }
                    if (!more || nbuf > kResWarpBuf - kResStep) weigh();   // room for the next step's candidates
                    if (!more) break;
                }
                base_res = warp_sum_u63(base_res);
                base_p = warp_sum_u63(base_p);
                ties_p = __reduce_add_sync(0xFFFFFFFFu, ties_p);
                ties_q = __reduce_add_sync(0xFFFFFFFFu, ties_q);
                if (lane == 0) {
                    TileSums& rec = recs[tile];
                    rec.v[kTsBaseRes] = base_res;
                    rec.v[kTsBaseP] = base_p;
#pragma unroll
                    for (int f = kTsTieRes; f < kTsTiesP; ++f) rec.v[f] = tacc[f - kTsTieRes];
                    rec.v[kTsTiesP] = (unsigned long long)ties_p;
                    rec.v[kTsTiesQ] = (unsigned long long)ties_q;
                }
                __syncwarp();   // tacc is reset for the next tile only after lane 0 read it
            }
            if (lane == 0) __threadfence();   // the warp's records, before its chunks are counted done
        }
        __syncthreads();
        if (tid == 0) sm.last = atomicAdd(&a.jobs[j].done, c_hi - c_lo) + (c_hi - c_lo) == n_units;
        __syncthreads();
        if (!sm.last) continue;
        __threadfence();

        // 2. the job's last chunk: one thread per tile record (read through
        //    L2: they come from other SMs); tie offsets and states by a scan
        const int t = tid;
        unsigned long long R[kTsFields] = {};
        if (t < n_tiles)
#pragma unroll
            for (int f = 0; f < kTsFields; ++f) R[f] = __ldcg(&recs[t].v[f]);
        if (tid == 0) {
            sm.n_ex = 0;
            sm.found_tile = -1;
        }
        unsigned long long tot;
        const unsigned long long ex = block_excl_u64(sm, (R[kTsTiesP] << 32) | R[kTsTiesQ], tot);
        const int op = (int)(ex >> 32), oq = (int)(ex & 0xFFFFFFFFu);
        const int stp = op + (int)R[kTsTiesP] <= P.ties ? 1 : (op >= P.ties ? 0 : 2);
        const int stq = oq + (int)R[kTsTiesQ] <= Q.ties ? 1 : (oq >= Q.ties ? 0 : 2);
        const bool split = t < n_tiles && (stp == 2 || stq == 2);
        if (split) {   // at most one tile for p and one for q
            const int k = atomicAdd(&sm.n_ex, 1);
            if (k < 2) {
                sm.ex_tile[k] = t;
                sm.ex_off_p[k] = op;
                sm.ex_off_q[k] = oq;
            }
        }
        __syncthreads();
        const int n_ex = min(sm.n_ex, 2);
        for (int e = 0; e < n_ex; ++e) {
            unsigned long long sr, sp_;
            rescan_tile(sm, P, Q, residual, sm.ex_tile[e] * tile_len, min(V, (sm.ex_tile[e] + 1) * tile_len),
                        sm.ex_off_p[e], sm.ex_off_q[e], vec_ok, 0,
                        false, 0ull, sr, sp_);
            if (tid == 0) {
                sm.ex_res[e] = sr;
                sm.ex_p[e] = sp_;
            }
        }
        __syncthreads();
        // 3. tile sums, totals, the target and the tile that holds it
        unsigned long long s_res = 0ull, s_p = 0ull;
        if (t < n_tiles) {
            if (split) {
                for (int e = 0; e < n_ex; ++e)
                    if (sm.ex_tile[e] == t) {
                        s_res = sm.ex_res[e];
                        s_p = sm.ex_p[e];
                    }
            } else {
                const unsigned long long tr0 = stq ? R[kTsTieRes + 1] : R[kTsTieRes];
                const unsigned long long tr1 = stq ? R[kTsTieRes + 3] : R[kTsTieRes + 2];
                s_res = R[kTsBaseRes] + (stp ? tr1 : tr0);
                s_p = R[kTsBaseP] + (stp ? R[kTsTieP + 1] : R[kTsTieP]);
            }
        }
        const unsigned long long W = block_sum_u64(sm, s_res), Wp = block_sum_u64(sm, s_p);
        if (job.kind == kJobSum) {   // block verification's H_j: the exact total is all it needs
            if (tid == 0) a.blk_h[(size_t)job.req * (K + 1) + job.a] = W;
            __syncthreads();
            continue;
        }
        const bool zero = residual && W == 0ull;
        const bool use_p = !residual || zero;
        const unsigned long long Wu = use_p ? Wp : W;
        const unsigned long long u24 = uniform24(a.seed, (uint32_t)job.req, (uint32_t)job.a, 1u);
        const unsigned long long hi = __umul64hi(Wu, u24), lo = Wu * u24;
        const unsigned long long target = (hi << 40) | (lo >> 24);   // floor(W * u)
        const unsigned long long mine = use_p ? s_p : s_res;
        unsigned long long all;
        const unsigned long long pre = block_excl_u64(sm, mine, all);
        if (t < n_tiles && pre <= target && target < pre + mine) {
            sm.found_tile = t;
            sm.tile_target = target - pre;
            sm.tile_off_p = op;
            sm.tile_off_q = oq;
        }
        __syncthreads();
        int x = -1;
        if (sm.found_tile >= 0) {
            unsigned long long d0, d1;
            x = rescan_tile(sm, P, Q, residual, sm.found_tile * tile_len, min(V, (sm.found_tile + 1) * tile_len),
                            sm.tile_off_p, sm.tile_off_q, vec_ok, 1,
                            use_p, sm.tile_target, d0, d1);
        }
        if (tid == 0) {
            if (x < 0) x = a.info[slot_target(job.req, K, job.a)].desc.argmax;   // not reached: sums are exact
            a.out_tokens[(size_t)job.req * (K + 1) + job.a] = x;
            if (zero && a.row_status) a.row_status[(size_t)job.req * (K + 1) + job.a] |= kResidZero;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_resample(const ChainArgs& a, int wave, cudaStream_t s)
{
    static int blocks[128] = {0};   // CTAs per SM, once per device (before any graph capture)
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = sizeof(ResSmem);
    int& nb = blocks[(dev >= 0 && dev < 128) ? dev : 0];
    if (nb == 0) {
        cudaError_t err = cudaFuncSetAttribute(resample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, resample_kernel, kResThreads, smem);
        if (err != cudaSuccess) return err;
        if (nb < 1) nb = 1;
    }
    const int unit = kResWarps * resample_tile_len(a.vocab);   // a chunk: one tile per warp
    const int n_units = (a.vocab + unit - 1) / unit;
    return launch_pdl(resample_kernel, dim3(a.num_sms * nb), dim3(kResThreads), smem, s, a, n_units, wave);
}

}  // namespace sv
