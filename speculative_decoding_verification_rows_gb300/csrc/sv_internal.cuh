// sv_internal.cuh -- device-side types and helpers shared by the libsv kernels.
//
// Workspace records, the order-preserving integer keys of logits, Philox4x32-10,
// warp reductions and the launchers each translation unit exports.  Nothing
// here is visible through the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sv.h"

namespace sv {

// ----------------------------------------------------------------------------
// Sizes
// ----------------------------------------------------------------------------
constexpr int kFastK = 32;          // largest top-k served by the one-pass select kernel
constexpr int kFastThreads = 512;   // threads of the one-pass select kernel
constexpr int kFastVecs = 8;        // 16-byte vectors per lane per warp chunk (4 KB a warp)
constexpr int kMaxRowWarps = 4096;  // warps of the one-pass select grid (sizes the partial lists)
constexpr int kHistThreads = 512;   // threads of the exact-histogram kernel
constexpr int kHistWords = 32768;   // 65536 16-bit counters, two per 32-bit word
constexpr int kHistMaxSlice = 65535;// elements per CTA so a 16-bit counter cannot wrap
constexpr int kMaxCluster = 8;      // portable cluster size limit

// Row / position status bits (the public SV_ROW_* values).
constexpr int kNonfinite = SV_ROW_NONFINITE, kEmpty = SV_ROW_EMPTY, kBadToken = SV_ROW_BAD_TOKEN,
              kBadParam = SV_ROW_BAD_PARAM, kBadLayout = SV_ROW_BAD_LAYOUT, kQZero = SV_ROW_Q_ZERO,
              kResidZero = SV_ROW_RESID_ZERO, kUnsupported = SV_ROW_UNSUPPORTED,
              kTimeout = SV_ROW_TIMEOUT;
constexpr int kErrorMask = SV_ROW_ERROR_MASK;

// ----------------------------------------------------------------------------
// Workspace records
// ----------------------------------------------------------------------------
// One logits row to process.
struct RowTask {
    int64_t row;      // row index in its logits tensor
    int32_t slot;     // RowInfo slot the result goes to
    int32_t req;      // request (index into the sampling parameters)
    int32_t token;    // token whose probability is reported, -1 for none
    int32_t k_eff;    // kept count of the top-k stage (1 for greedy rows)
    float temp;       // 0 = greedy
    float top_p;      // >= 1 = top-p off
    int32_t is_draft; // 1: row of the draft logits
    int32_t req_rows; // rows the request listed (its chain runs once they are all done)
};

// A list of row tasks, stored as three arrays (row index; slot, request,
// token, k; temperature, top-p, draft flag) so that the tasks of consecutive
// threads are written with whole-sector vector stores.
struct TaskList {
    int64_t* row;
    int4* meta;
    float4* samp;

    __device__ __forceinline__ RowTask get(int64_t t) const
    {
        RowTask r;
        r.row = row[t];
        const int4 m = meta[t];
        const float4 f = samp[t];
        r.slot = m.x;
        r.req = m.y;
        r.token = m.z;
        r.k_eff = m.w;
        r.temp = f.x;
        r.top_p = f.y;
        r.is_draft = __float_as_int(f.z);
        r.req_rows = __float_as_int(f.w);
        return r;
    }
    __device__ __forceinline__ void put(int64_t t, const RowTask& r) const
    {
        row[t] = r.row;
        meta[t] = make_int4(r.slot, r.req, r.token, r.k_eff);
        samp[t] = make_float4(r.temp, r.top_p, __int_as_float(r.is_draft), __int_as_float(r.req_rows));
    }
};
constexpr size_t kTaskBytes = sizeof(int64_t) + sizeof(int4) + sizeof(float4);

// Result of one row (its distribution, enough to sample from it).
struct RowInfo {
    sv_row_desc_t desc;         // 32 B, the public descriptor
    double p_token;             // probability of the task's token (NaN if none)
    double z;                   // normaliser: sum over kept of exp((l - m) / T)
    double z_rest;              // kept mass after the top token (z - 1, summed without cancellation)
    int32_t n_list;             // kept tokens listed below (ascending index), -1 if not listed
    int32_t cut_count;          // tokens whose logit equals the cutoff (all of them, kept or not)
    int32_t list_idx[kFastK];
    double list_p[kFastK];
};

// Top candidates of one warp's part of one row: composite keys, descending.
struct Partial {
    uint32_t status;
    uint32_t count;
    unsigned long long keys[kFastK];
};

// Per fast task: parts of the row finished so far, and the best lower bound
// on the row's k-th largest logit that a part has published (order key of
// the value, 0 = none).  Zeroed by the prep kernel.
struct RowSync {
    int32_t done;
    uint32_t bound;
};

// Per-request state written by the prep kernel.
struct ReqState {
    int32_t v;        // verified drafts (window = v + 1 target rows)
    int32_t greedy;   // temperature == 0
    int32_t err;      // request-level error bits (params, layout)
    int32_t fast;     // 1: its rows took the one-pass kernel, which also ran its chain
    uint64_t tok_bad; // bit j: draft token j out of range
    int32_t first_reject;   // histogram path, chain verify: lowest position whose test is known to reject (v: none yet)
    int32_t slow_base;      // index of its first row in the histogram-path task list (-1: none)
};

constexpr int kMaxK = 63;           // drafted positions per request (bit masks above)

// A full-row job of the resample kernel: draw the emitted token of a request
// whose kept set is not listed, or (block verification) sum a residual mass.
struct ResampleJob {
    int32_t req;
    int32_t a;        // position of the rows (the emitted token's, or the summed one's)
    int32_t residual; // 1: max(0, w p_a - q_a); 0: p_a (bonus)
    int32_t done;     // row chunks of the job the resample has finished (0 when listed)
    int32_t kind;     // kJobDraw or kJobSum
    int32_t pad;
    unsigned long long wfix;   // w as a 64-bit fraction (floor(w 2^64)); 0 means w = 1
};
constexpr int kJobDraw = 0;   // draw the emitted token by inverse CDF
constexpr int kJobSum = 1;    // only the exact residual total (block verification's H_j)

// A weight w in [0, 1] as a 64-bit fraction floor(w 2^64); w >= 1 as 0, the
// code for "no weight".
__device__ __forceinline__ unsigned long long weight_fix(double w)
{
    if (!(w < 1.0)) return 0ull;
    if (!(w > 0.0)) return 1ull;   // w = 0: the smallest weight, p w floors to 0
    return __double2ull_rz(w * 0x1p64);
}

// Chunks and tiles of the full-row resample.  A chunk (eight tiles) is what
// one CTA of the resample kernel streams at a time, one tile per warp; each
// tile (1,024 elements, or 2,048 when the row would otherwise have more than
// 256 tiles) leaves a record for the job's last chunk: exact fixed-point sums
// of the residual and of p over the tile, with the elements tied at a
// partially kept cutoff summed apart in both of their possible states (kept
// or not, for p and for q), and the tie counts.
constexpr int kResampleTile = 2048;    // the longest tile
constexpr int kResampleMaxTiles = 256;
enum TileField {
    kTsBaseRes = 0,   // residual over elements not tied at a partial cutoff
    kTsBaseP = 1,     // p over the same
    kTsTieRes = 2,    // 2..5: tied elements' residual, [p ties kept * 2 + q ties kept]
    kTsTieP = 6,      // 6..7: tied elements' p, [p ties kept]
    kTsTiesP = 8,     // elements at p's cutoff (partial groups only)
    kTsTiesQ = 9,     // elements at q's cutoff (partial groups only)
    kTsFields = 10
};
struct TileSums {
    unsigned long long v[kTsFields];
};
__host__ __device__ __forceinline__ int resample_tile_len(int vocab)
{
    return vocab <= kResampleMaxTiles * (kResampleTile / 2) ? kResampleTile / 2 : kResampleTile;
}
__host__ __device__ __forceinline__ int resample_tiles(int vocab)
{
    const int t = resample_tile_len(vocab);
    return (vocab + t - 1) / t;
}

// Request slots of the RowInfo array: target positions 0..K, then draft
// positions 0..K-1.
__host__ __device__ __forceinline__ int slot_target(int r, int K, int j) { return r * (2 * K + 1) + j; }
__host__ __device__ __forceinline__ int slot_draft(int r, int K, int j) { return r * (2 * K + 1) + K + 1 + j; }

// Counters at the head of the workspace.
struct Counters {
    int32_t n_fast;
    int32_t n_slow;
    int32_t n_jobs;
    int32_t timeout;   // set by a row kernel whose bounded wait gave up
    int32_t n_ovf;     // histogram rows handed from the one-CTA kernel to the cluster kernel
    int32_t n_jobs2;   // block verification: jobs listed after the residual sums (from index n_jobs)
    int32_t next_slow; // histogram path, chain verify: next row of slow_units to hand out
    int32_t n_slow_req;// requests whose rows take the histogram path (listed in slow_req)
    int32_t n_units;   // histogram path, chain verify: rows listed in slow_units
    int32_t pad[7];
};

// Carving of the caller's workspace.
struct WsLayout {
    size_t counters, fast_tasks, slow_tasks, ovf, info, partials, row_sync, req, req_done, pair_done, slow_req,
        slow_units, jobs, tiles, blk, total;
    int slots, max_tasks, max_jobs;
    size_t n_partials;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// slots: target positions 0..K and draft positions 0..K-1 of every request.
// Block verification (block = 1) lists up to K + 1 full-row jobs per request
// and keeps each request's weights w_j and residual sums H_j.
inline WsLayout ws_layout(int n_req, int k_max, int vocab, int block = 0)
{
    WsLayout L{};
    L.slots = n_req * (2 * k_max + 1);
    L.max_tasks = L.slots;
    // A grid of W warps splits T tasks into parts; W * (parts per warp) stays
    // below T + 3 W (see the range arithmetic of the row kernel).
    L.n_partials = (size_t)L.max_tasks + 3 * (size_t)kMaxRowWarps;
    size_t off = 0;
    L.counters = off;   off = align256(off + sizeof(Counters));
    L.fast_tasks = off; off = align256(off + kTaskBytes * (size_t)L.max_tasks + 16);   // + alignment of the arrays
    L.slow_tasks = off; off = align256(off + kTaskBytes * (size_t)L.max_tasks + 16);
    L.ovf = off;        off = align256(off + sizeof(int32_t) * (size_t)L.max_tasks);
    L.info = off;       off = align256(off + sizeof(RowInfo) * (size_t)L.slots);
    L.partials = off;   off = align256(off + sizeof(Partial) * L.n_partials);
    L.row_sync = off;   off = align256(off + sizeof(RowSync) * (size_t)L.max_tasks);
    L.req = off;        off = align256(off + sizeof(ReqState) * (size_t)n_req);
    L.req_done = off;   off = align256(off + sizeof(int32_t) * (size_t)n_req);
    L.pair_done = off;  off = align256(off + sizeof(int32_t) * (size_t)n_req * (size_t)(k_max + 1));
    L.slow_req = off;   off = align256(off + sizeof(int2) * (size_t)n_req);
    L.slow_units = off; off = align256(off + sizeof(int2) * (size_t)L.max_tasks);
    L.max_jobs = block ? n_req * (k_max + 1) : n_req;
    L.jobs = off;       off = align256(off + sizeof(ResampleJob) * (size_t)L.max_jobs);
    L.tiles = off;      off = align256(off + sizeof(TileSums) * (size_t)L.max_jobs * (size_t)resample_tiles(vocab));
    L.blk = off;        off = block ? align256(off + 2 * sizeof(double) * (size_t)n_req * (size_t)(k_max + 1)) : off;
    L.total = off;
    return L;
}

// ----------------------------------------------------------------------------
// Order-preserving keys.  Larger key <=> larger logit; -0 and +0 share a key.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t key_of_f32_bits(uint32_t b)
{
    if ((b & 0x7FFFFFFFu) == 0u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float f32_of_key(uint32_t k)
{
    uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(b);
}
// 16-bit key of a bf16 pattern, and back.
__device__ __forceinline__ uint32_t key16_of_bf16(uint32_t h)
{
    h &= 0xFFFFu;
    if ((h & 0x7FFFu) == 0u) h = 0u;
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
}
// Order keys of both bf16 halves of a word, -0 kept apart from +0 (key
// 0x7FFF, just below +0's 0x8000): a byte permute replicates each half's sign
// bit over the half, which selects the flip mask.
__device__ __forceinline__ uint32_t keys2_raw(uint32_t w)
{
    uint32_t sgn;
    asm("prmt.b32 %0, %1, %2, 0xBB99;" : "=r"(sgn) : "r"(w), "r"(0u));
    return w ^ (sgn | 0x80008000u);
}
__device__ __forceinline__ uint32_t max_u16x2(uint32_t x, uint32_t y)
{
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
    return r;
}
__device__ __forceinline__ uint32_t min_u16x2(uint32_t x, uint32_t y)
{
    uint32_t r;
    asm("min.u16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
    return r;
}
// Number of 16-bit halves of t that are zero (no carry crosses the halves).
__device__ __forceinline__ int zero_halves(uint32_t t)
{
    const uint32_t y = (t & 0x7FFF7FFFu) + 0x7FFF7FFFu;   // bit 15 of a half: its low 15 bits are not all 0
    return __popc(~(y | t) & 0x80008000u);
}

__device__ __forceinline__ float f32_of_key16(uint32_t k)
{
    uint32_t h = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
    return __uint_as_float(h << 16);
}
// Composite key: logit key above, inverted index below, so that a larger
// composite means (larger logit, or equal logit and smaller index).
__device__ __forceinline__ unsigned long long ckey(float v, uint32_t idx)
{
    return ((unsigned long long)key_of_f32_bits(__float_as_uint(v)) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ float ckey_value(unsigned long long c) { return f32_of_key((uint32_t)(c >> 32)); }
__device__ __forceinline__ int ckey_index(unsigned long long c) { return (int)(0xFFFFFFFFu - (uint32_t)c); }

// Exact value of a 16-bit key as a double.
__device__ __forceinline__ double key_value(uint32_t k16) { return (double)f32_of_key16(k16); }

// x^n for a small non-negative integer n (binary powering).
__device__ __forceinline__ double powi(double x, int n)
{
    double r = 1.0;
    while (n) {
        if (n & 1) r *= x;
        x *= x;
        n >>= 1;
    }
    return r;
}

// exp((v - m) / T) in fp64 for the 8 keys b*128 + 8g .. + 7 of binade b (the
// 128 keys sharing a sign and exponent; the mantissa step is constant along
// it).  Binade 0 holds -inf (mass 0).  Where the step is small against T the
// masses follow a geometric recurrence from two exps per binade; otherwise
// each key gets its own exp.
__device__ __forceinline__ void binade_masses(int b, int g, double m, double T, double e[8])
{
    if (b == 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) e[j] = 0.0;
        return;
    }
    const uint32_t kb = (uint32_t)b * 128u;
    const double v_first = key_value(kb);
    const double step = key_value(kb + 1u) - v_first;
    const double x = step / T;
    if (x <= 1.0) {
        const double R = exp(x);
        const double base = exp((v_first - m) / T);
        double cur = base * powi(R, 8 * g);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            e[j] = cur;
            cur *= R;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) e[j] = exp((key_value(kb + 8u * g + j) - m) / T);
    }
}

// ----------------------------------------------------------------------------
// Double-float arithmetic (Dekker, "A floating-point technique for extending
// the available precision", 1971; the error-free sum is Knuth's two-sum): a
// value held as the unevaluated sum hi + lo of two floats, about 48
// significant bits, so that sums which must agree with fp64 far below 1e-9
// run on the fp32 pipes instead of the narrow fp64 one.
// ----------------------------------------------------------------------------
struct dfloat {
    float hi, lo;
};
__device__ __forceinline__ dfloat df_of(double x)
{
    const float h = (float)x;
    return dfloat{h, (float)(x - (double)h)};
}
__device__ __forceinline__ double df_val(dfloat a) { return (double)a.hi + (double)a.lo; }
// a + f for a float f, renormalised.
__device__ __forceinline__ dfloat df_add_f(dfloat a, float f)
{
    const float s = a.hi + f;
    const float bb = s - a.hi;
    const float e = (a.hi - (s - bb)) + (f - bb) + a.lo;
    const float hi = s + e;
    return dfloat{hi, e - (hi - s)};
}
// a * b, renormalised (the product's rounding error recovered by an FMA).
__device__ __forceinline__ dfloat df_mul(dfloat a, dfloat b)
{
    const float p = a.hi * b.hi;
    float e = fmaf(a.hi, b.hi, -p);
    e = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, e));
    const float hi = p + e;
    return dfloat{hi, e - (hi - p)};
}

// More double-float pieces, and exp in double-float arithmetic (on GB300 the
// fp64 pipe runs at a 64th of the fp32 rate, so an fp64 exp per element, or
// per table entry, would dominate the kernels that need them).
constexpr double kLn2 = 0.69314718055994530942;   // ln 2
__device__ __forceinline__ dfloat df_two_sum(float a, float b)   // a + b exactly
{
    const float s = a + b;
    const float bb = s - a;
    return dfloat{s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ dfloat df_add(dfloat a, dfloat b)
{
    const dfloat s = df_two_sum(a.hi, b.hi);
    const float e = s.lo + a.lo + b.lo;
    const float hi = s.hi + e;
    return dfloat{hi, e - (hi - s.hi)};
}

// (x - m) / T as a double-float: the difference exactly, the quotient's
// remainder recovered by an FMA (inv_t = 1 / T rounded; the remainder
// corrects the first quotient to about 2^-46).
__device__ __forceinline__ dfloat scaled_logit(float x, float m, float T, float inv_t)
{
    const dfloat d = df_two_sum(x, -m);
    const float q1 = d.hi * inv_t;
    const float q2 = (fmaf(-q1, T, d.hi) + d.lo) * inv_t;
    const float hi = q1 + q2;
    return dfloat{hi, q2 - (hi - q1)};
}

// exp(a) for -87 <= a <= 88, about 2^-46 relative (0 below -87, where fp32
// ends).
// Reduction a = k ln2 / 64 + r (Tang, "Table-driven implementation of the
// exponential function in IEEE floating-point arithmetic", 1989), with
// |r| <= ln2 / 128; exp(r) = 1 + r + r^2/2 + r^3 (1/6 + r/24 + r^2/120 +
// r^3/720), the last factor in fp32 (it is below 2^-22 of the sum); then
// times 2^(j/64) from the table and 2^n.
constexpr float kExpK = (float)(64.0 / kLn2);
constexpr float kCHi = 1420.0f / 131072.0f;   // ln2 / 64 to 11 bits: k * kCHi is exact for |k| < 2^13
constexpr double kCRest = kLn2 / 64.0 - (double)kCHi;
constexpr float kCRestHi = (float)kCRest, kCRestLo = (float)(kCRest - (double)kCRestHi);

__device__ __forceinline__ dfloat exp_df(dfloat a, const dfloat* tab)
{
    if (!(a.hi >= -87.0f)) return dfloat{0.0f, 0.0f};
    const float kf = rintf(a.hi * kExpK);
    dfloat r = df_two_sum(a.hi, -kf * kCHi);
    r = df_add(r, dfloat{a.lo, 0.0f});
    r = df_add(r, df_mul(dfloat{kCRestHi, kCRestLo}, dfloat{-kf, 0.0f}));
    const float rh = r.hi;
    const float q = fmaf(fmaf(fmaf(rh, 1.0f / 720.0f, 1.0f / 120.0f), rh, 1.0f / 24.0f), rh, 1.0f / 6.0f);
    const dfloat r2 = df_mul(r, r);
    dfloat s = df_add(r, dfloat{0.5f * r2.hi, 0.5f * r2.lo});
    s = df_add_f(s, rh * rh * rh * q);
    dfloat e = df_add_f(s, 1.0f);
    const int k = (int)kf;
    e = df_mul(e, tab[k & 63]);
    const int n = k >> 6;   // floor(k / 64), in [-126, 127] for -87 <= a <= 88: 2^n is a normal float
    const float p2 = __int_as_float((n + 127) << 23);
    return dfloat{e.hi * p2, e.lo * p2};
}

// 2^(j / 64), j = 0..63, as double-floats: hi is the value rounded to fp32,
// lo the rest rounded to fp32 (together within 2^-47 of 2^(j / 64)).
__device__ const dfloat c_exp2_64[64] = {
    {0x1p+0f, 0.0f}, {0x1.02c9a4p+0f, -0x1.887fap-28f}, {0x1.059b0ep+0f, -0x1.9d4f52p-25f}, {0x1.087452p+0f, -0x1.e2990ep-26f},
    {0x1.0b5586p+0f, 0x1.9f3122p-25f}, {0x1.0e3ec4p+0f, -0x1.a585ccp-25f}, {0x1.11301ep+0f, -0x1.fdb496p-25f}, {0x1.1429aap+0f, 0x1.d525bcp-25f},
    {0x1.172b84p+0f, -0x1.c15742p-27f}, {0x1.1a35bep+0f, 0x1.6df96ep-25f}, {0x1.1d4874p+0f, -0x1.d2e8cap-25f}, {0x1.2063b8p+0f, 0x1.0c519ap-25f},
    {0x1.2387a6p+0f, 0x1.ceac48p-25f}, {0x1.26b456p+0f, 0x1.789f38p-26f}, {0x1.29e9ep+0f, -0x1.5c0424p-25f}, {0x1.2d285ap+0f, 0x1.b900c2p-26f},
    {0x1.306fep+0f, 0x1.4636e2p-25f}, {0x1.33c08cp+0f, -0x1.b37d2p-25f}, {0x1.371a74p+0f, -0x1.18aac6p-25f}, {0x1.3a7db4p+0f, -0x1.634c02p-25f},
    {0x1.3dea64p+0f, 0x1.824684p-25f}, {0x1.4160a2p+0f, 0x1.f72e2ap-28f}, {0x1.44e086p+0f, 0x1.8624b4p-30f}, {0x1.486a2cp+0f, -0x1.47d866p-25f},
    {0x1.4bfdaep+0f, -0x1.593abcp-25f}, {0x1.4f9b28p+0f, -0x1.2c5a6cp-25f}, {0x1.5342b6p+0f, -0x1.2c561p-25f}, {0x1.56f474p+0f, -0x1.295b04p-25f},
    {0x1.5ab07ep+0f, -0x1.5bd5ecp-27f}, {0x1.5e76f2p+0f, -0x1.4a5bd6p-25f}, {0x1.6247ecp+0f, -0x1.f8b55p-25f}, {0x1.662388p+0f, 0x1.2a9112p-27f},
    {0x1.6a09e6p+0f, 0x1.9fcef4p-26f}, {0x1.6dfb24p+0f, -0x1.cd72e8p-27f}, {0x1.71f75ep+0f, 0x1.1d8beep-25f}, {0x1.75feb6p+0f, -0x1.37b306p-25f},
    {0x1.7a1148p+0f, -0x1.829fdp-25f}, {0x1.7e2f34p+0f, -0x1.261634p-25f}, {0x1.82589ap+0f, -0x1.accc7cp-26f}, {0x1.868d9ap+0f, -0x1.2edb44p-26f},
    {0x1.8ace54p+0f, 0x1.15506ep-27f}, {0x1.8f1aeap+0f, -0x1.baa232p-26f}, {0x1.93737cp+0f, -0x1.e64744p-25f}, {0x1.97d82ap+0f, -0x1.0d8d84p-31f},
    {0x1.9c4918p+0f, 0x1.51f848p-27f}, {0x1.a0c668p+0f, -0x1.2886a6p-26f}, {0x1.a5503cp+0f, -0x1.b83b54p-25f}, {0x1.a9e6b6p+0f, -0x1.50c048p-25f},
    {0x1.ae89fap+0f, -0x1.a94b14p-26f}, {0x1.b33a2cp+0f, -0x1.ec3a82p-26f}, {0x1.b7f77p+0f, -0x1.a09438p-25f}, {0x1.bcc1eap+0f, -0x1.f687c6p-25f},
    {0x1.c199bep+0f, -0x1.3d56b2p-27f}, {0x1.c67f12p+0f, 0x1.cafa2ap-25f}, {0x1.cb720ep+0f, -0x1.8837ccp-27f}, {0x1.d072d4p+0f, 0x1.40f13p-25f},
    {0x1.d5818ep+0f, -0x1.822dbcp-27f}, {0x1.da9e6p+0f, 0x1.ed9942p-27f}, {0x1.dfc974p+0f, -0x1.908c94p-25f}, {0x1.e502eep+0f, 0x1.e2cffep-26f},
    {0x1.ea4afap+0f, 0x1.52486cp-27f}, {0x1.efa1bep+0f, 0x1.cc2b44p-25f}, {0x1.f50766p+0f, -0x1.246ebp-26f}, {0x1.fa7c18p+0f, 0x1.9e90d8p-28f}
};

// The table above in shared memory, where the lanes' lookups do not
// serialise (every thread calls it).
__device__ __forceinline__ void fill_exp_table(dfloat* tab)
{
    for (int j = threadIdx.x; j < 64; j += blockDim.x) tab[j] = c_exp2_64[j];
    __syncthreads();
}

// 1 / d for a positive double-float d: the fp32 reciprocal of its high part
// and one Newton correction 1 - d r computed with FMAs (about 2^-46).
__device__ __forceinline__ dfloat df_recip_df(dfloat d)
{
    const float r = 1.0f / d.hi;
    const float e = fmaf(-d.hi, r, 1.0f) - d.lo * r;
    return df_two_sum(r, r * e);
}
__device__ __forceinline__ dfloat df_recip(double z) { return df_recip_df(df_of(z)); }

// floor(e * 2^s) for 0 <= e <= 1 held as a double-float (s = 58 or 62).
__device__ __forceinline__ unsigned long long fix_df(dfloat e, float scale)
{
    const unsigned long long h = __float2ull_rz(e.hi * scale);   // up to 2^62
    const long long l = __float2ll_rd(e.lo * scale);              // |l| below 2^40
    if (l < 0 && (unsigned long long)(-l) > h) return 0ull;
    return h + (unsigned long long)l;                             // two's complement: h - |l| for l < 0
}

// ----------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): counter (req, pos, draw, 0),
// key (seed low, seed high); u = (word0 >> 8) * 2^-24.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t philox_word0(unsigned long long seed, uint32_t req, uint32_t pos, uint32_t draw)
{
    uint32_t c0 = req, c1 = pos, c2 = draw, c3 = 0u;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    return c0;
}
__device__ __forceinline__ uint32_t uniform24(unsigned long long seed, uint32_t req, uint32_t pos, uint32_t draw)
{
    return philox_word0(seed, req, pos, draw) >> 8;
}
__device__ __forceinline__ double uniform_f64(unsigned long long seed, uint32_t req, uint32_t pos, uint32_t draw)
{
    return (double)uniform24(seed, req, pos, draw) * (1.0 / 16777216.0);
}

// ----------------------------------------------------------------------------
// Warp helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, x, o);
        x = y > x ? y : x;
    }
    return x;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}

// The same for values below 2^63 whose warp total is below 2^63 (fixed-point
// probabilities), where most warps hold zeros: a vote, then three 21-bit
// limbs summed by the warp-reduce unit (each limb total stays below 2^26).
__device__ __forceinline__ unsigned long long warp_sum_u63(unsigned long long x)
{
    if (!__any_sync(0xFFFFFFFFu, x != 0ull)) return 0ull;
    const uint32_t l0 = (uint32_t)x & 0x1FFFFFu, l1 = (uint32_t)(x >> 21) & 0x1FFFFFu, l2 = (uint32_t)(x >> 42);
    return (unsigned long long)__reduce_add_sync(0xFFFFFFFFu, l0) +
           ((unsigned long long)__reduce_add_sync(0xFFFFFFFFu, l1) << 21) +
           ((unsigned long long)__reduce_add_sync(0xFFFFFFFFu, l2) << 42);
}

// Value of a row element, by dtype (0 = bf16, 1 = fp32).
template <int DT>
__device__ __forceinline__ float load_logit(const void* row, int64_t i)
{
    if (DT == 0) return __uint_as_float((uint32_t)(((const uint16_t*)row)[i]) << 16);
    return ((const float*)row)[i];
}

// ----------------------------------------------------------------------------
// mbarriers and bulk asynchronous copies (cp.async.bulk) into shared memory.
// Every wait is bounded: it gives up after kWaitPolls polls.
// ----------------------------------------------------------------------------
constexpr long long kWaitPolls = 1ll << 20;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0u;
}
// false when the phase did not complete within kWaitPolls polls
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity)
{
    for (long long i = 0; i < kWaitPolls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// Global -> shared bulk copy of `bytes` (multiple of 16, both ends 16-byte
// aligned) completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, unsigned long long* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(const void* p)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_u32(p)));
    return r;
}

// ----------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with
// the programmatic-serialisation attribute, so it may become resident while the
// kernel before it on the stream drains.  It first waits for that kernel to
// complete (its memory included), then lets its own dependent launch early.
// Without a programmatic predecessor the wait returns at once.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

inline void pdl_attr(cudaLaunchAttribute& at)
{
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
}

// Launch with the attribute above (plus `extra` attributes, if any).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    pdl_attr(at[0]);
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ----------------------------------------------------------------------------
// Launchers (host), one per kernel family.
// ----------------------------------------------------------------------------
struct ChainArgs {
    int n_req, K;          // K = k_max: slots per request = 2K + 1 (layout 2: n_req = rows)
    int n_params;          // length of the sampling-parameter arrays
    int vocab, dtype;
    int layout;            // 0 uniform, 1 ragged, 2 plain rows (build_target_probs)
    int block;             // 1: block verification instead of the token-by-token chain
    int est;               // 1: estimator features (layout 2, greedy requests at T = 1)
    int fuse;              // 1: the one-pass kernel runs the chain of each request whose rows it took
    int lazy;              // 1: histogram rows past a request's known first rejection get a validity scan only
    int lazy_grid;         // CTAs of the histogram kernel: rows that fit in one wave are not listed by position
    int shard;             // vocabulary-sharded verify (listed kept sets only): 1 a shard's rows
                           // (no outputs), 2 the merge of the shards' records (no logits)
    int rows_per_req;      // layout 2 without row_to_req: request = row / rows_per_req
    const void* tgt;
    const void* drf;
    int64_t stride_t, stride_d;
    int bucket;
    const int32_t* qo_indptr;
    const int32_t* verify_len;   // nullable in the uniform layout
    const int32_t* draft_tokens; // [n, K]
    const int32_t* row_to_req;   // layout 2
    const int32_t* token_per_row;// layout 2
    sv_sampling_t sp;
    unsigned long long seed;
    int32_t* accept_len;
    int32_t* out_tokens;
    int32_t* num_emitted;
    int32_t* row_status;
    Counters* counters;
    TaskList fast_tasks;
    TaskList slow_tasks;
    RowSync* row_sync;
    RowInfo* info;
    ReqState* req;
    int32_t* req_done;   // rows of each request finished by the one-pass kernel (zeroed by prep)
    const RowInfo* q_rows;   // draft rows' results made beforehand ([n_req][K], sv_estimator_predict_q), or NULL
    int32_t* pair_done;  // [n_req][K + 1]: rows of position j finished on the histogram path (lazy)
    int2* slow_req;      // requests whose rows take the histogram path (lazy), n_slow_req of them:
                         // {request << 7 | greedy << 6 | v, index of its first task}
    int2* slow_units;    // their rows in position order (lazy): {request << 7 | position << 1 | draft, task}
    ResampleJob* jobs;
    TileSums* tiles;   // [max_jobs][resample_tiles(vocab)]
    double* blk_w;     // block verification: [n_req][K + 1] weights w_j
    unsigned long long* blk_h;   // block verification: [n_req][K + 1] residual sums H_j (2^-62 units)
    int num_sms;
};

// The result of draft row j of request r: the verify's own (a row slot), or
// one made beforehand for the same rows and parameters.
__device__ __forceinline__ const RowInfo& draft_info(const ChainArgs& a, int r, int j)
{
    return a.q_rows ? a.q_rows[(size_t)r * a.K + j] : a.info[slot_draft(r, a.K, j)];
}

struct RowsArgs {
    const void* tgt;
    const void* drf;
    int64_t stride_t, stride_d;
    int vocab;
    int dtype;
    TaskList fast_tasks;
    TaskList slow_tasks;
    Counters* counters;
    RowInfo* info;
    Partial* partials;
    RowSync* row_sync;   // per fast task (zeroed by the prep kernel)
    int32_t* ovf_idx;    // slow tasks the one-CTA histogram kernel could not hold (counted in n_ovf)
    int max_tasks;
    int num_sms;
    ChainArgs chain;     // the chain walk the one-pass kernel runs when chain.fuse is set
    Partial* shard_out;  // vocabulary shard: per-slot records instead of row results (NULL otherwise)
    uint32_t shard_v0;   // the shard's first vocabulary element
};

cudaError_t launch_fast_rows(const RowsArgs& a, cudaStream_t s);
cudaError_t launch_shard_merge(const RowsArgs& a, const void* records, int n_shards, int slots, cudaStream_t s);
cudaError_t launch_hist_rows(const RowsArgs& a, cudaStream_t s);
cudaError_t launch_rows32(const RowsArgs& a, cudaStream_t s);   // fp32 rows with unlisted kept sets
// CTAs of the one-CTA histogram kernel's grid on the current device (0 on error).
int hist_wide_grid(int num_sms);



cudaError_t launch_prep(const ChainArgs& a, cudaStream_t s);
cudaError_t launch_chain(const ChainArgs& a, cudaStream_t s);
cudaError_t launch_resample(const ChainArgs& a, int wave, cudaStream_t s);
cudaError_t launch_resample32(const ChainArgs& a, int wave, cudaStream_t s);   // the same for fp32 rows
cudaError_t launch_block_finish(const ChainArgs& a, cudaStream_t s);
cudaError_t launch_rows_out(const ChainArgs& a, float* prob_of_token, sv_row_desc_t* desc, float* dense,
                            cudaStream_t s);

cudaError_t launch_est_init(double* state, int K, cudaStream_t s);
cudaError_t launch_est_predict(const RowInfo* info, const double* state, int n, int K, float* x, float* p,
                               const Counters* counters, cudaStream_t s);
cudaError_t launch_est_observe(double* state, const float* x, const int32_t* accept_len, const int32_t* num_emitted,
                               const int32_t* verify_lens, int n, int K, int refit_every, cudaStream_t s);

cudaError_t launch_plan(const float* conf, int ld, const int32_t* draft_len, int n, int K, int budget,
                        const int32_t* budget_dev, int32_t* verify_lens, int32_t* qo_indptr, int32_t* total,
                        int32_t* status, unsigned long long* keys, cudaStream_t s);

constexpr int kBudgetMaxCand = 16384;   // candidates (n * K) the budget choice sorts in shared memory
constexpr int kBudgetMaxShelves = 4096; // shelves and batch-overhead entries of a cost table
cudaError_t launch_budget(const float* conf, int ld, const int32_t* draft_len, int n, int K, const int32_t* cost_tokens,
                          const float* cost_ms, int n_cost, float fixed_ms, const int32_t* batch_sizes,
                          const float* batch_ms, int n_batch, int bucket, int32_t* budget_out, int32_t* budget_status,
                          cudaStream_t s);
cudaError_t launch_stats(const int32_t* accept_len, const int32_t* num_emitted, const int32_t* verify_lens,
                         const int32_t* draft_len, int n, int K, long long* out, cudaStream_t s);

int device_sm_count();

}  // namespace sv
