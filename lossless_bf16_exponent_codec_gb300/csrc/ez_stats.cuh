// ez_stats.cuh -- exact moments, exponent histogram and window choice.
//
// ZipCCL digest 3.1: the 3-bit code window follows from the tensor's
// standard deviation.  sigma is defined from the EXACT sums s1 = sum v and
// s2 = sum v^2 over the finite values, each rounded once to double, so any
// reduction order gives the same bits:
//
//   v = (-1)^s * M * 2^(E-134),  M = 128 + mantissa  (E >= 1)
//
// so s1 and s2 follow from per-exponent integer sums of +-M and M^2.  Per
// value the hot loop is one shared-memory atomic.  A CTA picks a 16-binade
// window [Elo, Elo+16) around the mode of a sample of its exponents; a value
// inside it increments the count of its (d = E - Elo, sign|mantissa byte)
// cell of a 16 x 256 histogram.  Since a cell fixes sign and M, the cell
// counts determine the window's exact per-exponent count, sum of +-M and
// sum of M^2; they are folded once per tile.  Values outside the window
// (and zeros, subnormals, Inf/NaN) go straight to per-exponent bins.
//
// The cell of an in-window value is s << 11 | d << 7 | m (sign, binade
// offset, mantissa).  With y = (h | 0x8000) - Elo * 128, a 16-bit lane holds
// 1 << 15 | d << 7 | m and has bits 11..14 clear exactly when the value lies
// in the window, so the cell is one PRMT (the sign, replicated) and one LOP3
// away from y; the cell increment is a predicated shared reduction.  The
// CTA then adds its bins to per-shard global bins (64-bit atomics); the last
// CTA of the shard turns the bins into one big integer per sum, rounds it to
// nearest even, and derives var, sigma and the window base E0.
#pragma once

#include "ez_common.cuh"

namespace ez {

struct StatsBins {                 // per shard, in the workspace (zeroed per call)
    unsigned long long hist[256];
    unsigned long long s1[256];    // two's-complement int64 sums of +-M
    unsigned long long s2[256];    // sums of M^2
    unsigned int done;             // CTAs that have flushed
    unsigned int pad[63];
};

// Per-CTA accumulators (dynamic shared memory).  A CTA adds at most
// kStatsMaxValues values before it flushes, so no cell or bin can overflow
// 32 bits: counts <= 2^16, |sum +-M| <= 2^16 * 255 < 2^31 and sums of M^2
// <= 2^16 * 255^2 < 2^32 (all plain 32-bit shared atomics).
constexpr int kStatsWin = 16;                  // binades in a CTA's window
constexpr uint32_t kStatsMaxValues = 1u << 16;
static_assert((unsigned long long)kStatsMaxValues * 255u * 255u < (1ull << 32), "sum of M^2 fits 32 bits");
struct StatsSmem {
    uint32_t hist[2 * kStatsWin * 128];        // [sign][d][mantissa]
    uint32_t s2[256];
    uint32_t cnt[256];
    int s1[256];
    uint32_t sample[256];
    uint32_t elo;
    uint32_t last;
    uint32_t junk[32];     // target of the reductions of out-of-window lanes (never read)
};

// Zero the CTA's accumulators and choose Elo from one exponent per thread
// (h0 = that thread's first value, or 0xFFFFFFFF for none).
__device__ __forceinline__ void st_begin(StatsSmem& S, uint32_t h0)
{
    const int t = threadIdx.x;
    S.cnt[t] = 0;
    S.s1[t] = 0;
    S.s2[t] = 0;
    S.sample[t] = 0;
    uint4* c = reinterpret_cast<uint4*>(S.hist);
    constexpr int kVec = (int)(sizeof(S.hist) / 16);
    for (int i = t; i < kVec; i += kThreads) c[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (h0 != 0xFFFFFFFFu) atomicAdd(&S.sample[exp_of(h0)], 1u);
    __syncthreads();
    if (t < 32) {
        // mode of the sample, ties to the lowest exponent
        uint32_t best = 0, bestE = 127;
        for (int k = 0; k < 8; k++) {
            const uint32_t E = (uint32_t)(t * 8 + k);
            const uint32_t v = S.sample[E];
            if (v > best) { best = v; bestE = E; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            uint32_t ob = __shfl_xor_sync(kFull, best, o);
            uint32_t oe = __shfl_xor_sync(kFull, bestE, o);
            if (ob > best || (ob == best && oe < bestE)) { best = ob; bestE = oe; }
        }
        if (t == 0) {
            int elo = (int)bestE - 10;
            elo = elo < 1 ? 1 : (elo > 239 ? 239 : elo);
            S.elo = (uint32_t)elo;
        }
    }
    __syncthreads();
}

// A value outside the window: straight into the per-exponent bins (a zero
// only counts).
__device__ __forceinline__ void st_add_slow(uint32_t h, StatsSmem& S)
{
    const uint32_t E = exp_of(h);
    atomicAdd(&S.cnt[E], 1u);
    const uint32_t M = (E ? 128u : 0u) | (h & 0x7Fu);
    if (E != 255u && M) {
        atomicAdd(&S.s1[E], (h & 0x8000u) ? -(int)M : (int)M);
        atomicAdd(&S.s2[E], M * M);
    }
}

// One value h (16 bits), any value.
__device__ __forceinline__ void st_add(uint32_t h, uint32_t elo, StatsSmem& S)
{
    // v = sign*256 + E - Elo; in the window iff its low byte is below 16
    // (Elo <= 239 keeps E = 255 and E < Elo outside)
    const uint32_t v = (h >> 7) - elo;
    if ((v & 0xF0u) == 0) {
        atomicAdd(&S.hist[((h >> 4) & 0x800u) | ((v & 0xFu) << 7) | (h & 0x7Fu)], 1u);
    } else {
        st_add_slow(h, S);
    }
}

// Lane-exact window offsets of the two values of word x: y = (x | 0x8000) -
// Elo * 0x00800080 (e7 = (Elo << 7) * 0x10001).  Setting the low lane's sign
// bit keeps it from borrowing out of the high lane.
__device__ __forceinline__ uint32_t st_y(uint32_t x, uint32_t e7) { return (x | 0x8000u) - e7; }

// Cell of one lane: t = that lane's y in bits 0..15 (bits above don't
// matter), m = its sign replicated over bits 8..15 of a word otherwise zero.
// Bits 0..10 and 12..14 come from t, bit 11 is ~t & m = the sign (bit 11 of
// an in-window t is clear), bit 15 and up give ~t & m = 0.
__device__ __forceinline__ uint32_t st_cell(uint32_t t, uint32_t m)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xC2;" : "=r"(r) : "r"(t), "r"(0x77FFu), "r"(m));
    return r;
}
__device__ __forceinline__ uint32_t st_sign_lo(uint32_t x)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, 0x4494;" : "=r"(r) : "r"(x));
    return r;
}
__device__ __forceinline__ uint32_t st_sign_hi(uint32_t x)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, 0x44B4;" : "=r"(r) : "r"(x));
    return r;
}

// hist[cell] += 1 when (y & mask) == 0 (the lane is in the window), else a
// lane-private junk word += 1: the address is selected, so the reduction
// itself is unconditional and the hot loop has no branch per value.
__device__ __forceinline__ void st_red_sel(uint32_t addr, uint32_t junk, uint32_t y, uint32_t mask)
{
    asm volatile("{ .reg .pred q; .reg .b32 t, a; and.b32 t, %1, %2; setp.eq.u32 q, t, 0;"
                 " selp.b32 a, %0, %3, q; red.shared.add.u32 [a], 1; }"
                 :: "r"(addr), "r"(y), "r"(mask), "r"(junk) : "memory");
}

// Eight values (one 16-byte load): in-window values take their cell, the
// others (rare) the per-exponent bins.
__device__ __forceinline__ void st_add8(const uint4& w, uint32_t e7, uint32_t hist_base, uint32_t junk,
                                        StatsSmem& S)
{
    const uint32_t xs[4] = {w.x, w.y, w.z, w.w};
    uint32_t y[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        y[q] = st_y(xs[q], e7);
        st_red_sel(hist_base + 4u * st_cell(y[q], st_sign_lo(xs[q])), junk, y[q], 0x7800u);
        st_red_sel(hist_base + 4u * st_cell(y[q] >> 16, st_sign_hi(xs[q])), junk, y[q], 0x78000000u);
    }
    if ((y[0] | y[1] | y[2] | y[3]) & 0x78007800u) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            if (y[q] & 0x7800u) st_add_slow(xs[q] & 0xFFFFu, S);
            if (y[q] & 0x78000000u) st_add_slow(xs[q] >> 16, S);
        }
    }
}

// Fold the CTA into the global bins; returns true in every thread of the CTA
// that is the `expected`-th to finish (it must then call st_finalize).
__device__ __forceinline__ bool st_end(StatsSmem& S, StatsBins* G, uint32_t expected)
{
    const int t = threadIdx.x;
    const uint32_t elo = S.elo;
    __syncthreads();
    // cells [s][d][m]: 8 threads per (s, d) row, 16 mantissas each
    {
        const uint32_t s = (uint32_t)t >> 7, d = ((uint32_t)t >> 3) & 15u, part = (uint32_t)t & 7u;
        const uint4* row = reinterpret_cast<const uint4*>(&S.hist[(s << 11) | (d << 7) | (part << 4)]);
        uint32_t c = 0, s1 = 0, s2 = 0;
        uint32_t M = 128u + (part << 4);
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const uint4 x = row[q];
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; i++, M++) {
                c += xs[i];
                s1 += xs[i] * M;
                s2 += xs[i] * (M * M);
            }
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            c += __shfl_xor_sync(kFull, c, o);
            s1 += __shfl_xor_sync(kFull, s1, o);
            s2 += __shfl_xor_sync(kFull, s2, o);
        }
        if (part == 0 && c) {
            const uint32_t E = elo + d;
            atomicAdd(&S.cnt[E], c);
            atomicAdd(&S.s1[E], s ? -(int)s1 : (int)s1);
            atomicAdd(&S.s2[E], s2);
        }
    }
    __syncthreads();
    // per-exponent bins -> global
    if (S.cnt[t]) atomicAdd(&G->hist[t], (unsigned long long)S.cnt[t]);
    if (S.s1[t]) atomicAdd(&G->s1[t], (unsigned long long)(long long)S.s1[t]);
    if (S.s2[t]) atomicAdd(&G->s2[t], (unsigned long long)S.s2[t]);
    // the barrier orders every thread's bin atomics before thread 0's fence
    // (fences are cumulative), which orders them before the completion count
    __syncthreads();
    if (t == 0) {
        __threadfence();
        S.last = (atomicAdd(&G->done, 1u) == expected - 1) ? 1u : 0u;
    }
    __syncthreads();
    const bool last = S.last != 0;
    if (last) __threadfence();
    return last;
}

// ---- exact rounding of big sums ---------------------------------------------
// A big sum is a vector of 32-bit limbs held by one warp, limb i in lane i
// (lanes kLimbs..31 hold 0): kLimbs limbs hold every sum of at most 2^40
// terms below 2^16 * 2^506.

constexpr int kLimbs = 24;

// Carry-in bits of an addition whose limbs generate a carry (mask G) or pass
// one on (mask P, disjoint from G): the carries of the bit vectors G | P and
// G added as integers are exactly those of the limbs.
__device__ __forceinline__ uint32_t carry_in_mask(uint32_t G, uint32_t P) { return ((G | P) + G) ^ P; }

// Lane i holds x_i < 2^48 (zero in lanes >= kLimbs); returns limb i of the
// sum of x_i * 2^(32 i).  After adding each lane's high word into the next
// lane, a limb that carries out holds less than 2^16, so the remaining carries
// are single bits.
__device__ __forceinline__ uint32_t warp_carry(unsigned long long x)
{
    const uint32_t lane = threadIdx.x & 31u;
    uint32_t up = __shfl_up_sync(kFull, (uint32_t)(x >> 32), 1);
    if (lane == 0) up = 0;
    const unsigned long long v = (x & 0xFFFFFFFFull) + up;
    const uint32_t l = (uint32_t)v;
    const uint32_t C = carry_in_mask(__ballot_sync(kFull, (v >> 32) != 0), __ballot_sync(kFull, l == 0xFFFFFFFFu));
    return l + ((C >> lane) & 1u);
}

// Limbs of a - b (a >= b).
__device__ __forceinline__ uint32_t warp_sub(uint32_t a, uint32_t b)
{
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t C = carry_in_mask(__ballot_sync(kFull, a < b), __ballot_sync(kFull, a == b));
    return a - b - ((C >> lane) & 1u);
}

// 2^e as a double, e in the normal range
__device__ __forceinline__ double pow2d(int e)
{
    return __longlong_as_double((long long)(e + 1023) << 52);
}

// (sum of w_i 2^(32 i)) * 2^scale to the nearest double, ties to even: the
// top 53 bits, the next bit and whether any bit below it is set.
__device__ __forceinline__ double warp_round(uint32_t w, int scale)
{
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t nz = __ballot_sync(kFull, w != 0);
    if (!nz) return 0.0;
    const int top = 31 - __clz((int)nz);
    const int L = top * 32 + (32 - __clz((int)__shfl_sync(kFull, w, top)));   // bit length
    const unsigned long long low = (unsigned long long)__shfl_sync(kFull, w, 0) |
                                   (unsigned long long)__shfl_sync(kFull, w, 1) << 32;
    if (L <= 53) return __dmul_rn((double)low, pow2d(scale));                // exact: two limbs
    unsigned long long top64;                                                 // bits [L-64, L)
    bool sticky = false;
    if (L >= 64) {
        const int pos = L - 64, i = pos >> 5, sh = pos & 31;                 // i + 2 <= kLimbs
        const uint32_t w0 = __shfl_sync(kFull, w, i), w1 = __shfl_sync(kFull, w, i + 1),
                       w2 = __shfl_sync(kFull, w, i + 2);
        const unsigned long long lo = (unsigned long long)w0 | (unsigned long long)w1 << 32;
        top64 = sh ? (lo >> sh) | ((unsigned long long)w2 << (64 - sh)) : lo;
        sticky = __ballot_sync(kFull, w != 0 && (int)lane < i) != 0;         // bits [0, 32 i)
        if (sh) sticky |= (w0 & ((1u << sh) - 1u)) != 0;                      // bits [32 i, pos)
    } else {
        top64 = low << (64 - L);
    }
    unsigned long long q = top64 >> 11;                // the top 53 bits
    const bool half = (top64 >> 10) & 1ull;
    sticky |= (top64 & 0x3FFull) != 0;
    if (half && (sticky || (q & 1ull))) q++;           // 2^53 stays exact
    return __dmul_rn((double)q, pow2d(L - 53 + scale));
}

// Window base from the variance: the largest e in 1..249 with
// var >= K * 2^(2(e-127)-1), else 0.  K * 2^j is K with j added to its
// exponent field (exact: every threshold is a normal double), and positive
// doubles order as their bit patterns, so the search needs no FP64 multiply.
__device__ __forceinline__ uint32_t window_base(double var, double K)
{
    const long long vb = __double_as_longlong(var), kb = __double_as_longlong(K);
    int lo = 0, hi = 249;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (vb >= kb + ((long long)(2 * mid - 255) << 52)) lo = mid;
        else hi = mid - 1;
    }
    return (uint32_t)lo;
}

// The last CTA finalises.  Every thread takes one exponent bin and splits its
// terms into 32-bit pieces at their limbs of the three big sums (positive and
// negative parts of s1, and s2); the bins of one warp reach at most five
// consecutive limbs, so each warp adds its pieces limb by limb (warp
// reductions of the 16-bit halves) and stores its five slot sums with their
// first limb.  Warp 0 then gathers the limbs of s1's two parts (lane i adds
// the eight warps' slots at limb i), resolves the carries, subtracts and
// rounds; warp 1 does the same for s2 at the same time.  A limb total is at
// most 256 pieces of 32 bits < 2^40.
struct FinSmem {
    unsigned long long h[256];
    unsigned long long slot[kThreads / 32][3][5];   // per warp and sum: slot sums
    int base[kThreads / 32][3];                     // limb of each warp's slot 0
    unsigned long long nw[kThreads / 32];           // finite values per warp
    double s1d, s2d, b;
};
static_assert(sizeof(FinSmem) <= sizeof(StatsSmem::hist), "finalise scratch fits the histogram");

// Sum over the warp of 32-bit values
__device__ __forceinline__ unsigned long long warp_sum32(uint32_t v)
{
    return ((unsigned long long)__reduce_add_sync(kFull, v >> 16) << 16) + __reduce_add_sync(kFull, v & 0xFFFFu);
}

// The 32-bit pieces of v * 2^sh at limbs sh/32, sh/32 + 1, sh/32 + 2, added
// over the warp (all 32 lanes call it; lanes without a term pass v = 0).  The
// lanes' first limbs lie within 3 of lane 0's, so five slot sums cover them;
// lane 0 stores them to slot[0..4] and lane 0's limb to *base.
__device__ __forceinline__ void warp_slot_sums(unsigned long long* slot, int* base, unsigned long long v, int sh)
{
    const int limb = sh >> 5, bit = sh & 31;
    const uint32_t p0 = (uint32_t)(v << bit);
    const uint32_t p1 = (uint32_t)(bit ? (v >> (32 - bit)) : (v >> 32));
    const uint32_t p2 = (uint32_t)(bit ? (v >> (64 - bit)) : 0ull);
    const int b0 = __shfl_sync(kFull, limb, 0);
    const int k = limb - b0;
#pragma unroll
    for (int j = 0; j < 5; j++) {
        const unsigned long long c = warp_sum32((j == k ? p0 : 0u) + (j == k + 1 ? p1 : 0u) + (j == k + 2 ? p2 : 0u));
        if ((threadIdx.x & 31) == 0) slot[j] = c;
    }
    if ((threadIdx.x & 31) == 0) *base = b0;
}

// Lane i of the calling warp: limb i of sum q, before carries.
__device__ __forceinline__ unsigned long long gather_limb(const FinSmem& F, int q)
{
    const int i = (int)(threadIdx.x & 31);
    unsigned long long a = 0;
#pragma unroll
    for (int v = 0; v < kThreads / 32; v++) {
        const int j = i - F.base[v][q];
        if (j >= 0 && j < 5) a += F.slot[v][q][j];
    }
    return a;
}

static __device__ __noinline__ void st_finalize(const StatsBins* G, uint64_t n, double K, ez_stats_t* out,
                                                StatsSmem& S, uint32_t hist_window)
{
    const int t = threadIdx.x, wid = t >> 5, lane = t & 31;
    FinSmem& F = *reinterpret_cast<FinSmem*>(S.hist);
    __syncthreads();
    const unsigned long long h = __ldcg(&G->hist[t]);
    const long long s1 = (long long)__ldcg(&G->s1[t]);
    const unsigned long long s2 = __ldcg(&G->s2[t]);
    F.h[t] = h;
    out->hist[t] = h;
    {
        // v * 2^133 = +-M * 2^sh; v^2 * 2^266 = M^2 * 2^(2 sh); bin 255 holds no terms
        const int sh = (t ? t : 1) - 1;
        const bool live = t < 255;
        warp_slot_sums(F.slot[wid][0], &F.base[wid][0], live && s1 > 0 ? (unsigned long long)s1 : 0ull, sh);
        warp_slot_sums(F.slot[wid][1], &F.base[wid][1], live && s1 < 0 ? (unsigned long long)(-s1) : 0ull, sh);
        warp_slot_sums(F.slot[wid][2], &F.base[wid][2], live ? s2 : 0ull, 2 * sh);
        // counts are at most 2^40: two 20-bit halves
        const unsigned long long c = live ? h : 0ull;
        const unsigned long long nw = ((unsigned long long)__reduce_add_sync(kFull, (uint32_t)(c >> 20)) << 20) +
                                      __reduce_add_sync(kFull, (uint32_t)(c & 0xFFFFFu));
        if (lane == 0) F.nw[wid] = nw;
    }
    __syncthreads();
    if (wid > 1) return;
    unsigned long long n_fin = 0;
#pragma unroll
    for (int v = 0; v < kThreads / 32; v++) n_fin += F.nw[v];
    const double N = (double)n_fin;
    if (wid == 0) {
        const uint32_t P = warp_carry(gather_limb(F, 0)), Q = warp_carry(gather_limb(F, 1));
        const uint32_t d = __ballot_sync(kFull, P != Q);
        double s1d = 0.0;
        if (d) {
            const int k = 31 - __clz((int)d);
            const bool neg = __shfl_sync(kFull, P, k) < __shfl_sync(kFull, Q, k);
            const double m = warp_round(neg ? warp_sub(Q, P) : warp_sub(P, Q), -133);
            s1d = neg ? -m : m;
        }
        if (lane == 0) {
            F.s1d = s1d;
            if (n_fin >= 2) F.b = __dmul_rn(s1d, __ddiv_rn(s1d, N));
        }
    } else {
        const double s2d = warp_round(warp_carry(gather_limb(F, 2)), -266);
        if (lane == 0) F.s2d = s2d;
    }
    // warps 0 and 1 only; the rest of the CTA has returned
    asm volatile("bar.sync 1, 64;" ::: "memory");
    if (lane != 0) return;
    const double s1d = F.s1d, s2d = F.s2d;
    double var = 0.0;
    bool ok = false;
    if (n_fin >= 2) {
        var = __ddiv_rn(__dsub_rn(s2d, F.b), __dsub_rn(N, 1.0));
        ok = var > 0.0 && var <= 1.7976931348623157e308;
    }
    if (wid == 1) {
        out->sigma = ok ? __dsqrt_rn(var) : 0.0;
        return;
    }
    uint32_t rule = 1, E0 = 0;
    if (ok && !hist_window) {
        E0 = window_base(var, K);
        rule = 0;
    } else {
        // the densest run of 7 exponent bins, ties to the lowest base
        unsigned long long run = 0, best = 0;
        for (int E = 0; E < 7; E++) run += F.h[E];
        best = run;
        for (int b = 1; b <= 249; b++) {
            run += F.h[b + 6] - F.h[b - 1];
            if (run > best) { best = run; E0 = (uint32_t)b; }
        }
    }
    unsigned long long inwin = 0;
    for (uint32_t E = E0; E <= E0 + 6; E++) inwin += F.h[E];
    out->n = n;
    out->n_finite = n_fin;
    out->s1 = s1d;
    out->s2 = s2d;
    out->var = var;
    out->K = K;
    out->E0 = E0;
    out->rule = rule;
    out->n_escape = n - inwin;
}

}  // namespace ez
