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
// value the hot loop is integer work on shared memory only.  A CTA picks a
// 16-binade window [Elo, Elo+16) around the mode of a sample of its
// exponents.  A value inside it adds 2^22 + M to the lane-private cell of
// (sign, E) -- count in bits 22..31, sum of M in bits 0..21 -- and M^2 to the
// lane-private square cell of E; lane-private cells never conflict.  Values
// outside the window (and zeros, subnormals, Inf/NaN) go to per-exponent
// bins with shared-memory atomics.  At the end of a tile the CTA folds
// everything into per-shard global bins (64-bit atomics); the last CTA of the
// shard turns the bins into one big integer per sum, rounds it to nearest
// even, and derives var, sigma and the window base E0.
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

// Per-CTA accumulators (dynamic shared memory).  A CTA adds at most 32768
// values per tile (at most 128 per lane), so no cell or bin can overflow:
// 1023 values per packed cell, 128 * 65025 < 2^32 per square cell, and
// 32768 * 65025 < 2^32 per square bin.
struct StatsSmem {
    uint32_t cells[kThreads / 32][32][32];   // [warp][sign*16 + d][lane]
    uint32_t sq[kThreads / 32][16][32];      // [warp][d][lane]
    uint32_t cnt[256];
    int s1[256];
    uint32_t s2[256];
    uint32_t sample[256];
    uint32_t elo;
    uint32_t last;
};

constexpr uint32_t kCellOne = 1u << 22;

// Zero the CTA's accumulators and choose Elo from one exponent per thread
// (h0 = that thread's first value, or 0xFFFFFFFF for none).
__device__ __forceinline__ void st_begin(StatsSmem& S, uint32_t h0)
{
    const int t = threadIdx.x;
    S.cnt[t] = 0;
    S.s1[t] = 0;
    S.s2[t] = 0;
    S.sample[t] = 0;
    uint4* c = reinterpret_cast<uint4*>(&S.cells[0][0][0]);
    constexpr int kVec = (int)((sizeof(S.cells) + sizeof(S.sq)) / 16);
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

// One value h (16 bits).  `cell` = &S.cells[warp][0][lane], `sq` = &S.sq[warp][0][lane].
__device__ __forceinline__ void st_add(uint32_t h, uint32_t elo, uint32_t* cell, uint32_t* sq,
                                       StatsSmem& S)
{
    // v = sign*256 + E - Elo; in the window iff its low byte is below 16
    // (Elo <= 239 keeps E = 255 and E < Elo outside)
    const uint32_t v = (h >> 7) - elo;
    if ((v & 0xF0u) == 0) {
        const uint32_t k = (v & 0xFu) | ((v >> 4) & 0x10u);     // sign*16 + d
        const uint32_t m = h & 0x7Fu;
        atomicAdd(cell + 32 * k, kCellOne | 0x80u | m);
        atomicAdd(sq + 32 * (v & 0xFu), (m | 0x80u) * (m | 0x80u));
    } else {
        const uint32_t E = exp_of(h);
        atomicAdd(&S.cnt[E], 1u);
        if (E != 255u) {
            const uint32_t M = (E ? 128u : 0u) | (h & 0x7Fu);
            atomicAdd(&S.s1[E], (h & 0x8000u) ? -(int)M : (int)M);
            atomicAdd(&S.s2[E], M * M);
        }
    }
}

// Fold the CTA into the global bins; returns true in every thread of the CTA
// that is the `expected`-th to finish (it must then call st_finalize).
__device__ __forceinline__ bool st_end(StatsSmem& S, StatsBins* G, uint32_t expected)
{
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const uint32_t elo = S.elo;
    __syncthreads();
    // lane-private cells -> per-exponent CTA bins
#pragma unroll 4
    for (int d = 0; d < 16; d++) {
        const uint32_t cp = S.cells[wid][d][lane];
        const uint32_t cn = S.cells[wid][16 + d][lane];
        const uint32_t q = S.sq[wid][d][lane];
        const uint32_t cnt = (cp >> 22) + (cn >> 22);
        const int s1 = (int)(cp & 0x3FFFFFu) - (int)(cn & 0x3FFFFFu);
        const uint32_t wc = __reduce_add_sync(kFull, cnt);
        const int ws = __reduce_add_sync(kFull, s1);
        const uint32_t wq = __reduce_add_sync(kFull, q);
        if (lane == 0 && wc) {
            atomicAdd(&S.cnt[elo + d], wc);
            atomicAdd(&S.s1[elo + d], ws);
            atomicAdd(&S.s2[elo + d], wq);
        }
    }
    __syncthreads();
    // per-exponent bins -> global
    if (S.cnt[t]) atomicAdd(&G->hist[t], (unsigned long long)S.cnt[t]);
    if (S.s1[t]) atomicAdd(&G->s1[t], (unsigned long long)(long long)S.s1[t]);
    if (S.s2[t]) atomicAdd(&G->s2[t], (unsigned long long)S.s2[t]);
    __threadfence();
    __syncthreads();
    if (t == 0) S.last = (atomicAdd(&G->done, 1u) == expected - 1) ? 1u : 0u;
    __syncthreads();
    const bool last = S.last != 0;
    if (last) __threadfence();
    return last;
}

// ---- exact rounding of big sums --------------------------------------------

struct Big {
    uint32_t w[24];   // 768-bit non-negative integer, little-endian limbs
};

__device__ __forceinline__ void big_add_at(Big& b, unsigned long long x, int limb)
{
    unsigned long long c = x;
    for (int i = limb; i < 24 && c; i++) {
        const unsigned long long s = (unsigned long long)b.w[i] + (c & 0xffffffffull);
        b.w[i] = (uint32_t)s;
        c = (c >> 32) + (s >> 32);
    }
}

// b += v * 2^sh
__device__ __forceinline__ void big_add_shl(Big& b, unsigned long long v, int sh)
{
    const int limb = sh >> 5, bit = sh & 31;
    big_add_at(b, (v & 0xffffffffull) << bit, limb);
    big_add_at(b, (v >> 32) << bit, limb + 1);
}

__device__ __forceinline__ int big_cmp(const Big& a, const Big& b)
{
    for (int i = 23; i >= 0; i--)
        if (a.w[i] != b.w[i]) return a.w[i] > b.w[i] ? 1 : -1;
    return 0;
}

__device__ __forceinline__ void big_sub(Big& a, const Big& b)   // a >= b
{
    unsigned long long borrow = 0;
    for (int i = 0; i < 24; i++) {
        const unsigned long long bi = (unsigned long long)b.w[i] + borrow;
        borrow = (unsigned long long)a.w[i] < bi ? 1ull : 0ull;
        a.w[i] = (uint32_t)((unsigned long long)a.w[i] - bi);
    }
}

__device__ __forceinline__ uint32_t big_bit(const Big& b, int pos)
{
    return (pos < 0) ? 0u : (b.w[pos >> 5] >> (pos & 31)) & 1u;
}

// 2^e as a double, e in the normal range
__device__ __forceinline__ double pow2d(int e)
{
    return __longlong_as_double((long long)(e + 1023) << 52);
}

// b * 2^scale to the nearest double, ties to even
static __device__ double big_round(const Big& b, int scale)
{
    int top = -1;
    for (int i = 23; i >= 0; i--) {
        if (b.w[i]) { top = i; break; }
    }
    if (top < 0) return 0.0;
    const int L = top * 32 + (32 - __clz(b.w[top]));
    unsigned long long q = 0;
    const int keep = L < 53 ? L : 53;
    for (int i = L - 1; i >= L - keep; i--) q = (q << 1) | big_bit(b, i);
    int e = L - keep + scale;
    if (L > 53) {
        const uint32_t half = big_bit(b, L - 54);
        uint32_t sticky = 0;
        const int below = L - 54;          // bits [0, below) are the sticky bits
        for (int i = 0; i < (below >> 5); i++) sticky |= b.w[i];
        if (below & 31) sticky |= b.w[below >> 5] & ((1u << (below & 31)) - 1u);
        if (half && (sticky || (q & 1ull))) q++;
    }
    return __dmul_rn((double)q, pow2d(e));
}

// Window base from the variance: the largest e in 1..249 with
// var >= K * 2^(2(e-127)-1), else 0.
__device__ __forceinline__ uint32_t window_base(double var, double K)
{
    int lo = 0, hi = 249;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (var >= __dmul_rn(K, pow2d(2 * mid - 255))) lo = mid;
        else hi = mid - 1;
    }
    return (uint32_t)lo;
}

// The last CTA finalises: all its threads load the bins into shared memory
// (reusing the cell area), thread 0 does the exact arithmetic from there.
struct FinSmem {
    unsigned long long h[256];
    unsigned long long s1[256];
    unsigned long long s2[256];
};
static_assert(sizeof(FinSmem) <= sizeof(StatsSmem::cells), "finalise scratch fits the cells");

static __device__ void st_finalize(const StatsBins* G, uint64_t n, double K, ez_stats_t* out,
                                   StatsSmem& S)
{
    const int t = threadIdx.x;
    FinSmem& F = *reinterpret_cast<FinSmem*>(&S.cells[0][0][0]);
    __syncthreads();
    const unsigned long long h = __ldcg(&G->hist[t]);
    F.h[t] = h;
    F.s1[t] = __ldcg(&G->s1[t]);
    F.s2[t] = __ldcg(&G->s2[t]);
    out->hist[t] = h;
    __syncthreads();
    if (t != 0) return;
    Big P, Q, R;
    for (int i = 0; i < 24; i++) { P.w[i] = 0; Q.w[i] = 0; R.w[i] = 0; }
    unsigned long long n_fin = 0;
    for (int E = 0; E < 255; E++) {
        n_fin += F.h[E];
        if (!F.h[E]) continue;
        const int sh = (E ? E : 1) - 1;     // v * 2^133 = +-M * 2^sh
        const long long s1 = (long long)F.s1[E];
        if (s1 > 0) big_add_shl(P, (unsigned long long)s1, sh);
        else if (s1 < 0) big_add_shl(Q, (unsigned long long)(-s1), sh);
        if (F.s2[E]) big_add_shl(R, F.s2[E], 2 * sh);   // v^2 * 2^266 = M^2 * 2^(2 sh)
    }
    double s1d;
    if (big_cmp(P, Q) >= 0) {
        big_sub(P, Q);
        s1d = big_round(P, -133);
    } else {
        big_sub(Q, P);
        s1d = -big_round(Q, -133);
    }
    const double s2d = big_round(R, -266);
    double var = 0.0, sigma = 0.0;
    uint32_t rule = 1, E0 = 0;
    if (n_fin >= 2) {
        const double N = (double)n_fin;
        var = __ddiv_rn(__dsub_rn(s2d, __dmul_rn(s1d, __ddiv_rn(s1d, N))), __dsub_rn(N, 1.0));
        if (var > 0.0 && var <= 1.7976931348623157e308) {
            sigma = __dsqrt_rn(var);
            E0 = window_base(var, K);
            rule = 0;
        }
    }
    if (rule == 1) {
        // the densest run of 7 exponent bins, ties to the lowest base
        unsigned long long run = 0, best = 0;
        for (int E = 0; E < 7; E++) run += F.h[E];
        best = run;
        E0 = 0;
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
    out->sigma = sigma;
    out->K = K;
    out->E0 = E0;
    out->rule = rule;
    out->n_escape = n - inwin;
}

}  // namespace ez
