// k_fp8.cu -- the 3-bit exponent code on FP8 values (ZipCCL digest 3.3, last
// paragraph: FP8 E5M2 coded to 3 bits gives e = 0.75, E4M3 gives e ~ 0.88).
//
// Formats as in the OCP 8-bit floating-point specification: E5M2 (bias 15,
// infinities and NaN at exponent field 31) and E4M3 (bias 7, no infinities,
// NaN only at S.1111.111).  A value keeps its sign and mantissa bits raw, as
// 1 + m bit-planes (sign+mantissa field sm = sign << m | mantissa, plane q =
// bit q of sm); its exponent field E becomes the 3-bit code E - E0 + 1 of the
// window E0..E0+6 (three more planes) or code 0 with E appended to the
// chunk's escape list.  A coded value takes 1 + m + 3 bits: 6/8 and 7/8.
//
// Chunk layout (little-endian, all padding zero): 128-byte header {"EZF8",
// u8 version 1, u8 format (1 E5M2, 2 E4M3), u8 E0, u8 0, u64 n_c, u64 n_esc,
// u64 chunk_bytes, u32 chunk index, u32 W}; the 1 + m sign/mantissa planes
// and the 3 code planes, each ceil(n_c/8) bytes padded to 128 (bit j&7 of
// byte j>>3 belongs to value j); the escape index (u64 per 8192 values:
// escapes among the values before that point; padded to 128); the escapes
// (raw exponent fields in value order; padded to 128).
//
// Kernels.  A thread owns 32 consecutive values (32 bytes, two 16-byte
// accesses).  Its 8 bit-planes come from an 8x8 bit-matrix transpose of each
// 8-value group (three delta swaps on 64 bits) followed by a 4x4 byte
// transpose (byte permutes); decoding runs the same two transposes backwards
// (both are their own inverses).  Codes are computed bit-sliced, 32 values
// per operation: d = E - E0 by a ripple subtraction over the exponent
// planes, in-window = no borrow and d <= 6, code = d + 1.  Escape offsets use
// the decoupled look-back of ez_common.cuh over tiles of 4 index spans
// (encode) or the index (decode).
// Statistics: every byte pattern is counted exactly (one shared-memory
// reduction per value into lane-private copies, so no two lanes of a warp
// share an address or a bank); the last CTA forms the exact sums of the
// finite values and of their squares from the 256 pattern counts as 128-bit
// integers, rounds each once to double and places the window as for BF16.
#include <type_traits>

#include "ez_internal.h"
#include "ez_common.cuh"

namespace ezk {
using namespace ez;

struct Fp8Fmt {
    uint32_t ebits, mbits, bias, emax0, tag;   // tag: the header's format byte
};

__host__ __device__ constexpr Fp8Fmt fp8_fmt(uint32_t codec)
{
    return codec == EZ_CODEC_FP8_E5M2 ? Fp8Fmt{5u, 2u, 15u, 25u, 1u} : Fp8Fmt{4u, 3u, 7u, 9u, 2u};
}

// ---- bit-plane transposes ------------------------------------------------------
// 8 values of one byte each in x (value r in byte r) -> byte c holds bit c of
// every value (bit r = value r).  Delta swaps of the 1x1, 2x2 and 4x4 blocks
// of the 8x8 bit matrix; applying it twice gives x back.
__device__ __forceinline__ unsigned long long tr8x8(unsigned long long x)
{
    unsigned long long t;
    t = (x ^ (x >> 7)) & 0x00AA00AA00AA00AAull;
    x ^= t ^ (t << 7);
    t = (x ^ (x >> 14)) & 0x0000CCCC0000CCCCull;
    x ^= t ^ (t << 14);
    t = (x ^ (x >> 28)) & 0x00000000F0F0F0F0ull;
    x ^= t ^ (t << 28);
    return x;
}

// 4x4 byte transpose: out[k] byte g = in[g] byte k.
__device__ __forceinline__ void tr4x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t* o)
{
    const uint32_t A = __byte_perm(a0, a1, 0x5140), B = __byte_perm(a0, a1, 0x7362);
    const uint32_t C = __byte_perm(a2, a3, 0x5140), D = __byte_perm(a2, a3, 0x7362);
    o[0] = __byte_perm(A, C, 0x5410);
    o[1] = __byte_perm(A, C, 0x7632);
    o[2] = __byte_perm(B, D, 0x5410);
    o[3] = __byte_perm(B, D, 0x7632);
}

// 32 bytes (value 4q+j in byte j of w[q]) -> planes P[k], bit i = bit k of value i.
__device__ __forceinline__ void to_planes(const uint32_t* w, uint32_t* P)
{
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int g = 0; g < 4; g++) {
        const unsigned long long x = tr8x8((unsigned long long)w[2 * g] | (unsigned long long)w[2 * g + 1] << 32);
        lo[g] = (uint32_t)x;
        hi[g] = (uint32_t)(x >> 32);
    }
    tr4x4(lo[0], lo[1], lo[2], lo[3], P);
    tr4x4(hi[0], hi[1], hi[2], hi[3], P + 4);
}

__device__ __forceinline__ void from_planes(const uint32_t* P, uint32_t* w)
{
    uint32_t lo[4], hi[4];
    tr4x4(P[0], P[1], P[2], P[3], lo);
    tr4x4(P[4], P[5], P[6], P[7], hi);
#pragma unroll
    for (int g = 0; g < 4; g++) {
        const unsigned long long x = tr8x8((unsigned long long)lo[g] | (unsigned long long)hi[g] << 32);
        w[2 * g] = (uint32_t)x;
        w[2 * g + 1] = (uint32_t)(x >> 32);
    }
}

__device__ __forceinline__ uint32_t bitmask_of(uint32_t v, int j) { return ((v >> j) & 1u) ? 0xFFFFFFFFu : 0u; }

// Borrow out of a - b - c (bit-sliced): (~a & b) | (~(a ^ b) & c).
__device__ __forceinline__ uint32_t borrow3(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x8E;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
// Carry out of a + b + c (bit-sliced majority).
__device__ __forceinline__ uint32_t carry3(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xE8;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// ---- layout ----------------------------------------------------------------------
__host__ __device__ __forceinline__ uint64_t f8_plane(uint64_t n_c) { return rup(cdiv(n_c, 8), 128); }
__host__ __device__ __forceinline__ uint64_t f8_idx_bytes(uint64_t n_c) { return rup(8 * cdiv(n_c, kTile), 128); }
__host__ __device__ __forceinline__ uint64_t f8_bytes(uint64_t n_c, uint64_t n_esc, uint32_t nsm)
{
    return 128 + (nsm + 3) * f8_plane(n_c) + f8_idx_bytes(n_c) + rup(n_esc, 128);
}

__device__ __forceinline__ uint32_t f8_le_byte(uint64_t v, int k) { return (uint32_t)(v >> (8 * k)) & 0xFFu; }

__device__ __forceinline__ uint32_t f8_header_byte(int b, const Fp8Fmt& f, uint32_t E0, uint64_t n_c,
                                                   uint64_t n_esc, uint64_t bytes, uint32_t c, uint32_t W)
{
    switch (b) {
        case 0: return 'E';
        case 1: return 'Z';
        case 2: return 'F';
        case 3: return '8';
        case 4: return 1;
        case 5: return f.tag;
        case 6: return E0;
        default: break;
    }
    if (b < 8) return 0;
    if (b < 16) return f8_le_byte(n_c, b - 8);
    if (b < 24) return f8_le_byte(n_esc, b - 16);
    if (b < 32) return f8_le_byte(bytes, b - 24);
    if (b < 36) return f8_le_byte(c, b - 32);
    if (b < 40) return f8_le_byte(W, b - 36);
    return 0;
}

// The thread's 32 values (cnt of them valid) as 8 words; missing values are 0.
__device__ __forceinline__ void load32(const uint8_t* p, uint32_t cnt, uint32_t* w)
{
    if (cnt == 32) {
        const uint4 a = ld_v4_nc(p), b = ld_v4_nc(p + 16);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        return;
    }
#pragma unroll
    for (int q = 0; q < 8; q++) w[q] = 0;
    // fixed indexes, so that w stays in registers
#pragma unroll
    for (uint32_t i = 0; i < 32; i++)
        if (i < cnt) w[i >> 2] |= (uint32_t)p[i] << (8 * (i & 3));
}

// =================================================================== statistics

struct F8Bins {                      // in the workspace's statistics bins (zeroed per call)
    unsigned long long cnt[256];     // count of each byte pattern
    unsigned int done;               // CTAs that have flushed
};

constexpr int kF8Copies = 32;        // lane-private copies of the pattern counts

struct u128p {
    unsigned long long lo, hi;
};
__device__ __forceinline__ u128p add128(u128p a, u128p b)
{
    u128p r;
    r.lo = a.lo + b.lo;
    r.hi = a.hi + b.hi + (r.lo < a.lo ? 1ull : 0ull);
    return r;
}
__device__ __forceinline__ u128p sub128(u128p a, u128p b)
{
    u128p r;
    r.lo = a.lo - b.lo;
    r.hi = a.hi - b.hi - (a.lo < b.lo ? 1ull : 0ull);
    return r;
}
__device__ __forceinline__ bool ge128(u128p a, u128p b) { return a.hi != b.hi ? a.hi > b.hi : a.lo >= b.lo; }
// v * 2^s for v < 2^64, s < 128
__device__ __forceinline__ u128p shl128(unsigned long long v, uint32_t s)
{
    u128p r;
    if (s == 0) {
        r.lo = v;
        r.hi = 0;
    } else if (s < 64) {
        r.lo = v << s;
        r.hi = v >> (64 - s);
    } else {
        r.lo = 0;
        r.hi = v << (s - 64);
    }
    return r;
}
// v * m for v < 2^64, m < 2^16 (a 128-bit product)
__device__ __forceinline__ u128p mul128(unsigned long long v, uint32_t m)
{
    u128p r;
    r.lo = v * (unsigned long long)m;
    r.hi = __umul64hi(v, (unsigned long long)m);
    return r;
}
__device__ __forceinline__ u128p shl128p(u128p v, uint32_t s)
{
    if (s == 0) return v;
    u128p r;
    if (s < 64) {
        r.hi = (v.hi << s) | (v.lo >> (64 - s));
        r.lo = v.lo << s;
    } else {
        r.hi = v.lo << (s - 64);
        r.lo = 0;
    }
    return r;
}
__device__ __forceinline__ u128p shfl_xor128(u128p v, int o)
{
    u128p r;
    r.lo = __shfl_xor_sync(kFull, v.lo, o);
    r.hi = __shfl_xor_sync(kFull, v.hi, o);
    return r;
}

// v rounded once to the nearest double (ties to even): the top 64 bits with
// every lower bit folded into bit 0 (below the rounding position, so the
// conversion's tie-break is unchanged), converted, then scaled back exactly.
__device__ __forceinline__ double round128(u128p v)
{
    if (v.hi == 0) return __ull2double_rn(v.lo);
    const int s = 64 - __clzll((long long)v.hi);   // 1..64
    unsigned long long top, rest;
    if (s == 64) {
        top = v.hi;
        rest = v.lo;
    } else {
        top = (v.hi << (64 - s)) | (v.lo >> s);
        rest = v.lo << (64 - s);
    }
    top |= rest != 0 ? 1ull : 0ull;
    return ldexp(__ull2double_rn(top), s);
}

template <uint32_t kCodec>
__global__ void __launch_bounds__(kThreads) k_fp8_stats(const uint8_t* x, uint64_t n, F8Bins* G,
                                                       ez_fp8_stats_t* out, double K, uint32_t hist_window)
{
    extern __shared__ __align__(16) uint32_t s_cnt[];   // [256 patterns][32 lanes]
    __shared__ unsigned long long s_hist[32];
    __shared__ u128p s_part[3][kThreads / 32];
    __shared__ unsigned long long s_fin[kThreads / 32];
    __shared__ uint32_t s_last;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    for (int i = t; i < 256 * kF8Copies / 4; i += kThreads)
        reinterpret_cast<uint4*>(s_cnt)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(s_cnt) + 4u * (uint32_t)lane;
    const uint64_t nw = n / 16;
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    uint64_t i = (uint64_t)blockIdx.x * kThreads + (uint64_t)t;
    // four 16-byte loads in flight per thread
    for (; i + 3 * stride < nw; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; u++) v[u] = ld_v4_nc(x + 16 * (i + (uint64_t)u * stride));
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const uint32_t ws[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int q = 0; q < 4; q++)
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    const uint32_t pat = __byte_perm(ws[q], 0u, 0x4440u | (uint32_t)b);
                    asm volatile("red.shared.add.u32 [%0], 1;" :: "r"(base + (pat << 7)) : "memory");
                }
        }
    }
    for (; i < nw; i += stride) {
        const uint4 v = ld_v4_nc(x + 16 * i);
        const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; q++)
#pragma unroll
            for (int b = 0; b < 4; b++) {
                const uint32_t pat = __byte_perm(ws[q], 0u, 0x4440u | (uint32_t)b);
                asm volatile("red.shared.add.u32 [%0], 1;" :: "r"(base + (pat << 7)) : "memory");
            }
    }
    if (blockIdx.x == 0)
        for (uint64_t j = nw * 16 + (uint64_t)t; j < n; j += kThreads)
            asm volatile("red.shared.add.u32 [%0], 1;" :: "r"(base + ((uint32_t)x[j] << 7)) : "memory");
    grid_dep_wait();   // the bins were cleared by the kernel before
    __syncthreads();
    {
        // thread t folds pattern t's copies (each at most the CTA's values)
        const uint4* row = reinterpret_cast<const uint4*>(s_cnt + t * kF8Copies);
        unsigned long long s = 0;
#pragma unroll
        for (int q = 0; q < kF8Copies / 4; q++) {
            const uint4 c = row[q];
            s += (unsigned long long)c.x + c.y + c.z + c.w;
        }
        if (s) atomicAdd(&G->cnt[t], s);
    }
    __threadfence();
    __syncthreads();
    if (t == 0) s_last = atomicAdd(&G->done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA: exact sums from the pattern counts
    constexpr Fp8Fmt f = fp8_fmt(kCodec);
    if (t < 32) s_hist[t] = 0;
    __syncthreads();
    const uint32_t pat = (uint32_t)t;
    const unsigned long long c = __ldcg(&G->cnt[pat]);
    const uint32_t E = (pat >> f.mbits) & ((1u << f.ebits) - 1u);
    const uint32_t man = pat & ((1u << f.mbits) - 1u);
    const bool finite = f.ebits == 5 ? E != 31u : !(E == 15u && man == 7u);
    if (c) atomicAdd(&s_hist[E], c);
    // v * 2^U = +-M * 2^sh, M = E ? 2^m + man : man, sh = max(E, 1) - 1,
    // U = bias + m - 1
    const uint32_t M = (E ? (1u << f.mbits) : 0u) + man;
    const uint32_t sh = (E ? E : 1u) - 1u;
    u128p pos = {0, 0}, neg = {0, 0}, sq = {0, 0};
    unsigned long long fin = 0;
    if (finite && c) {
        fin = c;
        if (M) {
            const u128p t1 = shl128(c * M, sh);
            if (pat & 0x80u) neg = t1;
            else pos = t1;
            sq = shl128p(mul128(c, M * M), 2 * sh);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        pos = add128(pos, shfl_xor128(pos, o));
        neg = add128(neg, shfl_xor128(neg, o));
        sq = add128(sq, shfl_xor128(sq, o));
        fin += __shfl_xor_sync(kFull, fin, o);
    }
    if (lane == 0) {
        s_part[0][wid] = pos;
        s_part[1][wid] = neg;
        s_part[2][wid] = sq;
        s_fin[wid] = fin;
    }
    __syncthreads();
    if (t < 32) out->hist[t] = t < (1 << f.ebits) ? s_hist[t] : 0ull;
    if (t != 0) return;
    u128p P = {0, 0}, Q = {0, 0}, R = {0, 0};
    unsigned long long nf = 0;
    for (int k = 0; k < kThreads / 32; k++) {
        P = add128(P, s_part[0][k]);
        Q = add128(Q, s_part[1][k]);
        R = add128(R, s_part[2][k]);
        nf += s_fin[k];
    }
    const int U = (int)(f.bias + f.mbits) - 1;
    double s1;
    if (ge128(P, Q)) s1 = ldexp(round128(sub128(P, Q)), -U);
    else s1 = -ldexp(round128(sub128(Q, P)), -U);
    const double s2 = ldexp(round128(R), -2 * U);
    double var = 0.0, sigma = 0.0;
    uint32_t E0 = 0, rule = 1;
    if (nf >= 2) {
        const double N = __ull2double_rn(nf);
        var = __ddiv_rn(__dsub_rn(s2, __dmul_rn(s1, __ddiv_rn(s1, N))), __dsub_rn(N, 1.0));
        if (var > 0.0 && isfinite(var)) {
            sigma = __dsqrt_rn(var);
            if (!hist_window) {
                // the integer nearest x_opt, ties up: the largest k with
                // var >= K 2^(2k-1), as the field value bias + k
                for (uint32_t e = 1; e <= f.emax0; e++) {
                    const int k = (int)e - (int)f.bias;
                    if (var >= ldexp(K, 2 * k - 1)) E0 = e;
                }
                rule = 0;
            }
        }
    }
    if (rule == 1) {
        unsigned long long best = 0;
        E0 = 0;
        for (uint32_t b = 0; b <= f.emax0; b++) {
            unsigned long long s = 0;
            for (uint32_t e = b; e <= b + 6; e++) s += s_hist[e];
            if (s > best) {
                best = s;
                E0 = b;
            }
        }
    }
    unsigned long long inw = 0;
    for (uint32_t e = E0; e <= E0 + 6; e++) inw += s_hist[e];
    out->n = n;
    out->n_finite = nf;
    out->s1 = s1;
    out->s2 = s2;
    out->var = var;
    out->sigma = sigma;
    out->K = K;
    out->E0 = E0;
    out->rule = rule;
    out->n_escape = n - inw;
}

// =================================================================== encode

struct F8Enc {
    const uint8_t* x;
    uint8_t* out;
    uint64_t slot;
    uint64_t* sizes;
    const ez_fp8_stats_t* st;
    uint32_t* dstatus;
    uint64_t n, L;
    uint32_t W, first, count, tpc;
    unsigned long long* state;
    uint32_t* counter;
    uint32_t* abort;
};

// One CTA per tile of kF8Spans index spans (4 x 8192 values), tiles taken in
// order from a counter (dealt round-robin over the chunks), so a tile's
// look-back only waits on tiles whose CTAs already run.  Two spans at a time
// (each thread's 32 bytes of both requested together; one block scan of the
// pair's two escape counts, on one of two alternating warp-total buffers, so
// a pair costs one barrier): the planes are stored at once, the scan places
// each thread's escapes in the tile's shared staging area; one look-back per
// tile then gives the escape prefix, the index entries of its spans and the
// place of the staged escapes (on a chunk's last tile also the header,
// padding and size).
constexpr uint32_t kF8Spans = 4;
static_assert(kF8Spans % 2 == 0, "spans are coded in pairs");
constexpr uint32_t kF8TileV = kF8Spans * kTile;

template <uint32_t kCodec>
__global__ void __launch_bounds__(kThreads) k_fp8_encode(F8Enc a)
{
    __shared__ uint32_t s_tile;
    __shared__ unsigned long long s_warp[2][kThreads / 32];   // by span-pair parity
    __shared__ unsigned long long s_prefix;
    __shared__ uint32_t s_base[kF8Spans + 1];
    __shared__ __align__(16) uint8_t s_esc[kF8TileV + 16];
    const int t = threadIdx.x;
    grid_dep_wait();   // the counters and tile states were cleared by the kernel before
    constexpr Fp8Fmt f = fp8_fmt(kCodec);
    constexpr uint32_t nsm = 1 + f.mbits;
    uint32_t E0 = __ldg(&a.st->E0);
    if (E0 > f.emax0) {
        if (t == 0) atomicOr(a.dstatus, EZ_DSTAT_BAD_STATS);
        E0 = 0;
    }
    const uint32_t tpt = (uint32_t)cdiv(a.tpc, kF8Spans);   // tiles per chunk
    const uint32_t id = next_tile(a.counter, &s_tile);
    const TilePos tp = tile_pos(id, a.count, tpt);
    const uint32_t ci = tp.ci, lt = tp.lt;
    const uint32_t c = a.first + ci;
    const uint64_t n_c = shard_values(a.n, a.L, c);
    uint8_t* o = a.out + (uint64_t)ci * a.slot;
    const uint64_t plane = f8_plane(n_c);
    uint8_t* pl = o + 128;
    uint8_t* idx = pl + (nsm + 3) * plane;
    uint8_t* esc = idx + f8_idx_bytes(n_c);
    const uint32_t tv = 32u * (uint32_t)t;
    uint32_t base = 0;                 // escapes of the tile's earlier spans (uniform)
    // spans in pairs: both spans' bytes requested together, one block scan of
    // the two escape counts (16-bit fields; a span holds at most 8192).  A tile
    // whose spans are all full takes an instance without per-span counts and
    // masks (0.147 -> 0.139 ms at 2^28 values).
    auto code_pairs = [&](auto full_tag) {
        constexpr bool kFullT = decltype(full_tag)::value;
#pragma unroll 1
        for (uint32_t sp = 0; sp < kF8Spans; sp += 2) {
            uint32_t w[2][8];
            uint32_t cnt[2];
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint64_t v0 = ((uint64_t)lt * kF8Spans + sp + h) * kTile;
                if constexpr (kFullT) {
                    cnt[h] = 32;
                } else {
                    const uint32_t nv = v0 < n_c ? (uint32_t)umin64(kTile, n_c - v0) : 0u;
                    cnt[h] = tv < nv ? min(32u, nv - tv) : 0u;
                }
                if (kFullT || cnt[h] == 32) {
                    const uint8_t* q = a.x + (uint64_t)ci * a.L + v0 + tv;
                    const uint4 x0 = ld_v4_nc(q), x1 = ld_v4_nc(q + 16);
                    w[h][0] = x0.x; w[h][1] = x0.y; w[h][2] = x0.z; w[h][3] = x0.w;
                    w[h][4] = x1.x; w[h][5] = x1.y; w[h][6] = x1.z; w[h][7] = x1.w;
                } else {
                    load32(a.x + (uint64_t)ci * a.L + v0 + tv, cnt[h], w[h]);
                }
            }
            uint32_t escm[2] = {0, 0}, e[2][5];
#pragma unroll
            for (int h = 0; h < 2; h++) {
#pragma unroll
                for (int j = 0; j < 5; j++) e[h][j] = 0;
                const uint32_t cnt_v = cnt[h];
                if (kFullT || cnt_v) {
                    const uint64_t v0 = ((uint64_t)lt * kF8Spans + sp + h) * kTile;
                    uint32_t R[8];
                    to_planes(w[h], R);
                    const uint32_t vm = (kFullT || cnt_v == 32) ? 0xFFFFFFFFu : ((1u << cnt_v) - 1u);
                    // d = E - E0 over the exponent planes R[m .. m+ebits)
                    uint32_t d[5], br = 0;
#pragma unroll
                    for (int j = 0; j < 5; j++) {
                        if (j < (int)f.ebits) {
                            const uint32_t ej = R[f.mbits + j], k = bitmask_of(E0, j);
                            e[h][j] = ej;
                            d[j] = ej ^ k ^ br;
                            br = borrow3(ej, k, br);
                        } else {
                            d[j] = 0;
                        }
                    }
                    const uint32_t in = ~br & ~(d[3] | d[4]) & ~(d[0] & d[1] & d[2]) & vm;
                    escm[h] = ~in & vm;
                    // sign/mantissa planes: mantissa bits, then the sign
                    uint8_t* pt = pl + (v0 + tv) / 8;
#pragma unroll
                    for (uint32_t q = 0; q < 4; q++)
                        if (q < nsm) *reinterpret_cast<uint32_t*>(pt + q * plane) = (q < f.mbits ? R[q] : R[7]) & vm;
                    // code = d + 1 inside the window
                    *reinterpret_cast<uint32_t*>(pt + nsm * plane) = ~d[0] & in;
                    *reinterpret_cast<uint32_t*>(pt + (nsm + 1) * plane) = (d[1] ^ d[0]) & in;
                    *reinterpret_cast<uint32_t*>(pt + (nsm + 2) * plane) = (d[2] ^ (d[1] & d[0])) & in;
                }
            }
            unsigned long long tot;
            const unsigned long long ex = block_excl_scan((unsigned long long)__popc(escm[0]) |
                                                              (unsigned long long)__popc(escm[1]) << 16,
                                                          s_warp[(sp >> 1) & 1u], &tot);
            // the thread's escapes, in value order (raw exponent fields), staged
#pragma unroll
            for (int h = 0; h < 2; h++) {
                uint32_t m = escm[h], r = base + (uint32_t)((ex >> (16 * h)) & 0xFFFFull);
                while (m) {
                    const int i = __ffs(m) - 1;
                    m &= m - 1;
                    uint32_t eb = 0;
#pragma unroll
                    for (int j = 0; j < 5; j++) eb |= ((e[h][j] >> i) & 1u) << j;
                    s_esc[r++] = (uint8_t)eb;
                }
                if (t == 0) s_base[sp + h] = base;
                base += (uint32_t)((tot >> (16 * h)) & 0xFFFFull);
            }
            // the next pair's scan writes the other s_warp buffer; this one is
            // written again two pairs on, after the next scan's barrier
        }
    };
    if (((uint64_t)lt + 1) * kF8TileV <= n_c) code_pairs(std::true_type{});
    else code_pairs(std::false_type{});
    const unsigned long long P = tile_prefix(a.state, ci * tpt + lt, ci * tpt, base, &s_prefix,
                                             a.dstatus, a.abort);
    if ((uint32_t)t < kF8Spans) {
        const uint64_t span = (uint64_t)lt * kF8Spans + t;
        if (span * kTile < n_c) *reinterpret_cast<unsigned long long*>(idx + 8ull * span) = P + s_base[t];
    }
    for (uint32_t i = (uint32_t)t; i < base; i += kThreads) esc[P + i] = s_esc[i];
    if (lt == tpt - 1) {
        const uint64_t n_esc = P + base;
        const uint64_t bytes = f8_bytes(n_c, n_esc, nsm);
        const uint64_t pb = cdiv(n_c, 8), ib = 8 * cdiv(n_c, kTile), ibytes = f8_idx_bytes(n_c);
        for (int q = t; q < 128; q += kThreads) {
            o[q] = (uint8_t)f8_header_byte(q, f, E0, n_c, n_esc, bytes, c, a.W);
            if (pb + q < plane)
                for (uint32_t k = 0; k < nsm + 3; k++) pl[k * plane + pb + q] = 0;
            if (ib + q < ibytes) idx[ib + q] = 0;
            if (n_esc + q < rup(n_esc, 128)) esc[n_esc + q] = 0;
        }
        if (t == 0) a.sizes[ci] = bytes;
    }
}

// =================================================================== decode

struct F8Dec {
    const uint8_t* in;
    const uint64_t* offsets;
    uint8_t* out;
    uint32_t* dstatus;
    uint64_t n, L;
    uint32_t W, first, count, tpc;
    FastDiv tpcd;         // tpc, for the CTA index split
};

// One CTA per 8192-value span, no inter-span dependence (the span's escape
// prefix is the chunk's index entry).  Header checks in the oracle's order;
// the index is checked against the span's own escape count, so the escapes
// read always lie inside the escape section.
// kVPT values per thread in kVPT / 32 words of 32 values (64: 128 threads per
// span, so the per-thread setup -- offsets, header checks, scan, index
// checks -- is spread over 64 one-byte values: 0.160 -> 0.124 ms at 2^28).
template <uint32_t kCodec, int kVPT>
__global__ void __launch_bounds__(kTile / kVPT) k_fp8_decode(F8Dec a)
{
    constexpr int kThr = kTile / kVPT, kW = kVPT / 32;
    static_assert(kW == 1 || kW == 2, "32 or 64 values per thread");
    __shared__ uint32_t s_bad, s_E0;
    __shared__ unsigned long long s_nesc;
    __shared__ uint32_t s_warp32[kThr / 32];
    __shared__ __align__(16) uint8_t s_esc[kTile + 16];
    const int t = threadIdx.x;
    constexpr Fp8Fmt f = fp8_fmt(kCodec);
    constexpr uint32_t nsm = 1 + f.mbits;
    uint32_t ci, lt;
    chunk_tile(blockIdx.x, a.tpcd, ci, lt);
    const uint32_t c = a.first + ci;
    const uint64_t n_c = shard_values(a.n, a.L, c);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t nv = v0 < n_c ? (uint32_t)umin64(kTile, n_c - v0) : 0u;
    const uint64_t off = __ldg(a.offsets + ci), end = __ldg(a.offsets + ci + 1);
    const uint64_t avail = end >= off ? end - off : 0ull;
    const uint8_t* p = a.in + off;
    const uint64_t plane = f8_plane(n_c);
    const uint64_t sec_idx = 128 + (nsm + 3) * plane;
    const uint64_t sec_esc = sec_idx + f8_idx_bytes(n_c);
    const uint64_t n_idx = cdiv(n_c, kTile);
    const bool fixed_ok = (off & 15u) == 0 && end >= off && avail >= sec_esc;
    const uint32_t tv = (uint32_t)kVPT * (uint32_t)t;
    const uint32_t cnt_v = tv < nv ? min((uint32_t)kVPT, nv - tv) : 0u;
    uint32_t pw[kW][7];
#pragma unroll
    for (int j = 0; j < kW; j++)
#pragma unroll
        for (int q = 0; q < 7; q++) pw[j][q] = 0;
    unsigned long long idx_here = 0, idx_next = 0;
    if (fixed_ok) {
        if (cnt_v) {
            // whole words: a word past the chunk's last value lies in the
            // plane's zero padding
            const uint8_t* pt = p + 128 + (v0 + tv) / 8;
#pragma unroll
            for (uint32_t q = 0; q < 7; q++) {
                if (q < nsm + 3) {
                    if (kW == 2) {   // 8-byte aligned: (v0 + tv) / 8 = 1024 lt + 8 t
                        const uint2 u = __ldg(reinterpret_cast<const uint2*>(pt + q * plane));
                        pw[0][q] = u.x;
                        pw[kW - 1][q] = u.y;
                    } else {
                        pw[0][q] = __ldg(reinterpret_cast<const uint32_t*>(pt + q * plane));
                    }
                }
            }
        }
        if (lt < n_idx) idx_here = __ldg(reinterpret_cast<const unsigned long long*>(p + sec_idx) + lt);
        if (lt + 1 < n_idx) idx_next = __ldg(reinterpret_cast<const unsigned long long*>(p + sec_idx) + lt + 1);
    }
    if (t == 0) {
        uint32_t bad = 0;
        s_E0 = 0;
        s_nesc = 0;
        if (off & 15u) {
            bad = EZ_DSTAT_MISALIGNED;
        } else if (end < off || avail < 128) {
            bad = EZ_DSTAT_BAD_SIZE;
        } else {
            const uint4 h0 = *reinterpret_cast<const uint4*>(p), h1 = *reinterpret_cast<const uint4*>(p + 16);
            const uint4 h2 = *reinterpret_cast<const uint4*>(p + 32);
            const uint64_t n_hdr = (uint64_t)h0.z | (uint64_t)h0.w << 32;
            const uint64_t n_esc = (uint64_t)h1.x | (uint64_t)h1.y << 32;
            const uint64_t bytes = (uint64_t)h1.z | (uint64_t)h1.w << 32;
            const uint32_t ver = h0.y & 0xFFu, fmt = (h0.y >> 8) & 0xFFu, E0 = (h0.y >> 16) & 0xFFu;
            if (h0.x != 0x38465A45u || ver != 1u || fmt != f.tag || E0 > f.emax0 || n_hdr != n_c ||
                h2.x != c || h2.y != a.W)
                bad = EZ_DSTAT_BAD_HEADER;
            else if (n_esc > n_c)
                bad = EZ_DSTAT_BAD_COUNT;
            else if (bytes != f8_bytes(n_c, n_esc, nsm) || bytes > avail)
                bad = EZ_DSTAT_BAD_SIZE;
            s_E0 = E0;
            s_nesc = n_esc;
        }
        s_bad = bad;
    }
    uint32_t vm[kW], escm[kW];
    uint32_t my = 0;
#pragma unroll
    for (int j = 0; j < kW; j++) {
        const uint32_t cj = cnt_v > 32u * j ? min(32u, cnt_v - 32u * j) : 0u;
        vm[j] = cj >= 32 ? 0xFFFFFFFFu : ((1u << cj) - 1u);
        escm[j] = ~(pw[j][nsm] | pw[j][nsm + 1] | pw[j][nsm + 2]) & vm[j];
        my += __popc(escm[j]);
    }
    const int lane = t & 31, wid = t >> 5;
    uint32_t xs = my;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, xs, o);
        if (lane >= o) xs += y;
    }
    if (lane == 31) s_warp32[wid] = xs;
    __syncthreads();   // also publishes s_bad
    uint32_t wpre = 0, agg32 = 0;
#pragma unroll
    for (int i = 0; i < kThr / 32; i++) {
        const uint32_t v = s_warp32[i];
        wpre += i < wid ? v : 0u;
        agg32 += v;
    }
    const uint32_t excl = wpre + xs - my;
    const uint32_t bad = s_bad;
    if (bad) {
        if (lt == 0 && t == 0) atomicOr(a.dstatus, bad);
        return;
    }
    const uint32_t E0 = s_E0;
    const unsigned long long n_esc = s_nesc;
    const unsigned long long agg = agg32;
    const unsigned long long P = lt < n_idx ? idx_here : n_esc;
    const unsigned long long want = lt + 1 < n_idx ? idx_next : n_esc;
    const bool idx_ok = (lt != 0 || n_idx == 0 || P == 0) && P <= n_esc && agg <= n_esc - P &&
                        (lt >= n_idx || P + agg == want);
    if (!idx_ok) {
        if (t == 0) atomicOr(a.dstatus, EZ_DSTAT_BAD_COUNT);
        return;
    }
    // the span's escapes [P, P + agg) into shared memory
    const uint8_t* esrc = p + sec_esc + P;
    for (uint32_t i = (uint32_t)t; i < agg32; i += kThr) s_esc[i] = esrc[i];
    __syncthreads();
    if (!cnt_v) return;
    uint8_t* ot = a.out + (uint64_t)ci * a.L + v0 + tv;
    uint32_t r = excl;
    const uint32_t emask = (1u << f.ebits) - 1u;
#pragma unroll
    for (int j = 0; j < kW; j++) {
        if (32u * j >= cnt_v) break;
        const uint32_t c0 = pw[j][nsm] & vm[j], c1 = pw[j][nsm + 1] & vm[j], c2 = pw[j][nsm + 2] & vm[j];
        // E = code - 1 + E0 inside the window (bit-sliced over 32 values)
        const uint32_t d0 = ~c0, b0 = ~c0;
        const uint32_t d1 = c1 ^ b0, b1 = ~c1 & b0;
        const uint32_t d2 = c2 ^ b1;
        const uint32_t dd[5] = {d0, d1, d2, 0u, 0u};
        uint32_t e[5], cy = 0;
#pragma unroll
        for (int k = 0; k < 5; k++) {
            const uint32_t kk = bitmask_of(E0, k);
            e[k] = dd[k] ^ kk ^ cy;
            cy = carry3(dd[k], kk, cy);
        }
        // escaped values take their exponent field from the list
        uint32_t m = escm[j];
        while (m) {
            const int i = __ffs(m) - 1;
            m &= m - 1;
            const uint32_t b = s_esc[r++] & emask;
            const uint32_t bit = 1u << i;
#pragma unroll
            for (int k = 0; k < 5; k++) e[k] = (e[k] & ~bit) | (((b >> k) & 1u) ? bit : 0u);
        }
        uint32_t R[8];
#pragma unroll
        for (int k = 0; k < 8; k++) R[k] = 0;
#pragma unroll
        for (uint32_t q = 0; q < 3; q++)
            if (q < f.mbits) R[q] = pw[j][q] & vm[j];
        R[7] = pw[j][f.mbits] & vm[j];
#pragma unroll
        for (int k = 0; k < 5; k++)
            if (k < (int)f.ebits) R[f.mbits + k] = e[k] & vm[j];
        uint32_t w[8];
        from_planes(R, w);
        const uint32_t cj = min(32u, cnt_v - 32u * j);
        uint8_t* oj = ot + 32u * j;
        if (cj == 32) {
            st_v4(oj, make_uint4(w[0], w[1], w[2], w[3]));
            st_v4(oj + 16, make_uint4(w[4], w[5], w[6], w[7]));
        } else {
#pragma unroll
            for (uint32_t i = 0; i < 32; i++)
                if (i < cj) oj[i] = (uint8_t)(w[i >> 2] >> (8 * (i & 3)));
        }
    }
}

// =================================================================== launchers

uint64_t fp8_slot_bytes(uint32_t codec, uint64_t L)
{
    const Fp8Fmt f = fp8_fmt(codec);
    return f8_bytes(L, L, 1 + f.mbits);
}

template <uint32_t kCodec>
static cudaError_t fp8_stats_launch(const ez_plan_s* p, const uint8_t* x, uint64_t n, ez_fp8_stats_t* out,
                                    const WsView& w, cudaStream_t s)
{
    static PerDeviceAttr smem_attr;
    const int smem = 256 * kF8Copies * 4;
    cudaError_t e = max_dyn_smem_per_device(smem_attr, k_fp8_stats<kCodec>, smem);
    if (e != cudaSuccess) return e;
    const uint64_t words = n / 16;
    uint64_t grid = cdiv(words, (uint64_t)kThreads * 4);
    const uint64_t cap = persistent_grid(k_fp8_stats<kCodec>, kThreads, smem);
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    return launch_dependent(k_fp8_stats<kCodec>, (unsigned)grid, kThreads, (size_t)smem, s, x, n,
                            reinterpret_cast<F8Bins*>(w.bins), out, p->K, p->hist_window);
}

cudaError_t launch_fp8_stats(const ez_plan_s* p, const uint8_t* x, uint64_t n, ez_fp8_stats_t* out,
                             const WsView& w, cudaStream_t s)
{
    if (p->codec == EZ_CODEC_FP8_E5M2) return fp8_stats_launch<EZ_CODEC_FP8_E5M2>(p, x, n, out, w, s);
    return fp8_stats_launch<EZ_CODEC_FP8_E4M3>(p, x, n, out, w, s);
}

cudaError_t launch_fp8_encode(const ez_plan_s* p, const uint8_t* x, uint32_t first, uint32_t count,
                              const ez_fp8_stats_t* st, uint8_t* out, uint64_t* sizes, uint32_t* dstatus,
                              const WsView& w, cudaStream_t s)
{
    F8Enc a;
    a.x = x;
    a.out = out;
    a.slot = p->slot_bytes;
    a.sizes = sizes;
    a.st = st;
    a.dstatus = dstatus;
    a.n = p->n;
    a.L = p->L;
    a.W = p->W;
    a.first = first;
    a.count = count;
    a.tpc = p->tpc;
    a.state = w.state_a;
    a.counter = w.counters + 0;
    a.abort = w.counters + 7;
    const uint64_t tiles = (uint64_t)count * cdiv(p->tpc, kF8Spans);
    if (tiles > 0x7fffffffull) return cudaErrorInvalidValue;
    if (p->codec == EZ_CODEC_FP8_E5M2)
        return launch_dependent(k_fp8_encode<EZ_CODEC_FP8_E5M2>, (unsigned)tiles, kThreads, 0, s, a);
    return launch_dependent(k_fp8_encode<EZ_CODEC_FP8_E4M3>, (unsigned)tiles, kThreads, 0, s, a);
}

cudaError_t launch_fp8_decode(const ez_plan_s* p, const uint8_t* in, const uint64_t* offsets, uint32_t first,
                              uint32_t count, uint8_t* out, uint32_t* dstatus, cudaStream_t s)
{
    F8Dec a;
    a.in = in;
    a.offsets = offsets;
    a.out = out;
    a.dstatus = dstatus;
    a.n = p->n;
    a.L = p->L;
    a.W = p->W;
    a.first = first;
    a.count = count;
    a.tpc = p->tpc;
    a.tpcd = make_fastdiv(p->tpc);
    const uint64_t tiles = (uint64_t)count * p->tpc;
    if (tiles > 0x7fffffffull) return cudaErrorInvalidValue;
    if (p->codec == EZ_CODEC_FP8_E5M2)
        k_fp8_decode<EZ_CODEC_FP8_E5M2, 64><<<(unsigned)tiles, kTile / 64, 0, s>>>(a);
    else
        k_fp8_decode<EZ_CODEC_FP8_E4M3, 64><<<(unsigned)tiles, kTile / 64, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ezk
