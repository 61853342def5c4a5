// k_reuse.cu -- a3 / a4 / a5: CIERA cross-iteration exponent reuse
// ("CIERA: Cross-Iteration Exponent Reuse for Lossless Allgather in Sharded
// MoE Training", exponent-reuse and gain-formula paragraphs).
//
// Sender: per block of B values, the block is "changed" when one of its
// exponents differs from the sender's cache of the previous iteration (or the
// call is cold).  The payload carries a changed-block bitmap, the
// sign+mantissa byte of every value and the exponents of the changed blocks
// packed in block order.  Change detection compares the exponents with an
// exponent cache (1 byte per value; same bitmap as the pages' block hash,
// minus collisions) or, with EZ_FLAG_HASH_CACHE, compares two SplitMix64
// hashes per block with the pages' HashCache (16 bytes per block).  Step A
// (k_reuse_split, or k_reuse_hash_split for the raw codec in hash mode) is one
// CTA per 8192-value tile with no inter-tile dependence and publishes the
// tile's changed-block count; k_tile_scan turns the counts into prefixes; the
// place step puts each tile's changed exponents at (prefix + rank) * B and
// writes the index entry, and the tile holding the shard's last value writes
// the header and the size.
//
// Coded variant (EZ_CODEC_REUSE_CODE3): the changed exponents are coded with
// the 3-bit code of ZipCCL (research digest 3.1) instead of nvCOMP's ANS,
// whose window comes from the shard's sigma (k_stats over each shard, a
// launch of its own).  The split codes each tile's changed exponents and
// stages its planes and escapes; the place step moves them into the payload.
//
// Receiver (k_reuse_decode32, k_reuse_decode for B < 32): for W payloads in
// one launch, each 8192-value span reads its slice of the bitmap and its
// prefix from the payload's index, takes unchanged exponents from its
// exponent cache (ExpCache) and changed ones from the payload, writes them
// back into the cache and stores the merged BF16 values straight into the
// gathered full buffer.
#include "ez_internal.h"
#include "ez_common.cuh"
#include "ez_bytes.cuh"

#include <type_traits>

namespace ezk {
using namespace ez;

struct RuEnc {
    const uint16_t* x;
    uint8_t* cache;
    uint8_t* out;
    uint64_t slot;
    uint64_t* sizes;
    uint32_t* dstatus;
    uint64_t n, L;
    uint32_t W, B, log2B, first, count, tpc;
    int cold;
    unsigned long long* state;
    uint32_t* counter;
    uint32_t* abort;
    ShardInfo* info;      // per-shard records (the tail of the EXP length)
    ez_stats_t* stats;    // per shard record (caller's or workspace), coded only
    // coded only: staged planes (3 x 1 KB per tile), staged escapes (the
    // tile's own kTile bytes of a W*L stream), escape-count tile states
    uint8_t* plbuf;
    uint8_t* escbuf;
    unsigned long long* state_b;
    // hash-based change detection: `cache` holds 2 u64 hashes per block,
    // shard first+i at byte i * hstride
    int hash;
    uint64_t hstride;
    FastDiv countd;       // count, for the tile-position split
};


struct RuDec {
    const uint8_t* in;
    const uint64_t* offsets;   // NULL: one payload at `in` with single_avail bytes
    uint64_t single_avail;
    uint8_t* cache;
    uint16_t* out;
    uint32_t* dstatus;
    uint64_t n, L;
    uint32_t W, B, log2B, first, count, tpc;
    unsigned long long* state_a;
    unsigned long long* state_b;
    uint32_t* counter;
    uint32_t* abort;
    FastDiv tpcd;         // tpc, for the CTA index split
};

// Payload sections: header 64 | bitmap | SM | index | EXP.  The index holds
// one entry per kTile (8192) values of the shard: u64 changed blocks before
// it, and for the coded variant a second u64, the escapes among the EXP
// exponents of those blocks.
// Blocks of a shard of n_s values: B is a power of two, so a shift instead of
// a 64-bit division (a software routine on the GPU, paid by every thread).
__device__ __forceinline__ uint64_t ru_blocks(uint64_t n_s, uint32_t B)
{
    return (n_s + B - 1) >> (__ffs((int)B) - 1);
}
__device__ __forceinline__ uint64_t ru_off_sm(uint64_t n_s, uint32_t B)
{
    return 64 + rup(cdiv(ru_blocks(n_s, B), 8), 16);
}
__device__ __forceinline__ uint64_t ru_off_idx(uint64_t n_s, uint32_t B)
{
    return ru_off_sm(n_s, B) + rup(n_s, 16);
}
__device__ __forceinline__ uint32_t ru_idx_stride(bool coded) { return coded ? 16u : 8u; }
__device__ __forceinline__ uint64_t ru_idx_bytes(uint64_t n_s, bool coded)
{
    return rup(ru_idx_stride(coded) * cdiv(n_s, kTile), 16);
}
__device__ __forceinline__ uint64_t ru_off_exp(uint64_t n_s, uint32_t B, bool coded)
{
    return ru_off_idx(n_s, B) + ru_idx_bytes(n_s, coded);
}
__device__ __forceinline__ uint64_t ru_bytes(uint64_t n_s, uint32_t B, uint64_t m, bool coded,
                                             uint64_t n_esc)
{
    return rup(ru_off_exp(n_s, B, coded) + (coded ? 3 * rup(cdiv(m, 8), 16) + n_esc : m), 128);
}

__device__ __forceinline__ uint32_t lb8(uint64_t v, int k) { return (uint32_t)(v >> (8 * k)) & 0xFFu; }

__device__ __forceinline__ uint32_t ru_header_byte(int b, uint32_t flags, uint32_t E0, uint32_t B,
                                                   uint32_t shard, uint64_t n_s, uint64_t n_changed,
                                                   uint64_t m, uint64_t n_esc, uint64_t total)
{
    switch (b) {
        case 0: return 'E';
        case 1: return 'Z';
        case 2: return 'R';
        case 3: return 'U';
        case 4: return 2;
        case 5: return flags;
        case 6: return E0;
        case 7: return 0;
        default: break;
    }
    if (b < 12) return lb8(B, b - 8);
    if (b < 16) return lb8(shard, b - 12);
    if (b < 24) return lb8(n_s, b - 16);
    if (b < 32) return lb8(n_changed, b - 24);
    if (b < 40) return lb8(m, b - 32);
    if (b < 48) return lb8(n_esc, b - 40);
    if (b < 56) return lb8(total, b - 48);
    return 0;
}

__device__ __forceinline__ uint4 ld_group16(const uint16_t* p, uint32_t v, uint32_t nv)
{
    if (v + 8 <= nv) return ld_v4_nc(p + v);
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 8; i++) h[i] = (v + i < nv) ? (uint32_t)p[v + i] : 0u;
    return make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
}
__device__ __forceinline__ unsigned long long ld_group8(const uint8_t* p, uint32_t v, uint32_t nv)
{
    if (v + 8 <= nv) return __ldg(reinterpret_cast<const unsigned long long*>(p + v));
    unsigned long long r = 0;
    for (uint32_t i = 0; v + i < nv && i < 8; i++) r |= (unsigned long long)p[v + i] << (8 * i);
    return r;
}
__device__ __forceinline__ void st_group8(uint8_t* p, uint32_t v, uint32_t nv, unsigned long long x)
{
    if (v + 8 <= nv) {
        *reinterpret_cast<unsigned long long*>(p + v) = x;
    } else {
        for (uint32_t i = 0; v + i < nv && i < 8; i++) p[v + i] = (uint8_t)(x >> (8 * i));
    }
}
// The first cnt (<= 16) bytes at p as a 16-byte word, zero above; stores of
// the first cnt bytes of w.
__device__ __forceinline__ uint4 ld_bytes16(const uint8_t* p, uint32_t cnt)
{
    uint32_t w[4] = {0, 0, 0, 0};
    for (uint32_t i = 0; i < cnt && i < 16; i++) w[i >> 2] |= (uint32_t)p[i] << (8 * (i & 3));
    return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void st_bytes16(uint8_t* p, const uint4& w, uint32_t cnt)
{
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    for (uint32_t i = 0; i < cnt && i < 16; i++) p[i] = (uint8_t)(ws[i >> 2] >> (8 * (i & 3)));
}
__device__ __forceinline__ uint32_t vmask_of(uint32_t v, uint32_t nv)
{
    return v >= nv ? 0u : (nv - v >= 8 ? 0xFFu : ((1u << (nv - v)) - 1u));
}
__device__ __forceinline__ unsigned long long bytemask_of(uint32_t vm)
{
    unsigned long long r = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) r |= ((vm >> i) & 1u) ? (0xFFull << (8 * i)) : 0ull;
    return r;
}

// Tile bitmap (up to 1024 blocks) from the 1024 group-lane changed bits held
// in s_gl (word w = group-lanes 32w..32w+31), built by warp 0 into s_bm; the
// exclusive per-word popcount prefix goes to s_pre.  Returns the changed
// block count of the tile (warp 0 only).
__device__ __forceinline__ uint32_t build_bitmap(const uint32_t* s_gl, uint32_t* s_bm, uint32_t* s_pre,
                                                 uint32_t log2B)
{
    const int lane = threadIdx.x & 31;
    const uint32_t word = s_gl[lane];
    const uint32_t s = 1u << (log2B - 3);   // group-lanes per block
    if (s <= 32) {
        const uint32_t per = 32u / s;
        const uint32_t bmask = (s == 32) ? 0xffffffffu : ((1u << s) - 1u);
        uint32_t bits = 0;
        for (uint32_t b = 0; b < per; b++)
            if ((word >> (b * s)) & bmask) bits |= 1u << b;
        const uint32_t pos = (uint32_t)lane * per;
        atomicOr(&s_bm[pos >> 5], bits << (pos & 31));
    } else {
        const uint32_t k = ((uint32_t)lane * 32u) / s;
        if (word) atomicOr(&s_bm[k >> 5], 1u << (k & 31));
    }
    __syncwarp();
    const uint32_t c = __popc(s_bm[lane]);
    uint32_t x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    s_pre[lane] = x - c;
    return __shfl_sync(kFull, x, 31);
}

__device__ __forceinline__ bool block_changed(const uint32_t* s_bm, uint32_t k)
{
    return (s_bm[k >> 5] >> (k & 31)) & 1u;
}
__device__ __forceinline__ uint32_t block_rank(const uint32_t* s_bm, const uint32_t* s_pre, uint32_t k)
{
    return s_pre[k >> 5] + __popc(s_bm[k >> 5] & ((1u << (k & 31)) - 1u));
}

// 3-bit code plane bits / escape flag per exponent value (see k_code3.cu)
__device__ __forceinline__ uint32_t ru_lut_entry(uint32_t e, uint32_t E0)
{
    const uint32_t d = e - E0;
    const uint32_t code = d < 7u ? d + 1u : 0u;
    return (code & 1u) | ((code & 2u) << 7) | ((code & 4u) << 14) | (code ? 0u : (1u << 24));
}
__device__ __forceinline__ uint32_t lut_b(const uint32_t* lut, uint32_t byte_off)
{
    return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(lut) + byte_off);
}
// plane bytes 0..2 and escape mask (byte 3) of 8 exponent bytes
__device__ __forceinline__ uint32_t codes_of_bytes(const uint32_t* lut, uint32_t lo, uint32_t hi)
{
    uint32_t acc = 0;
    acc += lut_b(lut, (lo << 2) & 0x3FCu);
    acc += lut_b(lut, (lo >> 6) & 0x3FCu) << 1;
    acc += lut_b(lut, (lo >> 14) & 0x3FCu) << 2;
    acc += lut_b(lut, (lo >> 22) & 0x3FCu) << 3;
    acc += lut_b(lut, (hi << 2) & 0x3FCu) << 4;
    acc += lut_b(lut, (hi >> 6) & 0x3FCu) << 5;
    acc += lut_b(lut, (hi >> 14) & 0x3FCu) << 6;
    acc += lut_b(lut, (hi >> 22) & 0x3FCu) << 7;
    return acc;
}

// Exponent bytes of cnt (1..32) consecutive BF16 values at p, 32 bytes as
// two 16-byte words (0 past cnt).
__device__ __forceinline__ void ew_from_x(const uint16_t* p, uint32_t cnt, uint4* ew)
{
    uint32_t xw[16];
    if (cnt == 32) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const uint4 w = ld_v4_nc(p + 8 * q);
            xw[4 * q] = w.x; xw[4 * q + 1] = w.y; xw[4 * q + 2] = w.z; xw[4 * q + 3] = w.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const uint32_t lo = 2u * i < cnt ? (uint32_t)p[2 * i] : 0u;
            const uint32_t hi = 2u * i + 1 < cnt ? (uint32_t)p[2 * i + 1] : 0u;
            xw[i] = lo | hi << 16;
        }
    }
    ew[0] = make_uint4(exp4_of(xw[0], xw[1]), exp4_of(xw[2], xw[3]), exp4_of(xw[4], xw[5]),
                       exp4_of(xw[6], xw[7]));
    ew[1] = make_uint4(exp4_of(xw[8], xw[9]), exp4_of(xw[10], xw[11]), exp4_of(xw[12], xw[13]),
                       exp4_of(xw[14], xw[15]));
}

// ---- hash-based change detection (CIERA: HashCache, two independent 64-bit
// SplitMix64 hashes per block) ---------------------------------------------
// Word i of a block is its 8 exponent bytes (little-endian; 0 past the
// shard); term_i = mix(word + seed + (i + 1) * gamma) is one SplitMix64
// output; the block's hash is mix(sum of its B/8 terms).  The sum makes the
// hash a plain reduction over the block's threads.
constexpr unsigned long long kGamma = 0x9E3779B97F4A7C15ull;
constexpr unsigned long long kHashSeed1 = 0x5851F42D4C957F2Dull;
__device__ __forceinline__ unsigned long long sm64_mix(unsigned long long z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Hash-based decision inside the coded split, for the block holding the
// group at tile value v (every thread of the CTA calls it for the same
// group): each lane's 8-value word is one term of its block; the B/8 terms of
// a block are summed across lanes (B <= 256) or across the 2 or 4 warps of
// the block (B = 512, 1024); the block's first lane compares the hash pair
// with the cache and writes it back when it differs (or cold).  Returns, in
// every lane of the block, whether the block changed.
__device__ __forceinline__ bool hash_group_changed(const RuEnc& a, uint32_t ci, uint64_t v0, uint32_t v,
                                                   uint64_t n_s, unsigned long long word,
                                                   unsigned long long* s_h, uint32_t* s_ch)
{
    const uint32_t B = a.B, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const unsigned long long i = ((v0 + v) & (B - 1u)) >> 3;     // the word's index in its block
    const unsigned long long base = word + (i + 1) * kGamma;
    unsigned long long s0 = sm64_mix(base), s1 = sm64_mix(base + kHashSeed1);
    const uint32_t per = B >> 3;                                   // words (lanes) per block
    for (uint32_t o = (per < 32 ? per : 32) >> 1; o; o >>= 1) {
        s0 += __shfl_xor_sync(kFull, s0, o);
        s1 += __shfl_xor_sync(kFull, s1, o);
    }
    unsigned long long* hc0 = reinterpret_cast<unsigned long long*>(a.cache + (uint64_t)ci * a.hstride);
    if (per <= 32) {
        bool ch = false;
        if ((lane & (per - 1)) == 0 && v0 + v < n_s) {
            unsigned long long* hc = hc0 + 2 * ((v0 + v) >> a.log2B);
            const unsigned long long h0 = sm64_mix(s0), h1 = sm64_mix(s1);
            if (a.cold || hc[0] != h0 || hc[1] != h1) {
                hc[0] = h0;
                hc[1] = h1;
                ch = true;
            }
        }
        return __shfl_sync(kFull, ch, lane & ~(per - 1));
    }
    const uint32_t wpb = per >> 5;                                 // warps per block
    if (lane == 0) {
        s_h[wid] = s0;
        s_h[kThreads / 32 + wid] = s1;
    }
    __syncthreads();
    if (lane == 0 && (wid & (wpb - 1)) == 0) {
        unsigned long long b0 = 0, b1 = 0;
        for (uint32_t k = 0; k < wpb; k++) {
            b0 += s_h[wid + k];
            b1 += s_h[kThreads / 32 + wid + k];
        }
        bool ch = false;
        if (v0 + v < n_s) {
            unsigned long long* hc = hc0 + 2 * ((v0 + v) >> a.log2B);
            const unsigned long long h0 = sm64_mix(b0), h1 = sm64_mix(b1);
            if (a.cold || hc[0] != h0 || hc[1] != h1) {
                hc[0] = h0;
                hc[1] = h1;
                ch = true;
            }
        }
        s_ch[wid] = ch ? 1u : 0u;
    }
    __syncthreads();
    return s_ch[wid & ~(wpb - 1)] != 0;
}

// Raw reuse encode with hash-based change detection, step A in one pass
// (same outputs as k_reuse_split<false> in hash mode): thread t holds the 32
// values [32t, 32t + 32) of the tile, stores their sign+mantissa bytes and
// hashes their four exponent words (B >= 32: the block's B/32 threads add
// their sums with shuffles and the block's first thread decides; B = 8, 16:
// the thread decides its own 32/B blocks), updating the hash cache; the
// block bits go into the tile's bitmap, whose count is published for the
// scan; the shard's final tile records its tail.  The place step then reads
// the changed exponents from x.
__global__ void __launch_bounds__(kThreads, 5) k_reuse_hash_split(RuEnc a)
{
    __shared__ uint32_t s_bm[32];
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    if (t < 32) s_bm[t] = 0;
    const TilePos tp = tile_pos(blockIdx.x, a.countd, a.tpc);
    const uint32_t ci = tp.ci, lt = tp.lt;
    const uint64_t n_s = shard_values(a.n, a.L, a.first + ci);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t nv = v0 < n_s ? (uint32_t)umin64(kTile, n_s - v0) : 0u;
    const uint32_t B = a.B, log2B = a.log2B;
    const uint64_t off_sm = ru_off_sm(n_s, B);
    const uint32_t tv = 32u * (uint32_t)t;
    auto span_body = [&](auto full_tag) {
    constexpr bool kFullSpan = decltype(full_tag)::value;
    const uint32_t cnt_v = kFullSpan ? 32u : tv < nv ? min(32u, nv - tv) : 0u;
    const uint16_t* xt = a.x + (uint64_t)ci * a.L + v0 + tv;
    uint8_t* o = a.out + (uint64_t)ci * a.slot;
    uint32_t xw[16];
    if (cnt_v == 32) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const uint4 w = ld_v4_nc(xt + 8 * q);
            xw[4 * q] = w.x; xw[4 * q + 1] = w.y; xw[4 * q + 2] = w.z; xw[4 * q + 3] = w.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const uint32_t lo = 2u * i < cnt_v ? (uint32_t)xt[2 * i] : 0u;
            const uint32_t hi = 2u * i + 1 < cnt_v ? (uint32_t)xt[2 * i + 1] : 0u;
            xw[i] = lo | hi << 16;
        }
    }
    if (cnt_v) {
        uint32_t sm[8];
#pragma unroll
        for (int j = 0; j < 8; j++) sm[j] = sm4_of(xw[2 * j], xw[2 * j + 1]);
        uint8_t* dst = o + off_sm + v0 + tv;
        if (cnt_v == 32) {
            st_v4(dst, make_uint4(sm[0], sm[1], sm[2], sm[3]));
            st_v4(dst + 16, make_uint4(sm[4], sm[5], sm[6], sm[7]));
        } else {
            st_bytes16(dst, make_uint4(sm[0], sm[1], sm[2], sm[3]), cnt_v);
            st_bytes16(dst + 16, make_uint4(sm[4], sm[5], sm[6], sm[7]), cnt_v > 16 ? cnt_v - 16 : 0u);
        }
    }
    // the block's hash pair (words of 8 exponent bytes, 0 past the shard)
    unsigned long long ew[4];
#pragma unroll
    for (int q = 0; q < 4; q++)
        ew[q] = (unsigned long long)exp4_of(xw[4 * q + 2], xw[4 * q + 3]) << 32 | exp4_of(xw[4 * q], xw[4 * q + 1]);
    unsigned long long* hc0 = reinterpret_cast<unsigned long long*>(a.cache + (uint64_t)ci * a.hstride);
    if (B < 32) {
        // the thread's 32 values are 32/B whole blocks of B/8 words each: it
        // decides them all and ORs their bits into the tile's bitmap
        unsigned long long t0[4], t1[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const unsigned long long base = ew[q] + ((B == 8 ? 0ull : (unsigned long long)(q & 1)) + 1) * kGamma;
            t0[q] = sm64_mix(base);
            t1[q] = sm64_mix(base + kHashSeed1);
        }
        const uint32_t bpt = 32u >> log2B;
        uint32_t bits = 0;
#pragma unroll
        for (uint32_t j = 0; j < 4; j++) {
            if (j >= bpt) break;
            const uint64_t vb = v0 + tv + (uint64_t)j * B;
            if (vb >= n_s) break;
            const unsigned long long s0 = B == 8 ? t0[j] : t0[2 * j] + t0[2 * j + 1];
            const unsigned long long s1 = B == 8 ? t1[j] : t1[2 * j] + t1[2 * j + 1];
            unsigned long long* hc = hc0 + 2 * (vb >> log2B);
            const unsigned long long h0 = sm64_mix(s0), h1 = sm64_mix(s1);
            if (a.cold || hc[0] != h0 || hc[1] != h1) {
                hc[0] = h0;
                hc[1] = h1;
                bits |= 1u << j;
            }
        }
        __syncthreads();   // s_bm cleared
        const uint32_t pos = (uint32_t)t * bpt;             // the thread's first block in the tile
        if (bits) atomicOr(&s_bm[pos >> 5], bits << (pos & 31));
    } else {
        unsigned long long s0 = 0, s1 = 0;
        const unsigned long long i0 = (tv & (B - 1u)) >> 3;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const unsigned long long base = ew[q] + (i0 + q + 1) * kGamma;
            s0 += sm64_mix(base);
            s1 += sm64_mix(base + kHashSeed1);
        }
        const uint32_t per = B >> 5;                      // threads per block, 1..32
        for (uint32_t o2 = per >> 1; o2; o2 >>= 1) {
            s0 += __shfl_xor_sync(kFull, s0, o2);
            s1 += __shfl_xor_sync(kFull, s1, o2);
        }
        bool ch = false;
        if ((lane & (per - 1)) == 0 && v0 + tv < n_s) {
            unsigned long long* hc = hc0 + 2 * ((v0 + tv) >> log2B);
            const unsigned long long h0 = sm64_mix(s0), h1 = sm64_mix(s1);
            if (a.cold || hc[0] != h0 || hc[1] != h1) {
                hc[0] = h0;
                hc[1] = h1;
                ch = true;
            }
        }
        const uint32_t bal = __ballot_sync(kFull, ch);
        __syncthreads();   // s_bm cleared
        if (lane == 0 && bal) {
            const uint32_t nbw = 32u / per;               // blocks per warp
            uint32_t bits = 0;
            for (uint32_t j = 0; j < nbw; j++)
                if ((bal >> (j * per)) & 1u) bits |= 1u << j;
            const uint32_t pos = (uint32_t)wid * nbw;
            atomicOr(&s_bm[pos >> 5], bits << (pos & 31));
        }
    }
    __syncthreads();
    // the shard's block count is needed only from here on (short live range)
    const uint64_t nb = ru_blocks(n_s, B);
    const uint64_t bm_bytes = cdiv(nb, 8);
    const uint32_t fin_tile = n_s ? (uint32_t)((n_s - 1) / kTile) : 0u;
    if (t < 32) {
        const uint32_t c = __popc(s_bm[lane]);
        uint32_t x = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, x, d);
            if (lane >= d) x += y;
        }
        const uint32_t agg = __shfl_sync(kFull, x, 31);
        if (t == 0) {
            st_relaxed(a.state + tp.state, (lt == 0 ? kFlagIncl : kFlagAgg) | agg);
            // the shard's tail (its changed-block total is the tile scan's
            // last inclusive prefix)
            if (lt == fin_tile)
                a.info[ci].tail = (n_s && block_changed(s_bm, (uint32_t)((n_s - 1 - v0) >> log2B)))
                                      ? nb * B - n_s : 0ull;
        }
    }
    __syncthreads();
    const uint32_t nbt = (uint32_t)kTile >> log2B;
    const uint64_t bm0 = (uint64_t)lt * (nbt / 8);
    if ((uint32_t)t < nbt / 8 && bm0 + t < bm_bytes)
        o[64 + bm0 + t] = reinterpret_cast<const uint8_t*>(s_bm)[t];
    if (lt == fin_tile) {
        if (t < 16 && rup(bm_bytes, 16) > bm_bytes + t) o[64 + bm_bytes + t] = 0;
        if (t < 16 && rup(n_s, 16) > n_s + t) o[off_sm + n_s + t] = 0;
    }
    };
    if (nv == (uint32_t)kTile) span_body(std::true_type{});
    else span_body(std::false_type{});
}

// Step A of both reuse encoders, one CTA per 8192-value tile with no
// inter-tile dependence: compare the exponents with the sender cache, store
// the sign+mantissa bytes, build the tile's slice of the changed-block bitmap
// (one ballot per 8-value group), write the changed blocks' exponents into
// the cache, and publish the tile's changed-block count as its look-back
// aggregate.  The updated cache then holds every current exponent at its own
// position, so the later steps read the changed exponents from it.  (The
// hashing coded instance is held to 40 registers, 6 CTAs per SM: 2.4% faster
// than at 64.  The coding instance keeps the plain division in tile_pos: with
// the multiply it is compiled to 56 registers, or, held to 40, runs 2% slower.)
template <bool kCoded, bool kHash>
__global__ void __launch_bounds__(kThreads, (kCoded && !kHash) ? 4 : 6) k_reuse_split(RuEnc a)
{
    __shared__ uint32_t s_gl[32], s_bm[32], s_pre[32];
    __shared__ uint32_t s_lut[kCoded ? 256 : 1];
    __shared__ uint32_t s_comp[kCoded ? 2 * 256 : 1];
    __shared__ unsigned long long s_warp[kCoded ? kThreads / 32 : 1];
    __shared__ __align__(16) uint32_t s_esc32[kCoded ? (kTile + 16) / 4 : 4];
    __shared__ unsigned long long s_h[kHash ? 2 * kThreads / 32 : 1];
    __shared__ uint32_t s_ch[kHash ? kThreads / 32 : 1];
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    // s_gl needs no clearing: lane 0 of every warp writes its entry of every
    // group below (a clear here could land after another warp's entry)
    if (t < 32) s_bm[t] = 0;
    grid_dep_launch();
    const TilePos tp = tile_pos(blockIdx.x, a.count, a.tpc);
    const uint32_t ci = tp.ci, lt = tp.lt;
    const uint32_t r = a.first + ci;
    const uint64_t n_s = shard_values(a.n, a.L, r);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t nv = v0 < n_s ? (uint32_t)umin64(kTile, n_s - v0) : 0u;
    const uint32_t B = a.B, log2B = a.log2B;
    const uint64_t nb = ru_blocks(n_s, B);
    const uint64_t bm_bytes = cdiv(nb, 8);
    const uint64_t off_sm = ru_off_sm(n_s, B);
    const uint16_t* xt = a.x + (uint64_t)ci * a.L + v0;
    uint8_t* ct = a.cache + (uint64_t)ci * a.L + v0;
    uint8_t* o = a.out + (uint64_t)ci * a.slot;

    // a full tile (every one but a shard's short last) takes an instance
    // without the per-group bounds
    auto split_tile = [&](auto full_tag) {
    constexpr bool kFullTile = decltype(full_tag)::value;
    uint4 w[kGroups];
    unsigned long long cv[kGroups];
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        w[g] = kFullTile ? ld_v4_nc(xt + v) : ld_group16(xt, v, nv);
        cv[g] = ((kFullTile || v < nv) && !a.cold && !kHash)
                    ? (kFullTile ? __ldg(reinterpret_cast<const unsigned long long*>(ct + v)) : ld_group8(ct, v, nv))
                    : 0ull;
    }
    // coded: the split may start while the shard statistics finish; nothing
    // above depends on them, everything below may
    grid_dep_wait();
    if (kCoded) {
        uint32_t E0 = a.stats[ci].E0;
        if (E0 > 249u) {
            if (t == 0 && lt == 0) atomicOr(a.dstatus, EZ_DSTAT_BAD_STATS);
            E0 = 0;
        }
        s_lut[t] = ru_lut_entry((uint32_t)t, E0);
        fill_comp_table(s_comp, t);
    }
    unsigned long long e8[kGroups];
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        const uint32_t vm = kFullTile ? 0xFFu : vmask_of(v, nv);
        const unsigned long long bmask = vm == 0xFFu ? ~0ull : bytemask_of(vm);
        const unsigned long long e = ((unsigned long long)exp4_of(w[g].z, w[g].w) << 32 |
                                      exp4_of(w[g].x, w[g].y)) & bmask;
        e8[g] = e;
        bool ch;
        if (kHash) {   // the block's hash pair against the hash cache
            const bool hch = hash_group_changed(a, ci, v0, v, n_s, e, s_h, s_ch);
            ch = vm && hch;
        } else {
            ch = vm && (a.cold || ((e ^ cv[g]) & bmask) != 0ull);
        }
        const uint32_t bal = __ballot_sync(kFull, ch);
        if (lane == 0) s_gl[g * (kThreads / 32) + wid] = bal;
        if (vm) {
            const unsigned long long smw = (unsigned long long)sm4_of(w[g].z, w[g].w) << 32 |
                                           sm4_of(w[g].x, w[g].y);
            if (kFullTile) *reinterpret_cast<unsigned long long*>(o + off_sm + v0 + v) = smw;
            else st_group8(o + off_sm + v0, v, nv, smw);
        }
    }
    __syncthreads();
    const uint32_t fin_tile = n_s ? (uint32_t)((n_s - 1) / kTile) : 0u;
    if (t < 32) {
        const uint32_t agg = build_bitmap(s_gl, s_bm, s_pre, log2B);
        if (t == 0) {
            st_relaxed(a.state + tp.state, (lt == 0 ? kFlagIncl : kFlagAgg) | agg);
            // the shard's tail (its changed-block total is the tile scan's
            // last inclusive prefix)
            if (lt == fin_tile)
                a.info[ci].tail = (n_s && block_changed(s_bm, (uint32_t)((n_s - 1 - v0) >> log2B)))
                                      ? nb * B - n_s : 0ull;
        }
    }
    __syncthreads();
    const uint32_t nbt = (uint32_t)kTile >> log2B;
    const uint64_t bm0 = (uint64_t)lt * (nbt / 8);
    if ((uint32_t)t < nbt / 8 && bm0 + t < bm_bytes)
        o[64 + bm0 + t] = reinterpret_cast<const uint8_t*>(s_bm)[t];
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        if (!kHash && (kFullTile || v < nv) && block_changed(s_bm, v >> log2B)) {
            if (kFullTile) *reinterpret_cast<unsigned long long*>(ct + v) = e8[g];
            else st_group8(ct, v, nv, e8[g]);
        }
    }
    if (lt == fin_tile) {
        if (t < 16 && rup(bm_bytes, 16) > bm_bytes + t) o[64 + bm_bytes + t] = 0;
        if (t < 16 && rup(n_s, 16) > n_s + t) o[off_sm + n_s + t] = 0;
    }
    if (!kCoded) return;
    // coded: the changed exponents' 3-bit code at tile-local stream positions
    // (rank of the block among the tile's changed blocks * B + offset), the
    // planes and the escapes staged for the place step
    uint8_t* pst = a.plbuf + (uint64_t)tp.state * 3 * (kTile / 8);
    uint32_t emasks = 0;
    unsigned long long packed = 0;
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        if (!kFullTile && v >= nv) continue;
        const uint32_t k = v >> log2B;
        if (!block_changed(s_bm, k)) continue;
        const uint32_t local = block_rank(s_bm, s_pre, k) * B + (v - (k << log2B));
        const uint32_t acc = codes_of_bytes(s_lut, (uint32_t)e8[g], (uint32_t)(e8[g] >> 32)) &
                             (kFullTile ? 0xFFFFFFFFu : vmask_of(v, nv) * 0x01010101u);
        const uint32_t pb = local >> 3;
        pst[pb] = (uint8_t)acc;
        pst[kTile / 8 + pb] = (uint8_t)(acc >> 8);
        pst[2 * (kTile / 8) + pb] = (uint8_t)(acc >> 16);
        const uint32_t esc = acc >> 24;
        emasks |= esc << (8 * g);
        packed |= (unsigned long long)__popc(esc) << (16 * g);
    }
    unsigned long long total;
    const unsigned long long excl = block_excl_scan(packed, s_warp, &total);
    const uint32_t agg2 = (uint32_t)((total & 0xFFFFull) + ((total >> 16) & 0xFFFFull) +
                                     ((total >> 32) & 0xFFFFull) + (total >> 48));
    if (t == 0) st_relaxed(a.state_b + tp.state, (unsigned long long)agg2);
    uint8_t* s_esc = reinterpret_cast<uint8_t*>(s_esc32);
    uint32_t gbase = 0;
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t mm = (emasks >> (8 * g)) & 0xFFu;
        const uint32_t kmax = __reduce_max_sync(kFull, (uint32_t)__popc(mm));
        if (kmax) {
            const uint32_t q = gbase + (uint32_t)((excl >> (16 * g)) & 0xFFFFull);
            stage_selected(s_esc, q, mm, (uint32_t)e8[g], (uint32_t)(e8[g] >> 32), kmax, s_comp);
        }
        gbase += (uint32_t)((total >> (16 * g)) & 0xFFFFull);
    }
    __syncthreads();
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.escbuf + (uint64_t)ci * a.L + v0);
    for (uint32_t i = (uint32_t)t; i < (agg2 + 3) / 4; i += kThreads) dst[i] = s_esc32[i];
    };
    if (nv == (uint32_t)kTile) split_tile(std::true_type{});
    else split_tile(std::false_type{});

}

// Changed blocks of a shard of n_s values and its EXP length, after the tile
// scan: the scan's last inclusive prefix of the shard (sc: its state array)
// and m = n_changed * B - the tail the split recorded.  Both are clamped to
// the shard (n_changed <= its blocks, m <= n_s), so a scan that gave up on a
// bounded wait (and reported it) cannot move a store out of the payload.
__device__ __forceinline__ void ru_totals(const RuEnc& a, uint32_t ci, const unsigned long long* sc,
                                          uint64_t n_s, uint64_t& n_changed, uint64_t& m)
{
    n_changed = umin64(ld_relaxed(sc + a.tpc - 1), ru_blocks(n_s, a.B));
    const uint64_t full = n_changed * a.B, tail = a.info[ci].tail;
    m = umin64(full > tail ? full - tail : 0ull, n_s);
}

// This tile's slice of the bitmap, read back from the payload: s_bm, the
// per-word exclusive popcounts s_pre and the changed-block count (returned
// in every thread).  Bits past nb are ignored.
__device__ __forceinline__ uint32_t load_bitmap(const uint8_t* o, uint32_t lt, uint64_t nb,
                                                uint32_t log2B, uint32_t* s_bm, uint32_t* s_pre,
                                                uint32_t* s_agg)
{
    const int t = threadIdx.x;
    const uint64_t bm_bytes = cdiv(nb, 8);
    const uint32_t nbt = (uint32_t)kTile >> log2B;
    const uint64_t bm0 = (uint64_t)lt * (nbt / 8);
    if ((uint32_t)t < nbt / 8) {
        uint32_t b = 0;
        if (bm0 + t < bm_bytes) {
            b = o[64 + bm0 + t];
            if (bm0 + t == bm_bytes - 1 && (nb & 7)) b &= (1u << (nb & 7)) - 1u;
        }
        if (b) atomicOr(&s_bm[t >> 2], b << (8 * (t & 3)));
    }
    __syncthreads();
    if (t < 32) {
        const uint32_t c = __popc(s_bm[t]);
        uint32_t x = c;
#pragma unroll
        for (int q = 1; q < 32; q <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, x, q);
            if (t >= q) x += y;
        }
        s_pre[t] = x - c;
        if (t == 31) *s_agg = x;
    }
    __syncthreads();
    return *s_agg;
}

// Step B of the raw reuse encoder, after the tile scan turned the split's
// changed-block counts into inclusive prefixes: the tile's changed exponents,
// read from the cache, go to EXP at (prefix + rank) * B + offset.  The index
// entry is the prefix; the tile holding the shard's last value writes the
// header, the padding and the size (totals from the split's shard record).
template <bool kHash>
__global__ void __launch_bounds__(kThreads, 6) k_reuse_place(RuEnc a)
{
    __shared__ uint32_t s_bm[32], s_pre[32], s_agg;
    const int t = threadIdx.x;
    grid_dep_wait();   // prefixes, cache and staging come from the kernels before
    if (t < 32) s_bm[t] = 0;
    const TilePos tp = tile_pos(blockIdx.x, a.countd, a.tpc);
    const uint32_t ci = tp.ci, lt = tp.lt;
    const uint32_t r = a.first + ci;
    const uint64_t n_s = shard_values(a.n, a.L, r);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t nv = v0 < n_s ? (uint32_t)umin64(kTile, n_s - v0) : 0u;
    const uint32_t B = a.B, log2B = a.log2B;
    const uint64_t nb = ru_blocks(n_s, B);
    const uint64_t off_idx = ru_off_idx(n_s, B), off_exp = ru_off_exp(n_s, B, false);
    const uint8_t* ct = a.cache + (uint64_t)ci * a.L + v0;
    uint8_t* o = a.out + (uint64_t)ci * a.slot;
    const unsigned long long* sc = a.state + (uint64_t)ci * a.tpc;
    // every group's exponents, loaded with the bitmap and the prefix: the
    // cache bytes, or (hash-based detection: the cache holds hashes) the
    // exponent fields of x
    unsigned long long ev[kGroups];
    const uint16_t* xt = a.x + (uint64_t)ci * a.L + v0;
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        if (kHash) {
            const uint4 xw = v < nv ? ld_group16(xt, v, nv) : make_uint4(0, 0, 0, 0);
            ev[g] = (unsigned long long)exp4_of(xw.z, xw.w) << 32 | exp4_of(xw.x, xw.y);
        } else {
            ev[g] = v < nv ? ld_group8(ct, v, nv) : 0ull;
        }
    }
    const unsigned long long P = lt ? ld_relaxed(sc + lt - 1) : 0ull;
    __syncthreads();
    load_bitmap(o, lt, nb, log2B, s_bm, s_pre, &s_agg);
    if (t == 0 && v0 < n_s) *reinterpret_cast<unsigned long long*>(o + off_idx + 8ull * lt) = P;
    uint64_t n_changed, m;
    ru_totals(a, ci, sc, n_s, n_changed, m);
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        if (v >= nv) continue;
        const uint32_t k = v >> log2B;
        if (!block_changed(s_bm, k)) continue;
        const uint64_t pos = (P + block_rank(s_bm, s_pre, k)) * B + (v - (k << log2B));
        const uint32_t cnt = min(8u, nv - v);
        if (pos + cnt <= m) st_group8(o + off_exp + pos, 0u, cnt, ev[g]);
    }
    const uint32_t fin_tile = n_s ? (uint32_t)((n_s - 1) / kTile) : 0u;
    if (lt == fin_tile) {
        const uint64_t total = ru_bytes(n_s, B, m, false, 0);
        if (t < 64)
            o[t] = (uint8_t)ru_header_byte(t, a.cold ? 2u : 0u, 0u, B, r, n_s, n_changed, m, 0, total);
        if (t < 128 && off_exp + m + t < total) o[off_exp + m + t] = 0;
        const uint64_t ib = 8 * cdiv(n_s, kTile);
        if (t < 16 && ib + t < ru_idx_bytes(n_s, false)) o[off_idx + ib + t] = 0;
        if (t == 0) a.sizes[ci] = total;
    }
}

// Block size B >= 32: as k_reuse_place, with thread t on the 32 consecutive
// values [32t, 32t + 32) of the tile, which lie in one block: a changed
// block's 32 exponents go to a stream position that is a multiple of 32, as
// two aligned 16-byte stores.
template <bool kHash>
__global__ void __launch_bounds__(kThreads, 6) k_reuse_place32(RuEnc a)
{
    __shared__ uint32_t s_bm[32], s_pre[32], s_agg;
    const int t = threadIdx.x;
    grid_dep_wait();   // prefixes, cache and staging come from the kernels before
    if (t < 32) s_bm[t] = 0;
    const TilePos tp = tile_pos(blockIdx.x, a.countd, a.tpc);
    const uint32_t ci = tp.ci, lt = tp.lt;
    const uint32_t r = a.first + ci;
    const uint64_t n_s = shard_values(a.n, a.L, r);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t nv = v0 < n_s ? (uint32_t)umin64(kTile, n_s - v0) : 0u;
    const uint32_t B = a.B, log2B = a.log2B;
    const uint64_t nb = ru_blocks(n_s, B);
    const uint64_t off_idx = ru_off_idx(n_s, B), off_exp = ru_off_exp(n_s, B, false);
    const uint32_t tv = 32u * (uint32_t)t;
    auto span_body = [&](auto full_tag) {
    constexpr bool kFullSpan = decltype(full_tag)::value;
    const uint32_t cnt_v = kFullSpan ? 32u : tv < nv ? min(32u, nv - tv) : 0u;
    const uint8_t* ct = a.cache + (uint64_t)ci * a.L + v0 + tv;
    uint8_t* o = a.out + (uint64_t)ci * a.slot;
    const unsigned long long* sc = a.state + (uint64_t)ci * a.tpc;
    // the thread's exponents, loaded with the bitmap and the prefix: from the
    // cache, or (hash-based detection: the cache holds hashes) from x
    uint4 ew[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (kHash) {
        if (cnt_v) ew_from_x(a.x + (uint64_t)ci * a.L + v0 + tv, cnt_v, ew);
    } else if (cnt_v == 32) {
        ew[0] = ld_v4_nc(ct);
        ew[1] = ld_v4_nc(ct + 16);
    } else if (cnt_v) {
        ew[0] = ld_bytes16(ct, cnt_v);
        ew[1] = ld_bytes16(ct + 16, cnt_v > 16 ? cnt_v - 16 : 0u);
    }
    const unsigned long long P = lt ? ld_relaxed(sc + lt - 1) : 0ull;
    __syncthreads();
    load_bitmap(o, lt, nb, log2B, s_bm, s_pre, &s_agg);
    if (t == 0 && v0 < n_s) *reinterpret_cast<unsigned long long*>(o + off_idx + 8ull * lt) = P;
    uint64_t n_changed, m;
    ru_totals(a, ci, sc, n_s, n_changed, m);
    const uint32_t k = tv >> log2B;
    if (cnt_v && block_changed(s_bm, k)) {
        const uint64_t pos = (P + block_rank(s_bm, s_pre, k)) * B + (tv & (B - 1u));
        uint8_t* dst = o + off_exp + pos;
        if (cnt_v == 32 && pos + 32 <= m) {
            st_v4(dst, ew[0]);
            st_v4(dst + 16, ew[1]);
        } else if (pos + cnt_v <= m) {
            st_bytes16(dst, ew[0], cnt_v);
            st_bytes16(dst + 16, ew[1], cnt_v > 16 ? cnt_v - 16 : 0u);
        }
    }
    const uint32_t fin_tile = n_s ? (uint32_t)((n_s - 1) / kTile) : 0u;
    if (lt == fin_tile) {
        const uint64_t total = ru_bytes(n_s, B, m, false, 0);
        if (t < 64)
            o[t] = (uint8_t)ru_header_byte(t, a.cold ? 2u : 0u, 0u, B, r, n_s, n_changed, m, 0, total);
        if (t < 128 && off_exp + m + t < total) o[off_exp + m + t] = 0;
        const uint64_t ib = 8 * cdiv(n_s, kTile);
        if (t < 16 && ib + t < ru_idx_bytes(n_s, false)) o[off_idx + ib + t] = 0;
        if (t == 0) a.sizes[ci] = total;
    }
    };
    if (nv == (uint32_t)kTile) span_body(std::true_type{});
    else span_body(std::false_type{});
}

// Bytes [b, b+16) of a run of `len` bytes at dst, from d (bytes past len
// are not written).
constexpr uint32_t kSpecBytes = 2048;

__device__ __forceinline__ void store_run16(uint8_t* dst, uint32_t b, uint32_t len, const uint4& d)
{
    if (b >= len) return;
    if (b + 16 <= len && (reinterpret_cast<uintptr_t>(dst + b) & 15u) == 0) {
        *reinterpret_cast<uint4*>(dst + b) = d;   // a whole aligned 16-byte piece
        return;
    }
    const uint32_t ws[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (uint32_t i = 0; i < 16; i++)
        if (b + i < len) dst[b + i] = (uint8_t)(ws[i >> 2] >> (8 * (i & 3)));
}

// Coded variant, place step (after the scans of the changed-block and the
// escape counts): the tile's staged plane bytes go to stream byte
// (prefix * B) / 8 of each plane, its staged escapes to their prefix; both
// prefixes are the span's index entries; the tile holding the shard's last
// value writes the header, the padding and the size.
constexpr int kPlaceThreads = 64;
static_assert(3 * (kTile / 8) == 3 * 16 * kPlaceThreads && kSpecBytes == 2 * 16 * kPlaceThreads,
              "k_reuse_place_coded covers 3 KB of planes and the escape window with 64 threads");
__global__ void __launch_bounds__(kPlaceThreads) k_reuse_place_coded(RuEnc a)
{
    __shared__ __align__(16) uint32_t s_e[kSpecBytes / 4 + 4];
    const int t = threadIdx.x;
    grid_dep_wait();   // prefixes, cache and staging come from the kernels before
    const TilePos tp = tile_pos(blockIdx.x, a.countd, a.tpc);
    const uint32_t ci = tp.ci, lt = tp.lt;
    const uint32_t r = a.first + ci;
    const uint64_t n_s = shard_values(a.n, a.L, r);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t B = a.B;
    const uint64_t spans = cdiv(n_s, kTile);
    const uint64_t off_idx = ru_off_idx(n_s, B), off_exp = ru_off_exp(n_s, B, true);
    uint8_t* o = a.out + (uint64_t)ci * a.slot;
    const unsigned long long* sa = a.state + (uint64_t)ci * a.tpc;
    const unsigned long long* sb = a.state_b + (uint64_t)ci * a.tpc;
    uint64_t n_changed, m;
    ru_totals(a, ci, sa, n_s, n_changed, m);
    const uint64_t plane = rup(cdiv(m, 8), 16);
    uint8_t* pl = o + off_exp;
    uint8_t* esc_sec = pl + 3 * plane;
    // staged planes (3 KB) and a 2 KB window of staged escapes, loaded with
    // the prefixes
    const uint8_t* pst = a.plbuf + (uint64_t)tp.state * 3 * (kTile / 8);
    const uint8_t* est = a.escbuf + (uint64_t)ci * a.L + v0;
    // 64 threads: 48 plane bytes and 32 speculative escape bytes each
    uint4 dp[3], de[2];
#pragma unroll
    for (int j = 0; j < 3; j++) dp[j] = ld_v4_nc(pst + 16u * (uint32_t)(t + j * kPlaceThreads));
#pragma unroll
    for (int j = 0; j < 2; j++) de[j] = ld_v4_nc(est + 16u * (uint32_t)(t + j * kPlaceThreads));
    const unsigned long long P = lt ? ld_relaxed(sa + lt - 1) : 0ull;
    const unsigned long long Pend = ld_relaxed(sa + lt);
    const unsigned long long Q = lt ? ld_relaxed(sb + lt - 1) : 0ull;
    const unsigned long long Qend = ld_relaxed(sb + lt);
    // this span's stream slice [P*B, end): whole blocks, the last span up to m
    uint64_t start = P * B, end = lt + 1 < spans ? Pend * B : m;
    if (lt >= spans || end < start || end > m || end - start > kTile) end = start = 0;
    const uint32_t nbytes = (uint32_t)cdiv(end - start, 8);
    const uint32_t agg2 = Qend >= Q && Qend - Q <= kTile ? (uint32_t)(Qend - Q) : 0u;
    if (t == 0 && v0 < n_s) {
        unsigned long long* idx = reinterpret_cast<unsigned long long*>(o + off_idx);
        idx[2 * lt] = P;
        idx[2 * lt + 1] = Q;
    }
#pragma unroll
    for (int j = 0; j < 3; j++) {
        const uint32_t b0 = 16u * (uint32_t)(t + j * kPlaceThreads);
        const uint32_t pi = b0 / (kTile / 8), off = b0 % (kTile / 8);
        store_run16(pl + (uint64_t)pi * plane + start / 8, off, nbytes, dp[j]);
    }
    // escapes: run [Q, Q + agg2) of the escape section from staged bytes
    // [0, agg2).  The 2 KB window goes through shared memory, so that every
    // aligned 16-byte word of the run is one store built from five words of
    // the window; only the unaligned head and tail are byte stores.  (Staged
    // bytes past the tile's own run are read but never stored; the staging
    // buffer is followed by the plane staging buffer, so the reads stay in
    // the workspace.)
#pragma unroll
    for (int j = 0; j < 2; j++)
        *reinterpret_cast<uint4*>(&s_e[4u * (uint32_t)(t + j * kPlaceThreads)]) = de[j];
    if (t < 4) s_e[kSpecBytes / 4 + t] = 0u;
    __syncthreads();
    {
        uint8_t* d = esc_sec + Q;
        const uint32_t head = min((uint32_t)((16u - (reinterpret_cast<uintptr_t>(d) & 15u)) & 15u), agg2);
        const uint32_t nw = (agg2 - head) / 16u;
        const uint32_t tail0 = head + 16u * nw;
        const uint8_t* s_b = reinterpret_cast<const uint8_t*>(s_e);
        for (uint32_t b = (uint32_t)t; b < head; b += kPlaceThreads) d[b] = b < kSpecBytes ? s_b[b] : est[b];
        for (uint32_t b = tail0 + (uint32_t)t; b < agg2; b += kPlaceThreads)
            d[b] = b < kSpecBytes ? s_b[b] : est[b];
        const uint32_t sh = 8u * (head & 3u);
        for (uint32_t j = (uint32_t)t; j < nw; j += kPlaceThreads) {
            const uint32_t sb = head + 16u * j, q = sb >> 2;
            uint32_t w[5];
            if (sb + 16u <= kSpecBytes) {   // every byte of this word is in the window
#pragma unroll
                for (int k = 0; k < 5; k++) w[k] = s_e[q + k];
            } else {
                const uint32_t* g = reinterpret_cast<const uint32_t*>(est);
#pragma unroll
                for (int k = 0; k < 5; k++) w[k] = __ldg(g + q + k);
            }
            uint4 v;
            v.x = __funnelshift_r(w[0], w[1], sh);
            v.y = __funnelshift_r(w[1], w[2], sh);
            v.z = __funnelshift_r(w[2], w[3], sh);
            v.w = __funnelshift_r(w[3], w[4], sh);
            *reinterpret_cast<uint4*>(d + sb) = v;
        }
    }
    const uint32_t fin_tile = n_s ? (uint32_t)((n_s - 1) / kTile) : 0u;
    if (lt == fin_tile) {
        uint32_t E0 = a.stats[ci].E0;
        if (E0 > 249u) E0 = 0;
        const uint64_t n_esc = ld_relaxed(sb + a.tpc - 1);
        const uint64_t tot = ru_bytes(n_s, B, m, true, n_esc);
        if (t < 64)
            o[t] = (uint8_t)ru_header_byte(t, 1u | (a.cold ? 2u : 0u), E0, B, r, n_s, n_changed, m,
                                           n_esc, tot);
        const uint64_t pbytes = cdiv(m, 8);
        if (t < 16 && pbytes + t < plane) {
            pl[pbytes + t] = 0;
            pl[plane + pbytes + t] = 0;
            pl[2 * plane + pbytes + t] = 0;
        }
        for (uint32_t u = (uint32_t)t; u < 128; u += kPlaceThreads)
            if (off_exp + 3 * plane + n_esc + u < tot) o[off_exp + 3 * plane + n_esc + u] = 0;
        const uint64_t ib = 16 * cdiv(n_s, kTile);
        if (t < 16 && ib + t < ru_idx_bytes(n_s, true)) o[off_idx + ib + t] = 0;
        if (t == 0) a.sizes[ci] = tot;
    }
}

__device__ __forceinline__ uint4 ld16_plain(const void* p) { return *reinterpret_cast<const uint4*>(p); }

// The oracle's checks of a reuse payload's header, in its order; 0 or the
// first failing status.  Reads the 64 header bytes only when they lie inside
// the payload.  *E0 and hdr[0..2] = n_changed, m, n_esc are set when it
// returns 0.
__device__ __forceinline__ uint32_t ru_check_header(const uint8_t* p, uint64_t off, uint64_t avail,
                                                 bool order_bad, uint32_t B, uint32_t r, uint64_t n_s,
                                                 uint64_t nb, bool kCoded, uint32_t* E0_out,
                                                 unsigned long long* hdr)
{
    uint32_t bad = 0;
    *E0_out = 0;
    if (order_bad) bad = EZ_DSTAT_BAD_SIZE;
    if (!bad && (off & 15u)) bad = EZ_DSTAT_MISALIGNED;
    if (!bad && avail < 64) bad = EZ_DSTAT_BAD_SIZE;
    if (!bad) {
        const uint4 h0 = ld16_plain(p), h1 = ld16_plain(p + 16), h2 = ld16_plain(p + 32),
                    h3 = ld16_plain(p + 48);
        const uint32_t flags = (h0.y >> 8) & 0xFFu, E0 = (h0.y >> 16) & 0xFFu;
        const uint64_t n_hdr = (uint64_t)h1.x | (uint64_t)h1.y << 32;
        const uint64_t n_changed = (uint64_t)h1.z | (uint64_t)h1.w << 32;
        const uint64_t m = (uint64_t)h2.x | (uint64_t)h2.y << 32;
        const uint64_t n_esc = (uint64_t)h2.z | (uint64_t)h2.w << 32;
        const uint64_t total = (uint64_t)h3.x | (uint64_t)h3.y << 32;
        const bool coded = flags & 1u;
        if (h0.x != 0x55525A45u || (h0.y & 0xFFu) != 2u || (flags & ~3u) || (h0.y >> 24) != 0 ||
            h0.z != B || h0.w != r || n_hdr != n_s || coded != kCoded)
            bad = EZ_DSTAT_BAD_HEADER;
        else if (coded ? E0 > 249 : (E0 != 0 || n_esc != 0))
            bad = EZ_DSTAT_BAD_HEADER;
        else if (n_changed > nb || m > n_s || n_esc > m)
            bad = EZ_DSTAT_BAD_COUNT;
        else if (total != ru_bytes(n_s, B, m, coded, n_esc) || total > avail)
            bad = EZ_DSTAT_BAD_SIZE;
        *E0_out = E0;
        hdr[0] = n_changed;
        hdr[1] = m;
        hdr[2] = n_esc;
    }
    return bad;
}

// One CTA per kTile span of one payload, no inter-tile dependence.  The
// span's index entry gives the changed blocks (and, coded, the escapes)
// before it; it is checked against the span's own counts -- entry 0 must be
// 0, entry + count must equal the next entry, the last one n_changed (n_esc)
// -- so the exponents read always lie inside the EXP section.  Every thread
// reads the payload offsets, then the bitmap slice, sign+mantissa bytes and
// index entries are loaded before thread 0's header checks complete.
template <bool kCoded>
__global__ void __launch_bounds__(kThreads, 5) k_reuse_decode(RuDec a)
{
    __shared__ uint32_t s_bad, s_E0;
    __shared__ unsigned long long s_hdr[4];   // n_changed, m, n_esc
    __shared__ uint32_t s_bm[32], s_pre[32], s_agg;
    __shared__ unsigned long long s_warp[kThreads / 32];
    __shared__ __align__(16) uint32_t s_esc32[kCoded ? (kTile + 32) / 4 : 4];
    const int t = threadIdx.x;
    if (t < 32) s_bm[t] = 0;   // warp 0, which alone ORs the bitmap bytes in below
    uint32_t ci, lt;
    chunk_tile(blockIdx.x, a.tpcd, ci, lt);
    const uint32_t r = a.first + ci;
    const uint64_t n_s = shard_values(a.n, a.L, r);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t nv = v0 < n_s ? (uint32_t)umin64(kTile, n_s - v0) : 0u;
    const uint32_t B = a.B, log2B = a.log2B;
    const uint64_t nb = ru_blocks(n_s, B);
    const uint64_t bm_bytes = cdiv(nb, 8);
    const uint64_t spans = cdiv(n_s, kTile);
    const uint64_t off = a.offsets ? __ldg(a.offsets + ci) : 0ull;
    uint64_t avail = a.single_avail;
    bool order_bad = false;
    if (a.offsets) {
        const uint64_t end = __ldg(a.offsets + ci + 1);
        order_bad = end < off;
        avail = order_bad ? 0ull : end - off;
    }
    const uint8_t* p = a.in + off;
    const uint64_t off_sm = ru_off_sm(n_s, B), off_idx = ru_off_idx(n_s, B);
    const uint64_t off_exp = ru_off_exp(n_s, B, kCoded);
    const uint32_t stride = ru_idx_stride(kCoded);
    const bool fixed_ok = !order_bad && (off & 15u) == 0 && avail >= off_exp;

    // loads that need only the fixed sections
    const uint32_t nbt = (uint32_t)kTile >> log2B;
    const uint64_t bm0 = (uint64_t)lt * (nbt / 8);
    uint32_t bmb = 0;
    unsigned long long smv[kGroups];
    unsigned long long ib_here = 0, ib_next = 0, ie_here = 0, ie_next = 0;
#pragma unroll
    for (int g = 0; g < kGroups; g++) smv[g] = 0;
    if (fixed_ok) {
        if ((uint32_t)t < nbt / 8 && bm0 + t < bm_bytes) {
            bmb = p[64 + bm0 + t];
            if (bm0 + t == bm_bytes - 1 && (nb & 7)) bmb &= (1u << (nb & 7)) - 1u;
        }
        const uint8_t* sm_t = p + off_sm + v0;
#pragma unroll
        for (int g = 0; g < kGroups; g++) {
            const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
            if (v < nv) smv[g] = ld_group8(sm_t, v, nv);
        }
        const unsigned long long* idx = reinterpret_cast<const unsigned long long*>(p + off_idx);
        const uint32_t sw = stride / 8;
        if (lt < spans) {
            ib_here = __ldg(idx + sw * lt);
            if (kCoded) ie_here = __ldg(idx + sw * lt + 1);
        }
        if (lt + 1 < spans) {
            ib_next = __ldg(idx + sw * (lt + 1));
            if (kCoded) ie_next = __ldg(idx + sw * (lt + 1) + 1);
        }
    }
    if (t == 0) {
        uint32_t e0;
        s_bad = ru_check_header(p, off, avail, order_bad, B, r, n_s, nb, kCoded, &e0, s_hdr);
        s_E0 = e0;
    }
    if (bmb) atomicOr(&s_bm[t >> 2], bmb << (8 * (t & 3)));
    __syncthreads();
    if (s_bad) {
        if (lt == 0 && t == 0) atomicOr(a.dstatus, s_bad);
        return;
    }
    if (t < 32) {
        const uint32_t c = __popc(s_bm[t]);
        uint32_t x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, x, o);
            if (t >= o) x += y;
        }
        s_pre[t] = x - c;
        if (t == 31) s_agg = x;
    }
    __syncthreads();
    const unsigned long long agg = s_agg;
    const uint64_t n_changed = s_hdr[0], m = s_hdr[1], n_esc = s_hdr[2];
    const uint32_t E0 = s_E0;
    // index checks on the changed-block prefix
    const unsigned long long P = lt < spans ? ib_here : n_changed;
    bool ok = (lt != 0 || spans == 0 || P == 0) && P <= n_changed && agg <= n_changed - P &&
              (lt >= spans || P + agg == (lt + 1 < spans ? ib_next : n_changed));
    if (ok && lt + 1 == spans) {
        const bool last_changed = block_changed(s_bm, (uint32_t)((n_s - 1 - v0) >> log2B));
        ok = (P + agg) * B - (last_changed ? nb * B - n_s : 0) == m;
    }
    if (!ok) {
        if (t == 0) atomicOr(a.dstatus, EZ_DSTAT_BAD_COUNT);
        return;
    }
    const uint8_t* ex = p + off_exp;
    uint8_t* ct = a.cache + (uint64_t)ci * a.L + v0;
    uint16_t* ot = a.out + (uint64_t)ci * a.L + v0;

    unsigned long long ev[kGroups];
    bool chg[kGroups];
    uint64_t pos[kGroups];
    bool in_range = true;
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        const uint32_t k = v >> log2B;
        chg[g] = v < nv && block_changed(s_bm, k);
        pos[g] = (P + block_rank(s_bm, s_pre, k)) * B + (v - (k << log2B));
        ev[g] = 0;
        if (v < nv && !chg[g]) ev[g] = ld_group8(ct, v, nv);
        if (chg[g] && pos[g] + min(8u, nv - v) > m) {
            // an m smaller than the bitmap says: never read past the section
            in_range = false;
            chg[g] = false;
        }
        if (!kCoded && chg[g]) ev[g] = ld_group8(ex + pos[g], 0u, min(8u, nv - v));
    }
    if (!in_range) atomicOr(a.dstatus, EZ_DSTAT_BAD_COUNT);

    if (kCoded) {
        // planes of this span's changed exponents; escapes from the index
        const uint64_t plane = rup(cdiv(m, 8), 16);
        const uint8_t* esc_sec = ex + 3 * plane;
        uint32_t pbs[kGroups];
#pragma unroll
        for (int g = 0; g < kGroups; g++) {
            pbs[g] = 0;
            if (!chg[g]) continue;
            const uint64_t pb = pos[g] >> 3;
            pbs[g] = (uint32_t)ex[pb] | (uint32_t)ex[plane + pb] << 8 | (uint32_t)ex[2 * plane + pb] << 16;
        }
        // stage the span's escapes while the plane bytes are in flight: the
        // index gives their range [Q, Qn); the scan below checks it against
        // the planes, and a range the header does not allow is not staged.
        // The escape section starts on a 16-byte boundary (EXP section and
        // planes are multiples of 16), so whole words up to rup(n_esc, 4)
        // stay inside the padded payload.
        const unsigned long long Q = lt < spans ? ie_here : n_esc;
        const unsigned long long Qn = lt + 1 < spans ? ie_next : n_esc;
        const uint8_t* esc_w = esc_sec + (Q & ~3ull);
        const uint32_t sh = (uint32_t)(Q & 3ull);
        const uint32_t words = (Q <= Qn && Qn <= n_esc && Qn - Q <= nv) ? (uint32_t)((Qn - Q + sh + 3) >> 2) : 0u;
        {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(esc_w);
            const uint32_t i0 = (uint32_t)t, i1 = (uint32_t)t + kThreads;
            const uint32_t w0 = i0 < words ? __ldg(src + i0) : 0u;
            const uint32_t w1 = i1 < words ? __ldg(src + i1) : 0u;
            if (i0 < words) s_esc32[i0] = w0;
            if (i1 < words) s_esc32[i1] = w1;
            for (uint32_t i = (uint32_t)t + 2 * kThreads; i < words; i += kThreads) s_esc32[i] = __ldg(src + i);
        }
        uint32_t emasks = 0;
        unsigned long long packed = 0;
#pragma unroll
        for (int g = 0; g < kGroups; g++) {
            if (!chg[g]) continue;
            const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
            const uint32_t cnt = min(8u, nv - v);
            const uint32_t vm = cnt >= 8 ? 0xFFu : ((1u << cnt) - 1u);
            const uint32_t esc = ~(pbs[g] | pbs[g] >> 8 | pbs[g] >> 16) & vm;
            emasks |= esc << (8 * g);
            packed |= (unsigned long long)__popc(esc) << (16 * g);
        }
        // the scan's barrier also publishes the staged escapes
        unsigned long long total;
        const unsigned long long excl = block_excl_scan(packed, s_warp, &total);
        const unsigned long long agg2 = (total & 0xFFFFull) + ((total >> 16) & 0xFFFFull) +
                                        ((total >> 32) & 0xFFFFull) + (total >> 48);
        const bool eok = (lt != 0 || spans == 0 || Q == 0) && Q <= n_esc && agg2 <= n_esc - Q &&
                         (lt >= spans || Q + agg2 == Qn);
        if (!eok) {
            if (t == 0) atomicOr(a.dstatus, EZ_DSTAT_BAD_COUNT);
            return;
        }
        uint32_t gbase = 0;
        // the window base decides the code -> exponent step once, not per
        // group: two instances of the loop
        const unsigned long long K = (unsigned long long)(E0 - 1) * 0x0101010101010101ull;
        auto expand = [&](auto zero) {
        constexpr bool kZero = decltype(zero)::value;
#pragma unroll
        for (int g = 0; g < kGroups; g++) {
            const uint32_t q = gbase + (uint32_t)((excl >> (16 * g)) & 0xFFFFull);
            gbase += (uint32_t)((total >> (16 * g)) & 0xFFFFull);
            if (!chg[g]) continue;
            const unsigned long long c8 = codes8(pbs[g] & 0xFFu, (pbs[g] >> 8) & 0xFFu, (pbs[g] >> 16) & 0xFFu);
            unsigned long long e = kZero
                ? ((c8 | 0x8080808080808080ull) - 0x0101010101010101ull) & 0x7F7F7F7F7F7F7F7Full
                : c8 + K;
            const uint32_t mm = (emasks >> (8 * g)) & 0xFFu;
            if (mm) {
                uint32_t c_lo, c_hi;
                load_unaligned8(s_esc32, q + sh, c_lo, c_hi);
                e = insert_selected_a(e, mm, c_lo, c_hi);
            }
            const uint32_t cnt = min(8u, nv - (8u * (uint32_t)(g * kThreads + t)));
            ev[g] = cnt >= 8 ? e : (e & byte_mask((1u << cnt) - 1u));
        }
        };
        if (E0 == 0) expand(std::true_type{});
        else expand(std::false_type{});
    }

#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        if (v >= nv) continue;
        if (chg[g]) st_group8(ct, v, nv, ev[g]);
        uint4 o4;
        merge4((uint32_t)smv[g], (uint32_t)ev[g], o4.x, o4.y);
        merge4((uint32_t)(smv[g] >> 32), (uint32_t)(ev[g] >> 32), o4.z, o4.w);
        if (v + 8 <= nv) {
            st_v4(ot + v, o4);
        } else {
            const uint32_t hw[4] = {o4.x, o4.y, o4.z, o4.w};
            for (uint32_t i = 0; i < nv - v; i++) ot[v + i] = (uint16_t)(hw[i >> 1] >> (16 * (i & 1)));
        }
    }
}

// Block size B >= 32: thread t owns the 32 consecutive values [32t, 32t + 32)
// of the span.  They lie in one block, so one bitmap bit says where all of
// them come from, and a changed block's stream position is a multiple of 32:
// the thread reads its exponents as two aligned 16-byte words (raw) or one
// aligned 32-bit word of each code plane (coded), its sign+mantissa bytes
// and cache bytes as 16-byte words, and writes its 32 outputs as four
// 16-byte stores.  Checks and statuses are those of k_reuse_decode.
template <bool kCoded>
__global__ void __launch_bounds__(kThreads, 6) k_reuse_decode32(RuDec a)
{
    __shared__ uint32_t s_bad, s_E0;
    __shared__ unsigned long long s_hdr[4];   // n_changed, m, n_esc
    __shared__ uint32_t s_bm[32];
    __shared__ uint32_t s_warp32[kThreads / 32];
    __shared__ __align__(16) uint32_t s_esc32[kCoded ? (kTile + 32) / 4 : 4];
    const int t = threadIdx.x;
    if (t < 32) s_bm[t] = 0;   // warp 0, which alone ORs the bitmap bytes in below
    uint32_t ci, lt;
    chunk_tile(blockIdx.x, a.tpcd, ci, lt);
    const uint32_t r = a.first + ci;
    const uint64_t n_s = shard_values(a.n, a.L, r);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t nv = v0 < n_s ? (uint32_t)umin64(kTile, n_s - v0) : 0u;
    const uint32_t B = a.B, log2B = a.log2B;
    const uint64_t nb = ru_blocks(n_s, B);
    const uint64_t bm_bytes = cdiv(nb, 8);
    const uint64_t spans = cdiv(n_s, kTile);
    const uint64_t off = a.offsets ? __ldg(a.offsets + ci) : 0ull;
    uint64_t avail = a.single_avail;
    bool order_bad = false;
    if (a.offsets) {
        const uint64_t end = __ldg(a.offsets + ci + 1);
        order_bad = end < off;
        avail = order_bad ? 0ull : end - off;
    }
    const uint8_t* p = a.in + off;
    const uint64_t off_sm = ru_off_sm(n_s, B), off_idx = ru_off_idx(n_s, B);
    const uint64_t off_exp = ru_off_exp(n_s, B, kCoded);
    const uint32_t stride = ru_idx_stride(kCoded);
    const bool fixed_ok = !order_bad && (off & 15u) == 0 && avail >= off_exp;

    const uint32_t nbt = (uint32_t)kTile >> log2B;
    const uint64_t bm0 = (uint64_t)lt * (nbt / 8);
    const uint32_t tv = 32u * (uint32_t)t;
    auto span_body = [&](auto full_tag) {
    constexpr bool kFullSpan = decltype(full_tag)::value;
    const uint32_t cnt_v = kFullSpan ? 32u : tv < nv ? min(32u, nv - tv) : 0u;
    uint32_t bmb = 0;
    uint4 smw[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    unsigned long long ib_here = 0, ib_next = 0, ie_here = 0, ie_next = 0;
    if (fixed_ok) {
        if ((uint32_t)t < nbt / 8 && bm0 + t < bm_bytes) {
            bmb = p[64 + bm0 + t];
            if (bm0 + t == bm_bytes - 1 && (nb & 7)) bmb &= (1u << (nb & 7)) - 1u;
        }
        const uint8_t* sm_t = p + off_sm + v0 + tv;
        if (cnt_v == 32) {
            smw[0] = ld_v4_nc(sm_t);
            smw[1] = ld_v4_nc(sm_t + 16);
        } else if (cnt_v) {
            smw[0] = ld_bytes16(sm_t, cnt_v);
            smw[1] = ld_bytes16(sm_t + 16, cnt_v > 16 ? cnt_v - 16 : 0u);
        }
        const unsigned long long* idx = reinterpret_cast<const unsigned long long*>(p + off_idx);
        const uint32_t sw = stride / 8;
        if (lt < spans) {
            ib_here = __ldg(idx + sw * lt);
            if (kCoded) ie_here = __ldg(idx + sw * lt + 1);
        }
        if (lt + 1 < spans) {
            ib_next = __ldg(idx + sw * (lt + 1));
            if (kCoded) ie_next = __ldg(idx + sw * (lt + 1) + 1);
        }
    }
    if (t == 0) {
        uint32_t e0;
        s_bad = ru_check_header(p, off, avail, order_bad, B, r, n_s, nb, kCoded, &e0, s_hdr);
        s_E0 = e0;
    }
    if (bmb) atomicOr(&s_bm[t >> 2], bmb << (8 * (t & 3)));
    __syncthreads();
    if (s_bad) {
        if (lt == 0 && t == 0) atomicOr(a.dstatus, s_bad);
        return;
    }
    // the span's bitmap is at most kTile / 32 = 256 bits, 8 words: every
    // thread sums their popcounts itself (the span's changed blocks, and those
    // before its own block) instead of waiting on a warp's scan
    const uint32_t nbw = (uint32_t)((kTile >> log2B) + 31) >> 5;
    const uint32_t kb = (32u * (uint32_t)t) >> log2B;   // this thread's block in the span
    uint32_t agg32 = 0, pre32 = 0;
#pragma unroll
    for (uint32_t w = 0; w < kTile / 32 / 32; w++) {
        if (w < nbw) {
            const uint32_t bw = s_bm[w];
            agg32 += __popc(bw);
            pre32 += w < (kb >> 5) ? __popc(bw) : (w == (kb >> 5) ? __popc(bw & ((1u << (kb & 31)) - 1u)) : 0u);
        }
    }
    const unsigned long long agg = agg32;
    const uint64_t n_changed = s_hdr[0], m = s_hdr[1], n_esc = s_hdr[2];
    const uint32_t E0 = s_E0;
    // index checks on the changed-block prefix
    const unsigned long long P = lt < spans ? ib_here : n_changed;
    bool ok = (lt != 0 || spans == 0 || P == 0) && P <= n_changed && agg <= n_changed - P &&
              (lt >= spans || P + agg == (lt + 1 < spans ? ib_next : n_changed));
    if (ok && lt + 1 == spans) {
        const bool last_changed = block_changed(s_bm, (uint32_t)((n_s - 1 - v0) >> log2B));
        ok = (P + agg) * B - (last_changed ? nb * B - n_s : 0) == m;
    }
    if (!ok) {
        if (t == 0) atomicOr(a.dstatus, EZ_DSTAT_BAD_COUNT);
        return;
    }
    const uint8_t* ex = p + off_exp;
    uint8_t* ct = a.cache + (uint64_t)ci * a.L + v0 + tv;
    uint16_t* ot = a.out + (uint64_t)ci * a.L + v0 + tv;

    // this thread's block: changed (exponents from the stream) or not (cache)
    const uint32_t k = tv >> log2B;
    bool chg = cnt_v && block_changed(s_bm, k);
    const uint64_t pos = (P + pre32) * B + (tv & (B - 1u));
    if (chg && pos + cnt_v > m) {
        // an m smaller than the bitmap says: never read past the section
        atomicOr(a.dstatus, EZ_DSTAT_BAD_COUNT);
        chg = false;
    }
    uint4 ew[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (cnt_v && !chg) {
        if (cnt_v == 32) {
            ew[0] = ld_v4_nc(ct);
            ew[1] = ld_v4_nc(ct + 16);
        } else {
            ew[0] = ld_bytes16(ct, cnt_v);
            ew[1] = ld_bytes16(ct + 16, cnt_v > 16 ? cnt_v - 16 : 0u);
        }
    }
    if (!kCoded && chg) {
        if (cnt_v == 32) {
            ew[0] = ld_v4_nc(ex + pos);
            ew[1] = ld_v4_nc(ex + pos + 16);
        } else {
            ew[0] = ld_bytes16(ex + pos, cnt_v);
            ew[1] = ld_bytes16(ex + pos + 16, cnt_v > 16 ? cnt_v - 16 : 0u);
        }
    }
    if (kCoded) {
        // one word of each plane (pos is a multiple of 32, and the plane
        // sections are padded to 16 bytes, so the word lies inside)
        const uint64_t plane = rup(cdiv(m, 8), 16);
        const uint8_t* esc_sec = ex + 3 * plane;
        uint32_t p0 = 0, p1 = 0, p2 = 0;
        if (chg) {
            const uint32_t* pw = reinterpret_cast<const uint32_t*>(ex + (pos >> 3));
            p0 = __ldg(pw);
            p1 = __ldg(pw + plane / 4);
            p2 = __ldg(pw + plane / 2);
        }
        // stage the span's escapes while the plane words are in flight: the
        // index gives their range [Q, Qn); the scan below checks it against
        // the planes, and a range the header does not allow is not staged.
        // The escape section starts on a 16-byte boundary, so whole words up
        // to rup(n_esc, 4) stay inside the padded payload.
        const unsigned long long Q = lt < spans ? ie_here : n_esc;
        const unsigned long long Qn = lt + 1 < spans ? ie_next : n_esc;
        const uint8_t* esc_w = esc_sec + (Q & ~3ull);
        const uint32_t sh = (uint32_t)(Q & 3ull);
        const uint32_t words = (Q <= Qn && Qn <= n_esc && Qn - Q <= nv) ? (uint32_t)((Qn - Q + sh + 3) >> 2) : 0u;
        {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(esc_w);
            const uint32_t i0 = (uint32_t)t, i1 = (uint32_t)t + kThreads;
            const uint32_t w0 = i0 < words ? __ldg(src + i0) : 0u;
            const uint32_t w1 = i1 < words ? __ldg(src + i1) : 0u;
            if (i0 < words) s_esc32[i0] = w0;
            if (i1 < words) s_esc32[i1] = w1;
            for (uint32_t i = (uint32_t)t + 2 * kThreads; i < words; i += kThreads) s_esc32[i] = __ldg(src + i);
        }
        const uint32_t vmask = cnt_v >= 32 ? 0xFFFFFFFFu : ((1u << cnt_v) - 1u);
        const uint32_t esc = chg ? (~(p0 | p1 | p2) & vmask) : 0u;
        const uint32_t my = __popc(esc);
        // block scan of the escape counts; its barrier also publishes the
        // staged escapes
        const int lane = t & 31, wid = t >> 5;
        uint32_t x = my;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp32[wid] = x;
        __syncthreads();
        uint32_t wpre = 0, agg2 = 0;
#pragma unroll
        for (int i = 0; i < kThreads / 32; i++) {
            const uint32_t v = s_warp32[i];
            wpre += i < wid ? v : 0u;
            agg2 += v;
        }
        const uint32_t excl = wpre + x - my;
        const bool eok = (lt != 0 || spans == 0 || Q == 0) && Q <= n_esc && agg2 <= n_esc - Q &&
                         (lt >= spans || Q + agg2 == Qn);
        if (!eok) {
            if (t == 0) atomicOr(a.dstatus, EZ_DSTAT_BAD_COUNT);
            return;
        }
        if (chg) {
            uint32_t ev32[8];
            // the window base decides the code -> exponent step once, not per
            // group: two instances of the loop
            const unsigned long long K = (unsigned long long)(E0 - 1) * 0x0101010101010101ull;
            auto expand = [&](auto zero) {
            constexpr bool kZero = decltype(zero)::value;
#pragma unroll
            for (int g = 0; g < 4; g++) {
                const unsigned long long c8 = codes8((p0 >> (8 * g)) & 0xFFu, (p1 >> (8 * g)) & 0xFFu,
                                                     (p2 >> (8 * g)) & 0xFFu);
                unsigned long long e = kZero
                    ? ((c8 | 0x8080808080808080ull) - 0x0101010101010101ull) & 0x7F7F7F7F7F7F7F7Full
                    : c8 + K;
                const uint32_t mm = (esc >> (8 * g)) & 0xFFu;
                if (mm) {
                    const uint32_t q = excl + __popc(esc & ((1u << (8 * g)) - 1u));
                    uint32_t c_lo, c_hi;
                    load_unaligned8(s_esc32, q + sh, c_lo, c_hi);
                    e = insert_selected_a(e, mm, c_lo, c_hi);
                }
                ev32[2 * g] = (uint32_t)e;
                ev32[2 * g + 1] = (uint32_t)(e >> 32);
            }
            };
            if (E0 == 0) expand(std::true_type{});
            else expand(std::false_type{});
            ew[0] = make_uint4(ev32[0], ev32[1], ev32[2], ev32[3]);
            ew[1] = make_uint4(ev32[4], ev32[5], ev32[6], ev32[7]);
        }
    }
    if (!cnt_v) return;
    if (chg) {
        if (cnt_v == 32) {
            st_v4(ct, ew[0]);
            st_v4(ct + 16, ew[1]);
        } else {
            st_bytes16(ct, ew[0], cnt_v);
            st_bytes16(ct + 16, ew[1], cnt_v > 16 ? cnt_v - 16 : 0u);
        }
    }
    const uint32_t smv[8] = {smw[0].x, smw[0].y, smw[0].z, smw[0].w, smw[1].x, smw[1].y, smw[1].z, smw[1].w};
    const uint32_t evv[8] = {ew[0].x, ew[0].y, ew[0].z, ew[0].w, ew[1].x, ew[1].y, ew[1].z, ew[1].w};
#pragma unroll
    for (int g = 0; g < 4; g++) {
        uint4 o4;
        merge4(smv[2 * g], evv[2 * g], o4.x, o4.y);
        merge4(smv[2 * g + 1], evv[2 * g + 1], o4.z, o4.w);
        const uint32_t v = 8u * (uint32_t)g;
        if (v + 8 <= cnt_v) {
            st_v4(ot + v, o4);
        } else if (v < cnt_v) {
            const uint32_t hw[4] = {o4.x, o4.y, o4.z, o4.w};
            for (uint32_t i = 0; i < cnt_v - v; i++) ot[v + i] = (uint16_t)(hw[i >> 1] >> (16 * (i & 1)));
        }
    }
    };
    // the raw decoder takes an instance for a full span (every one but a
    // shard's short last); the coded one is faster without it
    if constexpr (!kCoded) {
        if (nv == (uint32_t)kTile) span_body(std::true_type{});
        else span_body(std::false_type{});
    } else {
        span_body(std::false_type{});
    }
}

static uint32_t ilog2(uint32_t v)
{
    uint32_t r = 0;
    while ((1u << r) < v) r++;
    return r;
}

cudaError_t launch_reuse_encode(const ez_plan_s* p, const uint16_t* x, uint32_t first,
                                uint32_t count, uint8_t* cache, int cold, uint8_t* out,
                                uint64_t* sizes, ez_stats_t* st, uint32_t* dstatus,
                                const WsView& w, cudaStream_t s)
{
    const bool coded = p->codec == EZ_CODEC_REUSE_CODE3;
    RuEnc a;
    a.x = x;
    a.cache = cache;
    a.out = out;
    a.slot = p->slot_bytes;
    a.sizes = sizes;
    a.dstatus = dstatus;
    a.n = p->n;
    a.L = p->L;
    a.W = p->W;
    a.B = p->B;
    a.log2B = ilog2(p->B);
    a.first = first;
    a.count = count;
    a.tpc = p->tpc;
    a.countd = make_fastdiv(count);
    a.cold = cold ? 1 : 0;
    a.state = w.state_a;
    a.counter = w.counters + 0;
    a.abort = w.counters + 7;
    a.info = w.info;
    a.stats = st ? st : w.shard_stats;
    a.hash = p->hash_cache ? 1 : 0;
    a.hstride = p->hstride;
    const unsigned tiles = (unsigned)((uint64_t)count * p->tpc);
    cudaError_t e;
    if (coded) {
        // the shards' windows (a pass over the values of their own)
        e = launch_shard_stats(p, x, first, count, a.stats, w, s);
        if (e != cudaSuccess) return e;
    }
    if (!coded) {
        if (a.hash) k_reuse_hash_split<<<tiles, kThreads, 0, s>>>(a);
        else k_reuse_split<false, false><<<tiles, kThreads, 0, s>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        e = launch_tile_scan(p, w.state_a, count, w.seg_a, w.counters + 4, w.counters + 7, dstatus, s);
        if (e != cudaSuccess) return e;
        if (p->B < 32)
            return a.hash ? launch_dependent(k_reuse_place<true>, tiles, kThreads, 0, s, a)
                          : launch_dependent(k_reuse_place<false>, tiles, kThreads, 0, s, a);
        return a.hash ? launch_dependent(k_reuse_place32<true>, tiles, kThreads, 0, s, a)
                      : launch_dependent(k_reuse_place32<false>, tiles, kThreads, 0, s, a);
    }
    a.plbuf = w.plbuf;
    a.escbuf = w.escbuf;
    a.state_b = w.state_b;
    e = a.hash ? launch_dependent(k_reuse_split<true, true>, tiles, kThreads, 0, s, a)
               : launch_dependent(k_reuse_split<true, false>, tiles, kThreads, 0, s, a);
    if (e != cudaSuccess) return e;
    // changed-block and escape prefixes in one launch
    e = launch_tile_scan2(p, w.state_a, w.seg_a, w.counters + 4, w.state_b, w.seg_b, w.counters + 5, count,
                          w.counters + 7, dstatus, s);
    if (e != cudaSuccess) return e;
    return launch_dependent(k_reuse_place_coded, tiles, kPlaceThreads, 0, s, a);
}

cudaError_t launch_reuse_decode(const ez_plan_s* p, const uint8_t* in, const uint64_t* offsets,
                                uint64_t single_avail, uint32_t first, uint32_t count,
                                uint8_t* cache, uint16_t* out, uint32_t* dstatus,
                                const WsView& w, cudaStream_t s)
{
    RuDec a;
    a.in = in;
    a.offsets = offsets;
    a.single_avail = single_avail;
    a.cache = cache;
    a.out = out;
    a.dstatus = dstatus;
    a.n = p->n;
    a.L = p->L;
    a.W = p->W;
    a.B = p->B;
    a.log2B = ilog2(p->B);
    a.first = first;
    a.count = count;
    a.tpc = p->tpc;
    a.tpcd = make_fastdiv(p->tpc);
    a.state_a = w.state_a;
    a.state_b = w.state_b;
    a.counter = w.counters + 3;
    a.abort = w.counters + 7;
    const unsigned tiles = (unsigned)((uint64_t)count * p->tpc);
    const bool coded = p->codec == EZ_CODEC_REUSE_CODE3;
    if (p->B >= 32) {
        if (coded) k_reuse_decode32<true><<<tiles, kThreads, 0, s>>>(a);
        else k_reuse_decode32<false><<<tiles, kThreads, 0, s>>>(a);
    } else {
        if (coded) k_reuse_decode<true><<<tiles, kThreads, 0, s>>>(a);
        else k_reuse_decode<false><<<tiles, kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace ezk
