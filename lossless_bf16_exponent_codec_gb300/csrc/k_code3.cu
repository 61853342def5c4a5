// k_code3.cu -- a2 / a6: ZipCCL 3-bit exponent code (research digest 3.1,
// 3.2), encode into per-peer chunk slots and decode back.
//
// Per value: SM byte = sign|mantissa (stored raw, fixed stride); exponent E
// becomes code E-E0+1 when E0 <= E <= E0+6, else code 0 and E is appended to
// the chunk's escape list in value order.  The code's three bits go to three
// bit-planes (bit j&7 of byte j>>3).  Each thread handles 8 consecutive values
// per group, so it produces exactly one byte of each plane per group and no
// cross-lane bit shuffling is needed.
//
// Escape positions need the count of escapes in all earlier tiles of the
// chunk: a decoupled look-back scan (ez_common.cuh) gives every tile its
// prefix in one pass; only the escape bytes wait for it, the sign+mantissa
// bytes and planes are stored before the look-back.  The last tile of each
// chunk writes the header, the zero padding and the chunk size.
#include "ez_internal.h"
#include "ez_common.cuh"

namespace ezk {
using namespace ez;

struct C3Enc {
    const uint16_t* x;
    uint8_t* out;
    uint64_t slot;
    uint64_t* sizes;
    const ez_stats_t* st;
    uint32_t* dstatus;
    uint64_t n, L;
    uint32_t W, first, tpc;
    unsigned long long* state;
    uint32_t* counter;
    uint32_t* abort;
};

struct C3Dec {
    const uint8_t* in;
    const uint64_t* offsets;
    uint16_t* out;
    uint32_t* dstatus;
    uint64_t n, L;
    uint32_t W, first, tpc;
    unsigned long long* state;
    uint32_t* counter;
    uint32_t* abort;
};

__device__ __forceinline__ uint64_t c3_bytes(uint64_t n_c, uint64_t n_esc)
{
    return 128 + rup(n_c, 128) + 3 * rup(cdiv(n_c, 8), 128) + rup(n_esc, 128);
}

__device__ __forceinline__ uint32_t le_byte(uint64_t v, int k) { return (uint32_t)(v >> (8 * k)) & 0xFFu; }

__device__ __forceinline__ uint32_t c3_header_byte(int b, uint32_t E0, uint64_t n_c, uint64_t n_esc,
                                                   uint64_t bytes, uint32_t c, uint32_t W)
{
    switch (b) {
        case 0: return 'E';
        case 1: return 'Z';
        case 2: return 'C';
        case 3: return '3';
        case 4: return 1;
        case 5: return E0;
        default: break;
    }
    if (b < 8) return 0;
    if (b < 16) return le_byte(n_c, b - 8);
    if (b < 24) return le_byte(n_esc, b - 16);
    if (b < 32) return le_byte(bytes, b - 24);
    if (b < 36) return le_byte(c, b - 32);
    if (b < 40) return le_byte(W, b - 36);
    return 0;
}

// Load the 8 values of a group; lanes past nv read as 0.
__device__ __forceinline__ uint4 load_group(const uint16_t* p, uint32_t v, uint32_t nv)
{
    if (v + 8 <= nv) return ld_v4_nc(p + v);
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 8; i++) h[i] = (v + i < nv) ? (uint32_t)p[v + i] : 0u;
    return make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
}

__global__ void __launch_bounds__(kThreads) k_code3_encode(C3Enc a)
{
    __shared__ uint32_t s_tile;
    __shared__ unsigned long long s_warp[kThreads / 32];
    __shared__ unsigned long long s_prefix;
    const int t = threadIdx.x;
    const uint32_t tile = next_tile(a.counter, &s_tile);
    const uint32_t ci = tile / a.tpc, lt = tile - ci * a.tpc;
    const uint32_t c = a.first + ci;
    const uint64_t n_c = shard_values(a.n, a.L, c);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t nv = v0 < n_c ? (uint32_t)umin64(kTile, n_c - v0) : 0u;
    uint32_t E0 = __ldg(&a.st->E0);
    if (E0 > 249u) {
        if (t == 0) atomicOr(a.dstatus, EZ_DSTAT_BAD_STATS);
        E0 = 0;
    }
    const uint16_t* xt = a.x + (uint64_t)ci * a.L + v0;
    uint8_t* o = a.out + (uint64_t)ci * a.slot;
    const uint64_t plane = rup(cdiv(n_c, 8), 128);
    uint8_t* sm_sec = o + 128;
    uint8_t* pl_sec = sm_sec + rup(n_c, 128);
    uint8_t* esc_sec = pl_sec + 3 * plane;
    uint8_t* pl_t = pl_sec + v0 / 8;

    uint4 w[kGroups];
#pragma unroll
    for (int g = 0; g < kGroups; g++) w[g] = load_group(xt, 8u * (uint32_t)(g * kThreads + t), nv);

    uint32_t emask[kGroups];
    unsigned long long packed = 0;
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t j = (uint32_t)(g * kThreads + t);
        const uint32_t v = 8u * j;
        emask[g] = 0;
        if (v < nv) {
            const uint32_t vmask = (nv - v >= 8) ? 0xFFu : ((1u << (nv - v)) - 1u);
            uint32_t p0 = 0, p1 = 0, p2 = 0, esc = 0, s_lo = 0, s_hi = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint32_t h = half_of(w[g], i);
                const uint32_t d = exp_of(h) - E0;
                const uint32_t code = d < 7u ? d + 1u : 0u;
                p0 |= (code & 1u) << i;
                p1 |= ((code >> 1) & 1u) << i;
                p2 |= (code >> 2) << i;
                esc |= (code == 0u ? 1u : 0u) << i;
                if (i < 4) s_lo |= sm_of(h) << (8 * i);
                else s_hi |= sm_of(h) << (8 * (i - 4));
            }
            p0 &= vmask;
            p1 &= vmask;
            p2 &= vmask;
            esc &= vmask;
            if (vmask == 0xFFu) {
                *reinterpret_cast<uint2*>(sm_sec + v0 + v) = make_uint2(s_lo, s_hi);
            } else {
                for (uint32_t i = 0; i < nv - v; i++)
                    sm_sec[v0 + v + i] = (uint8_t)((i < 4 ? s_lo >> (8 * i) : s_hi >> (8 * (i - 4))) & 0xFFu);
            }
            pl_t[j] = (uint8_t)p0;
            pl_t[plane + j] = (uint8_t)p1;
            pl_t[2 * plane + j] = (uint8_t)p2;
            emask[g] = esc;
            packed |= (unsigned long long)__popc(esc) << (16 * g);
        }
    }

    unsigned long long total;
    const unsigned long long excl = block_excl_scan(packed, s_warp, &total);
    const unsigned long long agg = (total & 0xFFFFull) + ((total >> 16) & 0xFFFFull) +
                                   ((total >> 32) & 0xFFFFull) + (total >> 48);
    const unsigned long long P = tile_prefix(a.state, tile, ci * a.tpc, agg, &s_prefix, a.dstatus, a.abort);

    unsigned long long gbase = 0;
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        uint32_t m = emask[g];
        unsigned long long r = P + gbase + ((excl >> (16 * g)) & 0xFFFFull);
        while (m) {
            const int i = __ffs(m) - 1;
            m &= m - 1;
            esc_sec[r++] = (uint8_t)exp_of(half_of(w[g], i));
        }
        gbase += (total >> (16 * g)) & 0xFFFFull;
    }

    if (lt == a.tpc - 1) {
        const uint64_t n_esc = P + agg;
        const uint64_t bytes = c3_bytes(n_c, n_esc);
        if (t < 128) {
            o[t] = (uint8_t)c3_header_byte(t, E0, n_c, n_esc, bytes, c, a.W);
            if (n_c + t < rup(n_c, 128)) sm_sec[n_c + t] = 0;
            const uint64_t pb = cdiv(n_c, 8);
            if (pb + t < plane) {
                pl_sec[pb + t] = 0;
                pl_sec[plane + pb + t] = 0;
                pl_sec[2 * plane + pb + t] = 0;
            }
            if (n_esc + t < rup(n_esc, 128)) esc_sec[n_esc + t] = 0;
        }
        if (t == 0) a.sizes[ci] = bytes;
    }
}

__device__ __forceinline__ uint64_t rd_u64(const uint8_t* p)
{
    uint64_t v = 0;
#pragma unroll
    for (int k = 7; k >= 0; k--) v = (v << 8) | p[k];
    return v;
}
__device__ __forceinline__ uint32_t rd_u32(const uint8_t* p)
{
    return (uint32_t)p[0] | (uint32_t)p[1] << 8 | (uint32_t)p[2] << 16 | (uint32_t)p[3] << 24;
}

__global__ void __launch_bounds__(kThreads) k_code3_decode(C3Dec a)
{
    __shared__ uint32_t s_tile, s_bad, s_E0;
    __shared__ unsigned long long s_nesc;
    __shared__ unsigned long long s_warp[kThreads / 32];
    __shared__ unsigned long long s_prefix;
    const int t = threadIdx.x;
    const uint32_t tile = next_tile(a.counter, &s_tile);
    const uint32_t ci = tile / a.tpc, lt = tile - ci * a.tpc;
    const uint32_t c = a.first + ci;
    const uint64_t n_c = shard_values(a.n, a.L, c);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t nv = v0 < n_c ? (uint32_t)umin64(kTile, n_c - v0) : 0u;
    const uint64_t off = a.offsets[ci];
    const uint8_t* p = a.in + off;
    if (t == 0) {
        // the oracle's order of checks
        uint32_t bad = 0;
        const uint64_t end = a.offsets[ci + 1];
        if (off & 15u) {
            bad = EZ_DSTAT_MISALIGNED;
        } else if (end < off || end - off < 128) {
            bad = EZ_DSTAT_BAD_SIZE;
        } else {
            const uint64_t avail = end - off;
            const uint64_t n_esc = rd_u64(p + 16), bytes = rd_u64(p + 24);
            if (!(p[0] == 'E' && p[1] == 'Z' && p[2] == 'C' && p[3] == '3') || p[4] != 1 ||
                p[5] > 249 || rd_u64(p + 8) != n_c || rd_u32(p + 32) != c || rd_u32(p + 36) != a.W)
                bad = EZ_DSTAT_BAD_HEADER;
            else if (n_esc > n_c)
                bad = EZ_DSTAT_BAD_COUNT;
            else if (bytes != c3_bytes(n_c, n_esc) || bytes > avail)
                bad = EZ_DSTAT_BAD_SIZE;
            s_E0 = p[5];
            s_nesc = n_esc;
        }
        s_bad = bad;
    }
    __syncthreads();
    if (s_bad) {
        if (lt == a.tpc - 1 && t == 0) atomicOr(a.dstatus, s_bad);
        return;
    }
    const uint32_t E0 = s_E0;
    const uint64_t n_esc = s_nesc;
    const uint64_t plane = rup(cdiv(n_c, 8), 128);
    const uint8_t* sm_sec = p + 128;
    const uint8_t* pl_sec = sm_sec + rup(n_c, 128);
    const uint8_t* esc_sec = pl_sec + 3 * plane;
    const uint8_t* pl_t = pl_sec + v0 / 8;
    uint16_t* ot = a.out + (uint64_t)ci * a.L + v0;

    uint2 smv[kGroups];
    uint32_t codes[kGroups];   // plane bytes p0 | p1 << 8 | p2 << 16
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t j = (uint32_t)(g * kThreads + t);
        const uint32_t v = 8u * j;
        smv[g] = make_uint2(0, 0);
        codes[g] = 0;
        if (v + 8 <= nv) {
            smv[g] = __ldg(reinterpret_cast<const uint2*>(sm_sec + v0 + v));
        } else if (v < nv) {
            uint32_t lo = 0, hi = 0;
            for (uint32_t i = 0; i < nv - v; i++) {
                const uint32_t b = sm_sec[v0 + v + i];
                if (i < 4) lo |= b << (8 * i);
                else hi |= b << (8 * (i - 4));
            }
            smv[g] = make_uint2(lo, hi);
        }
        if (v < nv)
            codes[g] = (uint32_t)__ldg(pl_t + j) | (uint32_t)__ldg(pl_t + plane + j) << 8 |
                       (uint32_t)__ldg(pl_t + 2 * plane + j) << 16;
    }
    uint32_t emask[kGroups];
    unsigned long long packed = 0;
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        const uint32_t vmask = v >= nv ? 0u : (nv - v >= 8 ? 0xFFu : ((1u << (nv - v)) - 1u));
        const uint32_t any = (codes[g] | codes[g] >> 8 | codes[g] >> 16) & 0xFFu;
        emask[g] = ~any & vmask;
        packed |= (unsigned long long)__popc(emask[g]) << (16 * g);
    }
    unsigned long long total;
    const unsigned long long excl = block_excl_scan(packed, s_warp, &total);
    const unsigned long long agg = (total & 0xFFFFull) + ((total >> 16) & 0xFFFFull) +
                                   ((total >> 32) & 0xFFFFull) + (total >> 48);
    const unsigned long long P = tile_prefix(a.state, tile, ci * a.tpc, agg, &s_prefix, a.dstatus, a.abort);
    if (lt == a.tpc - 1 && t == 0 && P + agg != n_esc) atomicOr(a.dstatus, EZ_DSTAT_BAD_COUNT);

    unsigned long long gbase = 0;
    bool overrun = false;
#pragma unroll
    for (int g = 0; g < kGroups; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        unsigned long long r = P + gbase + ((excl >> (16 * g)) & 0xFFFFull);
        gbase += (total >> (16 * g)) & 0xFFFFull;
        if (v >= nv) continue;
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t cb = codes[g] >> i;
            const uint32_t code = (cb & 1u) | ((cb >> 7) & 2u) | ((cb >> 14) & 4u);
            uint32_t E;
            if (code) {
                E = E0 + code - 1;
            } else if ((emask[g] >> i) & 1u) {
                if (r < n_esc) E = esc_sec[r];
                else { E = 0; overrun = true; }
                r++;
            } else {
                E = 0;   // past the end of the chunk
            }
            const uint32_t sm = ((i < 4 ? smv[g].x >> (8 * i) : smv[g].y >> (8 * (i - 4)))) & 0xFFu;
            h[i] = merge_of(sm, E);
        }
        if (v + 8 <= nv) {
            st_v4(ot + v, make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16,
                                     h[6] | h[7] << 16));
        } else {
            for (uint32_t i = 0; i < nv - v; i++) ot[v + i] = (uint16_t)h[i];
        }
    }
    if (overrun) atomicOr(a.dstatus, EZ_DSTAT_BAD_COUNT);
}

cudaError_t launch_code3_encode(const ez_plan_s* p, const uint16_t* x, uint32_t first,
                                uint32_t count, const ez_stats_t* st, uint8_t* out,
                                uint64_t* sizes, uint32_t* dstatus, const WsView& w, cudaStream_t s)
{
    C3Enc a;
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
    a.tpc = p->tpc;
    a.state = w.state_a;
    a.counter = w.counters + 0;
    a.abort = w.counters + 7;
    const uint64_t tiles = (uint64_t)count * p->tpc;
    k_code3_encode<<<(unsigned)tiles, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_code3_decode(const ez_plan_s* p, const uint8_t* in, const uint64_t* offsets,
                                uint32_t first, uint32_t count, uint16_t* out,
                                uint32_t* dstatus, const WsView& w, cudaStream_t s)
{
    C3Dec a;
    a.in = in;
    a.offsets = offsets;
    a.out = out;
    a.dstatus = dstatus;
    a.n = p->n;
    a.L = p->L;
    a.W = p->W;
    a.first = first;
    a.tpc = p->tpc;
    a.state = w.state_a;
    a.counter = w.counters + 1;
    a.abort = w.counters + 7;
    const uint64_t tiles = (uint64_t)count * p->tpc;
    k_code3_decode<<<(unsigned)tiles, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ezk
