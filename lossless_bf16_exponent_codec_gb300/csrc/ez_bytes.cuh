// ez_bytes.cuh -- branch-light byte compaction and expansion for escapes.
//
// A group of 8 values has an 8-bit escape mask m.  The encoder must append
// the escaping exponent bytes, in value order, to the tile's escape list; the
// decoder must put the next popc(m) bytes of that list back at the set bits
// of m.  Both are byte permutations that depend only on m, so they are done
// with PRMT (__byte_perm) instead of a per-escape loop: the encoder takes its
// selectors from a compile-time table indexed by m (copied to shared memory
// by each CTA), the decoder computes them with integer multiplies.
#pragma once

#include <cstdint>

namespace ez {

struct ByteTables {
    uint32_t comp_lo[256];   // PRMT selector: selected bytes 0..3 of (lo, hi)
    uint32_t comp_hi[256];   // selected bytes 4..7
    unsigned long long bmask[256];    // 0xFF in byte i where bit i of m is set
};

constexpr ByteTables make_byte_tables()
{
    ByteTables t{};
    for (int m = 0; m < 256; m++) {
        uint32_t clo = 0, chi = 0;
        unsigned long long bm = 0;
        int rank = 0;
        for (int i = 0; i < 8; i++) {
            if ((m >> i) & 1) {
                if (rank < 4) clo |= (uint32_t)i << (4 * rank);
                else chi |= (uint32_t)i << (4 * (rank - 4));
                bm |= 0xFFull << (8 * i);
                rank++;
            }
        }
        t.comp_lo[m] = clo;
        t.comp_hi[m] = chi;
        t.bmask[m] = bm;
    }
    return t;
}

__device__ const ByteTables kByteTables = make_byte_tables();

// The compaction selectors in shared memory (comp[m] = comp_lo[m],
// comp[256 + m] = comp_hi[m]), filled by the CTA's first 256 threads before a
// barrier: a shared load on the staging path instead of a global one.
__device__ __forceinline__ void fill_comp_table(uint32_t* comp, int t)
{
    if (t < 256) {
        comp[t] = kByteTables.comp_lo[t];
        comp[256 + t] = kByteTables.comp_hi[t];
    }
}

// Append the bytes of (lo, hi) selected by m to s[r ...].  kmax is the
// largest popc(m) over the warp (warp-uniform), so the store loop does not
// diverge.  comp: the selector table of fill_comp_table.
__device__ __forceinline__ void stage_selected(uint8_t* s, uint32_t r, uint32_t m, uint32_t lo,
                                               uint32_t hi, uint32_t kmax, const uint32_t* comp)
{
    const uint32_t c_lo = __byte_perm(lo, hi, comp[m]);
    const uint32_t c_hi = __byte_perm(lo, hi, comp[256 + m]);
    const uint32_t cnt = __popc(m);
#pragma unroll
    for (uint32_t k = 0; k < 8; k++) {
        if (k >= kmax) break;
        if (k < cnt) s[r + k] = (uint8_t)((k < 4 ? c_lo >> (8 * k) : c_hi >> (8 * (k - 4))) & 0xFFu);
    }
}

// The 8 bytes starting at byte offset r of a 4-byte-aligned shared buffer
// (which must extend 12 bytes past the last byte read).
__device__ __forceinline__ void load_unaligned8(const uint32_t* s32, uint32_t r, uint32_t& lo,
                                                uint32_t& hi)
{
    const uint32_t q = r >> 2, o = r & 3u;
    const uint32_t sel = 0x3210u + 0x1111u * o;
    const uint32_t w0 = s32[q], w1 = s32[q + 1], w2 = s32[q + 2];
    lo = __byte_perm(w0, w1, sel);
    hi = __byte_perm(w1, w2, sel);
}

// ---- table-free forms (integer multiplies instead of shared-memory lookups) ----
// Bits 0..3 of n4 (n4 < 16) to bits 0, 8, 16, 24: the four shifted copies
// n4 << 7k (k = 0..3) do not overlap, so the product has no carries and bit
// 8k of it is bit k of n4.
__device__ __forceinline__ uint32_t spread4(uint32_t n4) { return (n4 * 0x00204081u) & 0x01010101u; }

// 3-bit codes of 8 values from one byte of each code plane: byte i of the
// result is bit i of b0 | bit i of b1 << 1 | bit i of b2 << 2.
__device__ __forceinline__ unsigned long long codes8(uint32_t b0, uint32_t b1, uint32_t b2)
{
    const uint32_t lo = spread4(b0 & 15u) | spread4(b1 & 15u) << 1 | spread4(b2 & 15u) << 2;
    const uint32_t hi = spread4(b0 >> 4) | spread4(b1 >> 4) << 1 | spread4(b2 >> 4) << 2;
    return (unsigned long long)hi << 32 | lo;
}

// e8 with the bytes at the set bits of m (m < 256) replaced, in order, by the
// compact bytes (c_lo, c_hi).  Byte i takes compact byte rank(i) = the set
// bits of m below i: the bit spreads of m's nibbles times 0x01010100 are the
// exclusive byte prefix sums, packed to nibbles they are PRMT selectors.
__device__ __forceinline__ unsigned long long insert_selected_a(unsigned long long e8, uint32_t m,
                                                                uint32_t c_lo, uint32_t c_hi)
{
    const uint32_t bl = spread4(m & 15u), bh = spread4(m >> 4);
    const uint32_t pl = bl * 0x01010100u;
    const uint32_t ph = bh * 0x01010100u + (uint32_t)__popc(m & 15u) * 0x01010101u;
    const uint32_t sel_lo = __byte_perm(pl | (pl >> 4), 0u, 0x4420u);
    const uint32_t sel_hi = __byte_perm(ph | (ph >> 4), 0u, 0x4420u);
    const unsigned long long x = (unsigned long long)__byte_perm(c_lo, c_hi, sel_hi) << 32 |
                                 __byte_perm(c_lo, c_hi, sel_lo);
    const unsigned long long bm = (unsigned long long)(bh * 255u) << 32 | (bl * 255u);
    return (e8 & ~bm) | (x & bm);
}

__device__ __forceinline__ unsigned long long byte_mask(uint32_t m)
{
    return __ldg(&kByteTables.bmask[m]);
}

}  // namespace ez
