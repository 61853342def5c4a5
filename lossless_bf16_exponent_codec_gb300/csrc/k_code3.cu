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
//
// The decoder has a second variant that adds the decoded values into an FP32
// accumulator instead of storing BF16 (the local step of a compressed
// reduce-scatter, digest 3.2).
#include "ez_internal.h"
#include "ez_common.cuh"
#include "ez_bytes.cuh"
#include "ez_tma.cuh"

#include <type_traits>

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
    uint32_t W, first, count, tpc;
    unsigned long long* state;
    uint32_t* counter;
    uint32_t* abort;
    uint32_t* shard_ctr;
};

struct C3Dec {
    const uint8_t* in;
    const uint64_t* offsets;
    uint16_t* out;
    float* acc;          // accumulate variant: FP32 sums instead of BF16 output
    int acc_first;       // the first source: acc = 0 + value
    uint32_t* dstatus;
    uint64_t n, L;
    uint32_t W, first, count, tpc;
    unsigned long long* state;
    uint32_t* counter;
    uint32_t* abort;
    FastDiv tpcd;                 // tpc, for the CTA index split
    unsigned long long full_plane, full_sec_pl, full_sec_idx, full_sec_esc;   // sections of an L-value chunk
    unsigned long long full_nidx;   // its index entries, ceil(L / kTile) (tpc is at least 1, this may be 0)
};

// Escape index: one u64 per kTile (8192) values of the chunk, the number of
// escapes among the values before it.
__device__ __forceinline__ uint64_t c3_idx_bytes(uint64_t n_c) { return rup(8 * cdiv(n_c, kTile), 128); }

__device__ __forceinline__ uint64_t c3_bytes(uint64_t n_c, uint64_t n_esc)
{
    return 128 + rup(n_c, 128) + 3 * rup(cdiv(n_c, 8), 128) + c3_idx_bytes(n_c) + rup(n_esc, 128);
}

__device__ __forceinline__ uint64_t v0_of(uint32_t lt) { return (uint64_t)lt * kTile; }

__device__ __forceinline__ uint32_t le_byte(uint64_t v, int k) { return (uint32_t)(v >> (8 * k)) & 0xFFu; }

__device__ __forceinline__ uint32_t c3_header_byte(int b, uint32_t E0, uint64_t n_c, uint64_t n_esc,
                                                   uint64_t bytes, uint32_t c, uint32_t W)
{
    switch (b) {
        case 0: return 'E';
        case 1: return 'Z';
        case 2: return 'C';
        case 3: return '3';
        case 4: return 2;
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

// Per exponent value e, the code's three plane bits spread to bits 0, 8 and 16
// and the escape flag at bit 24: adding lut[E_i] << i over the 8 values of a
// group yields plane bytes 0..2 and the escape mask in one register.
__device__ __forceinline__ uint32_t c3_lut_entry(uint32_t e, uint32_t E0)
{
    const uint32_t d = e - E0;
    const uint32_t code = d < 7u ? d + 1u : 0u;
    return (code & 1u) | ((code & 2u) << 7) | ((code & 4u) << 14) | (code ? 0u : (1u << 24));
}

__device__ __forceinline__ uint32_t lut_at(const uint32_t* lut, uint32_t byte_off)
{
    return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(lut) + byte_off);
}

__device__ __forceinline__ uint32_t group_codes(const uint32_t* lut, const uint4& w)
{
    uint32_t acc = 0;
    acc += lut_at(lut, (w.x >> 5) & 0x3FCu);
    acc += lut_at(lut, (w.x >> 21) & 0x3FCu) << 1;
    acc += lut_at(lut, (w.y >> 5) & 0x3FCu) << 2;
    acc += lut_at(lut, (w.y >> 21) & 0x3FCu) << 3;
    acc += lut_at(lut, (w.z >> 5) & 0x3FCu) << 4;
    acc += lut_at(lut, (w.z >> 21) & 0x3FCu) << 5;
    acc += lut_at(lut, (w.w >> 5) & 0x3FCu) << 6;
    acc += lut_at(lut, (w.w >> 21) & 0x3FCu) << 7;
    return acc;
}

__device__ __forceinline__ uint32_t byte_of(uint32_t lo, uint32_t hi, int i)
{
    return ((i < 4 ? lo : hi) >> (8 * (i & 3))) & 0xFFu;
}

constexpr uint32_t kEndMark = 0xFFFFFFFFu;
constexpr int kStages = 2;                       // input ring depth (16 KB per stage)
constexpr int kEncThreads = kCompute + 64;       // + chain warp + producer warp

struct EncSmem {
    __align__(128) uint8_t in[kStages][kTile * 2];
    __align__(16) uint8_t esc[kSlots][kTile + 16];
};

__device__ __forceinline__ uint4 lds128(const uint8_t* p)
{
    return *reinterpret_cast<const uint4*>(p);
}

// Persistent, warp-specialised:
//  * producer warp: takes the next tile of a chunk this CTA serves and starts
//    a bulk copy of its BF16 values into a ring stage;
//  * 8 compute warps: code the tile from shared memory, store sign+mantissa
//    bytes and planes, stage the escapes in an escape slot, publish the
//    tile's escape count;
//  * chain warp: resolves each tile's escape prefix in order (decoupled
//    look-back), writes the escapes, and on a chunk's last tile its header,
//    padding and size.
__global__ void __launch_bounds__(kEncThreads, 3) k_code3_encode(C3Enc a)
{
    extern __shared__ __align__(128) unsigned char dyn[];
    EncSmem& S = *reinterpret_cast<EncSmem*>(dyn);
    __shared__ unsigned long long s_full[kStages];
    __shared__ uint32_t s_ici[kStages], s_ilt[kStages], s_empty[kStages];
    __shared__ uint32_t s_lut[256];
    __shared__ uint32_t s_sci[kSlots], s_slt[kSlots], s_sagg[kSlots];
    __shared__ uint32_t s_efull[kSlots], s_edone[kSlots];
    __shared__ unsigned long long s_warp[kCompute / 32];
    __shared__ uint32_t s_comp[2 * 256];
    const int t = threadIdx.x;
    grid_dep_wait();   // the counters were cleared by the kernel before
    uint32_t E0 = __ldg(&a.st->E0);
    if (E0 > 249u) {
        if (t == 0) atomicOr(a.dstatus, EZ_DSTAT_BAD_STATS);
        E0 = 0;
    }
    if (t < 256) s_lut[t] = c3_lut_entry((uint32_t)t, E0);
    fill_comp_table(s_comp, t);
    if (t < kStages) {
        mbar_init(&s_full[t], 1);
        s_empty[t] = 0;
    }
    if (t < kSlots) {
        s_efull[t] = 0;
        s_edone[t] = 0;
    }
    mbar_fence_init();
    __syncthreads();
    volatile uint32_t* vempty = s_empty;
    volatile uint32_t* vefull = s_efull;
    volatile uint32_t* vedone = s_edone;

    if (t >= kCompute + 32) {
        // ---- producer warp (one lane)
        if (t != kCompute + 32) return;
        uint32_t it = 0;
        for (ShardIter sh(blockIdx.x, gridDim.x, a.count); sh.valid(); sh.advance()) {
            const uint32_t ci = sh.next;
            const uint64_t n_c = shard_values(a.n, a.L, a.first + ci);
            for (;; it++) {
                const uint32_t s = it % kStages, round = it / kStages;
                if (!wait_flag(&vempty[s], round, a.abort)) atomicOr(a.dstatus, EZ_DSTAT_TIMEOUT);
                const uint32_t lt = atomicAdd(&a.shard_ctr[ci], 1u);
                if (lt >= a.tpc) break;
                const uint64_t v0 = (uint64_t)lt * kTile;
                const uint32_t nv = v0 < n_c ? (uint32_t)umin64(kTile, n_c - v0) : 0u;
                const uint32_t bytes = (nv & ~7u) * 2u;
                s_ici[s] = ci;
                s_ilt[s] = lt;
                mbar_arrive_expect_tx(&s_full[s], bytes);
                if (bytes) bulk_g2s(S.in[s], a.x + (uint64_t)ci * a.L + v0, bytes, &s_full[s]);
            }
        }
        const uint32_t s = it % kStages, round = it / kStages;
        if (!wait_flag(&vempty[s], round, a.abort)) atomicOr(a.dstatus, EZ_DSTAT_TIMEOUT);
        s_ici[s] = kEndMark;
        mbar_arrive(&s_full[s]);
        return;
    }

    if (t < kCompute) {
        // ---- compute warps
        uint32_t it = 0;
        for (;; it++) {
            const uint32_t s = it % kStages;
            if (!mbar_wait(&s_full[s], (it / kStages) & 1u, a.abort)) {
                // give up on the pipeline, but let a copy still in flight land
                // before this CTA leaves
                if (t == 0) {
                    atomicOr(a.dstatus, EZ_DSTAT_TIMEOUT);
                    atomicExch(a.abort, 1u);
                }
                uint32_t zero = 0;
                mbar_wait(&s_full[s], (it / kStages) & 1u, &zero);
                break;
            }
            const uint32_t ci = s_ici[s];
            if (ci == kEndMark) break;
            const uint32_t lt = s_ilt[s];
            const uint32_t es = it % kSlots, eround = it / kSlots;
            const uint32_t c = a.first + ci;
            const uint64_t n_c = shard_values(a.n, a.L, c);
            const uint64_t v0 = (uint64_t)lt * kTile;
            const uint32_t nv = v0 < n_c ? (uint32_t)umin64(kTile, n_c - v0) : 0u;
            uint8_t* o = a.out + (uint64_t)ci * a.slot;
            const uint64_t plane = rup(cdiv(n_c, 8), 128);
            uint8_t* sm_sec = o + 128;
            uint8_t* pl_t = sm_sec + rup(n_c, 128) + v0 / 8;
            const uint16_t* xt = a.x + (uint64_t)ci * a.L + v0;

            uint4 w[kGroups];
            uint32_t emasks = 0;
            unsigned long long packed = 0;
            // a full tile (every one but a chunk's short last) takes an
            // instance of the loops without the per-group bounds
            auto code_tile = [&](auto full_tag) {
            constexpr bool kFullTile = decltype(full_tag)::value;
#pragma unroll
            for (int g = 0; g < kGroups; g++) {
                const uint32_t v = 8u * (uint32_t)(g * kCompute + t);
                w[g] = (kFullTile || v + 8 <= nv) ? lds128(S.in[s] + 2 * v) : load_group(xt, v, nv);
            }
#pragma unroll
            for (int g = 0; g < kGroups; g++) {
                const uint32_t j = (uint32_t)(g * kCompute + t);
                const uint32_t v = 8u * j;
                if (!kFullTile && v >= nv) continue;
                uint32_t acc = group_codes(s_lut, w[g]);
                const uint32_t sm_lo = sm4_of(w[g].x, w[g].y), sm_hi = sm4_of(w[g].z, w[g].w);
                if (kFullTile || nv - v >= 8) {
                    *reinterpret_cast<uint2*>(sm_sec + v0 + v) = make_uint2(sm_lo, sm_hi);
                } else {
                    const uint32_t vm = (1u << (nv - v)) - 1u;
                    acc &= vm * 0x01010101u;
                    for (uint32_t i = 0; i < nv - v; i++)
                        sm_sec[v0 + v + i] = (uint8_t)byte_of(sm_lo, sm_hi, (int)i);
                }
                pl_t[j] = (uint8_t)acc;
                pl_t[plane + j] = (uint8_t)(acc >> 8);
                pl_t[2 * plane + j] = (uint8_t)(acc >> 16);
                const uint32_t esc = acc >> 24;
                emasks |= esc << (8 * g);
                packed |= (unsigned long long)__popc(esc) << (16 * g);
            }
            };
            if (nv == (uint32_t)kTile) code_tile(std::true_type{});
            else code_tile(std::false_type{});
            if (t == 0 && !wait_flag(&vedone[es], eround, a.abort)) atomicOr(a.dstatus, EZ_DSTAT_TIMEOUT);
            unsigned long long total;
            const unsigned long long excl = compute_excl_scan(packed, s_warp, &total);
            if (t == 0) {
                __threadfence_block();
                vempty[s] = (it / kStages) + 1;     // every compute thread has read the stage
            }
            const unsigned long long agg = (total & 0xFFFFull) + ((total >> 16) & 0xFFFFull) +
                                           ((total >> 32) & 0xFFFFull) + (total >> 48);
            uint32_t gbase = 0;
#pragma unroll
            for (int g = 0; g < kGroups; g++) {
                const uint32_t m = (emasks >> (8 * g)) & 0xFFu;
                const uint32_t kmax = __reduce_max_sync(kFull, (uint32_t)__popc(m));
                if (kmax) {
                    const uint32_t r = gbase + (uint32_t)((excl >> (16 * g)) & 0xFFFFull);
                    stage_selected(S.esc[es], r, m, exp4_of(w[g].x, w[g].y), exp4_of(w[g].z, w[g].w),
                                   kmax, s_comp);
                }
                gbase += (uint32_t)((total >> (16 * g)) & 0xFFFFull);
            }
            compute_sync();    // staging complete; s_warp free
            if (t == 0) {
                st_relaxed(a.state + ci * a.tpc + lt, (lt == 0 ? kFlagIncl : kFlagAgg) | agg);
                s_sci[es] = ci;
                s_slt[es] = lt;
                s_sagg[es] = (uint32_t)agg;
                __threadfence_block();
                vefull[es] = eround + 1;
            }
        }
        if (t == 0) {
            const uint32_t es = it % kSlots, eround = it / kSlots;
            if (!wait_flag(&vedone[es], eround, a.abort)) atomicOr(a.dstatus, EZ_DSTAT_TIMEOUT);
            s_sci[es] = kEndMark;
            __threadfence_block();
            vefull[es] = eround + 1;
        }
        return;
    }

    // ---- chain warp
    const int lane = t & 31;
    for (uint32_t it = 0;; it++) {
        const uint32_t s = it % kSlots, round = it / kSlots;
        bool ok = true;
        if (lane == 0) ok = wait_flag(&vefull[s], round + 1, a.abort);
        ok = __shfl_sync(kFull, ok, 0);
        __threadfence_block();
        if (!ok) {
            if (lane == 0) atomicOr(a.dstatus, EZ_DSTAT_TIMEOUT);
            break;
        }
        const uint32_t ci = s_sci[s];
        if (ci == kEndMark) break;
        const uint32_t lt = s_slt[s], agg = s_sagg[s];
        const uint32_t c = a.first + ci;
        const uint64_t n_c = shard_values(a.n, a.L, c);
        uint8_t* o = a.out + (uint64_t)ci * a.slot;
        const uint64_t plane = rup(cdiv(n_c, 8), 128);
        uint8_t* sm_sec = o + 128;
        uint8_t* pl_sec = sm_sec + rup(n_c, 128);
        uint8_t* idx_sec = pl_sec + 3 * plane;
        uint8_t* esc_sec = idx_sec + c3_idx_bytes(n_c);
        unsigned long long P = 0;
        if (lt != 0) {
            bool stuck;
            P = lookback(a.state, ci * a.tpc + lt, ci * a.tpc, &stuck, a.abort);
            if (lane == 0) {
                if (stuck) atomicOr(a.dstatus, EZ_DSTAT_TIMEOUT);
                st_relaxed(a.state + ci * a.tpc + lt, kFlagIncl | ((P + agg) & kValMask));
            }
        }
        if (lane == 0 && v0_of(lt) < n_c)
            *reinterpret_cast<unsigned long long*>(idx_sec + 8ull * lt) = P;
        {
            // the tile's escapes to [P, P + agg): every aligned 16-byte word
            // of the run is one store assembled from five words of the slot
            // with funnel shifts (the words read lie below agg + 4, inside
            // the slot); the unaligned head and tail are byte stores
            uint8_t* d = esc_sec + P;
            const uint32_t head = min((uint32_t)((16u - (reinterpret_cast<uintptr_t>(d) & 15u)) & 15u), agg);
            const uint32_t nw = (agg - head) / 16u, tail0 = head + 16u * nw;
            for (uint32_t b = (uint32_t)lane; b < head; b += 32) d[b] = S.esc[s][b];
            for (uint32_t b = tail0 + (uint32_t)lane; b < agg; b += 32) d[b] = S.esc[s][b];
            const uint32_t* e32 = reinterpret_cast<const uint32_t*>(S.esc[s]);
            const uint32_t sh = 8u * (head & 3u);
            for (uint32_t j = (uint32_t)lane; j < nw; j += 32) {
                const uint32_t sb = head + 16u * j, q = sb >> 2;
                const uint32_t w0 = e32[q], w1 = e32[q + 1], w2 = e32[q + 2], w3 = e32[q + 3], w4 = e32[q + 4];
                st_v4(d + sb, make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                                         __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh)));
            }
        }
        if (lt == a.tpc - 1) {
            const uint64_t n_esc = P + agg;
            const uint64_t bytes = c3_bytes(n_c, n_esc);
            const uint64_t pb = cdiv(n_c, 8);
            const uint64_t ib = 8 * cdiv(n_c, kTile);
            for (int q = lane; q < 128; q += 32) {
                o[q] = (uint8_t)c3_header_byte(q, E0, n_c, n_esc, bytes, c, a.W);
                if (n_c + q < rup(n_c, 128)) sm_sec[n_c + q] = 0;
                if (pb + q < plane) {
                    pl_sec[pb + q] = 0;
                    pl_sec[plane + pb + q] = 0;
                    pl_sec[2 * plane + pb + q] = 0;
                }
                if (ib + q < c3_idx_bytes(n_c)) idx_sec[ib + q] = 0;
                if (n_esc + q < rup(n_esc, 128)) esc_sec[n_esc + q] = 0;
            }
            if (lane == 0) a.sizes[ci] = bytes;
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            vedone[s] = round + 1;
        }
    }
}

__device__ __forceinline__ uint4 ld_v4_plain(const void* p)
{
    return *reinterpret_cast<const uint4*>(p);
}

// One CTA per tile of 8192 values, no inter-tile dependence: the tile's
// escape prefix is the chunk's index entry.  Every thread reads the chunk's
// offsets, issues its sign+mantissa, plane and index loads as soon as the
// fixed sections are known to lie inside the payload, and only then waits
// for thread 0's header checks (in the oracle's order).  The index is
// checked against the tile's own escape count (entry 0 must be 0, each entry
// plus the tile's count must equal the next entry, the last one n_esc), so
// the escapes read are always inside the escape section.
// kAcc: the local step of a compressed reduce-scatter fused into the decode;
// each decoded value is converted to FP32 (exact) and added to a.acc with one
// IEEE addition (0 + value for the first source), as ez_accumulate_bf16 does.
template <bool kAcc>
__global__ void __launch_bounds__(kThreads, kAcc ? 4 : 5) k_code3_decode(C3Dec a)
{
    __shared__ uint32_t s_bad, s_E0;
    __shared__ unsigned long long s_nesc;
    __shared__ uint32_t s_warp32[kThreads / 32];
    __shared__ __align__(16) uint32_t s_esc32[(kTile + 32) / 4];
    const int t = threadIdx.x;
    uint32_t ci, lt;
    chunk_tile(blockIdx.x, a.tpcd, ci, lt);
    const uint32_t c = a.first + ci;
    const uint64_t n_c = shard_values(a.n, a.L, c);
    const uint64_t v0 = (uint64_t)lt * kTile;
    const uint32_t nv = v0 < n_c ? (uint32_t)umin64(kTile, n_c - v0) : 0u;
    const uint64_t off = __ldg(a.offsets + ci), end = __ldg(a.offsets + ci + 1);
    const uint64_t avail = end >= off ? end - off : 0ull;
    const uint8_t* p = a.in + off;
    // sections: precomputed for a full chunk (every chunk but a short last one)
    const bool full = n_c == a.L;
    const uint64_t plane = full ? a.full_plane : rup(cdiv(n_c, 8), 128);
    const uint64_t sec_pl = full ? a.full_sec_pl : 128 + rup(n_c, 128);
    const uint64_t sec_idx = full ? a.full_sec_idx : sec_pl + 3 * plane;
    const uint64_t sec_esc = full ? a.full_sec_esc : sec_idx + c3_idx_bytes(n_c);
    const uint64_t n_idx = full ? a.full_nidx : cdiv(n_c, kTile);
    // all fixed sections inside the payload: safe to read before the header
    const bool fixed_ok = (off & 15u) == 0 && end >= off && avail >= sec_esc;
    // thread t owns the 32 consecutive values [32t, 32t + 32) of the tile:
    // 32 sign+mantissa bytes, one 32-bit word of each plane
    const uint32_t tv = 32u * (uint32_t)t;
    const uint32_t cnt_v = tv < nv ? umin64(32u, nv - tv) : 0u;   // values of this thread
    const uint8_t* sm_t = p + 128 + v0 + tv;
    const uint8_t* pl_t = p + sec_pl + v0 / 8 + tv / 8;
    uint4 smw[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    uint32_t p0 = 0, p1 = 0, p2 = 0;
    unsigned long long idx_here = 0, idx_next = 0;
    if (fixed_ok) {
        if (cnt_v == 32) {
            smw[0] = ld_v4_nc(sm_t);
            smw[1] = ld_v4_nc(sm_t + 16);
            p0 = __ldg(reinterpret_cast<const uint32_t*>(pl_t));
            p1 = __ldg(reinterpret_cast<const uint32_t*>(pl_t + plane));
            p2 = __ldg(reinterpret_cast<const uint32_t*>(pl_t + 2 * plane));
        } else if (cnt_v) {
            uint32_t w8[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (uint32_t i = 0; i < cnt_v; i++) w8[i >> 2] |= (uint32_t)sm_t[i] << (8 * (i & 3));
            smw[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
            smw[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
            for (uint32_t i = 0; i < cdiv(cnt_v, 8); i++) {
                p0 |= (uint32_t)pl_t[i] << (8 * i);
                p1 |= (uint32_t)pl_t[plane + i] << (8 * i);
                p2 |= (uint32_t)pl_t[2 * plane + i] << (8 * i);
            }
        }
        if (lt < n_idx) idx_here = __ldg(reinterpret_cast<const unsigned long long*>(p + sec_idx) + lt);
        if (lt + 1 < n_idx) idx_next = __ldg(reinterpret_cast<const unsigned long long*>(p + sec_idx) + lt + 1);
    }
    if (t == 0) {
        // the oracle's order of checks
        uint32_t bad = 0;
        s_E0 = 0;
        s_nesc = 0;
        if (off & 15u) {
            bad = EZ_DSTAT_MISALIGNED;
        } else if (end < off || avail < 128) {
            bad = EZ_DSTAT_BAD_SIZE;
        } else {
            const uint4 h0 = ld_v4_plain(p), h1 = ld_v4_plain(p + 16), h2 = ld_v4_plain(p + 32);
            const uint64_t n_hdr = (uint64_t)h0.z | (uint64_t)h0.w << 32;
            const uint64_t n_esc = (uint64_t)h1.x | (uint64_t)h1.y << 32;
            const uint64_t bytes = (uint64_t)h1.z | (uint64_t)h1.w << 32;
            const uint32_t E0 = (h0.y >> 8) & 0xFFu;
            if (h0.x != 0x33435A45u || (h0.y & 0xFFu) != 2u || E0 > 249 || n_hdr != n_c ||
                h2.x != c || h2.y != a.W)
                bad = EZ_DSTAT_BAD_HEADER;
            else if (n_esc > n_c)
                bad = EZ_DSTAT_BAD_COUNT;
            else if (bytes != c3_bytes(n_c, n_esc) || bytes > avail)
                bad = EZ_DSTAT_BAD_SIZE;
            s_E0 = E0;
            s_nesc = n_esc;
        }
        s_bad = bad;
    }
    // stage the span's escapes as soon as the index gives their range
    // [idx_here, idx_next) (the scan below checks it against the planes):
    // every span but the chunk's last, whose end is the header's count, when
    // the range lies inside the payload
    const bool early = fixed_ok && lt + 1 < n_idx && idx_next >= idx_here && idx_next - idx_here <= nv &&
                       sec_esc + ((idx_next + 3) & ~3ull) <= avail;
    if (early) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p + sec_esc + (idx_here & ~3ull));
        const uint32_t words = (uint32_t)((idx_next - idx_here + (idx_here & 3ull) + 3) >> 2);
        const uint32_t i0 = (uint32_t)t, i1 = (uint32_t)t + kThreads;
        const uint32_t w0 = i0 < words ? __ldg(src + i0) : 0u;
        const uint32_t w1 = i1 < words ? __ldg(src + i1) : 0u;
        if (i0 < words) s_esc32[i0] = w0;
        if (i1 < words) s_esc32[i1] = w1;
        for (uint32_t i = (uint32_t)t + 2 * kThreads; i < words; i += kThreads) s_esc32[i] = __ldg(src + i);
    }
    // escapes of the thread's 32 values: code 0 in all three planes
    const uint32_t vmask = cnt_v >= 32 ? 0xFFFFFFFFu : ((1u << cnt_v) - 1u);
    const uint32_t esc = ~(p0 | p1 | p2) & vmask;
    const uint32_t my = __popc(esc);
    // block exclusive scan of one count per thread
    const int lane = t & 31, wid = t >> 5;
    uint32_t x = my;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp32[wid] = x;
    __syncthreads();   // also publishes s_bad and the early-staged escapes
    uint32_t wpre = 0, agg32 = 0;
#pragma unroll
    for (int i = 0; i < kThreads / 32; i++) {
        const uint32_t v = s_warp32[i];
        wpre += i < wid ? v : 0u;
        agg32 += v;
    }
    const uint32_t excl = wpre + x - my;
    const uint32_t bad = s_bad;
    if (bad) {
        if (lt == 0 && t == 0) atomicOr(a.dstatus, bad);
        return;
    }
    const uint32_t E0 = s_E0;
    const unsigned long long n_esc = s_nesc;
    const unsigned long long agg = agg32;
    // index checks (tiles past the chunk's end carry no entry and no escapes)
    const unsigned long long P = lt < n_idx ? idx_here : n_esc;
    const unsigned long long want = lt + 1 < n_idx ? idx_next : n_esc;
    const bool idx_ok = (lt != 0 || n_idx == 0 || P == 0) && P <= n_esc && agg <= n_esc - P &&
                        (lt >= n_idx || P + agg == want);
    if (!idx_ok) {
        if (t == 0) atomicOr(a.dstatus, EZ_DSTAT_BAD_COUNT);
        return;
    }
    // this tile's escapes as aligned words: byte q of the tile is byte q + (P & 3)
    const uint8_t* esc_w = p + sec_esc + (P & ~3ull);
    const uint32_t sh = (uint32_t)(P & 3ull);
    if (!early) {   // CTA-uniform: every thread read the same index entries
        const uint32_t words = (uint32_t)((agg + sh + 3) >> 2);
        for (uint32_t i = (uint32_t)t; i < words; i += kThreads)
            s_esc32[i] = __ldg(reinterpret_cast<const uint32_t*>(esc_w) + i);
        __syncthreads();
    }
    if (!cnt_v) return;
    uint16_t* ot = kAcc ? nullptr : a.out + (uint64_t)ci * a.L + v0 + tv;
    float* at = kAcc ? a.acc + (uint64_t)ci * a.L + v0 + tv : nullptr;
    // accumulate variant: the thread's 32 sums are requested before the code
    // expansion, so their latency overlaps it
    float4 accv[kAcc ? 8 : 1];
    if (kAcc) {
#pragma unroll
        for (int q = 0; q < 8; q++) accv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!a.acc_first && cnt_v == 32) {
#pragma unroll
            for (int q = 0; q < 8; q++) accv[q] = reinterpret_cast<const float4*>(at)[q];
        }
    }
    const uint32_t smv[8] = {smw[0].x, smw[0].y, smw[0].z, smw[0].w, smw[1].x, smw[1].y, smw[1].z, smw[1].w};
    // the window base decides the code -> exponent step once per thread, not
    // per group: two instances of the loop
    const unsigned long long K = (unsigned long long)(E0 - 1) * 0x0101010101010101ull;
    auto expand = [&](auto zero) {
    constexpr bool kZero = decltype(zero)::value;
#pragma unroll
    for (int g = 0; g < 4; g++) {
        const uint32_t b0 = (p0 >> (8 * g)) & 0xFFu, b1 = (p1 >> (8 * g)) & 0xFFu, b2 = (p2 >> (8 * g)) & 0xFFu;
        unsigned long long e8 = codes8(b0, b1, b2);
        e8 = kZero ? ((e8 | 0x8080808080808080ull) - 0x0101010101010101ull) & 0x7F7F7F7F7F7F7F7Full : e8 + K;
        const uint32_t m = (esc >> (8 * g)) & 0xFFu;
        if (m) {
            const uint32_t r = excl + __popc(esc & ((1u << (8 * g)) - 1u));
            uint32_t c_lo, c_hi;
            load_unaligned8(s_esc32, r + sh, c_lo, c_hi);
            e8 = insert_selected_a(e8, m, c_lo, c_hi);
        }
        uint4 o4;
        merge4(smv[2 * g], (uint32_t)e8, o4.x, o4.y);
        merge4(smv[2 * g + 1], (uint32_t)(e8 >> 32), o4.z, o4.w);
        const uint32_t v = 8u * (uint32_t)g;
        if (kAcc) {
            const uint32_t hw[4] = {o4.x, o4.y, o4.z, o4.w};
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; i++)
                f[i] = __uint_as_float((i & 1) ? (hw[i >> 1] & 0xFFFF0000u) : (hw[i >> 1] << 16));
            if (cnt_v == 32) {
                float4* p4 = reinterpret_cast<float4*>(at + v);
                float4 lo = accv[2 * g], hi = accv[2 * g + 1];
                lo.x = __fadd_rn(lo.x, f[0]); lo.y = __fadd_rn(lo.y, f[1]);
                lo.z = __fadd_rn(lo.z, f[2]); lo.w = __fadd_rn(lo.w, f[3]);
                hi.x = __fadd_rn(hi.x, f[4]); hi.y = __fadd_rn(hi.y, f[5]);
                hi.z = __fadd_rn(hi.z, f[6]); hi.w = __fadd_rn(hi.w, f[7]);
                p4[0] = lo;
                p4[1] = hi;
            } else {
#pragma unroll
                for (uint32_t i = 0; i < 8; i++)
                    if (v + i < cnt_v) at[v + i] = __fadd_rn(a.acc_first ? 0.f : at[v + i], f[i]);
            }
        } else if (v + 8 <= cnt_v) {
            st_v4(ot + v, o4);
        } else if (v < cnt_v) {
            const uint32_t hw[4] = {o4.x, o4.y, o4.z, o4.w};
            for (uint32_t i = 0; i < cnt_v - v; i++) ot[v + i] = (uint16_t)(hw[i >> 1] >> (16 * (i & 1)));
        }
    }
    };
    if (E0 == 0) expand(std::true_type{});
    else expand(std::false_type{});
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
    a.count = count;
    a.tpc = p->tpc;
    a.state = w.state_a;
    a.counter = w.counters + 0;
    a.abort = w.counters + 7;
    a.shard_ctr = w.shard_ctr;
    static PerDeviceAttr smem_attr;
    const cudaError_t attr = max_dyn_smem_per_device(smem_attr, k_code3_encode, (int)sizeof(EncSmem));
    if (attr != cudaSuccess) return attr;
    return launch_dependent(k_code3_encode, persistent_grid(k_code3_encode, kEncThreads, sizeof(EncSmem)),
                            kEncThreads, sizeof(EncSmem), s, a);
}

cudaError_t launch_code3_decode(const ez_plan_s* p, const uint8_t* in, const uint64_t* offsets,
                                uint32_t first, uint32_t count, uint16_t* out,
                                uint32_t* dstatus, const WsView& w, cudaStream_t s,
                                float* acc, int acc_first)
{
    C3Dec a;
    a.in = in;
    a.offsets = offsets;
    a.out = out;
    a.acc = acc;
    a.acc_first = acc_first;
    a.dstatus = dstatus;
    a.n = p->n;
    a.L = p->L;
    a.W = p->W;
    a.first = first;
    a.count = count;
    a.tpc = p->tpc;
    a.state = w.state_a;
    a.counter = w.counters + 1;
    a.abort = w.counters + 7;
    a.tpcd = make_fastdiv(p->tpc);
    a.full_plane = rup(cdiv(p->L, 8), 128);
    a.full_sec_pl = 128 + rup(p->L, 128);
    a.full_sec_idx = a.full_sec_pl + 3 * a.full_plane;
    a.full_sec_esc = a.full_sec_idx + rup(8 * cdiv(p->L, kTile), 128);
    a.full_nidx = cdiv(p->L, kTile);
    const uint64_t tiles = (uint64_t)count * p->tpc;
    if (acc) k_code3_decode<true><<<(unsigned)tiles, kThreads, 0, s>>>(a);
    else k_code3_decode<false><<<(unsigned)tiles, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ezk
