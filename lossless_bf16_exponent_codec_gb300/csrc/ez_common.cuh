// ez_common.cuh -- tile geometry and device helpers shared by the kernels of
// libexpzip (sm_103a).
//
// Every kernel works on tiles of kTile = 8192 values.  A CTA of 256 threads
// takes one tile; thread t owns four "groups" of 8 consecutive values, group
// g at tile value 8*(g*256 + t), so each warp load or store of a group is one
// contiguous run (512 B of BF16, 256 B of sign+mantissa bytes, 32 B of a code
// plane).  Tiles never straddle a shard: shard i owns tiles
// [i*tpc, (i+1)*tpc) with tpc = max(1, ceil(L/kTile)).
//
// Order-preserving compaction (escapes, changed blocks) uses a decoupled
// look-back scan over tile aggregates (Merrill & Garland, "Single-pass
// parallel prefix scan with decoupled look-back", 2016).  Tile ids are taken
// from an atomic counter, so a tile only waits on tiles whose CTAs are
// already running.  Every wait is bounded; a wait that gives up sets a flag
// the caller turns into EZ_DSTAT_TIMEOUT.
#pragma once

#include <atomic>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "expzip.h"

namespace ez {

constexpr int kThreads = 256;
constexpr int kGroups = 4;
constexpr int kTile = kThreads * kGroups * 8;      // 8192 values
constexpr uint32_t kFull = 0xffffffffu;
constexpr uint32_t kSpinLimit = 1u << 21;          // ~0.1-0.3 s of polling

constexpr unsigned long long kFlagAgg = 1ull << 62;
constexpr unsigned long long kFlagIncl = 2ull << 62;
constexpr unsigned long long kValMask = (1ull << 62) - 1;

__host__ __device__ __forceinline__ uint64_t cdiv(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ uint64_t rup(uint64_t a, uint64_t b) { return cdiv(a, b) * b; }
__host__ __device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// values of shard r (r counted over the whole plan)
__host__ __device__ __forceinline__ uint64_t shard_values(uint64_t n, uint64_t L, uint32_t r)
{
    uint64_t a = (uint64_t)r * L;
    if (a >= n) return 0;
    return (n - a < L) ? n - a : L;
}

// ---- BF16 fields (CIERA split; ZipCCL 3.1) ---------------------------------
__device__ __forceinline__ uint32_t exp_of(uint32_t h) { return (h >> 7) & 0xFFu; }

// ---- SWAR helpers: two BF16 values per 32-bit word --------------------------
// Sign+mantissa bytes of the 4 values in words a (values 0,1) and b (2,3):
// per 16-bit half, ((h >> 8) & 0x80) | (h & 0x7F), then bytes 0 and 2 of each.
__device__ __forceinline__ uint32_t sm4_of(uint32_t a, uint32_t b)
{
    const uint32_t pa = ((a >> 8) & 0x00800080u) | (a & 0x007F007Fu);
    const uint32_t pb = ((b >> 8) & 0x00800080u) | (b & 0x007F007Fu);
    return __byte_perm(pa, pb, 0x6420);
}
// Exponent bytes of the 4 values in words a, b.
__device__ __forceinline__ uint32_t exp4_of(uint32_t a, uint32_t b)
{
    return __byte_perm(a >> 7, b >> 7, 0x6420);
}
// Two output words (values 0,1 and 2,3) from 4 sign+mantissa bytes and 4
// exponent bytes: per value ((sm & 0x80) << 8) | (E << 7) | (sm & 0x7F).
__device__ __forceinline__ void merge4(uint32_t sm4, uint32_t e4, uint32_t& lo, uint32_t& hi)
{
    // per 16-bit lane: A = sm with its sign replicated over the high byte
    // (bits 0..6 the mantissa, bit 15 the sign), E = exponent in the high
    // byte; E >> 1 puts it at bits 7..14, and one LOP3 takes bits 0..6 and 15
    // from A, the rest from E >> 1
    const uint32_t a0 = __byte_perm(sm4, 0u, 0x9180), a1 = __byte_perm(sm4, 0u, 0xB3A2);
    const uint32_t e0 = __byte_perm(e4, 0u, 0x1404) >> 1, e1 = __byte_perm(e4, 0u, 0x3424) >> 1;
    asm("lop3.b32 %0, %1, %2, %3, 0xE2;" : "=r"(lo) : "r"(a0), "r"(0x807F807Fu), "r"(e0));
    asm("lop3.b32 %0, %1, %2, %3, 0xE2;" : "=r"(hi) : "r"(a1), "r"(0x807F807Fu), "r"(e1));
}

// ---- tile order ----------------------------------------------------------------
// Tile ids are dealt round-robin over the `count` shards of a launch, so the
// shards' look-back chains advance side by side; state index is
// shard-contiguous (shard ci owns [ci*tpc, (ci+1)*tpc)).
// n / d for 32-bit n and d >= 1 by one multiply: rcp = floor((2^64 - 1) / d)
// + 1 (0 stands for d = 1).  With 2^64 = q d + r, n * rcp / 2^64 exceeds n / d
// by less than n / 2^64 < 1 / d, and the fractional part of n / d is at most
// 1 - 1 / d, so the floor is n / d exactly (for a power of two rcp = 2^64 / d).
struct FastDiv {
    uint32_t d, pad;
    unsigned long long rcp;
};
inline FastDiv make_fastdiv(uint32_t d) { return FastDiv{d, 0u, d > 1 ? ~0ull / d + 1 : 0ull}; }
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f)
{
    return f.rcp ? (uint32_t)__umul64hi((unsigned long long)n, f.rcp) : n;
}

struct TilePos {
    uint32_t ci, lt, state;
};
__device__ __forceinline__ TilePos tile_pos(uint32_t id, uint32_t count, uint32_t tpc)
{
    TilePos p;
    p.ci = id % count;
    p.lt = id / count;
    p.state = p.ci * tpc + p.lt;
    return p;
}
__device__ __forceinline__ TilePos tile_pos(uint32_t id, const FastDiv& count, uint32_t tpc)
{
    TilePos p;
    p.lt = fdiv(id, count);
    p.ci = id - p.lt * count.d;
    p.state = p.ci * tpc + p.lt;
    return p;
}
// Chunk ci and tile lt of CTA id over chunks of tpc tiles.
__device__ __forceinline__ void chunk_tile(uint32_t id, const FastDiv& tpc, uint32_t& ci, uint32_t& lt)
{
    ci = fdiv(id, tpc);
    lt = id - ci * tpc.d;
}

// ---- memory helpers ----------------------------------------------------------
__device__ __forceinline__ uint4 ld_v4_nc(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ void st_v4(void* p, const uint4& v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Exclusive prefix of tile t over [seg_first, t).  One full warp calls it.
// Returns the prefix; *stuck is set (uniformly) if a predecessor never
// published within the spin limit.
__device__ __forceinline__ uint32_t ld_relaxed32(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Exclusive prefix of tile t over [seg_first, t).  One full warp calls it.
// Each pass reads a window of 128 predecessors (4 per lane, nearest first) in
// one round trip to L2, so the inclusive-prefix front advances 128 tiles per
// round trip -- faster than tiles complete at HBM speed.  Entries before
// seg_first act as an inclusive prefix of 0.
// `abort` (per launch, zeroed with the tile states) is raised by the first
// wait that gives up; every other wait then stops at once, so a broken chain
// costs one spin limit, not one per tile.  *stuck is set uniformly on a
// give-up.
constexpr int kLookPerLane = 4;

static __device__ __noinline__ unsigned long long lookback(unsigned long long* st, long long t,
                                                           long long seg_first, bool* stuck,
                                                           uint32_t* abort)
{
    const int lane = threadIdx.x & 31;
    unsigned long long prefix = 0;
    long long pos = t - 1;
    *stuck = false;
    while (pos >= seg_first) {
        unsigned long long w[kLookPerLane];
#pragma unroll
        for (int k = 0; k < kLookPerLane; k++) {
            const long long idx = pos - (long long)(kLookPerLane * lane + k);
            w[k] = idx >= seg_first ? ld_relaxed(st + idx) : kFlagIncl;
        }
        bool empty = false;
#pragma unroll
        for (int k = 0; k < kLookPerLane; k++) {
            const long long idx = pos - (long long)(kLookPerLane * lane + k);
            uint32_t spins = 0;
            while ((w[k] >> 62) == 0 && spins < kSpinLimit) {
                __nanosleep(32);
                w[k] = ld_relaxed(st + idx);
                if ((++spins & 63u) == 0 && ld_relaxed32(abort)) break;
            }
            empty |= (w[k] >> 62) == 0;
        }
        __syncwarp();
        if (__any_sync(kFull, empty)) {
            *stuck = true;
            if (lane == 0) atomicExch(abort, 1u);
            return prefix;
        }
        int kf = kLookPerLane;            // nearest inclusive entry of this lane
        unsigned long long all = 0, part = 0;
#pragma unroll
        for (int k = kLookPerLane - 1; k >= 0; k--) {
            const unsigned long long v = w[k] & kValMask;
            all += v;
            if ((w[k] >> 62) == 2) {
                kf = k;
                part = 0;
            }
            part += v;
        }
        // part = sum of entries 0..kf when kf < kLookPerLane
        if (kf == kLookPerLane) part = all;
        const uint32_t incl = __ballot_sync(kFull, kf < kLookPerLane);
        if (incl) {
            const int j = __ffs(incl) - 1;
            const unsigned long long v = lane < j ? all : (lane == j ? part : 0ull);
            return prefix + warp_sum_u64(v);
        }
        prefix += warp_sum_u64(all);
        pos -= 32 * kLookPerLane;
    }
    return prefix;
}

// Block-wide exclusive scan of a 64-bit value over 256 threads.  s_warp holds
// 8 entries; a __syncthreads() is needed before s_warp is reused.
__device__ __forceinline__ unsigned long long block_excl_scan(unsigned long long v,
                                                              unsigned long long* s_warp,
                                                              unsigned long long* total)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned long long y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    unsigned long long pre = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < kThreads / 32; i++) {
        unsigned long long s = s_warp[i];
        if (i < wid) pre += s;
        tot += s;
    }
    *total = tot;
    return pre + x - v;
}

// ---- persistent, warp-specialised launches ----------------------------------
// A CTA has kCompute threads (8 compute warps) plus one chain warp.  Compute
// warps synchronise among themselves with named barrier 1; the chain warp
// never joins it.  Slots of a small shared-memory ring pass tiles between the
// two roles; every wait on a slot flag is bounded.
constexpr int kCompute = kThreads;            // 256 compute threads
constexpr int kPThreads = kCompute + 32;      // + the chain warp
constexpr int kSlots = 4;

__device__ __forceinline__ void compute_sync()
{
    asm volatile("bar.sync 1, %0;" :: "r"(kCompute) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile_s32(const volatile uint32_t* p) { return *p; }

// Wait until *flag >= want (bounded); returns false if the wait gave up.
__device__ __forceinline__ bool wait_flag(const volatile uint32_t* flag, uint32_t want, uint32_t* abort)
{
    uint32_t spins = 0;
    while (ld_volatile_s32(flag) < want) {
        if (++spins > kSpinLimit) return false;
        if ((spins & 63u) == 0 && ld_relaxed32(abort)) return false;
        __nanosleep(20);
    }
    return true;
}

// Shards served by CTA `c` of `G` persistent CTAs: with count <= G each shard
// gets G/count CTAs (shard c % count); otherwise CTA c serves c, c+G, ...
struct ShardIter {
    uint32_t next, step, count;
    __device__ __forceinline__ ShardIter(uint32_t c, uint32_t G, uint32_t count_)
    {
        count = count_;
        if (count <= G) {
            const uint32_t per = G / count;
            next = (c < per * count) ? c % count : count;
            step = count;   // one shard only
        } else {
            next = c;
            step = G;
        }
    }
    __device__ __forceinline__ bool valid() const { return next < count; }
    __device__ __forceinline__ void advance() { next = (step == count) ? count : next + step; }
};

// Exclusive scan over the kCompute compute threads (named barrier 1); s_warp
// holds 8 entries and must not be reused before the next compute_sync().
__device__ __forceinline__ unsigned long long compute_excl_scan(unsigned long long v,
                                                                unsigned long long* s_warp,
                                                                unsigned long long* total)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned long long y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    compute_sync();
    unsigned long long pre = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < kCompute / 32; i++) {
        unsigned long long s = s_warp[i];
        if (i < wid) pre += s;
        tot += s;
    }
    *total = tot;
    return pre + x - v;
}

// Tile id from the per-launch counter, broadcast to the CTA.
__device__ __forceinline__ uint32_t next_tile(uint32_t* counter, uint32_t* s_tile)
{
    if (threadIdx.x == 0) *s_tile = atomicAdd(counter, 1u);
    __syncthreads();
    return *s_tile;
}

// Publish a tile's aggregate, look back, publish its inclusive prefix.  All
// threads call it; returns the exclusive prefix to every thread.
__device__ __forceinline__ unsigned long long tile_prefix(unsigned long long* st, uint32_t tile,
                                                          uint32_t seg_first,
                                                          unsigned long long agg,
                                                          unsigned long long* s_prefix,
                                                          uint32_t* dstatus, uint32_t* abort)
{
    if (tile == seg_first) {
        if (threadIdx.x == 0) {
            st_relaxed(st + tile, kFlagIncl | agg);
            *s_prefix = 0;
        }
    } else {
        if (threadIdx.x == 0) st_relaxed(st + tile, kFlagAgg | agg);
        if (threadIdx.x < 32) {
            bool stuck;
            unsigned long long p = lookback(st, tile, seg_first, &stuck, abort);
            if (threadIdx.x == 0) {
                if (stuck) atomicOr(dstatus, EZ_DSTAT_TIMEOUT);
                st_relaxed(st + tile, kFlagIncl | ((p + agg) & kValMask));
                *s_prefix = p;
            }
        }
    }
    __syncthreads();
    return *s_prefix;
}

// Grid of a persistent kernel: resident CTAs per SM (from the occupancy
// calculator) times the SM count of the current device.
// ---- programmatic dependent launch -------------------------------------------
// The later kernels of a multi-kernel call are launched so that their CTAs may
// start while the kernel before them drains; each such kernel calls
// grid_dep_wait() before it touches anything an earlier kernel of the call
// wrote (the wait returns once those grids have completed and their memory
// operations are visible).  Launched without the attribute, the wait returns
// at once.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Called at the start of a kernel that has a dependent launch after it: once
// every CTA has called it, the dependent kernel may be scheduled (its CTAs
// then fill SMs as this kernel's CTAs finish, and wait as above).
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                                    cudaStream_t s, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// A kernel's dynamic shared-memory limit is an attribute of the kernel in one
// device's context, so it must be raised on every device the kernel runs on.
// One record per kernel: bit d is set once device d has it (ordinals >= 64
// set it on every launch).
struct PerDeviceAttr {
    std::atomic<unsigned long long> done{0};
};

template <typename K>
inline cudaError_t max_dyn_smem_per_device(PerDeviceAttr& rec, K kernel, int bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool tracked = dev >= 0 && dev < 64;
    if (tracked && ((rec.done.load(std::memory_order_acquire) >> dev) & 1ull)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && tracked) rec.done.fetch_or(1ull << dev, std::memory_order_release);
    return e;
}

template <typename K>
inline unsigned persistent_grid(K kernel, int threads, size_t dyn_smem = 0)
{
    int dev = 0, sms = 0, per = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, threads, dyn_smem);
    if (per < 1) per = 1;
    if (sms < 1) sms = 1;
    return (unsigned)(sms * per);
}

}  // namespace ez
