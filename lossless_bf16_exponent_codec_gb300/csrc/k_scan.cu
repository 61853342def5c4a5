// k_scan.cu -- prefix sums of per-tile counts, between the split and place
// steps of the encoders.
//
// A split launch publishes one count per 8192-value tile (escapes, changed
// blocks) in a tile-state array, chunk-major: st[c * tpc + t], the value in
// the low 62 bits.  This launch replaces every entry by the inclusive prefix
// of its chunk (flag bits cleared), so tile t of chunk c starts at
// st[c*tpc + t - 1] (0 for t = 0) and the chunk's total is st[c*tpc + tpc-1].
// One CTA scans a segment of kScanSpan entries of one chunk (8 per thread,
// one block scan); segments of a chunk are chained by a decoupled look-back
// over per-segment states (ids from an atomic counter, so a segment waits
// only on running ones; every wait bounded).  The coded reuse encoder scans
// its changed-block and escape counts in one launch of two halves.
#include "ez_internal.h"
#include "ez_common.cuh"

namespace ezk {
using namespace ez;

constexpr uint32_t kScanPer = 8;
constexpr uint32_t kScanSpan = kThreads * kScanPer;   // 2048 tile entries per CTA

// One state array to scan: per-tile counts, per-segment look-back states and
// the ticket counter of its segments.
struct ScanArr {
    unsigned long long* st;
    unsigned long long* seg_st;
    uint32_t* counter;
};

// Scans one or two state arrays of the same geometry in one launch: CTAs
// [0, count * spc) take the first array, the rest the second; each array has
// its own ticket counter, so a look-back only ever waits on the same array.
__global__ void __launch_bounds__(kThreads) k_tile_scan(ScanArr A0, ScanArr A1, uint32_t count,
                                                        uint32_t tpc, uint32_t spc, uint32_t* abort,
                                                        uint32_t* dstatus)
{
    __shared__ uint32_t s_tile;
    __shared__ unsigned long long s_warp[kThreads / 32];
    __shared__ unsigned long long s_prefix;
    const int t = threadIdx.x;
    grid_dep_launch();
    grid_dep_wait();   // the counts come from the kernel before
    const ScanArr A = blockIdx.x < count * spc ? A0 : A1;
    const uint32_t id = next_tile(A.counter, &s_tile);
    const uint32_t c = id / spc, sg = id % spc;   // segments of a chunk in order
    if (c >= count) return;
    unsigned long long* sc = A.st + (uint64_t)c * tpc;
    const uint32_t base = sg * kScanSpan + (uint32_t)t * kScanPer;
    unsigned long long v[kScanPer];
    unsigned long long sum = 0;
#pragma unroll
    for (uint32_t i = 0; i < kScanPer; i++) {
        v[i] = base + i < tpc ? (ld_relaxed(sc + base + i) & kValMask) : 0ull;
        sum += v[i];
    }
    unsigned long long total;
    const unsigned long long excl = block_excl_scan(sum, s_warp, &total);
    const unsigned long long P = tile_prefix(A.seg_st, c * spc + sg, c * spc, total, &s_prefix,
                                             dstatus, abort);
    unsigned long long run = P + excl;
#pragma unroll
    for (uint32_t i = 0; i < kScanPer; i++) {
        run += v[i];
        if (base + i < tpc) st_relaxed(sc + base + i, run);
    }
}

cudaError_t launch_tile_scan(const ez_plan_s* p, unsigned long long* st, uint32_t count,
                             unsigned long long* seg_st, uint32_t* counter, uint32_t* abort,
                             uint32_t* dstatus, cudaStream_t s)
{
    const uint32_t spc = (uint32_t)cdiv(p->tpc, kScanSpan);
    const uint64_t ctas = (uint64_t)count * spc;
    if (ctas > 0x7fffffffull) return cudaErrorInvalidValue;
    const ScanArr A{st, seg_st, counter};
    return launch_dependent(k_tile_scan, (unsigned)ctas, kThreads, 0, s, A, A, count, p->tpc, spc, abort,
                            dstatus);
}

cudaError_t launch_tile_scan2(const ez_plan_s* p, unsigned long long* st0, unsigned long long* seg0,
                              uint32_t* counter0, unsigned long long* st1, unsigned long long* seg1,
                              uint32_t* counter1, uint32_t count, uint32_t* abort, uint32_t* dstatus,
                              cudaStream_t s)
{
    const uint32_t spc = (uint32_t)cdiv(p->tpc, kScanSpan);
    const uint64_t ctas = 2ull * count * spc;
    if (ctas > 0x7fffffffull) return cudaErrorInvalidValue;
    return launch_dependent(k_tile_scan, (unsigned)ctas, kThreads, 0, s, ScanArr{st0, seg0, counter0},
                            ScanArr{st1, seg1, counter1}, count, p->tpc, spc, abort, dstatus);
}

uint64_t tile_scan_segments(uint64_t tpc) { return cdiv(tpc, kScanSpan); }

// Workspace clear before an encode: a kernel rather than a memset, so that
// the encode's first kernel can be a dependent launch (it starts its loads
// while this runs and waits before it touches the workspace).
__global__ void __launch_bounds__(kThreads) k_zero(uint4* p, uint64_t n16)
{
    grid_dep_launch();
    for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < n16; i += (uint64_t)gridDim.x * kThreads)
        p[i] = make_uint4(0, 0, 0, 0);
}

cudaError_t launch_zero(void* p, uint64_t bytes, cudaStream_t s)
{
    if (!bytes) return cudaSuccess;
    if ((bytes & 15u) || (reinterpret_cast<uintptr_t>(p) & 15u)) return cudaMemsetAsync(p, 0, bytes, s);
    const uint64_t n16 = bytes / 16;
    const unsigned grid = (unsigned)umin64(cdiv(n16, kThreads), 1024);
    k_zero<<<grid, kThreads, 0, s>>>(reinterpret_cast<uint4*>(p), n16);
    return cudaGetLastError();
}

}  // namespace ezk
