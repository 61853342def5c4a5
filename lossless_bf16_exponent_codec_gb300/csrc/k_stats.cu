// k_stats.cu -- a1: statistics and window of one BF16 tensor (ZipCCL digest
// 3.1, "one call of torch.std gives sigma, and the code table follows").
//
// Each CTA adds a tile of values into the exact accumulators of
// ez_stats.cuh and folds them into the global bins; the last CTA to finish
// computes s1, s2, var, sigma and E0 and writes the ez_stats_t record.
#include "ez_internal.h"
#include "ez_stats.cuh"

namespace ezk {
using namespace ez;

static_assert(sizeof(StatsBins) == 3 * 256 * 8 + 256, "StatsBins layout (api.cpp sizes it)");
static_assert(sizeof(ShardInfo) == 64, "ShardInfo layout (api.cpp sizes it)");
static_assert(sizeof(ez_stats_t) == 2120, "ez_stats_t layout");

constexpr int kStatsLoads = 16;                             // 16-B loads per thread
constexpr uint32_t kStatsTile = kThreads * kStatsLoads * 8;   // 32768 values

// One CTA per tile of 32768 values, 6 resident CTAs per SM; every thread
// keeps four 16-byte loads in flight and adds their 32 values to the CTA's
// histogram.
__global__ void __launch_bounds__(kThreads, 6)
k_stats(const uint16_t* __restrict__ x, uint64_t n, StatsBins* G, ez_stats_t* out, double K)
{
    extern __shared__ __align__(16) unsigned char dyn[];
    StatsSmem& S = *reinterpret_cast<StatsSmem*>(dyn);
    const uint64_t base = (uint64_t)blockIdx.x * kStatsTile;
    const uint32_t nv = base < n ? (uint32_t)umin64(kStatsTile, n - base) : 0u;
    const uint16_t* xt = x + base;
    const int t = threadIdx.x;
    st_begin(S, (uint32_t)(8 * t) < nv ? (uint32_t)xt[8 * t] : 0xFFFFFFFFu);
    const uint32_t elo = S.elo;
#pragma unroll 1
    for (int g0 = 0; g0 < kStatsLoads; g0 += 4) {
        uint4 w[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const uint32_t v = 8u * (uint32_t)((g0 + k) * kThreads + t);
            if (v + 8 <= nv) {
                w[k] = ld_v4_nc(xt + v);
            } else {
                uint32_t h[8];
#pragma unroll
                for (int i = 0; i < 8; i++) h[i] = (v + i < nv) ? (uint32_t)xt[v + i] : 0u;
                w[k] = make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16,
                                  h[6] | h[7] << 16);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const uint32_t v = 8u * (uint32_t)((g0 + k) * kThreads + t);
            if (v + 8 <= nv) {
                const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    st_add(ws[q] & 0xFFFFu, elo, S);
                    st_add(ws[q] >> 16, elo, S);
                }
            } else if (v < nv) {
                for (int i = 0; i < 8; i++)
                    if (v + i < nv) st_add(half_of(w[k], i), elo, S);
            }
        }
    }
    if (st_end(S, G, gridDim.x)) st_finalize(G, n, K, out, S);
}

cudaError_t launch_stats(const ez_plan_s* p, const uint16_t* x, uint64_t n, ez_stats_t* out,
                         const WsView& w, cudaStream_t s)
{
    const uint64_t tiles = n ? cdiv(n, kStatsTile) : 1;
    if (tiles > 0x7fffffffull) return cudaErrorInvalidValue;
    static const cudaError_t attr = cudaFuncSetAttribute(
        k_stats, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(StatsSmem));
    if (attr != cudaSuccess) return attr;
    k_stats<<<(unsigned)tiles, kThreads, sizeof(StatsSmem), s>>>(x, n, (StatsBins*)w.bins, out,
                                                               p->K);
    return cudaGetLastError();
}

}  // namespace ezk
