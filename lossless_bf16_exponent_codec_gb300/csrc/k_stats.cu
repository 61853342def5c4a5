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

constexpr int kStatsLoads = 27;                             // 16-B loads per thread
constexpr int kStatsBatch = 3;                              // loads in flight per thread
static_assert(kStatsLoads % kStatsBatch == 0, "whole batches");
// 55296 values: 2^26 values make 1214 tiles, 8 shards of 2^23 make 1216,
// i.e. at most 8 per SM on 152 SMs (8 resident), none left for a second wave
constexpr uint32_t kStatsTile = kThreads * kStatsLoads * 8;
static_assert(kStatsTile <= kStatsMaxValues, "a tile's sums fit the 32-bit shared bins");

// One CTA per tile of 55296 values of one shard, 8 resident CTAs per SM;
// every thread keeps three 16-byte loads in flight and adds their 24 values
// to the CTA's histogram.  Shard ci = tile / tps holds values [ci*L, ci*L + n_s)
// of x; its CTAs fold into bins G[ci], and the last of them writes out[ci].
// The a1 statistics of a whole tensor are the case of one shard.
__global__ void __launch_bounds__(kThreads, 8)
k_stats(const uint16_t* __restrict__ x, uint64_t n, uint64_t L, uint32_t first, uint32_t W,
        uint32_t tps, StatsBins* G, ez_stats_t* out, double K, uint32_t hist_window)
{
    extern __shared__ __align__(16) unsigned char dyn[];
    StatsSmem& S = *reinterpret_cast<StatsSmem*>(dyn);
    grid_dep_launch();   // a dependent launch (the coded split) may be scheduled
    const uint32_t ci = blockIdx.x / tps, lt = blockIdx.x % tps;
    const uint64_t n_s = W ? shard_values(n, L, first + ci) : n;
    const uint64_t base = (uint64_t)lt * kStatsTile;
    const uint32_t nv = base < n_s ? (uint32_t)umin64(kStatsTile, n_s - base) : 0u;
    const uint16_t* xt = x + (uint64_t)ci * L + base;
    const int t = threadIdx.x;
    st_begin(S, (uint32_t)(8 * t) < nv ? (uint32_t)xt[8 * t] : 0xFFFFFFFFu);
    const uint32_t elo = S.elo;
    const uint32_t e7 = (elo << 7) * 0x10001u;
    const uint32_t hb = (uint32_t)__cvta_generic_to_shared(S.hist);
    const uint32_t jb = (uint32_t)__cvta_generic_to_shared(S.junk) + 4u * (uint32_t)(t & 31);
    if (nv == kStatsTile) {
        // full tile: no per-group bounds
#pragma unroll 1
        for (int g0 = 0; g0 < kStatsLoads; g0 += kStatsBatch) {
            uint4 w[kStatsBatch];
#pragma unroll
            for (int k = 0; k < kStatsBatch; k++) w[k] = ld_v4_nc(xt + 8u * (uint32_t)((g0 + k) * kThreads + t));
#pragma unroll
            for (int k = 0; k < kStatsBatch; k++) st_add8(w[k], e7, hb, jb, S);
        }
        grid_dep_wait();   // the bins were cleared by the kernel before
        if (st_end(S, G + ci, tps)) st_finalize(G + ci, n_s, K, out + ci, S, hist_window);
        return;
    }
#pragma unroll 1
    for (int g = 0; g < kStatsLoads; g++) {
        const uint32_t v = 8u * (uint32_t)(g * kThreads + t);
        if (v + 8 <= nv) {
            st_add8(ld_v4_nc(xt + v), e7, hb, jb, S);
        } else if (v < nv) {
            for (uint32_t i = v; i < nv; i++) st_add(xt[i], elo, S);
        }
    }
    grid_dep_wait();   // the bins were cleared by the kernel before
    if (st_end(S, G + ci, tps)) st_finalize(G + ci, n_s, K, out + ci, S, hist_window);
}

static cudaError_t stats_launch(const uint16_t* x, uint64_t n, uint64_t L, uint32_t first,
                                uint32_t W, uint32_t count, uint64_t per_shard, StatsBins* G,
                                ez_stats_t* out, double K, uint32_t hist_window, cudaStream_t s)
{
    const uint64_t tps = per_shard ? cdiv(per_shard, kStatsTile) : 1;
    const uint64_t tiles = tps * count;
    if (tiles > 0x7fffffffull) return cudaErrorInvalidValue;
    static PerDeviceAttr smem_attr;
    const cudaError_t attr = max_dyn_smem_per_device(smem_attr, k_stats, (int)sizeof(StatsSmem));
    if (attr != cudaSuccess) return attr;
    return launch_dependent(k_stats, (unsigned)tiles, kThreads, sizeof(StatsSmem), s, x, n, L, first, W,
                            (uint32_t)tps, G, out, K, hist_window);
}

cudaError_t launch_stats(const ez_plan_s* p, const uint16_t* x, uint64_t n, ez_stats_t* out,
                         const WsView& w, cudaStream_t s)
{
    return stats_launch(x, n, n, 0, 0, 1, n, (StatsBins*)w.bins, out, p->K, p->hist_window, s);
}

cudaError_t launch_shard_stats(const ez_plan_s* p, const uint16_t* x, uint32_t first, uint32_t count,
                               ez_stats_t* out, const WsView& w, cudaStream_t s)
{
    return stats_launch(x, p->n, p->L, first, p->W, count, p->L, (StatsBins*)w.bins, out, p->K,
                        p->hist_window, s);
}

}  // namespace ezk
