// ez_internal.h -- plan object and kernel launchers of libexpzip (host side).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "expzip.h"

struct ez_plan_s {
    uint64_t n;
    uint32_t W, B, codec;
    uint64_t L;              // shard length
    uint32_t tpc;            // tiles per shard
    uint64_t slot_bytes;     // worst-case payload per shard
    double K;                // 16383 / (14 ln 2)
    // workspace layout (byte offsets); [0, zero_bytes) is cleared per call
    uint64_t off_ctr, off_info, off_shard_stats, off_bins, off_state_a, off_state_b, off_seg, off_escbuf, off_plbuf;
    uint64_t zero_bytes, ws_bytes;
    uint32_t n_bins;
    uint32_t hist_window;    // EZ_FLAG_WINDOW_HIST: window from the histogram
    uint32_t hash_cache;     // EZ_FLAG_HASH_CACHE: sender cache of block hashes
    uint64_t hstride;        // sender-cache bytes per shard (hash mode: 16 per block)
};

namespace ezk {

// Per-shard record of the reuse split, written by the tile that holds the
// shard's last value: the values by which the shard's last block falls short
// of B when that block changed, else 0.  The shard's changed-block count is
// the tile scan's last inclusive prefix, so its EXP length is
// m = n_changed * B - tail (no atomics on a per-shard total: with one shard
// every tile of the split would add to the same two words).
struct ShardInfo {
    unsigned long long tail;
    unsigned int pad[14];
};

struct WsView {
    uint32_t* counters;            // 8 tile counters
    uint32_t* shard_ctr;           // W per-shard tile counters
    ShardInfo* info;               // W records
    ez_stats_t* shard_stats;       // W records (reuse+code3 without caller stats)
    unsigned long long* state_a;
    unsigned long long* state_b;
    void* bins;                    // StatsBins[n_bins]
    uint8_t* escbuf;               // W * L bytes of staged escapes (coded reuse) or NULL
    uint8_t* plbuf;                // 3 KB of staged planes per tile (coded reuse) or NULL
    unsigned long long* seg_a;     // scan-segment states, two arrays of W * segments
    unsigned long long* seg_b;
};

WsView ws_view(const ez_plan_s* p, void* ws);

// Scan segments per chunk of tpc tiles (k_scan.cu).
cudaError_t launch_accumulate_bf16(float* acc, const uint16_t* x, uint64_t n, int first, cudaStream_t s);
cudaError_t launch_zero(void* p, uint64_t bytes, cudaStream_t s);
uint64_t tile_scan_segments(uint64_t tpc);

// Inclusive prefixes, per chunk, of the per-tile counts in st[count * tpc].
cudaError_t launch_tile_scan(const ez_plan_s* p, unsigned long long* st, uint32_t count,
                             unsigned long long* seg_st, uint32_t* counter, uint32_t* abort,
                             uint32_t* dstatus, cudaStream_t s);
// The same for two state arrays of the same geometry (own segment states and
// counters) in one launch.
cudaError_t launch_tile_scan2(const ez_plan_s* p, unsigned long long* st0, unsigned long long* seg0,
                              uint32_t* counter0, unsigned long long* st1, unsigned long long* seg1,
                              uint32_t* counter1, uint32_t count, uint32_t* abort, uint32_t* dstatus,
                              cudaStream_t s);

cudaError_t launch_stats(const ez_plan_s* p, const uint16_t* x, uint64_t n, ez_stats_t* out,
                         const WsView& w, cudaStream_t s);

// Statistics of shards [first, first+count) of the plan (values at x + i*L),
// one record per shard.
cudaError_t launch_shard_stats(const ez_plan_s* p, const uint16_t* x, uint32_t first, uint32_t count,
                               ez_stats_t* out, const WsView& w, cudaStream_t s);

cudaError_t launch_code3_encode(const ez_plan_s* p, const uint16_t* x, uint32_t first,
                                uint32_t count, const ez_stats_t* st, uint8_t* out,
                                uint64_t* sizes, uint32_t* dstatus, const WsView& w,
                                cudaStream_t s);

cudaError_t launch_code3_decode(const ez_plan_s* p, const uint8_t* in, const uint64_t* offsets,
                                uint32_t first, uint32_t count, uint16_t* out,
                                uint32_t* dstatus, const WsView& w, cudaStream_t s,
                                float* acc = nullptr, int acc_first = 0);

cudaError_t launch_reuse_encode(const ez_plan_s* p, const uint16_t* x, uint32_t first,
                                uint32_t count, uint8_t* cache, int cold, uint8_t* out,
                                uint64_t* sizes, ez_stats_t* st, uint32_t* dstatus,
                                const WsView& w, cudaStream_t s);

// FP8 codecs (k_fp8.cu): worst-case chunk bytes of L values, and the kernels.
uint64_t fp8_slot_bytes(uint32_t codec, uint64_t L);
cudaError_t launch_fp8_stats(const ez_plan_s* p, const uint8_t* x, uint64_t n, ez_fp8_stats_t* out,
                             const WsView& w, cudaStream_t s);
cudaError_t launch_fp8_encode(const ez_plan_s* p, const uint8_t* x, uint32_t first, uint32_t count,
                              const ez_fp8_stats_t* st, uint8_t* out, uint64_t* sizes, uint32_t* dstatus,
                              const WsView& w, cudaStream_t s);
cudaError_t launch_fp8_decode(const ez_plan_s* p, const uint8_t* in, const uint64_t* offsets, uint32_t first,
                              uint32_t count, uint8_t* out, uint32_t* dstatus, cudaStream_t s);

cudaError_t launch_reuse_decode(const ez_plan_s* p, const uint8_t* in, const uint64_t* offsets,
                                uint64_t single_avail, uint32_t first, uint32_t count,
                                uint8_t* cache, uint16_t* out, uint32_t* dstatus,
                                const WsView& w, cudaStream_t s);

}  // namespace ezk
