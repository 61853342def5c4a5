// api.cpp -- the C ABI of libexpzip: plans, argument checks, workspace
// layout, and kernel launches.  See include/expzip.h for the contract.
#include <cstdint>
#include <cstring>
#include <new>

#include "ez_internal.h"

namespace {

constexpr uint64_t kTileValues = 8192;   // ez::kTile
constexpr uint64_t kMaxN = 1ull << 40;

uint64_t cdiv(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
uint64_t rup(uint64_t a, uint64_t b) { return cdiv(a, b) * b; }
bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// bytes of the per-shard records and of StatsBins (must match the device types)
constexpr uint64_t kShardInfoBytes = 64;
constexpr uint64_t kStatsBinsBytes = 3 * 256 * 8 + 256;

bool is_reuse(const ez_plan_s* p)
{
    return p->codec == EZ_CODEC_REUSE || p->codec == EZ_CODEC_REUSE_CODE3;
}
bool is_fp8(const ez_plan_s* p) { return p->codec == EZ_CODEC_FP8_E5M2 || p->codec == EZ_CODEC_FP8_E4M3; }

ez_status cuda_status(cudaError_t e) { return e == cudaSuccess ? EZ_OK : EZ_ERR_CUDA; }

// Clear [0, bytes) of the workspace on the stream (a kernel; the encode's
// first kernel is a dependent launch after it).
ez_status clear_ws(void* ws, uint64_t bytes, cudaStream_t s)
{
    return cuda_status(ezk::launch_zero(ws, bytes, s));
}

ez_status check_ws(const ez_plan_s* p, const void* ws, uint64_t ws_bytes)
{
    if (!ws || !al(ws, 256)) return EZ_ERR_ARG;
    if (ws_bytes < p->ws_bytes) return EZ_ERR_CAPACITY;
    return EZ_OK;
}

}  // namespace

namespace ezk {

WsView ws_view(const ez_plan_s* p, void* ws)
{
    uint8_t* b = static_cast<uint8_t*>(ws);
    WsView v;
    v.counters = reinterpret_cast<uint32_t*>(b);
    v.shard_ctr = reinterpret_cast<uint32_t*>(b + p->off_ctr);
    v.info = reinterpret_cast<ShardInfo*>(b + p->off_info);
    v.shard_stats = reinterpret_cast<ez_stats_t*>(b + p->off_shard_stats);
    v.bins = b + p->off_bins;
    v.escbuf = p->off_escbuf ? b + p->off_escbuf : nullptr;
    v.plbuf = p->off_plbuf ? b + p->off_plbuf : nullptr;
    const uint64_t segs = tile_scan_segments(p->tpc) * p->W;
    v.seg_a = reinterpret_cast<unsigned long long*>(b + p->off_seg);
    v.seg_b = v.seg_a + segs;
    v.state_a = reinterpret_cast<unsigned long long*>(b + p->off_state_a);
    v.state_b = reinterpret_cast<unsigned long long*>(b + p->off_state_b);
    return v;
}

}  // namespace ezk

extern "C" {

ez_status ez_plan_create(ez_plan* out, const ez_plan_desc* d)
{
    if (!out || !d) return EZ_ERR_ARG;
    *out = nullptr;
    if ((d->flags & ~(EZ_FLAG_WINDOW_HIST | EZ_FLAG_HASH_CACHE)) || d->W == 0 || d->W > 65536 ||
        d->n > kMaxN)
        return EZ_ERR_ARG;
    if (d->codec < EZ_CODEC_CODE3 || d->codec > EZ_CODEC_FP8_E4M3) return EZ_ERR_ARG;
    const bool reuse = d->codec == EZ_CODEC_REUSE || d->codec == EZ_CODEC_REUSE_CODE3;
    const bool fp8 = d->codec == EZ_CODEC_FP8_E5M2 || d->codec == EZ_CODEC_FP8_E4M3;
    const bool hash = (d->flags & EZ_FLAG_HASH_CACHE) != 0;
    if (hash && !reuse) return EZ_ERR_ARG;
    if (reuse) {
        if (d->B == 0) return EZ_ERR_ARG;
        if (d->B < 8 || d->B > 1024 || (d->B & (d->B - 1))) return EZ_ERR_UNSUPPORTED;
    }
    ez_plan_s* p = new (std::nothrow) ez_plan_s();
    if (!p) return EZ_ERR_ARG;
    p->n = d->n;
    p->hist_window = (d->flags & EZ_FLAG_WINDOW_HIST) ? 1u : 0u;
    p->hash_cache = hash ? 1u : 0u;
    p->W = d->W;
    p->B = reuse ? d->B : 0;
    p->codec = d->codec;
    p->L = rup(cdiv(d->n, d->W), 128);
    const uint64_t tpc = p->L ? cdiv(p->L, kTileValues) : 1;
    p->tpc = (uint32_t)tpc;
    const uint64_t L = p->L;
    const uint64_t spans = cdiv(L, kTileValues);   // index entries per shard
    if (fp8) {
        p->slot_bytes = ezk::fp8_slot_bytes(d->codec, L);
    } else if (!reuse) {
        p->slot_bytes = 128 + L + 3 * rup(cdiv(L, 8), 128) + rup(8 * spans, 128) + L;
    } else {
        const uint64_t nb = cdiv(L, p->B);
        const uint64_t idx = rup((d->codec == EZ_CODEC_REUSE_CODE3 ? 16 : 8) * spans, 16);
        const uint64_t head = 64 + rup(cdiv(nb, 8), 16) + rup(L, 16) + idx;
        const uint64_t exp = (d->codec == EZ_CODEC_REUSE_CODE3) ? 3 * rup(cdiv(L, 8), 16) + L : L;
        p->slot_bytes = rup(head + exp, 128);
    }
    p->K = 16383.0 / (14.0 * 0.6931471805599453);
    const uint64_t W = d->W;
    const bool coded = d->codec == EZ_CODEC_REUSE_CODE3;
    p->n_bins = coded ? d->W : 1;
    uint64_t off = 256;                                   // 8 tile counters
    p->off_ctr = off;
    off = rup(off + W * 4, 256);                          // per-shard tile counters
    p->off_info = off;
    off = rup(off + W * kShardInfoBytes, 256);
    p->off_shard_stats = off;
    off = rup(off + (coded ? W * sizeof(ez_stats_t) : 0), 256);
    p->off_bins = off;
    off = rup(off + p->n_bins * kStatsBinsBytes, 256);
    p->off_state_a = off;
    off = rup(off + W * tpc * 8, 256);
    p->off_state_b = off;
    off = rup(off + (coded ? W * tpc * 8 : 0), 256);
    p->off_seg = off;                                     // two arrays of scan-segment states
    off = rup(off + 2 * W * ezk::tile_scan_segments(tpc) * 8, 256);
    // hash mode: the sender cache holds 16 bytes (two hashes) per block
    const uint64_t blocks = reuse ? cdiv(L, d->B) : 0;
    p->hstride = hash ? 16 * blocks : L;
    p->zero_bytes = off;
    // coded reuse: each tile's escapes staged at its own offset, its planes
    // in 3 KB per tile
    p->off_escbuf = coded ? off : 0;
    off = rup(off + (coded ? W * L : 0), 256);
    p->off_plbuf = coded ? off : 0;
    off = rup(off + (coded ? W * tpc * 3 * (kTileValues / 8) : 0), 256);
    p->ws_bytes = off;
    *out = p;
    return EZ_OK;
}

ez_status ez_plan_destroy(ez_plan p)
{
    delete p;
    return EZ_OK;
}

ez_status ez_plan_sizes(ez_plan p, ez_sizes* out)
{
    if (!p || !out) return EZ_ERR_ARG;
    out->shard_len = p->L;
    out->slot_bytes = p->slot_bytes;
    out->workspace_bytes = p->ws_bytes;
    out->cache_bytes = is_reuse(p) ? p->n : 0;
    out->tile_values = kTileValues;
    out->send_cache_bytes = !is_reuse(p) ? 0 : (p->hash_cache ? p->W * p->hstride : p->n);
    return EZ_OK;
}

ez_status ez_stats(ez_plan p, const uint16_t* d_x, uint64_t n_values, ez_stats_t* d_stats,
                   void* d_ws, uint64_t ws_bytes, void* stream)
{
    if (!p || !d_stats || !al(d_stats, 8) || n_values > kMaxN) return EZ_ERR_ARG;
    if (n_values && (!d_x || !al(d_x, 16))) return EZ_ERR_ARG;
    ez_status s = check_ws(p, d_ws, ws_bytes);
    if (s != EZ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = clear_ws(d_ws, p->off_state_a, st);
    if (s != EZ_OK) return s;
    return cuda_status(ezk::launch_stats(p, d_x, n_values, d_stats, ezk::ws_view(p, d_ws), st));
}

ez_status ez_encode_code3(ez_plan p, const uint16_t* d_x, uint32_t first, uint32_t count,
                          const ez_stats_t* d_stats, uint8_t* d_out, uint64_t out_bytes,
                          uint64_t* d_sizes, uint32_t* d_status, void* d_ws, uint64_t ws_bytes,
                          void* stream)
{
    if (!p || p->codec != EZ_CODEC_CODE3) return EZ_ERR_ARG;
    if (count == 0 || first >= p->W || count > p->W - first) return EZ_ERR_ARG;
    if (!d_stats || !al(d_stats, 8) || !d_out || !al(d_out, 16) || !d_sizes || !al(d_sizes, 8) ||
        !d_status || !al(d_status, 4))
        return EZ_ERR_ARG;
    if (p->n && (!d_x || !al(d_x, 16))) return EZ_ERR_ARG;
    if (out_bytes / p->slot_bytes < count) return EZ_ERR_CAPACITY;
    ez_status s = check_ws(p, d_ws, ws_bytes);
    if (s != EZ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = clear_ws(d_ws, p->zero_bytes, st);
    if (s != EZ_OK) return s;
    return cuda_status(ezk::launch_code3_encode(p, d_x, first, count, d_stats, d_out, d_sizes,
                                                d_status, ezk::ws_view(p, d_ws), st));
}

ez_status ez_decode_code3(ez_plan p, const uint8_t* d_in, const uint64_t* d_offsets, uint32_t first,
                          uint32_t count, uint16_t* d_out, uint32_t* d_status, void* d_ws,
                          uint64_t ws_bytes, void* stream)
{
    if (!p || p->codec != EZ_CODEC_CODE3) return EZ_ERR_ARG;
    if (count == 0 || first >= p->W || count > p->W - first) return EZ_ERR_ARG;
    if (!d_in || !al(d_in, 16) || !d_offsets || !al(d_offsets, 8) || !d_status || !al(d_status, 4))
        return EZ_ERR_ARG;
    if (p->n && (!d_out || !al(d_out, 16))) return EZ_ERR_ARG;
    ez_status s = check_ws(p, d_ws, ws_bytes);
    if (s != EZ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(ezk::launch_code3_decode(p, d_in, d_offsets, first, count, d_out, d_status,
                                                ezk::ws_view(p, d_ws), st));
}

ez_status ez_decode_code3_accumulate(ez_plan p, const uint8_t* d_in, const uint64_t* d_offsets,
                                     uint32_t first, uint32_t count, float* d_acc, int first_source,
                                     uint32_t* d_status, void* d_ws, uint64_t ws_bytes, void* stream)
{
    if (!p || p->codec != EZ_CODEC_CODE3) return EZ_ERR_ARG;
    if (count == 0 || first >= p->W || count > p->W - first) return EZ_ERR_ARG;
    if (!d_in || !al(d_in, 16) || !d_offsets || !al(d_offsets, 8) || !d_status || !al(d_status, 4))
        return EZ_ERR_ARG;
    if (p->n && (!d_acc || !al(d_acc, 16))) return EZ_ERR_ARG;
    ez_status s = check_ws(p, d_ws, ws_bytes);
    if (s != EZ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(ezk::launch_code3_decode(p, d_in, d_offsets, first, count, nullptr, d_status,
                                                ezk::ws_view(p, d_ws), st, d_acc, first_source ? 1 : 0));
}

ez_status ez_encode_reuse(ez_plan p, const uint16_t* d_x, uint32_t first, uint32_t count,
                          uint8_t* d_send_cache, int cold, uint8_t* d_out, uint64_t out_bytes,
                          uint64_t* d_sizes, ez_stats_t* d_stats, uint32_t* d_status, void* d_ws,
                          uint64_t ws_bytes, void* stream)
{
    if (!p || !is_reuse(p)) return EZ_ERR_ARG;
    if (count == 0 || first >= p->W || count > p->W - first) return EZ_ERR_ARG;
    if (!d_out || !al(d_out, 16) || !d_sizes || !al(d_sizes, 8) || !d_status || !al(d_status, 4))
        return EZ_ERR_ARG;
    if (p->n && (!d_x || !al(d_x, 16) || !d_send_cache || !al(d_send_cache, 16))) return EZ_ERR_ARG;
    if (d_stats && !al(d_stats, 8)) return EZ_ERR_ARG;
    if (out_bytes / p->slot_bytes < count) return EZ_ERR_CAPACITY;
    ez_status s = check_ws(p, d_ws, ws_bytes);
    if (s != EZ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = clear_ws(d_ws, p->zero_bytes, st);
    if (s != EZ_OK) return s;
    return cuda_status(ezk::launch_reuse_encode(p, d_x, first, count, d_send_cache, cold, d_out,
                                                d_sizes, d_stats, d_status, ezk::ws_view(p, d_ws),
                                                st));
}

ez_status ez_decode_reuse(ez_plan p, const uint8_t* d_payload, uint64_t payload_bytes, uint32_t shard,
                          uint8_t* d_recv_cache, uint16_t* d_out, uint32_t* d_status, void* d_ws,
                          uint64_t ws_bytes, void* stream)
{
    if (!p || !is_reuse(p) || shard >= p->W) return EZ_ERR_ARG;
    if (!d_payload || !al(d_payload, 16) || !d_status || !al(d_status, 4)) return EZ_ERR_ARG;
    if (p->n && (!d_recv_cache || !al(d_recv_cache, 16) || !d_out || !al(d_out, 16)))
        return EZ_ERR_ARG;
    ez_status s = check_ws(p, d_ws, ws_bytes);
    if (s != EZ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(ezk::launch_reuse_decode(p, d_payload, nullptr, payload_bytes, shard, 1,
                                                d_recv_cache, d_out, d_status,
                                                ezk::ws_view(p, d_ws), st));
}

ez_status ez_accumulate_bf16(float* d_acc, const uint16_t* d_x, uint64_t n, int first, void* stream)
{
    if (!n) return EZ_OK;
    if (!d_acc || !al(d_acc, 16) || !d_x || !al(d_x, 16)) return EZ_ERR_ARG;
    return cuda_status(ezk::launch_accumulate_bf16(d_acc, d_x, n, first, static_cast<cudaStream_t>(stream)));
}

ez_status ez_fp8_stats(ez_plan p, const uint8_t* d_x, uint64_t n_values, ez_fp8_stats_t* d_stats,
                       void* d_ws, uint64_t ws_bytes, void* stream)
{
    if (!p || !is_fp8(p) || !d_stats || !al(d_stats, 8) || n_values > kMaxN) return EZ_ERR_ARG;
    if (n_values && (!d_x || !al(d_x, 16))) return EZ_ERR_ARG;
    ez_status s = check_ws(p, d_ws, ws_bytes);
    if (s != EZ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = clear_ws(d_ws, p->off_state_a, st);
    if (s != EZ_OK) return s;
    return cuda_status(ezk::launch_fp8_stats(p, d_x, n_values, d_stats, ezk::ws_view(p, d_ws), st));
}

ez_status ez_fp8_encode(ez_plan p, const uint8_t* d_x, uint32_t first, uint32_t count,
                        const ez_fp8_stats_t* d_stats, uint8_t* d_out, uint64_t out_bytes,
                        uint64_t* d_sizes, uint32_t* d_status, void* d_ws, uint64_t ws_bytes,
                        void* stream)
{
    if (!p || !is_fp8(p)) return EZ_ERR_ARG;
    if (count == 0 || first >= p->W || count > p->W - first) return EZ_ERR_ARG;
    if (!d_stats || !al(d_stats, 8) || !d_out || !al(d_out, 16) || !d_sizes || !al(d_sizes, 8) ||
        !d_status || !al(d_status, 4))
        return EZ_ERR_ARG;
    if (p->n && (!d_x || !al(d_x, 16))) return EZ_ERR_ARG;
    if (out_bytes / p->slot_bytes < count) return EZ_ERR_CAPACITY;
    ez_status s = check_ws(p, d_ws, ws_bytes);
    if (s != EZ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = clear_ws(d_ws, p->zero_bytes, st);
    if (s != EZ_OK) return s;
    return cuda_status(ezk::launch_fp8_encode(p, d_x, first, count, d_stats, d_out, d_sizes, d_status,
                                              ezk::ws_view(p, d_ws), st));
}

ez_status ez_fp8_decode(ez_plan p, const uint8_t* d_in, const uint64_t* d_offsets, uint32_t first,
                        uint32_t count, uint8_t* d_out, uint32_t* d_status, void* d_ws,
                        uint64_t ws_bytes, void* stream)
{
    if (!p || !is_fp8(p)) return EZ_ERR_ARG;
    if (count == 0 || first >= p->W || count > p->W - first) return EZ_ERR_ARG;
    if (!d_in || !al(d_in, 16) || !d_offsets || !al(d_offsets, 8) || !d_status || !al(d_status, 4))
        return EZ_ERR_ARG;
    if (p->n && (!d_out || !al(d_out, 16))) return EZ_ERR_ARG;
    ez_status s = check_ws(p, d_ws, ws_bytes);
    if (s != EZ_OK) return s;
    return cuda_status(ezk::launch_fp8_decode(p, d_in, d_offsets, first, count, d_out, d_status,
                                              static_cast<cudaStream_t>(stream)));
}

ez_status ez_gather_decode(ez_plan p, const uint8_t* d_recv, const uint64_t* d_offsets,
                           uint8_t* d_recv_cache, uint16_t* d_full_out, uint32_t* d_status, void* d_ws,
                           uint64_t ws_bytes, void* stream)
{
    if (!p) return EZ_ERR_ARG;
    if (!d_recv || !al(d_recv, 16) || !d_offsets || !al(d_offsets, 8) || !d_status ||
        !al(d_status, 4))
        return EZ_ERR_ARG;
    if (p->n && (!d_full_out || !al(d_full_out, 16))) return EZ_ERR_ARG;
    if (is_reuse(p) && p->n && (!d_recv_cache || !al(d_recv_cache, 16))) return EZ_ERR_ARG;
    ez_status s = check_ws(p, d_ws, ws_bytes);
    if (s != EZ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const ezk::WsView w = ezk::ws_view(p, d_ws);
    if (is_fp8(p))
        return cuda_status(ezk::launch_fp8_decode(p, d_recv, d_offsets, 0, p->W,
                                                  reinterpret_cast<uint8_t*>(d_full_out), d_status, st));
    if (!is_reuse(p))
        return cuda_status(
            ezk::launch_code3_decode(p, d_recv, d_offsets, 0, p->W, d_full_out, d_status, w, st));
    return cuda_status(ezk::launch_reuse_decode(p, d_recv, d_offsets, 0, 0, p->W, d_recv_cache,
                                                d_full_out, d_status, w, st));
}

const char* ez_status_str(ez_status s)
{
    switch (s) {
        case EZ_OK: return "ok";
        case EZ_ERR_ARG: return "invalid argument";
        case EZ_ERR_CUDA: return "CUDA error";
        case EZ_ERR_CAPACITY: return "buffer or workspace too small";
        case EZ_ERR_CORRUPT: return "corrupt payload";
        case EZ_ERR_TIMEOUT: return "timed out";
        case EZ_ERR_UNSUPPORTED: return "unsupported";
    }
    return "unknown status";
}

uint32_t ez_version(void) { return 0x000300u; }

}  // extern "C"
