/*
 * expzip.h -- C ABI of libexpzip, lossless BF16 exponent codecs for sm_103a.
 *
 * Two codecs for BF16 weights in front of a sharded-data-parallel allgather:
 *
 *  code3  "ZipCCL: Efficient Lossless Data Compression of Communication
 *         Collectives" (research digest), section 3.1: each 8-bit exponent
 *         becomes a 3-bit code from a window of 7 exponents placed by the
 *         tensor's standard deviation (x_opt = log2 sigma + 1/2 log2(14 ln2 /
 *         16383)); code 000 escapes to the raw exponent.  Sign+mantissa stay
 *         one raw byte.  Output is written in per-peer chunks padded to 128 B
 *         (section 3.2: the codec writes the collective's chunk layout and
 *         only adds a size exchange).
 *  reuse  "CIERA: Cross-Iteration Exponent Reuse for Lossless Allgather in
 *         Sharded MoE Training", exponent-reuse paragraphs: each shard is cut
 *         into blocks of B values; a block whose exponents all equal the
 *         previous iteration's is not sent.  The payload is a changed-block
 *         bitmap, the sign+mantissa byte of every value and the exponents of
 *         the changed blocks (expected size S_{s+m} + S_bm + q*S_e, gain-
 *         formula paragraph).  The receiver merges them with its exponent
 *         cache (ExpCache).  REUSE_CODE3 codes the changed exponents with the
 *         3-bit code instead of nvCOMP's ANS.
 *
 * Geometry.  A plan describes one flat tensor of n BF16 values split into W
 * shards (= per-peer chunks) of L = 128*ceil(ceil(n/W)/128) values; shard r
 * covers [r*L, min((r+1)*L, n)) and trailing shards may be short or empty.
 *
 * Buffers.  Every pointer named d_* is a DEVICE pointer owned by the caller;
 * the library never allocates, frees or keeps a pointer after a call returns.
 * BF16 tensors are passed as their raw 16-bit patterns (uint16_t).  Value,
 * cache and payload buffers must be 16-byte aligned.  Every call is
 * asynchronous on `stream` (a cudaStream_t, NULL = legacy default stream):
 * a returned EZ_OK means the work was enqueued.  Calls that share a workspace
 * must not overlap in time (serialise them on one stream).
 *
 * Errors.  Problems visible on the host (bad plan, NULL or misaligned
 * pointer, capacity or workspace too small) return at once and enqueue
 * nothing.  Launch failures return EZ_ERR_CUDA.  Problems found in the data
 * (a corrupt or truncated payload, a look-back wait that timed out) are OR-ed
 * into the caller's device status word *d_status as EZ_DSTAT_* bits; read it
 * after synchronising.  Decoders never read outside [offset, offset+avail)
 * of a payload, whatever its contents, and never trap.  After a nonzero
 * status the decoded output and the receiver cache are unspecified: reset
 * the cache and send the next iteration cold.
 *
 * Byte formats (little-endian; all padding bytes are zero):
 *  code3 chunk: 128-B header {"EZC3", u8 version 2, u8 E0, u16 0, u64 n_c,
 *    u64 n_esc, u64 chunk_bytes, u32 chunk index, u32 W, zeros}; SM bytes
 *    (n_c, padded to 128); planes P0,P1,P2 (ceil(n_c/8) bytes each, padded
 *    to 128; bit p of code j is bit (j&7) of byte (j>>3) of plane p);
 *    escape index (u64 per 8192 values: escapes among the values before
 *    that point; ceil(n_c/8192) entries, padded to 128); escapes (n_esc raw
 *    exponents in value order, padded to 128).
 *    code = E-E0+1 for E0 <= E <= E0+6, else 0.
 *  reuse payload: 64-B header {"EZRU", u8 version 2, u8 flags (bit0 coded,
 *    bit1 cold), u8 E0, u8 0, u32 B, u32 shard, u64 n_s, u64 n_changed,
 *    u64 m, u64 n_esc, u64 total_bytes, u64 0}; bitmap (ceil(nb/8) bytes,
 *    block k = bit (k&7) of byte (k>>3), padded to 16); SM bytes (n_s,
 *    padded to 16); index (per 8192 values: u64 changed blocks before that
 *    point and, coded, u64 escapes among their exponents; padded to 16);
 *    EXP = the m exponents of the changed blocks in block order, or (coded)
 *    their 3 code planes (ceil(m/8) bytes each, padded to 16) followed by
 *    n_esc escapes; total padded to 128.
 *  The indices let a decoder place every 8192-value span independently;
 *  decoders check each entry against the span's own counts.
 */
#ifndef EXPZIP_H
#define EXPZIP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EZ_OK = 0,
    EZ_ERR_ARG = 1,          /* NULL / misaligned pointer, bad range, bad plan   */
    EZ_ERR_CUDA = 2,         /* a CUDA runtime call or launch failed             */
    EZ_ERR_CAPACITY = 3,     /* output or workspace smaller than required        */
    EZ_ERR_CORRUPT = 4,      /* reserved for host-side payload checks            */
    EZ_ERR_TIMEOUT = 5,      /* reserved for host-side waits                     */
    EZ_ERR_UNSUPPORTED = 6   /* valid request this build does not implement      */
} ez_status;

typedef enum {
    EZ_CODEC_CODE3 = 1,        /* ZipCCL 3-bit exponent code                     */
    EZ_CODEC_REUSE = 2,        /* CIERA exponent reuse, raw changed exponents    */
    EZ_CODEC_REUSE_CODE3 = 3,  /* CIERA reuse, changed exponents 3-bit coded     */
    EZ_CODEC_FP8_E5M2 = 4,     /* 3-bit exponent code on FP8 E5M2 values         */
    EZ_CODEC_FP8_E4M3 = 5      /* 3-bit exponent code on FP8 E4M3 values         */
} ez_codec;

/* bits OR-ed into a decoder's device status word */
#define EZ_DSTAT_BAD_HEADER  1u   /* magic, version, shard index, n, B, flags   */
#define EZ_DSTAT_BAD_SIZE    2u   /* declared size vs closed form or avail      */
#define EZ_DSTAT_BAD_COUNT   4u   /* escape / changed-block counts inconsistent */
#define EZ_DSTAT_TIMEOUT     8u   /* a bounded look-back wait gave up           */
#define EZ_DSTAT_MISALIGNED 16u   /* a payload offset is not 16-byte aligned    */
#define EZ_DSTAT_BAD_STATS  32u   /* encoder found a window base E0 > 249       */

typedef struct {
    uint64_t n;       /* values in the flat tensor (<= 2^40)                     */
    uint32_t W;       /* shards / per-peer chunks, 1..65536                      */
    uint32_t B;       /* reuse block size: power of two, 8..1024 (code3: ignored)*/
    uint32_t codec;   /* ez_codec                                                */
    uint32_t flags;   /* 0 or EZ_FLAG_WINDOW_HIST                                */
} ez_plan_desc;

/* Plan flag: the 3-bit code window of this plan's statistics (ez_stats and
 * the coded reuse encode's per-shard statistics) is always the densest run
 * of 7 exponent bins (ties to the lowest base, rule = 1), the window with the
 * fewest escapes, instead of the one placed by sigma.  sigma and var are
 * still computed and reported.  It suits tensors far from N(0, sigma^2),
 * e.g. norm weights near 1.0, where the sigma window misses every value. */
#define EZ_FLAG_WINDOW_HIST 1u

/* Plan flag (reuse codecs, any block size; EZ_ERR_ARG with the code3 and
 * FP8 codecs): CIERA's hash-based change detection.  The
 * sender cache holds two 64-bit hashes per block (HashCache, 16 bytes per
 * block instead of one byte per value): a block is sent when it is cold or
 * its hash pair differs, and the pair is then replaced.  Hash s of a block:
 * word i = the 8 exponent bytes of values 8i..8i+7 of the block (little-
 * endian, 0 past the shard), term_i = mix(word_i + seed_s + (i+1) * gamma),
 * hash = mix(sum of the B/8 terms mod 2^64), with mix the SplitMix64 output
 * function, gamma = 0x9E3779B97F4A7C15, seeds 0 and 0x5851F42D4C957F2D.  The
 * payload is the one the exponent compare gives unless a hash pair collides
 * (about 2^-128 per block); receivers are unchanged. */
#define EZ_FLAG_HASH_CACHE 2u

typedef struct ez_plan_s* ez_plan;   /* immutable after creation; may be shared */

typedef struct {
    uint64_t shard_len;        /* L                                               */
    uint64_t slot_bytes;       /* worst-case payload bytes of one shard (x128)    */
    uint64_t workspace_bytes;  /* device scratch every call of this plan needs    */
    uint64_t cache_bytes;      /* exponent-cache bytes of the full tensor (reuse) */
    uint64_t tile_values;      /* values per CUDA tile (8192)                     */
    uint64_t send_cache_bytes; /* sender cache of all W shards: cache_bytes, or   */
                               /* W * 16 * ceil(L / B) with EZ_FLAG_HASH_CACHE    */
} ez_sizes;

/* Statistics of one tensor (ZipCCL digest 3.1: "one call of torch.std gives
 * sigma").  s1 and s2 are the exact sums of the finite values and of their
 * squares, each rounded once to double; var = (s2 - s1*(s1/N)) / (N-1) with
 * N the finite count (Bessel-corrected, as torch.std); E0 = clamp(127 + x0,
 * 0, 249) with x0 the largest integer k such that var >= K * 2^(2k-1),
 * K = 16383 / (14 ln 2) -- the integer nearest x_opt, ties up.  When N < 2
 * or var <= 0 the window falls back to the 7 consecutive exponent bins with
 * the most values (ties to the lowest), rule = 1.  Written on the device. */
typedef struct {
    uint64_t hist[256];   /* count of each exponent field value                  */
    uint64_t n;           /* values                                             */
    uint64_t n_finite;    /* values with exponent field != 255                  */
    double s1;            /* exact sum of finite values, rounded once           */
    double s2;            /* exact sum of squares, rounded once                 */
    double var;           /* 0 when N < 2                                       */
    double sigma;         /* sqrt(var); 0 when var <= 0                         */
    double K;             /* 16383 / (14 ln 2)                                  */
    uint32_t E0;          /* window base: codes 1..7 cover E0..E0+6             */
    uint32_t rule;        /* 0 from sigma, 1 from the histogram (fallback, or   */
                          /* always with EZ_FLAG_WINDOW_HIST)                   */
    uint64_t n_escape;    /* values outside the window                          */
} ez_stats_t;

/* Create a plan.  Checks the descriptor and derives L, the worst-case slot
 * size and the workspace size.  Host only; EZ_ERR_ARG on a bad descriptor,
 * EZ_ERR_UNSUPPORTED for a block size outside 8..1024 powers of two. */
ez_status ez_plan_create(ez_plan* out, const ez_plan_desc* desc);

/* Free a plan (host only).  NULL is accepted. */
ez_status ez_plan_destroy(ez_plan p);

/* Sizes the caller must allocate for this plan (host only). */
ez_status ez_plan_sizes(ez_plan p, ez_sizes* out);

/* a1: statistics and window of n_values BF16 values at d_x (any count up to
 * 2^40, independent of the plan's n; the plan supplies the workspace layout).
 * Writes *d_stats.  ZipCCL digest 3.1 (Eqs. 1-5, Figure 2). */
ez_status ez_stats(ez_plan p, const uint16_t* d_x, uint64_t n_values,
                   ez_stats_t* d_stats, void* d_ws, uint64_t ws_bytes, void* stream);

/* a2: 3-bit exponent encode of chunks [first, first+count).  d_x holds the
 * values of those chunks contiguously (chunk first+i at d_x + i*L).  The
 * window base E0 is read from d_stats->E0 on the device (an ez_stats result,
 * e.g. over the whole tensor).  Chunk first+i is written to the slot
 * d_out + i*slot_bytes (out_bytes >= count*slot_bytes) and its size to
 * d_sizes[i].  d_status receives EZ_DSTAT_TIMEOUT / EZ_DSTAT_BAD_STATS.
 * ZipCCL digest 3.1 (code, chunk layout) and 3.2 (per-peer chunks). */
ez_status ez_encode_code3(ez_plan p, const uint16_t* d_x, uint32_t first, uint32_t count,
                          const ez_stats_t* d_stats, uint8_t* d_out, uint64_t out_bytes,
                          uint64_t* d_sizes, uint32_t* d_status,
                          void* d_ws, uint64_t ws_bytes, void* stream);

/* a6: decode code3 chunks [first, first+count).  Chunk first+i occupies
 * d_in[d_offsets[i] .. d_offsets[i+1]) (count+1 device offsets; the exclusive
 * prefix sum of the exchanged sizes, or slot starts).  Values of chunk
 * first+i go to d_out + i*L.  ZipCCL digest 3.2 ("decompress all"). */
ez_status ez_decode_code3(ez_plan p, const uint8_t* d_in, const uint64_t* d_offsets,
                          uint32_t first, uint32_t count, uint16_t* d_out,
                          uint32_t* d_status, void* d_ws, uint64_t ws_bytes, void* stream);

/* The local step of a compressed reduce-scatter fused into a6 (ZipCCL
 * digest 3.2, zipcclReduceScatter): chunks [first, first+count) as
 * ez_decode_code3, but chunk first+i is added into the FP32 accumulator
 * d_acc + i*L instead of written as BF16: d_acc[j] = (first_source ? 0 :
 * d_acc[j]) + (float)value_j, one IEEE single-precision addition each --
 * the same bits as ez_decode_code3 followed by ez_accumulate_bf16.  d_acc is
 * a 16-byte aligned device pointer owned by the caller.  A chunk that fails
 * its checks leaves its part of d_acc untouched and sets d_status. */
ez_status ez_decode_code3_accumulate(ez_plan p, const uint8_t* d_in, const uint64_t* d_offsets,
                                     uint32_t first, uint32_t count, float* d_acc, int first_source,
                                     uint32_t* d_status, void* d_ws, uint64_t ws_bytes, void* stream);

/* a3: exponent-reuse encode of shards [first, first+count) (one sender
 * encodes count = 1).  d_x and d_send_cache hold those shards contiguously
 * (shard first+i at offset i*L values / bytes).  A block is sent when cold
 * != 0 or one of its exponents differs from d_send_cache; the cache then
 * holds the current exponents.  Payload of shard first+i goes to the slot
 * d_out + i*slot_bytes, its size to d_sizes[i].  For EZ_CODEC_REUSE_CODE3 the
 * shard's statistics are computed in the same pass and, if d_stats is not
 * NULL, written to d_stats[i]; the changed exponents are 3-bit coded with
 * that shard's window.  With EZ_FLAG_HASH_CACHE, d_send_cache holds each
 * shard's block hash pairs instead (shard first+i at byte i*16*ceil(L/B)).
 * CIERA exponent-reuse paragraphs, Algorithm 1 sender side (split, detect,
 * pack; ANS replaced by the 3-bit code). */
ez_status ez_encode_reuse(ez_plan p, const uint16_t* d_x, uint32_t first, uint32_t count,
                          uint8_t* d_send_cache, int cold, uint8_t* d_out, uint64_t out_bytes,
                          uint64_t* d_sizes, ez_stats_t* d_stats, uint32_t* d_status,
                          void* d_ws, uint64_t ws_bytes, void* stream);

/* a4: decode one reuse payload of `shard` (payload_bytes available at
 * d_payload) against the receiver cache d_recv_cache (that shard's L bytes),
 * writing the shard's values to d_out and the changed blocks' exponents to
 * the cache.  CIERA: "replaces only the changed blocks ... merging all the
 * exponents with the received sign-plus-mantissa values". */
ez_status ez_decode_reuse(ez_plan p, const uint8_t* d_payload, uint64_t payload_bytes,
                          uint32_t shard, uint8_t* d_recv_cache, uint16_t* d_out,
                          uint32_t* d_status, void* d_ws, uint64_t ws_bytes, void* stream);

/* a5: gather-decode all W payloads of an allgather into the full tensor in
 * one launch.  Payload r occupies d_recv[d_offsets[r] .. d_offsets[r+1])
 * (W+1 device offsets).  Shard r is written to d_full_out + r*L.  For the
 * reuse codecs d_recv_cache is the receiver's full n-byte exponent cache;
 * for code3 and the FP8 codecs it is ignored (may be NULL); an FP8 plan
 * writes n bytes (d_full_out is then the FP8 tensor's bytes).  ZipCCL digest 3.2 zipcclAllGather
 * ("decompress all"); CIERA Decmp (the only codec step on the critical path). */
ez_status ez_gather_decode(ez_plan p, const uint8_t* d_recv, const uint64_t* d_offsets,
                           uint8_t* d_recv_cache, uint16_t* d_full_out, uint32_t* d_status,
                           void* d_ws, uint64_t ws_bytes, void* stream);

/* ---- FP8 ----------------------------------------------------------------
 * ZipCCL digest 3.3, last paragraph: the 3-bit exponent code applied to FP8
 * (E5M2 coded to 3 bits gives e = 0.75, E4M3 gives e ~ 0.88).  Formats as
 * in the OCP 8-bit floating-point specification: E5M2 (exponent bias 15,
 * infinities and NaN at exponent field 31) and E4M3 (bias 7, no
 * infinities, NaN only at S.1111.111).  A plan with codec EZ_CODEC_FP8_E5M2
 * or EZ_CODEC_FP8_E4M3 describes n FP8 values (one byte each, passed as raw
 * bit patterns) in W chunks of L = 128*ceil(ceil(n/W)/128) values; B is
 * ignored and EZ_FLAG_WINDOW_HIST may be set.  Each value keeps its sign
 * and m mantissa bits raw (sm = sign << m | mantissa, stored as 1 + m bit-
 * planes, plane q = bit q of sm); its exponent field E becomes the code
 * E - E0 + 1 for E0 <= E <= E0+6 (three code planes) or code 0 with E
 * appended to the chunk's escape list.
 * Chunk layout (little-endian, all padding zero): 128-byte header {"EZF8",
 * u8 version 1, u8 format (1 = E5M2, 2 = E4M3), u8 E0, u8 0, u64 n_c,
 * u64 n_esc, u64 chunk_bytes, u32 chunk index, u32 W, zeros}; the 1 + m
 * sign/mantissa planes then the 3 code planes (ceil(n_c/8) bytes each,
 * padded to 128; bit j&7 of byte j>>3 is value j); the escape index (u64
 * per 8192 values: escapes among the values before that point, padded to
 * 128); the escapes (raw exponent fields in value order, padded to 128). */

/* Statistics of FP8 values: as ez_stats_t, with the exact sums taken over
 * the finite values and E0 a field value in 0 .. 2^e - 7 (25 for E5M2, 9 for
 * E4M3): the largest e with var >= K * 2^(2(e - bias) - 1) (the integer
 * nearest x_opt, ties up), 0 if none; when N < 2, var <= 0 or with
 * EZ_FLAG_WINDOW_HIST, the densest 7 consecutive exponent bins (ties to the
 * lowest), rule = 1. */
typedef struct {
    uint64_t hist[32];    /* count of each exponent field value (16 for E4M3)   */
    uint64_t n;           /* values                                             */
    uint64_t n_finite;    /* values that are neither Inf nor NaN                */
    double s1;            /* exact sum of the finite values, rounded once       */
    double s2;            /* exact sum of their squares, rounded once           */
    double var;           /* (s2 - s1*(s1/N)) / (N-1); 0 when N < 2             */
    double sigma;         /* sqrt(var); 0 when var <= 0                         */
    double K;             /* 16383 / (14 ln 2)                                  */
    uint32_t E0;          /* window base field value                            */
    uint32_t rule;        /* 0 from sigma, 1 from the histogram                 */
    uint64_t n_escape;    /* values outside the window                          */
} ez_fp8_stats_t;

/* Statistics and window of n_values FP8 values at d_x (the plan's codec
 * fixes the format; any count up to 2^40).  Writes *d_stats (8-byte
 * aligned device memory).  EZ_ERR_ARG for a plan that is not an FP8 plan. */
ez_status ez_fp8_stats(ez_plan p, const uint8_t* d_x, uint64_t n_values, ez_fp8_stats_t* d_stats,
                       void* d_ws, uint64_t ws_bytes, void* stream);

/* Encode FP8 chunks [first, first+count): d_x holds those chunks' values
 * contiguously (chunk first+i at d_x + i*L), E0 is read from d_stats->E0 on
 * the device; chunk first+i goes to the slot d_out + i*slot_bytes and its
 * size to d_sizes[i].  d_status receives EZ_DSTAT_TIMEOUT (a look-back wait
 * gave up) or EZ_DSTAT_BAD_STATS (E0 above 2^e - 7; encoded with E0 = 0). */
ez_status ez_fp8_encode(ez_plan p, const uint8_t* d_x, uint32_t first, uint32_t count,
                        const ez_fp8_stats_t* d_stats, uint8_t* d_out, uint64_t out_bytes,
                        uint64_t* d_sizes, uint32_t* d_status, void* d_ws, uint64_t ws_bytes,
                        void* stream);

/* Decode FP8 chunks [first, first+count): chunk first+i occupies
 * d_in[d_offsets[i] .. d_offsets[i+1]); its values go to d_out + i*L.  A
 * chunk that fails its checks (header, sizes, index, escape count) is not
 * written and sets d_status bits as the code3 decoder does. */
ez_status ez_fp8_decode(ez_plan p, const uint8_t* d_in, const uint64_t* d_offsets, uint32_t first,
                        uint32_t count, uint8_t* d_out, uint32_t* d_status, void* d_ws,
                        uint64_t ws_bytes, void* stream);

/* Bytes of the library's fixed device scratch array used by
 * ez_encode_code3_noalloc (one array per device). */
#define EZ_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)

/* ez_encode_code3 without a caller workspace: the same encode and the same
 * results, with its scratch (tile counters, per-chunk tile counters and
 * look-back state) taken from a fixed array inside the library instead of
 * d_ws.  No counterpart in the papers: it exists for callers that cannot
 * allocate device memory at the point where they compress -- a
 * communication runtime's send path or a non-blocking host thread, where
 * cudaMalloc/cudaFree could synchronize the device and stall against
 * communication kernels still waiting on peers, or an application whose
 * memory belongs to a pooling allocator.  The call allocates nothing (no
 * cudaMalloc, no cudaFree, no allocating library).
 * Limit: the plan's encode scratch -- 8 bytes per 8192 values of the
 * encoded chunks plus about 3.5 KB of counters and records for 8 chunks --
 * must fit in EZ_NOALLOC_SCRATCH_BYTES, else EZ_ERR_CAPACITY and nothing is
 * launched (4 MiB covers e.g. 2^31 values in 8 chunks).
 * The first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress); make that first call before
 * any stream capture.  The address is kept for the life of the process, so
 * the device's primary context must live as long: do not call this entry
 * point on a device after cudaDeviceReset on it (the array would be at a new
 * address and the kept one would be stale).  Each call clears the scratch it needs on `stream`
 * before its launch; every call on a device shares the one array, so calls
 * whose work overlaps on the GPU (unordered streams) race and must not be
 * issued.  Devices with ordinal >= 64 give EZ_ERR_UNSUPPORTED.  Arguments
 * and device status bits as ez_encode_code3. */
ez_status ez_encode_code3_noalloc(ez_plan p, const uint16_t* d_x, uint32_t first, uint32_t count,
                                  const ez_stats_t* d_stats, uint8_t* d_out, uint64_t out_bytes,
                                  uint64_t* d_sizes, uint32_t* d_status, void* stream);

/* The local step of a compressed reduce-scatter (ZipCCL digest 3.2,
 * zipcclReduceScatter: an all-to-all of compressed chunks, then local
 * decompression and a sum in higher precision).  For i < n:
 *   d_acc[i] = (first ? 0 : d_acc[i]) + (float)bf16(d_x[i])
 * with one IEEE single-precision addition (round to nearest even) per
 * element, so calls over the W decoded chunks in source order give the bits
 * of a sequential float32 sum in that order.  d_acc (n floats, read and
 * written) and d_x (n raw BF16 values) are device pointers, 16-byte aligned,
 * owned by the caller; n = 0 does nothing.  EZ_ERR_ARG on a null or
 * misaligned pointer, EZ_ERR_CUDA on a launch error.  Needs no plan. */
ez_status ez_accumulate_bf16(float* d_acc, const uint16_t* d_x, uint64_t n, int first, void* stream);

/* Static text for a status code. */
const char* ez_status_str(ez_status s);

/* Library version as 0xMMmmpp. */
uint32_t ez_version(void);

#ifdef __cplusplus
}
#endif
#endif /* EXPZIP_H */
