/*
 * ezoracle -- plain, slow, single-threaded CPU reference of the two lossless
 * BF16 exponent codecs.  TEST INFRASTRUCTURE ONLY: only the tests, the smoke
 * check and the benchmark's CPU-baseline leg load it.  It shares no code with
 * the CUDA library and never calls it.
 *
 * Pages followed (cited by title and section):
 *   [CIERA]  "CIERA: Cross-Iteration Exponent Reuse for Lossless Allgather in
 *            Sharded MoE Training" -- exponent reuse paragraphs (split into
 *            exponent and sign+mantissa, block partition, changed-block
 *            bitmap, ExpCache merge), the gain-formula paragraph (payload
 *            S_{s+m} + S_bm + q*S_e, S_bm = ceil(ceil(N/B)/8)), and the
 *            bitwise-identical-training paragraph (lossless round trip).
 *   [ZIP]    "ZipCCL: Efficient Lossless Data Compression of Communication
 *            Collectives" (research digest) -- section 3.1 (3-bit exponent
 *            code with escapes, window from sigma, Eqs. 1-5, Figure 2),
 *            section 3.2 (zipcclAllGather: sizes then blocks; static parts
 *            first), section 3.3 (break-even model, Eqs. 8-9).
 *
 * The pages fix no byte format; the format below is this library's reading,
 * and the CUDA path must reproduce it byte for byte.
 */
#ifndef EZORACLE_H
#define EZORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* statistics of one BF16 tensor [ZIP section 3.1] */
typedef struct {
    uint64_t hist[256];      /* count of each 8-bit exponent field value      */
    uint64_t n;              /* values                                        */
    uint64_t n_finite;       /* values with exponent field != 255             */
    double   s1;             /* exact sum of finite values, rounded once      */
    double   s2;             /* exact sum of squares, rounded once            */
    double   var;            /* (s2 - s1*(s1/N)) / (N-1); 0 when N < 2        */
    double   sigma;          /* sqrt(var), 0 when var <= 0                    */
    double   K;              /* 16383 / (14 ln 2)                             */
    uint32_t E0;             /* window base: codes cover E0 .. E0+6           */
    uint32_t rule;           /* 0: from sigma; 1: histogram fallback          */
    uint64_t n_escape;       /* values outside the window                     */
} orc_stats;

/* status bits reported by the decoders */
#define ORC_BAD_HEADER   1u   /* magic, version, index, n or B mismatch     */
#define ORC_BAD_SIZE     2u   /* declared size vs closed form / available   */
#define ORC_BAD_COUNT    4u   /* escape or changed-block count mismatch     */

uint64_t orc_shard_len(uint64_t n, uint32_t W);
uint64_t orc_shard_count(uint64_t n, uint32_t W, uint32_t r);

int  orc_stats_compute(const uint16_t* x, uint64_t n, orc_stats* st);
/* mode 1: window from the histogram's densest 7-bin run (ties to the lowest) */
int  orc_stats_compute_mode(const uint16_t* x, uint64_t n, int mode, orc_stats* st);
double orc_window_K(void);
uint32_t orc_window_from_var(double var);

/* code3: W per-peer chunks, chunk c written at out + c*slot_bytes */
uint64_t orc_code3_chunk_bytes(uint64_t n_c, uint64_t n_esc);
uint64_t orc_code3_slot_bytes(uint64_t n, uint32_t W);
int  orc_code3_encode_chunk(const uint16_t* xc, uint64_t n, uint32_t W, uint32_t c, uint32_t E0,
                            uint8_t* o, uint64_t slot_bytes, uint64_t* size);
int  orc_code3_encode(const uint16_t* x, uint64_t n, uint32_t W, uint32_t E0,
                      uint8_t* out, uint64_t slot_bytes, uint64_t* sizes);
/* one chunk c (ZipCCL digest 3.2: a peer's chunk of an all-to-all) */
uint32_t orc_code3_decode_chunk(const uint8_t* p, uint64_t avail, uint64_t n, uint32_t W,
                                uint32_t c, uint16_t* out_c);
uint32_t orc_code3_decode(const uint8_t* in, const uint64_t* offsets,
                          uint64_t n, uint32_t W, uint16_t* out);

/* reuse: one shard */
uint64_t orc_reuse_bytes(uint64_t n_s, uint32_t B, uint64_t m, int coded,
                         uint64_t n_esc);
uint64_t orc_reuse_slot_bytes(uint64_t n, uint32_t W, uint32_t B, int coded);
int  orc_reuse_encode(const uint16_t* shard, uint64_t n_s, uint32_t B,
                      uint32_t shard_index, uint8_t* send_cache, int cold,
                      int coded, orc_stats* st /* coded: shard stats, may be NULL */,
                      uint8_t* out, uint64_t cap, uint64_t* size);
int  orc_reuse_encode_mode(const uint16_t* shard, uint64_t n_s, uint32_t B,
                           uint32_t shard_index, uint8_t* send_cache, int cold,
                           int coded, int window_mode, orc_stats* st, uint8_t* out,
                           uint64_t cap, uint64_t* size);
/* CIERA's hash-based change detection: two 64-bit SplitMix64 hashes per
 * block in hash_cache (u64[2 * ceil(n_s / B)]); same payload as above. */
uint64_t orc_splitmix64_next(uint64_t* state);
uint64_t orc_block_hash(const uint16_t* shard, uint64_t n_s, uint32_t B, uint64_t k, int s);
int  orc_reuse_encode_hash(const uint16_t* shard, uint64_t n_s, uint32_t B,
                           uint32_t shard_index, uint64_t* hash_cache, int cold,
                           int coded, int window_mode, orc_stats* st, uint8_t* out,
                           uint64_t cap, uint64_t* size);
uint32_t orc_reuse_decode(const uint8_t* payload, uint64_t avail, uint64_t n_s,
                          uint32_t B, uint32_t shard_index,
                          uint8_t* recv_cache, uint16_t* out);

/* gather: W payloads at offsets[0..W] into out[n] */
uint32_t orc_gather_decode_reuse(const uint8_t* recv, const uint64_t* offsets,
                                 uint64_t n, uint32_t W, uint32_t B,
                                 uint8_t* recv_cache, uint16_t* out);

/* ---- FP8 (E5M2 / E4M3) with the 3-bit exponent code [ZIP 3.3]: oracle of
 * a format for later kernels; no library entry point yet ---- */
#define ORC_FP8_E5M2 1
#define ORC_FP8_E4M3 2
typedef struct {
    uint64_t hist[32];       /* count of each exponent field value (16 for E4M3) */
    uint64_t n, n_finite;
    double   s1, s2, var, sigma, K;
    uint32_t E0, rule;
    uint64_t n_escape;
} orc_fp8_stats_t;
int      orc_fp8_stats(const uint8_t* x, uint64_t n, int fmt, int window_mode, orc_fp8_stats_t* st);
uint64_t orc_fp8_chunk_bytes(uint64_t n_c, uint64_t n_esc, int fmt);
int      orc_fp8_encode(const uint8_t* x, uint64_t n, uint32_t W, int fmt, uint32_t E0,
                        uint8_t* out, uint64_t slot_bytes, uint64_t* sizes);
uint32_t orc_fp8_decode(const uint8_t* in, const uint64_t* offsets, uint64_t n, uint32_t W,
                        int fmt, uint8_t* out);

#ifdef __cplusplus
}
#endif
#endif
