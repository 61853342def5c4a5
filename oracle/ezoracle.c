/*
 * ezoracle.c -- plain CPU reference of the lossless BF16 exponent codecs.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use this file.  It is deliberately slow and literal: one
 * value at a time, in value order, no blocking and no fusion, so that each
 * step can be checked against the pages by eye.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * Byte layouts (all integers little-endian, all padding bytes zero):
 *
 * BF16 split [CIERA, exponent-reuse paragraph; ZIP 3.1]
 *   h = 16 bits: sign s = h>>15, exponent E = (h>>7)&0xFF, mantissa m = h&0x7F.
 *   sign+mantissa byte SM = (s<<7)|m.  merge(SM,E) = ((SM&0x80)<<8)|(E<<7)|(SM&0x7F).
 *
 * Shards / per-peer chunks
 *   L = 128 * ceil(ceil(n/W)/128); shard r covers [r*L, min((r+1)*L, n)).
 *
 * code3 chunk [ZIP 3.1 code and layout; 3.2 AllGather/AlltoAll; 3.1 measured
 * size: "padding, indices"]
 *   header 128 B: "EZC3", u8 version=2, u8 E0, u16 0, u64 n_c, u64 n_esc,
 *                 u64 chunk_bytes, u32 chunk index, u32 W, zeros
 *   SM    : n_c bytes, padded to 128
 *   P0..P2: ceil(n_c/8) bytes each, padded to 128; bit p of code(j) is bit
 *           (j&7) of byte (j>>3) of plane p
 *   IDX   : u64 per 8192 values, T = ceil(n_c/8192) entries; IDX[k] = number
 *           of escapes among values [0, 8192k); padded to 128
 *   ESC   : n_esc raw exponent bytes in value order, padded to 128
 *   code(j) = E-E0+1 when E0 <= E <= E0+6, else 0 (escape)
 *
 * reuse payload [CIERA, exponent-reuse and gain-formula paragraphs]
 *   header 64 B: "EZRU", u8 version=2, u8 flags (bit0 exponents code3-coded,
 *                bit1 cold), u8 E0, u8 0, u32 B, u32 shard index, u64 n_s,
 *                u64 n_changed, u64 m, u64 n_esc, u64 total_bytes, u64 0
 *   BM : ceil(nb/8) bytes, nb = ceil(n_s/B); bit k = block k changed, bit
 *        (k&7) of byte (k>>3); padded to 16
 *   SM : n_s bytes, padded to 16
 *   IDX: per 8192 values, T = ceil(n_s/8192) entries: u64 number of changed
 *        blocks among blocks [0, 8192k/B), and, when coded, a second u64:
 *        number of escapes among the EXP exponents of those blocks; padded
 *        to 16 (B divides 8192, so no block straddles an entry)
 *   EXP: raw  -> the m exponent bytes of the changed blocks, block order
 *        coded-> planes P0..P2 of the code3 code of those m exponents (each
 *               ceil(m/8) bytes padded to 16), then n_esc escape bytes
 *   total padded to 128.
 */
#include "ezoracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ split */

static uint8_t bf16_exp(uint16_t h) { return (uint8_t)((h >> 7) & 0xFF); }
static uint8_t bf16_sm(uint16_t h) { return (uint8_t)(((h >> 8) & 0x80) | (h & 0x7F)); }
static uint16_t bf16_merge(uint8_t sm, uint8_t e)
{
    return (uint16_t)(((uint16_t)(sm & 0x80) << 8) | ((uint16_t)e << 7) | (sm & 0x7F));
}

static uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
static uint64_t round_up(uint64_t a, uint64_t b) { return ceil_div(a, b) * b; }

uint64_t orc_shard_len(uint64_t n, uint32_t W)
{
    return round_up(ceil_div(n, W), 128);
}

uint64_t orc_shard_count(uint64_t n, uint32_t W, uint32_t r)
{
    uint64_t L = orc_shard_len(n, W);
    uint64_t a = (uint64_t)r * L;
    if (a >= n) return 0;
    return (n - a < L) ? n - a : L;
}

/* little-endian field access */
static void put_u32(uint8_t* p, uint32_t v)
{
    for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i));
}
static void put_u64(uint8_t* p, uint64_t v)
{
    for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i));
}
static uint32_t get_u32(const uint8_t* p)
{
    uint32_t v = 0;
    for (int i = 3; i >= 0; i--) v = (v << 8) | p[i];
    return v;
}
static uint64_t get_u64(const uint8_t* p)
{
    uint64_t v = 0;
    for (int i = 7; i >= 0; i--) v = (v << 8) | p[i];
    return v;
}

/* ------------------------------------------------------------ big integer */
/* Non-negative integers of 768 bits, used only to sum the moments exactly. */

#define BIG_LIMBS 24
typedef struct { uint32_t w[BIG_LIMBS]; } big_t;

static void big_add_pow2(big_t* a, unsigned pos)
{
    unsigned i = pos / 32;
    uint32_t add = 1u << (pos % 32);
    while (i < BIG_LIMBS) {
        uint32_t old = a->w[i];
        a->w[i] = old + add;
        if (a->w[i] >= old) return;   /* no carry out */
        add = 1;
        i++;
    }
    abort();                          /* cannot happen for n < 2**40 */
}

/* a += v * 2**sh, one set bit of v at a time */
static void big_add_shifted(big_t* a, uint64_t v, unsigned sh)
{
    for (unsigned i = 0; i < 64; i++)
        if ((v >> i) & 1u) big_add_pow2(a, sh + i);
}

static int big_cmp(const big_t* a, const big_t* b)
{
    for (int i = BIG_LIMBS - 1; i >= 0; i--) {
        if (a->w[i] != b->w[i]) return a->w[i] > b->w[i] ? 1 : -1;
    }
    return 0;
}

/* a -= b, requires a >= b */
static void big_sub(big_t* a, const big_t* b)
{
    uint32_t borrow = 0;
    for (int i = 0; i < BIG_LIMBS; i++) {
        uint64_t ai = a->w[i], bi = (uint64_t)b->w[i] + borrow;
        a->w[i] = (uint32_t)(ai - bi);
        borrow = ai < bi;
    }
}

static int big_bit(const big_t* a, int pos)
{
    return (a->w[pos / 32] >> (pos % 32)) & 1u;
}

static int big_bitlen(const big_t* a)
{
    for (int pos = 32 * BIG_LIMBS - 1; pos >= 0; pos--)
        if (big_bit(a, pos)) return pos + 1;
    return 0;
}

/* a * 2**scale rounded to the nearest double, ties to even */
static double big_round(const big_t* a, int scale)
{
    int L = big_bitlen(a);
    if (L == 0) return 0.0;
    uint64_t q = 0;
    if (L <= 53) {
        for (int i = L - 1; i >= 0; i--) q = 2 * q + (uint64_t)big_bit(a, i);
        return ldexp((double)q, scale);
    }
    for (int i = L - 1; i >= L - 53; i--) q = 2 * q + (uint64_t)big_bit(a, i);
    int half = big_bit(a, L - 54);
    int sticky = 0;
    for (int i = L - 55; i >= 0; i--) sticky |= big_bit(a, i);
    if (half && (sticky || (q & 1u))) q++;
    return ldexp((double)q, L - 53 + scale);
}

/* ------------------------------------------------------------ statistics */

/* K = 16383 / (14 ln 2): sigma^2 >= K * 2^(2k-1)  <=>  x_opt + 1/2 >= k,
 * with x_opt = log2(sigma) + (1/2) log2(14 ln 2 / 16383)  [ZIP 3.1, Eq. for
 * x_opt].  So the integer nearest x_opt (ties up) is the largest such k. */
double orc_window_K(void)
{
    return 16383.0 / (14.0 * log(2.0));
}

uint32_t orc_window_from_var(double var)
{
    double K = orc_window_K();
    uint32_t E0 = 0;
    for (int e = 1; e <= 249; e++) {       /* E0 = 127 + x0, clamped to 0..249 */
        int k = e - 127;
        if (var >= ldexp(K, 2 * k - 1)) E0 = (uint32_t)e;
    }
    return E0;
}

int orc_stats_compute(const uint16_t* x, uint64_t n, orc_stats* st)
{
    return orc_stats_compute_mode(x, n, 0, st);
}

/* mode 0: the window from sigma, the histogram only as the fallback
 * [ZIP 3.1]; mode 1: the window always from the histogram (the densest
 * run of 7 exponent bins), sigma still computed and reported. */
int orc_stats_compute_mode(const uint16_t* x, uint64_t n, int mode, orc_stats* st)
{
    int64_t S1[256];
    uint64_t S2[256];
    memset(st, 0, sizeof(*st));
    memset(S1, 0, sizeof(S1));
    memset(S2, 0, sizeof(S2));
    st->n = n;
    /* exact per-exponent moments of v = (-1)^s * M * 2^(k(E)),
     * M = E ? 128+m : m, k(E) = (E ? E : 1) - 134 */
    for (uint64_t i = 0; i < n; i++) {
        uint16_t h = x[i];
        unsigned E = bf16_exp(h);
        st->hist[E]++;
        if (E == 255) continue;            /* Inf / NaN stay out of sigma */
        st->n_finite++;
        int64_t M = (E ? 128 : 0) + (h & 0x7F);
        S1[E] += (h & 0x8000) ? -M : M;
        S2[E] += (uint64_t)(M * M);
    }
    /* s1 = sum_E S1[E] * 2^(k(E)), exactly, as (P - Q) * 2^-133 */
    big_t P, Q, R;
    memset(&P, 0, sizeof(P));
    memset(&Q, 0, sizeof(Q));
    memset(&R, 0, sizeof(R));
    for (unsigned E = 0; E < 255; E++) {
        unsigned sh = (E ? E : 1) - 1;     /* k(E) + 133 */
        if (S1[E] >= 0) big_add_shifted(&P, (uint64_t)S1[E], sh);
        else big_add_shifted(&Q, (uint64_t)(-S1[E]), sh);
        big_add_shifted(&R, S2[E], 2 * sh);  /* s2 = R * 2^-266 */
    }
    if (big_cmp(&P, &Q) >= 0) {
        big_sub(&P, &Q);
        st->s1 = big_round(&P, -133);
    } else {
        big_sub(&Q, &P);
        st->s1 = -big_round(&Q, -133);
    }
    st->s2 = big_round(&R, -266);
    st->K = orc_window_K();
    st->rule = 1;
    if (st->n_finite >= 2) {
        double N = (double)st->n_finite;
        double var = (st->s2 - st->s1 * (st->s1 / N)) / (N - 1.0);
        st->var = var;
        if (var > 0 && isfinite(var)) {
            st->sigma = sqrt(var);
            if (mode == 0) {
                st->E0 = orc_window_from_var(var);
                st->rule = 0;
            }
        }
    }
    if (st->rule == 1) {
        /* fallback: the 7 consecutive exponent bins with the most values */
        uint64_t best = 0;
        uint32_t best_b = 0;
        for (uint32_t b = 0; b <= 249; b++) {
            uint64_t c = 0;
            for (uint32_t E = b; E <= b + 6; E++) c += st->hist[E];
            if (c > best) { best = c; best_b = b; }
        }
        st->E0 = best_b;
    }
    uint64_t in_window = 0;
    for (uint32_t E = st->E0; E <= st->E0 + 6; E++) in_window += st->hist[E];
    st->n_escape = n - in_window;
    return 0;
}

/* ------------------------------------------------------------------ code3 */

static unsigned code_of(unsigned E, unsigned E0)
{
    return (E >= E0 && E <= E0 + 6) ? E - E0 + 1 : 0;
}

#define IDX_SPAN 8192u

uint64_t orc_code3_chunk_bytes(uint64_t n_c, uint64_t n_esc)
{
    return 128 + round_up(n_c, 128) + 3 * round_up(ceil_div(n_c, 8), 128)
           + round_up(8 * ceil_div(n_c, IDX_SPAN), 128) + round_up(n_esc, 128);
}

uint64_t orc_code3_slot_bytes(uint64_t n, uint32_t W)
{
    uint64_t L = orc_shard_len(n, W);
    return orc_code3_chunk_bytes(L, L);
}

/* Chunk c of an n-value tensor split W ways: its n_c values at xc, encoded
 * into o (slot_bytes available); the chunk's size goes to *size. */
int orc_code3_encode_chunk(const uint16_t* xc, uint64_t n, uint32_t W, uint32_t c, uint32_t E0,
                           uint8_t* o, uint64_t slot_bytes, uint64_t* size)
{
    if (W == 0 || c >= W || E0 > 249) return -1;
    uint64_t n_c = orc_shard_count(n, W, c);
    uint64_t n_esc = 0;
    for (uint64_t j = 0; j < n_c; j++)
        if (code_of(bf16_exp(xc[j]), E0) == 0) n_esc++;
    uint64_t bytes = orc_code3_chunk_bytes(n_c, n_esc);
    if (bytes > slot_bytes) return -2;
    memset(o, 0, bytes);
    o[0] = 'E'; o[1] = 'Z'; o[2] = 'C'; o[3] = '3';
    o[4] = 2;
    o[5] = (uint8_t)E0;
    put_u64(o + 8, n_c);
    put_u64(o + 16, n_esc);
    put_u64(o + 24, bytes);
    put_u32(o + 32, c);
    put_u32(o + 36, W);
    uint64_t off_sm = 128;
    uint64_t plane = round_up(ceil_div(n_c, 8), 128);
    uint64_t off_p = off_sm + round_up(n_c, 128);
    uint64_t off_i = off_p + 3 * plane;
    uint64_t off_e = off_i + round_up(8 * ceil_div(n_c, IDX_SPAN), 128);
    uint64_t k = 0;
    for (uint64_t j = 0; j < n_c; j++) {
        uint16_t h = xc[j];
        if (j % IDX_SPAN == 0) put_u64(o + off_i + 8 * (j / IDX_SPAN), k);
        unsigned E = bf16_exp(h);
        unsigned code = code_of(E, E0);
        o[off_sm + j] = bf16_sm(h);
        for (unsigned p = 0; p < 3; p++)
            if ((code >> p) & 1u) o[off_p + p * plane + j / 8] |= (uint8_t)(1u << (j % 8));
        if (code == 0) o[off_e + k++] = (uint8_t)E;
    }
    *size = bytes;
    return 0;
}

int orc_code3_encode(const uint16_t* x, uint64_t n, uint32_t W, uint32_t E0,
                     uint8_t* out, uint64_t slot_bytes, uint64_t* sizes)
{
    if (W == 0 || E0 > 249) return -1;
    uint64_t L = orc_shard_len(n, W);
    for (uint32_t c = 0; c < W; c++) {
        int rc = orc_code3_encode_chunk(x + (uint64_t)c * L, n, W, c, E0,
                                        out + (uint64_t)c * slot_bytes, slot_bytes, sizes + c);
        if (rc) return rc;
    }
    return 0;
}

/* One chunk c of an n-value tensor split W ways, at p with avail bytes,
 * decoded to out_c (n_c values).  Returns the status bits of that chunk. */
uint32_t orc_code3_decode_chunk(const uint8_t* p, uint64_t avail, uint64_t n, uint32_t W,
                                uint32_t c, uint16_t* out_c)
{
    uint32_t status = 0;
    uint64_t n_c = orc_shard_count(n, W, c);
    if (avail < 128) return ORC_BAD_SIZE;
    if (!(p[0] == 'E' && p[1] == 'Z' && p[2] == 'C' && p[3] == '3') || p[4] != 2
        || p[5] > 249 || get_u64(p + 8) != n_c || get_u32(p + 32) != c
        || get_u32(p + 36) != W)
        return ORC_BAD_HEADER;
    unsigned E0 = p[5];
    uint64_t n_esc = get_u64(p + 16);
    if (n_esc > n_c) return ORC_BAD_COUNT;
    uint64_t bytes = get_u64(p + 24);
    if (bytes != orc_code3_chunk_bytes(n_c, n_esc) || bytes > avail) return ORC_BAD_SIZE;
    uint64_t plane = round_up(ceil_div(n_c, 8), 128);
    const uint8_t* sm = p + 128;
    const uint8_t* pl = sm + round_up(n_c, 128);
    const uint8_t* idx = pl + 3 * plane;
    const uint8_t* esc = idx + round_up(8 * ceil_div(n_c, IDX_SPAN), 128);
    uint64_t k = 0;
    for (uint64_t j = 0; j < n_c; j++) {
        /* the index must hold the escape count of the values before */
        if (j % IDX_SPAN == 0 && get_u64(idx + 8 * (j / IDX_SPAN)) != k)
            status |= ORC_BAD_COUNT;
        unsigned code = 0;
        for (unsigned b = 0; b < 3; b++)
            code |= ((pl[b * plane + j / 8] >> (j % 8)) & 1u) << b;
        unsigned E;
        if (code) {
            E = E0 + code - 1;
        } else if (k < n_esc) {
            E = esc[k++];
        } else {
            status |= ORC_BAD_COUNT;
            E = 0;
        }
        out_c[j] = bf16_merge(sm[j], (uint8_t)E);
    }
    if (k != n_esc) status |= ORC_BAD_COUNT;
    return status;
}

uint32_t orc_code3_decode(const uint8_t* in, const uint64_t* offsets,
                          uint64_t n, uint32_t W, uint16_t* out)
{
    uint32_t status = 0;
    uint64_t L = orc_shard_len(n, W);
    for (uint32_t c = 0; c < W; c++) {
        if (offsets[c + 1] < offsets[c]) { status |= ORC_BAD_SIZE; continue; }
        status |= orc_code3_decode_chunk(in + offsets[c], offsets[c + 1] - offsets[c], n, W, c,
                                         out + (uint64_t)c * L);
    }
    return status;
}

/* ------------------------------------------------------------------ reuse */

static uint64_t reuse_idx_bytes(uint64_t n_s, int coded)
{
    return round_up((coded ? 16 : 8) * ceil_div(n_s, IDX_SPAN), 16);
}

uint64_t orc_reuse_bytes(uint64_t n_s, uint32_t B, uint64_t m, int coded,
                         uint64_t n_esc)
{
    uint64_t nb = ceil_div(n_s, B);
    uint64_t exp_bytes = coded ? 3 * round_up(ceil_div(m, 8), 16) + n_esc : m;
    return round_up(64 + round_up(ceil_div(nb, 8), 16) + round_up(n_s, 16)
                    + reuse_idx_bytes(n_s, coded) + exp_bytes, 128);
}

uint64_t orc_reuse_slot_bytes(uint64_t n, uint32_t W, uint32_t B, int coded)
{
    uint64_t L = orc_shard_len(n, W);
    return orc_reuse_bytes(L, B, L, coded, coded ? L : 0);
}

int orc_reuse_encode(const uint16_t* shard, uint64_t n_s, uint32_t B,
                     uint32_t shard_index, uint8_t* send_cache, int cold,
                     int coded, orc_stats* st, uint8_t* out, uint64_t cap,
                     uint64_t* size)
{
    return orc_reuse_encode_mode(shard, n_s, B, shard_index, send_cache, cold, coded, 0, st, out,
                                 cap, size);
}

/* The payload of one shard given its changed-block flags (CIERA exponent
 * reuse; the coded variant codes the changed exponents with ZipCCL's 3-bit
 * code, window from the shard's statistics). */
static int reuse_payload(const uint16_t* shard, uint64_t n_s, uint32_t B, uint32_t shard_index,
                         const uint8_t* changed, int cold, int coded, int window_mode,
                         orc_stats* st, uint8_t* out, uint64_t cap, uint64_t* size)
{
    uint64_t nb = ceil_div(n_s, B);
    uint8_t* exps = (uint8_t*)malloc(n_s ? n_s : 1);
    if (!exps) return -3;
    uint64_t n_changed = 0, m = 0;
    for (uint64_t k = 0; k < nb; k++) {
        if (!changed[k]) continue;
        uint64_t a = k * B, b = (k + 1) * B < n_s ? (k + 1) * B : n_s;
        n_changed++;
        for (uint64_t i = a; i < b; i++) exps[m++] = bf16_exp(shard[i]);
    }
    uint32_t E0 = 0;
    uint64_t n_esc = 0;
    if (coded) {
        /* the code window comes from this shard's sigma [ZIP 3.1] */
        orc_stats local;
        orc_stats* s = st ? st : &local;
        orc_stats_compute_mode(shard, n_s, window_mode, s);
        E0 = s->E0;
        for (uint64_t j = 0; j < m; j++)
            if (code_of(exps[j], E0) == 0) n_esc++;
    }
    uint64_t total = orc_reuse_bytes(n_s, B, m, coded, n_esc);
    if (total > cap) { free(exps); return -2; }
    memset(out, 0, total);
    out[0] = 'E'; out[1] = 'Z'; out[2] = 'R'; out[3] = 'U';
    out[4] = 2;
    out[5] = (uint8_t)((coded ? 1 : 0) | (cold ? 2 : 0));
    out[6] = (uint8_t)E0;
    put_u32(out + 8, B);
    put_u32(out + 12, shard_index);
    put_u64(out + 16, n_s);
    put_u64(out + 24, n_changed);
    put_u64(out + 32, m);
    put_u64(out + 40, n_esc);
    put_u64(out + 48, total);
    uint64_t off_bm = 64;
    uint64_t off_sm = off_bm + round_up(ceil_div(nb, 8), 16);
    uint64_t off_i = off_sm + round_up(n_s, 16);
    uint64_t off_x = off_i + reuse_idx_bytes(n_s, coded);
    for (uint64_t k = 0; k < nb; k++)
        if (changed[k]) out[off_bm + k / 8] |= (uint8_t)(1u << (k % 8));
    for (uint64_t i = 0; i < n_s; i++) out[off_sm + i] = bf16_sm(shard[i]);
    /* index: changed blocks (and escapes among their exponents) before
     * each multiple of 8192 values */
    {
        uint64_t k = 0, before = 0, q = 0, esc_before = 0;
        for (uint64_t t = 0; t < ceil_div(n_s, IDX_SPAN); t++) {
            /* walk the blocks that lie before value t*8192 */
            for (; k < t * IDX_SPAN / B; k++) {
                if (!changed[k]) continue;
                before++;
                uint64_t a = k * B, b = (k + 1) * B < n_s ? (k + 1) * B : n_s;
                for (uint64_t i = a; i < b; i++, q++)
                    if (coded && code_of(exps[q], E0) == 0) esc_before++;
            }
            put_u64(out + off_i + (coded ? 16 : 8) * t, before);
            if (coded) put_u64(out + off_i + 16 * t + 8, esc_before);
        }
    }
    if (!coded) {
        for (uint64_t j = 0; j < m; j++) out[off_x + j] = exps[j];
    } else {
        uint64_t plane = round_up(ceil_div(m, 8), 16);
        uint64_t off_e = off_x + 3 * plane, k = 0;
        for (uint64_t j = 0; j < m; j++) {
            unsigned code = code_of(exps[j], E0);
            for (unsigned p = 0; p < 3; p++)
                if ((code >> p) & 1u) out[off_x + p * plane + j / 8] |= (uint8_t)(1u << (j % 8));
            if (code == 0) out[off_e + k++] = exps[j];
        }
    }
    *size = total;
    free(exps);
    return 0;
}

int orc_reuse_encode_mode(const uint16_t* shard, uint64_t n_s, uint32_t B,
                          uint32_t shard_index, uint8_t* send_cache, int cold,
                          int coded, int window_mode, orc_stats* st, uint8_t* out,
                          uint64_t cap, uint64_t* size)
{
    if (B == 0) return -1;
    uint64_t nb = ceil_div(n_s, B);
    uint8_t* changed = (uint8_t*)calloc(nb ? nb : 1, 1);
    if (!changed) return -3;
    /* changed_k = cold or some exponent differs from the sender's cache */
    for (uint64_t k = 0; k < nb; k++) {
        uint64_t a = k * B, b = (k + 1) * B < n_s ? (k + 1) * B : n_s;
        int ch = cold;
        for (uint64_t i = a; i < b; i++)
            if (bf16_exp(shard[i]) != send_cache[i]) ch = 1;
        changed[k] = (uint8_t)ch;
    }
    int rc = reuse_payload(shard, n_s, B, shard_index, changed, cold, coded, window_mode, st, out,
                           cap, size);
    if (rc == 0) {
        /* the sender's cache now holds this iteration's exponents */
        for (uint64_t k = 0; k < nb; k++) {
            if (!changed[k]) continue;
            uint64_t a = k * B, b = (k + 1) * B < n_s ? (k + 1) * B : n_s;
            for (uint64_t i = a; i < b; i++) send_cache[i] = bf16_exp(shard[i]);
        }
    }
    free(changed);
    return rc;
}

/* ---- hash-based change detection (CIERA: HashCache, two independent
 * 64-bit SplitMix64 hashes per block) ----------------------------------- */

/* The SplitMix64 generator (Steele, Lea and Flood): the state advances by
 * the golden gamma and each output is the state passed through the mixing
 * function below. */
#define SM64_GAMMA 0x9E3779B97F4A7C15ull
static uint64_t sm64_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t orc_splitmix64_next(uint64_t* state)
{
    *state += SM64_GAMMA;
    return sm64_mix(*state);
}

/* Hash s (0 or 1) of block k: word i is the 8 exponent bytes of values
 * kB + 8i .. kB + 8i + 7 (little-endian, 0 for values past the shard);
 * term_i = mix(word_i + seed_s + (i + 1) * gamma), one SplitMix64 output per
 * word; the hash is mix(sum of the B/8 terms mod 2^64).  A change in any
 * single word changes its term (mix is a bijection) and so the sum. */
static const uint64_t kHashSeed[2] = {0ull, 0x5851F42D4C957F2Dull};

uint64_t orc_block_hash(const uint16_t* shard, uint64_t n_s, uint32_t B, uint64_t k, int s)
{
    uint64_t sum = 0;
    for (uint32_t i = 0; i < B / 8; i++) {
        uint64_t w = 0;
        for (unsigned j = 0; j < 8; j++) {
            uint64_t v = k * B + 8ull * i + j;
            if (v < n_s) w |= (uint64_t)bf16_exp(shard[v]) << (8 * j);
        }
        sum += sm64_mix(w + kHashSeed[s] + (uint64_t)(i + 1) * SM64_GAMMA);
    }
    return sm64_mix(sum);
}

int orc_reuse_encode_hash(const uint16_t* shard, uint64_t n_s, uint32_t B,
                          uint32_t shard_index, uint64_t* hash_cache, int cold,
                          int coded, int window_mode, orc_stats* st, uint8_t* out,
                          uint64_t cap, uint64_t* size)
{
    if (B < 8 || (B & 7)) return -1;
    uint64_t nb = ceil_div(n_s, B);
    uint8_t* changed = (uint8_t*)calloc(nb ? nb : 1, 1);
    uint64_t* h = (uint64_t*)malloc(2 * (nb ? nb : 1) * sizeof(uint64_t));
    if (!changed || !h) { free(changed); free(h); return -3; }
    /* changed_k = cold or the block's hash pair differs from HashCache[k] */
    for (uint64_t k = 0; k < nb; k++) {
        h[2 * k] = orc_block_hash(shard, n_s, B, k, 0);
        h[2 * k + 1] = orc_block_hash(shard, n_s, B, k, 1);
        changed[k] = (uint8_t)(cold || h[2 * k] != hash_cache[2 * k] || h[2 * k + 1] != hash_cache[2 * k + 1]);
    }
    int rc = reuse_payload(shard, n_s, B, shard_index, changed, cold, coded, window_mode, st, out,
                           cap, size);
    if (rc == 0)
        for (uint64_t k = 0; k < nb; k++)
            if (changed[k]) { hash_cache[2 * k] = h[2 * k]; hash_cache[2 * k + 1] = h[2 * k + 1]; }
    free(changed);
    free(h);
    return rc;
}

uint32_t orc_reuse_decode(const uint8_t* p, uint64_t avail, uint64_t n_s,
                          uint32_t B, uint32_t shard_index,
                          uint8_t* recv_cache, uint16_t* out)
{
    if (avail < 64) return ORC_BAD_SIZE;
    if (!(p[0] == 'E' && p[1] == 'Z' && p[2] == 'R' && p[3] == 'U') || p[4] != 2
        || (p[5] & ~3u) != 0 || p[7] != 0 || get_u32(p + 8) != B
        || get_u32(p + 12) != shard_index || get_u64(p + 16) != n_s)
        return ORC_BAD_HEADER;
    int coded = p[5] & 1;
    unsigned E0 = p[6];
    uint64_t n_changed = get_u64(p + 24), m = get_u64(p + 32);
    uint64_t n_esc = get_u64(p + 40), total = get_u64(p + 48);
    if (coded ? E0 > 249 : (E0 != 0 || n_esc != 0)) return ORC_BAD_HEADER;
    uint64_t nb = ceil_div(n_s, B);
    if (n_changed > nb || m > n_s || n_esc > m) return ORC_BAD_COUNT;
    if (total != orc_reuse_bytes(n_s, B, m, coded, n_esc) || total > avail)
        return ORC_BAD_SIZE;
    uint64_t off_bm = 64;
    uint64_t off_sm = off_bm + round_up(ceil_div(nb, 8), 16);
    uint64_t off_i = off_sm + round_up(n_s, 16);
    uint64_t off_x = off_i + reuse_idx_bytes(n_s, coded);
    const uint8_t* bm = p + off_bm;
    const uint8_t* sm = p + off_sm;
    const uint8_t* idx = p + off_i;
    const uint64_t stride = coded ? 16 : 8;
    /* the bitmap must agree with the declared counts before anything is
     * written to the receiver's cache */
    uint64_t cnt = 0, len = 0;
    for (uint64_t k = 0; k < nb; k++) {
        if ((bm[k / 8] >> (k % 8)) & 1u) {
            uint64_t a = k * B, b = (k + 1) * B < n_s ? (k + 1) * B : n_s;
            cnt++;
            len += b - a;
        }
    }
    if (cnt != n_changed || len != m) return ORC_BAD_COUNT;
    uint32_t status = 0;
    uint64_t plane = round_up(ceil_div(m, 8), 16);
    const uint8_t* esc = p + off_x + 3 * plane;
    uint64_t j = 0, k_esc = 0, blocks_before = 0;
    for (uint64_t k = 0; k < nb; k++) {
        uint64_t a = k * B, b = (k + 1) * B < n_s ? (k + 1) * B : n_s;
        int ch = (bm[k / 8] >> (k % 8)) & 1u;
        /* the index must hold the changed blocks (and escapes) before */
        if (a % IDX_SPAN == 0) {
            const uint8_t* e = idx + stride * (a / IDX_SPAN);
            if (get_u64(e) != blocks_before || (coded && get_u64(e + 8) != k_esc))
                status |= ORC_BAD_COUNT;
        }
        blocks_before += (uint64_t)ch;
        for (uint64_t i = a; i < b; i++) {
            if (ch) {
                unsigned E;
                if (!coded) {
                    E = p[off_x + j];
                } else {
                    unsigned code = 0;
                    for (unsigned q = 0; q < 3; q++)
                        code |= ((p[off_x + q * plane + j / 8] >> (j % 8)) & 1u) << q;
                    if (code) E = E0 + code - 1;
                    else if (k_esc < n_esc) E = esc[k_esc++];
                    else { status |= ORC_BAD_COUNT; E = 0; }
                }
                j++;
                recv_cache[i] = (uint8_t)E;   /* ExpCache takes the new block */
            }
            out[i] = bf16_merge(sm[i], recv_cache[i]);
        }
    }
    if (coded && k_esc != n_esc) status |= ORC_BAD_COUNT;
    return status;
}

uint32_t orc_gather_decode_reuse(const uint8_t* recv, const uint64_t* offsets,
                                 uint64_t n, uint32_t W, uint32_t B,
                                 uint8_t* recv_cache, uint16_t* out)
{
    uint32_t status = 0;
    uint64_t L = orc_shard_len(n, W);
    for (uint32_t r = 0; r < W; r++) {
        uint64_t n_r = orc_shard_count(n, W, r);
        if (offsets[r + 1] < offsets[r]) { status |= ORC_BAD_SIZE; continue; }
        status |= orc_reuse_decode(recv + offsets[r], offsets[r + 1] - offsets[r],
                                   n_r, B, r, recv_cache + (uint64_t)r * L,
                                   out + (uint64_t)r * L);
    }
    return status;
}

/* ------------------------------------------------------------------ FP8 */
/* The 3-bit exponent code applied to FP8 [ZIP 3.3 last paragraph: "FP8 E5M2
 * coded to 3 bits gives e = 0.75, E4M3 gives e ~ 0.88"].  Formats as in the
 * OCP 8-bit floating-point specification: E5M2 (bias 15, infinities and NaN
 * at exponent field 31) and E4M3 (bias 7, no infinities, NaN only at
 * S.1111.111).  A value keeps its sign and mantissa bits raw (1+m bits, as
 * bit-planes); its exponent field becomes the 3-bit code of the window
 * E0..E0+6 or escapes to the raw field.  The window follows the same Gaussian
 * model as for BF16 (the 7-binade argument does not depend on the format):
 * E0 = bias + x0, clamped to 0 .. (2^e - 1) - 6. */

typedef struct { unsigned ebits, mbits, bias; } fp8_fmt;

static int fp8_format(int fmt, fp8_fmt* f)
{
    if (fmt == ORC_FP8_E5M2) { f->ebits = 5; f->mbits = 2; f->bias = 15; return 0; }
    if (fmt == ORC_FP8_E4M3) { f->ebits = 4; f->mbits = 3; f->bias = 7; return 0; }
    return -1;
}

static unsigned fp8_exp(const fp8_fmt* f, uint8_t b) { return (b >> f->mbits) & ((1u << f->ebits) - 1u); }
static unsigned fp8_man(const fp8_fmt* f, uint8_t b) { return b & ((1u << f->mbits) - 1u); }
static unsigned fp8_sm(const fp8_fmt* f, uint8_t b) { return ((b >> 7) << f->mbits) | fp8_man(f, b); }
static uint8_t fp8_merge(const fp8_fmt* f, unsigned sm, unsigned e)
{
    return (uint8_t)(((sm >> f->mbits) << 7) | (e << f->mbits) | (sm & ((1u << f->mbits) - 1u)));
}
static int fp8_finite(const fp8_fmt* f, uint8_t b)
{
    unsigned emax = (1u << f->ebits) - 1u;
    if (f->ebits == 5) return fp8_exp(f, b) != emax;                          /* E5M2: Inf / NaN */
    return !(fp8_exp(f, b) == emax && fp8_man(f, b) == (1u << f->mbits) - 1u);  /* E4M3: NaN only */
}

int orc_fp8_stats(const uint8_t* x, uint64_t n, int fmt, int window_mode, orc_fp8_stats_t* st)
{
    fp8_fmt f;
    if (fp8_format(fmt, &f)) return -1;
    memset(st, 0, sizeof(*st));
    st->n = n;
    const unsigned nbins = 1u << f.ebits, emax0 = nbins - 1u - 6u;
    uint64_t cnt[256];
    memset(cnt, 0, sizeof(cnt));
    for (uint64_t i = 0; i < n; i++) {
        cnt[x[i]]++;
        st->hist[fp8_exp(&f, x[i])]++;
    }
    /* v * 2^U = +-M * 2^(max(E,1) - 1), M = E ? 2^m + man : man,
     * U = bias + m - 1: exact big sums of the 256 patterns, rounded once */
    big_t P, Q, R;
    memset(&P, 0, sizeof(P));
    memset(&Q, 0, sizeof(Q));
    memset(&R, 0, sizeof(R));
    for (unsigned b = 0; b < 256; b++) {
        if (!cnt[b] || !fp8_finite(&f, (uint8_t)b)) continue;
        st->n_finite += cnt[b];
        unsigned E = fp8_exp(&f, (uint8_t)b);
        uint64_t M = (E ? (1u << f.mbits) : 0u) + fp8_man(&f, (uint8_t)b);
        unsigned sh = (E ? E : 1u) - 1u;
        if (M == 0) continue;
        if (b & 0x80u) big_add_shifted(&Q, cnt[b] * M, sh);
        else big_add_shifted(&P, cnt[b] * M, sh);
        big_add_shifted(&R, cnt[b] * M * M, 2 * sh);
    }
    int U = (int)(f.bias + f.mbits) - 1;
    if (big_cmp(&P, &Q) >= 0) {
        big_sub(&P, &Q);
        st->s1 = big_round(&P, -U);
    } else {
        big_sub(&Q, &P);
        st->s1 = -big_round(&Q, -U);
    }
    st->s2 = big_round(&R, -2 * U);
    st->K = orc_window_K();
    st->rule = 1;
    if (st->n_finite >= 2) {
        double N = (double)st->n_finite;
        double var = (st->s2 - st->s1 * (st->s1 / N)) / (N - 1.0);
        st->var = var;
        if (var > 0 && isfinite(var)) {
            st->sigma = sqrt(var);
            if (window_mode == 0) {
                /* the integer nearest x_opt, ties up: the largest k with
                 * var >= K 2^(2k-1), as a field value bias + k */
                uint32_t E0 = 0;
                for (unsigned e = 1; e <= emax0; e++) {
                    int k = (int)e - (int)f.bias;
                    if (var >= ldexp(st->K, 2 * k - 1)) E0 = e;
                }
                st->E0 = E0;
                st->rule = 0;
            }
        }
    }
    if (st->rule == 1) {
        uint64_t best = 0;
        uint32_t best_b = 0;
        for (uint32_t b = 0; b <= emax0; b++) {
            uint64_t c = 0;
            for (uint32_t E = b; E <= b + 6; E++) c += st->hist[E];
            if (c > best) { best = c; best_b = b; }
        }
        st->E0 = best_b;
    }
    uint64_t in_window = 0;
    for (uint32_t E = st->E0; E <= st->E0 + 6; E++) in_window += st->hist[E];
    st->n_escape = n - in_window;
    return 0;
}

/* chunk: header 128 | 1+m sign/mantissa planes | 3 code planes | index (u64
 * escapes before each 8192 values) | escapes (raw exponent fields, value
 * order); every section padded to 128 bytes, plane p holding bit p of the
 * field for value j at bit j&7 of byte j>>3. */
uint64_t orc_fp8_chunk_bytes(uint64_t n_c, uint64_t n_esc, int fmt)
{
    fp8_fmt f;
    if (fp8_format(fmt, &f)) return 0;
    uint64_t plane = round_up(ceil_div(n_c, 8), 128);
    return 128 + (1 + f.mbits + 3) * plane + round_up(8 * ceil_div(n_c, IDX_SPAN), 128) + round_up(n_esc, 128);
}

int orc_fp8_encode(const uint8_t* x, uint64_t n, uint32_t W, int fmt, uint32_t E0,
                   uint8_t* out, uint64_t slot_bytes, uint64_t* sizes)
{
    fp8_fmt f;
    if (fp8_format(fmt, &f) || W == 0) return -1;
    const unsigned nsm = 1 + f.mbits, emax0 = (1u << f.ebits) - 1u - 6u;
    if (E0 > emax0) return -1;
    uint64_t L = orc_shard_len(n, W);
    for (uint32_t c = 0; c < W; c++) {
        uint64_t n_c = orc_shard_count(n, W, c);
        const uint8_t* xc = x + (uint64_t)c * L;
        uint64_t n_esc = 0;
        for (uint64_t j = 0; j < n_c; j++) {
            unsigned E = fp8_exp(&f, xc[j]);
            if (!(E >= E0 && E <= E0 + 6)) n_esc++;
        }
        uint64_t bytes = orc_fp8_chunk_bytes(n_c, n_esc, fmt);
        if (bytes > slot_bytes) return -2;
        uint8_t* o = out + (uint64_t)c * slot_bytes;
        memset(o, 0, bytes);
        o[0] = 'E'; o[1] = 'Z'; o[2] = 'F'; o[3] = '8';
        o[4] = 1;
        o[5] = (uint8_t)fmt;
        o[6] = (uint8_t)E0;
        put_u64(o + 8, n_c);
        put_u64(o + 16, n_esc);
        put_u64(o + 24, bytes);
        put_u32(o + 32, c);
        put_u32(o + 36, W);
        uint64_t plane = round_up(ceil_div(n_c, 8), 128);
        uint8_t* pl = o + 128;
        uint8_t* idx = pl + (nsm + 3) * plane;
        uint8_t* esc = idx + round_up(8 * ceil_div(n_c, IDX_SPAN), 128);
        uint64_t k = 0;
        for (uint64_t j = 0; j < n_c; j++) {
            if (j % IDX_SPAN == 0) put_u64(idx + 8 * (j / IDX_SPAN), k);
            unsigned sm = fp8_sm(&f, xc[j]), E = fp8_exp(&f, xc[j]);
            unsigned code = (E >= E0 && E <= E0 + 6) ? E - E0 + 1 : 0;
            for (unsigned p = 0; p < nsm; p++)
                if ((sm >> p) & 1u) pl[p * plane + j / 8] |= (uint8_t)(1u << (j % 8));
            for (unsigned p = 0; p < 3; p++)
                if ((code >> p) & 1u) pl[(nsm + p) * plane + j / 8] |= (uint8_t)(1u << (j % 8));
            if (code == 0) esc[k++] = (uint8_t)E;
        }
        sizes[c] = bytes;
    }
    return 0;
}

uint32_t orc_fp8_decode(const uint8_t* in, const uint64_t* offsets, uint64_t n, uint32_t W,
                        int fmt, uint8_t* out)
{
    fp8_fmt f;
    if (fp8_format(fmt, &f) || W == 0) return ORC_BAD_HEADER;
    const unsigned nsm = 1 + f.mbits, emax0 = (1u << f.ebits) - 1u - 6u;
    uint32_t status = 0;
    uint64_t L = orc_shard_len(n, W);
    for (uint32_t c = 0; c < W; c++) {
        uint64_t n_c = orc_shard_count(n, W, c);
        if (offsets[c + 1] < offsets[c]) { status |= ORC_BAD_SIZE; continue; }
        uint64_t avail = offsets[c + 1] - offsets[c];
        if (avail < 128) { status |= ORC_BAD_SIZE; continue; }
        const uint8_t* p = in + offsets[c];
        if (!(p[0] == 'E' && p[1] == 'Z' && p[2] == 'F' && p[3] == '8') || p[4] != 1 || p[5] != (uint8_t)fmt
            || p[6] > emax0 || get_u64(p + 8) != n_c || get_u32(p + 32) != c || get_u32(p + 36) != W) {
            status |= ORC_BAD_HEADER;
            continue;
        }
        unsigned E0 = p[6];
        uint64_t n_esc = get_u64(p + 16);
        if (n_esc > n_c) { status |= ORC_BAD_COUNT; continue; }
        uint64_t bytes = get_u64(p + 24);
        if (bytes != orc_fp8_chunk_bytes(n_c, n_esc, fmt) || bytes > avail) { status |= ORC_BAD_SIZE; continue; }
        uint64_t plane = round_up(ceil_div(n_c, 8), 128);
        const uint8_t* pl = p + 128;
        const uint8_t* idx = pl + (nsm + 3) * plane;
        const uint8_t* esc = idx + round_up(8 * ceil_div(n_c, IDX_SPAN), 128);
        uint8_t* oc = out + (uint64_t)c * L;
        uint64_t k = 0;
        for (uint64_t j = 0; j < n_c; j++) {
            if (j % IDX_SPAN == 0 && get_u64(idx + 8 * (j / IDX_SPAN)) != k) status |= ORC_BAD_COUNT;
            unsigned sm = 0, code = 0;
            for (unsigned q = 0; q < nsm; q++) sm |= ((pl[q * plane + j / 8] >> (j % 8)) & 1u) << q;
            for (unsigned q = 0; q < 3; q++) code |= ((pl[(nsm + q) * plane + j / 8] >> (j % 8)) & 1u) << q;
            unsigned E;
            if (code) {
                E = E0 + code - 1;
            } else if (k < n_esc) {
                E = esc[k++] & ((1u << f.ebits) - 1u);
            } else {
                status |= ORC_BAD_COUNT;
                E = 0;
            }
            oc[j] = fp8_merge(&f, sm, E);
        }
        if (k != n_esc) status |= ORC_BAD_COUNT;
    }
    return status;
}
