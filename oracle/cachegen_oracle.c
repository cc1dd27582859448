/*
 * cachegen_oracle.c -- plain, slow CPU definition of the CacheGen KV codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no source, header, table or helper with the
 * CUDA library (nor with lmkv_oracle.c); it is built with plain gcc,
 * -ffp-contract=off, single-threaded.
 *
 * What it follows: "LMCache 中的 KV Cache 压缩：CacheGen 编解码原理、配置方式与
 * 源码解析", sections 1 (QuantizationSpec / CacheGenConfig: bins per layer
 * group), 2 (per-layer symmetric quantisation), 3 (per-(layer, channel) CDF
 * from a histogram and cumsum, scaled to 2^16 with an arange ramp), 4
 * (arithmetic coding in batches of at most 256 tokens, a byte stream plus
 * per-stream lengths per batch) and 5 (decoding through the lengths' prefix
 * sums, then t = (t - C) / C * max).
 *
 * The page gives the algorithm in outline; the readings taken here are:
 *  R1 quantisation (section 2): MAX = bins/2 - 1 (integer division); for
 *     every (K/V, layer, token) row, max1 = the largest |x| over the row's
 *     channels (the amax over the last axis of [layers, tokens, channels]);
 *     factor = MAX / max1, y = x * factor, z = y + MAX, q = round(z) to the
 *     nearest integer, ties to even; every step one fp32 operation (the bf16
 *     input widened exactly).  q is clamped to [0, 2*MAX]; a row whose max1
 *     is 0 gets q = MAX.  Inputs are finite.  The clamp is applied to z
 *     before the rounding (the same result for every finite z, the bounds
 *     being integers).  A nonzero max1 below MAX / FLT_MAX (a row of
 *     subnormal values) makes factor infinite: y is then +-inf, clamped to
 *     2*MAX or 0, or NaN for x = 0, taken as 0 (as a maximum with 0 treats
 *     a NaN operand).
 *  R2 CDF (section 3): nsym = 2*MAX + 1 symbols and Lp = nsym + 1 CDF
 *     entries.  Over the n tokens of the chunk, cum[k] = number of tokens
 *     whose symbol is below k (k = 0..nsym); with M = 2^16 - (Lp - 1),
 *     C[k] = round(cum[k] * M / n) + k, the division exact and the rounding
 *     to nearest, ties to even.  So C[0] = 0, C[nsym] = 2^16 and every
 *     symbol has a frequency C[k+1] - C[k] of at least 1.  One CDF per
 *     (K/V, layer, channel) per chunk, shared by the chunk's batches.
 *  R3 coder (section 4): the integer arithmetic coder of Witten, Neal and
 *     Cleary ("Arithmetic coding for data compression", Communications of
 *     the ACM 30(6), 1987) with 32-bit low / high, cumulative frequencies
 *     out of 2^16, bits packed most significant first, the final partial
 *     byte padded with zeros.  One stream per (batch, K/V, layer, channel):
 *     the channel's symbols for the batch's tokens in token order.  The
 *     decoder reads zero bits past the end of a stream.
 *  R4 dequantisation (section 5): y = ((q - MAX) / MAX) * max1, the division
 *     and the product each one fp32 operation, then rounded to bf16 (nearest,
 *     ties to even).
 *  R5 bins (section 1): K uses 32 bins for layers 0-9 and 16 after; V uses 32
 *     bins for layers 0-1 and 16 after; a model with fewer than 10 layers uses
 *     32 bins everywhere.
 *
 * Encoded chunk (one byte blob per chunk of n tokens, L layers, H channels;
 * all integers little-endian):
 *   max1    float32 [2][L][n]                       at 0
 *   cdf     uint16, for each (kv, l) in order, [H][nsym(kv,l) - 1]
 *           holding C[1..nsym-1] (C[0] = 0 and C[nsym] = 2^16 implied)
 *   lengths uint32 [nb][2][L][H], nb = ceil(n / 256), at the next multiple
 *           of 4 bytes
 *   bytes   the streams back to back in (batch, kv, l, channel) order
 * The blob's size is the offset of bytes plus the sum of the lengths.
 *
 * Return codes: 0 / a size on success, -1 invalid arguments, -2 capacity too
 * small, -3 inconsistent blob.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define CG_BATCH 256
#define CG_TOTAL 65536u
#define CG_HALF 0x80000000ull
#define CG_QUARTER 0x40000000ull

/* ---- bf16 <-> fp32 (IEEE binary32 narrowed to 8 significant bits) ---- */

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a finite float to the nearest bf16 (ties to even), saturating to
 * infinity the way IEEE rounding does. */
static uint16_t f32_to_bf16(float v)
{
    double a = fabs((double)v);
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                         /* a = m * 2^e, m in [0.5, 1) */
    if (e < -125) e = -125;               /* subnormal grid: quantum 2^-133 */
    double quantum = ldexp(1.0, e - 8);   /* 8 significant bits */
    double n = floor(a / quantum);
    double frac = a / quantum - n;
    if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
    double r = n * quantum;
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
    float f = (float)r;                   /* exact: r has at most 8 bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* ---- R5: default bins ---- */

/* bins[kv * L + l] for kv = 0 (K), 1 (V). */
void cgo_default_bins(int32_t num_layers, int32_t* bins)
{
    for (int32_t l = 0; l < num_layers; ++l) {
        int all32 = num_layers < 10;
        bins[l] = (all32 || l < 10) ? 32 : 16;
        bins[num_layers + l] = (all32 || l < 2) ? 32 : 16;
    }
}

static int32_t nsym_of(int32_t bins) { return 2 * (bins / 2 - 1) + 1; }

/* ---- R1: quantisation of one (K/V, layer) slice x[n][H] (bf16 bits) ---- */

void cgo_quantize(const uint16_t* x, int32_t n, int32_t H, int32_t bins, uint8_t* sym,
                  float* max1)
{
    int32_t MAX = bins / 2 - 1;
    for (int32_t t = 0; t < n; ++t) {
        const uint16_t* row = x + (int64_t)t * H;
        float m = 0.0f;
        for (int32_t c = 0; c < H; ++c) {
            float a = fabsf(bf16_to_f32(row[c]));
            if (a > m) m = a;
        }
        max1[t] = m;
        volatile float factor = m == 0.0f ? 0.0f : (float)MAX / m;
        for (int32_t c = 0; c < H; ++c) {
            int32_t q = MAX;
            if (m != 0.0f) {
                volatile float y = bf16_to_f32(row[c]) * factor;
                volatile float z = y + (float)MAX;
                /* clamp, then round (default mode: nearest, ties even);
                   fmaxf takes 0 for a NaN z */
                float zc = fminf(fmaxf(z, 0.0f), (float)(2 * MAX));
                q = (int32_t)nearbyintf(zc);
            }
            sym[(int64_t)t * H + c] = (uint8_t)q;
        }
    }
}

/* ---- R2: the CDF of one channel ---- */

/* Symbols sym[t * stride], t < n (n >= 1); writes C[0..nsym]. */
void cgo_cdf(const uint8_t* sym, int32_t n, int64_t stride, int32_t nsym, uint32_t* C)
{
    int64_t count[256];
    for (int k = 0; k < 256; ++k) count[k] = 0;
    for (int32_t t = 0; t < n; ++t) count[sym[(int64_t)t * stride]]++;
    int32_t Lp = nsym + 1;
    uint64_t M = CG_TOTAL - (uint64_t)(Lp - 1);
    uint64_t cum = 0;
    for (int32_t k = 0; k <= nsym; ++k) {
        uint64_t num = cum * M;                 /* cum * M / n, rounded */
        uint64_t q = num / (uint64_t)n, r = num % (uint64_t)n;
        if (2 * r > (uint64_t)n || (2 * r == (uint64_t)n && (q & 1))) q += 1;
        C[k] = (uint32_t)(q + (uint64_t)k);
        if (k < nsym) cum += (uint64_t)count[k];
    }
}

/* ---- R3: the arithmetic coder ---- */

typedef struct {
    uint8_t* out;
    int64_t cap;       /* bytes */
    int64_t nbits;
    int overflow;
} bit_writer;

static void write_bit(bit_writer* w, int bit)
{
    int64_t byte = w->nbits >> 3;
    if (byte >= w->cap) {
        w->overflow = 1;
    } else {
        if ((w->nbits & 7) == 0) w->out[byte] = 0;
        if (bit) w->out[byte] |= (uint8_t)(0x80u >> (w->nbits & 7));
    }
    w->nbits++;
}

/* A decided bit, then the bits_to_follow opposite bits that were held back
 * while the interval straddled the middle. */
static void bit_plus_follow(bit_writer* w, int bit, int64_t* bits_to_follow)
{
    write_bit(w, bit);
    while (*bits_to_follow > 0) {
        write_bit(w, !bit);
        --*bits_to_follow;
    }
}

/* Code the n symbols sym[t * stride] with the CDF C[0..nsym] (C[nsym] =
 * 2^16) into out; returns the byte length, -1 for a symbol >= nsym, or -2
 * when cap is too small. */
int64_t cgo_encode(const uint8_t* sym, int32_t n, int64_t stride, const uint32_t* C,
                   int32_t nsym, uint8_t* out, int64_t cap)
{
    bit_writer w = {out, cap, 0, 0};
    uint64_t low = 0, high = 0xFFFFFFFFull;
    int64_t follow = 0;
    for (int32_t t = 0; t < n; ++t) {
        uint32_t s = sym[(int64_t)t * stride];
        if (s >= (uint32_t)nsym) return -1;
        uint64_t range = high - low + 1;
        high = low + ((range * C[s + 1]) >> 16) - 1;
        low = low + ((range * C[s]) >> 16);
        for (;;) {
            if (high < CG_HALF) {
                bit_plus_follow(&w, 0, &follow);
            } else if (low >= CG_HALF) {
                bit_plus_follow(&w, 1, &follow);
                low -= CG_HALF;
                high -= CG_HALF;
            } else if (low >= CG_QUARTER && high < 3 * CG_QUARTER) {
                follow++;
                low -= CG_QUARTER;
                high -= CG_QUARTER;
            } else {
                break;
            }
            low = 2 * low;
            high = 2 * high + 1;
        }
    }
    /* two more bits pick a point inside the final interval */
    follow++;
    bit_plus_follow(&w, low < CG_QUARTER ? 0 : 1, &follow);
    if (w.overflow) return -2;
    return (w.nbits + 7) >> 3;
}

static int read_bit(const uint8_t* in, int64_t nbytes, int64_t* pos)
{
    int64_t byte = *pos >> 3;
    int bit = byte < nbytes ? (in[byte] >> (7 - (*pos & 7))) & 1 : 0;
    ++*pos;
    return bit;
}

/* Decode n symbols from in[0..nbytes) into sym[t * stride]. */
void cgo_decode(const uint8_t* in, int64_t nbytes, int32_t n, const uint32_t* C, int32_t nsym,
                uint8_t* sym, int64_t stride)
{
    uint64_t low = 0, high = 0xFFFFFFFFull, value = 0;
    int64_t pos = 0;
    for (int i = 0; i < 32; ++i) value = 2 * value + (uint64_t)read_bit(in, nbytes, &pos);
    for (int32_t t = 0; t < n; ++t) {
        uint64_t range = high - low + 1;
        uint64_t cum = ((value - low + 1) * CG_TOTAL - 1) / range;
        int32_t s = 0;
        while (s + 1 < nsym && C[s + 1] <= cum) ++s;
        sym[(int64_t)t * stride] = (uint8_t)s;
        high = low + ((range * C[s + 1]) >> 16) - 1;
        low = low + ((range * C[s]) >> 16);
        for (;;) {
            if (high < CG_HALF) {
                /* the top bit is 0 for low, high and value alike */
            } else if (low >= CG_HALF) {
                value -= CG_HALF;
                low -= CG_HALF;
                high -= CG_HALF;
            } else if (low >= CG_QUARTER && high < 3 * CG_QUARTER) {
                value -= CG_QUARTER;
                low -= CG_QUARTER;
                high -= CG_QUARTER;
            } else {
                break;
            }
            low = 2 * low;
            high = 2 * high + 1;
            value = 2 * value + (uint64_t)read_bit(in, nbytes, &pos);
        }
    }
}

/* ---- R4: dequantisation of one (K/V, layer) slice ---- */

void cgo_dequantize(const uint8_t* sym, const float* max1, int32_t n, int32_t H, int32_t bins,
                    uint16_t* out)
{
    int32_t MAX = bins / 2 - 1;
    for (int32_t t = 0; t < n; ++t)
        for (int32_t c = 0; c < H; ++c) {
            volatile float a = (float)((int32_t)sym[(int64_t)t * H + c] - MAX) / (float)MAX;
            volatile float y = a * max1[t];
            out[(int64_t)t * H + c] = f32_to_bf16(y);
        }
}

/* ---- the encoded chunk ---- */

/* off[0] max1, off[1] cdf, off[2] lengths, off[3] bytes, off[4] an upper
 * bound on the blob size (a stream of nt symbols takes at most 18 * nt + 2
 * bits: every symbol leaves an interval of at least 2^14 out of at most 2^32
 * and each bit doubles it).  Returns 0 or -1. */
int cgo_layout(int32_t L, int32_t n, int32_t H, const int32_t* bins, int64_t* off)
{
    if (L <= 0 || n <= 0 || H <= 0) return -1;
    int64_t cdf_entries = 0;
    for (int32_t i = 0; i < 2 * L; ++i) {
        if (bins[i] < 4 || bins[i] > 32) return -1;
        cdf_entries += (int64_t)H * (nsym_of(bins[i]) - 1);
    }
    int64_t nb = ((int64_t)n + CG_BATCH - 1) / CG_BATCH;
    off[0] = 0;
    off[1] = (int64_t)4 * 2 * L * n;
    off[2] = (off[1] + 2 * cdf_entries + 3) / 4 * 4;
    off[3] = off[2] + (int64_t)4 * nb * 2 * L * H;
    int64_t bound = off[3];
    for (int64_t b = 0; b < nb; ++b) {
        int64_t nt = (b + 1) * CG_BATCH <= n ? CG_BATCH : n - b * CG_BATCH;
        bound += (int64_t)2 * L * H * ((18 * nt + 2 + 7) / 8);
    }
    off[4] = bound;
    return 0;
}

static void put_u32(uint8_t* p, uint32_t v)
{
    for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}

static uint32_t get_u32(const uint8_t* p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/* Encode chunk[2][L][n][H] (bf16 bits) into blob; returns the blob size, -1
 * for invalid arguments or -2 when cap is too small. */
int64_t cgo_encode_chunk(const uint16_t* chunk, int32_t L, int32_t n, int32_t H,
                         const int32_t* bins, uint8_t* blob, int64_t cap)
{
    int64_t off[5];
    if (cgo_layout(L, n, H, bins, off) != 0) return -1;
    if (cap < off[3]) return -2;
    memset(blob, 0, (size_t)off[3]);
    uint8_t* sym = (uint8_t*)malloc((size_t)2 * L * n * H);
    uint32_t* cdf = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)2 * L * H * 33);
    float* max1 = (float*)malloc(sizeof(float) * (size_t)n);
    if (sym == NULL || cdf == NULL || max1 == NULL) {
        free(sym); free(cdf); free(max1);
        return -1;
    }
    /* quantise every (kv, l) slice, then one CDF per (kv, l, channel) */
    int64_t cdf_pos = off[1];
    for (int32_t s = 0; s < 2 * L; ++s) {
        int32_t nsym = nsym_of(bins[s]);
        cgo_quantize(chunk + (int64_t)s * n * H, n, H, bins[s], sym + (int64_t)s * n * H, max1);
        for (int32_t t = 0; t < n; ++t) memcpy(blob + 4 * ((int64_t)s * n + t), &max1[t], 4);
        for (int32_t c = 0; c < H; ++c) {
            uint32_t* C = cdf + ((int64_t)s * H + c) * 33;
            cgo_cdf(sym + (int64_t)s * n * H + c, n, H, nsym, C);
            for (int32_t k = 1; k < nsym; ++k, cdf_pos += 2) {
                blob[cdf_pos] = (uint8_t)C[k];
                blob[cdf_pos + 1] = (uint8_t)(C[k] >> 8);
            }
        }
    }
    /* one stream per (batch, kv, l, channel), in that order */
    int64_t pos = off[3], li = off[2];
    int64_t rc = 0;
    for (int32_t b0 = 0; b0 < n && rc == 0; b0 += CG_BATCH) {
        int32_t nt = n - b0 < CG_BATCH ? n - b0 : CG_BATCH;
        for (int32_t s = 0; s < 2 * L && rc == 0; ++s)
            for (int32_t c = 0; c < H; ++c, li += 4) {
                const uint8_t* col = sym + ((int64_t)s * n + b0) * H + c;
                int64_t len = cgo_encode(col, nt, H, cdf + ((int64_t)s * H + c) * 33,
                                         nsym_of(bins[s]), blob + pos, cap - pos);
                if (len < 0) { rc = -2; break; }
                put_u32(blob + li, (uint32_t)len);
                pos += len;
            }
    }
    free(sym); free(cdf); free(max1);
    return rc != 0 ? rc : pos;
}

/* Decode blob[0..size) into chunk[2][L][n][H] (bf16 bits); returns 0, -1 or
 * -3 when the lengths do not add up to size. */
int cgo_decode_chunk(const uint8_t* blob, int64_t size, int32_t L, int32_t n, int32_t H,
                     const int32_t* bins, uint16_t* chunk)
{
    int64_t off[5];
    if (cgo_layout(L, n, H, bins, off) != 0) return -1;
    if (size < off[3]) return -3;
    int64_t nb = ((int64_t)n + CG_BATCH - 1) / CG_BATCH;
    int64_t nstreams = nb * 2 * L * H, total = off[3];
    for (int64_t i = 0; i < nstreams; ++i) total += get_u32(blob + off[2] + 4 * i);
    if (total != size) return -3;
    uint8_t* sym = (uint8_t*)malloc((size_t)n * H);
    float* max1 = (float*)malloc(sizeof(float) * (size_t)n);
    int64_t* start = (int64_t*)malloc(sizeof(int64_t) * (size_t)nstreams);
    if (sym == NULL || max1 == NULL || start == NULL) {
        free(sym); free(max1); free(start);
        return -1;
    }
    /* stream i starts after the prefix sum of the lengths before it */
    start[0] = off[3];
    for (int64_t i = 1; i < nstreams; ++i) start[i] = start[i - 1] + get_u32(blob + off[2] + 4 * (i - 1));
    int64_t cdf_pos = off[1];
    for (int32_t s = 0; s < 2 * L; ++s) {
        int32_t nsym = nsym_of(bins[s]);
        for (int32_t c = 0; c < H; ++c) {
            uint32_t C[33];
            C[0] = 0;
            for (int32_t k = 1; k < nsym; ++k, cdf_pos += 2)
                C[k] = (uint32_t)blob[cdf_pos] | ((uint32_t)blob[cdf_pos + 1] << 8);
            C[nsym] = CG_TOTAL;
            for (int64_t b = 0; b < nb; ++b) {
                int64_t idx = (b * 2 * L + s) * H + c;
                int32_t b0 = (int32_t)(b * CG_BATCH);
                int32_t nt = n - b0 < CG_BATCH ? n - b0 : CG_BATCH;
                cgo_decode(blob + start[idx], get_u32(blob + off[2] + 4 * idx), nt, C, nsym,
                           sym + (int64_t)b0 * H + c, H);
            }
        }
        for (int32_t t = 0; t < n; ++t) memcpy(&max1[t], blob + 4 * ((int64_t)s * n + t), 4);
        cgo_dequantize(sym, max1, n, H, bins[s], chunk + (int64_t)s * n * H);
    }
    free(sym); free(max1); free(start);
    return 0;
}
