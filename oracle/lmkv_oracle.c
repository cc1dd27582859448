/*
 * lmkv_oracle.c -- plain, slow, obviously correct CPU definition of the
 * paged-KV chunk gather / scatter and of its fp8-e4m3 variant.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no source, header, table or helper with
 * the CUDA library; it is built with plain gcc, no OpenMP, no intrinsics,
 * -ffp-contract=off, single-threaded.
 *
 * What it follows (page titles of the sources, with the part cited):
 *  - "LMCache: An Efficient KV Cache Layer for Enterprise-Scale LLM Inference"
 *    (papercache.org notes), section "可配置的块大小" (configurable chunk
 *    size): pages of many layers are copied by a kernel into a contiguous
 *    streaming buffer of 256-token chunks on store, and split back into the
 *    paged memory on load.  Section "层级流水线" (layer-wise pipeline): the
 *    same movement one layer at a time.
 *  - "LMCache 源码解析一个文件讲透KV缓存复用机制" (walk-through of
 *    cache_engine.py), section "store()": tokens are cut into chunk_size
 *    (default 256) chunks, the tail shorter than a chunk is kept only when
 *    save_unfull_chunk is set, and the already-computed prefix given to the
 *    store must be a multiple of chunk_size (else ValueError).
 *  - "LMCache 分布式 KV Cache 序列化框架：Serde 双层接口设计与自定义扩展实战",
 *    section 7.1 (fp8 serde): elements are cast
 *    to float8_e4m3fn, one byte per element.  The scaled form used here (one
 *    fp32 absmax/448 scale per (K/V, layer, chunk), round-to-nearest-even,
 *    saturating) is the workload definition of the fused variant.
 *
 * Every step is written as the plain definition: enumerate chunks, then for
 * every (chunk, K/V, layer, token) copy one token row of row_bytes bytes.
 * There is no blocking, fusion or reordering.
 *
 * Layouts (bytes; row = num_kv_heads * head_dim elements):
 *   pool layer l    : [2][num_blocks][block_size][row]
 *   chunk buffer g  : [2][num_layers][n_g][row]        (n_g = tokens in chunk g)
 *   fp8 codes g     : [2][num_layers][n_g][row] uint8
 *   fp8 scales      : [num_chunks][2][num_layers] float32
 *
 * Return codes: 0 ok, -1 invalid arguments, 5 some token referenced a block
 * id outside [0, num_blocks) and was skipped (the remaining tokens are still
 * moved).
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define ORC_OK 0
#define ORC_INVALID (-1)
#define ORC_BAD_BLOCK 5

/* ------------------------------------------------------------------------ */
/* Chunk enumeration (cache_engine.py walk-through, "store()" section).      */
/* Request r covers tokens [start[r], end[r]).  start[r] must be a multiple  */
/* of chunk_size.  Chunk j of request r covers                                */
/*   [start + j*C, min(start + (j+1)*C, end)).                                */
/* A chunk shorter than C exists only as the last one and only when          */
/* save_unfull_chunk != 0.  Chunks are numbered request by request.          */
/* Returns the number of chunks, or -1.  Output arrays may be NULL.          */
/* ------------------------------------------------------------------------ */
int64_t lmkvo_enumerate(const int64_t* start, const int64_t* end, int32_t num_req,
                        int32_t chunk_size, int32_t save_unfull,
                        int32_t* chunk_req, int64_t* chunk_tok0, int32_t* chunk_ntok,
                        int64_t cap)
{
    if (num_req < 0 || chunk_size <= 0) return ORC_INVALID;
    if (num_req > 0 && (start == NULL || end == NULL)) return ORC_INVALID;
    int64_t g = 0;
    for (int32_t r = 0; r < num_req; ++r) {
        if (start[r] < 0 || end[r] < start[r]) return ORC_INVALID;
        if (start[r] % chunk_size != 0) return ORC_INVALID;
        for (int64_t t0 = start[r]; t0 < end[r]; t0 += chunk_size) {
            int64_t t1 = t0 + chunk_size;
            if (t1 > end[r]) {
                if (!save_unfull) break;
                t1 = end[r];
            }
            if (chunk_req != NULL || chunk_tok0 != NULL || chunk_ntok != NULL) {
                if (g >= cap) return ORC_INVALID;
                if (chunk_req) chunk_req[g] = r;
                if (chunk_tok0) chunk_tok0[g] = t0;
                if (chunk_ntok) chunk_ntok[g] = (int32_t)(t1 - t0);
            }
            ++g;
        }
    }
    return g;
}

/* Shared argument check for the movement functions. */
static int check_common(void* const* layer_base, int32_t num_layers, int64_t num_blocks,
                        int32_t block_size, int32_t row_bytes, const int32_t* block_table,
                        int32_t max_blocks, const int64_t* start, const int64_t* end,
                        int32_t num_req, int32_t chunk_size)
{
    if (layer_base == NULL || num_layers <= 0 || num_blocks <= 0 || block_size <= 0 ||
        row_bytes <= 0 || max_blocks < 0 || chunk_size <= 0 || num_req < 0)
        return ORC_INVALID;
    if (num_req > 0 && (block_table == NULL || start == NULL || end == NULL)) return ORC_INVALID;
    for (int32_t l = 0; l < num_layers; ++l)
        if (layer_base[l] == NULL) return ORC_INVALID;
    for (int32_t r = 0; r < num_req; ++r) {
        if (start[r] < 0 || end[r] < start[r] || start[r] % chunk_size != 0) return ORC_INVALID;
        /* every token t < end[r] needs block-table column t / block_size */
        if (end[r] > 0 && (end[r] - 1) / block_size >= max_blocks) return ORC_INVALID;
    }
    return ORC_OK;
}

/* Byte address of token row (kv, blk, slot) inside pool layer l. */
static uint8_t* pool_row(void* const* layer_base, int32_t l, int32_t kv, int64_t num_blocks,
                         int32_t block_size, int32_t row_bytes, int64_t blk, int32_t slot)
{
    int64_t row_index = ((int64_t)kv * num_blocks + blk) * block_size + slot;
    return (uint8_t*)layer_base[l] + row_index * (int64_t)row_bytes;
}

/* Byte address of token row (kv, l, t) inside chunk buffer g with n_g rows. */
static uint8_t* chunk_row(void* const* chunk_ptrs, int64_t g, int32_t kv, int32_t l,
                          int32_t num_layers, int32_t n_g, int32_t t, int32_t row_bytes)
{
    int64_t row_index = ((int64_t)kv * num_layers + l) * n_g + t;
    return (uint8_t*)chunk_ptrs[g] + row_index * (int64_t)row_bytes;
}

/*
 * Gather (direction 0) or scatter (direction 1) of whole chunks.
 *   gather : X_g[kv][l][t] = P_l[kv][BT[r][tok/B]][tok%B]
 *   scatter: P_l[kv][BT[r][tok/B]][tok%B] = X_g[kv][l][t]
 * with tok = chunk start + t.  layer < 0 moves every layer; layer >= 0 moves
 * only that layer's slices (the layer-wise pipeline granularity).
 */
static int move_chunks(int direction, void* const* layer_base, int32_t num_layers,
                       int64_t num_blocks, int32_t block_size, int32_t row_bytes,
                       const int32_t* block_table, int32_t max_blocks,
                       const int64_t* start, const int64_t* end, int32_t num_req,
                       int32_t chunk_size, int32_t save_unfull, void* const* chunk_ptrs,
                       int32_t layer)
{
    int rc = check_common(layer_base, num_layers, num_blocks, block_size, row_bytes,
                          block_table, max_blocks, start, end, num_req, chunk_size);
    if (rc != ORC_OK) return rc;
    if (layer >= num_layers) return ORC_INVALID;
    int64_t num_chunks = lmkvo_enumerate(start, end, num_req, chunk_size, save_unfull,
                                         NULL, NULL, NULL, 0);
    if (num_chunks < 0) return ORC_INVALID;
    if (num_chunks > 0 && chunk_ptrs == NULL) return ORC_INVALID;
    int bad = 0;
    int64_t g = 0;
    for (int32_t r = 0; r < num_req; ++r) {
        for (int64_t t0 = start[r]; t0 < end[r]; t0 += chunk_size) {
            int64_t t1 = t0 + chunk_size;
            if (t1 > end[r]) {
                if (!save_unfull) break;
                t1 = end[r];
            }
            int32_t n_g = (int32_t)(t1 - t0);
            for (int32_t kv = 0; kv < 2; ++kv) {
                for (int32_t l = 0; l < num_layers; ++l) {
                    if (layer >= 0 && l != layer) continue;
                    for (int32_t t = 0; t < n_g; ++t) {
                        int64_t tok = t0 + t;
                        int64_t blk = block_table[(int64_t)r * max_blocks + tok / block_size];
                        int32_t slot = (int32_t)(tok % block_size);
                        if (blk < 0 || blk >= num_blocks) { bad = 1; continue; }
                        uint8_t* p = pool_row(layer_base, l, kv, num_blocks, block_size,
                                              row_bytes, blk, slot);
                        uint8_t* x = chunk_row(chunk_ptrs, g, kv, l, num_layers, n_g, t,
                                               row_bytes);
                        if (direction == 0) memcpy(x, p, (size_t)row_bytes);
                        else memcpy(p, x, (size_t)row_bytes);
                    }
                }
            }
            ++g;
        }
    }
    return bad ? ORC_BAD_BLOCK : ORC_OK;
}

int lmkvo_gather(void* const* layer_base, int32_t num_layers, int64_t num_blocks,
                 int32_t block_size, int32_t row_bytes, const int32_t* block_table,
                 int32_t max_blocks, const int64_t* start, const int64_t* end,
                 int32_t num_req, int32_t chunk_size, int32_t save_unfull,
                 void* const* chunk_ptrs, int32_t layer)
{
    return move_chunks(0, layer_base, num_layers, num_blocks, block_size, row_bytes,
                       block_table, max_blocks, start, end, num_req, chunk_size,
                       save_unfull, chunk_ptrs, layer);
}

int lmkvo_scatter(void* const* layer_base, int32_t num_layers, int64_t num_blocks,
                  int32_t block_size, int32_t row_bytes, const int32_t* block_table,
                  int32_t max_blocks, const int64_t* start, const int64_t* end,
                  int32_t num_req, int32_t chunk_size, int32_t save_unfull,
                  void* const* chunk_ptrs, int32_t layer)
{
    return move_chunks(1, layer_base, num_layers, num_blocks, block_size, row_bytes,
                       block_table, max_blocks, start, end, num_req, chunk_size,
                       save_unfull, chunk_ptrs, layer);
}

/* ------------------------------------------------------------------------ */
/* Number formats, written from their definitions.                           */
/*                                                                            */
/* Rounding to a binary grid with round-to-nearest, ties-to-even: a finite   */
/* a >= 0 is placed between the two neighbouring grid points of its binade   */
/* (or of the subnormal range) and the nearer one is taken; on a tie the one */
/* whose last significand bit is 0.  `mant_bits` = stored significand bits,  */
/* `emin` = exponent of the smallest normal number.  All arithmetic is in    */
/* double, where every step below is exact for float inputs.                 */
/* ------------------------------------------------------------------------ */
static double round_to_grid_rne(double a, int mant_bits, int emin)
{
    if (a == 0.0) return 0.0;
    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) => floor(log2 a) = e2-1 */
    int e = e2 - 1;
    if (e < emin) e = emin;       /* subnormal range shares the quantum of the first binade */
    double quantum = ldexp(1.0, e - mant_bits);
    double m = a / quantum;       /* exact: division by a power of two */
    double n = floor(m);
    double frac = m - n;          /* exact */
    if (frac > 0.5) n += 1.0;
    else if (frac == 0.5 && fmod(n, 2.0) != 0.0) n += 1.0;
    return n * quantum;
}

/* float -> bf16 bits, round to nearest even (bf16: 7 stored bits, emin -126,
 * max finite (2 - 2^-7) * 2^127, no saturation: overflow gives infinity). */
uint16_t lmkvo_f32_to_bf16(float v)
{
    uint32_t bits;
    memcpy(&bits, &v, 4);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs((double)v);
    double rounded = isinf(v) ? INFINITY : round_to_grid_rne(a, 7, -126);
    double max_finite = ldexp(2.0 - ldexp(1.0, -7), 127);
    if (rounded > max_finite) return (uint16_t)(sign | 0x7F80u);
    /* the rounded value is a bf16 value, hence exactly a float: take its top bits */
    float rf = (float)rounded;
    uint32_t rb;
    memcpy(&rb, &rf, 4);
    return (uint16_t)(sign | (uint16_t)(rb >> 16));
}

/* bf16 bits -> float (exact: a bf16 is the top half of a float). */
float lmkvo_bf16_to_f32(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float v;
    memcpy(&v, &bits, 4);
    return v;
}

/* float -> float8 e4m3fn bits (OCP FP8 E4M3: bias 7, 3 stored bits, smallest
 * normal 2^-6, subnormal quantum 2^-9, largest finite 448, no infinities,
 * S.1111.111 is NaN).  Round to nearest even, saturating: every |v| >= 448
 * maps to +-448.  The sign of -0 is kept (code 0x80).  NaN maps to 0x7F. */
uint8_t lmkvo_f32_to_e4m3(float v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    double r = (a >= 448.0) ? 448.0 : round_to_grid_rne(a, 3, -6);
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    uint8_t code;
    if (r < ldexp(1.0, -6)) {
        code = (uint8_t)(r / ldexp(1.0, -9));            /* subnormal: E=0, M = r / 2^-9 */
    } else {
        int e2;
        (void)frexp(r, &e2);
        int e = e2 - 1;                                  /* r in [2^e, 2^(e+1)) */
        double mant = r / ldexp(1.0, e) - 1.0;           /* in [0, 1), a multiple of 1/8 */
        code = (uint8_t)(((e + 7) << 3) | (int)(mant * 8.0));
    }
    return (uint8_t)(sign | code);
}

/* float8 e4m3fn bits -> float (exact). */
float lmkvo_e4m3_to_f32(uint8_t c)
{
    int s = (c >> 7) & 1;
    int E = (c >> 3) & 0xF;
    int M = c & 7;
    double v;
    if (E == 15 && M == 7) return NAN;
    if (E == 0) v = M * ldexp(1.0, -9);
    else v = (1.0 + M / 8.0) * ldexp(1.0, E - 7);
    return (float)(s ? -v : v);
}

/* ------------------------------------------------------------------------ */
/* fp8 variant.                                                              */
/* Quantising gather, per tile (chunk g, kv, layer l) of n_g bf16 rows:       */
/*   amax  = max |x| over the tile (exact; bf16 -> float is exact)            */
/*   scale = amax / 448.0f                  (one IEEE fp32 division)          */
/*   code  = e4m3_rne_satfinite(x / scale)  (one IEEE fp32 division each)     */
/*   amax == 0 => scale = 0 and every code = 0.                               */
/*   scales[(g*2 + kv)*L + l] = scale.                                        */
/* Dequantising scatter:                                                      */
/*   y = bf16_rne(e4m3_value(code) * scale)  (one fp32 multiply)              */
/* Rows whose block id is out of range are skipped (not read, not written).   */
/* The pool element type must be bf16 (2 bytes); row_elems = heads*head_dim.  */
/* ------------------------------------------------------------------------ */
int lmkvo_gather_fp8(void* const* layer_base, int32_t num_layers, int64_t num_blocks,
                     int32_t block_size, int32_t row_elems, const int32_t* block_table,
                     int32_t max_blocks, const int64_t* start, const int64_t* end,
                     int32_t num_req, int32_t chunk_size, int32_t save_unfull,
                     void* const* code_ptrs, float* scales)
{
    int32_t row_bytes = row_elems * 2;
    int rc = check_common(layer_base, num_layers, num_blocks, block_size, row_bytes,
                          block_table, max_blocks, start, end, num_req, chunk_size);
    if (rc != ORC_OK) return rc;
    int64_t num_chunks = lmkvo_enumerate(start, end, num_req, chunk_size, save_unfull,
                                         NULL, NULL, NULL, 0);
    if (num_chunks < 0) return ORC_INVALID;
    if (num_chunks > 0 && (code_ptrs == NULL || scales == NULL)) return ORC_INVALID;
    int bad = 0;
    int64_t g = 0;
    for (int32_t r = 0; r < num_req; ++r) {
        for (int64_t t0 = start[r]; t0 < end[r]; t0 += chunk_size) {
            int64_t t1 = t0 + chunk_size;
            if (t1 > end[r]) {
                if (!save_unfull) break;
                t1 = end[r];
            }
            int32_t n_g = (int32_t)(t1 - t0);
            for (int32_t kv = 0; kv < 2; ++kv) {
                for (int32_t l = 0; l < num_layers; ++l) {
                    /* pass 1: absmax over the tile */
                    float amax = 0.0f;
                    for (int32_t t = 0; t < n_g; ++t) {
                        int64_t tok = t0 + t;
                        int64_t blk = block_table[(int64_t)r * max_blocks + tok / block_size];
                        if (blk < 0 || blk >= num_blocks) { bad = 1; continue; }
                        const uint8_t* p = pool_row(layer_base, l, kv, num_blocks, block_size,
                                                    row_bytes, blk, (int32_t)(tok % block_size));
                        for (int32_t i = 0; i < row_elems; ++i) {
                            uint16_t h;
                            memcpy(&h, p + 2 * i, 2);
                            float a = fabsf(lmkvo_bf16_to_f32(h));
                            if (a > amax) amax = a;
                        }
                    }
                    volatile float scale = amax / 448.0f;
                    scales[(g * 2 + kv) * num_layers + l] = scale;
                    /* pass 2: codes */
                    for (int32_t t = 0; t < n_g; ++t) {
                        int64_t tok = t0 + t;
                        int64_t blk = block_table[(int64_t)r * max_blocks + tok / block_size];
                        if (blk < 0 || blk >= num_blocks) continue;
                        const uint8_t* p = pool_row(layer_base, l, kv, num_blocks, block_size,
                                                    row_bytes, blk, (int32_t)(tok % block_size));
                        uint8_t* q = (uint8_t*)code_ptrs[g] +
                                     (((int64_t)kv * num_layers + l) * n_g + t) * row_elems;
                        for (int32_t i = 0; i < row_elems; ++i) {
                            uint16_t h;
                            memcpy(&h, p + 2 * i, 2);
                            if (scale == 0.0f) { q[i] = 0; continue; }
                            volatile float y = lmkvo_bf16_to_f32(h) / scale;
                            q[i] = lmkvo_f32_to_e4m3(y);
                        }
                    }
                }
            }
            ++g;
        }
    }
    return bad ? ORC_BAD_BLOCK : ORC_OK;
}

int lmkvo_scatter_fp8(void* const* layer_base, int32_t num_layers, int64_t num_blocks,
                      int32_t block_size, int32_t row_elems, const int32_t* block_table,
                      int32_t max_blocks, const int64_t* start, const int64_t* end,
                      int32_t num_req, int32_t chunk_size, int32_t save_unfull,
                      void* const* code_ptrs, const float* scales)
{
    int32_t row_bytes = row_elems * 2;
    int rc = check_common(layer_base, num_layers, num_blocks, block_size, row_bytes,
                          block_table, max_blocks, start, end, num_req, chunk_size);
    if (rc != ORC_OK) return rc;
    int64_t num_chunks = lmkvo_enumerate(start, end, num_req, chunk_size, save_unfull,
                                         NULL, NULL, NULL, 0);
    if (num_chunks < 0) return ORC_INVALID;
    if (num_chunks > 0 && (code_ptrs == NULL || scales == NULL)) return ORC_INVALID;
    int bad = 0;
    int64_t g = 0;
    for (int32_t r = 0; r < num_req; ++r) {
        for (int64_t t0 = start[r]; t0 < end[r]; t0 += chunk_size) {
            int64_t t1 = t0 + chunk_size;
            if (t1 > end[r]) {
                if (!save_unfull) break;
                t1 = end[r];
            }
            int32_t n_g = (int32_t)(t1 - t0);
            for (int32_t kv = 0; kv < 2; ++kv) {
                for (int32_t l = 0; l < num_layers; ++l) {
                    float scale = scales[(g * 2 + kv) * num_layers + l];
                    for (int32_t t = 0; t < n_g; ++t) {
                        int64_t tok = t0 + t;
                        int64_t blk = block_table[(int64_t)r * max_blocks + tok / block_size];
                        if (blk < 0 || blk >= num_blocks) { bad = 1; continue; }
                        uint8_t* p = pool_row(layer_base, l, kv, num_blocks, block_size,
                                              row_bytes, blk, (int32_t)(tok % block_size));
                        const uint8_t* q = (const uint8_t*)code_ptrs[g] +
                                           (((int64_t)kv * num_layers + l) * n_g + t) * row_elems;
                        for (int32_t i = 0; i < row_elems; ++i) {
                            volatile float y = lmkvo_e4m3_to_f32(q[i]) * scale;
                            uint16_t h = lmkvo_f32_to_bf16(y);
                            memcpy(p + 2 * i, &h, 2);
                        }
                    }
                }
            }
            ++g;
        }
    }
    return bad ? ORC_BAD_BLOCK : ORC_OK;
}

/* Exported elementwise helpers so the format routines can be pinned against
 * independent implementations on whole arrays. */
void lmkvo_f32_to_e4m3_array(const float* v, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = lmkvo_f32_to_e4m3(v[i]);
}

void lmkvo_e4m3_to_f32_array(const uint8_t* c, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = lmkvo_e4m3_to_f32(c[i]);
}

void lmkvo_f32_to_bf16_array(const float* v, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = lmkvo_f32_to_bf16(v[i]);
}

/* y[i] = x[i] / s in fp32 (the quantiser's division, exported for pins). */
void lmkvo_div_f32_array(const float* x, float s, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        volatile float y = x[i] / s;
        out[i] = y;
    }
}
