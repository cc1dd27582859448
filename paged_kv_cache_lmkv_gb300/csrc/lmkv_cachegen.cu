// lmkv_cachegen.cu -- the CacheGen KV codec on sm_103a ("LMCache 中的 KV Cache
// 压缩：CacheGen 编解码原理、配置方式与源码解析", sections 1-5).
//
// Encode, per group of up to kMaxChunks chunks (three kernels):
//   cg_cdf_kernel     per (chunk, kv, layer) slice: per-token absmax over the
//                     row (section 2), the symbols (into the workspace), a
//                     per-channel histogram in shared memory and the 2^16 CDF
//                     with its arange ramp (section 3), written to the blob.
//   cg_code_kernel    per (chunk, 256-token batch, kv, layer) region: every
//                     thread runs kStreams independent arithmetic coders, one
//                     per channel (section 4), into fixed-size slots.
//   cg_compact_kernel per region: the prefix sums of the stream lengths place
//                     each slot's bytes into the blob.
// Decode (two kernels): cg_total_kernel sums each region's lengths, then
// cg_decode_kernel finds each stream by the prefix sums (section 5), decodes
// kStreams channels per thread and writes the dequantised bf16 rows.
// A slice or region takes 1, 2 or 4 CTAs (CgParams::split, chosen per launch
// so that a small batch still covers the SMs): the CDF pass splits the rows
// over a thread-block cluster, the other kernels split the channels.
//
// The coder is the integer arithmetic coder of Witten, Neal and Cleary
// (CACM 30(6), 1987) with 32-bit registers and frequencies out of 2^16.  Its
// bit-at-a-time renormalisation is taken here in two jumps: the run of
// leading bits where low and high agree (count leading zeros of low ^ high)
// is shifted out at once, then the run of middle-straddling steps (low =
// 01..., high = 10...) is counted and folded into the pending bits.  The bits
// produced are those of the one-bit-per-step loop.
#include "lmkv.h"
#include "lmkv_internal.h"

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

namespace {

namespace cg = cooperative_groups;

constexpr int kBatch = LMKV_CACHEGEN_BATCH;
constexpr int kMaxChunks = 64;                 // chunks per launch
constexpr int kMaxSlices = 2 * LMKV_CACHEGEN_MAX_LAYERS;
constexpr int kStreams = 4;                    // channels (streams) per thread
constexpr int kRows = 8;                       // rows per block-wide absmax round
constexpr int kMaxThreads = LMKV_CACHEGEN_MAX_CHANNELS / kStreams;
constexpr uint64_t kMaxBlobBytes = 0xFFFFFF00ull;   // blobs are addressed with 32-bit offsets

struct CgParams {
    const uint8_t* const* chunk_ptrs;   // DEVICE array of chunk buffers (chunk form), else null
    uint8_t* const* blob_ptrs;          // DEVICE array of blobs
    uint64_t* sizes;                    // DEVICE blob sizes (encode writes, decode reads)
    int32_t* status;
    uint8_t* ws;
    int32_t L, H, nchunks, cdf_entries;
    int32_t split;                      // CTAs per slice (CDF pass) / per region (coder, compaction, decoder)
    int32_t ntok[kMaxChunks];
    uint64_t tot_off[kMaxChunks];       // workspace byte offsets per chunk
    uint64_t sym_off[kMaxChunks];
    uint64_t slot_off[kMaxChunks];
    int32_t cdf_prefix[kMaxSlices];     // cdf entries before slice s
    uint8_t bins[kMaxSlices];
    // Pool form (layer_base != null): chunk gi is tokens [chunk_tok0, chunk_tok0 +
    // ntok) of block-table row chunk_req, rows read from / written to the pages.
    const uint8_t* const* layer_base;   // DEVICE array of per-layer pool bases
    const int32_t* block_table;
    int64_t num_blocks;
    int32_t bt_stride, block_size;
    int32_t chunk_req[kMaxChunks];
    int64_t chunk_tok0[kMaxChunks];
};

// The token rows of one (chunk, K/V, layer) slice, walked in token order:
// consecutive rows of the chunk buffer, or the rows of the chunk's pages in
// the pool (one block-table entry per block; an id outside [0, num_blocks)
// gives null rows).
struct Rows {
    const uint8_t* cur;        // chunk form: this row; pool form: the current block's first row
    const uint8_t* layer;      // pool form: K or V half of the layer
    const int32_t* bt;         // pool form: the request's block-table row
    uint32_t row_bytes;
    int32_t col, slot, B;
    int64_t nb;
    bool pool;
};

__device__ __forceinline__ const uint8_t* block_rows(const Rows& R, int32_t blk) {
    return (blk >= 0 && blk < R.nb) ? R.layer + (uint64_t)blk * R.B * R.row_bytes : nullptr;
}

// Rows of slice s of chunk gi from token t (chunk-relative) on.
__device__ __forceinline__ void rows_init(Rows& R, const CgParams& p, int gi, int s, int n, int t) {
    R.row_bytes = (uint32_t)p.H * 2;
    R.pool = p.layer_base != nullptr;
    if (!R.pool) {
        R.cur = p.chunk_ptrs[gi] + ((uint64_t)s * n + t) * R.row_bytes;
        return;
    }
    const int kv = s / p.L, l = s % p.L;
    R.B = p.block_size;
    R.nb = p.num_blocks;
    R.layer = p.layer_base[l] + (uint64_t)kv * p.num_blocks * p.block_size * R.row_bytes;
    R.bt = p.block_table + (uint64_t)p.chunk_req[gi] * p.bt_stride;
    const int64_t tok = p.chunk_tok0[gi] + t;
    R.col = (int32_t)(tok / R.B);
    R.slot = (int32_t)(tok % R.B);
    R.cur = block_rows(R, R.bt[R.col]);
}

__device__ __forceinline__ const uint8_t* rows_ptr(const Rows& R) {
    if (!R.pool) return R.cur;
    return R.cur ? R.cur + (uint64_t)R.slot * R.row_bytes : nullptr;
}

// Step to the next row; `more` says whether it exists (so no block-table entry
// past the request's last block is read).
__device__ __forceinline__ void rows_next(Rows& R, bool more) {
    if (!R.pool) {
        R.cur += R.row_bytes;
        return;
    }
    if (++R.slot == R.B) {
        R.slot = 0;
        ++R.col;
        if (more) R.cur = block_rows(R, R.bt[R.col]);
    }
}

// The chunk's blob and rows are there and 4-byte aligned (the kernels move
// 32-bit words); otherwise the chunk is skipped and BAD_POINTER reported.
__device__ __forceinline__ bool aligned4(const void* q) {
    return q != nullptr && (reinterpret_cast<uintptr_t>(q) & 3) == 0;
}
// Every kernel of a call takes the same whole-chunk decision, so a chunk is
// either processed by all of them or by none (no kernel reads what a skipped
// one did not write).
__device__ __forceinline__ bool chunk_ok(const CgParams& p, int gi) {
    if (!aligned4(p.blob_ptrs[gi])) return false;
    if (p.layer_base == nullptr) return aligned4(p.chunk_ptrs[gi]);
    bool ok = true;
    for (int l = 0; l < p.L; ++l) ok &= aligned4(p.layer_base[l]);
    return ok;
}

__host__ __device__ inline int nsym_of(int bins) { return 2 * (bins / 2 - 1) + 1; }
__host__ __device__ inline int batches_of(int n) { return (n + kBatch - 1) / kBatch; }

// Blob offsets (the layout in lmkv.h).
__host__ __device__ inline uint64_t cdf_offset(int L, int n) { return 8ull * (uint64_t)L * n; }
__host__ __device__ inline uint64_t lengths_offset(int L, int n, int cdf_entries) {
    return (cdf_offset(L, n) + 2ull * (uint64_t)cdf_entries + 3) & ~3ull;
}
__host__ __device__ inline uint64_t bytes_offset(int L, int n, int H, int cdf_entries) {
    return lengths_offset(L, n, cdf_entries) + 4ull * batches_of(n) * 2ull * L * H;
}
// Largest stream of nt symbols: every symbol leaves an interval of at least
// 2^14 of at most 2^32 and each emitted or pending bit doubles it, so at most
// 18 bits per symbol, plus the two final bits.
__host__ __device__ inline uint64_t stream_bound(int nt) { return (18ull * nt + 2 + 7) / 8; }
// Slot stride in the workspace: the bound plus 4 bytes (the compaction reads
// one word past a stream), rounded up to 16 bytes.
__host__ __device__ inline uint64_t slot_stride(int n) {
    const int nt = n < kBatch ? n : kBatch;
    return (stream_bound(nt) + 4 + 15) & ~15ull;
}

__device__ __forceinline__ void set_status(int32_t* st, int code) {
    if (st != nullptr) atomicCAS(st, 0, code);
}

// |x| of two packed bf16 as the larger fp32 bit pattern (non-negative floats
// order like their bit patterns).
__device__ __forceinline__ uint32_t abs_max_bits(uint32_t two_bf16) {
    const uint32_t a = (two_bf16 << 16) & 0x7FFF0000u;
    const uint32_t b = two_bf16 & 0x7FFF0000u;
    return a > b ? a : b;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// q = clamp(round(x * factor + MAX), 0, 2*MAX), one fp32 operation per step.
// The clamp is taken first (the bounds are integers, so it commutes with the
// rounding; a NaN product, 0 * inf for a row of tiny values, clamps to 0),
// then adding 1.5 * 2^23 rounds to an integer with ties to even (in
// [2^23, 2^24) the spacing of floats is 1) and leaves it in the low bits.
__device__ __forceinline__ uint32_t quantise(float x, float factor, float maxf, float two_maxf) {
    const float z = fminf(fmaxf(__fadd_rn(__fmul_rn(x, factor), maxf), 0.0f), two_maxf);
    return __float_as_uint(__fadd_rn(z, 12582912.0f)) - 0x4B400000u;
}

// Channel j (0..kStreams-1) of thread tid: the pairs (2*tid, 2*tid + 1) in
// each half of the row.  Lanes then touch consecutive 32-bit words of every
// [symbol][channel] uint16 table row, so table reads and histogram updates
// are free of shared-memory bank conflicts whatever symbol each lane holds.
__device__ __forceinline__ int chan(int tid, int j, int H) {
    return 2 * tid + (j & 1) + (j >> 1) * (H >> 1);
}

// ---- arithmetic encoder state, one per stream ----
// Bit strings are moved with the funnel shifts of two 32-bit words (a shift
// by a variable amount of a 64-bit integer is not one instruction).
struct Enc {
    uint32_t low, high, follow, nacc, words;
    uint32_t acc_hi, acc_lo;   // output bits not yet stored: the last nacc of acc_hi:acc_lo
};

__device__ __forceinline__ void enc_init(Enc& e) {
    e.low = 0;
    e.high = 0xFFFFFFFFu;
    e.follow = 0;
    e.nacc = 0;
    e.words = 0;
    e.acc_hi = 0;
    e.acc_lo = 0;
}

// Append the c (0..32) bits v (nothing above them set); a completed 32-bit
// word goes to the slot, most significant byte first.
__device__ __forceinline__ void put_bits(Enc& e, uint32_t v, uint32_t c, uint32_t* slot,
                                         uint32_t cap_words, bool& overflow) {
    e.acc_hi = __funnelshift_lc(e.acc_lo, e.acc_hi, c);
    e.acc_lo = __funnelshift_lc(0u, e.acc_lo, c) | v;
    e.nacc += c;
    const bool full = e.nacc >= 32;
    e.nacc -= full ? 32u : 0u;
    const uint32_t w = __funnelshift_rc(e.acc_lo, e.acc_hi, e.nacc);
    if (full) {
        if (e.words < cap_words) slot[e.words] = __byte_perm(w, 0, 0x0123);
        else overflow = true;
    }
    e.words += full ? 1u : 0u;
}

// 2^f - 1 for 0 <= f <= 32.
__device__ __forceinline__ uint32_t ones(uint32_t f) { return __funnelshift_rc(0xFFFFFFFFu, 0u, 32 - f); }

// The rare case of more than 32 bits at once (a long run of held bits):
// `bit`, then `f` opposite bits, then the k-1 bits `rest`.
__device__ __forceinline__ void emit_long(Enc& e, uint32_t bit, uint32_t f, uint32_t k, uint32_t rest,
                                      uint32_t* slot, uint32_t cap_words, bool& overflow) {
    put_bits(e, bit, 1, slot, cap_words, overflow);
    for (uint32_t left = f; left > 0;) {
        const uint32_t c = left < 32 ? left : 32;
        put_bits(e, bit ? 0u : ones(c), c, slot, cap_words, overflow);
        left -= c;
    }
    put_bits(e, rest, k - 1, slot, cap_words, overflow);
}

// Narrow [low, high] to the symbol's [lo, hi) out of 2^16, then renormalise.
//
// low and high are kept without the quarter subtraction of the middle-
// straddling steps: such a step is a left shift followed by adding 2^31
// modulo 2^32, and leaving the addition out changes only bit 31 of low and
// high, both alike.  So low ^ high, high - low and every bit below bit 31 are
// those of the textbook registers, and bit 31 of the true low is bit 31 of
// this low flipped exactly when held bits are pending (follow > 0).  The
// renormalisation is then one shift by k + m: the k leading bits where low
// and high agree are decided (the first releases the held bits, as its
// opposite), and the m steps after them that straddle the middle are held.
__device__ __forceinline__ void enc_symbol(Enc& e, uint32_t lo, uint32_t hi, uint32_t* slot,
                                           uint32_t cap_words, bool& overflow) {
    const uint32_t rm1 = e.high - e.low;                       // range - 1
    const uint64_t top = (uint64_t)rm1 * hi + hi;              // range * hi
    const uint64_t bot = (uint64_t)rm1 * lo + lo;              // range * lo
    e.high = e.low + (uint32_t)(top >> 16) - 1;
    e.low = e.low + (uint32_t)(bot >> 16);
    const uint32_t k = __clz(e.low ^ e.high);                  // 0..18
    const uint32_t f = e.follow;
    // The k decided bits are the top k bits of the true low.  "b" followed by
    // f copies of "not b" is the number 2^f - 1 + b, so the run is
    // top_k(true low) + (2^f - 1) * 2^(k-1).
    const uint32_t topk = __funnelshift_rc(e.low ^ (f ? 0x80000000u : 0u), 0u, 32 - k);  // 0 if k == 0
    if (f + k <= 32) {
        const uint32_t held = k ? ones(f) << (k - 1) : 0u;
        put_bits(e, topk + held, k ? f + k : 0u, slot, cap_words, overflow);
    } else if (k) {
        emit_long(e, topk >> (k - 1), f, k, topk & ((1u << (k - 1)) - 1), slot, cap_words, overflow);
    }
    // straddling steps: the leading run of positions after bit k where low
    // holds 1 and high holds 0
    const uint32_t m = __clz(~(e.low << (k + 1)) | (e.high << (k + 1)));
    const uint32_t c = k + m;
    e.follow = (k ? 0u : f) + m;
    e.low <<= c;
    e.high = (e.high << c) | ((1u << c) - 1);
}

// Two final bits select a point inside the last interval; returns the
// stream's length in bytes.  Bit 30 of the kept low is that of the true low.
__device__ __forceinline__ uint32_t enc_finish(Enc& e, uint32_t* slot, uint32_t cap_words,
                                               bool& overflow) {
    const uint32_t bit = (e.low >> 30) & 1u;                   // true low >= 2^30
    const uint32_t f = e.follow + 1;
    if (f + 1 <= 32) {
        const uint32_t run = bit ? 0u : ones(f);
        put_bits(e, (bit << f) | run, f + 1, slot, cap_words, overflow);
    } else {
        emit_long(e, bit, f, 1, 0, slot, cap_words, overflow);
    }
    e.follow = 0;
    const uint32_t bits = e.words * 32 + e.nacc;
    if (e.nacc) {
        const uint32_t w = e.acc_lo << (32 - e.nacc);
        if (e.words < cap_words) slot[e.words] = __byte_perm(w, 0, 0x0123);
        else overflow = true;
    }
    return (bits + 7) >> 3;
}

// ---- arithmetic decoder state, one per stream ----
// The reader does not stop at the stream's end: the bits after it are those
// of the next stream (or of the blob's tail).  That cannot change a decoded
// symbol, because the encoder's two final bits select a sub-interval of the
// last interval that every continuation stays inside ([1/4, 1/2) or
// [1/2, 3/4) of the renormalised window), and the decoder stops after n
// symbols.  Reads stay inside the blob.  low, high and value are kept without
// the quarter subtraction, as in the encoder: the decoder needs only
// value - low, high - low and low ^ high, which that leaves unchanged.
struct Dec {
    uint32_t low, high, value, nbuf;
    uint32_t q;              // blob offset of the next word to load
    uint32_t next;           // the word at q - 4 as loaded, ahead of its use
    uint32_t buf_hi, buf_lo; // upcoming bits, most significant first; nbuf valid
};

// The aligned word at blob offset q as stored (little-endian load); bytes at
// or past `size` read as zero.  The byte swap to stream order is left to the
// consumer so that a load issued ahead is not waited for here.
__device__ __forceinline__ uint32_t load_word(const uint8_t* blob, uint32_t q, uint32_t size) {
    if (q + 4 <= size) return __ldg(reinterpret_cast<const uint32_t*>(blob + q));
    uint32_t w = 0;
    for (uint32_t i = 0; i < 4; ++i)
        if (q + i < size) w |= (uint32_t)blob[q + i] << (8 * i);
    return w;
}

// Keep more than 32 bits buffered; the word after the one consumed is
// loaded now and used by the next refill.
__device__ __forceinline__ void dec_refill(Dec& d, const uint8_t* blob, uint32_t size) {
    if (d.nbuf <= 32) {
        const uint32_t w = __byte_perm(d.next, 0, 0x0123);     // placed at bit 64 - nbuf - 32
        d.buf_hi |= __funnelshift_rc(w, 0u, d.nbuf);
        d.buf_lo |= __funnelshift_lc(0u, w, 32 - d.nbuf);
        d.nbuf += 32;
        d.next = load_word(blob, d.q, size);
        d.q += 4;
    }
}

// The next c (0..32) bits.
__device__ __forceinline__ uint32_t dec_take(Dec& d, uint32_t c) {
    const uint32_t r = __funnelshift_lc(d.buf_hi, 0u, c);
    d.buf_hi = __funnelshift_lc(d.buf_lo, d.buf_hi, c);
    d.buf_lo = __funnelshift_lc(0u, d.buf_lo, c);
    d.nbuf -= c;
    return r;
}

// The stream starting at blob offset `start` (the blob is 4-byte aligned and
// `size` bytes long).
__device__ __forceinline__ void dec_init(Dec& d, const uint8_t* blob, uint32_t start, uint32_t size) {
    const uint32_t a = start & ~3u, sh = start - a;
    d.buf_hi = __byte_perm(load_word(blob, a, size), 0, 0x0123) << (8 * sh);
    d.buf_lo = 0;
    d.nbuf = 32 - 8 * sh;
    d.next = load_word(blob, a + 4, size);
    d.q = a + 8;
    dec_refill(d, blob, size);
    d.value = dec_take(d, 32);
    d.low = 0;
    d.high = 0xFFFFFFFFu;
}

// One symbol.  table[k * H] holds C[k] of this stream's channel for k < nsym
// and 0xFFFF for nsym <= k < 2^kSteps (C[nsym] = 2^16).  The symbol is the
// largest k with floor(range * C[k] / 2^16) <= value - low: the interval the
// encoder chose.  A padding row can only be picked when value - low lies in
// the top of the last symbol's interval, so the search result is clamped to
// nsym - 1.
template <int kSteps>
__device__ __forceinline__ uint32_t dec_symbol(Dec& d, const uint16_t* table, int H, int nsym,
                                               const uint8_t* blob, uint32_t size) {
    dec_refill(d, blob, size);
    const uint32_t v = d.value - d.low;
    const uint32_t rm1 = d.high - d.low;
    int s = 0;
#pragma unroll
    for (int step = 1 << (kSteps - 1); step >= 1; step >>= 1) {
        const uint32_t C = table[(s + step) * H];
        if ((uint32_t)(((uint64_t)rm1 * C + C) >> 16) <= v) s += step;
    }
    s = s < nsym - 1 ? s : nsym - 1;
    const uint32_t lo = table[s * H];
    const uint32_t hi = s + 1 < nsym ? (uint32_t)table[(s + 1) * H] : 65536u;
    const uint64_t top = (uint64_t)rm1 * hi + hi;
    const uint64_t bot = (uint64_t)rm1 * lo + lo;
    d.high = d.low + (uint32_t)(top >> 16) - 1;
    d.low = d.low + (uint32_t)(bot >> 16);
    const uint32_t k = __clz(d.low ^ d.high);
    const uint32_t c = k + __clz(~(d.low << (k + 1)) | (d.high << (k + 1)));
    d.low <<= c;
    d.high = (d.high << c) | ((1u << c) - 1);
    d.value = (d.value << c) | dec_take(d, c);
    return (uint32_t)s;
}

// Block-wide sum; every thread gets the result.  `red` holds >= 32 words.
__device__ __forceinline__ uint64_t block_sum(uint64_t v, uint64_t* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    uint64_t t = 0;
    for (int w = 0; w < nw; ++w) t += red[w];
    return t;
}

// Exclusive block-wide prefix sum of v in thread order, and the block total.
// `red` holds >= 32 words.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* red, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) red[warp] = x;
    __syncthreads();
    uint32_t before = 0, all = 0;
    for (int w = 0; w < nw; ++w) {
        before += w < warp ? red[w] : 0u;
        all += red[w];
    }
    *total = all;
    return before + x - v;
}

// Byte offsets, in channel order, of this thread's kStreams streams within
// their region, from the region's lengths.
__device__ __forceinline__ void stream_offsets(const uint32_t (&l)[kStreams], uint32_t* red,
                                               uint32_t (&off)[kStreams]) {
    uint32_t total0, total1;
    const uint32_t o0 = block_scan(l[0] + l[1], red, &total0);      // channels 0 .. H/2-1
    const uint32_t o1 = block_scan(l[2] + l[3], red + 32, &total1); // channels H/2 .. H-1
    off[0] = o0;
    off[1] = o0 + l[0];
    off[2] = total0 + o1;
    off[3] = total0 + o1 + l[2];
}

// Cluster barrier halves (every thread of every CTA of the cluster takes part).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- encode 1: absmax, symbols, histogram, CDF ----
// grid (2L * split, chunks) in clusters of `split` CTAs along x, one cluster
// per (chunk, kv, layer) slice; block = H / kStreams threads rounded up to a
// warp, thread t holding channels chan(t, 0..3).  CTA `part` of a slice takes
// a contiguous 1/split of its rows.  The histograms are then merged through
// distributed shared memory: each CTA sums, over the cluster, the channels of
// its 1/split of the threads, and those threads write their CDFs.
// Shared memory: uint16 hist[nsym_max][H] (counts <= n <= 4096).
__global__ void __launch_bounds__(kMaxThreads) cg_cdf_kernel(const __grid_constant__ CgParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint32_t part_max[2][kRows][kMaxThreads / 32];
    const int gi = blockIdx.y, S = p.split;
    const int s = blockIdx.x / S, part = blockIdx.x % S;    // part = rank in the cluster
    const int n = p.ntok[gi], H = p.H, L = p.L;
    const int bins = p.bins[s], MAX = bins / 2 - 1, nsym = 2 * MAX + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (blockDim.x + 31) >> 5;
    const int T = H / kStreams, Tl = T / S;
    const bool active = tid < T;
    uint16_t* hist = reinterpret_cast<uint16_t*>(smem);

    uint8_t* blob = p.blob_ptrs[gi];
    if (!chunk_ok(p, gi)) {            // the same decision in every CTA of the cluster
        if (tid == 0 && part == 0) set_status(p.status, LMKV_ERR_BAD_POINTER);
        return;
    }
    if (part == 0) {                   // the coder adds each region's total into these
        uint32_t* totals = reinterpret_cast<uint32_t*>(p.ws + p.tot_off[gi]);
        for (int b = tid; b < batches_of(n); b += blockDim.x) totals[b * 2 * L + s] = 0;
    }
    if (active)
        for (int k = 0; k < nsym; ++k) {
            *reinterpret_cast<uint32_t*>(hist + k * H + chan(tid, 0, H)) = 0;
            *reinterpret_cast<uint32_t*>(hist + k * H + chan(tid, 2, H)) = 0;
        }

    // this CTA's rows [r0, r1); this thread's two bf16 pairs of a row:
    // channels (2t, 2t+1) and (H/2 + 2t, H/2 + 2t + 1)
    const int per = (n + S - 1) / S;
    const int r0 = part * per < n ? part * per : n, r1 = r0 + per < n ? r0 + per : n;
    Rows rows;
    if (r0 < r1) rows_init(rows, p, gi, s, n, r0);
    bool bad_row = false;
    uint32_t* sym = reinterpret_cast<uint32_t*>(p.ws + p.sym_off[gi] + (uint64_t)s * n * H) + tid;
    float* max1_out = reinterpret_cast<float*>(blob) + (uint64_t)s * n;
    const float maxf = (float)MAX, two_maxf = (float)(2 * MAX);
    uint32_t* hist32 = reinterpret_cast<uint32_t*>(smem);

    // rows are loaded one group of kRows ahead of their use
    uint2 nxt[kRows];
    auto load_group = [&](int t0) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            nxt[r] = make_uint2(0, 0);
            if (t0 + r < r1) {
                const uint8_t* row = rows_ptr(rows);
                if (row == nullptr) {
                    bad_row = true;                     // a bad block id: the row reads as zeros
                } else if (active) {
                    nxt[r].x = __ldg(reinterpret_cast<const uint32_t*>(row + 4 * tid));
                    nxt[r].y = __ldg(reinterpret_cast<const uint32_t*>(row + H + 4 * tid));
                }
                rows_next(rows, t0 + r + 1 < r1);
            }
        }
    };
    if (r0 < r1) load_group(r0);
    for (int t0 = r0, buf = 0; t0 < r1; t0 += kRows, buf ^= 1) {
        uint2 v[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) v[r] = nxt[r];
        if (t0 + kRows < r1) load_group(t0 + kRows);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const uint32_t a = abs_max_bits(v[r].x), b = abs_max_bits(v[r].y);
            const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, a > b ? a : b);
            if (lane == 0) part_max[buf][r][warp] = m;
        }
        __syncthreads();
        // lane r of every warp finishes row r: the max over the warps' partial
        // maxima and factor = MAX / max1 (IEEE division; 0 for an all-zero row,
        // which then quantises to MAX everywhere); the other lanes get them by
        // shuffles
        uint32_t mb = 0;
        if (lane < kRows)
            for (int w = 0; w < nw; ++w) mb = mb > part_max[buf][lane][w] ? mb : part_max[buf][lane][w];
        const float mrow = __uint_as_float(mb);
        const float frow = mb ? __fdiv_rn(maxf, mrow) : 0.0f;
        if (warp == 0 && lane < kRows && t0 + lane < r1) max1_out[t0 + lane] = mrow;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int t = t0 + r;
            const float factor = __shfl_sync(0xFFFFFFFFu, frow, r);
            if (t >= r1 || !active) continue;
            uint32_t q[kStreams];
            q[0] = quantise(bf16_lo(v[r].x), factor, maxf, two_maxf);
            q[1] = quantise(bf16_hi(v[r].x), factor, maxf, two_maxf);
            q[2] = quantise(bf16_lo(v[r].y), factor, maxf, two_maxf);
            q[3] = quantise(bf16_hi(v[r].y), factor, maxf, two_maxf);
            sym[(uint64_t)t * (H / 4)] = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
            // channels (2t, 2t+1) share a 32-bit word of the uint16 histogram
            // row, low half first; no carry between the halves (counts <= 4096)
            atomicAdd(hist32 + q[0] * (H / 2) + tid, 1u);
            atomicAdd(hist32 + q[1] * (H / 2) + tid, 0x10000u);
            atomicAdd(hist32 + q[2] * (H / 2) + H / 4 + tid, 1u);
            atomicAdd(hist32 + q[3] * (H / 2) + H / 4 + tid, 0x10000u);
        }
    }
    if (bad_row && tid == 0) set_status(p.status, LMKV_ERR_BAD_BLOCK);
    if (S > 1) {
        cluster_arrive();              // every CTA's histogram is complete ...
        cluster_wait();
        // ... and this CTA sums its threads' channels over the cluster: the
        // pairs [2 part Tl, 2 (part + 1) Tl) of each half of the row, as
        // 32-bit words of two counts (no carry between the halves: <= 4096)
        for (int i = tid; i < nsym * 2 * Tl; i += blockDim.x) {
            const int k = i / (2 * Tl), r = i % (2 * Tl);
            const int c = (r < Tl ? 0 : H / 2) + 2 * (part * Tl + r % Tl);
            uint32_t* w = reinterpret_cast<uint32_t*>(hist + k * H + c);
            uint32_t sum = *w;
            for (int q = 1; q < S; ++q) sum += *cg::this_cluster().map_shared_rank(w, (unsigned)((part + q) % S));
            *w = sum;
        }
        cluster_arrive();              // this CTA has read its peers' counts
        __syncthreads();
    }
    // C[k] = round(cum[k] * (2^16 - (Lp - 1)) / n) + k, ties to even; the
    // blob keeps C[1..nsym-1] per channel.
    if (active && tid / Tl == part) {
        const uint32_t M = 65536u - (uint32_t)nsym;
        uint16_t* cdf = reinterpret_cast<uint16_t*>(blob + cdf_offset(L, n)) + p.cdf_prefix[s];
#pragma unroll
        for (int j = 0; j < kStreams; ++j) {
            const int c = chan(tid, j, H);
            uint16_t* dst = cdf + (uint64_t)c * (nsym - 1);
            uint32_t cum = 0;
            for (int k = 0; k < nsym; ++k) {
                const uint32_t num = cum * M;
                uint32_t q = num / (uint32_t)n;
                const uint32_t r = num - q * (uint32_t)n;
                if (2 * r > (uint32_t)n || (2 * r == (uint32_t)n && (q & 1))) ++q;
                if (k > 0) dst[k - 1] = (uint16_t)(q + k);
                cum += hist[k * H + c];
            }
        }
    }
    if (S > 1) cluster_wait();         // peers may still be reading this CTA's counts
}

// Load this CTA's part of one slice's CDF table from the blob into shared
// memory: table[k * Hl + cl] = C[k] for k < nsym (C[0] = 0) and 0xFFFF for
// nsym <= k < rows, cl the local index of the thread's channel (Hl = H /
// split channels per CTA).
__device__ __forceinline__ void load_table_part(uint16_t* table, const uint8_t* blob, const CgParams& p,
                                                int s, int n, int nsym, int tid, int tl, int Hl, int rows) {
    const uint16_t* src = reinterpret_cast<const uint16_t*>(blob + cdf_offset(p.L, n)) + p.cdf_prefix[s];
#pragma unroll
    for (int j = 0; j < kStreams; ++j) {
        const int c = chan(tid, j, p.H), cl = chan(tl, j, Hl);
        const uint16_t* sc = src + (uint64_t)c * (nsym - 1);
        table[cl] = 0;
        for (int k = 1; k < rows; ++k) table[k * Hl + cl] = k < nsym ? sc[k - 1] : (uint16_t)0xFFFF;
    }
}

// ---- encode 2: the coders of one (chunk, batch, kv, layer) region ----
// grid (nb_max * 2L * split, chunks): CTA `part` of a region runs the threads
// [part * Tl, (part + 1) * Tl) of the region (Tl = H / kStreams / split), each
// with kStreams coders.  Shared memory: uint16 table[nsym][H / split].
// kThreads = 256 (up to 1024 channels) lets three CTAs share an SM's
// registers; 512 covers up to 2048 channels.
template <int kThreads>
__global__ void __launch_bounds__(kThreads, kThreads == 256 ? 3 : 1)
cg_code_kernel(const __grid_constant__ CgParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint64_t red[32];
    const int gi = blockIdx.y, n = p.ntok[gi], H = p.H, L = p.L, S = p.split;
    const int region = blockIdx.x / S, part = blockIdx.x % S;
    const int b = region / (2 * L), s = region % (2 * L);
    if (b >= batches_of(n)) return;
    const int nsym = nsym_of(p.bins[s]);
    const int t0 = b * kBatch, nt = n - t0 < kBatch ? n - t0 : kBatch;
    const int Hl = H / S, Tl = Hl / kStreams;
    const int tl = threadIdx.x, tid = part * Tl + tl;
    const bool active = tl < Tl;
    uint8_t* blob = p.blob_ptrs[gi];
    if (!chunk_ok(p, gi)) return;   // reported by the CDF kernel
    uint16_t* table = reinterpret_cast<uint16_t*>(smem);
    if (active) load_table_part(table, blob, p, s, n, nsym, tid, tl, Hl, nsym);
    __syncthreads();

    const uint64_t stride = slot_stride(n);
    const uint32_t cap_words = (uint32_t)((stride - 4) / 4);     // keep the slack word free
    uint32_t len[kStreams] = {0, 0, 0, 0};
    bool overflow = false;
    if (active) {
        uint32_t* slot[kStreams];
        const uint16_t* tab[kStreams];
        Enc e[kStreams];
#pragma unroll
        for (int j = 0; j < kStreams; ++j) {
            const int c = chan(tid, j, H);
            slot[j] = reinterpret_cast<uint32_t*>(p.ws + p.slot_off[gi] + ((uint64_t)region * H + c) * stride);
            tab[j] = table + chan(tl, j, Hl);
            enc_init(e[j]);
        }
        const uint32_t* sym = reinterpret_cast<const uint32_t*>(p.ws + p.sym_off[gi] +
                                                                ((uint64_t)s * n + t0) * H) + tid;
        const int hw = H / 4;
        uint32_t w_next = sym[0];
        for (int t = 0; t < nt; ++t) {
            const uint32_t w = w_next;
            if (t + 1 < nt) w_next = sym[(uint64_t)(t + 1) * hw];
#pragma unroll
            for (int j = 0; j < kStreams; ++j) {
                const uint32_t q = (w >> (8 * j)) & 0xFFu;
                const uint32_t lo = tab[j][q * Hl];
                const uint32_t hi = (int)q + 1 < nsym ? (uint32_t)tab[j][(q + 1) * Hl] : 65536u;
                enc_symbol(e[j], lo, hi, slot[j], cap_words, overflow);
            }
        }
        uint32_t* lengths = reinterpret_cast<uint32_t*>(blob + lengths_offset(L, n, p.cdf_entries)) +
                            (uint64_t)region * H;
#pragma unroll
        for (int j = 0; j < kStreams; ++j) {
            len[j] = enc_finish(e[j], slot[j], cap_words, overflow);
            // never past the slot (excluded by the bound; keeps the blob in bounds)
            len[j] = len[j] < cap_words * 4 ? len[j] : cap_words * 4;
            lengths[chan(tid, j, H)] = len[j];
        }
    }
    if (overflow) set_status(p.status, LMKV_ERR_SCRATCH_LIMIT);   // excluded by the bound
    const uint64_t total = block_sum((uint64_t)len[0] + len[1] + len[2] + len[3], red);
    if (tl == 0)   // the CDF pass zeroed the region totals
        atomicAdd(reinterpret_cast<uint32_t*>(p.ws + p.tot_off[gi]) + region, (uint32_t)total);
}

// Byte offset of region `region` within the chunk's streams, and the total
// of all regions (both from the per-region totals).
__device__ __forceinline__ void region_base(const uint32_t* totals, int region, int nregions,
                                            uint64_t* red, uint64_t* before, uint64_t* all) {
    uint64_t a = 0, c = 0;
    for (int i = threadIdx.x; i < nregions; i += blockDim.x) {
        const uint64_t v = totals[i];
        c += v;
        if (i < region) a += v;
    }
    *before = block_sum(a, red);
    *all = block_sum(c, red);
}

// 16-byte asynchronous copy from global to shared memory (both 16-byte aligned).
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"((uint32_t)__cvta_generic_to_shared(sdst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

constexpr uint32_t kStage = 32768;     // compaction staging bytes per CTA

// ---- encode 3: place every stream at its prefix-sum offset ----
// grid (nb_max * 2L * split, chunks), block as the coder of a whole region
// (every CTA scans the region's lengths).  CTA `part` moves the streams of
// channels [part H / split, (part + 1) H / split) in batches that fit the
// staging buffer: the batch's slots are copied into shared memory with 16-byte
// asynchronous copies (many in flight: the slots were just written and every
// read waits on memory), then each stream is written to its byte offset in the
// blob from there.  Shared memory: uint32 off[H], len[H], kStage + 16 bytes of
// staging.
__global__ void __launch_bounds__(kMaxThreads) cg_compact_kernel(const __grid_constant__ CgParams p) {
    __shared__ uint64_t red[32];
    __shared__ uint32_t sred[64];
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t* off = reinterpret_cast<uint32_t*>(smem);
    uint32_t* lens = off + p.H;
    const int gi = blockIdx.y, n = p.ntok[gi], H = p.H, L = p.L, S = p.split;
    const int region = blockIdx.x / S, part = blockIdx.x % S, b = region / (2 * L);
    const int nb = batches_of(n), nregions = nb * 2 * L;
    if (b >= nb) return;
    uint8_t* blob = p.blob_ptrs[gi];
    if (!chunk_ok(p, gi)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) p.sizes[gi] = 0;     // nothing was encoded
        return;
    }
    const int tid = threadIdx.x;
    const bool active = tid < H / kStreams;
    uint64_t before, all;
    region_base(reinterpret_cast<const uint32_t*>(p.ws + p.tot_off[gi]), region, nregions, red,
                &before, &all);
    const uint64_t bytes0 = bytes_offset(L, n, H, p.cdf_entries);
    if (blockIdx.x == 0 && tid == 0) p.sizes[gi] = bytes0 + all;

    const uint32_t* lengths = reinterpret_cast<const uint32_t*>(blob + lengths_offset(L, n, p.cdf_entries)) +
                              (uint64_t)region * H;
    uint32_t l[kStreams] = {0, 0, 0, 0}, o[kStreams];
    if (active)
#pragma unroll
        for (int j = 0; j < kStreams; ++j) l[j] = lengths[chan(tid, j, H)];
    stream_offsets(l, sred, o);
    if (active)
#pragma unroll
        for (int j = 0; j < kStreams; ++j) {
            off[chan(tid, j, H)] = o[j];
            lens[chan(tid, j, H)] = l[j];
        }
    __syncthreads();
    const uint32_t stride = (uint32_t)slot_stride(n);
    uint8_t* dst0 = blob + bytes0 + before;
    const uint8_t* src0 = p.ws + p.slot_off[gi] + (uint64_t)region * H * stride;
    uint8_t* stage = smem + (size_t)H * 8;          // 16-byte aligned (H % 4 == 0)
    const uint32_t lane = tid & 31;
    const int warp = tid >> 5, nw = (blockDim.x + 31) >> 5;
    const int span = H / S, ce = (part + 1) * span;
    for (int c = part * span; c < ce;) {
        // The batch [c, e): stream x goes to stage + pos(x), pos(x) =
        // roundup16(off[x] - off[c]) + 16 (x - c), which leaves room for its
        // roundup16(len) copied bytes before pos(x + 1).  So "fits" (pos(x)
        // + roundup16(len[x]) <= kStage) holds for a prefix of the streams,
        // always including x = c (a stream is at most 578 bytes).
        const uint32_t base = off[c];
        auto pos = [&](int x) { return ((off[x] - base + 15u) & ~15u) + 16u * (uint32_t)(x - c); };
        int e = c;
        for (int x0 = c; x0 < ce; x0 += blockDim.x) {
            const int x = x0 + tid;
            const bool fits = x < ce && pos(x) + ((lens[x] + 15u) & ~15u) <= kStage;
            const int k = __syncthreads_count(fits);
            e += k;
            if (k < (int)blockDim.x) break;
        }
        // copy in: 8 lanes per stream, 16 bytes each
        for (int x = c + (tid >> 3); x < e; x += (int)blockDim.x >> 3) {
            const uint32_t chunks = (lens[x] + 15u) >> 4, at = pos(x);
            for (uint32_t j = tid & 7; j < chunks; j += 8)
                cp_async16(stage + at + 16 * j, src0 + (uint64_t)x * stride + 16 * j);
        }
        cp_async_wait_all();
        __syncthreads();
        // copy out: a warp per stream.  The destination is byte-aligned: the
        // bytes before its first 4-byte boundary and after its last are
        // written one by one (those words are shared with the neighbouring
        // streams), the words in between whole, each assembled from two
        // aligned words of the staged copy.
        for (int x = c + warp; x < e; x += nw) {
            const uint32_t len = lens[x];
            const uint8_t* src = stage + pos(x);
            uint8_t* dst = dst0 + off[x];
            uint32_t head = (uint32_t)(-reinterpret_cast<uintptr_t>(dst)) & 3u;
            head = head < len ? head : len;
            const uint32_t words = (len - head) >> 2;
            const uint32_t body = head + 4 * words, tail = len - body;
            if (lane < head) dst[lane] = src[lane];
            if (lane < tail) dst[body + lane] = src[body + lane];
            const uint32_t* sw = reinterpret_cast<const uint32_t*>(src);
            uint32_t* dw = reinterpret_cast<uint32_t*>(dst + head);
            for (uint32_t i = lane; i < words; i += 32) {
                const uint32_t lo = sw[i], hi = sw[i + 1];   // at most 4 bytes past the copy: in the buffer
                dw[i] = head ? __funnelshift_r(lo, hi, 8 * head) : lo;
            }
        }
        __syncthreads();                                  // the buffer is reused
        c = e;
    }
}

// ---- decode 1: per-region totals of the stream lengths ----
// grid (nb_max * 2L, chunks), 256 threads.
__global__ void __launch_bounds__(256) cg_total_kernel(const __grid_constant__ CgParams p) {
    __shared__ uint64_t red[32];
    const int gi = blockIdx.y, n = p.ntok[gi], H = p.H, L = p.L;
    const int region = blockIdx.x;
    if (region / (2 * L) >= batches_of(n)) return;
    const uint8_t* blob = p.blob_ptrs[gi];
    if (!chunk_ok(p, gi)) {
        if (threadIdx.x == 0) set_status(p.status, LMKV_ERR_BAD_POINTER);
        return;
    }
    const uint32_t* lengths = reinterpret_cast<const uint32_t*>(blob + lengths_offset(L, n, p.cdf_entries)) +
                              (uint64_t)region * H;
    uint64_t a = 0;
    for (int c = threadIdx.x; c < H; c += blockDim.x) a += lengths[c];
    a = block_sum(a, red);
    if (threadIdx.x == 0) {
        // a region total above its streams' bound cannot come from the encoder
        const int nt = n - (region / (2 * L)) * kBatch;
        const uint64_t cap = (uint64_t)H * stream_bound(nt < kBatch ? nt : kBatch);
        reinterpret_cast<uint32_t*>(p.ws + p.tot_off[gi])[region] = a > cap ? 0xFFFFFFFFu : (uint32_t)a;
    }
}

// Decode this thread's kStreams streams over the batch's nt tokens and write
// the dequantised rows.
// The table holds this CTA's Hl channels (thread tl's at chan(tl, j, Hl)).
template <int kSteps>
__device__ __forceinline__ void decode_rows(const uint8_t* blob, uint32_t size, uint32_t start,
                                            const uint32_t (&o)[kStreams], const uint16_t* table, int tid,
                                            int tl, int H, int Hl, int nsym, const float* deq,
                                            const float* max1s, int nt, Rows& rows, bool& bad_row) {
    Dec d[kStreams];
    const uint16_t* tab[kStreams];
#pragma unroll
    for (int j = 0; j < kStreams; ++j) {
        dec_init(d[j], blob, start + o[j], size);
        tab[j] = table + chan(tl, j, Hl);
    }
    for (int t = 0; t < nt; ++t) {
        const float m = max1s[t];
        float y[kStreams];
#pragma unroll
        for (int j = 0; j < kStreams; ++j)
            y[j] = __fmul_rn(deq[dec_symbol<kSteps>(d[j], tab[j], Hl, nsym, blob, size)], m);
        uint8_t* row = const_cast<uint8_t*>(rows_ptr(rows));
        if (row != nullptr) {
            *reinterpret_cast<__nv_bfloat162*>(row + 4 * tid) = __floats2bfloat162_rn(y[0], y[1]);
            *reinterpret_cast<__nv_bfloat162*>(row + H + 4 * tid) = __floats2bfloat162_rn(y[2], y[3]);
        } else {
            bad_row = true;                        // a bad block id: the row is not written
        }
        rows_next(rows, t + 1 < nt);
    }
}

// Sum over the region's lengths (H of them) of those channels c with
// lo <= c < hi, for each of three ranges; every thread gets the sums.
__device__ __forceinline__ void range_sums(const uint32_t* lengths, int H, const int (&lo)[3],
                                           const int (&hi)[3], uint64_t* red, uint64_t (&out)[3]) {
    uint64_t a[3] = {0, 0, 0};
    for (int c = threadIdx.x; c < H; c += blockDim.x) {
        const uint32_t v = lengths[c];
#pragma unroll
        for (int i = 0; i < 3; ++i) a[i] += (c >= lo[i] && c < hi[i]) ? v : 0u;
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) out[i] = block_sum(a[i], red);
}

// ---- decode 2: the decoders of one (chunk, batch, kv, layer) region ----
// grid (nb_max * 2L * split, chunks): CTA `part` of a region runs the threads
// [part * Tl, (part + 1) * Tl) (Tl = H / kStreams / split).  Shared memory:
// uint16 table[16 or 32][H / split].
template <int kThreads>
__global__ void __launch_bounds__(kThreads, kThreads == 256 ? 3 : 1)
cg_decode_kernel(const __grid_constant__ CgParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint64_t red[32];
    __shared__ uint32_t sred[64];
    __shared__ float deq[32];
    __shared__ float max1s[kBatch];
    const int gi = blockIdx.y, n = p.ntok[gi], H = p.H, L = p.L, S = p.split;
    const int region = blockIdx.x / S, part = blockIdx.x % S, b = region / (2 * L), s = region % (2 * L);
    const int nb = batches_of(n), nregions = nb * 2 * L;
    if (b >= nb) return;
    const uint8_t* blob = p.blob_ptrs[gi];
    if (!chunk_ok(p, gi)) return;   // reported by the totals kernel
    const int Hl = H / S, Tl = Hl / kStreams;
    const int tl = threadIdx.x, tid = part * Tl + tl;
    const bool active = tl < Tl;
    const int bins = p.bins[s], MAX = bins / 2 - 1, nsym = 2 * MAX + 1;
    const int t0 = b * kBatch, nt = n - t0 < kBatch ? n - t0 : kBatch;

    uint64_t before, all;
    region_base(reinterpret_cast<const uint32_t*>(p.ws + p.tot_off[gi]), region, nregions, red,
                &before, &all);
    const uint64_t bytes0 = bytes_offset(L, n, H, p.cdf_entries);
    const uint64_t size = p.sizes[gi];
    if (bytes0 + all != size) {          // the lengths do not add up to the blob
        if (tl == 0 && part == 0) set_status(p.status, LMKV_ERR_BAD_DATA);
        return;
    }
    uint16_t* table = reinterpret_cast<uint16_t*>(smem);
    if (active) load_table_part(table, blob, p, s, n, nsym, tid, tl, Hl, nsym > 16 ? 32 : 16);
    if (tl < nsym) deq[tl] = __fdiv_rn((float)(tl - MAX), (float)MAX);
    const float* max1 = reinterpret_cast<const float*>(blob) + (uint64_t)s * n + t0;
    for (int t = tl; t < nt; t += blockDim.x) max1s[t] = max1[t];

    const uint32_t* lengths = reinterpret_cast<const uint32_t*>(blob + lengths_offset(L, n, p.cdf_entries)) +
                              (uint64_t)region * H;
    uint32_t l[kStreams] = {0, 0, 0, 0}, o[kStreams];
    if (active)
#pragma unroll
        for (int j = 0; j < kStreams; ++j) l[j] = lengths[chan(tid, j, H)];
    // The streams lie in channel order.  Within each half of the row the
    // thread's pair follows those of the threads before it in this CTA (the
    // scans) and, with a split, the 2 part Tl channels of the CTAs before it.
    uint32_t tot0, tot1;
    const uint32_t s0 = block_scan(l[0] + l[1], sred, &tot0);   // also orders the shared-memory writes above
    const uint32_t s1 = block_scan(l[2] + l[3], sred + 32, &tot1);
    uint32_t first = 0, second = tot0;
    if (S > 1) {
        const int lo[3] = {0, H / 2, 0}, hi[3] = {2 * part * Tl, H / 2 + 2 * part * Tl, H / 2};
        uint64_t sums[3];
        range_sums(lengths, H, lo, hi, red, sums);
        first = (uint32_t)sums[0];
        second = (uint32_t)(sums[2] + sums[1]);
    }
    o[0] = first + s0;
    o[1] = o[0] + l[0];
    o[2] = second + s1;
    o[3] = o[2] + l[2];
    if (!active) return;
    const uint64_t bound = stream_bound(nt);
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kStreams; ++j) bad |= l[j] > bound;
    if (bad) {
        set_status(p.status, LMKV_ERR_BAD_DATA);
        return;
    }
    const uint32_t start = (uint32_t)(bytes0 + before);
    Rows rows;
    rows_init(rows, p, gi, s, n, t0);
    bool bad_row = false;
    if (nsym > 16)
        decode_rows<5>(blob, (uint32_t)size, start, o, table, tid, tl, H, Hl, nsym, deq, max1s, nt, rows,
                       bad_row);
    else
        decode_rows<4>(blob, (uint32_t)size, start, o, table, tid, tl, H, Hl, nsym, deq, max1s, nt, rows,
                       bad_row);
    if (bad_row && tl == 0) set_status(p.status, LMKV_ERR_BAD_BLOCK);
}

// ---- host side ----

int check_shape(int32_t L, int32_t H, const int32_t* bins, int32_t* cdf_prefix, int32_t* cdf_entries,
                int* max_nsym) {
    if (L < 1 || L > LMKV_CACHEGEN_MAX_LAYERS || H < 4 || H > LMKV_CACHEGEN_MAX_CHANNELS || H % 4 != 0 ||
        bins == nullptr)
        return LMKV_ERR_INVALID_ARG;
    int64_t e = 0;
    int mx = 0;
    for (int s = 0; s < 2 * L; ++s) {
        if (bins[s] < 4 || bins[s] > 32) return LMKV_ERR_INVALID_ARG;
        if (cdf_prefix) cdf_prefix[s] = (int32_t)e;
        e += (int64_t)H * (nsym_of(bins[s]) - 1);
        mx = nsym_of(bins[s]) > mx ? nsym_of(bins[s]) : mx;
    }
    if (cdf_entries) *cdf_entries = (int32_t)e;
    if (max_nsym) *max_nsym = mx;
    return LMKV_OK;
}

// Workspace of one chunk: [totals | symbols | slots], each 256-byte aligned.
struct ChunkWs {
    uint64_t tot, sym, slot, end;
};

ChunkWs chunk_ws(uint64_t at, int L, int H, int n) {
    auto up = [](uint64_t v) { return (v + 255) & ~255ull; };
    const uint64_t nregions = (uint64_t)batches_of(n) * 2 * L;
    ChunkWs w;
    w.tot = up(at);
    w.sym = up(w.tot + 4 * nregions);
    w.slot = up(w.sym + 2ull * L * n * H);
    w.end = w.slot + nregions * H * slot_stride(n);
    return w;
}

int workspace_size(int32_t L, int32_t H, const int32_t* ntok, int32_t num_chunks, uint64_t* out) {
    if (num_chunks < 0 || (num_chunks > 0 && ntok == nullptr)) return LMKV_ERR_INVALID_ARG;
    uint64_t at = 0;
    for (int32_t g = 0; g < num_chunks; ++g) {
        if (ntok[g] < 1 || ntok[g] > LMKV_CACHEGEN_MAX_TOKENS) return LMKV_ERR_INVALID_ARG;
        at = chunk_ws(at, L, H, ntok[g]).end;
    }
    *out = at;
    return LMKV_OK;
}

int threads_for(int H) { return ((H / kStreams + 31) / 32) * 32; }

// CTAs per unit of work (a slice for the CDF pass, a region for the coder,
// compaction and decoder), among the splits that leave every CTA a whole
// number of warps of threads.  Measured on 32 layers x 1024 channels with
// 256-token chunks (64 units a chunk): 4 CTAs a unit are fastest while the
// units do not fill two CTAs per SM (up to 4 chunks: 1 chunk encodes in
// 0.26 ms against 0.37 ms with one CTA), 2 CTAs from there on (within 1 % of
// the best from 6 to 40 chunks; the 128-thread CTAs balance better over the
// SMs than 256-thread ones, 64-thread ones cost more per CTA).
int choose_split(int64_t units, int H, int sms) {
    auto whole_warps = [H](int S) { return H % (kStreams * S) == 0 && (H / (kStreams * S)) % 32 == 0; };
    if (units <= 2 * (int64_t)sms && whole_warps(4)) return 4;
    return whole_warps(2) ? 2 : 1;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return 0;
    return n;
}

// Allow the largest dynamic shared memory any codec call can need and ask for
// the largest shared memory carve-out, so that as many CTAs fit per SM as
// their tables allow.  Done once per (device, kernel), so that later calls
// (and calls inside a stream capture) make no attribute call at all.
int set_smem(const void* fn) {
    static std::mutex mu;
    static std::set<std::pair<int, const void*>> done;
    int dev = 0;
    if (lmkv_internal_cuda_status(cudaGetDevice(&dev)) != LMKV_OK) return LMKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({dev, fn})) return LMKV_OK;
    const size_t most = (size_t)32 * LMKV_CACHEGEN_MAX_CHANNELS * 2;    // 32 table rows of 2-byte entries
    if (lmkv_internal_cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                      (int)most)) != LMKV_OK ||
        lmkv_internal_cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                      cudaSharedmemCarveoutMaxShared)) != LMKV_OK)
        return LMKV_ERR_CUDA;
    done.insert({dev, fn});
    return LMKV_OK;
}

enum class Dir { kEncode, kDecode };

// The pool form of a call: rows come from / go to the pages of the listed chunks.
struct PoolForm {
    const lmkv_pool_t* pool;
    const int32_t* block_table;
    int32_t max_blocks;
    const std::vector<LmkvChunkRef>* chunks;
};

int run(Dir dir, void* const* chunk_ptrs, void* const* blob_ptrs, uint64_t* sizes, const int32_t* ntok,
        int32_t num_chunks, int32_t L, int32_t H, const int32_t* bins, void* workspace,
        uint64_t workspace_bytes, int32_t* d_status, void* stream, const PoolForm* pf = nullptr) {
    CgParams p{};
    int max_nsym = 0;
    int rc = check_shape(L, H, bins, p.cdf_prefix, &p.cdf_entries, &max_nsym);
    if (rc != LMKV_OK) return rc;
    if (num_chunks < 0) return LMKV_ERR_INVALID_ARG;
    if (num_chunks == 0) return LMKV_OK;
    if ((chunk_ptrs == nullptr && pf == nullptr) || blob_ptrs == nullptr || sizes == nullptr ||
        ntok == nullptr || workspace == nullptr)
        return LMKV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return LMKV_ERR_MISALIGNED;
    uint64_t need = 0;
    rc = workspace_size(L, H, ntok, num_chunks, &need);
    if (rc != LMKV_OK) return rc;
    for (int32_t g = 0; g < num_chunks; ++g) {
        lmkv_cachegen_layout_t lay;
        rc = lmkv_cachegen_layout(L, ntok[g], H, bins, &lay);
        if (rc != LMKV_OK) return rc;
    }
    if (need > workspace_bytes) return LMKV_ERR_INVALID_ARG;
    for (int s = 0; s < 2 * L; ++s) p.bins[s] = (uint8_t)bins[s];
    p.L = L;
    p.H = H;
    p.status = d_status;
    p.ws = static_cast<uint8_t*>(workspace);
    if (pf != nullptr) {
        p.layer_base = reinterpret_cast<const uint8_t* const*>(pf->pool->layer_base);
        p.block_table = pf->block_table;
        p.num_blocks = pf->pool->num_blocks;
        p.bt_stride = pf->max_blocks;
        p.block_size = pf->pool->block_size;
    }
    const int threads = threads_for(H);
    const int sms = sm_count();
    if (sms == 0) {
        lmkv_internal_cuda_status(cudaGetLastError());
        return LMKV_ERR_CUDA;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dir == Dir::kEncode) {
        if (set_smem((const void*)cg_cdf_kernel) != LMKV_OK || set_smem((const void*)cg_code_kernel<512>) != LMKV_OK ||
            set_smem((const void*)cg_code_kernel<256>) != LMKV_OK || set_smem((const void*)cg_compact_kernel) != LMKV_OK)
            return LMKV_ERR_CUDA;
    } else if (set_smem((const void*)cg_decode_kernel<512>) != LMKV_OK ||
               set_smem((const void*)cg_decode_kernel<256>) != LMKV_OK) {
        return LMKV_ERR_CUDA;
    }
    uint64_t at = 0;
    for (int32_t g0 = 0; g0 < num_chunks; g0 += kMaxChunks) {
        const int cnt = num_chunks - g0 < kMaxChunks ? num_chunks - g0 : kMaxChunks;
        int nb_max = 0;
        for (int i = 0; i < cnt; ++i) {
            const int n = ntok[g0 + i];
            const ChunkWs w = chunk_ws(at, L, H, n);
            p.ntok[i] = n;
            p.tot_off[i] = w.tot;
            p.sym_off[i] = w.sym;
            p.slot_off[i] = w.slot;
            if (pf != nullptr) {
                p.chunk_req[i] = (*pf->chunks)[g0 + i].req;
                p.chunk_tok0[i] = (*pf->chunks)[g0 + i].tok0;
            }
            at = w.end;
            nb_max = batches_of(n) > nb_max ? batches_of(n) : nb_max;
        }
        p.nchunks = cnt;
        p.chunk_ptrs = chunk_ptrs ? reinterpret_cast<const uint8_t* const*>(chunk_ptrs) + g0 : nullptr;
        p.blob_ptrs = reinterpret_cast<uint8_t* const*>(blob_ptrs) + g0;
        p.sizes = sizes + g0;
        int64_t units = 0;
        for (int i = 0; i < cnt; ++i) units += (int64_t)batches_of(p.ntok[i]) * 2 * L;
        const int S = choose_split(units, H, sms);
        p.split = S;
        const int part_threads = threads_for(H / S);       // = H / (kStreams S) when S > 1
        const size_t table_bytes = (size_t)max_nsym * (H / S) * 2;
        const size_t search_bytes = (size_t)(max_nsym > 16 ? 32 : 16) * (H / S) * 2;
        const dim3 regions(nb_max * 2 * L * S, cnt);
        if (dir == Dir::kEncode) {
            // one cluster of S CTAs per slice
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            cfg.gridDim = dim3(2 * L * S, cnt);
            cfg.blockDim = dim3(threads);
            cfg.dynamicSmemBytes = (size_t)max_nsym * H * 2;
            cfg.stream = st;
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = S;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = S > 1 ? 1 : 0;
            if (lmkv_internal_cuda_status(cudaLaunchKernelEx(&cfg, cg_cdf_kernel, p)) != LMKV_OK)
                return LMKV_ERR_CUDA;
            if (part_threads > 256) cg_code_kernel<512><<<regions, part_threads, table_bytes, st>>>(p);
            else cg_code_kernel<256><<<regions, part_threads, table_bytes, st>>>(p);
            cg_compact_kernel<<<regions, threads, (size_t)H * 8 + kStage + 16, st>>>(p);
            lmkv_internal_add_launches(3);
        } else {
            cg_total_kernel<<<dim3(nb_max * 2 * L, cnt), 256, 0, st>>>(p);
            if (part_threads > 256) cg_decode_kernel<512><<<regions, part_threads, search_bytes, st>>>(p);
            else cg_decode_kernel<256><<<regions, part_threads, search_bytes, st>>>(p);
            lmkv_internal_add_launches(2);
        }
        if (lmkv_internal_cuda_status(cudaGetLastError()) != LMKV_OK) return LMKV_ERR_CUDA;
    }
    return LMKV_OK;
}

}  // namespace

extern "C" {

int lmkv_cachegen_default_bins(int32_t num_layers, int32_t* bins) {
    if (num_layers < 1 || num_layers > LMKV_CACHEGEN_MAX_LAYERS || bins == nullptr) return LMKV_ERR_INVALID_ARG;
    const bool all32 = num_layers < 10;
    for (int32_t l = 0; l < num_layers; ++l) {
        bins[l] = (all32 || l < 10) ? 32 : 16;
        bins[num_layers + l] = (all32 || l < 2) ? 32 : 16;
    }
    return LMKV_OK;
}

int lmkv_cachegen_layout(int32_t num_layers, int32_t num_tokens, int32_t channels, const int32_t* bins,
                         lmkv_cachegen_layout_t* out) {
    int32_t entries = 0;
    const int rc = check_shape(num_layers, channels, bins, nullptr, &entries, nullptr);
    if (rc != LMKV_OK) return rc;
    if (out == nullptr || num_tokens < 1 || num_tokens > LMKV_CACHEGEN_MAX_TOKENS) return LMKV_ERR_INVALID_ARG;
    out->max1_offset = 0;
    out->cdf_offset = cdf_offset(num_layers, num_tokens);
    out->lengths_offset = lengths_offset(num_layers, num_tokens, entries);
    out->bytes_offset = bytes_offset(num_layers, num_tokens, channels, entries);
    uint64_t bound = out->bytes_offset;
    for (int t0 = 0; t0 < num_tokens; t0 += kBatch) {
        const int nt = num_tokens - t0 < kBatch ? num_tokens - t0 : kBatch;
        bound += 2ull * num_layers * channels * stream_bound(nt);
    }
    out->max_bytes = bound;
    // the kernels address a blob with 32-bit offsets
    return bound <= kMaxBlobBytes ? LMKV_OK : LMKV_ERR_INVALID_ARG;
}

int lmkv_cachegen_workspace_bytes(int32_t num_layers, int32_t channels, const int32_t* num_tokens,
                                  int32_t num_chunks, uint64_t* bytes) {
    if (bytes == nullptr || num_layers < 1 || num_layers > LMKV_CACHEGEN_MAX_LAYERS || channels < 4 ||
        channels > LMKV_CACHEGEN_MAX_CHANNELS || channels % 4 != 0)
        return LMKV_ERR_INVALID_ARG;
    return workspace_size(num_layers, channels, num_tokens, num_chunks, bytes);
}

int lmkv_cachegen_encode(void* const* chunk_ptrs, const int32_t* num_tokens, int32_t num_chunks,
                         int32_t num_layers, int32_t channels, const int32_t* bins,
                         void* const* blob_ptrs, uint64_t* sizes, void* workspace,
                         uint64_t workspace_bytes, int32_t* d_status, void* stream) {
    return run(Dir::kEncode, chunk_ptrs, blob_ptrs, sizes, num_tokens, num_chunks, num_layers, channels,
               bins, workspace, workspace_bytes, d_status, stream);
}

int lmkv_cachegen_decode(void* const* blob_ptrs, const uint64_t* sizes, const int32_t* num_tokens,
                         int32_t num_chunks, int32_t num_layers, int32_t channels,
                         const int32_t* bins, void* const* chunk_ptrs, void* workspace,
                         uint64_t workspace_bytes, int32_t* d_status, void* stream) {
    return run(Dir::kDecode, chunk_ptrs, blob_ptrs, const_cast<uint64_t*>(sizes), num_tokens, num_chunks,
               num_layers, channels, bins, workspace, workspace_bytes, d_status, stream);
}

// The pool forms: the chunks of a store / retrieve call, enumerated and
// validated as lmkv_gather_chunks does.
static int pool_entry(Dir dir, const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                      const int64_t* start, const int64_t* end, int32_t num_req, int32_t chunk_size,
                      int32_t save_unfull_chunk, const int32_t* bins, void* const* blob_ptrs,
                      uint64_t* sizes, void* workspace, uint64_t workspace_bytes, int32_t* d_status,
                      void* stream) {
    std::vector<LmkvChunkRef> chunks;
    const int rc = lmkv_internal_list_chunks(pool, block_table, max_blocks, start, end, num_req, chunk_size,
                                             save_unfull_chunk, &chunks);
    if (rc != LMKV_OK) return rc;
    if (pool->elem_bytes != 2) return LMKV_ERR_UNSUPPORTED;
    std::vector<int32_t> ntok(chunks.size());
    for (size_t g = 0; g < chunks.size(); ++g) ntok[g] = chunks[g].n;
    const PoolForm pf{pool, block_table, max_blocks, &chunks};
    return run(dir, nullptr, blob_ptrs, sizes, ntok.data(), (int32_t)chunks.size(), pool->num_layers,
               pool->num_kv_heads * pool->head_dim, bins, workspace, workspace_bytes, d_status, stream, &pf);
}

int lmkv_cachegen_store_chunks(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                               const int64_t* start, const int64_t* end, int32_t num_req, int32_t chunk_size,
                               int32_t save_unfull_chunk, const int32_t* bins, void* const* blob_ptrs,
                               uint64_t* sizes, void* workspace, uint64_t workspace_bytes, int32_t* d_status,
                               void* stream) {
    return pool_entry(Dir::kEncode, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                      save_unfull_chunk, bins, blob_ptrs, sizes, workspace, workspace_bytes, d_status, stream);
}

int lmkv_cachegen_retrieve_chunks(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                                  const int64_t* start, const int64_t* end, int32_t num_req,
                                  int32_t chunk_size, int32_t save_unfull_chunk, const int32_t* bins,
                                  void* const* blob_ptrs, const uint64_t* sizes, void* workspace,
                                  uint64_t workspace_bytes, int32_t* d_status, void* stream) {
    return pool_entry(Dir::kDecode, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                      save_unfull_chunk, bins, blob_ptrs, const_cast<uint64_t*>(sizes), workspace,
                      workspace_bytes, d_status, stream);
}

}  // extern "C"
