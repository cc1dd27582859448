// lmkv_kernels.cuh -- sm_103a kernels for the paged-KV chunk gather / scatter.
//
// The movement ("LMCache: An Efficient KV Cache Layer for Enterprise-Scale
// LLM Inference", section on the configurable chunk size): a
// kernel copies the scattered pages of many layers into a contiguous chunk
// buffer on store and splits chunk buffers back into pages on load.  With
// chunk_size a multiple of block_size, every (chunk, K/V, layer, block)
// pair is one contiguous run of rows on BOTH sides: block_size rows of the
// pool page and the matching rows of the chunk tile X_g[kv][l].  The unit of
// work ("item") is such a run, optionally split into equal parts.
//
// Item numbering is chunk-major so that consecutive items touch consecutive
// bytes of the chunk buffers:
//   item = (((g * 2 + kv) * layer_n + ll) * blocks_per_chunk + j) * parts + q
//
// Copies use move_lsu_kernel: CTA-wide 16-byte vector loads into registers,
// then stores, one CTA per item (grid-stride when the grid is capped).  (A
// TMA bulk-copy engine -- cp.async.bulk global->shared->global through a ring
// of shared-memory stages -- measured slower on GB300 for every stage count
// and grid shape tried, for whole-batch and per-layer calls.)
// The fp8 variant quantises one (chunk, K/V, layer) tile per thread-block
// cluster: each CTA stages its rows in registers and in shared memory (TMA
// bulk copies), and the absmax is reduced across the cluster through
// distributed shared memory, so HBM is read once.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <cooperative_groups.h>

namespace lmkv {

constexpr int kStatusBadBlock = 5;    // LMKV_ERR_BAD_BLOCK
constexpr int kStatusBadPointer = 6;  // LMKV_ERR_BAD_POINTER
constexpr int kStatusTimeout = 7;     // LMKV_ERR_TIMEOUT (bounded waits gave up)

// By-value launch parameters (kept in the constant bank via __grid_constant__).
// kCap = requests one launch can carry; calls with few requests use a small
// block so the launch copies a few hundred bytes of parameters, not kilobytes.
template <int kCap>
struct BatchT {
    static constexpr int kCapacity = kCap;
    const uint8_t* const* layer_base;   // DEVICE [num_layers] pool layer bases
    uint8_t* const* chunk_ptrs;         // DEVICE [total chunks] chunk (or code) buffers
    const int32_t* block_table;         // DEVICE [num_req_total][bt_stride]
    int32_t* status;                    // DEVICE int32 or null
    float* scales;                      // DEVICE [total chunks][2][L] (fp8 only)
    int64_t num_blocks;
    int64_t bt_stride;
    int32_t num_layers;
    int32_t row_bytes;                  // pool row bytes (HD * elem_bytes)
    int32_t block_size;
    int32_t chunk_size;
    int32_t blocks_per_chunk;           // chunk_size / block_size
    int32_t parts;                      // items per (chunk, kv, layer, block); divides block_size
    int32_t layer_lo;                   // first layer moved
    int32_t layer_n;                    // number of layers moved
    int32_t num_req;                    // requests packed in this launch (all with >= 1 chunk)
    int32_t chunk_base;                 // global index of this launch's chunk 0
    int32_t num_chunks;                 // chunks in this launch
    int32_t prefetch_ahead;             // copy kernel: L2 prefetch distance in items (0 = none)
    uint8_t* staging;                   // DEVICE one-layer staging buffer, or null (see item_run)
    int64_t stage_tok_base;             // enumerated tokens of the call before this launch
    int64_t req_tok0[kCap];             // first enumerated token of packed request i
    int64_t req_tok_prefix[kCap];       // enumerated tokens of packed requests before i
    int64_t req_tok_end[kCap];          // end (exclusive) of its enumerated tokens
    int32_t req_row[kCap];              // its block-table row
    int32_t req_col0[kCap];             // block-table column of its first token (tok0 / B)
    int32_t req_chunk_begin[kCap + 1];  // local chunk index of its first chunk
};

constexpr int kSmallBatch = 8;
constexpr int kMaxReqPerLaunch = 256;
using BatchSmall = BatchT<kSmallBatch>;
using Batch = BatchT<kMaxReqPerLaunch>;

template <class B>
__host__ __device__ inline int64_t batch_items(const B& p) {
    return (int64_t)p.num_chunks * 2 * p.layer_n * p.blocks_per_chunk * p.parts;
}

// Programmatic dependent launch: let the next kernel on the stream be
// scheduled during this one's tail, and wait for every prerequisite grid
// (complete, memory visible) before touching global memory.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// x / d for a runtime divisor that is usually a power of two.
struct UDiv {
    uint32_t d;
    int32_t shift;      // log2(d) when d is a power of two, else -1
    __device__ __forceinline__ explicit UDiv(uint32_t dv) : d(dv), shift(-1) {
#ifdef __CUDA_ARCH__
        if (__popc(dv) == 1) shift = __ffs(dv) - 1;
#endif
    }
    __device__ __forceinline__ uint32_t div(uint32_t x) const { return shift >= 0 ? x >> shift : x / d; }
};

struct ChunkRef {
    int32_t req_row;
    int32_t ntok;
    int32_t col0;       // block-table column of the chunk's first token
    int32_t req;        // packed request index in the launch
    int64_t tok0;
};

// Chunk gl (local) -> its request: the last packed request whose first chunk <= gl.
template <class B>
__device__ __forceinline__ ChunkRef resolve_chunk(const B& p, int32_t gl) {
    int lo = 0, hi = p.num_req - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (p.req_chunk_begin[mid] <= gl) lo = mid; else hi = mid - 1;
    }
    ChunkRef c;
    c.req = lo;
    c.req_row = p.req_row[lo];
    c.tok0 = p.req_tok0[lo] + (int64_t)(gl - p.req_chunk_begin[lo]) * p.chunk_size;
    c.col0 = p.req_col0[lo] + (gl - p.req_chunk_begin[lo]) * p.blocks_per_chunk;
    int64_t left = p.req_tok_end[lo] - c.tok0;
    c.ntok = (int32_t)(left < p.chunk_size ? left : p.chunk_size);
    return c;
}

template <class B>
__device__ __forceinline__ void report(const B& p, int code) {
    if (p.status != nullptr) atomicCAS(p.status, 0, code);
}

// One item's two runs.  Returns false (after reporting, if it is an error)
// when the item has nothing to move.
struct Run {
    uint8_t* pool;
    uint8_t* chunk;
    uint32_t bytes;
    int32_t kv, ll, gl;     // the item's K/V half, layer (within the call) and local chunk
};

// item -> (chunk gl, kv, layer ll, page j, part q).  Items below 2^32 (every
// launch in practice) are split with 32-bit shifts or divisions: the 64-bit
// divisions by runtime values are a long serial chain at the start of every
// CTA.
template <class B>
__device__ __forceinline__ void decode_item(const B& p, int64_t item, int& q, int& j, int& ll,
                                            int& kv, int& gl) {
    if (item <= 0xFFFFFFFFll) {
        const UDiv dq((uint32_t)p.parts), dj((uint32_t)p.blocks_per_chunk), dl((uint32_t)p.layer_n);
        const uint32_t i0 = (uint32_t)item;
        const uint32_t i1 = dq.div(i0), i2 = dj.div(i1), i3 = dl.div(i2);
        q = (int)(i0 - i1 * (uint32_t)p.parts);
        j = (int)(i1 - i2 * (uint32_t)p.blocks_per_chunk);
        ll = (int)(i2 - i3 * (uint32_t)p.layer_n);
        kv = (int)(i3 & 1u);
        gl = (int)(i3 >> 1);
    } else {
        q = (int)(item % p.parts);
        int64_t t = item / p.parts;
        j = (int)(t % p.blocks_per_chunk);
        t /= p.blocks_per_chunk;
        ll = (int)(t % p.layer_n);
        t /= p.layer_n;
        kv = (int)(t & 1);
        gl = (int)(t >> 1);
    }
}

template <class B, bool kReport = true>
__device__ __forceinline__ bool item_run(const B& p, int64_t item, Run& run) {
    int q, j, ll, kv, gl;
    decode_item(p, item, q, j, ll, kv, gl);
    run.kv = kv;
    run.ll = ll;
    run.gl = gl;
    const ChunkRef c = resolve_chunk(p, gl);
    const int part_rows = p.block_size / p.parts;
    const int row0 = j * p.block_size + q * part_rows;     // first row inside the chunk
    if (row0 >= c.ntok) return false;                       // past a partial chunk's end
    const int rows = min(part_rows, c.ntok - row0);
    const int l = p.layer_lo + ll;
    const int64_t col = c.col0 + j;
    const int64_t rb = p.row_bytes;
    // The block id and both base pointers are read before any of them is
    // checked, so the three loads are in flight together (every index is in
    // range whatever the values turn out to be).
    const int64_t blk = p.block_table[(int64_t)c.req_row * p.bt_stride + col];
    uint8_t* lb = const_cast<uint8_t*>(p.layer_base[l]);
    // Chunk side: chunk g's buffer [2][L][n_g][row], or -- in staging mode --
    // the one-layer staging buffer, where chunk g's [2][n_g][row] slices sit
    // at 2 * row * (tokens enumerated before chunk g).
    const bool staged = p.staging != nullptr;
    uint8_t* cb = staged ? nullptr : p.chunk_ptrs[p.chunk_base + gl];
    int64_t chunk_layers = p.num_layers, layer_slot = l;
    if (staged) {
        const int64_t tok_before = p.stage_tok_base + p.req_tok_prefix[c.req] +
                                   (int64_t)(gl - p.req_chunk_begin[c.req]) * p.chunk_size;
        cb = p.staging + 2 * rb * tok_before;
        chunk_layers = 1;
        layer_slot = 0;
    }
    if (blk < 0 || blk >= p.num_blocks) {
        if (kReport) report(p, kStatusBadBlock);
        return false;
    }
    if (lb == nullptr || cb == nullptr || ((reinterpret_cast<uintptr_t>(lb) |
                                            reinterpret_cast<uintptr_t>(cb)) & 15)) {
        if (kReport) report(p, kStatusBadPointer);
        return false;
    }
    run.pool = lb + ((kv * p.num_blocks + blk) * p.block_size + q * part_rows) * rb;
    run.chunk = cb + (((int64_t)kv * chunk_layers + layer_slot) * c.ntok + row0) * rb;
    run.bytes = (uint32_t)(rows * rb);
    return true;
}

// ---------------------------------------------------------------------------
// 16-byte global accesses with streaming cache hints.
__device__ __forceinline__ int4 ld_stream(const int4* ptr) {
    int4 r;
    asm("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(ptr));
    return r;
}

__device__ __forceinline__ void st_stream(int4* ptr, const int4& v) {
    asm volatile("st.global.cs.v4.s32 [%0], {%1, %2, %3, %4};"
                 :: "l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// CTA-wide copy of `bytes` (a multiple of 16) from src to dst.
template <int kThreads, int kUnroll>
__device__ __forceinline__ void cta_copy(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                         uint32_t bytes) {
    const int nvec = (int)(bytes >> 4);
    const int4* s = reinterpret_cast<const int4*>(src);
    int4* d = reinterpret_cast<int4*>(dst);
    for (int base = threadIdx.x; base < nvec; base += kThreads * kUnroll) {
        int4 r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = base + u * kThreads;
            if (v < nvec) r[u] = ld_stream(s + v);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = base + u * kThreads;
            if (v < nvec) st_stream(d + v, r[u]);
        }
    }
}

// L2 prefetch of `bytes` (a multiple of 16) from a 16-byte aligned global
// address, issued to the TMA unit (no registers wait for it).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}

// LSU engine.  kGather: pool -> chunk, else chunk -> pool.  Grid-stride over
// items, so the grid may be the item count (one CTA per item) or smaller.
// With p.prefetch_ahead > 0 (one-layer calls), thread 0 first asks the TMA
// unit to bring the source run of item + prefetch_ahead into L2, so the CTA
// that later takes that item finds its rows there: a one-layer call is short
// enough that the loads of its CTAs alone keep too few bytes in flight.  The
// address comes from the same checked lookup as that item's own (after the
// dependency wait); errors are left for the owning CTA to report.
template <class B, bool kGather, int kThreads, int kUnroll>
__global__ void __launch_bounds__(kThreads)
move_lsu_kernel(const __grid_constant__ B p, int64_t num_items) {
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t item = blockIdx.x; item < num_items; item += gridDim.x) {
        if (p.prefetch_ahead > 0 && threadIdx.x == 0 && item + p.prefetch_ahead < num_items) {
            Run ahead;
            if (item_run<B, false>(p, item + p.prefetch_ahead, ahead))
                bulk_prefetch_l2(kGather ? ahead.pool : ahead.chunk, ahead.bytes);
        }
        Run run;
        if (!item_run(p, item, run)) continue;
        if (kGather) cta_copy<kThreads, kUnroll>(run.pool, run.chunk, run.bytes);
        else cta_copy<kThreads, kUnroll>(run.chunk, run.pool, run.bytes);
    }
}

// ---------------------------------------------------------------------------
// TMA bulk-copy and mbarrier primitives (inline PTX).
__device__ __forceinline__ uint32_t smem_addr(const void* ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}

// Bounded wait on an mbarrier phase: false if it did not complete in time.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < (1u << 20); ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void bulk_g2s(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(sdst)), "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// fp8 e4m3 quantising gather.  One thread-block cluster of kCluster CTAs per
// tile (chunk g, kv, layer l); CTA `rank` owns rows [rank*R, rank*R + R) of the
// tile (R = ceil(n_g / kCluster)).  Values stay in registers between the
// absmax pass and the quantising pass when the slice fits in
// kThreads * kVPT vectors of 16 bytes; otherwise the rest is re-read.
// The absmax is exchanged through distributed shared memory with one split
// cluster barrier; there is no CTA-wide barrier.
constexpr int kQuantMaxRows = 256;   // rows per CTA slice (chunk_size <= kCluster * 256)

// Running max of |x| over 8 bf16 values, as bf16x2 bit patterns (the sign bit
// cleared, so max.bf16x2 of the magnitudes is exact).
__device__ __forceinline__ uint32_t absmax_bf16x8(uint32_t acc, const uint4& v) {
    const uint32_t m = 0x7FFF7FFFu;
    auto as_bf2 = [](uint32_t w) { return *reinterpret_cast<const __nv_bfloat162*>(&w); };
    __nv_bfloat162 a = __hmax2(as_bf2(v.x & m), as_bf2(v.y & m));
    __nv_bfloat162 b = __hmax2(as_bf2(v.z & m), as_bf2(v.w & m));
    a = __hmax2(__hmax2(a, b), as_bf2(acc));
    return *reinterpret_cast<const uint32_t*>(&a);
}


// Correctly rounded x / s for a per-tile constant s, from the correctly
// rounded reciprocal r = RN(1/s): q0 = RN(x*r) is within an ulp of x/s, the
// remainder q0*s - x is exact in one FMA, and one correction step
// RN(q0 - rem*r) yields RN(x/s) (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990).  The remainder is exact only while it stays out of the fp32
// subnormal range: it is a multiple of ulp(q0) * ulp(s), which needs
// exponent(q0) + exponent(s) >= -103.  With s >= 2^-90 that holds for every
// |q| >= 2^-13, and quotients below 2^-11 round to a signed e4m3 zero however
// their last bits come out; smaller scales take the IEEE division instead
// (kFastDivMinScale).
//
// The kernel evaluates the steps on y = -x, whose remainder q0*s - y is
// q0*s + x, so the unpacked x is used as it is, and under round-to-nearest
// every zero quotient keeps the sign of y.  e4m3 is sign-magnitude and its
// rounding and saturation are symmetric, so the codes of x / s are those of
// y / s with the sign bit flipped.  Two lanes at a time use the packed fp32
// pipe (mul/fma .f32x2).  The tests compare the codes exhaustively with IEEE
// division over every bf16 input and every scale a bf16 absmax can produce.
constexpr float kFastDivMinScale = 0x1p-90f;

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Four fp32 values -> four e4m3 codes (round to nearest even, saturating),
// byte i of the result from value i.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r) : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
    return r;
}
__device__ __forceinline__ uint32_t e4m3x4(uint64_t a, uint64_t b) {
    float a0, a1, b0, b1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(b0), "=f"(b1) : "l"(b));
    return e4m3x4(a0, a1, b0, b1);
}

// Per-tile constants of the quantiser.
struct QuantK {
    float scale;
    uint64_t s2;     // {s, s}
    uint64_t nr2;    // {-RN(1/s), -RN(1/s)}
};

__device__ __forceinline__ QuantK make_quant(float scale, bool fast) {
    QuantK k;
    k.scale = scale;
    const float nr = fast ? -__frcp_rn(scale) : 0.0f;
    k.s2 = f2_pack(scale, scale);
    k.nr2 = f2_pack(nr, nr);
    return k;
}

// 8 bf16 values (one 16-byte vector) -> 8 e4m3 codes.
template <bool kFastDiv>
__device__ __forceinline__ uint2 quant_bf16x8(const uint4& v, const QuantK& k) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (kFastDiv) {
            uint64_t q[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint32_t word = w[2 * h + i];
                const uint64_t x2 = f2_pack(__uint_as_float(word << 16),
                                            __uint_as_float(word & 0xFFFF0000u));
                const uint64_t q0 = f2_mul(x2, k.nr2);           // RN(y * r), y = -x
                const uint64_t rem = f2_fma(q0, k.s2, x2);       // q0 * s - y, exact
                q[i] = f2_fma(rem, k.nr2, q0);                   // RN(y / s)
            }
            out[h] = e4m3x4(q[0], q[1]) ^ 0x80808080u;           // codes of x / s
        } else {
            const uint32_t w0 = w[2 * h], w1 = w[2 * h + 1];
            out[h] = e4m3x4(__fdiv_rn(__uint_as_float(w0 << 16), k.scale),
                            __fdiv_rn(__uint_as_float(w0 & 0xFFFF0000u), k.scale),
                            __fdiv_rn(__uint_as_float(w1 << 16), k.scale),
                            __fdiv_rn(__uint_as_float(w1 & 0xFFFF0000u), k.scale));
        }
    }
    return make_uint2(out[0], out[1]);
}

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Where the CTA's vectors come from: vector v of the slice is row v / vpr,
// 16-byte column v % vpr.  With kThreads a multiple of vpr each thread keeps
// one column and steps rows by kThreads / vpr.
struct SliceMap {
    const uint8_t* kv_base;     // pool layer l, K or V half
    const int32_t* bt;          // block-table entries of the chunk (column tok0 / B)
    uint32_t r0, vpr, row_bytes, block_size, num_blocks;
    UDiv bdiv, vdiv;
    __device__ __forceinline__ SliceMap(const uint8_t* kvb, const int32_t* btc, uint32_t r0_,
                                        uint32_t vpr_, uint32_t rb, uint32_t bs, uint32_t nb)
        : kv_base(kvb), bt(btc), r0(r0_), vpr(vpr_), row_bytes(rb), block_size(bs), num_blocks(nb),
          bdiv(bs), vdiv(vpr_) {}
    // Source of slice vector v (row-major over the slice), or null for a bad block.
    __device__ __forceinline__ const uint8_t* src(uint32_t row_local, uint32_t col) const {
        const uint32_t row = r0 + row_local;
        const uint32_t jb = bdiv.div(row);
        const int32_t blk = bt[jb];
        if ((uint32_t)blk >= num_blocks) return nullptr;
        const uint32_t slot = row - jb * block_size;
        return kv_base + ((int64_t)blk * block_size + slot) * row_bytes + col * 16u;
    }
};

// Quantise the CTA's slice from registers (and re-read the part that did not
// fit), writing 8 codes per 16-byte source vector.
template <bool kFastDiv, int kThreads, int kVPT>
__device__ __forceinline__ void quant_slice(const uint4 (&regs)[kVPT], uint32_t valid, uint32_t nvec,
                                            const SliceMap& sm, uint8_t* tile_codes, const QuantK& k) {
#pragma unroll
    for (int u = 0; u < kVPT; ++u) {
        const uint32_t v = threadIdx.x + u * kThreads;
        if (v < nvec && (valid >> u) & 1u) {
            const uint2 q = k.scale == 0.0f ? make_uint2(0, 0) : quant_bf16x8<kFastDiv>(regs[u], k);
            *reinterpret_cast<uint2*>(tile_codes + (int64_t)v * 8) = q;
        }
    }
    for (uint32_t v = threadIdx.x + kVPT * kThreads; v < nvec; v += kThreads) {
        const uint32_t row = sm.vdiv.div(v);
        const uint8_t* src = sm.src(row, v - row * sm.vpr);
        if (src == nullptr) continue;
        const int4 x = ld_stream(reinterpret_cast<const int4*>(src));
        const uint4 xv = make_uint4((uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w);
        const uint2 q = k.scale == 0.0f ? make_uint2(0, 0) : quant_bf16x8<kFastDiv>(xv, k);
        *reinterpret_cast<uint2*>(tile_codes + (int64_t)v * 8) = q;
    }
}

template <class B, int kThreads, int kVPT, int kCluster>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
quant_gather_kernel(const __grid_constant__ B p) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ uint32_t warp_max[kThreads / 32];
    static_assert(kThreads / 32 <= 32, "one lane per warp slot");
    pdl_launch_dependents();
    pdl_wait();

    const int rank = (int)cluster.block_rank();
    const uint32_t tile = blockIdx.x / kCluster;
    const uint32_t ll = tile % (uint32_t)p.layer_n;
    const uint32_t kv = (tile / (uint32_t)p.layer_n) & 1u;
    const int gl = (int)(tile / (uint32_t)p.layer_n / 2u);
    const int l = p.layer_lo + (int)ll;
    const ChunkRef c = resolve_chunk(p, gl);
    const uint32_t rows_per = (uint32_t)(c.ntok + kCluster - 1) / kCluster;
    const uint32_t r0 = rank * rows_per;
    const uint32_t nrows = (uint32_t)max(0, min(c.ntok, (int)(r0 + rows_per)) - (int)r0);
    const uint32_t vpr = (uint32_t)p.row_bytes >> 4;      // 16-byte vectors per row
    const uint32_t row_elems = (uint32_t)p.row_bytes >> 1;
    const uint32_t nvec = nrows * vpr;
    const int lane = threadIdx.x & 31;

    uint8_t* codes = p.chunk_ptrs[p.chunk_base + gl];
    const uint8_t* lb = p.layer_base[l];
    const bool ptr_ok = codes != nullptr && lb != nullptr &&
                        ((reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(lb)) & 15) == 0;
    if (!ptr_ok && threadIdx.x == 0 && rank == 0) report(p, kStatusBadPointer);
    const SliceMap sm(lb + (int64_t)kv * p.num_blocks * p.block_size * p.row_bytes,
                      p.block_table + (int64_t)c.req_row * p.bt_stride + c.col0,
                      r0, vpr, (uint32_t)p.row_bytes, (uint32_t)p.block_size, (uint32_t)p.num_blocks);

    // Pass 1: load the slice and take the running max of |x| on bf16 bits.
    const bool col_fixed = (kThreads % vpr) == 0;
    const uint32_t t_row = threadIdx.x / vpr, t_col = threadIdx.x - t_row * vpr;
    const uint32_t rstep = kThreads / vpr;
    uint4 regs[kVPT];
    uint32_t valid = 0;
    uint32_t acc = 0;
    bool bad = false;
#pragma unroll
    for (int u = 0; u < kVPT; ++u) {
        const uint32_t v = threadIdx.x + u * kThreads;
        regs[u] = make_uint4(0, 0, 0, 0);
        if (ptr_ok && v < nvec) {
            uint32_t row, col;
            if (col_fixed) { row = t_row + u * rstep; col = t_col; }
            else { row = sm.vdiv.div(v); col = v - row * vpr; }
            const uint8_t* src = sm.src(row, col);
            if (src == nullptr) {
                bad = true;
            } else {
                const int4 x = ld_stream(reinterpret_cast<const int4*>(src));
                regs[u] = make_uint4((uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w);
                valid |= 1u << u;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kVPT; ++u) acc = absmax_bf16x8(acc, regs[u]);
    for (uint32_t v = threadIdx.x + kVPT * kThreads; ptr_ok && v < nvec; v += kThreads) {
        const uint32_t row = sm.vdiv.div(v);
        const uint8_t* src = sm.src(row, v - row * vpr);
        if (src == nullptr) { bad = true; continue; }
        const int4 x = ld_stream(reinterpret_cast<const int4*>(src));
        acc = absmax_bf16x8(acc, make_uint4((uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w));
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) report(p, kStatusBadBlock);
    uint32_t m = max(acc & 0xFFFFu, acc >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) warp_max[threadIdx.x >> 5] = m;

    // Exchange: every warp reads all warp maxima of all CTAs of the cluster.
    cluster_arrive_release();
    cluster_wait_acquire();
    uint32_t w = 0;
    constexpr int kSlots = kCluster * (kThreads / 32);
    for (int i = lane; i < kSlots; i += 32)
        w = max(w, *cluster.map_shared_rank(&warp_max[i % (kThreads / 32)], (unsigned)(i / (kThreads / 32))));
    w = __reduce_max_sync(0xFFFFFFFFu, w);
    cluster_arrive_relaxed();          // this CTA's shared memory may be released after everyone arrives

    const float amax = __uint_as_float(w << 16);
    const float scale = __fdiv_rn(amax, 448.0f);
    if (rank == 0 && threadIdx.x == 0 && p.scales != nullptr)
        p.scales[((int64_t)(p.chunk_base + gl) * 2 + kv) * p.num_layers + l] = scale;
    if (ptr_ok) {
        uint8_t* tile_codes = codes + (((int64_t)kv * p.num_layers + l) * c.ntok + r0) * row_elems;
        if (scale >= kFastDivMinScale) {          // reciprocal + correction
            quant_slice<true, kThreads, kVPT>(regs, valid, nvec, sm, tile_codes, make_quant(scale, true));
        } else {                                  // zero or tiny scale: IEEE division
            quant_slice<false, kThreads, kVPT>(regs, valid, nvec, sm, tile_codes, make_quant(scale, false));
        }
    }
    cluster_wait_acquire();
}

// Shared-memory passes of the staged quantisers: absmax, then quantisation,
// over a CTA's rows staged contiguously in shared memory.  Rows whose block id
// is out of range were not copied; with kCheckRows they are skipped.
template <bool kFastDiv, bool kCheckRows, int kThreads>
__device__ __forceinline__ void quant_smem_slice(const uint8_t* slice, uint32_t nvec, const UDiv& vdiv,
                                                 const uint32_t* row_ok, uint8_t* tile_codes,
                                                 const QuantK& k) {
    // Two adjacent vectors per step (rows hold an even number of vectors when
    // row bytes are a multiple of 32), so codes go out as 16-byte stores.
    if (!kCheckRows && (nvec & 1u) == 0 && (vdiv.d & 1u) == 0) {
        for (uint32_t v2 = threadIdx.x; v2 < (nvec >> 1); v2 += kThreads) {
            const uint4 a = *reinterpret_cast<const uint4*>(slice + (size_t)v2 * 32);
            const uint4 b = *reinterpret_cast<const uint4*>(slice + (size_t)v2 * 32 + 16);
            const uint2 qa = quant_bf16x8<kFastDiv>(a, k);
            const uint2 qb = quant_bf16x8<kFastDiv>(b, k);
            *reinterpret_cast<uint4*>(tile_codes + (int64_t)v2 * 16) = make_uint4(qa.x, qa.y, qb.x, qb.y);
        }
        return;
    }
    for (uint32_t v = threadIdx.x; v < nvec; v += kThreads) {
        if (kCheckRows) {
            const uint32_t row = vdiv.div(v);
            if (!((row_ok[row >> 5] >> (row & 31)) & 1u)) continue;
        }
        const uint4 x = *reinterpret_cast<const uint4*>(slice + (size_t)v * 16);
        *reinterpret_cast<uint2*>(tile_codes + (int64_t)v * 8) = quant_bf16x8<kFastDiv>(x, k);
    }
}

template <bool kCheckRows, int kThreads>
__device__ __forceinline__ uint32_t absmax_smem_slice(const uint8_t* slice, uint32_t nvec,
                                                      const UDiv& vdiv, const uint32_t* row_ok) {
    uint32_t acc = 0;
    for (uint32_t v = threadIdx.x; v < nvec; v += kThreads) {
        if (kCheckRows) {
            const uint32_t row = vdiv.div(v);
            if (!((row_ok[row >> 5] >> (row & 31)) & 1u)) continue;
        }
        acc = absmax_bf16x8(acc, *reinterpret_cast<const uint4*>(slice + (size_t)v * 16));
    }
    return acc;
}

// Warp 0 of a quantiser CTA, once its own rows have arrived: ask the TMA unit
// to bring into L2 the slice of the same-rank CTA of tile t2 (a CTA that
// starts about half a wave of clusters later), so that DRAM keeps working
// while this CTA reduces, waits for its cluster and quantises.  Same lookups
// and checks as the slice's own staging; bad ids and pointers are skipped
// (the owning CTA reports them).
template <int kCluster, class B>
__device__ __forceinline__ void prefetch_slice(const B& p, uint32_t t2, uint32_t rank, int lane) {
    if (t2 >= gridDim.x / kCluster) return;
    const uint32_t row_bytes = (uint32_t)p.row_bytes;
    const uint32_t bs = (uint32_t)p.block_size;
    const uint32_t P = bs / (uint32_t)p.parts;
    const UDiv pdiv(P), qdiv((uint32_t)p.parts);
    const uint32_t ll = t2 % (uint32_t)p.layer_n;
    const uint32_t kv = (t2 / (uint32_t)p.layer_n) & 1u;
    const int gl = (int)(t2 / (uint32_t)p.layer_n / 2u);
    const ChunkRef c = resolve_chunk(p, gl);
    const uint32_t rows_per = (uint32_t)(c.ntok + kCluster - 1) / kCluster;
    const uint32_t r0 = rank * rows_per;
    const uint32_t nrows = (uint32_t)max(0, min(c.ntok, (int)(r0 + rows_per)) - (int)r0);
    const uint8_t* lb = p.layer_base[p.layer_lo + (int)ll];
    if (nrows == 0 || lb == nullptr || (reinterpret_cast<uintptr_t>(lb) & 15)) return;
    const uint8_t* kv_base = lb + (int64_t)kv * p.num_blocks * p.block_size * row_bytes;
    const int32_t* bt = p.block_table + (int64_t)c.req_row * p.bt_stride + c.col0;
    const uint32_t pi_end = pdiv.div(r0 + nrows - 1) + 1;
    for (uint32_t pi = pdiv.div(r0) + lane; pi < pi_end; pi += 32) {
        const uint32_t a = max(r0, pi * P), e = min(r0 + nrows, (pi + 1) * P);
        const uint32_t jb = qdiv.div(pi);
        const int32_t blk = bt[jb];
        if ((uint32_t)blk < (uint32_t)p.num_blocks)
            bulk_prefetch_l2(kv_base + ((int64_t)blk * bs + (a - jb * bs)) * row_bytes, (e - a) * row_bytes);
    }
}

// Staged quantising gather (the default when the staged rows fit in shared
// memory).  One thread-block cluster of kCluster CTAs per (chunk, K/V, layer)
// tile; CTA r owns rows [r*n/kCluster, (r+1)*n/kCluster).  The first h rows of
// the CTA's slice (as many whole rows as kThreads * kVPT 16-byte vectors hold)
// are loaded into registers with ordinary loads while warp 0 looks up the page
// runs of the remaining rows in parallel and issues one cp.async.bulk copy per
// run of at most 32 KiB (a page, or a piece of a larger page) into shared
// memory, completing one mbarrier; both halves are in flight
// together.  The CTA takes the absmax over registers and shared memory, the
// cluster exchanges CTA maxima through distributed shared memory (one split
// cluster barrier; lane r reads CTA r's maximum), and every CTA quantises its
// rows.  Measured on the 8B batch with clusters of 8: 4 register vectors per
// thread (16 KiB of registers + 48 KiB of shared memory per CTA) beat staging
// everything in shared memory (0.394 vs 0.406 ms) and 8 or 12 register
// vectors; clusters of 4 (16 KiB + 112 KiB per CTA, two CTAs per SM) are
// faster again (0.371 ms): half as many CTAs meet at each cluster barrier.
template <class B, int kThreads, int kVPT, int kCluster>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
quant_gather_hybrid_kernel(const __grid_constant__ B p) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(128) uint8_t slice[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t cta_max;
    __shared__ uint32_t row_ok[kQuantMaxRows / 32];
    __shared__ uint32_t any_bad;
    static_assert(kCluster <= 32, "one lane per cluster rank");
    pdl_launch_dependents();
    pdl_wait();

    const uint32_t rank = cluster.block_rank();
    const uint32_t tile = blockIdx.x / kCluster;
    const uint32_t ll = tile % (uint32_t)p.layer_n;
    const uint32_t kv = (tile / (uint32_t)p.layer_n) & 1u;
    const int gl = (int)(tile / (uint32_t)p.layer_n / 2u);
    const int l = p.layer_lo + (int)ll;
    const ChunkRef c = resolve_chunk(p, gl);
    const uint32_t rows_per = (uint32_t)(c.ntok + kCluster - 1) / kCluster;
    const uint32_t r0 = rank * rows_per;
    const uint32_t nrows = (uint32_t)max(0, min(c.ntok, (int)(r0 + rows_per)) - (int)r0);
    const uint32_t row_bytes = (uint32_t)p.row_bytes;
    const uint32_t vpr = row_bytes >> 4;
    const uint32_t h = min(nrows, (uint32_t)(kThreads * kVPT) / vpr);   // rows held in registers
    const uint32_t nvec_reg = h * vpr;
    const uint32_t nrows_s = nrows - h;                                   // rows staged in shared memory
    const uint32_t nvec_s = nrows_s * vpr;
    const int lane = threadIdx.x & 31;

    uint8_t* codes = p.chunk_ptrs[p.chunk_base + gl];
    const uint8_t* lb = p.layer_base[l];
    const bool ptr_ok = codes != nullptr && lb != nullptr &&
                        ((reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(lb)) & 15) == 0;
    const SliceMap sm(lb + (int64_t)kv * p.num_blocks * p.block_size * row_bytes,
                      p.block_table + (int64_t)c.req_row * p.bt_stride + c.col0, r0, vpr, row_bytes,
                      (uint32_t)p.block_size, (uint32_t)p.num_blocks);
    if (threadIdx.x < 32) {
        // Warp 0 stages rows [r0 + h, r0 + nrows) in shared memory.
        if (lane == 0) {
            if (!ptr_ok && rank == 0) report(p, kStatusBadPointer);
            cta_max = 0;
            mbar_init(&bar, 1);
            fence_barrier_init();
        }
        for (int i = lane; i < kQuantMaxRows / 32; i += 32) row_ok[i] = 0;
        __syncwarp();
        // One bulk copy per piece of P = block_size / parts rows (pages of at
        // most 32 KiB are one piece; larger pages are cut so that several
        // copies are in flight, as with small pages).  Piece i covers slice
        // rows [i*P, (i+1)*P), inside page i / parts.
        const uint32_t bs = (uint32_t)p.block_size;
        const uint32_t P = bs / (uint32_t)p.parts;
        const UDiv pdiv(P), qdiv((uint32_t)p.parts);
        const uint32_t s0 = r0 + h;
        const uint32_t pi0 = nrows_s ? pdiv.div(s0) : 0u;
        const uint32_t pi_end = nrows_s ? pdiv.div(s0 + nrows_s - 1) + 1 : 0u;
        uint32_t bytes = 0;
        bool bad = false;
        for (uint32_t pi = pi0 + lane; ptr_ok && pi < pi_end; pi += 32) {
            const uint32_t a = max(s0, pi * P), e = min(s0 + nrows_s, (pi + 1) * P);
            const int32_t blk = sm.bt[qdiv.div(pi)];
            if ((uint32_t)blk < (uint32_t)p.num_blocks) {
                bytes += (e - a) * row_bytes;
                for (uint32_t r = a - s0; r < e - s0; ++r) atomicOr(&row_ok[r >> 5], 1u << (r & 31));
            } else {
                bad = true;
            }
        }
        const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, bytes);
        const bool any = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0) {
            any_bad = any ? 1u : 0u;
            mbar_arrive_expect_tx(&bar, total);
        }
        __syncwarp();
        for (uint32_t pi = pi0 + lane; ptr_ok && pi < pi_end; pi += 32) {
            const uint32_t a = max(s0, pi * P), e = min(s0 + nrows_s, (pi + 1) * P);
            const uint32_t jb = qdiv.div(pi);
            const int32_t blk = sm.bt[jb];
            if ((uint32_t)blk < (uint32_t)p.num_blocks)
                bulk_g2s(slice + (size_t)(a - s0) * row_bytes,
                         sm.kv_base + ((int64_t)blk * bs + (a - jb * bs)) * row_bytes, (e - a) * row_bytes, &bar);
        }
    }
    // Every thread: rows [r0, r0 + h) into registers.
    const bool col_fixed = (kThreads % vpr) == 0;
    const uint32_t t_row = threadIdx.x / vpr, t_col = threadIdx.x - t_row * vpr;
    const uint32_t rstep = kThreads / vpr;
    uint4 regs[kVPT];
    uint32_t valid = 0;
    bool bad_reg = false;
#pragma unroll
    for (int u = 0; u < kVPT; ++u) {
        const uint32_t v = threadIdx.x + u * kThreads;
        regs[u] = make_uint4(0, 0, 0, 0);
        if (ptr_ok && v < nvec_reg) {
            uint32_t row, col;
            if (col_fixed) { row = t_row + u * rstep; col = t_col; }
            else { row = sm.vdiv.div(v); col = v - row * vpr; }
            const uint8_t* src = sm.src(row, col);
            if (src == nullptr) {
                bad_reg = true;
            } else {
                const int4 x = ld_stream(reinterpret_cast<const int4*>(src));
                regs[u] = make_uint4((uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w);
                valid |= 1u << u;
            }
        }
    }
    uint32_t acc = 0;
#pragma unroll
    for (int u = 0; u < kVPT; ++u) acc = absmax_bf16x8(acc, regs[u]);
    if (__any_sync(0xFFFFFFFFu, bad_reg) && lane == 0) report(p, kStatusBadBlock);
    __syncthreads();                                  // barrier initialised, row_ok / any_bad written
    bool timed_out = false;
    if (!mbar_wait_bounded(&bar, 0)) {
        timed_out = true;
        if (threadIdx.x == 0) report(p, kStatusTimeout);
        (void)mbar_wait_bounded(&bar, 0);
    }
    if (threadIdx.x == 0 && any_bad) report(p, kStatusBadBlock);
    if (p.prefetch_ahead > 0 && threadIdx.x < 32)
        prefetch_slice<kCluster>(p, tile + (uint32_t)p.prefetch_ahead, rank, lane);
    const bool check_rows = any_bad != 0;
    {
        const uint32_t a2 = check_rows ? absmax_smem_slice<true, kThreads>(slice, nvec_s, sm.vdiv, row_ok)
                                       : absmax_smem_slice<false, kThreads>(slice, nvec_s, sm.vdiv, row_ok);
        const uint32_t m1 = max(acc & 0xFFFFu, acc >> 16), m2 = max(a2 & 0xFFFFu, a2 >> 16);
        uint32_t m = max(m1, m2);
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0) atomicMax(&cta_max, m);
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    uint32_t w = lane < kCluster ? *cluster.map_shared_rank(&cta_max, (unsigned)lane) : 0u;
    w = __reduce_max_sync(0xFFFFFFFFu, w);
    cluster_arrive_relaxed();          // this CTA's shared memory may be released after everyone arrives

    const float amax = __uint_as_float(w << 16);
    const float scale = __fdiv_rn(amax, 448.0f);
    if (rank == 0 && threadIdx.x == 0 && p.scales != nullptr)
        p.scales[((int64_t)(p.chunk_base + gl) * 2 + kv) * p.num_layers + l] = scale;
    if (ptr_ok && !timed_out) {
        uint8_t* tile_codes = codes + (((int64_t)kv * p.num_layers + l) * c.ntok + r0) * (row_bytes >> 1);
        uint8_t* smem_codes = tile_codes + (size_t)nvec_reg * 8;
        const bool fast = scale >= kFastDivMinScale;
        const QuantK k = make_quant(scale, fast);
        // register rows
#pragma unroll
        for (int u = 0; u < kVPT; ++u) {
            const uint32_t v = threadIdx.x + u * kThreads;
            if (v < nvec_reg && (valid >> u) & 1u) {
                const uint2 q = scale == 0.0f ? make_uint2(0, 0)
                              : fast ? quant_bf16x8<true>(regs[u], k) : quant_bf16x8<false>(regs[u], k);
                *reinterpret_cast<uint2*>(tile_codes + (int64_t)v * 8) = q;
            }
        }
        // shared-memory rows
        if (scale == 0.0f) {
            for (uint32_t v = threadIdx.x; v < nvec_s; v += kThreads) {
                const uint32_t row = sm.vdiv.div(v);
                if (!check_rows || ((row_ok[row >> 5] >> (row & 31)) & 1u))
                    *reinterpret_cast<uint2*>(smem_codes + (int64_t)v * 8) = make_uint2(0, 0);
            }
        } else if (fast) {
            if (check_rows) quant_smem_slice<true, true, kThreads>(slice, nvec_s, sm.vdiv, row_ok, smem_codes, k);
            else quant_smem_slice<true, false, kThreads>(slice, nvec_s, sm.vdiv, row_ok, smem_codes, k);
        } else {
            quant_smem_slice<false, true, kThreads>(slice, nvec_s, sm.vdiv, row_ok, smem_codes, k);
        }
    }
    cluster_wait_acquire();
}

// ---------------------------------------------------------------------------
// fp8 e4m3 dequantising scatter: per item (chunk, kv, layer, block part),
// 8 codes (8 bytes) in, 8 bf16 (16 bytes) out per thread step.
__device__ __forceinline__ uint2 ld_stream8(const uint2* ptr) {
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(ptr));
    return r;
}

__device__ __forceinline__ uint32_t dequant_pair(uint16_t two_codes, float scale) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two_codes, __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    return *reinterpret_cast<const uint32_t*>(&b);
}

template <class B, int kThreads, int kUnroll>
__global__ void __launch_bounds__(kThreads)
dequant_scatter_kernel(const __grid_constant__ B p, int64_t num_items) {
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t item = blockIdx.x; item < num_items; item += gridDim.x) {
        // Decode the item against a bf16 pool, then derive the code run from it.
        Run run;
        if (!item_run(p, item, run)) continue;
        const int kv = run.kv, gl = run.gl;
        const int l = p.layer_lo + run.ll;
        const float scale = p.scales[((int64_t)(p.chunk_base + gl) * 2 + kv) * p.num_layers + l];
        // chunk-side offset of the run in bf16 bytes -> the same rows in code bytes
        const uint8_t* cb = p.chunk_ptrs[p.chunk_base + gl];
        const int64_t code_off = (run.chunk - cb) >> 1;
        // 8 codes (8 bytes) per thread step -> one 16-byte store, so that a
        // warp's store instruction covers 512 contiguous bytes; kUnroll code
        // words per thread are loaded before their stores (the code and pool
        // pointers may alias, so the compiler never moves a load above an
        // earlier store by itself)
        const int n8 = (int)(run.bytes >> 4);
        const uint2* src = reinterpret_cast<const uint2*>(cb + code_off);
        int4* dst = reinterpret_cast<int4*>(run.pool);
        for (int base = threadIdx.x; base < n8; base += kThreads * kUnroll) {
            uint2 ci[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = base + u * kThreads;
                if (v < n8) ci[u] = ld_stream8(src + v);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = base + u * kThreads;
                if (v >= n8) continue;
                st_stream(dst + v, make_int4((int)dequant_pair((uint16_t)(ci[u].x & 0xFFFFu), scale),
                                             (int)dequant_pair((uint16_t)(ci[u].x >> 16), scale),
                                             (int)dequant_pair((uint16_t)(ci[u].y & 0xFFFFu), scale),
                                             (int)dequant_pair((uint16_t)(ci[u].y >> 16), scale)));
            }
        }
    }
}

}  // namespace lmkv
