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
// The fp8 variant (quantising gather, dequantising scatter) is in
// lmkv_fp8.cuh.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

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

}  // namespace lmkv
