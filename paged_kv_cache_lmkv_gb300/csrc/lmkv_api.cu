// lmkv_api.cu -- host side of the C ABI declared in include/lmkv.h.
//
// Validates arguments, enumerates chunks (cache_engine.py walk-through,
// "store()" section: chunk_size chunks, short tail only with
// save_unfull_chunk, chunk-aligned start), packs up to kMaxReqPerLaunch
// requests into one by-value parameter block per launch, and enqueues the
// kernels of lmkv_kernels.cuh on the caller's stream.  Nothing is allocated
// and nothing is synchronised.
#include "lmkv.h"
#include "lmkv_internal.h"
#include "lmkv_fp8.cuh"

#include <atomic>
#include <map>
#include <mutex>

namespace {

std::atomic<int64_t> g_launches{0};
std::atomic<int> g_last_cuda_error{0};

// Keep the code of a failed CUDA runtime call for lmkv_last_cuda_error().
inline int cuda_status(cudaError_t err) {
    if (err == cudaSuccess) return LMKV_OK;
    g_last_cuda_error.store((int)err, std::memory_order_relaxed);
    return LMKV_ERR_CUDA;
}

// Copy engine configuration (chosen by measurement on GB300: a sweep of the
// LSU and TMA bulk engines over threads, unroll, grid shape and stages found
// the LSU engine with one CTA per run (page, or 32 KiB piece of a larger
// page) at the top for the 8B gather; a grid of
// resident CTAs with equal vector ranges was 6-9% slower for whole-batch and
// per-layer calls).
constexpr int kLsuThreads = 256;
constexpr int kLsuUnroll = 8;
constexpr int kQuantThreads = 256;        // staged quantiser
constexpr int kQuantRegThreads = 512;     // register-staged fallback (slices beyond shared memory)
constexpr int kQuantVPT = 8;
// Cluster sizes of the staged quantiser: 4 CTAs per (chunk, K/V, layer) tile
// where a CTA's quarter of the tile fits the staging limit (every 8B / 70B /
// Qwen tile: 64 rows = 8 in registers + 56 in 112 KiB of shared memory), else
// 8 (longer chunks; also the register-staged fallback).  Measured on the 8B
// batch (median of 30 event-timed calls): clusters of 4 0.371 ms, of 8
// 0.398 ms; 4 with 6 register vectors 0.374, with 2 (120 KiB of shared
// memory, one CTA per SM) 0.584; 512-thread CTAs 0.40-0.50.
constexpr int kQuantCluster = 4;
constexpr int kQuantClusterWide = 8;
constexpr int kQuantHybridVPT = 4;        // register vectors per thread of the staged quantiser
constexpr int kDequantThreads = 256;
// 8-byte code words per thread loaded before their stores (each word -> one
// contiguous 16-byte store).  Measured on the 8B batch: 2 -> 0.329 ms, 4 ->
// 0.314, 8 -> 0.308 (8 covers a whole 16-row item of 2 KiB rows in one pass).
// The earlier form, 16-byte code vectors each stored as two 16-byte halves
// 32 bytes apart, measured 1 -> 0.319, 2 -> 0.316, 4 -> 0.357, 8 -> 0.361.
constexpr int kDequantUnroll = 8;

// Chunks of one request (cache_engine.py walk-through, "store()").
inline int64_t request_chunks(int64_t s, int64_t e, int32_t chunk_size, int32_t save_unfull) {
    const int64_t len = e - s;
    return len / chunk_size + ((save_unfull && len % chunk_size) ? 1 : 0);
}

// Validate the request list; returns the chunk count and the number of
// requests that have at least one chunk.
int check_requests(const int64_t* start, const int64_t* end, int32_t num_req, int32_t chunk_size,
                   int32_t save_unfull, int64_t* num_chunks, int32_t* nonempty) {
    if (num_req < 0 || chunk_size <= 0) return LMKV_ERR_INVALID_ARG;
    if (num_req > 0 && (start == nullptr || end == nullptr)) return LMKV_ERR_INVALID_ARG;
    int64_t n = 0;
    int32_t ne = 0;
    for (int32_t r = 0; r < num_req; ++r) {
        const int64_t s = start[r], e = end[r];
        if (s < 0 || e < s || s % chunk_size != 0) return LMKV_ERR_INVALID_ARG;
        const int64_t c = request_chunks(s, e, chunk_size, save_unfull);
        n += c;
        ne += c > 0;
    }
    if (n > INT32_MAX) return LMKV_ERR_INVALID_ARG;
    *num_chunks = n;
    if (nonempty) *nonempty = ne;
    return LMKV_OK;
}

int check_pool(const lmkv_pool_t* pool) {
    if (pool == nullptr || pool->layer_base == nullptr) return LMKV_ERR_INVALID_ARG;
    if (pool->num_layers <= 0 || pool->num_kv_heads <= 0 || pool->head_dim <= 0 ||
        pool->block_size <= 0 || pool->num_blocks <= 0 || pool->num_blocks > INT32_MAX)
        return LMKV_ERR_INVALID_ARG;
    if (pool->elem_bytes != 1 && pool->elem_bytes != 2 && pool->elem_bytes != 4)
        return LMKV_ERR_INVALID_ARG;
    const int64_t row = (int64_t)pool->num_kv_heads * pool->head_dim * pool->elem_bytes;
    if (row > (1 << 20)) return LMKV_ERR_INVALID_ARG;
    if (row % 16 != 0) return LMKV_ERR_MISALIGNED;
    if ((int64_t)pool->block_size * row > (int64_t)1 << 30) return LMKV_ERR_INVALID_ARG;
    return LMKV_OK;
}

// Everything a call needs besides the kernel choice.
struct Call {
    const lmkv_pool_t* pool;
    const int32_t* block_table;
    int32_t max_blocks;
    const int64_t* start;
    const int64_t* end;
    int32_t num_req;
    int32_t chunk_size;
    int32_t save_unfull;
    void* const* chunk_ptrs;
    int32_t* d_status;
    int32_t layer_lo;
    int32_t layer_n;
    int32_t parts;
    int64_t num_chunks;
    int32_t nonempty;
    void* staging;       // one-layer DEVICE staging buffer (staged pipeline), else null
    int32_t prefetch_ahead;   // copy kernel's L2 prefetch distance in items (0 = none)
};

int validate(Call& c) {
    int rc = check_pool(c.pool);
    if (rc != LMKV_OK) return rc;
    if (c.chunk_size <= 0 || c.chunk_size % c.pool->block_size != 0) return LMKV_ERR_INVALID_ARG;
    if (c.max_blocks < 0 || c.num_req < 0) return LMKV_ERR_INVALID_ARG;
    if (c.layer_lo < 0 || c.layer_n <= 0 || c.layer_lo + c.layer_n > c.pool->num_layers)
        return LMKV_ERR_INVALID_ARG;
    if (c.pool->block_size % c.parts != 0) c.parts = 1;
    rc = check_requests(c.start, c.end, c.num_req, c.chunk_size, c.save_unfull, &c.num_chunks,
                        &c.nonempty);
    if (rc != LMKV_OK) return rc;
    for (int32_t r = 0; r < c.num_req; ++r) {
        if (c.end[r] > c.start[r] && (c.end[r] - 1) / c.pool->block_size >= c.max_blocks)
            return LMKV_ERR_INVALID_ARG;
    }
    if (c.num_chunks > 0 && (c.block_table == nullptr || c.chunk_ptrs == nullptr))
        return LMKV_ERR_INVALID_ARG;
    return LMKV_OK;
}

// Pack the call's non-empty requests into parameter blocks of capacity
// B::kCapacity and hand each block to `launch`.
template <class B, class LaunchFn>
int for_each_block(const Call& c, float* scales, LaunchFn&& launch) {
    B b;
    b.layer_base = reinterpret_cast<const uint8_t* const*>(c.pool->layer_base);
    b.chunk_ptrs = reinterpret_cast<uint8_t* const*>(c.chunk_ptrs);
    b.block_table = c.block_table;
    b.status = c.d_status;
    b.scales = scales;
    b.num_blocks = c.pool->num_blocks;
    b.bt_stride = c.max_blocks;
    b.num_layers = c.pool->num_layers;
    b.row_bytes = c.pool->num_kv_heads * c.pool->head_dim * c.pool->elem_bytes;
    b.block_size = c.pool->block_size;
    b.chunk_size = c.chunk_size;
    b.blocks_per_chunk = c.chunk_size / c.pool->block_size;
    b.parts = c.parts;
    b.layer_lo = c.layer_lo;
    b.layer_n = c.layer_n;
    b.num_req = 0;
    b.chunk_base = 0;
    b.num_chunks = 0;
    b.prefetch_ahead = c.prefetch_ahead;
    b.staging = static_cast<uint8_t*>(c.staging);
    b.stage_tok_base = 0;
    b.req_chunk_begin[0] = 0;
    int64_t tok_in_launch = 0;
    for (int32_t r = 0; r < c.num_req; ++r) {
        const int64_t nch = request_chunks(c.start[r], c.end[r], c.chunk_size, c.save_unfull);
        if (nch == 0) continue;
        if (b.num_req == B::kCapacity) {
            const int rc = launch(b);
            if (rc != LMKV_OK) return rc;
            b.chunk_base += b.num_chunks;
            b.stage_tok_base += tok_in_launch;
            tok_in_launch = 0;
            b.num_chunks = 0;
            b.num_req = 0;
            b.req_chunk_begin[0] = 0;
        }
        const int i = b.num_req++;
        b.req_row[i] = r;
        b.req_chunk_begin[i] = b.num_chunks;
        b.req_tok0[i] = c.start[r];
        b.req_col0[i] = (int32_t)(c.start[r] / c.pool->block_size);
        b.req_tok_end[i] = c.save_unfull ? c.end[r]
                                          : c.start[r] + (c.end[r] - c.start[r]) / c.chunk_size * c.chunk_size;
        b.req_tok_prefix[i] = tok_in_launch;
        tok_in_launch += b.req_tok_end[i] - b.req_tok0[i];
        b.num_chunks += (int32_t)nch;
        b.req_chunk_begin[i + 1] = b.num_chunks;
    }
    if (b.num_req > 0) return launch(b);
    return LMKV_OK;
}

// Launch with programmatic stream serialization (the kernels wait for their
// predecessors with griddepcontrol.wait before touching memory).
template <class Kernel, class... Args>
int launch_pdl(Kernel kernel, int64_t grid, int threads, cudaStream_t stream, Args... args) {
    if (grid <= 0) return LMKV_OK;
    if (grid > INT32_MAX) return LMKV_ERR_INVALID_ARG;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, args...);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(err);
}

template <class Kernel, class... Args>
int launch_pdl_smem(Kernel kernel, int64_t grid, int threads, int64_t smem, cudaStream_t stream,
                    Args... args) {
    if (grid <= 0) return LMKV_OK;
    if (grid > INT32_MAX) return LMKV_ERR_INVALID_ARG;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, args...);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(err);
}

// Number of CTAs the LSU engine launches for `items` items (one per item).
int64_t lsu_grid(int64_t items) {
    const int64_t cap = (int64_t)1 << 30;
    return items < cap ? items : cap;
}

template <class B, bool kGather>
int launch_move(const Call& c, cudaStream_t stream) {
    return for_each_block<B>(c, nullptr, [&](const B& b) {
        const int64_t items = lmkv::batch_items(b);
        return launch_pdl(lmkv::move_lsu_kernel<B, kGather, kLsuThreads, kLsuUnroll>,
                          lsu_grid(items), kLsuThreads, stream, b, items);
    });
}

// Items of about 32 KiB: a page larger than that is split into equal parts
// (a divisor of block_size), so that calls on 32- and 64-token pages launch
// as many CTAs of the same size as calls on 16-token pages of 2 KiB rows
// (one per-layer call on 64-token pages otherwise has a quarter of the CTAs,
// each looping four times).  Pages of up to 32 KiB stay whole: splitting the
// 8B layer-wise calls' 32 KiB runs into 2, 4 or 8 parts measured 2-120%
// slower than one CTA per run.
constexpr int64_t kItemBytes = 32 * 1024;

int32_t choose_parts(const lmkv_pool_t* pool) {
    const int64_t row = (int64_t)pool->num_kv_heads * pool->head_dim * pool->elem_bytes;
    const int64_t page = row * pool->block_size;
    int32_t parts = 1;
    for (int32_t q = 2; q <= pool->block_size && page / q >= kItemBytes; ++q)
        if (pool->block_size % q == 0) parts = q;
    return parts;
}

// L2 prefetch distance, in items, of the copy kernel's one-layer calls: five
// eighths of the kernel's CTAs resident at once (occupancy x SM count: 4 x
// 152 -> 380 on GB300).  Measured on the 8B per-layer calls (gather /
// scatter, us per call): no prefetch 15.7 / 15.5; 228 items ahead 15.2 /
// 14.9; 304 and 380 15.1 / 14.8; 456 15.2 / 14.8; 608 15.5 / 15.3; each CTA
// prefetching its own run 15.4 / 15.2.  Whole-batch copies are bound by HBM
// and gain nothing (prefetching there measured -1% to +0.5%).  (The
// dequantising scatter gained 2.4% with a fixed distance at 47 registers and
// 5 CTAs per SM, but lost 2% once its registers fell to 40 and 6 CTAs per SM;
// it does not prefetch.)
// Cached per device after the first call made outside a stream capture (no
// device query is made while `stream` is capturing: such a call, before the
// value is known, prefetches nothing); 0 (no prefetch) if a query fails.
template <class Kernel>
int32_t prefetch_distance(Kernel kernel, int threads, std::atomic<int32_t>* cache, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return 0;
    }
    const int32_t v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        (void)cudaGetLastError();
        return 0;
    }
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const int32_t ahead = (int32_t)((int64_t)per_sm * sms * 5 / 8);
    if (ahead > 0) cache[dev].store(ahead, std::memory_order_relaxed);
    return ahead > 0 ? ahead : 0;
}

int32_t lsu_prefetch_ahead(cudaStream_t stream) {
    static std::atomic<int32_t> cache[64];
    return prefetch_distance(lmkv::move_lsu_kernel<lmkv::BatchSmall, true, kLsuThreads, kLsuUnroll>,
                             kLsuThreads, cache, stream);
}

int move_entry(bool gather, const lmkv_pool_t* pool, const int32_t* block_table,
               int32_t max_blocks, const int64_t* start, const int64_t* end, int32_t num_req,
               int32_t chunk_size, int32_t save_unfull, void* const* chunk_ptrs,
               int32_t layer, int32_t* d_status, void* stream, void* staging = nullptr) {
    const int rc0 = check_pool(pool);
    if (rc0 != LMKV_OK) return rc0;
    Call c{pool, block_table, max_blocks, start, end, num_req, chunk_size, save_unfull,
           chunk_ptrs, d_status, 0, pool->num_layers, 1, 0, 0, staging};
    if (layer >= 0) {
        if (layer >= pool->num_layers) return LMKV_ERR_INVALID_ARG;
        c.layer_lo = layer;
        c.layer_n = 1;
        c.prefetch_ahead = lsu_prefetch_ahead(reinterpret_cast<cudaStream_t>(stream));
    }
    c.parts = choose_parts(pool);
    const int rc = validate(c);
    if (rc != LMKV_OK || c.num_chunks == 0) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (c.nonempty <= lmkv::kSmallBatch)
        return gather ? launch_move<lmkv::BatchSmall, true>(c, s)
                      : launch_move<lmkv::BatchSmall, false>(c, s);
    return gather ? launch_move<lmkv::Batch, true>(c, s) : launch_move<lmkv::Batch, false>(c, s);
}

// Layer-wise pipeline: per layer, wait on its ready event, move it, record its
// done event, all on one stream.
int layers_entry(bool gather, const lmkv_pool_t* pool, const int32_t* block_table,
                 int32_t max_blocks, const int64_t* start, const int64_t* end, int32_t num_req,
                 int32_t chunk_size, int32_t save_unfull, void* const* chunk_ptrs, int32_t layer_lo,
                 int32_t layer_n, void* const* ready, void* const* done, int32_t* d_status,
                 void* stream) {
    int rc = check_pool(pool);
    if (rc != LMKV_OK) return rc;
    if (layer_lo < 0 || layer_n < 0 || (int64_t)layer_lo + layer_n > pool->num_layers)
        return LMKV_ERR_INVALID_ARG;
    if (layer_n == 0) return LMKV_OK;
    // validate the whole call once (same checks as every per-layer call)
    Call c{pool, block_table, max_blocks, start, end, num_req, chunk_size, save_unfull,
           chunk_ptrs, d_status, layer_lo, layer_n, 1, 0, 0, nullptr};
    rc = validate(c);
    if (rc != LMKV_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int32_t i = 0; i < layer_n; ++i) {
        if (ready != nullptr && ready[i] != nullptr &&
            cuda_status(cudaStreamWaitEvent(s, reinterpret_cast<cudaEvent_t>(ready[i]), 0)) != LMKV_OK)
            return LMKV_ERR_CUDA;
        rc = move_entry(gather, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                        save_unfull, chunk_ptrs, layer_lo + i, d_status, stream);
        if (rc != LMKV_OK) return rc;
        if (done != nullptr && done[i] != nullptr &&
            cuda_status(cudaEventRecord(reinterpret_cast<cudaEvent_t>(done[i]), s)) != LMKV_OK)
            return LMKV_ERR_CUDA;
    }
    return LMKV_OK;
}

// Staged layer-wise pipeline: per layer, the kernel moves the layer between
// the pool and a one-layer DEVICE staging buffer, and one 2-D copy per chunk
// (the copy engine, no SMs) moves the chunk's K and V slices of that layer
// between the staging buffer and the chunk's pinned host buffer.
// The staged pipeline.  With copy_stream == null: per layer, the kernel and
// the copies run in order on `stream` through one staging buffer.  With a
// copy stream and four caller-owned events: two staging buffers, kernels on
// `stream` and copies on `copy_stream`, so that a layer's copies overlap the
// next layer's kernel; sync[b] marks "kernel on buffer b done", sync[2 + b]
// "copies of buffer b done".
int staged_entry(bool store, const lmkv_pool_t* pool, const int32_t* block_table,
                 int32_t max_blocks, const int64_t* start, const int64_t* end, int32_t num_req,
                 int32_t chunk_size, int32_t save_unfull, void* const* host_chunks, void* staging,
                 int64_t staging_bytes, int32_t layer_lo, int32_t layer_n, void* const* ready,
                 void* const* done, int32_t* d_status, void* stream, void* copy_stream = nullptr,
                 void* const* sync = nullptr) {
    int rc = check_pool(pool);
    if (rc != LMKV_OK) return rc;
    if (layer_lo < 0 || layer_n < 0 || (int64_t)layer_lo + layer_n > pool->num_layers)
        return LMKV_ERR_INVALID_ARG;
    if (layer_n == 0) return LMKV_OK;
    Call c{pool, block_table, max_blocks, start, end, num_req, chunk_size, save_unfull,
           host_chunks, d_status, layer_lo, layer_n, choose_parts(pool), 0, 0, staging};
    rc = validate(c);
    if (rc != LMKV_OK || c.num_chunks == 0) return rc;
    const int64_t rb = (int64_t)pool->num_kv_heads * pool->head_dim * pool->elem_bytes;
    int64_t tokens = 0;
    for (int32_t r = 0; r < num_req; ++r) {
        const int64_t nch = request_chunks(start[r], end[r], chunk_size, save_unfull);
        if (nch > 0)
            tokens += save_unfull ? end[r] - start[r] : (end[r] - start[r]) / chunk_size * chunk_size;
    }
    const bool two = copy_stream != nullptr;
    const int64_t layer_bytes = 2 * rb * tokens;                 // one layer's K and V rows
    if (staging == nullptr || staging_bytes < (two ? 2 : 1) * layer_bytes) return LMKV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(staging) & 15) return LMKV_ERR_MISALIGNED;
    if (two && (sync == nullptr || sync[0] == nullptr || sync[1] == nullptr || sync[2] == nullptr ||
                sync[3] == nullptr))
        return LMKV_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t cs = two ? reinterpret_cast<cudaStream_t>(copy_stream) : s;
    auto ev = [&](int k) { return reinterpret_cast<cudaEvent_t>(sync[k]); };
    uint8_t* stage_base = static_cast<uint8_t*>(staging);
    const int64_t L = pool->num_layers;
    // Per chunk, rows {K, V} of layer l: n_g * rb bytes each; host pitch
    // L * n_g * rb, staging pitch n_g * rb.  A run of full chunks whose host
    // buffers follow each other in memory (chunk g+1 starts where chunk g
    // ends) is tried as one 3-D copy (depth = chunks); the driver accepts that
    // only within one allocation, so if it declines, the run falls back to one
    // 2-D copy per chunk and no further 3-D copy is tried in this call.
    bool try_3d = true;
    uint8_t* staging_now = stage_base;           // the buffer of the layer being moved
    auto copy_2d = [&](uint8_t* host, uint8_t* stage, int64_t n) {
        return store ? cudaMemcpy2DAsync(host, L * n * rb, stage, n * rb, n * rb, 2,
                                         cudaMemcpyDeviceToHost, cs)
                     : cudaMemcpy2DAsync(stage, n * rb, host, L * n * rb, n * rb, 2,
                                         cudaMemcpyHostToDevice, cs);
    };
    auto copy_run = [&](int32_t l, int64_t g0, int64_t count, int64_t n, int64_t tok_before) -> int {
        uint8_t* host = static_cast<uint8_t*>(host_chunks[g0]) + (int64_t)l * n * rb;
        uint8_t* stage = staging_now + 2 * rb * tok_before;
        if (count > 1 && try_3d) {
            cudaMemcpy3DParms m = {};
            const cudaPitchedPtr hp = make_cudaPitchedPtr(host, (size_t)(L * n * rb), (size_t)(n * rb), 2);
            const cudaPitchedPtr sp = make_cudaPitchedPtr(stage, (size_t)(n * rb), (size_t)(n * rb), 2);
            m.srcPtr = store ? sp : hp;
            m.dstPtr = store ? hp : sp;
            m.extent = make_cudaExtent((size_t)(n * rb), 2, (size_t)count);
            m.kind = store ? cudaMemcpyDeviceToHost : cudaMemcpyHostToDevice;
            if (cudaMemcpy3DAsync(&m, cs) == cudaSuccess) return LMKV_OK;
            (void)cudaGetLastError();
            try_3d = false;
        }
        const int64_t chunk_bytes = 2 * L * n * rb;
        for (int64_t k = 0; k < count; ++k) {
            if (cuda_status(copy_2d(host + k * chunk_bytes, stage + k * 2 * n * rb, n)) != LMKV_OK)
                return LMKV_ERR_CUDA;
        }
        return LMKV_OK;
    };
    auto copies = [&](int32_t l) -> int {
        int64_t g = 0, tok_before = 0;
        int64_t run_g0 = -1, run_len = 0, run_tok = 0;
        const int64_t full_bytes = 2 * L * (int64_t)chunk_size * rb;
        int rc2 = LMKV_OK;
        for (int32_t r = 0; r < num_req && rc2 == LMKV_OK; ++r) {
            const int64_t nch = request_chunks(start[r], end[r], chunk_size, save_unfull);
            for (int64_t j = 0; j < nch && rc2 == LMKV_OK; ++j, ++g) {
                const int64_t t0 = start[r] + j * chunk_size;
                const int64_t n = (t0 + chunk_size < end[r] ? t0 + chunk_size : end[r]) - t0;
                if (host_chunks[g] == nullptr) return LMKV_ERR_INVALID_ARG;
                const bool extends = run_len > 0 && n == chunk_size &&
                    static_cast<uint8_t*>(host_chunks[g]) ==
                        static_cast<uint8_t*>(host_chunks[run_g0]) + run_len * full_bytes;
                if (extends) {
                    ++run_len;
                } else {
                    if (run_len > 0) rc2 = copy_run(l, run_g0, run_len, chunk_size, run_tok);
                    if (n == chunk_size) {
                        run_g0 = g;
                        run_len = 1;
                        run_tok = tok_before;
                    } else {
                        run_len = 0;
                        if (rc2 == LMKV_OK) rc2 = copy_run(l, g, 1, n, tok_before);
                    }
                }
                tok_before += n;
            }
        }
        if (rc2 == LMKV_OK && run_len > 0) rc2 = copy_run(l, run_g0, run_len, chunk_size, run_tok);
        return rc2;
    };
    auto wait = [&](cudaStream_t on, cudaEvent_t e) {
        return cuda_status(cudaStreamWaitEvent(on, e, 0));
    };
    auto record = [&](cudaEvent_t e, cudaStream_t on) { return cuda_status(cudaEventRecord(e, on)); };
    if (two) {
        // the copy stream starts after everything already ordered on `stream`
        if (record(ev(0), s) != LMKV_OK || wait(cs, ev(0)) != LMKV_OK) return LMKV_ERR_CUDA;
    }
    for (int32_t i = 0; i < layer_n; ++i) {
        const int32_t l = layer_lo + i;
        const int b = two ? (i & 1) : 0;
        staging_now = stage_base + b * layer_bytes;
        cudaEvent_t ready_i = (ready != nullptr && ready[i] != nullptr) ? reinterpret_cast<cudaEvent_t>(ready[i])
                                                                        : nullptr;
        cudaEvent_t done_i = (done != nullptr && done[i] != nullptr) ? reinterpret_cast<cudaEvent_t>(done[i])
                                                                     : nullptr;
        if (store) {
            // buffer b is free once the copies of layer i - 2 are done
            if (two && i >= 2 && wait(s, ev(2 + b)) != LMKV_OK) return LMKV_ERR_CUDA;
            if (ready_i && wait(s, ready_i) != LMKV_OK) return LMKV_ERR_CUDA;
            rc = move_entry(true, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                            save_unfull, host_chunks, l, d_status, stream, staging_now);
            if (rc != LMKV_OK) return rc;
            if (two && (record(ev(b), s) != LMKV_OK || wait(cs, ev(b)) != LMKV_OK)) return LMKV_ERR_CUDA;
            rc = copies(l);
            if (rc != LMKV_OK) return rc;
            if (two && record(ev(2 + b), cs) != LMKV_OK) return LMKV_ERR_CUDA;
            if (done_i && record(done_i, cs) != LMKV_OK) return LMKV_ERR_CUDA;
        } else {
            // buffer b is free once the kernel of layer i - 2 has read it
            if (two && i >= 2 && wait(cs, ev(b)) != LMKV_OK) return LMKV_ERR_CUDA;
            rc = copies(l);
            if (rc != LMKV_OK) return rc;
            if (two && (record(ev(2 + b), cs) != LMKV_OK || wait(s, ev(2 + b)) != LMKV_OK)) return LMKV_ERR_CUDA;
            if (ready_i && wait(s, ready_i) != LMKV_OK) return LMKV_ERR_CUDA;
            rc = move_entry(false, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                            save_unfull, host_chunks, l, d_status, stream, staging_now);
            if (rc != LMKV_OK) return rc;
            if (two && record(ev(b), s) != LMKV_OK) return LMKV_ERR_CUDA;
            if (done_i && record(done_i, s) != LMKV_OK) return LMKV_ERR_CUDA;
        }
    }
    if (two && store) {
        // the call's work ends on `stream`: join the last copies of both buffers
        if (wait(s, ev(2)) != LMKV_OK || wait(s, ev(3)) != LMKV_OK) return LMKV_ERR_CUDA;
    }
    return LMKV_OK;
}

int check_fp8_pool(const lmkv_pool_t* pool, int32_t chunk_size) {
    const int rc = check_pool(pool);
    if (rc != LMKV_OK) return rc;
    if (pool->elem_bytes != 2) return LMKV_ERR_UNSUPPORTED;
    if (((int64_t)pool->num_kv_heads * pool->head_dim) % 16 != 0) return LMKV_ERR_UNSUPPORTED;
    if (chunk_size > kQuantClusterWide * lmkv::kQuantMaxRows) return LMKV_ERR_UNSUPPORTED;
    return LMKV_OK;
}

// Opt a kernel into `bytes` of dynamic shared memory (once per device).
template <class Kernel>
bool ensure_smem(Kernel kernel, int64_t bytes, std::atomic<int>* cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (cache[dev].load(std::memory_order_relaxed) >= bytes) return true;
    if (cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes)) !=
        LMKV_OK) {
        (void)cudaGetLastError();
        return false;
    }
    if (kQuantClusterWide > 8 &&
        cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != LMKV_OK) {
        (void)cudaGetLastError();
        return false;
    }
    cache[dev].store((int)bytes, std::memory_order_relaxed);
    return true;
}

constexpr int64_t kQuantSmemMax = 200 * 1024;

// Shared-memory bytes of the hybrid quantiser: the slice rows beyond those
// its registers hold.
// Shared memory of one CTA of the staged quantiser with `cluster` CTAs per
// tile: the rows of its slice beyond those its registers hold.
int64_t quant_hybrid_smem_bytes(const Call& c, int cluster) {
    const int64_t row = (int64_t)c.pool->num_kv_heads * c.pool->head_dim * c.pool->elem_bytes;
    const int64_t rows = (c.chunk_size + cluster - 1) / cluster;
    const int64_t reg_rows = (int64_t)kQuantThreads * kQuantHybridVPT * 16 / row;
    return (rows > reg_rows ? rows - reg_rows : 0) * row;
}

// L2 prefetch distance of the staged quantiser, in tiles: half the clusters
// resident at once (occupancy at this shared-memory size x SM count /
// cluster size: 2 x 152 / 4 -> 38 on GB300 at 112 KiB).  Measured on the 8B
// batch (ms): no prefetch 0.373; 19 tiles ahead 0.373, 28 0.351, 38 0.346,
// 48 0.347, 57 0.357, 76 0.376; prefetching before the CTA's own rows have
// arrived was slower at every distance (0.380-0.464).  Cached per device and
// shared-memory size after the first call made outside a stream capture; 0
// (no prefetch) while unknown or if a query fails.
template <class Kernel>
int32_t quant_prefetch_tiles(Kernel kernel, int64_t smem_bytes, int cluster, cudaStream_t stream) {
    static std::mutex mu;
    static std::map<std::pair<int, int64_t>, int32_t> known;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    const auto it = known.find({dev, smem_bytes});
    if (it != known.end()) return it->second;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        (void)cudaGetLastError();
        return 0;
    }
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kQuantThreads, (size_t)smem_bytes) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const int32_t tiles = (int32_t)((int64_t)per_sm * sms / cluster / 2);
    known[{dev, smem_bytes}] = tiles > 0 ? tiles : 0;
    return tiles > 0 ? tiles : 0;
}

template <class B, int kCluster>
int launch_hybrid(const Call& c, float* scales, cudaStream_t stream, int64_t hsmem) {
    auto hyb = lmkv::quant_gather_hybrid_kernel<B, kQuantThreads, kQuantHybridVPT, kCluster>;
    static std::atomic<int> hyb_cache[64];
    const int64_t bytes = hsmem > 16 ? hsmem : 16;
    if (!ensure_smem(hyb, bytes, hyb_cache)) return LMKV_ERR_CUDA;
    Call cq = c;
    cq.prefetch_ahead = quant_prefetch_tiles(hyb, bytes, kCluster, stream);
    return for_each_block<B>(cq, scales, [&](const B& b) {
        const int64_t ctas = (int64_t)b.num_chunks * 2 * b.layer_n * kCluster;
        return launch_pdl_smem(hyb, ctas, kQuantThreads, bytes, stream, b);
    });
}

template <class B>
int launch_quant(const Call& c, float* scales, cudaStream_t stream) {
    if (c.chunk_size <= kQuantCluster * lmkv::kQuantMaxRows) {
        const int64_t h = quant_hybrid_smem_bytes(c, kQuantCluster);
        if (h <= kQuantSmemMax) return launch_hybrid<B, kQuantCluster>(c, scales, stream, h);
    }
    const int64_t h = quant_hybrid_smem_bytes(c, kQuantClusterWide);
    if (h <= kQuantSmemMax) return launch_hybrid<B, kQuantClusterWide>(c, scales, stream, h);
    // rows beyond shared memory: register-staged kernel, re-reading what does not fit
    return for_each_block<B>(c, scales, [&](const B& b) {
        const int64_t ctas = (int64_t)b.num_chunks * 2 * b.layer_n * kQuantClusterWide;
        return launch_pdl(lmkv::quant_gather_kernel<B, kQuantRegThreads, kQuantVPT, kQuantClusterWide>,
                          ctas, kQuantRegThreads, stream, b);
    });
}

template <class B>
int launch_dequant(const Call& c, float* scales, cudaStream_t stream) {
    return for_each_block<B>(c, scales, [&](const B& b) {
        const int64_t items = lmkv::batch_items(b);
        return launch_pdl(lmkv::dequant_scatter_kernel<B, kDequantThreads, kDequantUnroll>, lsu_grid(items),
                          kDequantThreads, stream, b, items);
    });
}

int fp8_entry(bool gather, const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
              const int64_t* start, const int64_t* end, int32_t num_req, int32_t chunk_size,
              int32_t save_unfull, void* const* code_ptrs, float* scales, int32_t* d_status,
              void* stream) {
    int rc = check_fp8_pool(pool, chunk_size);
    if (rc != LMKV_OK) return rc;
    Call c{pool, block_table, max_blocks, start, end, num_req, chunk_size, save_unfull,
           code_ptrs, d_status, 0, pool->num_layers, choose_parts(pool), 0, 0, nullptr};
    rc = validate(c);
    if (rc != LMKV_OK || c.num_chunks == 0) return rc;
    if (scales == nullptr) return LMKV_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    if (c.nonempty <= lmkv::kSmallBatch)
        return gather ? launch_quant<lmkv::BatchSmall>(c, scales, s)
                      : launch_dequant<lmkv::BatchSmall>(c, scales, s);
    return gather ? launch_quant<lmkv::Batch>(c, scales, s) : launch_dequant<lmkv::Batch>(c, scales, s);
}

}  // namespace

// Built-in staging area of lmkv_store_layers_staged_noalloc.  In host code the
// name only stands for the device array: the kernels get its device address,
// looked up once per device with that device current.
static __device__ __align__(256) uint8_t g_noalloc_staging[LMKV_NOALLOC_STAGING_BYTES];

namespace {

// Device address of g_noalloc_staging on the current device (null on error).
// Looked up on every call rather than cached: after a device reset the
// library's module is loaded again and the array may sit elsewhere.  The
// first lookup on a device loads the module there (the set-up).
void* noalloc_staging_address() {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_staging) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return ptr;
}

}  // namespace

void lmkv_internal_add_launches(int64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int lmkv_internal_cuda_status(cudaError_t err) { return cuda_status(err); }

int lmkv_internal_list_chunks(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                              const int64_t* start, const int64_t* end, int32_t num_req,
                              int32_t chunk_size, int32_t save_unfull, std::vector<LmkvChunkRef>* out) {
    Call c{pool, block_table, max_blocks, start, end, num_req, chunk_size, save_unfull,
           nullptr, nullptr, 0, pool ? pool->num_layers : 1, 1, 0, 0, nullptr};
    static void* const kAny = nullptr;
    c.chunk_ptrs = &kAny;                 // the codec passes its blobs separately
    const int rc = validate(c);
    if (rc != LMKV_OK) return rc;
    out->clear();
    for (int32_t r = 0; r < num_req; ++r) {
        const int64_t nch = request_chunks(start[r], end[r], chunk_size, save_unfull);
        for (int64_t j = 0; j < nch; ++j) {
            const int64_t t0 = start[r] + j * chunk_size;
            const int64_t n = end[r] - t0 < chunk_size ? end[r] - t0 : chunk_size;
            out->push_back(LmkvChunkRef{r, t0, (int32_t)n});
        }
    }
    return LMKV_OK;
}

extern "C" {

int lmkv_count_chunks(const int64_t* start, const int64_t* end, int32_t num_req,
                      int32_t chunk_size, int32_t save_unfull_chunk, int32_t* out_num_chunks) {
    if (out_num_chunks == nullptr) return LMKV_ERR_INVALID_ARG;
    int64_t n = 0;
    const int rc = check_requests(start, end, num_req, chunk_size, save_unfull_chunk, &n, nullptr);
    if (rc != LMKV_OK) return rc;
    *out_num_chunks = (int32_t)n;
    return LMKV_OK;
}

int lmkv_enumerate_chunks(const int64_t* start, const int64_t* end, int32_t num_req,
                          int32_t chunk_size, int32_t save_unfull_chunk, int32_t* out_req,
                          int64_t* out_tok0, int32_t* out_ntok, int32_t capacity) {
    int64_t n = 0;
    const int rc = check_requests(start, end, num_req, chunk_size, save_unfull_chunk, &n, nullptr);
    if (rc != LMKV_OK) return rc;
    if (n > capacity) return LMKV_ERR_INVALID_ARG;
    if (n > 0 && (out_req == nullptr || out_tok0 == nullptr || out_ntok == nullptr))
        return LMKV_ERR_INVALID_ARG;
    int64_t g = 0;
    for (int32_t r = 0; r < num_req; ++r) {
        const int64_t nch = request_chunks(start[r], end[r], chunk_size, save_unfull_chunk);
        for (int64_t j = 0; j < nch; ++j, ++g) {
            const int64_t t0 = start[r] + j * chunk_size;
            const int64_t t1 = t0 + chunk_size < end[r] ? t0 + chunk_size : end[r];
            out_req[g] = r;
            out_tok0[g] = t0;
            out_ntok[g] = (int32_t)(t1 - t0);
        }
    }
    return LMKV_OK;
}

int lmkv_decode_store_ranges(const int64_t* stored_end, const int64_t* cur_end, int32_t num_req,
                             int32_t chunk_size, int64_t* out_start, int64_t* out_end,
                             int32_t* out_num_chunks) {
    if (num_req < 0 || chunk_size <= 0 || out_num_chunks == nullptr) return LMKV_ERR_INVALID_ARG;
    if (num_req > 0 && (stored_end == nullptr || cur_end == nullptr || out_start == nullptr ||
                        out_end == nullptr))
        return LMKV_ERR_INVALID_ARG;
    int64_t n = 0;
    for (int32_t r = 0; r < num_req; ++r) {
        const int64_t s = stored_end[r], e = cur_end[r];
        if (s < 0 || e < s || s % chunk_size != 0) return LMKV_ERR_INVALID_ARG;
    }
    for (int32_t r = 0; r < num_req; ++r) {
        const int64_t full = (cur_end[r] - stored_end[r]) / chunk_size;
        out_start[r] = stored_end[r];
        out_end[r] = stored_end[r] + full * chunk_size;
        n += full;
    }
    if (n > INT32_MAX) return LMKV_ERR_INVALID_ARG;
    *out_num_chunks = (int32_t)n;
    return LMKV_OK;
}

// Dynamic offloading of free pages: host-only bookkeeping of the three
// positions; every call keeps start <= current <= end <= limit.
static bool offload_ok(const lmkv_offload_t* st) {
    return st != nullptr && 0 <= st->start && st->start <= st->current && st->current <= st->end &&
           st->end <= st->limit && st->window >= 0;
}

static int64_t offload_target_end(const lmkv_offload_t* st) {
    const int64_t t = st->start + st->window;
    return t < st->limit ? t : st->limit;
}

int lmkv_offload_init(lmkv_offload_t* st, int64_t num_free, int64_t window) {
    if (st == nullptr || num_free < 0 || window < 0) return LMKV_ERR_INVALID_ARG;
    st->start = 0;
    st->current = 0;
    st->limit = num_free;
    st->window = window;
    st->end = offload_target_end(st);
    return LMKV_OK;
}

int lmkv_offload_plan(const lmkv_offload_t* st, int64_t max_pages, int64_t* first, int64_t* count) {
    if (!offload_ok(st) || max_pages < 0 || first == nullptr || count == nullptr)
        return LMKV_ERR_INVALID_ARG;
    const int64_t left = st->end - st->current;
    *first = st->current;
    *count = left < max_pages ? left : max_pages;
    return LMKV_OK;
}

int lmkv_offload_copied(lmkv_offload_t* st, int64_t count) {
    if (!offload_ok(st) || count < 0 || st->current + count > st->end) return LMKV_ERR_INVALID_ARG;
    st->current += count;
    return LMKV_OK;
}

int lmkv_offload_allocate(lmkv_offload_t* st, int64_t want, int64_t* granted, int64_t* stalled) {
    if (!offload_ok(st) || want < 0 || granted == nullptr || stalled == nullptr)
        return LMKV_ERR_INVALID_ARG;
    const int64_t ready = st->current - st->start;
    const int64_t g = want < ready ? want : ready;
    st->start += g;
    const int64_t e = st->end + g;
    st->end = e < st->limit ? e : st->limit;
    *granted = g;
    *stalled = want - g;
    return LMKV_OK;
}

int lmkv_offload_add_free(lmkv_offload_t* st, int64_t n) {
    if (!offload_ok(st) || n < 0) return LMKV_ERR_INVALID_ARG;
    st->limit += n;
    const int64_t t = offload_target_end(st);
    if (st->end < t) st->end = t;
    return LMKV_OK;
}

int lmkv_gather_chunks(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                       const int64_t* start, const int64_t* end, int32_t num_req,
                       int32_t chunk_size, int32_t save_unfull_chunk, void* const* chunk_ptrs,
                       int32_t* d_status, void* stream) {
    return move_entry(true, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                      save_unfull_chunk, chunk_ptrs, -1, d_status, stream);
}

int lmkv_scatter_chunks(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                        const int64_t* start, const int64_t* end, int32_t num_req,
                        int32_t chunk_size, int32_t save_unfull_chunk, void* const* chunk_ptrs,
                        int32_t* d_status, void* stream) {
    return move_entry(false, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                      save_unfull_chunk, chunk_ptrs, -1, d_status, stream);
}

int lmkv_gather_layer(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                      const int64_t* start, const int64_t* end, int32_t num_req,
                      int32_t chunk_size, int32_t save_unfull_chunk, void* const* chunk_ptrs,
                      int32_t layer, int32_t* d_status, void* stream) {
    if (layer < 0) return LMKV_ERR_INVALID_ARG;
    return move_entry(true, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                      save_unfull_chunk, chunk_ptrs, layer, d_status, stream);
}

int lmkv_scatter_layer(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                       const int64_t* start, const int64_t* end, int32_t num_req,
                       int32_t chunk_size, int32_t save_unfull_chunk, void* const* chunk_ptrs,
                       int32_t layer, int32_t* d_status, void* stream) {
    if (layer < 0) return LMKV_ERR_INVALID_ARG;
    return move_entry(false, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                      save_unfull_chunk, chunk_ptrs, layer, d_status, stream);
}

int lmkv_store_layers(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                      const int64_t* start, const int64_t* end, int32_t num_req,
                      int32_t chunk_size, int32_t save_unfull_chunk, void* const* chunk_ptrs,
                      int32_t layer_lo, int32_t layer_n, void* const* layer_ready,
                      void* const* layer_done, int32_t* d_status, void* stream) {
    return layers_entry(true, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                        save_unfull_chunk, chunk_ptrs, layer_lo, layer_n, layer_ready, layer_done,
                        d_status, stream);
}

int lmkv_retrieve_layers(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                         const int64_t* start, const int64_t* end, int32_t num_req,
                         int32_t chunk_size, int32_t save_unfull_chunk, void* const* chunk_ptrs,
                         int32_t layer_lo, int32_t layer_n, void* const* layer_ready,
                         void* const* layer_done, int32_t* d_status, void* stream) {
    return layers_entry(false, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                        save_unfull_chunk, chunk_ptrs, layer_lo, layer_n, layer_ready, layer_done,
                        d_status, stream);
}

int lmkv_store_layers_staged(const lmkv_pool_t* pool, const int32_t* block_table,
                             int32_t max_blocks, const int64_t* start, const int64_t* end,
                             int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                             void* const* host_chunks, void* staging, int64_t staging_bytes,
                             int32_t layer_lo, int32_t layer_n, void* const* layer_ready,
                             void* const* layer_done, int32_t* d_status, void* stream) {
    return staged_entry(true, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                        save_unfull_chunk, host_chunks, staging, staging_bytes, layer_lo, layer_n,
                        layer_ready, layer_done, d_status, stream);
}

int lmkv_retrieve_layers_staged(const lmkv_pool_t* pool, const int32_t* block_table,
                                int32_t max_blocks, const int64_t* start, const int64_t* end,
                                int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                                void* const* host_chunks, void* staging, int64_t staging_bytes,
                                int32_t layer_lo, int32_t layer_n, void* const* layer_ready,
                                void* const* layer_done, int32_t* d_status, void* stream) {
    return staged_entry(false, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                        save_unfull_chunk, host_chunks, staging, staging_bytes, layer_lo, layer_n,
                        layer_ready, layer_done, d_status, stream);
}

int lmkv_store_layers_overlapped(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                                 const int64_t* start, const int64_t* end, int32_t num_req, int32_t chunk_size,
                                 int32_t save_unfull_chunk, void* const* host_chunks, void* staging,
                                 int64_t staging_bytes, int32_t layer_lo, int32_t layer_n,
                                 void* const* layer_ready, void* const* layer_done, void* const* sync_events,
                                 int32_t* d_status, void* stream, void* copy_stream) {
    if (copy_stream == nullptr || copy_stream == stream) return LMKV_ERR_INVALID_ARG;
    return staged_entry(true, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                        save_unfull_chunk, host_chunks, staging, staging_bytes, layer_lo, layer_n,
                        layer_ready, layer_done, d_status, stream, copy_stream, sync_events);
}

int lmkv_retrieve_layers_overlapped(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                                    const int64_t* start, const int64_t* end, int32_t num_req,
                                    int32_t chunk_size, int32_t save_unfull_chunk, void* const* host_chunks,
                                    void* staging, int64_t staging_bytes, int32_t layer_lo, int32_t layer_n,
                                    void* const* layer_ready, void* const* layer_done,
                                    void* const* sync_events, int32_t* d_status, void* stream,
                                    void* copy_stream) {
    if (copy_stream == nullptr || copy_stream == stream) return LMKV_ERR_INVALID_ARG;
    return staged_entry(false, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                        save_unfull_chunk, host_chunks, staging, staging_bytes, layer_lo, layer_n,
                        layer_ready, layer_done, d_status, stream, copy_stream, sync_events);
}

int lmkv_gather_chunks_fp8e4m3(const lmkv_pool_t* pool, const int32_t* block_table,
                               int32_t max_blocks, const int64_t* start, const int64_t* end,
                               int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                               void* const* code_ptrs, float* scales, int32_t* d_status,
                               void* stream) {
    return fp8_entry(true, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                     save_unfull_chunk, code_ptrs, scales, d_status, stream);
}

int lmkv_scatter_chunks_fp8e4m3(const lmkv_pool_t* pool, const int32_t* block_table,
                                int32_t max_blocks, const int64_t* start, const int64_t* end,
                                int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                                void* const* code_ptrs, const float* scales, int32_t* d_status,
                                void* stream) {
    return fp8_entry(false, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                     save_unfull_chunk, code_ptrs, const_cast<float*>(scales), d_status, stream);
}

const char* lmkv_status_string(int status) {
    switch (status) {
        case LMKV_OK: return "ok";
        case LMKV_ERR_INVALID_ARG: return "invalid argument";
        case LMKV_ERR_MISALIGNED: return "row bytes or pointer not 16-byte aligned";
        case LMKV_ERR_CUDA: return "CUDA launch failed";
        case LMKV_ERR_UNSUPPORTED: return "unsupported pool format for this entry point";
        case LMKV_ERR_BAD_BLOCK: return "block id out of range (token skipped)";
        case LMKV_ERR_BAD_POINTER: return "null or misaligned device pointer in an array (skipped)";
        case LMKV_ERR_TIMEOUT: return "bounded device wait gave up";
        case LMKV_ERR_SCRATCH_LIMIT: return "batch needs more than the built-in staging area";
        case LMKV_ERR_BAD_DATA: return "encoded blob inconsistent with its size (stream skipped)";
        default: return "unknown status";
    }
}

// lmkv_store_layers_staged_noalloc: the staged store with the library's own
// staging area, for callers that must not allocate device memory.
int lmkv_store_layers_staged_noalloc(const lmkv_pool_t* pool, const int32_t* block_table,
                                     int32_t max_blocks, const int64_t* start, const int64_t* end,
                                     int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                                     void* const* host_chunks, int32_t layer_lo, int32_t layer_n,
                                     void* const* layer_ready, void* const* layer_done,
                                     int32_t* d_status, void* stream) {
    const int rc = check_pool(pool);
    if (rc != LMKV_OK) return rc;
    int64_t chunks = 0;
    if (check_requests(start, end, num_req, chunk_size, save_unfull_chunk, &chunks, nullptr) != LMKV_OK)
        return LMKV_ERR_INVALID_ARG;
    // Tokens the staging area can hold (K and V rows of one layer); each
    // request's count is checked against what is left before it is added, so
    // no product or sum can overflow whatever the offsets are.
    const int64_t row = (int64_t)pool->num_kv_heads * pool->head_dim * pool->elem_bytes;
    const int64_t cap = (int64_t)LMKV_NOALLOC_STAGING_BYTES / (2 * row);
    int64_t tokens = 0;
    for (int32_t r = 0; r < num_req; ++r) {
        if (request_chunks(start[r], end[r], chunk_size, save_unfull_chunk) == 0) continue;
        const int64_t n = save_unfull_chunk ? end[r] - start[r] : (end[r] - start[r]) / chunk_size * chunk_size;
        if (n > cap - tokens) return LMKV_ERR_SCRATCH_LIMIT;
        tokens += n;
    }
    void* staging = noalloc_staging_address();
    if (staging == nullptr) return LMKV_ERR_CUDA;
    return staged_entry(true, pool, block_table, max_blocks, start, end, num_req, chunk_size,
                        save_unfull_chunk, host_chunks, staging, (int64_t)LMKV_NOALLOC_STAGING_BYTES,
                        layer_lo, layer_n, layer_ready, layer_done, d_status, stream);
}

int lmkv_abi_version(void) { return LMKV_ABI_VERSION; }

int64_t lmkv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int lmkv_last_cuda_error(void) { return g_last_cuda_error.load(std::memory_order_relaxed); }

const char* lmkv_cuda_error_name(int err) { return cudaGetErrorName((cudaError_t)err); }

}  // extern "C"
