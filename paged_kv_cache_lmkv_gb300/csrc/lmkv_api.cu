// lmkv_api.cu -- host side of the C ABI declared in include/lmkv.h.
//
// Validates arguments, enumerates chunks (cache_engine.py walk-through,
// "store()" section: chunk_size chunks, short tail only with
// save_unfull_chunk, chunk-aligned start), packs up to kMaxReqPerLaunch
// requests into one by-value parameter block per launch, and enqueues the
// kernels of lmkv_kernels.cuh on the caller's stream.  Nothing is allocated
// and nothing is synchronised.
#include "lmkv.h"
#include "lmkv_kernels.cuh"

#include <atomic>
#include <cstring>
#include <vector>

namespace {

using lmkv::Batch;

std::atomic<int64_t> g_launches{0};

// Copy engine configuration (chosen by measurement on GB300; see the kernel
// header for the two engines).
constexpr int kLsuThreads = 256;
constexpr int kLsuUnroll = 8;
constexpr int kQuantThreads = 512;
constexpr int kQuantVPT = 8;
constexpr int kQuantCluster = 8;
constexpr int kDequantThreads = 256;

struct ChunkSpan {
    int32_t req;
    int64_t tok0;
    int32_t ntok;
};

// Host-side chunk enumeration; returns LMKV_OK and fills `out` (if given).
int enumerate(const int64_t* start, const int64_t* end, int32_t num_req, int32_t chunk_size,
              int32_t save_unfull, std::vector<ChunkSpan>* out, int64_t* count) {
    if (num_req < 0 || chunk_size <= 0) return LMKV_ERR_INVALID_ARG;
    if (num_req > 0 && (start == nullptr || end == nullptr)) return LMKV_ERR_INVALID_ARG;
    int64_t n = 0;
    for (int32_t r = 0; r < num_req; ++r) {
        const int64_t s = start[r], e = end[r];
        if (s < 0 || e < s || s % chunk_size != 0) return LMKV_ERR_INVALID_ARG;
        const int64_t len = e - s;
        int64_t full = len / chunk_size;
        const int64_t tail = len % chunk_size;
        const int64_t nch = full + ((save_unfull && tail) ? 1 : 0);
        if (out != nullptr) {
            for (int64_t j = 0; j < nch; ++j) {
                const int64_t t0 = s + j * chunk_size;
                const int64_t t1 = (t0 + chunk_size < e) ? t0 + chunk_size : e;
                out->push_back({r, t0, (int32_t)(t1 - t0)});
            }
        }
        n += nch;
    }
    if (n > INT32_MAX) return LMKV_ERR_INVALID_ARG;
    *count = n;
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

// Validate a call and build its launch parameter blocks.
int prepare(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
            const int64_t* start, const int64_t* end, int32_t num_req, int32_t chunk_size,
            int32_t save_unfull, void* const* chunk_ptrs, int32_t* d_status, int32_t layer_lo,
            int32_t layer_n, int32_t parts, std::vector<Batch>* launches) {
    int rc = check_pool(pool);
    if (rc != LMKV_OK) return rc;
    if (chunk_size <= 0 || chunk_size % pool->block_size != 0) return LMKV_ERR_INVALID_ARG;
    if (max_blocks < 0 || num_req < 0) return LMKV_ERR_INVALID_ARG;
    if (layer_lo < 0 || layer_n <= 0 || layer_lo + layer_n > pool->num_layers)
        return LMKV_ERR_INVALID_ARG;
    if (pool->block_size % parts != 0) parts = 1;
    std::vector<ChunkSpan> chunks;
    int64_t nch = 0;
    rc = enumerate(start, end, num_req, chunk_size, save_unfull, &chunks, &nch);
    if (rc != LMKV_OK) return rc;
    for (int32_t r = 0; r < num_req; ++r) {
        if (end[r] > start[r] && (end[r] - 1) / pool->block_size >= max_blocks)
            return LMKV_ERR_INVALID_ARG;
    }
    if (nch == 0) return LMKV_OK;
    if (block_table == nullptr || chunk_ptrs == nullptr) return LMKV_ERR_INVALID_ARG;

    Batch base;
    std::memset(&base, 0, sizeof(base));
    base.layer_base = reinterpret_cast<const uint8_t* const*>(pool->layer_base);
    base.chunk_ptrs = reinterpret_cast<uint8_t* const*>(chunk_ptrs);
    base.block_table = block_table;
    base.status = d_status;
    base.num_blocks = pool->num_blocks;
    base.bt_stride = max_blocks;
    base.num_layers = pool->num_layers;
    base.row_bytes = pool->num_kv_heads * pool->head_dim * pool->elem_bytes;
    base.block_size = pool->block_size;
    base.chunk_size = chunk_size;
    base.blocks_per_chunk = chunk_size / pool->block_size;
    base.parts = parts;
    base.layer_lo = layer_lo;
    base.layer_n = layer_n;

    // Pack requests with at least one chunk, kMaxReqPerLaunch per launch.
    Batch cur = base;
    int32_t g = 0;
    size_t ci = 0;
    while (ci < chunks.size()) {
        const int32_t r = chunks[ci].req;
        size_t cj = ci;
        while (cj < chunks.size() && chunks[cj].req == r) ++cj;
        if (cur.num_req == lmkv::kMaxReqPerLaunch) {
            launches->push_back(cur);
            const int32_t next_base = cur.chunk_base + cur.num_chunks;
            cur = base;
            cur.chunk_base = next_base;
        }
        const int i = cur.num_req++;
        cur.req_row[i] = r;
        cur.req_chunk_begin[i] = cur.num_chunks;
        cur.req_tok0[i] = chunks[ci].tok0;
        cur.req_tok_end[i] = chunks[cj - 1].tok0 + chunks[cj - 1].ntok;
        cur.num_chunks += (int32_t)(cj - ci);
        cur.req_chunk_begin[i + 1] = cur.num_chunks;
        g += (int32_t)(cj - ci);
        ci = cj;
    }
    if (cur.num_req > 0) launches->push_back(cur);
    (void)g;
    return LMKV_OK;
}

int finish_launch() {
    const cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? LMKV_OK : LMKV_ERR_CUDA;
}

// Number of CTAs the LSU engine launches for `items` items.
int64_t lsu_grid(int64_t items) {
    const int64_t cap = (int64_t)1 << 30;
    return items < cap ? items : cap;
}

template <bool kGather>
int launch_move(const std::vector<Batch>& launches, cudaStream_t stream) {
    for (const Batch& b : launches) {
        const int64_t items = lmkv::batch_items(b);
        if (items == 0) continue;
        lmkv::move_lsu_kernel<kGather, kLsuThreads, kLsuUnroll>
            <<<(unsigned)lsu_grid(items), kLsuThreads, 0, stream>>>(b, items);
        g_launches.fetch_add(1, std::memory_order_relaxed);
        const int rc = finish_launch();
        if (rc != LMKV_OK) return rc;
    }
    return LMKV_OK;
}

// Parts per block: split runs when the call has too few items to fill the GPU.
int32_t choose_parts(const lmkv_pool_t* pool, int32_t layer_n) {
    return layer_n == 1 && pool->block_size % 2 == 0 ? 2 : 1;
}

int move_entry(bool gather, const lmkv_pool_t* pool, const int32_t* block_table,
               int32_t max_blocks, const int64_t* start, const int64_t* end, int32_t num_req,
               int32_t chunk_size, int32_t save_unfull, void* const* chunk_ptrs,
               int32_t layer, int32_t* d_status, void* stream) {
    const int rc0 = check_pool(pool);
    if (rc0 != LMKV_OK) return rc0;
    int32_t lo = 0, n = pool->num_layers;
    if (layer >= 0) {
        if (layer >= pool->num_layers) return LMKV_ERR_INVALID_ARG;
        lo = layer;
        n = 1;
    }
    std::vector<Batch> launches;
    const int rc = prepare(pool, block_table, max_blocks, start, end, num_req, chunk_size,
                           save_unfull, chunk_ptrs, d_status, lo, n, choose_parts(pool, n),
                           &launches);
    if (rc != LMKV_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return gather ? launch_move<true>(launches, s) : launch_move<false>(launches, s);
}

int check_fp8_pool(const lmkv_pool_t* pool, int32_t chunk_size) {
    const int rc = check_pool(pool);
    if (rc != LMKV_OK) return rc;
    if (pool->elem_bytes != 2) return LMKV_ERR_UNSUPPORTED;
    if (((int64_t)pool->num_kv_heads * pool->head_dim) % 16 != 0) return LMKV_ERR_UNSUPPORTED;
    if (chunk_size > kQuantCluster * lmkv::kQuantMaxRows) return LMKV_ERR_UNSUPPORTED;
    return LMKV_OK;
}

}  // namespace

extern "C" {

int lmkv_count_chunks(const int64_t* start, const int64_t* end, int32_t num_req,
                      int32_t chunk_size, int32_t save_unfull_chunk, int32_t* out_num_chunks) {
    if (out_num_chunks == nullptr) return LMKV_ERR_INVALID_ARG;
    int64_t n = 0;
    const int rc = enumerate(start, end, num_req, chunk_size, save_unfull_chunk, nullptr, &n);
    if (rc != LMKV_OK) return rc;
    *out_num_chunks = (int32_t)n;
    return LMKV_OK;
}

int lmkv_enumerate_chunks(const int64_t* start, const int64_t* end, int32_t num_req,
                          int32_t chunk_size, int32_t save_unfull_chunk, int32_t* out_req,
                          int64_t* out_tok0, int32_t* out_ntok, int32_t capacity) {
    std::vector<ChunkSpan> chunks;
    int64_t n = 0;
    const int rc = enumerate(start, end, num_req, chunk_size, save_unfull_chunk, &chunks, &n);
    if (rc != LMKV_OK) return rc;
    if (n > capacity) return LMKV_ERR_INVALID_ARG;
    if (n > 0 && (out_req == nullptr || out_tok0 == nullptr || out_ntok == nullptr))
        return LMKV_ERR_INVALID_ARG;
    for (int64_t g = 0; g < n; ++g) {
        out_req[g] = chunks[g].req;
        out_tok0[g] = chunks[g].tok0;
        out_ntok[g] = chunks[g].ntok;
    }
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

int lmkv_gather_chunks_fp8e4m3(const lmkv_pool_t* pool, const int32_t* block_table,
                               int32_t max_blocks, const int64_t* start, const int64_t* end,
                               int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                               void* const* code_ptrs, float* scales, int32_t* d_status,
                               void* stream) {
    int rc = check_fp8_pool(pool, chunk_size);
    if (rc != LMKV_OK) return rc;
    std::vector<Batch> launches;
    rc = prepare(pool, block_table, max_blocks, start, end, num_req, chunk_size,
                 save_unfull_chunk, code_ptrs, d_status, 0, pool->num_layers, 1, &launches);
    if (rc != LMKV_OK) return rc;
    if (!launches.empty() && scales == nullptr) return LMKV_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (Batch& b : launches) {
        b.scales = scales;
        const int64_t tiles = (int64_t)b.num_chunks * 2 * b.layer_n;
        const int64_t ctas = tiles * kQuantCluster;
        if (ctas > INT32_MAX) return LMKV_ERR_INVALID_ARG;
        lmkv::quant_gather_kernel<kQuantThreads, kQuantVPT, kQuantCluster>
            <<<(unsigned)ctas, kQuantThreads, 0, s>>>(b);
        g_launches.fetch_add(1, std::memory_order_relaxed);
        rc = finish_launch();
        if (rc != LMKV_OK) return rc;
    }
    return LMKV_OK;
}

int lmkv_scatter_chunks_fp8e4m3(const lmkv_pool_t* pool, const int32_t* block_table,
                                int32_t max_blocks, const int64_t* start, const int64_t* end,
                                int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                                void* const* code_ptrs, const float* scales, int32_t* d_status,
                                void* stream) {
    int rc = check_fp8_pool(pool, chunk_size);
    if (rc != LMKV_OK) return rc;
    std::vector<Batch> launches;
    rc = prepare(pool, block_table, max_blocks, start, end, num_req, chunk_size,
                 save_unfull_chunk, code_ptrs, d_status, 0, pool->num_layers, 1, &launches);
    if (rc != LMKV_OK) return rc;
    if (!launches.empty() && scales == nullptr) return LMKV_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (Batch& b : launches) {
        b.scales = const_cast<float*>(scales);
        const int64_t items = lmkv::batch_items(b);
        lmkv::dequant_scatter_kernel<kDequantThreads>
            <<<(unsigned)lsu_grid(items), kDequantThreads, 0, s>>>(b, items);
        g_launches.fetch_add(1, std::memory_order_relaxed);
        rc = finish_launch();
        if (rc != LMKV_OK) return rc;
    }
    return LMKV_OK;
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
        default: return "unknown status";
    }
}

int lmkv_abi_version(void) { return LMKV_ABI_VERSION; }

int64_t lmkv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
