/*
 * lmkv.h -- C ABI of liblmkv.so: batched paged-KV chunk gather / scatter on
 * GB300 (sm_103a).
 *
 * What the calls compute.  An inference engine keeps each layer's KV cache
 * in small fixed-size pages ("blocks") of block_size tokens, addressed per
 * request through a block table.  LMCache moves KV cache in large chunks
 * instead of pages: a GPU kernel copies the scattered pages of many layers
 * into a contiguous streaming buffer of 256-token chunks, which is then moved
 * as a whole; on load the chunks are split back into pages by a kernel
 * ("LMCache: An Efficient KV Cache Layer for Enterprise-Scale LLM Inference",
 * section on the configurable chunk size).  The layer-wise pipeline moves one
 * layer at a time so that transfer overlaps compute (same paper, section on
 * the layer-wise pipeline).  The store entry point of the engine cuts tokens
 * into chunk_size chunks, keeps a tail shorter than a chunk only when
 * save_unfull_chunk is set, and requires the already-cached prefix to be a
 * multiple of chunk_size ("LMCache 源码解析", cache_engine.py walk-through,
 * section "store()").
 *
 * Notation: L = num_layers, HD = num_kv_heads * head_dim, e = elem_bytes,
 * B = block_size, C = chunk_size, row = HD * e bytes (one token of K or V of
 * one layer).
 *
 * Layouts (all row-major, contiguous):
 *   pool layer l  : [2][num_blocks][B][HD]   (index 0 = K, 1 = V)
 *   block table   : int32 [num_req][max_blocks]; entry [r][t / B] is the
 *                   block that holds token t of request r
 *   chunk g       : [2][L][n_g][HD]           (n_g = tokens in chunk g)
 *   fp8 codes g   : uint8 [2][L][n_g][HD]     (float8 e4m3fn bit patterns)
 *   fp8 scales    : float32 [num_chunks][2][L]
 *
 * Chunk enumeration.  Request r covers tokens [start[r], end[r]) with
 * start[r] % C == 0.  Its chunk j covers [start + j*C, min(start+(j+1)*C, end));
 * a chunk shorter than C exists only as the request's last chunk and only
 * when save_unfull_chunk != 0.  Chunks are numbered request by request; that
 * number g indexes chunk_ptrs / code_ptrs / scales.
 *
 * Ownership and synchronisation.  The caller owns every buffer.  The library
 * allocates nothing, never synchronises, and returns right after enqueueing
 * its kernels on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 * default stream).  Pointers marked DEVICE must be device memory of the
 * current device; HOST arrays are read before the call returns.
 *
 * CUDA graphs.  Calls can be captured in a CUDA graph.  The first call of an
 * entry point on a device sets kernel attributes (the shared-memory size of
 * the fp8 quantiser and of the CacheGen kernels) and looks up the kernels'
 * occupancy, which sizes the L2 prefetch distances; make that first call
 * outside any stream capture (a warm-up call).  A call whose occupancy
 * lookup has not happened yet makes none while its stream is capturing, and
 * runs without the L2 prefetch.
 *
 * Errors.  Every call returns an lmkv_status value.  Argument errors are
 * detected on the host before anything is launched (nothing is written).
 * Errors found by the kernels (a block id outside [0, num_blocks), a null or
 * misaligned device pointer inside the pointer arrays) skip the affected
 * rows, move everything else, and store the code into *d_status (a DEVICE
 * int32 the caller zeroes beforehand; may be NULL) -- readable after the
 * stream has been synchronised.  Kernels never trap and never wait on a flag.
 *
 * Preconditions the library cannot check cheaply: block ids written by a
 * scatter must be distinct across the batch (otherwise the result depends on
 * write order); chunk buffers must not overlap the pool.
 */
#ifndef LMKV_H
#define LMKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LMKV_ABI_VERSION 1

typedef enum lmkv_status {
    LMKV_OK = 0,
    LMKV_ERR_INVALID_ARG = 1,   /* host: bad size, null pointer, unaligned start, short table */
    LMKV_ERR_MISALIGNED = 2,    /* host: row bytes or a host-visible pointer not 16-byte aligned */
    LMKV_ERR_CUDA = 3,          /* host: a CUDA launch or attribute call failed */
    LMKV_ERR_UNSUPPORTED = 4,   /* host: e.g. the fp8 variant on a pool that is not bf16 */
    LMKV_ERR_BAD_BLOCK = 5,     /* device: a block id outside [0, num_blocks); token skipped */
    LMKV_ERR_BAD_POINTER = 6,   /* device: null or misaligned entry in a pointer array; skipped */
    LMKV_ERR_TIMEOUT = 7,       /* device: an asynchronous copy did not complete within 1 s (the
                                   tile's codes are not written; the CTA waits up to 10 s more
                                   for the copy before it exits).  The GPU is then not serving
                                   memory requests: treat the context as unusable. */
    LMKV_ERR_SCRATCH_LIMIT = 8, /* host: the batch needs more than the library's built-in scratch */
    LMKV_ERR_BAD_DATA = 9       /* device: an encoded blob is inconsistent (stream skipped) */
} lmkv_status;

/* The paged KV pool.  layer_base is a DEVICE array of num_layers DEVICE
 * pointers, each to one layer's [2][num_blocks][B][HD] pool (16-byte
 * aligned).  The struct itself is read on the host during the call. */
typedef struct lmkv_pool {
    void* const* layer_base;
    int64_t num_blocks;
    int32_t num_layers;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t elem_bytes;     /* 2 for bf16 / fp16; 1 and 4 also accepted by the copies */
} lmkv_pool_t;

/* Number of chunks of a batch (host only, no CUDA).  Returns
 * LMKV_ERR_INVALID_ARG for num_req < 0, chunk_size <= 0, start < 0,
 * end < start, or start % chunk_size != 0. */
int lmkv_count_chunks(const int64_t* start, const int64_t* end, int32_t num_req,
                      int32_t chunk_size, int32_t save_unfull_chunk,
                      int32_t* out_num_chunks);

/* The chunk list itself (host only): for chunk g, its request, first token
 * and token count n_g.  `capacity` is the length of the three HOST output
 * arrays; LMKV_ERR_INVALID_ARG if it is smaller than the chunk count. */
int lmkv_enumerate_chunks(const int64_t* start, const int64_t* end, int32_t num_req,
                          int32_t chunk_size, int32_t save_unfull_chunk,
                          int32_t* out_req, int64_t* out_tok0, int32_t* out_ntok,
                          int32_t capacity);

/* Deferred decode-KV store (LMCache paper, section on delayed storing of
 * decode KV: instead of writing every generated token's KV, buffer it and
 * store in batch once a whole chunk has been generated).  The decode KV stays
 * in the paged pool; this host-only helper turns each request's stored prefix
 * and current length into the range of chunks completed since the last store:
 *   out_start[r] = stored_end[r]
 *   out_end[r]   = stored_end[r] + floor((cur_end[r] - stored_end[r]) / C) * C
 * and *out_num_chunks = the number of those chunks.  Passing out_start /
 * out_end with save_unfull_chunk = 0 to lmkv_gather_chunks (or a staged
 * store) stores exactly them; the caller then sets stored_end = out_end.
 * INVALID_ARG if a stored_end is not a multiple of chunk_size, is negative, or
 * exceeds cur_end.  All arrays are HOST, num_req entries. */
int lmkv_decode_store_ranges(const int64_t* stored_end, const int64_t* cur_end, int32_t num_req,
                             int32_t chunk_size, int64_t* out_start, int64_t* out_end,
                             int32_t* out_num_chunks);

/* Dynamic offloading of free pages (LMCache paper, section on the dynamic
 * offloading mechanism and its Figure 7).  The engine keeps freed pages, whose
 * KV is still valid, in an ordered free list; before a freed page is handed
 * to a new query its KV is backed up to CPU memory, so it stays reusable.
 * Only part of the free list is backed up, tracked by three positions in the
 * free-list order, with start <= current <= end at all times:
 *   start   : the next free page the engine will hand out;
 *   current : pages before it have been backed up;
 *   end     : pages before it are planned for backup.
 * The four states of the mechanism: #1 initialised (current == start),
 * #2 in progress (current moves toward end), #3 a query arrives (it takes
 * backed-up pages from start, and end moves forward by the number taken),
 * #4 steady (current == end: every planned page is backed up).  A larger
 * window (end - start) makes it less likely that a query must wait for
 * backups, at the cost of more copying.  The struct is caller-owned; these
 * calls are host-only and never touch the GPU.  The backup copy of positions
 * [current, current + count) is an ordinary store with block_size-token
 * chunks (one page per chunk) whose block table is the free list, e.g.
 * lmkv_store_layers_staged with start = current * B, end = (current+count) * B,
 * chunk_size = B. */
typedef struct lmkv_offload {
    int64_t start;
    int64_t current;
    int64_t end;
    int64_t limit;    /* free-list positions that exist (pages freed so far) */
    int64_t window;   /* planned backup pages beyond start: end - start <= window */
} lmkv_offload_t;

/* State #1: start = current = 0, end = min(window, num_free).  INVALID_ARG for
 * negative sizes or a null state. */
int lmkv_offload_init(lmkv_offload_t* st, int64_t num_free, int64_t window);

/* The next backup range: *first = current, *count = min(max_pages, end - current).
 * A count of 0 means steady state (#4). */
int lmkv_offload_plan(const lmkv_offload_t* st, int64_t max_pages, int64_t* first,
                      int64_t* count);

/* Record that `count` planned pages starting at `current` were backed up
 * (state #2).  INVALID_ARG if that would pass end. */
int lmkv_offload_copied(lmkv_offload_t* st, int64_t count);

/* A query takes up to `want` pages from start (state #3).  Only backed-up
 * pages can be handed out: *granted = min(want, current - start); start and
 * end advance by *granted (end capped at limit); *stalled = want - *granted
 * pages must wait for backups. */
int lmkv_offload_allocate(lmkv_offload_t* st, int64_t want, int64_t* granted, int64_t* stalled);

/* `n` more pages were freed (appended to the free-list order): limit += n,
 * and end grows toward start + window. */
int lmkv_offload_add_free(lmkv_offload_t* st, int64_t n);

/* Store path: X_g[kv][l][t][:] = P_l[kv][BT[r][tok/B]][tok % B][:] for every
 * chunk g (request r, tok = first token of g + t), kv, layer l, t < n_g.
 * Configurable chunk size section of the LMCache paper (pages -> contiguous
 * chunk buffer).
 *   pool        : the paged pool (see lmkv_pool_t)
 *   block_table : DEVICE int32 [num_req][max_blocks]
 *   start, end  : HOST int64 [num_req]
 *   chunk_ptrs  : DEVICE array [num_chunks] of DEVICE pointers, chunk g's
 *                 buffer [2][L][n_g][HD], 16-byte aligned
 *   d_status    : DEVICE int32 or NULL
 * Host errors: INVALID_ARG (null pool/arrays, sizes <= 0, chunk_size not a
 * multiple of block_size, unaligned start, end needing a column >= max_blocks),
 * MISALIGNED (row bytes not a multiple of 16), CUDA. */
int lmkv_gather_chunks(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                       const int64_t* start, const int64_t* end, int32_t num_req,
                       int32_t chunk_size, int32_t save_unfull_chunk,
                       void* const* chunk_ptrs, int32_t* d_status, void* stream);

/* Retrieve path: the inverse copy, P_l[kv][BT[r][tok/B]][tok % B][:] =
 * X_g[kv][l][t][:], writing exactly the enumerated tokens (other slots of a
 * partially covered block keep their contents).  Same arguments; chunk
 * buffers are read.  Same section of the LMCache paper (chunks -> pages). */
int lmkv_scatter_chunks(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                        const int64_t* start, const int64_t* end, int32_t num_req,
                        int32_t chunk_size, int32_t save_unfull_chunk,
                        void* const* chunk_ptrs, int32_t* d_status, void* stream);

/* Layer-wise store: lmkv_gather_chunks restricted to one layer `layer`
 * (0 <= layer < L); only the X_g[kv][layer] slices of every chunk are
 * written.  Calls for layer = 0..L-1 together equal one lmkv_gather_chunks.
 * LMCache paper, layer-wise pipeline section (one layer's KV per transfer).
 * INVALID_ARG if layer is out of range; otherwise as lmkv_gather_chunks. */
int lmkv_gather_layer(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                      const int64_t* start, const int64_t* end, int32_t num_req,
                      int32_t chunk_size, int32_t save_unfull_chunk,
                      void* const* chunk_ptrs, int32_t layer, int32_t* d_status, void* stream);

/* Layer-wise retrieve: lmkv_scatter_chunks restricted to one layer. */
int lmkv_scatter_layer(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                       const int64_t* start, const int64_t* end, int32_t num_req,
                       int32_t chunk_size, int32_t save_unfull_chunk,
                       void* const* chunk_ptrs, int32_t layer, int32_t* d_status, void* stream);

/* Layer-wise pipeline (LMCache paper, layer-wise pipeline section: compute and
 * data movement on separate CUDA streams; while layer i computes, layer i+1's
 * KV is being moved; connector hooks start_store_kv / wait_store_kv and
 * start_load_kv / wait_load_kv).
 *
 * lmkv_store_layers: for each layer l = layer_lo .. layer_lo+layer_n-1 in order,
 * make `stream` (the copy stream) wait on layer_ready[l - layer_lo] if that
 * entry is non-NULL, enqueue lmkv_gather_layer(l), then record
 * layer_done[l - layer_lo] on `stream` if non-NULL.  lmkv_retrieve_layers does
 * the same with lmkv_scatter_layer.  A typical store records layer_ready[i] on
 * the compute stream after layer i's KV is written; a typical retrieve lets the
 * compute stream wait on layer_done[i] before computing layer i.
 *   layer_ready, layer_done : HOST arrays of layer_n cudaEvent_t handles (as
 *                             void*), or NULL; entries may be NULL.  The events
 *                             must exist (created by the caller).
 *   chunk_ptrs              : as lmkv_gather_chunks; the buffers may be pinned
 *                             host memory mapped into the device address space,
 *                             in which case the kernels are the host transfer.
 * Nothing is allocated or synchronised.  Errors: as lmkv_gather_layer, checked
 * for the whole call before anything is enqueued; LMKV_ERR_CUDA if an event
 * wait or record fails (earlier layers may already be enqueued). */
int lmkv_store_layers(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                      const int64_t* start, const int64_t* end, int32_t num_req,
                      int32_t chunk_size, int32_t save_unfull_chunk, void* const* chunk_ptrs,
                      int32_t layer_lo, int32_t layer_n, void* const* layer_ready,
                      void* const* layer_done, int32_t* d_status, void* stream);

int lmkv_retrieve_layers(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                         const int64_t* start, const int64_t* end, int32_t num_req,
                         int32_t chunk_size, int32_t save_unfull_chunk, void* const* chunk_ptrs,
                         int32_t layer_lo, int32_t layer_n, void* const* layer_ready,
                         void* const* layer_done, int32_t* d_status, void* stream);

/* Staged layer-wise pipeline to / from pinned host memory (the same section
 * of the LMCache paper: a GPU buffer of one layer's KV between the paged pool
 * and the DMA engine).  Per layer l (in order; layer_ready / layer_done as in
 * lmkv_store_layers):
 *   store    : gather layer l into `staging`, then one cudaMemcpy2DAsync per
 *              chunk moves that chunk's K and V slices of layer l from
 *              `staging` to host_chunks[g] (device-to-host);
 *   retrieve : the 2-D copies move the slices from host_chunks[g] into
 *              `staging` (host-to-device), then layer l is scattered from it.
 * A run of full chunks whose host buffers follow each other in memory is
 * first tried as one cudaMemcpy3DAsync per layer (much cheaper to issue than
 * one copy per chunk); the driver accepts that only when the run lies in one
 * allocation, and otherwise the run is copied chunk by chunk.
 * The copies run on the copy engine, so the transfer uses no SMs while it
 * overlaps compute on another stream; only the short gather / scatter kernel
 * needs SMs.
 *   host_chunks   : HOST array [num_chunks] of pinned HOST pointers, chunk g's
 *                   buffer [2][L][n_g][HD] (the layout of lmkv_gather_chunks)
 *   staging       : DEVICE buffer, 16-byte aligned, of staging_bytes >=
 *                   2 * row_bytes * (tokens enumerated in the batch) -- one
 *                   layer of the batch; chunk g's slices sit at
 *                   2 * row_bytes * (tokens of the chunks before g)
 * Everything is enqueued on `stream`; consecutive layers reuse the staging
 * buffer in stream order.  A retrieve waits on layer_ready[i] just before layer
 * i's scatter (its host-to-staging copies do not touch the pool).  Errors: as lmkv_store_layers; INVALID_ARG if the
 * staging buffer is null or too small or a host pointer is null; MISALIGNED
 * if staging is not 16-byte aligned. */
int lmkv_store_layers_staged(const lmkv_pool_t* pool, const int32_t* block_table,
                             int32_t max_blocks, const int64_t* start, const int64_t* end,
                             int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                             void* const* host_chunks, void* staging, int64_t staging_bytes,
                             int32_t layer_lo, int32_t layer_n, void* const* layer_ready,
                             void* const* layer_done, int32_t* d_status, void* stream);

int lmkv_retrieve_layers_staged(const lmkv_pool_t* pool, const int32_t* block_table,
                                int32_t max_blocks, const int64_t* start, const int64_t* end,
                                int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                                void* const* host_chunks, void* staging, int64_t staging_bytes,
                                int32_t layer_lo, int32_t layer_n, void* const* layer_ready,
                                void* const* layer_done, int32_t* d_status, void* stream);

/* The staged pipeline with two staging buffers and the copies on their own
 * stream, so that layer l's copies overlap layer l+1's gather (store) and
 * layer l's scatter overlaps layer l+1's copies (retrieve): on one stream the
 * kernel and the copies of every layer take turns on the link.
 *   staging      : DEVICE, 16-byte aligned, staging_bytes >= 2 layers of the
 *                  batch (2 * 2 * row_bytes * tokens); layer i uses half i % 2
 *   stream       : the kernels (and, for store, the end of the call: it
 *                  waits for the last copies); copy_stream: the copies, a
 *                  different caller-owned stream
 *   sync_events  : HOST array of 4 caller-owned cudaEvent_t (as void*): the
 *                  library records and waits on them to order the two
 *                  streams (event b: kernel on half b done; event 2 + b: copies
 *                  of half b done); the copy stream first waits for the work
 *                  already on `stream`
 *   layer_ready  : waited on `stream` before layer i's kernel
 *   layer_done   : store: recorded on copy_stream after layer i's copies
 *                  (its rows are on the host); retrieve: recorded on `stream`
 *                  after layer i's scatter
 * Other arguments, layouts and errors as lmkv_store_layers_staged; also
 * INVALID_ARG for a null copy stream, copy_stream == stream, or a null event.
 * Nothing is allocated; the calls can be captured in a CUDA graph. */
int lmkv_store_layers_overlapped(const lmkv_pool_t* pool, const int32_t* block_table,
                                 int32_t max_blocks, const int64_t* start, const int64_t* end,
                                 int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                                 void* const* host_chunks, void* staging, int64_t staging_bytes,
                                 int32_t layer_lo, int32_t layer_n, void* const* layer_ready,
                                 void* const* layer_done, void* const* sync_events, int32_t* d_status,
                                 void* stream, void* copy_stream);

int lmkv_retrieve_layers_overlapped(const lmkv_pool_t* pool, const int32_t* block_table,
                                    int32_t max_blocks, const int64_t* start, const int64_t* end,
                                    int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                                    void* const* host_chunks, void* staging, int64_t staging_bytes,
                                    int32_t layer_lo, int32_t layer_n, void* const* layer_ready,
                                    void* const* layer_done, void* const* sync_events,
                                    int32_t* d_status, void* stream, void* copy_stream);

/* Size of the built-in staging area of lmkv_store_layers_staged_noalloc. */
#define LMKV_NOALLOC_STAGING_BYTES (64u << 20)

/* lmkv_store_layers_staged without a caller-provided staging buffer, for
 * callers that cannot allocate device memory: code running where a device
 * allocation is not allowed or not possible (inside a memory-pool or
 * arena-managed runtime that forbids other allocations, under a strict device
 * memory budget, or in a host callback path that must not call cudaMalloc).
 * The paper has no counterpart; this is a convenience of this library.
 *
 * The staging area is a fixed device array of LMKV_NOALLOC_STAGING_BYTES
 * (64 MiB) inside the library: every GPU that loads the library holds it until
 * the process exits.  Every call looks up that array's device address on the
 * device that is current at the time (cudaGetSymbolAddress; the first lookup
 * on a device loads the library's device code there, a one-time set-up per
 * device, so make that first call before any stream capture).  Because the
 * address is not cached, calls made after a cudaDeviceReset use the array of
 * the new context.  All other arguments, the layout of the host chunks and
 * the per-layer behaviour are those of lmkv_store_layers_staged.  The call
 * allocates and frees nothing.
 *
 * Every call on a device uses the same staging area, and it keeps whatever
 * the last call left there; nothing in it needs to start at zero (each layer's
 * rows are written by the gather before the copies read them).  Calls whose
 * work overlaps on the GPU (on different streams, or on different host
 * threads without ordering) race on the staging area: order them on one
 * stream or with events.
 *
 * Errors: LMKV_ERR_SCRATCH_LIMIT if 2 * row_bytes * (tokens enumerated in the
 * batch) exceeds LMKV_NOALLOC_STAGING_BYTES (nothing is enqueued: split the
 * batch); LMKV_ERR_CUDA if the set-up fails; otherwise as
 * lmkv_store_layers_staged. */
int lmkv_store_layers_staged_noalloc(const lmkv_pool_t* pool, const int32_t* block_table,
                                     int32_t max_blocks, const int64_t* start, const int64_t* end,
                                     int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                                     void* const* host_chunks, int32_t layer_lo, int32_t layer_n,
                                     void* const* layer_ready, void* const* layer_done,
                                     int32_t* d_status, void* stream);

/* Quantising store (bf16 pool only, elem_bytes == 2).  For every tile
 * (chunk g, kv, layer l):
 *   amax  = max |x| over the tile's n_g x HD values
 *   scale = amax / 448.0f                      (IEEE fp32 division)
 *   code  = e4m3fn_round_nearest_even_saturating(x / scale)   (IEEE fp32 division)
 *   amax == 0 gives scale 0 and all codes 0.
 * scales[(g*2 + kv)*L + l] = scale.  The LMCache fp8 serde casts every element
 * to float8_e4m3fn at one byte per element ("LMCache 分布式 KV Cache 序列化框架：
 * Serde 双层接口设计与自定义扩展实战", section 7.1);
 * this variant adds the per-tile scale and fuses the cast into the gather.
 *   code_ptrs : DEVICE array [num_chunks] of DEVICE pointers, chunk g's
 *               codes [2][L][n_g][HD] uint8, 16-byte aligned
 *   scales    : DEVICE float32 [num_chunks][2][L]
 * Rows with a bad block id are skipped (not part of amax, codes not written).
 * Non-finite values follow the same formulas in IEEE arithmetic: a NaN takes
 * no part in amax and its code is 0x7F (the canonical e4m3fn NaN); an
 * infinity makes amax and the scale infinite, so the tile's finite values
 * code as +-0 (0x00 / 0x80) and its infinities (inf / inf = NaN) as 0x7F.
 * UNSUPPORTED if elem_bytes != 2 or HD is not a multiple of 16. */
int lmkv_gather_chunks_fp8e4m3(const lmkv_pool_t* pool, const int32_t* block_table,
                               int32_t max_blocks, const int64_t* start, const int64_t* end,
                               int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                               void* const* code_ptrs, float* scales, int32_t* d_status,
                               void* stream);

/* Dequantising retrieve: P[...] = bf16_round_nearest_even(float(e4m3(code)) * scale),
 * one fp32 multiply per element, into the enumerated tokens' rows.  A NaN
 * result (a NaN code, or 0 * an infinite scale) is stored as a bf16 NaN; which
 * NaN bit pattern is not specified. */
int lmkv_scatter_chunks_fp8e4m3(const lmkv_pool_t* pool, const int32_t* block_table,
                                int32_t max_blocks, const int64_t* start, const int64_t* end,
                                int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                                void* const* code_ptrs, const float* scales, int32_t* d_status,
                                void* stream);

/* ---- CacheGen KV codec ------------------------------------------------
 * "LMCache 中的 KV Cache 压缩：CacheGen 编解码原理、配置方式与源码解析",
 * sections 1-5.  A chunk buffer [2][L][n][H] of bf16 (H = num_kv_heads *
 * head_dim channels, the layout of lmkv_gather_chunks) is quantised per
 * (K/V, layer) with that slice's bin count, the symbols of every
 * (K/V, layer, channel) get a CDF over the chunk's n tokens, and every
 * channel's symbols are arithmetic-coded in batches of at most 256 tokens:
 *
 *   MAX     = bins/2 - 1,  nsym = 2*MAX + 1 symbols, Lp = nsym + 1
 *   max1[t] = max over the row's H channels of |x|           (section 2)
 *   q       = clamp(round(x * (MAX / max1) + MAX), 0, 2*MAX)  each step one
 *             IEEE fp32 operation, ties to even; max1 == 0 gives q = MAX
 *   C[k]    = round(cum[k] * (2^16 - (Lp - 1)) / n) + k, k = 0..nsym, cum[k]
 *             the tokens whose symbol is below k, the division exact, ties
 *             to even (section 3); C[0] = 0, C[nsym] = 2^16
 *   coder   = Witten-Neal-Cleary arithmetic coding ("Arithmetic coding for
 *             data compression", CACM 30(6), 1987), 32-bit low/high,
 *             frequencies out of 2^16, bits most significant first, the
 *             last byte zero-padded (section 4)
 *   decode  = y = bf16(((q - MAX) / MAX) * max1), two fp32 operations
 *             (section 5)
 * Inputs must be finite.  bins are 4..32 per (K/V, layer):
 * bins[kv * L + l]; lmkv_cachegen_default_bins gives the page's rule.
 *
 * Encoded chunk ("blob", one per chunk; integers little-endian):
 *   max1     float32 [2][L][n]                       at max1_offset (0)
 *   cdf      uint16: for each (kv, l) in order, [H][nsym(kv,l) - 1] holding
 *            C[1..nsym-1]                            at cdf_offset
 *   lengths  uint32 [nb][2][L][H], nb = ceil(n/256)  at lengths_offset
 *   bytes    the streams back to back in (batch, kv, l, channel) order,
 *            each channel's symbols for the batch's tokens; a stream starts
 *            at the prefix sum of the lengths before it    at bytes_offset
 * size = bytes_offset + sum(lengths) <= max_bytes.
 */
#define LMKV_CACHEGEN_BATCH 256
#define LMKV_CACHEGEN_MAX_CHANNELS 2048
#define LMKV_CACHEGEN_MAX_TOKENS 4096
#define LMKV_CACHEGEN_MAX_LAYERS 128

typedef struct lmkv_cachegen_layout {
    uint64_t max1_offset;
    uint64_t cdf_offset;
    uint64_t lengths_offset;
    uint64_t bytes_offset;
    uint64_t max_bytes;   /* bound on the size: a stream of nt symbols takes at
                             most ceil((18 * nt + 2) / 8) bytes */
} lmkv_cachegen_layout_t;

/* The page's bins (section 1): K 32 bins for layers 0-9 and 16 after, V 32
 * bins for layers 0-1 and 16 after; fewer than 10 layers: 32 everywhere.
 * bins: HOST int32 [2 * num_layers].  INVALID_ARG for num_layers outside
 * 1..LMKV_CACHEGEN_MAX_LAYERS or a null pointer.  Host only. */
int lmkv_cachegen_default_bins(int32_t num_layers, int32_t* bins);

/* Offsets of one chunk's blob.  INVALID_ARG unless 1 <= num_layers <=
 * LMKV_CACHEGEN_MAX_LAYERS, 1 <= num_tokens <= LMKV_CACHEGEN_MAX_TOKENS,
 * 4 <= channels <= LMKV_CACHEGEN_MAX_CHANNELS with channels % 4 == 0, every
 * bins entry in 4..32, and max_bytes below 4 GiB - 256 (the kernels address
 * a blob with 32-bit offsets).  Host only. */
int lmkv_cachegen_layout(int32_t num_layers, int32_t num_tokens, int32_t channels,
                         const int32_t* bins, lmkv_cachegen_layout_t* out);

/* Device workspace the two calls below need for these chunks (HOST
 * num_tokens[num_chunks]); the same size serves encode and decode. */
int lmkv_cachegen_workspace_bytes(int32_t num_layers, int32_t channels, const int32_t* num_tokens,
                                  int32_t num_chunks, uint64_t* bytes);

/* Encode chunk g (DEVICE chunk_ptrs[g] -> [2][L][n_g][H] bf16, 16-byte
 * aligned) into DEVICE blob_ptrs[g] (4-byte aligned, at least max_bytes of its layout) and
 * store its size into DEVICE sizes[g] (uint64).  num_tokens and bins are
 * HOST arrays; workspace is DEVICE memory of lmkv_cachegen_workspace_bytes
 * bytes (16-byte aligned, contents irrelevant, not shared with calls in
 * flight).  Enqueues three kernels per group of up to 64 chunks on `stream`:
 * quantise + CDF per (chunk, kv, l), code per (chunk, batch, kv, l),
 * compact the streams.  Host errors as lmkv_cachegen_layout, plus
 * INVALID_ARG for null arrays or a workspace that is too small; device
 * errors (a null chunk pointer: BAD_POINTER) go to *d_status. */
int lmkv_cachegen_encode(void* const* chunk_ptrs, const int32_t* num_tokens, int32_t num_chunks,
                         int32_t num_layers, int32_t channels, const int32_t* bins,
                         void* const* blob_ptrs, uint64_t* sizes, void* workspace,
                         uint64_t workspace_bytes, int32_t* d_status, void* stream);

/* Decode blob g (DEVICE blob_ptrs[g], 4-byte aligned, DEVICE sizes[g] bytes) into DEVICE
 * chunk_ptrs[g] ([2][L][n_g][H] bf16, 16-byte aligned).  Streams are found
 * through the prefix sums of the lengths (section 5).  A blob whose lengths
 * do not add up to its size, or a stream that would run past it, is not
 * decoded (its rows keep their contents) and sets *d_status to BAD_DATA.
 * Two kernels per group of up to 64 chunks: region totals, then decode +
 * dequantise per (chunk, batch, kv, l). */
int lmkv_cachegen_decode(void* const* blob_ptrs, const uint64_t* sizes, const int32_t* num_tokens,
                         int32_t num_chunks, int32_t num_layers, int32_t channels,
                         const int32_t* bins, void* const* chunk_ptrs, void* workspace,
                         uint64_t workspace_bytes, int32_t* d_status, void* stream);

/* Store with CacheGen: the chunks of a store call (enumerated and validated
 * exactly as lmkv_gather_chunks does; same pool, block_table, max_blocks,
 * start, end, num_req, chunk_size, save_unfull_chunk) are encoded straight
 * from the pool's pages into DEVICE blob_ptrs[g] / sizes[g], without a chunk
 * buffer in between: the quantise pass reads each token row from its page.
 * The result equals lmkv_gather_chunks followed by lmkv_cachegen_encode.
 * bf16 pools only (UNSUPPORTED otherwise); H = num_kv_heads * head_dim and
 * chunk_size within the codec's limits; the workspace as
 * lmkv_cachegen_workspace_bytes for the chunks' token counts.  A row in a
 * block with an id outside [0, num_blocks) is coded as zeros and sets
 * *d_status to BAD_BLOCK. */
int lmkv_cachegen_store_chunks(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                               const int64_t* start, const int64_t* end, int32_t num_req,
                               int32_t chunk_size, int32_t save_unfull_chunk, const int32_t* bins,
                               void* const* blob_ptrs, uint64_t* sizes, void* workspace,
                               uint64_t workspace_bytes, int32_t* d_status, void* stream);

/* Retrieve with CacheGen: decode blob g straight into the pages of chunk g
 * of the call (the inverse of lmkv_cachegen_store_chunks; equal to
 * lmkv_cachegen_decode followed by lmkv_scatter_chunks).  Rows in a block with
 * a bad id are not written and set BAD_BLOCK; an inconsistent blob is not
 * decoded and sets BAD_DATA. */
int lmkv_cachegen_retrieve_chunks(const lmkv_pool_t* pool, const int32_t* block_table,
                                  int32_t max_blocks, const int64_t* start, const int64_t* end,
                                  int32_t num_req, int32_t chunk_size, int32_t save_unfull_chunk,
                                  const int32_t* bins, void* const* blob_ptrs, const uint64_t* sizes,
                                  void* workspace, uint64_t workspace_bytes, int32_t* d_status,
                                  void* stream);

/* Human-readable name of a status code (static storage). */
const char* lmkv_status_string(int status);

/* LMKV_ABI_VERSION of the loaded library. */
int lmkv_abi_version(void);

/* Number of kernel launches the library has enqueued since load (all entry
 * points, all streams); a host-side counter for accounting, not a sync. */
int64_t lmkv_launch_count(void);

/* The cudaError_t (as int) of the most recent CUDA runtime call that made an
 * entry point return LMKV_ERR_CUDA, 0 if none; a launch can report an error
 * left by an earlier asynchronous fault.  lmkv_cuda_error_name gives its name
 * (static storage). */
int lmkv_last_cuda_error(void);
const char* lmkv_cuda_error_name(int err);

#ifdef __cplusplus
}
#endif

#endif /* LMKV_H */
