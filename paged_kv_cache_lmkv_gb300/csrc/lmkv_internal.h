// lmkv_internal.h -- declarations shared by the library's translation units
// (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "lmkv.h"

// Adds n to the counter lmkv_launch_count() reports.
void lmkv_internal_add_launches(int64_t n);

// LMKV_OK for cudaSuccess; otherwise records err for lmkv_last_cuda_error()
// and returns LMKV_ERR_CUDA.
int lmkv_internal_cuda_status(cudaError_t err);

// One chunk of a store / retrieve call: request row, first token, tokens.
struct LmkvChunkRef {
    int32_t req;
    int64_t tok0;
    int32_t n;
};

// Validates a call's pool, requests and block table exactly as
// lmkv_gather_chunks does and lists its chunks in chunk order.
int lmkv_internal_list_chunks(const lmkv_pool_t* pool, const int32_t* block_table, int32_t max_blocks,
                              const int64_t* start, const int64_t* end, int32_t num_req,
                              int32_t chunk_size, int32_t save_unfull, std::vector<LmkvChunkRef>* out);
