"""GB300-native batched paged-KV chunk gather / scatter (LMCache's store / retrieve
data path): a C-ABI CUDA library (include/lmkv.h, csrc/) and its Python binding."""
from . import lmkv  # noqa: F401
from .lmkv import (CachegenCodec, Offload, Pool, LmkvError, check, count_chunks,  # noqa: F401
                   decode_store_ranges, enumerate_chunks,
                   gather_chunks, gather_chunks_fp8e4m3, gather_layer, pointer_array,
                   overlap_events, retrieve_layers, retrieve_layers_overlapped,
                   retrieve_layers_staged, scatter_chunks,
                   scatter_chunks_fp8e4m3, scatter_layer, staging_bytes, store_layers,
                   store_layers_overlapped, store_layers_staged)

__all__ = ["lmkv", "CachegenCodec", "Offload", "Pool", "LmkvError", "check", "count_chunks", "decode_store_ranges",
           "enumerate_chunks",
           "gather_chunks", "scatter_chunks", "gather_layer", "scatter_layer",
           "gather_chunks_fp8e4m3", "scatter_chunks_fp8e4m3", "pointer_array",
           "store_layers", "retrieve_layers", "store_layers_staged",
           "retrieve_layers_staged", "staging_bytes", "store_layers_overlapped",
           "retrieve_layers_overlapped", "overlap_events"]
