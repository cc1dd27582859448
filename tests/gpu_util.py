"""Helpers shared by the GPU parity tests: device pools, host copies for the
oracle, and compact sub-batches for sampling full-size workloads."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_lmkv_gb300 as pkg
from paged_kv_cache_lmkv_gb300 import workloads as wl

DEV = torch.device("cuda:0")


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pkg.lmkv.load()


def host_bytes(t: torch.Tensor) -> np.ndarray:
    """Host copy of a tensor as raw bytes, last dim in bytes."""
    a = t.detach().contiguous().cpu()
    shape = list(a.shape)
    shape[-1] *= a.element_size()
    return a.view(torch.uint8).numpy().reshape(shape)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def alloc_chunks(chunks, w, dtype=torch.bfloat16, fill=None, row_elems=None):
    row = w.row_elems if row_elems is None else row_elems
    bufs = []
    for _, _, n in chunks:
        t = torch.empty((2, w.num_layers, n, row), dtype=dtype, device=DEV)
        if fill is not None:
            t.view(torch.uint8).fill_(fill)
        bufs.append(t)
    return bufs, pkg.pointer_array(bufs, DEV)


def device_pool(w, seed, fill="normal"):
    return pkg.Pool(wl.make_pool(w, DEV, seed, fill), w.num_kv_heads, w.head_dim)


def new_status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def compact_subbatch(pool_layers, table, chunks, sample):
    """Host pool holding only the blocks of the sampled chunks, plus a
    one-request-per-chunk table addressing it.  Returns (HostPool, table,
    starts, ends, block ids per sampled chunk)."""
    B = pool_layers[0].shape[2]
    ids_per = []
    for g in sample:
        r, t0, n = chunks[g]
        c0 = t0 // B
        ids_per.append([int(x) for x in table[r, c0:c0 + math.ceil(n / B)]])
    flat = [i for ids in ids_per for i in ids]
    idx = torch.as_tensor(flat, dtype=torch.long, device=pool_layers[0].device)
    host = [host_bytes(t.index_select(1, idx)) for t in pool_layers]
    maxb = max(len(x) for x in ids_per)
    tab = np.full((len(sample), maxb), -1, np.int32)
    k = 0
    for i, ids in enumerate(ids_per):
        tab[i, :len(ids)] = np.arange(k, k + len(ids))
        k += len(ids)
    starts = np.zeros(len(sample), np.int64)
    ends = np.array([chunks[g][2] for g in sample], np.int64)
    return oracle.HostPool(host, B), tab, starts, ends, ids_per


def oracle_chunks_for(pool_layers, table, chunks, sample, chunk_size, L, row_bytes):
    """The oracle's gather of the sampled chunks (byte arrays [2][L][n][row_bytes])."""
    hp, tab, s, e, _ = compact_subbatch(pool_layers, table, chunks, sample)
    out = [np.zeros((2, L, chunks[g][2], row_bytes), np.uint8) for g in sample]
    assert oracle.gather(hp, tab, s, e, chunk_size, True, out) == 0
    return out


def nonsentinel_rows(layers) -> int:
    """Rows of a pool (all layers, K and V) that differ from the sentinel pattern."""
    total = 0
    for t in layers:
        b = t.view(torch.uint8)
        total += int((b != wl.SENTINEL_BYTE).any(dim=-1).sum().item())
    return total
