"""Per-token dictionary model of the chunk gather / scatter, for tiny pools.

An independent, deliberately naive restatement used to pin the C oracle:
the pool is a dict keyed by (layer, kv, block, slot), each request's token
list is sliced into runs of chunk_size tokens (the LMCache store loop cuts
tokens into chunk_size chunks and drops a short tail unless
save_unfull_chunk is set; cache_engine.py walk-through, "store()" section),
and every chunk is a dict keyed by (kv, layer, token-in-chunk).
"""
from __future__ import annotations

import numpy as np


def chunk_token_lists(starts, ends, chunk_size, save_unfull):
    """[(request, [token, ...])] in request order, or None if a start is unaligned."""
    out = []
    for r, (s, e) in enumerate(zip(starts, ends)):
        s, e = int(s), int(e)
        if s % chunk_size or s < 0 or e < s:
            return None
        toks = list(range(s, e))
        pieces = [toks[i:i + chunk_size] for i in range(0, len(toks), chunk_size)]
        if pieces and len(pieces[-1]) < chunk_size and not save_unfull:
            pieces = pieces[:-1]
        out.extend((r, p) for p in pieces)
    return out


def pool_to_dict(layers):
    d = {}
    for l, a in enumerate(layers):
        for kv in range(2):
            for blk in range(a.shape[1]):
                for slot in range(a.shape[2]):
                    d[(l, kv, blk, slot)] = a[kv, blk, slot].copy()
    return d


def dict_to_pool(d, layers):
    for (l, kv, blk, slot), row in d.items():
        layers[l][kv, blk, slot] = row


def gather(layers, table, starts, ends, chunk_size, save_unfull, chunks, layer=None):
    """Fill ``chunks`` (list of [2][L][n][row] arrays) in place; returns #bad rows."""
    pool = pool_to_dict(layers)
    B = layers[0].shape[2]
    nb = layers[0].shape[1]
    bad = 0
    for g, (r, toks) in enumerate(chunk_token_lists(starts, ends, chunk_size, save_unfull)):
        for kv in range(2):
            for l in range(len(layers)):
                if layer is not None and l != layer:
                    continue
                for t, tok in enumerate(toks):
                    blk = int(table[r][tok // B])
                    if not 0 <= blk < nb:
                        bad += 1
                        continue
                    chunks[g][kv, l, t] = pool[(l, kv, blk, tok % B)]
    return bad


def scatter(layers, table, starts, ends, chunk_size, save_unfull, chunks, layer=None):
    """Write ``chunks`` back into ``layers`` in place; returns #bad rows."""
    pool = pool_to_dict(layers)
    B = layers[0].shape[2]
    nb = layers[0].shape[1]
    bad = 0
    for g, (r, toks) in enumerate(chunk_token_lists(starts, ends, chunk_size, save_unfull)):
        for kv in range(2):
            for l in range(len(layers)):
                if layer is not None and l != layer:
                    continue
                for t, tok in enumerate(toks):
                    blk = int(table[r][tok // B])
                    if not 0 <= blk < nb:
                        bad += 1
                        continue
                    pool[(l, kv, blk, tok % B)] = np.array(chunks[g][kv, l, t])
    dict_to_pool(pool, layers)
    return bad
