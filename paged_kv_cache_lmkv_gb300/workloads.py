"""Seeded synthetic inputs for the paged-KV chunk gather / scatter.

This module only draws inputs: model-shaped workload descriptions, random
block tables and random pool contents.  It holds none of the movement or
quantisation arithmetic, so both the CUDA path and the CPU oracle can take
their inputs from it.

Workload shapes follow the models the LMCache paper evaluates
("LMCache: An Efficient KV Cache Layer for Enterprise-Scale LLM Inference",
experimental setup: Llama-3.1-8B / 70B, Qwen2.5-Coder-32B), with vLLM-style
16-token pages and 256-token chunks (configurable chunk size section).  The
pages' evaluation datasets are not used: seeded N(0, 1) bf16 values of the
same tensor shapes stand in for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

# Bit pattern written into pool rows that no request references; a finite
# bf16 (about -2.9e-16), so it survives any bitwise comparison unchanged.
SENTINEL_BF16 = 0xA5A5
SENTINEL_BYTE = 0xA5


@dataclass(frozen=True)
class Workload:
    name: str
    num_layers: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int                 # per layer
    req_tokens: tuple               # end offset of each request
    req_start: tuple = ()           # start offset of each request (default 0)
    chunk_size: int = 256
    save_unfull: bool = True
    outliers: bool = False          # 1% of channels x20 per (K/V, layer)
    elem_bytes: int = 2             # bf16
    notes: str = field(default="", compare=False)

    @property
    def row_elems(self) -> int:
        return self.num_kv_heads * self.head_dim

    @property
    def row_bytes(self) -> int:
        return self.row_elems * self.elem_bytes

    @property
    def starts(self) -> np.ndarray:
        if self.req_start:
            return np.asarray(self.req_start, np.int64)
        return np.zeros(len(self.req_tokens), np.int64)

    @property
    def ends(self) -> np.ndarray:
        return np.asarray(self.req_tokens, np.int64)

    @property
    def blocks_per_req(self) -> list:
        return [math.ceil(int(e) / self.block_size) for e in self.ends]

    @property
    def max_blocks(self) -> int:
        return max(self.blocks_per_req) if self.req_tokens else 1

    @property
    def pool_layer_bytes(self) -> int:
        return 2 * self.num_blocks * self.block_size * self.row_bytes

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload("tiny", 2, 2, 64, 16, 64, (512,),
                notes="2 layers, 2 KV heads, head_dim 64, one 512-token request")
LLAMA8B = Workload("llama3.1-8b", 32, 8, 128, 16, 8192, (10240,),
                   notes="10240-token request, 40 chunks of 256, 16 GiB pool")
LLAMA70B = Workload("llama3.1-70b", 80, 8, 128, 16, 32768, (4096, 9000, 20000, 32768),
                    notes="4-request batch with partial last chunks, 160 GiB pool")
QWEN32B = Workload("qwen2.5-32b", 64, 8, 128, 16, 4096, (16384,), outliers=True,
                   notes="fp8 workload; block_size swept over 16/32/64, 65536 tokens per layer")

WORKLOADS = {w.name: w for w in (TINY, LLAMA8B, LLAMA70B, QWEN32B)}


def qwen_with_block_size(block_size: int) -> Workload:
    """Qwen2.5-32B shape at another page size, keeping 65536 token slots per layer."""
    return QWEN32B.with_(block_size=block_size, num_blocks=65536 // block_size)


def block_table(w: Workload, seed: int, exclude=None, tiny_subset: int | None = None) -> np.ndarray:
    """int32 [num_req][max_blocks] block table with all ids distinct.

    Ids are drawn without replacement from the pool (minus ``exclude``).  With
    several requests the drawn ids are dealt out in a shuffled request order,
    so consecutive pool blocks belong to different requests (interleaved
    tables).  ``tiny_subset`` draws the ids from the first ``tiny_subset``
    pool blocks only.  Unused trailing columns hold -1.
    """
    rng = np.random.default_rng(seed)
    need = w.blocks_per_req
    total = int(sum(need))
    candidates = np.arange(w.num_blocks if tiny_subset is None else tiny_subset, dtype=np.int64)
    if exclude is not None:
        candidates = np.setdiff1d(candidates, np.asarray(sorted(exclude), np.int64))
    if total > len(candidates):
        raise ValueError("pool too small for the block table")
    ids = rng.permutation(candidates)[:total]
    labels = np.repeat(np.arange(len(need)), need)
    labels = labels[rng.permutation(total)]
    table = np.full((len(need), max(w.max_blocks, 1)), -1, np.int32)
    fill = [0] * len(need)
    # ids in ascending pool order, handed to the request named by the shuffled label
    for blk, r in zip(np.sort(ids), labels):
        table[r, fill[r]] = blk
        fill[r] += 1
    # shuffle within each request so the per-request order is random too
    for r in range(len(need)):
        table[r, :need[r]] = rng.permutation(table[r, :need[r]])
    return table


def generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def fill_normal_(t: torch.Tensor, seed: int) -> torch.Tensor:
    """Fill a bf16 tensor in place with N(0, 1) values from a seeded generator."""
    g = generator(t.device, seed)
    if t.dtype == torch.bfloat16:
        # draw in slabs to bound the float32 temporary on large pools
        flat = t.view(-1)
        step = 1 << 28
        for i in range(0, flat.numel(), step):
            n = min(step, flat.numel() - i)
            flat[i:i + n].copy_(torch.randn(n, generator=g, device=t.device, dtype=torch.float32))
    else:
        t.normal_(generator=g)
    return t


def fill_sentinel_(t: torch.Tensor) -> torch.Tensor:
    if t.dtype == torch.bfloat16:
        t.view(torch.int16).fill_(np.int16(np.uint16(SENTINEL_BF16).view(np.int16)).item())
    else:
        t.view(torch.uint8).fill_(SENTINEL_BYTE)
    return t


def outlier_channels(w: Workload, seed: int) -> np.ndarray:
    """[2][num_layers][n_out] channel indices (1% of the row, at least one) that get x20."""
    rng = np.random.default_rng(seed)
    n_out = max(1, round(0.01 * w.row_elems))
    out = np.empty((2, w.num_layers, n_out), np.int64)
    for kv in range(2):
        for l in range(w.num_layers):
            out[kv, l] = rng.choice(w.row_elems, n_out, replace=False)
    return out


def apply_outliers_(layer: torch.Tensor, kv: int, channels: np.ndarray, factor: float = 20.0):
    """Scale the given channels of one pool layer's K (kv=0) or V (kv=1) half by ``factor``."""
    idx = torch.as_tensor(channels, device=layer.device)
    half = layer[kv]                       # [num_blocks][block_size][row]
    half[..., idx] = (half[..., idx].float() * factor).to(layer.dtype)


def make_pool(w: Workload, device, seed: int | None, fill: str = "normal") -> list:
    """Per-layer pool tensors [2][num_blocks][block_size][row] (bf16 for elem_bytes 2)."""
    dtype = {1: torch.uint8, 2: torch.bfloat16, 4: torch.float32}[w.elem_bytes]
    layers = []
    for l in range(w.num_layers):
        t = torch.empty((2, w.num_blocks, w.block_size, w.row_elems), dtype=dtype, device=device)
        if fill == "normal":
            if dtype == torch.uint8:
                g = generator(device, seed * 1000003 + l)
                t.copy_(torch.randint(0, 256, t.shape, generator=g, device=device, dtype=torch.uint8))
            else:
                fill_normal_(t, seed * 1000003 + l)
        elif fill == "sentinel":
            fill_sentinel_(t)
        elif fill != "empty":
            raise ValueError(fill)
        layers.append(t)
    if fill == "normal" and w.outliers:
        ch = outlier_channels(w, 3 if seed is None else seed + 3)
        for l, t in enumerate(layers):
            for kv in range(2):
                apply_outliers_(t, kv, ch[kv, l])
    return layers


# CacheGen codec inputs: the page's benchmark ("LMCache 中的 KV Cache 压缩：CacheGen
# 编解码原理、配置方式与源码解析", section on verifying the compression) builds
# synthetic bf16 KV of 32 layers x 8 KV heads x head_size 128 and sweeps the
# chunk size over 64, 128, 256 and 768 tokens.
CACHEGEN_LAYERS = 32
CACHEGEN_CHANNELS = 8 * 128
CACHEGEN_CHUNK_SIZES = (64, 128, 256, 768)


def cachegen_chunks(num_layers: int, channels: int, ntoks, seed: int, device="cpu",
                    outliers: bool = False, zero_rows: int = 0, tiny_rows: int = 0) -> list:
    """Chunk buffers [2][L][n][H] bf16 ~ N(0, 1), one per entry of ntoks, drawn
    on the CPU from a seeded generator (so every device sees the same values),
    optionally with 1% of each (K/V, layer)'s channels scaled x20, the first
    `zero_rows` token rows of every slice set to zero and the next `tiny_rows`
    scaled by 1e-39 (bf16 subnormals, some of them zero)."""
    g = generator("cpu", seed)
    out = []
    for n in ntoks:
        x = torch.randn((2, num_layers, n, channels), generator=g, dtype=torch.float32)
        if outliers:
            k = max(1, round(0.01 * channels))
            for kv in range(2):
                for l in range(num_layers):
                    idx = torch.randperm(channels, generator=g)[:k]
                    x[kv, l, :, idx] *= 20.0
        if zero_rows:
            x[:, :, :zero_rows] = 0
        if tiny_rows:
            x[:, :, zero_rows:zero_rows + tiny_rows] *= 1e-39
        out.append(x.to(torch.bfloat16).to(device))
    return out
