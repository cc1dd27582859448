"""Pins for the oracle's chunk enumeration (CPU only).

Rule: cache_engine.py walk-through ("LMCache 源码解析"), section "store()":
chunk_size-token chunks, short tail kept only with save_unfull_chunk, the
cached prefix must be a multiple of chunk_size.
"""
import os

import numpy as np
import pytest

import brute
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "chunking.txt")


def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            C, s, e, flag = (int(x) for x in lhs.split())
            rhs = rhs.split()
            cases.append((C, s, e, flag, rhs))
    return cases


@pytest.mark.parametrize("C,s,e,flag,rhs", _golden_cases())
def test_golden_chunking(C, s, e, flag, rhs):
    chunks = oracle.enumerate_chunks([s], [e], C, bool(flag))
    if rhs[0] == "invalid":
        assert chunks is None
        return
    assert len(chunks) == int(rhs[0])
    if rhs[1] != "-":
        assert chunks[-1][2] == int(rhs[1])


def test_70b_batch_counts():
    ends = [4096, 9000, 20000, 32768]
    with_tail = oracle.enumerate_chunks([0] * 4, ends, 256, True)
    no_tail = oracle.enumerate_chunks([0] * 4, ends, 256, False)
    assert len(with_tail) == 16 + 36 + 79 + 128 == 259
    assert len(no_tail) == 16 + 35 + 78 + 128 == 257
    assert sum(n for _, _, n in with_tail) == sum(ends)
    # request-major order, chunk starts aligned to the chunk size
    assert [r for r, _, _ in with_tail] == sorted(r for r, _, _ in with_tail)
    assert all(t0 % 256 == 0 for _, t0, _ in with_tail)


def test_closed_form_random():
    rng = np.random.default_rng(7)
    for _ in range(500):
        C = int(rng.choice([1, 16, 64, 256, 768]))
        nreq = int(rng.integers(0, 6))
        starts = rng.integers(0, 5, nreq) * C
        ends = starts + rng.integers(0, 4 * C + 3, nreq)
        flag = bool(rng.integers(0, 2))
        chunks = oracle.enumerate_chunks(starts, ends, C, flag)
        expect = sum((e - s) // C + (1 if flag and (e - s) % C else 0)
                     for s, e in zip(starts, ends))
        assert len(chunks) == expect
        ref = brute.chunk_token_lists(starts, ends, C, flag)
        assert [(r, toks[0], len(toks)) for r, toks in ref] == chunks


def test_unaligned_start_rejected():
    assert oracle.enumerate_chunks([0, 17], [512, 600], 256, True) is None
    assert brute.chunk_token_lists([0, 17], [512, 600], 256, True) is None
