"""Deferred decode-KV store ranges (CPU only).

LMCache paper, delayed storing of decode KV: generated tokens' KV is buffered
and stored in batch once a whole chunk exists.  Pinned against a token-by-
token simulation: a chunk is stored at the step where its last token arrives.
"""
import numpy as np
import pytest

from paged_kv_cache_lmkv_gb300 import build, lmkv


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    lmkv.load()


def test_simulated_decode_runs():
    rng = np.random.default_rng(0)
    for C in (16, 256):
        nreq = 7
        prompt = rng.integers(0, 3 * C, nreq)
        stored = (prompt // C) * C                      # prefill stored its full chunks
        cur = prompt.copy()
        tok_stored = [set(range(int(s))) for s in stored]
        for step in range(40):
            cur = cur + rng.integers(0, C // 2 + 2, nreq)
            s, e, n = lmkv.decode_store_ranges(stored, cur, C)
            # token-by-token model: chunk [k*C, (k+1)*C) is stored once token (k+1)*C - 1 exists
            expect_n = 0
            for r in range(nreq):
                k0, k1 = int(stored[r]) // C, int(cur[r]) // C
                expect_n += k1 - k0
                assert s[r] == stored[r] and e[r] == k1 * C
                tok_stored[r] |= set(range(int(s[r]), int(e[r])))
            assert n == expect_n
            stored = e
        for r in range(nreq):
            assert tok_stored[r] == set(range(int(cur[r]) // C * C))


def test_nothing_ready_and_invalid():
    s, e, n = lmkv.decode_store_ranges([256, 0], [300, 255], 256)
    assert n == 0 and list(s) == [256, 0] and list(e) == [256, 0]
    with pytest.raises(lmkv.LmkvError):
        lmkv.decode_store_ranges([100], [300], 256)     # unaligned stored prefix
    with pytest.raises(lmkv.LmkvError):
        lmkv.decode_store_ranges([512], [300], 256)     # stored past the current length
