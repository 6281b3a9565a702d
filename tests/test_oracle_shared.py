"""Pins of the oracle's shared-expert scale pages (S4b).

The page row of a token is checked against properties that the layout fixes
without restating its formula: each 128-row page holds its four 32-token
quarters interleaved row by row (so reading a page's rows in order visits
tokens 0, 32, 64, 96, 1, 33, ...), blocks of ``shared_block_m`` tokens start
at multiples of the block size rounded up to 128 rows, every token gets its
own row, and the bytes are the UE8M0 exponents of the token-order staging.
"""
import numpy as np
import pytest


def _page_order(n):
    """Tokens of one 128-row page in row order, built by interleaving quarters."""
    quarters = [list(range(q * 32, q * 32 + 32)) for q in range(4)]
    order = [quarters[q][i] for i in range(32) for q in range(4)]
    return [t for t in order if t < n]


@pytest.mark.parametrize("block_m", [128, 256, 512])
def test_rows_are_the_interleaved_quarters(orc, block_m):
    T = 3 * block_m
    rows = np.array([orc.shared_sf_row(t, block_m) for t in range(T)])
    # a bijection onto [0, T) when the block is a whole number of pages
    assert sorted(rows.tolist()) == list(range(T))
    inv = np.empty(T, np.int64)
    inv[rows] = np.arange(T)
    for page in range(T // 128):
        assert (inv[page * 128:(page + 1) * 128] - page * 128).tolist() == _page_order(128)


@pytest.mark.parametrize("block_m", [1, 7, 64, 100, 200, 300])
def test_partial_pages_are_padded(orc, block_m):
    padded = (block_m + 127) // 128 * 128
    T = 2 * block_m + 3
    rows = np.array([orc.shared_sf_row(t, block_m) for t in range(T)])
    assert len(set(rows.tolist())) == T
    for t in range(T):
        b, m = divmod(t, block_m)
        assert b * padded <= rows[t] < (b + 1) * padded
        # inside the block the token keeps its page and quarter structure
        r = rows[t] - b * padded
        assert r // 128 == m // 128
        assert (r % 128) % 4 == (m % 128) // 32 and (r % 128) // 4 == m % 32


def test_bytes_are_the_staging_exponents(orc):
    rng = np.random.default_rng(5)
    T, K = 300, 7 * 128  # G = 7: the last word has three bytes in use
    hidden = (rng.standard_normal((T, K)) * np.exp(rng.uniform(-20, 20, (T, 1)))).astype(np.float32)
    bits = (hidden.view(np.uint32) >> 16).astype(np.uint16)
    st = orc.prepare_inputs(bits, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32))
    words = st["x_sf"]
    out = orc.shared_sf(words, K, 200, rows=600, fill=0xAB)
    G = K // 128
    written = np.zeros(600, bool)
    for t in range(T):
        r = orc.shared_sf_row(t, 200)
        written[r] = True
        unpacked = [(int(words[t, g // 4]) >> (8 * (g % 4))) & 0xFF for g in range(G)]
        assert out[r].tolist() == unpacked
    # rows no token maps to keep the caller's contents
    assert np.all(out[~written] == 0xAB)
    # exponents of N(0,1)-scaled data are never the unused code 0 or 255
    assert out[written].min() >= 1 and out[written].max() <= 254
