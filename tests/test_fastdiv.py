"""The multiply-shift division the combine kernel uses to split a flat work
index into (token, vector): checked exhaustively against integer division on
the sizes the library allows, using the same magic-number recipe as the host
code (round-up method of Granlund and Montgomery, 1994)."""
import numpy as np


def magic(d):
    l = 0
    while (1 << l) < d:
        l += 1
    m = ((((1 << l) - d) << 32) // d + 1) & 0xFFFFFFFF
    return m, l


def fastdiv(n, m, l):
    hi = (n.astype(np.uint64) * np.uint64(m)) >> np.uint64(32)
    return ((hi + n.astype(np.uint64)) >> np.uint64(l)).astype(np.int64)


def test_fastdiv_matches_integer_division():
    rng = np.random.default_rng(0)
    ds = list(range(1, 2049)) + [896, 256, 512, 4096, 6400, 7168 // 8, 12345, 65535, 1 << 20]
    n = np.concatenate([np.arange(0, 70000, dtype=np.int64),
                        rng.integers(0, 2**31, size=200000, dtype=np.int64),
                        np.array([2**31 - 1, 2**31 - 2], dtype=np.int64)])
    for d in ds:
        m, l = magic(d)
        assert np.array_equal(fastdiv(n, m, l), n // d), d
