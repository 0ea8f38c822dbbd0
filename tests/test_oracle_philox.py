"""Pins for the oracle's Philox4x32-10 (Salmon et al., "Parallel Random Numbers:
As Easy as 1, 2, 3", SC'11).

The known-answer vectors are the published ones for philox4x32 with 10
rounds (the authors' Random123 distribution, kat_vectors); they fix the round
function, the multipliers, the Weyl key schedule and the round count at once.
"""
import numpy as np
import pytest

import oracle

# counter (4 words), key (2 words) -> output (4 words)
KAT = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF), (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", KAT)
def test_known_answer(ctr, key, want):
    got = oracle.philox4x32_10(np.array([ctr], dtype=np.uint32), np.array(key, dtype=np.uint32))
    assert tuple(int(x) for x in got[0]) == want


def test_uniform_is_top24_of_word0():
    seed = 0x0123456789ABCDEF
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint32)
    for (j, b, s, off) in [(0, 0, 0, 0), (15, 3, 1, 7), (7, 100, 0, 2**32 - 1)]:
        w = oracle.philox4x32_10(np.array([[j, b, s, off]], dtype=np.uint32), key)[0, 0]
        u = oracle.uniform(seed, j, b, s, off)
        assert u == (int(w) >> 8) / 2.0**24
        assert 0.0 <= u < 1.0


def test_uniformity_chi_square():
    scipy_stats = pytest.importorskip("scipy.stats")
    n = 200_000
    ctr = np.zeros((n, 4), dtype=np.uint32)
    ctr[:, 0] = np.arange(n) % 16
    ctr[:, 1] = np.arange(n) // 16
    out = oracle.philox4x32_10(ctr, np.array([1234, 0], dtype=np.uint32))
    u = (out[:, 0] >> 8).astype(np.float64) / 2.0**24
    counts, _ = np.histogram(u, bins=64, range=(0.0, 1.0))
    _, pval = scipy_stats.chisquare(counts)
    assert pval > 1e-4
    # all four words look uniform too (byte histogram)
    by = out.view(np.uint8).reshape(-1)
    counts, _ = np.histogram(by, bins=256, range=(0, 256))
    _, pval = scipy_stats.chisquare(counts)
    assert pval > 1e-4
