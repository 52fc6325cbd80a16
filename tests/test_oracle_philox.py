"""CPU checks of the oracle's Philox4x32-10 dropout generator.

The bijection itself is pinned on a GPU against cuRAND's device generator
(tests/test_gpu_philox.py). Here: statistics that a plausible slip (a wrong
multiplier, a missing key bump, a dropped word) would break, the keep
fraction, and the word-layout convention of the keep-mask.
"""
import numpy as np
import pytest

from oracle.philox import drop_threshold, keep_mask, philox4x32_10


def test_threshold():
    assert drop_threshold(0.0) == 0
    assert drop_threshold(0.5) == 1 << 15
    assert drop_threshold(0.1) == 6553  # floor(0.1 * 2**16)
    assert drop_threshold(1.0 - 2.0 ** -20) == 65535
    with pytest.raises(ValueError):
        drop_threshold(1.0)


def test_words_uniform_and_independent():
    n = 1 << 16
    c = np.arange(n, dtype=np.uint64)
    w = philox4x32_10(c, 0, 0, 0, 1234, 0)
    allw = np.concatenate(w).astype(np.uint64)
    # chi-square on the top 8 bits: 256 bins, 262144 draws
    hist = np.bincount((allw >> np.uint64(24)).astype(np.int64), minlength=256)
    exp = allw.size / 256
    chi2 = ((hist - exp) ** 2 / exp).sum()
    assert chi2 < 255 + 6 * np.sqrt(2 * 255)
    # low bits too (a missing high-half xor would leave them structured)
    hist = np.bincount((allw & np.uint64(0xFF)).astype(np.int64), minlength=256)
    chi2 = ((hist - exp) ** 2 / exp).sum()
    assert chi2 < 255 + 6 * np.sqrt(2 * 255)
    # the four words are not copies or simple functions of each other
    for a in range(4):
        for b in range(a + 1, 4):
            corr = np.corrcoef(w[a].astype(np.float64), w[b].astype(np.float64))[0, 1]
            assert abs(corr) < 5 / np.sqrt(n)


def test_avalanche():
    """Flipping one counter or key bit flips about half the output bits."""
    rng = np.random.default_rng(0)
    base = [rng.integers(0, 2 ** 32, 4096, dtype=np.uint64) for _ in range(4)]
    key = (np.uint64(0x1234567), np.uint64(0x89ABCDE))
    ref = philox4x32_10(*base, *key)
    for word in range(4):
        flipped = list(base)
        flipped[word] = flipped[word] ^ np.uint64(1 << 13)
        out = philox4x32_10(*flipped, *key)
        bits = sum(np.unpackbits((a ^ b).view(np.uint8)).sum() for a, b in zip(ref, out))
        frac = bits / (4096 * 128)
        assert abs(frac - 0.5) < 0.01
    out = philox4x32_10(*base, key[0] ^ np.uint64(1), key[1])
    bits = sum(np.unpackbits((a ^ b).view(np.uint8)).sum() for a, b in zip(ref, out))
    assert abs(bits / (4096 * 128) - 0.5) < 0.01


@pytest.mark.parametrize("p", [0.1, 0.25, 0.9])
def test_keep_fraction(p):
    N = 512
    z = np.concatenate([keep_mask(b, h, 4, N, np.arange(N), 1234, 0, p) for b in range(2) for h in range(4)])
    n = z.size
    sigma = np.sqrt(n * p * (1 - p))
    assert abs(z.sum() - n * (1 - p)) < 5 * sigma


def test_mask_layout_convention():
    """Mask entry (b, h, i, j) is 16-bit half j%2 (low half for even j) of word (j%8)//2 of
    Philox at counter g = ((b*H+h)*N+i)*ceil(N/8)+j//8, kept iff >= floor(p * 2**16)."""
    B, H, N, p, seed, off = 2, 3, 37, 0.3, (7 << 32) | 99, (5 << 32) | 11
    rng = np.random.default_rng(1)
    T = drop_threshold(p)
    n8 = (N + 7) // 8
    for _ in range(300):
        b, h, i, j = (int(rng.integers(0, x)) for x in (B, H, N, N))
        g = ((b * H + h) * N + i) * n8 + j // 8
        w = philox4x32_10(g & 0xFFFFFFFF, g >> 32, off & 0xFFFFFFFF, off >> 32, seed & 0xFFFFFFFF, seed >> 32)
        value = (int(w[(j % 8) // 2]) >> (16 * (j % 2))) & 0xFFFF
        assert keep_mask(b, h, H, N, [i], seed, off, p)[0, j] == (value >= T)


def test_mask_depends_on_seed_and_offset():
    a = keep_mask(0, 0, 1, 64, np.arange(64), 1, 0, 0.5)
    assert not np.array_equal(a, keep_mask(0, 0, 1, 64, np.arange(64), 2, 0, 0.5))
    assert not np.array_equal(a, keep_mask(0, 0, 1, 64, np.arange(64), 1, 1, 0.5))
    assert keep_mask(0, 0, 1, 64, np.arange(64), 1, 0, 0.0).all()
