"""Pins for the mask tile summary (``oracle.mask_tiles``): hand-built masks
whose classes and bits follow from the definition by inspection, the tail
rule (keys and rows past L count as removed, but do not decide the class)
and agreement with a vectorised numpy formulation that shares none of its
code."""
import numpy as np

import oracle


def test_classes_of_structured_masks():
    L = 256
    none = np.zeros((L, L), dtype=np.uint8)
    bits, cls = oracle.mask_tiles(none)
    assert cls.shape == (2, 2) and np.all(cls == 0) and np.all(bits == 0)
    causal_removed = np.triu(np.ones((L, L), dtype=np.uint8), k=1)   # key > query removed
    bits, cls = oracle.mask_tiles(causal_removed)
    np.testing.assert_array_equal(cls, [[1, 2], [0, 1]])
    # diagonal tile: row r removes keys r+1..127 -> word w holds bits above r
    for r in (0, 31, 32, 100, 127):
        want = [sum(1 << c for c in range(32) if 32 * w + c > r) for w in range(4)]
        np.testing.assert_array_equal(bits[0, 0, r], want)
    assert np.all(bits[0, 1] == 0xFFFFFFFF) and np.all(bits[1, 0] == 0)


def test_single_entry_and_full_tile():
    L = 256
    m = np.zeros((L, L), dtype=np.uint8)
    m[130, 5] = 1                      # tile (1, 0), row 2, key 5
    m[0:128, 128:256] = 1              # tile (0, 1) entirely removed
    bits, cls = oracle.mask_tiles(m)
    np.testing.assert_array_equal(cls, [[0, 2], [1, 0]])
    assert bits[1, 0, 2, 0] == 1 << 5 and np.count_nonzero(bits[1, 0]) == 1


def test_tail_tiles():
    # L = 130: tile 1 holds rows/keys 128, 129 only; the rest reads as removed
    L = 130
    m = np.zeros((L, L), dtype=np.uint8)
    bits, cls = oracle.mask_tiles(m)
    np.testing.assert_array_equal(cls, [[0, 0], [0, 0]])   # nothing inside is removed
    np.testing.assert_array_equal(bits[0, 1, 0], [0xFFFFFFFC, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF])
    assert np.all(bits[1, 0, 2:] == 0xFFFFFFFF) and np.all(bits[1, 0, :2] == 0)
    m[128:, :] = 1                      # the two tail rows remove every key
    bits, cls = oracle.mask_tiles(m)
    np.testing.assert_array_equal(cls, [[0, 0], [2, 2]])


def test_matches_vectorised_form():
    rng = np.random.default_rng(17)
    for L in (100, 128, 300):
        m = (rng.random((L, L)) < 0.4).astype(np.uint8)
        m[: min(L, 128), : min(L, 128)] = 0          # one tile with nothing removed
        if L > 128:
            m[128:256, :128] = 1                      # one with everything removed
        bits, cls = oracle.mask_tiles(m)
        n = (L + 127) // 128
        pad = np.ones((n * 128, n * 128), dtype=bool)
        pad[:L, :L] = m != 0
        inside = np.zeros_like(pad)
        inside[:L, :L] = True
        t = pad.reshape(n, 128, n, 128).transpose(0, 2, 1, 3)
        ins = inside.reshape(n, 128, n, 128).transpose(0, 2, 1, 3)
        weights = (1 << np.arange(32, dtype=np.uint64))
        want_bits = (t.reshape(n, n, 128, 4, 32) * weights).sum(-1).astype(np.uint32)
        np.testing.assert_array_equal(bits, want_bits)
        any_removed = (t & ins).any(axis=(2, 3))
        any_kept = (~t & ins).any(axis=(2, 3))
        want_cls = np.where(~any_removed, 0, np.where(~any_kept, 2, 1))
        np.testing.assert_array_equal(cls, want_cls)
