"""Pins for the oracle's 3-bit packing ("triton-3bit-kv-cache-kernel" README,
sections 1.A, 1.B and 2 items 1-2).  CPU only."""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "octet_layout.txt")


def _golden_rows():
    octet, word = [], []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        t = line.split()
        # "<kind> <idx> bit <k> = lane <i> bit <j>"
        rec = (int(t[1]), int(t[3]), int(t[6]), int(t[8]))
        (octet if t[0] == "byte" else word).append(rec)
    return octet, word


def test_golden_octet_bit_placement(orc):
    """Every bit of every lane lands where the page's byte diagram puts it,
    and nowhere else (walking single ones)."""
    octet, _ = _golden_rows()
    assert len(octet) == 24
    for byte, bit, lane, lbit in octet:
        v = np.zeros((1, 8), np.uint8)
        v[0, lane] = 1 << lbit
        p = orc.pack3(v)[0]
        expect = np.zeros(3, np.uint8)
        expect[byte] = 1 << bit
        assert (p == expect).all(), (byte, bit, lane, lbit, p)
        back = orc.unpack3(expect[None, :])[0]
        assert (back == v[0]).all()


def test_golden_word_straddles(orc):
    """Lanes 10 and 21 straddle 32-bit words exactly as the page lists."""
    _, word = _golden_rows()
    for w, bit, lane, lbit in word:
        W = np.zeros((1, 3), np.uint32)
        W[0, w] = np.uint32(1) << np.uint32(bit)
        vals = orc.unpack3_words(W)[0]
        expect = np.zeros(32, np.uint8)
        expect[lane] = 1 << lbit
        assert (vals == expect).all(), (w, bit, lane, lbit, vals)


def test_exhaustive_bijection_closed_form(orc):
    """All 2^24 octet states: packing the lanes of state n gives the three
    little-endian bytes of n (left inverse), and unpacking those bytes gives
    the lanes back (right inverse over every byte triple)."""
    n = np.arange(1 << 24, dtype=np.uint32)
    lanes = ((n[:, None] >> (3 * np.arange(8, dtype=np.uint32))[None, :]) & 7).astype(np.uint8)
    byts = n.view(np.uint8).reshape(-1, 4)[:, :3]          # little-endian bytes of n
    packed = orc.pack3(lanes)
    assert np.array_equal(packed, byts)
    unpacked = orc.unpack3(np.ascontiguousarray(byts))
    assert np.array_equal(unpacked, lanes)


def test_pack_masks_high_bits(orc):
    """Values above 7 contribute only their low 3 bits (the formulas mask
    with & 0x7)."""
    rng = np.random.default_rng(0)
    v = rng.integers(0, 256, size=(4096, 8), dtype=np.uint8)
    assert np.array_equal(orc.pack3(v), orc.pack3(v & 7))


@pytest.mark.parametrize("background", [0, 7])
def test_walking_isolation_bytes_and_words(orc, background):
    """Walking ones/zeros: set one of the 32 lanes of a 96-bit group to each
    of 0..7 over a background of 000 or 111; every other lane must read back
    unchanged through both the octet path and the word path, and the 12 bytes
    equal the 3 words viewed little-endian."""
    for lane in range(32):
        for val in range(8):
            v = np.full(32, background, np.uint8)
            v[lane] = val
            packed = orc.pack3(v.reshape(4, 8)).reshape(12)
            # byte path
            assert np.array_equal(orc.unpack3(packed.reshape(4, 3)).reshape(32), v)
            # word path on the same 12 bytes, little-endian words
            words = packed.view("<u4").reshape(1, 3)
            assert np.array_equal(orc.unpack3_words(words)[0], v)
            # explicit little-endian equivalence
            w_le = [int(packed[4 * i]) | int(packed[4 * i + 1]) << 8 |
                    int(packed[4 * i + 2]) << 16 | int(packed[4 * i + 3]) << 24 for i in range(3)]
            assert [int(x) for x in words[0]] == w_le


def test_word_path_matches_bitstream(orc):
    """Lane i of a 96-bit group equals bits 3i..3i+2 of the 96-bit
    little-endian integer (brute force with Python big integers)."""
    rng = np.random.default_rng(1)
    W = rng.integers(0, 1 << 32, size=(2000, 3), dtype=np.uint64).astype(np.uint32)
    got = orc.unpack3_words(W)
    for g in range(W.shape[0]):
        big = int(W[g, 0]) | int(W[g, 1]) << 32 | int(W[g, 2]) << 64
        exp = [(big >> (3 * i)) & 7 for i in range(32)]
        assert got[g].tolist() == exp
