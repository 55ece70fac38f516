"""Pins for the oracle's storage-layout relabelling (the x-vectorised paged
layout) against a hand-written fixture and plain transposes.  CPU only."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "xvec_layout.txt")


def _fixture():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            off, rhs = line.split("=")
            t = rhs.split()
            rows.append((int(off), int(t[1]), int(t[3]), int(t[5]), int(t[7])))
    return rows


def test_xvec_matches_golden_storage_order(orc):
    P, BS, H, D, x = 2, 2, 2, 4, 2
    b, s, h, d = np.meshgrid(np.arange(P), np.arange(BS), np.arange(H), np.arange(D), indexing="ij")
    label = ((b * 10 + s) * 10 + h) * 10 + d            # unique per element
    flat = orc.to_xvec(label, x).ravel()
    rows = _fixture()
    assert len(rows) == P * BS * H * D
    for off, bb, ss, hh, dd in rows:
        assert flat[off] == ((bb * 10 + ss) * 10 + hh) * 10 + dd, off


def test_xvec_roundtrip_and_shape(orc):
    rng = np.random.default_rng(5)
    for (P, BS, H, D), x in [((3, 16, 2, 128), 8), ((2, 32, 3, 128), 16), ((1, 16, 1, 64), 8)]:
        a = rng.integers(0, 1 << 16, size=(P, BS, H, D)).astype(np.uint16)
        phys = orc.to_xvec(a, x)
        assert phys.shape == (P, H, D // x, BS, x)
        assert np.array_equal(orc.from_xvec(phys), a)


def test_xvec_with_one_piece_is_head_major(orc):
    # x = head_dim: one piece per row, so the layout is [P, Hkv, 1, BS, D],
    # the head-major transpose of the flash layout
    a = np.arange(2 * 16 * 4 * 8, dtype=np.int32).reshape(2, 16, 4, 8)
    assert np.array_equal(orc.to_xvec(a, 8)[:, :, 0], a.transpose(0, 2, 1, 3))


def test_xvec_pieces_are_16_bytes_of_one_row(orc):
    # with x = 16 bytes / element size, every 16-byte unit of the storage is
    # x consecutive elements of a single (block, slot, head) row
    rng = np.random.default_rng(6)
    for dt in (np.uint16, np.uint8):
        x = orc.xvec_elems(np.dtype(dt).itemsize)
        a = rng.integers(0, 200, size=(2, 16, 2, 128)).astype(dt)
        units = orc.to_xvec(a, x).view(np.uint8).reshape(-1, 16)
        rows = a.view(np.uint8).reshape(-1, 16)        # 16-byte pieces of the rows
        assert sorted(map(bytes, units)) == sorted(map(bytes, rows))
