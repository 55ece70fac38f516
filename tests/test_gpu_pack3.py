"""GPU parity of pack3 / unpack3 / unpack3_words with the oracle, bit exact,
including the exhaustive 2^24 octet state space in both directions."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_num_gb300 as P
    P.lib()
    return P


def test_exhaustive_bijection_on_gpu(pkv, orc):
    lanes = W.all_octets()                                   # [2^24, 8] host
    exp_packed = orc.pack3(lanes.numpy())                    # oracle, [2^24, 3]
    d_lanes = lanes.reshape(-1).cuda()
    packed = pkv.pack3(d_lanes)
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy().reshape(-1, 3), exp_packed)
    # right inverse: every byte triple unpacks to the oracle's lanes
    back = pkv.unpack3(packed)
    torch.cuda.synchronize()
    exp_lanes = orc.unpack3(exp_packed)
    assert np.array_equal(back.cpu().numpy().reshape(-1, 8), exp_lanes)
    assert np.array_equal(exp_lanes, lanes.numpy())


@pytest.mark.parametrize("n", [0, 1, 3, 4, 5, 7, 1001, 4099])
def test_ragged_sizes(pkv, orc, n):
    rng = np.random.default_rng(n)
    vals = rng.integers(0, 256, size=(max(n, 1) * 8,), dtype=np.uint8)[:n * 8]
    d = torch.from_numpy(vals.copy()).cuda()
    packed = pkv.pack3(d)
    torch.cuda.synchronize()
    exp = orc.pack3(vals.reshape(-1, 8)).reshape(-1) if n else np.zeros(0, np.uint8)
    assert np.array_equal(packed.cpu().numpy(), exp)
    back = pkv.unpack3(packed)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), (vals & 7))


def test_unpack_words_matches_oracle(pkv, orc):
    rng = np.random.default_rng(7)
    W_ = rng.integers(0, 1 << 32, size=(50000, 3), dtype=np.uint64).astype(np.uint32)
    exp = orc.unpack3_words(W_)
    d = torch.from_numpy(W_.view(np.int32).copy()).cuda().reshape(-1)
    got = pkv.unpack3_words(d)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().reshape(-1, 32), exp)


def test_walking_isolation_on_gpu(pkv, orc):
    """Walking one lane through every value over 000 / 111 backgrounds for all
    32 lanes: packed by the GPU, unpacked by the GPU's word path."""
    vals = []
    for bg in (0, 7):
        for lane in range(32):
            for v in range(8):
                x = np.full(32, bg, np.uint8)
                x[lane] = v
                vals.append(x)
    vals = np.stack(vals)                                   # [512, 32]
    packed = pkv.pack3(torch.from_numpy(vals.reshape(-1).copy()).cuda())
    words = pkv.unpack3_words(packed.view(torch.int32))
    torch.cuda.synchronize()
    assert np.array_equal(words.cpu().numpy().reshape(-1, 32), vals)
    assert np.array_equal(packed.cpu().numpy().reshape(-1, 3),
                          orc.pack3(vals.reshape(-1, 8)))


@pytest.mark.parametrize("n,off", [(4099, 4), (4099, 0), (33, 8), (16, 12)])
def test_unpack_alignments(pkv, orc, n, off):
    """unpack3 from packed data at 16-byte aligned and merely 4-byte aligned
    addresses (both kernels), with tails of every length mod 16."""
    rng = np.random.default_rng(n + off)
    packed_h = rng.integers(0, 256, size=(n * 3,), dtype=np.uint8)
    buf = torch.zeros(n * 3 + 16, dtype=torch.uint8, device="cuda")
    buf[off:off + n * 3] = torch.from_numpy(packed_h).cuda()
    got = pkv.unpack3(buf[off:off + n * 3])
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().reshape(-1, 8), orc.unpack3(packed_h.reshape(-1, 3)))


@pytest.mark.parametrize("m,off", [(50001, 0), (50001, 4), (3, 0), (6, 8)])
def test_unpack_words_ragged_and_unaligned(pkv, orc, m, off):
    rng = np.random.default_rng(m + off)
    W_ = rng.integers(0, 1 << 32, size=(m, 3), dtype=np.uint64).astype(np.uint32)
    buf = torch.zeros(m * 3 + 4, dtype=torch.int32, device="cuda")
    o = off // 4
    buf[o:o + m * 3] = torch.from_numpy(W_.view(np.int32).reshape(-1).copy()).cuda()
    got = pkv.unpack3_words(buf[o:o + m * 3])
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().reshape(-1, 32), orc.unpack3_words(W_))
