"""GPU parity of kv_append (16-bit copy, fp8 e4m3, 3-bit) and of the device
slot_mapping builder with the oracle: bit exact over the whole pool,
including the untouched blocks and the -1 padding tokens."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import pipeline as PL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_num_gb300 as P
    P.lib()
    return P


def _assert_pools_equal(gpu, orc_c):
    for name, arr in orc_c.items():
        assert np.array_equal(gpu[name], arr), name


def test_slot_mapping_kernel(pkv, orc):
    w = W.mixed_append(n_prefill=4, n_decode=20, prefill_lo=10, prefill_hi=300, ctx_lo=5,
                       ctx_hi=700, pad_to=256)
    bt = w.block_tables
    got = pkv.slot_mapping(bt.cuda(), w.new_req.cuda(), w.new_pos.cuda(), w.block_size)
    torch.cuda.synchronize()
    exp = orc.build_slot_mapping(bt.numpy(), w.new_req.numpy(), w.new_pos.numpy(), w.block_size)
    assert np.array_equal(got.cpu().numpy(), exp)


def test_slot_mapping_out_of_table_flags(pkv):
    bt = torch.zeros((2, 3), dtype=torch.int32, device="cuda")
    req = torch.tensor([0, 1, 5, 0], dtype=torch.int32, device="cuda")
    pos = torch.tensor([3, 48, 0, -1], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = pkv.slot_mapping(bt, req, pos, 16, err_flag=err)
    torch.cuda.synchronize()
    assert got.tolist() == [3, -1, -1, -1]
    assert int(err.item()) & pkv.pkv.DEVERR_POS_RANGE


@pytest.mark.parametrize("literal", [False, True])
def test_tiny_append(pkv, orc, literal):
    w = W.tiny(literal=literal)
    cache, _ = PL.gpu_run(w, pkv, decode=False)
    _assert_pools_equal(PL.gpu_cache_host(cache), PL.oracle_caches(w, orc))


@pytest.mark.parametrize("size", ["small", "full"])
def test_mixed_prefill_decode_append(pkv, orc, size):
    if size == "small":
        w = W.mixed_append(n_prefill=3, n_decode=10, prefill_lo=20, prefill_hi=200, ctx_lo=30,
                           ctx_hi=400)
    else:
        w = W.mixed_append()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache, _ = PL.gpu_run(w, pkv, decode=False, err_flag=err)
    assert int(err.item()) == 0
    _assert_pools_equal(PL.gpu_cache_host(cache), PL.oracle_caches(w, orc))
    assert w.new_pos.numpy()[-1] == -1          # padding present


def test_strided_source_rows(pkv, orc):
    """K and V sliced out of a fused [T, 3, Hkv, D] projection output."""
    w = W.gqa_bf16(batch=5, ctx_lo=3, ctx_hi=100, seed=21)
    T, H, D = w.k_new.shape
    fused = torch.randn((T, 3, H, D), dtype=w.dtype)
    fused[:, 1] = w.k_new
    fused[:, 2] = w.v_new
    cache = pkv.KVCache.allocate("bf16", w.num_blocks, w.block_size, H, D)
    cache.k_cache.copy_(w.k_cache0.cuda())
    cache.v_cache.copy_(w.v_cache0.cuda())
    fd = fused.cuda()
    sm = pkv.slot_mapping(w.block_tables.cuda(), w.new_req.cuda(), w.new_pos.cuda(), w.block_size)
    pkv.kv_append(fd[:, 1], fd[:, 2], sm, cache)
    torch.cuda.synchronize()
    _assert_pools_equal(PL.gpu_cache_host(cache), PL.oracle_caches(w, orc))


def test_unaligned_source_uses_scalar_path(pkv, orc):
    w = W.tiny()
    T, H, D = w.k_new.shape
    buf = torch.empty(T * H * D + 1, dtype=w.dtype, device="cuda")
    k = buf[1:].view(T, H, D)
    k.copy_(w.k_new.cuda())
    cache = pkv.KVCache.allocate("f16", w.num_blocks, w.block_size, H, D)
    cache.k_cache.copy_(w.k_cache0.cuda())
    cache.v_cache.copy_(w.v_cache0.cuda())
    sm = pkv.slot_mapping(w.block_tables.cuda(), w.new_req.cuda(), w.new_pos.cuda(), w.block_size)
    pkv.kv_append(k, w.v_new.cuda(), sm, cache)
    torch.cuda.synchronize()
    _assert_pools_equal(PL.gpu_cache_host(cache), PL.oracle_caches(w, orc))


def test_out_of_range_slot_is_skipped_and_flagged(pkv):
    H, D, P, BS = 2, 64, 4, 16
    cache = pkv.KVCache.allocate("f16", P, BS, H, D, fill=0)
    kn = torch.ones((3, H, D), dtype=torch.float16, device="cuda")
    sm = torch.tensor([5, P * BS, -1], dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.kv_append(kn, kn, sm, cache, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.pkv.DEVERR_SLOT_RANGE
    flat = cache.k_cache.view(P * BS, H, D)
    assert torch.all(flat[5] == 1) and int((flat != 0).sum()) == H * D


@pytest.mark.parametrize("Hkv,T", [(8, 1500), (2, 4096), (16, 1024)])
def test_bulk_copy_path_large_batch(pkv, orc, Hkv, T):
    """Batches of >= 1024 tokens whose head rows are contiguous take the
    TMA bulk-copy append (global -> shared -> global per (token, K|V) row):
    bit exact over the whole pool, with padding tokens and slots out of the
    pool skipped (and flagged), at several row sizes and ring wrap-arounds."""
    D, BS = 128, 16
    g = torch.Generator().manual_seed(300 + Hkv)
    P = (T + 200) // BS + 8
    perm = torch.randperm(P * BS, generator=g)[:T].to(torch.int64)
    slots = perm.clone()
    slots[::7] = -1                                   # padding tokens
    slots[3] = P * BS + 11                            # out of the pool
    kn = torch.randn((T, Hkv, D), generator=g).to(torch.bfloat16)
    vn = torch.randn((T, Hkv, D), generator=g).to(torch.bfloat16)
    kn[slots < 0] = float("nan")
    vn[slots < 0] = float("nan")
    k0 = torch.randint(0, 256, (P * BS * Hkv * D * 2,), generator=g, dtype=torch.uint8)
    v0 = torch.randint(0, 256, (P * BS * Hkv * D * 2,), generator=g, dtype=torch.uint8)
    cache = pkv.KVCache.allocate("bf16", P, BS, Hkv, D)
    cache.k_cache.view(torch.uint8).view(-1).copy_(k0.cuda())
    cache.v_cache.view(torch.uint8).view(-1).copy_(v0.cuda())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.kv_append(kn.cuda(), vn.cuda(), slots.cuda(), cache, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.pkv.DEVERR_SLOT_RANGE
    ok_ = k0.view(torch.int16).numpy().view(np.uint16).reshape(P, BS, Hkv, D).copy()
    ov_ = v0.view(torch.int16).numpy().view(np.uint16).reshape(P, BS, Hkv, D).copy()
    bad = orc.kv_append(2, 2, W.bits16(kn), W.bits16(vn), slots.numpy(), ok_, ov_)
    assert bad == 1
    got = PL.gpu_cache_host(cache)
    assert np.array_equal(got["k_cache"], ok_) and np.array_equal(got["v_cache"], ov_)


def test_idempotent_append(pkv):
    w = W.tiny()
    cache, _ = PL.gpu_run(w, pkv, decode=False)
    before = PL.gpu_cache_host(cache)
    sm = pkv.slot_mapping(w.block_tables.cuda(), w.new_req.cuda(), w.new_pos.cuda(), w.block_size)
    pkv.kv_append(w.k_new.cuda(), w.v_new.cuda(), sm, cache)
    torch.cuda.synchronize()
    after = PL.gpu_cache_host(cache)
    for k in before:
        assert np.array_equal(before[k], after[k])


@pytest.mark.parametrize("src,fp8", [(torch.bfloat16, "e4m3"), (torch.float16, "e4m3"),
                                     (torch.bfloat16, "e5m2"), (torch.float16, "e5m2"),
                                     (torch.bfloat16, "i8"), (torch.float16, "i8")])
def test_fp8_every_source_pattern(pkv, orc, src, fp8):
    """All 2^16 source bit patterns (NaN, inf, subnormal, overflow included)
    through the one-byte appends (e4m3, e5m2, int8) for several scales: bit
    exact with the oracle, which encodes from the formats' definitions."""
    H, D, BS = 4, 128, 16
    pats = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16).view(src)
    T = (1 << 16) // D                        # 512 tokens, one head row each x 4 heads
    kn = pats.reshape(T, 1, D).repeat(1, H, 1)
    vn = pats.flip(0).reshape(T, 1, D).repeat(1, H, 1)
    P = T // BS
    k_scale = torch.tensor([1.0, 1e-3, 37.5, 2.0 ** -20], dtype=torch.float32)
    v_scale = torch.tensor([0.5, 3e4, 1.0 / 3.0, 448.0], dtype=torch.float32)
    cache = pkv.KVCache.allocate(fp8, P, BS, H, D, k_scale=k_scale.cuda(),
                                 v_scale=v_scale.cuda(), fill=0)
    slots = torch.randperm(P * BS, generator=torch.Generator().manual_seed(3))[:T]
    pkv.kv_append(kn.cuda(), vn.cuda(), slots.cuda(), cache)
    torch.cuda.synchronize()
    kc = np.zeros((P, BS, H, D), np.int8 if fp8 == "i8" else np.uint8)
    vc = np.zeros_like(kc)
    code = 1 if src == torch.float16 else 2
    orc.kv_append(PL.KIND_CODE_ORACLE[fp8], code, W.bits16(kn), W.bits16(vn), slots.numpy(), kc, vc,
                  k_scale.numpy(), v_scale.numpy())
    assert np.array_equal(cache.k_cache.cpu().numpy(), kc)
    assert np.array_equal(cache.v_cache.cpu().numpy(), vc)


@pytest.mark.parametrize("D,src", [(128, torch.float16), (64, torch.float16),
                                   (128, torch.bfloat16)])
def test_u3_append_bit_exact(pkv, orc, D, src):
    H, BS, P, T = 3, 16, 40, 500
    g = torch.Generator().manual_seed(D)
    kn = torch.randn((T, H, D), generator=g).to(src)
    vn = (torch.randn((T, H, D), generator=g) * 50).to(src)
    kn[7] = 1.25                                   # constant rows: scale 0
    kn[8, 1, :5] = -2.0                            # ties / repeated extremes
    slots = torch.randperm(P * BS, generator=g)[:T]
    slots[[0, 99]] = -1
    cache = pkv.KVCache.allocate("u3", P, BS, H, D, fill=0)
    pkv.kv_append(kn.cuda(), vn.cuda(), slots.cuda(), cache)
    torch.cuda.synchronize()
    RB = 3 * D // 8
    c = {"k_cache": np.zeros((P, BS, H, RB), np.uint8), "v_cache": np.zeros((P, BS, H, RB), np.uint8),
         "k_qscale": np.zeros((P, BS, H), np.uint16), "v_qscale": np.zeros((P, BS, H), np.uint16),
         "k_qzero": np.zeros((P, BS, H), np.uint8), "v_qzero": np.zeros((P, BS, H), np.uint8)}
    code = 1 if src == torch.float16 else 2
    orc.kv_append(4, code, W.bits16(kn), W.bits16(vn), slots.numpy(), c["k_cache"], c["v_cache"],
                  None, None, c["k_qscale"], c["k_qzero"], c["v_qscale"], c["v_qzero"])
    _assert_pools_equal(PL.gpu_cache_host(cache), c)


@pytest.mark.parametrize("src", [torch.float16, torch.bfloat16])
def test_u3_append_ties_zeros_extremes(pkv, orc, src):
    """3-bit rows whose quotients x / scale are exact half-integers (ties,
    rounded to even), rows of zeros with a few nonzero values, rows whose
    range overflows fp32 or fp16, and rows of tiny values: the kernel's
    division shortcut must fall back to the division wherever it could
    change a code, so the pool stays bit-exact with the oracle."""
    H, D, BS, P = 2, 128, 16, 16
    g = torch.Generator().manual_seed(278)
    big = 60000.0 if src == torch.float16 else 3.0e38
    rows = []
    ramp = torch.arange(-7, 8, dtype=torch.float32) * 0.125           # x / 0.25 = k / 2
    rows.append(ramp.repeat(D // 15 + 1)[:D])
    rows.append(torch.cat([ramp, ramp.flip(0)]).repeat(D // 30 + 1)[:D] * 4.0)
    z = torch.zeros(D)
    z[[3, 50]] = torch.tensor([0.75, -1.5])
    rows.append(z)
    e = torch.randn(D, generator=g)
    e[[0, 1]] = torch.tensor([big, -big])
    rows.append(e)
    rows.append(torch.randn(D, generator=g) * 1e-6)
    rows.append(torch.randn(D, generator=g) * 2.0 ** -30)
    R = torch.stack(rows)                                              # [6, D]
    T = 48
    kn = R[torch.arange(T * H) % R.shape[0]].reshape(T, H, D).to(src)
    vn = R[(torch.arange(T * H) + 3) % R.shape[0]].reshape(T, H, D).neg().to(src)
    slots = torch.randperm(P * BS, generator=g)[:T]
    cache = pkv.KVCache.allocate("u3", P, BS, H, D, fill=0)
    pkv.kv_append(kn.cuda(), vn.cuda(), slots.cuda(), cache)
    torch.cuda.synchronize()
    RB = 3 * D // 8
    c = {"k_cache": np.zeros((P, BS, H, RB), np.uint8), "v_cache": np.zeros((P, BS, H, RB), np.uint8),
         "k_qscale": np.zeros((P, BS, H), np.uint16), "v_qscale": np.zeros((P, BS, H), np.uint16),
         "k_qzero": np.zeros((P, BS, H), np.uint8), "v_qzero": np.zeros((P, BS, H), np.uint8)}
    code = 1 if src == torch.float16 else 2
    orc.kv_append(4, code, W.bits16(kn), W.bits16(vn), slots.numpy(), c["k_cache"], c["v_cache"],
                  None, None, c["k_qscale"], c["k_qzero"], c["v_qscale"], c["v_qzero"])
    _assert_pools_equal(PL.gpu_cache_host(cache), c)


@pytest.mark.parametrize("D", [64, 128])
def test_u3_append_hand_worked_ties(pkv, D):
    """The hand-worked rows of tests/golden/u3_ties.txt (tie quotients in the
    zero point and the codes, fp16 scale ties both ways, clamped codes,
    constant rows), tiled along head_dim, appended by the GPU: its scale
    bits, zero points and unpacked codes equal the hand-worked values
    directly, with no oracle in between."""
    from tests.refs import bitstream_unpack3, load_u3_ties
    rows = load_u3_ties()
    R = np.stack([np.tile(r[3], D // 16) for r in rows])              # [n, D] fp16
    H, BS = 2, 16
    n = R.shape[0]
    T = n                                                              # token t: K row t, V row n-1-t
    P = (T + BS - 1) // BS + 1
    kn = torch.from_numpy(R.astype(np.float32)).reshape(T, 1, D).expand(T, H, D).to(torch.float16)
    vn = torch.from_numpy(R[::-1].astype(np.float32).copy()).reshape(T, 1, D).expand(T, H, D).to(torch.float16)
    slots = torch.arange(T, dtype=torch.int64) + BS                    # skip block 0
    cache = pkv.KVCache.allocate("u3", P, BS, H, D, fill=0)
    pkv.kv_append(kn.contiguous().cuda(), vn.contiguous().cuda(), slots.cuda(), cache)
    torch.cuda.synchronize()
    got = PL.gpu_cache_host(cache)
    RB = 3 * D // 8
    for part, order in (("k", range(n)), ("v", range(n - 1, -1, -1))):
        packed = got[part + "_cache"].reshape(P * BS, H, RB)
        sc = got[part + "_qscale"].reshape(P * BS, H)
        zr = got[part + "_qzero"].reshape(P * BS, H)
        for t, ri in enumerate(order):
            name, s_exp, z_exp, _, q_exp = rows[ri]
            for h in range(H):
                slot = BS + t
                assert int(sc[slot, h]) == s_exp, (part, name, h)
                assert int(zr[slot, h]) == z_exp, (part, name, h)
                q = bitstream_unpack3(packed[slot, h][None, :], D)[0]
                assert np.array_equal(q, np.tile(q_exp, D // 16)), (part, name, h)
    assert not got["k_cache"][0].any() and not got["v_cache"][0].any()  # block 0 untouched


@pytest.mark.parametrize("src", [torch.float16, torch.bfloat16])
def test_u3_append_every_source_pattern_in_range(pkv, orc, src):
    """Every finite fp16 (or bf16) value x between a row's minimum -3s and
    maximum 4s, for scales s from 2^-20 to 2^12 (at most 8 significant bits,
    so that -3s and 4s are exact and the row's scale is s, zero point 3):
    the 3-bit append's codes, scales and zero points equal the oracle's
    (division, then round half to even) bit for bit.  This covers every
    quotient x / s the codes can take at these scales, the exact
    half-integer ties included."""
    D, H, BS = 128, 2, 16
    g = torch.Generator().manual_seed(281)
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    allv = bits.view(src).to(torch.float64)
    allv = allv[torch.isfinite(allv)]
    rows = []
    for s in (2.0 ** -20, 3 * 2.0 ** -14, 0.0078125 * 5, 0.25, 1.0, 1.5, 7.0, 100.0, 255.0 / 64, 2.0 ** 12):
        sv = torch.tensor(s, dtype=torch.float64)
        if any(float((k * sv).to(src).double()) != k * s for k in (1, 3, 4)):
            continue                    # anchors not exact in this source type
        vals = allv[(allv >= -3 * s) & (allv <= 4 * s)]
        vals = vals[torch.randperm(vals.numel(), generator=g)]
        n = (vals.numel() + D - 3) // (D - 2)
        pad = n * (D - 2) - vals.numel()
        vals = torch.cat([vals, vals[:pad]]).reshape(n, D - 2)
        anchors = torch.tensor([-3 * s, 4 * s], dtype=torch.float64).expand(n, 2)
        rows.append(torch.cat([anchors, vals], 1))
    R = torch.cat(rows).to(src)                                   # [n_rows, D]
    T = (R.shape[0] + 2 * H - 1) // (2 * H)
    R = torch.cat([R, R[:T * 2 * H - R.shape[0]]])
    kn = R[:T * H].reshape(T, H, D)
    vn = R[T * H:].reshape(T, H, D)
    P = (T + BS - 1) // BS + 1
    slots = torch.randperm(P * BS, generator=g)[:T]
    cache = pkv.KVCache.allocate("u3", P, BS, H, D, fill=0)
    pkv.kv_append(kn.cuda(), vn.cuda(), slots.cuda(), cache)
    torch.cuda.synchronize()
    RB = 3 * D // 8
    c = {"k_cache": np.zeros((P, BS, H, RB), np.uint8), "v_cache": np.zeros((P, BS, H, RB), np.uint8),
         "k_qscale": np.zeros((P, BS, H), np.uint16), "v_qscale": np.zeros((P, BS, H), np.uint16),
         "k_qzero": np.zeros((P, BS, H), np.uint8), "v_qzero": np.zeros((P, BS, H), np.uint8)}
    code = 1 if src == torch.float16 else 2
    orc.kv_append(4, code, W.bits16(kn), W.bits16(vn), slots.numpy(), c["k_cache"], c["v_cache"],
                  None, None, c["k_qscale"], c["k_qzero"], c["v_qscale"], c["v_qzero"])
    got = PL.gpu_cache_host(cache)
    assert np.all(c["k_qzero"][slots.numpy() // BS, slots.numpy() % BS] == 3)
    _assert_pools_equal(got, c)


def test_u3_append_unaligned_rows_and_sources(pkv, orc):
    """3-bit rows at a head stride of 49 bytes (rows start at any byte: the
    kernel stores their 12-byte runs byte by byte) from sources that start
    one element past a 16-byte boundary (scalar loads): the same codes and
    metadata as the oracle, and the padding byte after each row untouched."""
    H, D, BS, P, T = 3, 128, 16, 12, 100
    RB = 3 * D // 8
    g = torch.Generator().manual_seed(279)
    kn = torch.randn((T, H, D), generator=g).to(torch.float16)
    vn = (torch.randn((T, H, D), generator=g) * 7).to(torch.float16)
    slots = torch.randperm(P * BS, generator=g)[:T]
    dev = "cuda"
    kbuf = torch.empty(T * H * D + 1, dtype=torch.float16, device=dev)
    vbuf = torch.empty_like(kbuf)
    ksrc, vsrc = kbuf[1:].view(T, H, D), vbuf[1:].view(T, H, D)
    ksrc.copy_(kn.to(dev))
    vsrc.copy_(vn.to(dev))
    ref = pkv.KVCache.allocate("u3", P, BS, H, D, fill=0)
    wide_k = torch.full((P, BS, H, RB + 1), 0xA5, dtype=torch.uint8, device=dev)
    wide_v = torch.full_like(wide_k, 0x5A)
    cache = pkv.KVCache("u3", wide_k[..., :RB], wide_v[..., :RB], k_qscale=ref.k_qscale.clone(),
                        k_qzero=ref.k_qzero.clone(), v_qscale=ref.v_qscale.clone(),
                        v_qzero=ref.v_qzero.clone())
    assert cache.k_cache.stride(2) == RB + 1
    pkv.kv_append(ksrc, vsrc, slots.to(dev), cache)
    torch.cuda.synchronize()
    c = {"k_cache": np.zeros((P, BS, H, RB), np.uint8), "v_cache": np.zeros((P, BS, H, RB), np.uint8),
         "k_qscale": np.zeros((P, BS, H), np.uint16), "v_qscale": np.zeros((P, BS, H), np.uint16),
         "k_qzero": np.zeros((P, BS, H), np.uint8), "v_qzero": np.zeros((P, BS, H), np.uint8)}
    orc.kv_append(4, 1, W.bits16(kn), W.bits16(vn), slots.numpy(), c["k_cache"], c["v_cache"],
                  None, None, c["k_qscale"], c["k_qzero"], c["v_qscale"], c["v_qzero"])
    written = np.zeros((P * BS,), bool)
    written[slots.numpy()] = True
    written = written.reshape(P, BS)
    got = PL.gpu_cache_host(cache)
    for name in ("k_cache", "v_cache"):
        fill = 0xA5 if name == "k_cache" else 0x5A
        exp = np.where(written[:, :, None, None], c[name], np.uint8(fill))
        assert np.array_equal(got[name], exp), name
    for name in ("k_qscale", "v_qscale", "k_qzero", "v_qzero"):
        assert np.array_equal(got[name], c[name]), name
    pad_k = wide_k[..., RB].cpu().numpy()
    pad_v = wide_v[..., RB].cpu().numpy()
    assert (pad_k == 0xA5).all() and (pad_v == 0x5A).all()


@pytest.mark.parametrize("kind,H", [("bf16", 16), ("e4m3", 16), ("u3", 4)])
def test_append_many_items_several_passes(pkv, orc, kind, H):
    """Batches large enough that every warp of the grid walks several work
    items, with more than one part (or row) per token: a strided 16-bit
    source (the warp kernel, not the bulk path), 16 kv heads for e4m3 (two
    parts per token row), 4 heads for 3-bit (four rows per warp spanning
    tokens). The whole pool stays bit-exact with the oracle, padding and
    skipped slots included."""
    D, BS = 128, 16
    T = 12000
    P = (T + 600) // BS + 1
    g = torch.Generator().manual_seed(280 + H)
    src_dt = torch.bfloat16
    # [T, H, 3, D]: K and V heads interleaved with a third row, so a token's
    # heads are not one contiguous run and the 16-bit append takes the warp
    # kernel rather than the bulk copies
    fused = torch.randn((T, H, 3, D), generator=g).to(src_dt)
    kn, vn = fused[:, :, 1], fused[:, :, 2]
    slots = torch.randperm(P * BS, generator=g)[:T]
    slots[::97] = -1                                               # padding tokens
    dev = "cuda"
    if kind == "e4m3":
        ks = (torch.rand(H, generator=g) * 0.02 + 0.005).float()
        vs = (torch.rand(H, generator=g) * 0.02 + 0.005).float()
        cache = pkv.KVCache.allocate(kind, P, BS, H, D, k_scale=ks.to(dev), v_scale=vs.to(dev), fill=0)
    else:
        ks = vs = None
        cache = pkv.KVCache.allocate(kind, P, BS, H, D, fill=0)
    fd = fused.to(dev)
    pkv.kv_append(fd[:, :, 1], fd[:, :, 2], slots.to(dev), cache)
    torch.cuda.synchronize()
    if kind == "u3":
        RB = 3 * D // 8
        c = {"k_cache": np.zeros((P, BS, H, RB), np.uint8), "v_cache": np.zeros((P, BS, H, RB), np.uint8),
             "k_qscale": np.zeros((P, BS, H), np.uint16), "v_qscale": np.zeros((P, BS, H), np.uint16),
             "k_qzero": np.zeros((P, BS, H), np.uint8), "v_qzero": np.zeros((P, BS, H), np.uint8)}
        orc.kv_append(4, 2, W.bits16(kn), W.bits16(vn), slots.numpy(), c["k_cache"], c["v_cache"],
                      None, None, c["k_qscale"], c["k_qzero"], c["v_qscale"], c["v_qzero"])
    else:
        dt = np.uint16 if kind == "bf16" else np.uint8
        c = {"k_cache": np.zeros((P, BS, H, D), dt), "v_cache": np.zeros((P, BS, H, D), dt)}
        orc.kv_append(PL.KIND_CODE_ORACLE[kind], 2, W.bits16(kn), W.bits16(vn), slots.numpy(),
                      c["k_cache"], c["v_cache"], None if ks is None else ks.numpy(),
                      None if vs is None else vs.numpy())
    _assert_pools_equal(PL.gpu_cache_host(cache), c)
