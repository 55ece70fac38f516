"""Pins for the oracle's slot_mapping builder and scatter ("Write Triton Kv
Cache Append Kernel": reasoning steps 5, 6 and 9; correctness requirements;
output format item 4).  CPU only."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.refs import bitstream_unpack3, e4m3_dequant, e5m2_dequant


def _slots_closed_form(bt, req, pos, BS):
    out = np.full(len(req), -1, np.int64)
    for t, (r, p) in enumerate(zip(req, pos)):
        if p >= 0:
            out[t] = int(bt[r][p // BS]) * BS + p % BS
    return out


def test_slot_mapping_builder(orc):
    w = W.mixed_append(n_prefill=3, n_decode=5, prefill_lo=5, prefill_hi=70, ctx_lo=3,
                       ctx_hi=90, pad_to=64)
    bt = w.block_tables.numpy()
    req, pos = w.new_req.numpy(), w.new_pos.numpy()
    sm = orc.build_slot_mapping(bt, req, pos, w.block_size)
    assert np.array_equal(sm, _slots_closed_form(bt, req, pos, w.block_size))
    real = pos >= 0
    # decomposition back into (physical block, offset) matches the table
    assert np.array_equal(sm[real] // w.block_size, bt[req[real], pos[real] // w.block_size])
    assert np.array_equal(sm[real] % w.block_size, pos[real] % w.block_size)
    # distinct tokens of distinct positions get distinct slots
    assert len(set(sm[real].tolist())) == int(real.sum())
    assert np.all(sm[~real] == -1)


def _scatter_case(orc, dt, seed=0):
    g = torch.Generator().manual_seed(seed)
    P, BS, H, D, T = 9, 16, 3, 64, 40
    k0 = torch.randn((P, BS, H, D), generator=g).to(dt)
    v0 = torch.randn((P, BS, H, D), generator=g).to(dt)
    kn = torch.randn((T, H, D), generator=g).to(dt)
    vn = torch.randn((T, H, D), generator=g).to(dt)
    slots = torch.randperm(P * BS, generator=g)[:T].numpy().astype(np.int64)
    slots[[3, 17, 39]] = -1            # padding tokens
    kn[[3, 17, 39]] = float("nan")     # their rows must never be read
    vn[[3, 17, 39]] = float("nan")
    return P, BS, H, D, T, k0, v0, kn, vn, slots


def test_scatter_16bit_readback_and_untouched(orc):
    for dt, code in ((torch.float16, orc.F16), (torch.bfloat16, orc.BF16)):
        P, BS, H, D, T, k0, v0, kn, vn, slots = _scatter_case(orc, dt)
        kc, vc = W.bits16(k0).copy(), W.bits16(v0).copy()
        bad = orc.kv_append(code, code, W.bits16(kn), W.bits16(vn), slots, kc, vc)
        assert bad == 0
        # expected pool: initial pool with the written rows replaced
        ek, ev = W.bits16(k0).copy(), W.bits16(v0).copy()
        for t, s in enumerate(slots):
            if s >= 0:
                ek[s // BS, s % BS] = W.bits16(kn)[t]
                ev[s // BS, s % BS] = W.bits16(vn)[t]
        assert np.array_equal(kc, ek) and np.array_equal(vc, ev)
        # readback through the same indirection
        real = slots >= 0
        assert np.array_equal(kc.reshape(P * BS, H, D)[slots[real]], W.bits16(kn)[real])
        # no NaN from the padding rows anywhere
        assert not np.isnan(W.bits16(kn)[real].view(np.float16)).any() or dt == torch.bfloat16
        # idempotence: applying the same append again changes nothing
        kc2, vc2 = kc.copy(), vc.copy()
        orc.kv_append(code, code, W.bits16(kn), W.bits16(vn), slots, kc2, vc2)
        assert np.array_equal(kc2, kc) and np.array_equal(vc2, vc)


def test_scatter_out_of_range_slots_skipped(orc):
    P, BS, H, D, T, k0, v0, kn, vn, slots = _scatter_case(orc, torch.float16, seed=1)
    slots = slots.copy()
    slots[5] = P * BS          # one past the pool
    slots[6] = P * BS + 1000
    kc, vc = W.bits16(k0).copy(), W.bits16(v0).copy()
    bad = orc.kv_append(orc.F16, orc.F16, W.bits16(kn), W.bits16(vn), slots, kc, vc)
    assert bad == 2


def test_scatter_e5m2_matches_cast_and_step(orc):
    """fp8 e5m2: codes equal torch's e5m2 cast of (x / scale) taken in fp32
    (in range), out-of-range values saturate to +-57344, and the dequantised
    cache is within half an e5m2 step of the source."""
    P, BS, H, D, T, k0, v0, kn, vn, slots = _scatter_case(orc, torch.bfloat16, seed=3)
    # head 2 of V gets a scale too small for its values: those saturate
    kscale = np.array([1e-4, 2e-4, 3e-5], np.float32)
    vscale = np.array([1.5e-4, 5e-5, 2e-5], np.float32)
    kc = np.zeros((P, BS, H, D), np.uint8)
    vc = np.zeros((P, BS, H, D), np.uint8)
    orc.kv_append(orc.E5M2, orc.BF16, W.bits16(kn), W.bits16(vn), slots, kc, vc, kscale, vscale)
    real = slots >= 0
    for cache, src, sc in ((kc, kn, kscale), (vc, vn, vscale)):
        x = src[torch.from_numpy(real)].float() / torch.from_numpy(sc)[None, :, None]
        inr = (x.abs() < 57344).numpy()
        ref = x.to(torch.float8_e5m2).view(torch.uint8).numpy()
        got = cache.reshape(P * BS, H, D)[slots[real]]
        assert np.array_equal(got[inr], ref[inr])
        sat = np.where(x.numpy() > 0, 0x7B, 0xFB)
        assert np.array_equal(got[~inr], sat[~inr])
        inr_rows = inr.all(axis=(0, 2))
        got, sc = got[:, inr_rows], sc[inr_rows]
        deq = e5m2_dequant(got, sc)
        xs = src[torch.from_numpy(real)].double().numpy()[:, inr_rows]
        # half of the e5m2 spacing at each value: 2^(floor(log2|x/s|)-3) * s
        mag = np.maximum(np.abs(xs) / sc[None, :, None], 2.0 ** -14)
        half_step = 2.0 ** (np.floor(np.log2(mag)) - 3) * sc[None, :, None]
        assert np.all(np.abs(deq - xs) <= half_step * (1 + 1e-6))


def test_scatter_i8_matches_round_and_step(orc):
    """int8: codes equal torch's round-half-even of (x / scale) in fp32,
    clamped to +-127, and the dequantised cache is within half a step
    (the scale) of the source where it is in range."""
    P, BS, H, D, T, k0, v0, kn, vn, slots = _scatter_case(orc, torch.bfloat16, seed=4)
    kscale = np.array([0.02, 0.005, 0.03], np.float32)
    vscale = np.array([0.025, 0.01, 0.004], np.float32)
    kc = np.zeros((P, BS, H, D), np.int8)
    vc = np.zeros((P, BS, H, D), np.int8)
    orc.kv_append(orc.I8, orc.BF16, W.bits16(kn), W.bits16(vn), slots, kc, vc, kscale, vscale)
    real = slots >= 0
    for cache, src, sc in ((kc, kn, kscale), (vc, vn, vscale)):
        x = src[torch.from_numpy(real)].float() / torch.from_numpy(sc)[None, :, None]
        ref = x.round().clamp(-127, 127).to(torch.int8).numpy()
        got = cache.reshape(P * BS, H, D)[slots[real]]
        assert np.array_equal(got, ref)
        inr = (x.abs() <= 127).numpy()
        xs = src[torch.from_numpy(real)].double().numpy()
        deq = got.astype(np.float64) * sc[None, :, None]
        err = np.abs(deq - xs) / sc[None, :, None]
        # half a step, plus the fp32 rounding of x / scale (<= 2^-24 * 127)
        assert np.all(err[inr] <= 0.5 + 1e-5)
        assert (~inr).any()              # some values saturate at these scales


def test_scatter_e4m3_matches_cast_and_step(orc):
    """fp8: codes equal torch's e4m3 cast of (x / scale) taken in fp32 (in
    range), and the dequantised cache is within half a quantisation step of
    the source (the page asks for one step)."""
    P, BS, H, D, T, k0, v0, kn, vn, slots = _scatter_case(orc, torch.bfloat16, seed=2)
    # head 1 of K gets a scale too small for its values: those saturate
    kscale = np.array([0.01, 0.004, 0.02], np.float32)
    vscale = np.array([0.012, 0.03, 0.015], np.float32)
    kc = np.zeros((P, BS, H, D), np.uint8)
    vc = np.zeros((P, BS, H, D), np.uint8)
    orc.kv_append(orc.E4M3, orc.BF16, W.bits16(kn), W.bits16(vn), slots, kc, vc, kscale, vscale)
    real = slots >= 0
    for cache, src, sc in ((kc, kn, kscale), (vc, vn, vscale)):
        x = src[torch.from_numpy(real)].float() / torch.from_numpy(sc)[None, :, None]
        inr = (x.abs() < 448).numpy()
        ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = cache.reshape(P * BS, H, D)[slots[real]]
        assert np.array_equal(got[inr], ref[inr])
        # out of range saturates to +-448 (codes 0x7E / 0xFE)
        sat = np.where(x.numpy() > 0, 0x7E, 0xFE)
        assert np.array_equal(got[~inr], sat[~inr])
        got, inr_rows = got, inr.all(axis=(0, 2))
        got, sc = got[:, inr_rows], sc[inr_rows]
        deq = e4m3_dequant(got, sc)
        xs = src[torch.from_numpy(real)].double().numpy()[:, inr_rows]
        # half of the e4m3 spacing at each value: 2^(floor(log2|x/s|)-4) * s
        mag = np.maximum(np.abs(xs) / sc[None, :, None], 2.0 ** -6)
        half_step = 2.0 ** (np.floor(np.log2(mag)) - 4) * sc[None, :, None]
        assert np.all(np.abs(deq - xs) <= half_step * (1 + 1e-6))
        # rows not written stay zero
        mask = np.ones(P * BS, bool)
        mask[slots[real]] = False
        assert not cache.reshape(P * BS, H, D)[mask].any()


def test_scatter_u3_rows_and_metadata(orc):
    P, BS, H, D, T, k0, v0, kn, vn, slots = _scatter_case(orc, torch.float16, seed=3)
    RB = 3 * D // 8
    kc = np.zeros((P, BS, H, RB), np.uint8)
    vc = np.zeros((P, BS, H, RB), np.uint8)
    ks = np.zeros((P, BS, H), np.uint16)
    kz = np.zeros((P, BS, H), np.uint8)
    vs = np.zeros((P, BS, H), np.uint16)
    vz = np.zeros((P, BS, H), np.uint8)
    orc.kv_append(orc.U3, orc.F16, W.bits16(kn), W.bits16(vn), slots, kc, vc,
                  k_qscale=ks, k_qzero=kz, v_qscale=vs, v_qzero=vz)
    real = slots >= 0
    src = W.bits16(kn)[real].view(np.float16).astype(np.float64)   # [n, H, D]
    rows = kc.reshape(P * BS, H, RB)[slots[real]]
    q = bitstream_unpack3(rows.reshape(-1, RB), D).reshape(-1, H, D)
    s = ks.reshape(P * BS, H)[slots[real]].view(np.float16).astype(np.float64)
    z = kz.reshape(P * BS, H)[slots[real]].astype(np.float64)
    deq = (q - z[..., None]) * s[..., None]
    assert np.all(np.abs(deq - src) <= 1.5 * s[..., None])
    # one quantisation step on average or better
    assert np.mean(np.abs(deq - src) / s[..., None]) < 0.3
    mask = np.ones(P * BS, bool)
    mask[slots[real]] = False
    assert not kc.reshape(P * BS, H, RB)[mask].any() and not ks.reshape(P * BS, H)[mask].any()


@pytest.mark.parametrize("kind", ["e4m3", "i8"])
def test_scatter_per_token_and_per_block_scales(orc, kind):
    """Scale granularities: per block, each row quantised with its block's
    scale for its head; per token, with the scale given for that token and
    head, which is stored at the token's slot.  Codes are checked against
    the per-row cast / round of x / scale, and equal-valued block or token
    scales reproduce the per-head cache exactly."""
    P, BS, H, D, T, k0, v0, kn, vn, slots = _scatter_case(orc, torch.bfloat16, seed=5)
    code = orc.E4M3 if kind == "e4m3" else orc.I8
    dt = np.uint8 if kind == "e4m3" else np.int8
    g = np.random.default_rng(6)
    real = slots >= 0
    rows = slots[real]                      # slot of each real token

    def cast(x):                            # x: torch float32
        if kind == "e4m3":
            return x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        return x.round().clamp(-127, 127).to(torch.int8).numpy()

    # per block
    kb = (g.random((P, H)) * 0.02 + 0.002).astype(np.float32)
    vb = (g.random((P, H)) * 0.02 + 0.002).astype(np.float32)
    kc, vc = np.zeros((P, BS, H, D), dt), np.zeros((P, BS, H, D), dt)
    orc.kv_append(code, orc.BF16, W.bits16(kn), W.bits16(vn), slots, kc, vc,
                  scale_mode=orc.SCALE_PER_BLOCK, k_scales=kb, v_scales=vb)
    for cache, src, sc in ((kc, kn, kb), (vc, vn, vb)):
        x = src[torch.from_numpy(real)].float() / torch.from_numpy(sc[rows // BS])[:, :, None]
        assert np.array_equal(cache.reshape(P * BS, H, D)[rows], cast(x))
    # per token: scales given per new token, stored at its slot
    kt = (g.random((T, H)) * 0.02 + 0.002).astype(np.float32)
    vt = (g.random((T, H)) * 0.02 + 0.002).astype(np.float32)
    ks_arr, vs_arr = np.zeros((P, BS, H), np.float32), np.zeros((P, BS, H), np.float32)
    kc, vc = np.zeros((P, BS, H, D), dt), np.zeros((P, BS, H, D), dt)
    orc.kv_append(code, orc.BF16, W.bits16(kn), W.bits16(vn), slots, kc, vc,
                  scale_mode=orc.SCALE_PER_TOKEN, k_new_scale=kt, v_new_scale=vt,
                  k_scales=ks_arr, v_scales=vs_arr)
    assert np.array_equal(ks_arr.reshape(P * BS, H)[rows], kt[real])
    assert np.array_equal(vs_arr.reshape(P * BS, H)[rows], vt[real])
    for cache, src, sc in ((kc, kn, kt), (vc, vn, vt)):
        x = src[torch.from_numpy(real)].float() / torch.from_numpy(sc[real])[:, :, None]
        assert np.array_equal(cache.reshape(P * BS, H, D)[rows], cast(x))
    # equal-valued granular scales == per-head scales
    hs = np.array([0.01, 0.004, 0.02], np.float32)
    ref_k, ref_v = np.zeros((P, BS, H, D), dt), np.zeros((P, BS, H, D), dt)
    orc.kv_append(code, orc.BF16, W.bits16(kn), W.bits16(vn), slots, ref_k, ref_v, hs, hs)
    kc, vc = np.zeros((P, BS, H, D), dt), np.zeros((P, BS, H, D), dt)
    orc.kv_append(code, orc.BF16, W.bits16(kn), W.bits16(vn), slots, kc, vc,
                  scale_mode=orc.SCALE_PER_BLOCK, k_scales=np.tile(hs, (P, 1)),
                  v_scales=np.tile(hs, (P, 1)))
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)
