"""Pins for the oracle's paged decode ("10. Triton KV Cache and
PagedAttention": Step 1 layout, Step 4 gather reference, reference-code
TODO 1-5), in fp64: brute force against a torch float64 gather + softmax,
closed-form special cases, and invariants.  CPU only."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from tests.refs import e4m3_dequant, e5m2_dequant, gather_attention, u3_dequant


def _decode16(orc, w, q=None, kc=None, vc=None, bt=None, ctx=None, pairs=None):
    code = orc.F16 if w.dtype == torch.float16 else orc.BF16
    q = W.bits16(w.q) if q is None else q
    kc = W.bits16(w.k_cache0) if kc is None else kc
    vc = W.bits16(w.v_cache0) if vc is None else vc
    bt = w.block_tables.numpy() if bt is None else bt
    ctx = w.context_lens.numpy() if ctx is None else ctx
    out, bad = orc.paged_decode(code, code, q, kc, vc, bt, ctx, w.block_size, w.sm_scale,
                                pairs=pairs)
    assert bad == 0
    return out


def _as_f64(bits, dt):
    return torch.from_numpy(bits.view(np.int16)).view(dt).to(torch.float64).numpy()


@pytest.mark.parametrize("literal", [False, True])
def test_tiny_matches_torch_gather(orc, literal):
    w = W.tiny(literal=literal)
    out = _decode16(orc, w)
    ref = gather_attention(w.q, w.k_cache0, w.v_cache0, w.block_tables.numpy(),
                           w.context_lens.numpy(), w.block_size, w.sm_scale)
    assert np.max(np.abs(out - ref)) < 1e-12


@pytest.mark.parametrize("G,BS,D", [(1, 16, 64), (4, 16, 128), (8, 32, 128), (2, 8, 32)])
def test_gqa_matches_torch_gather(orc, G, BS, D):
    w = W.gqa_bf16(batch=3, ctx_lo=1, ctx_hi=5 * BS + 3, num_kv_heads=2, num_heads=2 * G,
                   head_dim=D, block_size=BS, seed=100 + G)
    out = _decode16(orc, w)
    ref = gather_attention(w.q, w.k_cache0, w.v_cache0, w.block_tables.numpy(),
                           w.context_lens.numpy(), w.block_size, w.sm_scale)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_context_one_returns_first_value(orc):
    w = W.gqa_bf16(batch=2, ctx_lo=1, ctx_hi=1, seed=7, num_heads=8, num_kv_heads=2)
    out = _decode16(orc, w)
    v = _as_f64(W.bits16(w.v_cache0), torch.bfloat16)
    for b in range(2):
        blk = int(w.block_tables[b, 0])
        for h in range(8):
            assert np.array_equal(out[b, h], v[blk, 0, h // 4])


def test_zero_query_gives_mean_of_values(orc):
    w = W.gqa_bf16(batch=2, ctx_lo=20, ctx_hi=70, seed=8, num_heads=4, num_kv_heads=2)
    q = np.zeros_like(W.bits16(w.q))
    out = _decode16(orc, w, q=q)
    v = _as_f64(W.bits16(w.v_cache0), torch.bfloat16)
    for b in range(2):
        n = int(w.context_lens[b])
        rows = [v[int(w.block_tables[b, t // w.block_size]), t % w.block_size] for t in range(n)]
        mean = np.mean(np.stack(rows), axis=0)          # [Hkv, D]
        for h in range(4):
            assert np.allclose(out[b, h], mean[h // 2], rtol=0, atol=1e-12)


def test_dominant_score_selects_its_value(orc):
    """q parallel to one key with a huge norm: the output is that key's value."""
    w = W.gqa_bf16(batch=1, ctx_lo=50, ctx_hi=50, seed=9, num_heads=2, num_kv_heads=1,
                   head_dim=64)
    k = _as_f64(W.bits16(w.k_cache0), torch.bfloat16)
    v = _as_f64(W.bits16(w.v_cache0), torch.bfloat16)
    t_star = 37
    blk = int(w.block_tables[0, t_star // w.block_size])
    kstar = k[blk, t_star % w.block_size, 0]
    q = torch.from_numpy(kstar * 64.0).to(torch.bfloat16)[None, None, :].repeat(1, 2, 1)
    out = _decode16(orc, w, q=W.bits16(q))
    assert np.allclose(out[0, 0], v[blk, t_star % w.block_size, 0], atol=1e-9)


def test_empty_context_gives_zero(orc):
    w = W.gqa_bf16(batch=3, ctx_lo=5, ctx_hi=40, seed=10, num_heads=4, num_kv_heads=2)
    ctx = w.context_lens.numpy().copy()
    ctx[1] = 0
    out = _decode16(orc, w, ctx=ctx)
    assert np.all(out[1] == 0)
    full = _decode16(orc, w)
    assert np.array_equal(out[0], full[0]) and np.array_equal(out[2], full[2])


def test_block_permutation_invariance(orc):
    """Moving physical blocks and rewriting the table leaves the output."""
    w = W.gqa_bf16(batch=3, ctx_lo=30, ctx_hi=90, seed=11, num_heads=4, num_kv_heads=2)
    base = _decode16(orc, w)
    P = w.num_blocks
    perm = np.random.default_rng(0).permutation(P)
    # old block i moves to position perm[i]; the table follows it
    bt = perm[w.block_tables.numpy()].astype(np.int32)
    kc2 = np.empty_like(W.bits16(w.k_cache0))
    vc2 = np.empty_like(W.bits16(w.v_cache0))
    kc2[perm] = W.bits16(w.k_cache0)
    vc2[perm] = W.bits16(w.v_cache0)
    out = _decode16(orc, w, kc=kc2, vc=vc2, bt=bt)
    assert np.array_equal(out, base)


def test_poison_beyond_context_is_ignored(orc):
    w = W.gqa_bf16(batch=3, ctx_lo=17, ctx_hi=60, seed=12, num_heads=4, num_kv_heads=2)
    base = _decode16(orc, w)
    kc, vc = W.bits16(w.k_cache0).copy(), W.bits16(w.v_cache0).copy()
    live = np.zeros((w.num_blocks, w.block_size), bool)
    for b in range(w.batch):
        for t in range(int(w.context_lens[b])):
            live[int(w.block_tables[b, t // w.block_size]), t % w.block_size] = True
    kc[~live] = 0x7FC0   # bf16 NaN
    vc[~live] = 0x7FC0
    out = _decode16(orc, w, kc=kc, vc=vc)
    assert np.array_equal(out, base)


def test_pairs_subset_equals_full(orc):
    w = W.gqa_bf16(batch=4, ctx_lo=10, ctx_hi=50, seed=13, num_heads=8, num_kv_heads=2)
    full = _decode16(orc, w)
    pairs = np.array([0, 5, 13, 31], np.int32)
    part = _decode16(orc, w, pairs=pairs)
    flat = part.reshape(-1, w.head_dim)
    assert np.array_equal(flat[pairs], full.reshape(-1, w.head_dim)[pairs])
    others = np.setdiff1d(np.arange(32), pairs)
    assert np.isnan(flat[others]).all()


def _fill_quantised(orc, w, code):
    """Fill a quantised cache with the oracle's append (context + new)."""
    P, BS, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    src_code = orc.F16 if w.dtype == torch.float16 else orc.BF16
    req = np.concatenate([w.fill_req.numpy(), w.new_req.numpy()])
    pos = np.concatenate([w.fill_pos.numpy(), w.new_pos.numpy()])
    kn = np.concatenate([W.bits16(w.k_fill), W.bits16(w.k_new)])
    vn = np.concatenate([W.bits16(w.v_fill), W.bits16(w.v_new)])
    slots = orc.build_slot_mapping(w.block_tables.numpy(), req, pos, BS)
    c = {}
    if code in (orc.E4M3, orc.E5M2, orc.I8):
        dt = np.int8 if code == orc.I8 else np.uint8
        c["k"] = np.zeros((P, BS, H, D), dt)
        c["v"] = np.zeros((P, BS, H, D), dt)
        orc.kv_append(code, src_code, kn, vn, slots, c["k"], c["v"], w.k_scale.numpy(),
                      w.v_scale.numpy())
    else:
        RB = 3 * D // 8
        c["k"] = np.zeros((P, BS, H, RB), np.uint8)
        c["v"] = np.zeros((P, BS, H, RB), np.uint8)
        for n in ("ks", "vs"):
            c[n] = np.zeros((P, BS, H), np.uint16)
        for n in ("kz", "vz"):
            c[n] = np.zeros((P, BS, H), np.uint8)
        orc.kv_append(code, src_code, kn, vn, slots, c["k"], c["v"], k_qscale=c["ks"],
                      k_qzero=c["kz"], v_qscale=c["vs"], v_qzero=c["vz"])
    return c


def test_fp8_decode_on_dequantised_cache(orc):
    w = W.fp8_long(batch=3, ctx_lo=40, ctx_hi=150, calib_tokens=64, seed=14)
    c = _fill_quantised(orc, w, orc.E4M3)
    out, bad = orc.paged_decode(orc.E4M3, orc.BF16, W.bits16(w.q), c["k"], c["v"],
                                w.block_tables.numpy(), w.context_lens.numpy(), w.block_size,
                                w.sm_scale, k_scale=w.k_scale.numpy(), v_scale=w.v_scale.numpy())
    assert bad == 0
    kd = e4m3_dequant(c["k"], w.k_scale.numpy())
    vd = e4m3_dequant(c["v"], w.v_scale.numpy())
    ref = gather_attention(w.q, kd, vd, w.block_tables.numpy(), w.context_lens.numpy(),
                           w.block_size, w.sm_scale)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_e5m2_decode_on_dequantised_cache(orc):
    w = W.fp8_long(batch=3, ctx_lo=40, ctx_hi=150, calib_tokens=64, seed=16, fp8="e5m2")
    c = _fill_quantised(orc, w, orc.E5M2)
    out, bad = orc.paged_decode(orc.E5M2, orc.BF16, W.bits16(w.q), c["k"], c["v"],
                                w.block_tables.numpy(), w.context_lens.numpy(), w.block_size,
                                w.sm_scale, k_scale=w.k_scale.numpy(), v_scale=w.v_scale.numpy())
    assert bad == 0
    kd = e5m2_dequant(c["k"], w.k_scale.numpy())
    vd = e5m2_dequant(c["v"], w.v_scale.numpy())
    ref = gather_attention(w.q, kd, vd, w.block_tables.numpy(), w.context_lens.numpy(),
                           w.block_size, w.sm_scale)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_i8_decode_on_dequantised_cache(orc):
    w = W.fp8_long(batch=3, ctx_lo=40, ctx_hi=150, calib_tokens=64, seed=17, fp8="i8")
    c = _fill_quantised(orc, w, orc.I8)
    out, bad = orc.paged_decode(orc.I8, orc.BF16, W.bits16(w.q), c["k"], c["v"],
                                w.block_tables.numpy(), w.context_lens.numpy(), w.block_size,
                                w.sm_scale, k_scale=w.k_scale.numpy(), v_scale=w.v_scale.numpy())
    assert bad == 0
    kd = c["k"].astype(np.float64) * w.k_scale.numpy().astype(np.float64)[:, None]
    vd = c["v"].astype(np.float64) * w.v_scale.numpy().astype(np.float64)[:, None]
    ref = gather_attention(w.q, kd, vd, w.block_tables.numpy(), w.context_lens.numpy(),
                           w.block_size, w.sm_scale)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_u3_decode_on_dequantised_cache(orc):
    w = W.u3_mha(batch=3, ctx_lo=20, ctx_hi=100, num_heads=4, seed=15)
    c = _fill_quantised(orc, w, orc.U3)
    out, bad = orc.paged_decode(orc.U3, orc.F16, W.bits16(w.q), c["k"], c["v"],
                                w.block_tables.numpy(), w.context_lens.numpy(), w.block_size,
                                w.sm_scale, k_qscale=c["ks"], k_qzero=c["kz"],
                                v_qscale=c["vs"], v_qzero=c["vz"])
    assert bad == 0
    kd = u3_dequant(c["k"], c["ks"], c["kz"], w.head_dim)
    vd = u3_dequant(c["v"], c["vs"], c["vz"], w.head_dim)
    ref = gather_attention(w.q, kd, vd, w.block_tables.numpy(), w.context_lens.numpy(),
                           w.block_size, w.sm_scale)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_appended_token_is_attended_at_last_position(orc):
    """After appending at position context_len-1 through the slot mapping,
    the decode's last attended token is the new row (context_lens counts it)."""
    w = W.tiny()
    kc, vc = W.bits16(w.k_cache0).copy(), W.bits16(w.v_cache0).copy()
    slots = orc.build_slot_mapping(w.block_tables.numpy(), w.new_req.numpy(),
                                   w.new_pos.numpy(), w.block_size)
    orc.kv_append(orc.F16, orc.F16, W.bits16(w.k_new), W.bits16(w.v_new), slots, kc, vc)
    for b in range(w.batch):
        t = int(w.context_lens[b]) - 1
        blk = int(w.block_tables[b, t // w.block_size])
        assert np.array_equal(kc[blk, t % w.block_size], W.bits16(w.k_new)[b])
    # a query equal to a scaled copy of the new key attends mostly to it
    out = _decode16(orc, w, kc=kc, vc=vc)
    ref = gather_attention(torch.from_numpy(W.bits16(w.q).view(np.float16)),
                           torch.from_numpy(kc.view(np.float16)),
                           torch.from_numpy(vc.view(np.float16)), w.block_tables.numpy(),
                           w.context_lens.numpy(), w.block_size, w.sm_scale)
    assert np.max(np.abs(out - ref)) < 1e-12


@pytest.mark.parametrize("mode", ["block", "token"])
def test_granular_scale_decode_on_dequantised_cache(orc, mode):
    """fp8 decode with per-block or per-token scales equals fp64 attention
    on the cache dequantised independently with each row's own scale."""
    w = W.fp8_long(batch=3, ctx_lo=40, ctx_hi=150, calib_tokens=64, seed=18)
    P, BS, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    g = np.random.default_rng(19)
    req = np.concatenate([w.fill_req.numpy(), w.new_req.numpy()])
    pos = np.concatenate([w.fill_pos.numpy(), w.new_pos.numpy()])
    kn = np.concatenate([W.bits16(w.k_fill), W.bits16(w.k_new)])
    vn = np.concatenate([W.bits16(w.v_fill), W.bits16(w.v_new)])
    slots = orc.build_slot_mapping(w.block_tables.numpy(), req, pos, BS)
    kc, vc = np.zeros((P, BS, H, D), np.uint8), np.zeros((P, BS, H, D), np.uint8)
    if mode == "block":
        ks = (g.random((P, H)) * 0.01 + 0.003).astype(np.float32)
        vs = (g.random((P, H)) * 0.01 + 0.003).astype(np.float32)
        orc.kv_append(orc.E4M3, orc.BF16, kn, vn, slots, kc, vc, scale_mode=orc.SCALE_PER_BLOCK,
                      k_scales=ks, v_scales=vs)
        krow = np.repeat(ks[:, None, :], BS, axis=1)          # [P, BS, H]
        vrow = np.repeat(vs[:, None, :], BS, axis=1)
        sm = orc.SCALE_PER_BLOCK
    else:
        T = len(slots)
        ks = np.zeros((P, BS, H), np.float32)
        vs = np.zeros((P, BS, H), np.float32)
        kt = (g.random((T, H)) * 0.01 + 0.003).astype(np.float32)
        vt = (g.random((T, H)) * 0.01 + 0.003).astype(np.float32)
        orc.kv_append(orc.E4M3, orc.BF16, kn, vn, slots, kc, vc, scale_mode=orc.SCALE_PER_TOKEN,
                      k_new_scale=kt, v_new_scale=vt, k_scales=ks, v_scales=vs)
        krow, vrow = ks, vs
        sm = orc.SCALE_PER_TOKEN
    out, bad = orc.paged_decode(orc.E4M3, orc.BF16, W.bits16(w.q), kc, vc, w.block_tables.numpy(),
                                w.context_lens.numpy(), BS, w.sm_scale, scale_mode=sm,
                                k_scales=ks, v_scales=vs)
    assert bad == 0
    one = np.ones(H)
    kd = e4m3_dequant(kc, one) * krow[..., None].astype(np.float64)
    vd = e4m3_dequant(vc, one) * vrow[..., None].astype(np.float64)
    ref = gather_attention(w.q, kd, vd, w.block_tables.numpy(), w.context_lens.numpy(), BS,
                           w.sm_scale)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_scale_edges_zero_and_negative(orc):
    """sm_scale 0: uniform weights, each row the mean of its V rows;
    sm_scale -s: the same as +s on the negated query (softmax of -q.k),
    which is how a negative scale must be read.  Both against the gather
    reference at the same scale."""
    w = W.gqa_bf16(batch=3, ctx_lo=1, ctx_hi=70, seed=12, num_heads=4, num_kv_heads=2, head_dim=64)
    v = _as_f64(W.bits16(w.v_cache0), torch.bfloat16)
    w.sm_scale = 0.0
    out0 = _decode16(orc, w)
    for b in range(3):
        n = int(w.context_lens[b])
        rows = [v[int(w.block_tables[b, t // w.block_size]), t % w.block_size] for t in range(n)]
        mean = np.mean(np.stack(rows), axis=0)
        for h in range(4):
            assert np.allclose(out0[b, h], mean[h // 2], rtol=0, atol=1e-12)
    s = 0.125
    w.sm_scale = -s
    neg = _decode16(orc, w)
    w.sm_scale = s
    flipped = _decode16(orc, w, q=W.bits16(w.q) ^ np.uint16(0x8000))
    assert np.max(np.abs(neg - flipped)) < 1e-12
    w.sm_scale = -s
    ref = gather_attention(w.q, w.k_cache0, w.v_cache0, w.block_tables.numpy(),
                           w.context_lens.numpy(), w.block_size, w.sm_scale)
    assert np.max(np.abs(neg - ref)) < 1e-12
