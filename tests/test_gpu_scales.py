"""Scale granularities of fp8 / int8 caches on the GPU: per-block scales
([num_blocks, Hkv], given with the cache) and per-token scales (given with
each new token, stored at its slot), through kv_append / kv_append_scaled
and paged_decode, against the oracle: appended codes and stored scales bit
exact, decode within the fp64 tolerance."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import pipeline as PL
from tests.test_gpu_decode import _check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_num_gb300 as P
    P.lib()
    return P


def _tokens(w):
    req = torch.cat([w.fill_req, w.new_req])
    pos = torch.cat([w.fill_pos, w.new_pos])
    kn = torch.cat([w.k_fill, w.k_new])
    vn = torch.cat([w.v_fill, w.v_new])
    return req, pos, kn, vn


@pytest.mark.parametrize("splits", [0, 2])
@pytest.mark.parametrize("kind", ["e4m3", "i8"])
@pytest.mark.parametrize("mode", ["block", "token"])
def test_granular_scales_append_and_decode(pkv, orc, kind, mode, splits):
    """splits 0: the persistent kernel, which stages each block's scales
    with the K/V tiles; splits 2: the general kernel."""
    w = W.fp8_long(batch=4, ctx_lo=30, ctx_hi=600, calib_tokens=64, seed=99, fp8=kind)
    P, BS, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    fmax = 448.0 if kind == "e4m3" else 127.0
    g = torch.Generator().manual_seed(100)
    req, pos, kn, vn = _tokens(w)
    T = req.shape[0]
    dev = "cuda"
    if mode == "block":
        kb = (torch.rand((P, H), generator=g) * 3 + 2) / fmax       # blocks' scales
        vb = (torch.rand((P, H), generator=g) * 3 + 2) / fmax
        cache = pkv.KVCache.allocate(kind, P, BS, H, D, device=dev, fill=0, scale_mode="block",
                                     k_scales=kb.to(dev), v_scales=vb.to(dev))
    else:
        kt = (torch.rand((T, H), generator=g) * 3 + 2) / fmax       # tokens' scales
        vt = (torch.rand((T, H), generator=g) * 3 + 2) / fmax
        cache = pkv.KVCache.allocate(kind, P, BS, H, D, device=dev, fill=0, scale_mode="token")
    bt = w.block_tables.to(dev)
    slots = pkv.slot_mapping(bt, req.to(dev), pos.to(dev), BS)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if mode == "block":
        pkv.kv_append(kn.to(dev), vn.to(dev), slots, cache, err_flag=err)
    else:
        with pytest.raises(pkv.PkvError):        # the plain append refuses a per-token cache
            pkv.kv_append(kn.to(dev), vn.to(dev), slots, cache)
        pkv.kv_append_scaled(kn.to(dev), vn.to(dev), kt.to(dev), vt.to(dev), slots, cache,
                             err_flag=err)
    out = pkv.paged_decode(w.q.to(dev), cache, bt, w.context_lens.to(dev), sm_scale=w.sm_scale,
                           num_splits=splits, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # oracle
    code = PL.KIND_CODE_ORACLE[kind]
    dt = np.int8 if kind == "i8" else np.uint8
    kc, vc = np.zeros((P, BS, H, D), dt), np.zeros((P, BS, H, D), dt)
    sl = orc.build_slot_mapping(w.block_tables.numpy(), req.numpy(), pos.numpy(), BS)
    if mode == "block":
        ks_o, vs_o = kb.numpy(), vb.numpy()
        orc.kv_append(code, orc.BF16, W.bits16(kn), W.bits16(vn), sl, kc, vc,
                      scale_mode=orc.SCALE_PER_BLOCK, k_scales=ks_o, v_scales=vs_o)
        sm = orc.SCALE_PER_BLOCK
    else:
        ks_o, vs_o = np.ones((P, BS, H), np.float32), np.ones((P, BS, H), np.float32)
        orc.kv_append(code, orc.BF16, W.bits16(kn), W.bits16(vn), sl, kc, vc,
                      scale_mode=orc.SCALE_PER_TOKEN, k_new_scale=kt.numpy(),
                      v_new_scale=vt.numpy(), k_scales=ks_o, v_scales=vs_o)
        assert np.array_equal(cache.k_scales.cpu().contiguous().numpy(), ks_o)
        assert np.array_equal(cache.v_scales.cpu().contiguous().numpy(), vs_o)
        sm = orc.SCALE_PER_TOKEN
    assert np.array_equal(cache.k_cache.cpu().numpy(), kc)
    assert np.array_equal(cache.v_cache.cpu().numpy(), vc)
    ref, bad = orc.paged_decode(code, orc.BF16, W.bits16(w.q), kc, vc, w.block_tables.numpy(),
                                w.context_lens.numpy(), BS, w.sm_scale, scale_mode=sm,
                                k_scales=ks_o, v_scales=vs_o, nthreads=orc.max_threads())
    assert bad == 0
    _check(w, out, ref)


def test_slot_major_token_scales_take_the_general_kernel(pkv, orc):
    """Per-token scales stored slot-major (contiguous [num_blocks,
    block_size, Hkv]) are not one run per head: decode runs the general
    kernel and still matches the head-major (persistent kernel) result."""
    w = W.fp8_long(batch=3, ctx_lo=30, ctx_hi=400, calib_tokens=64, seed=101)
    P, BS, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    g = torch.Generator().manual_seed(102)
    req, pos, kn, vn = _tokens(w)
    kt = (torch.rand((req.shape[0], H), generator=g) + 1) / 200
    vt = (torch.rand((req.shape[0], H), generator=g) + 1) / 200
    dev = "cuda"
    bt = w.block_tables.to(dev)
    outs = []
    for slot_major in (False, True):
        cache = pkv.KVCache.allocate("e4m3", P, BS, H, D, device=dev, fill=0, scale_mode="token")
        if slot_major:
            cache.k_scales = torch.ones((P, BS, H), dtype=torch.float32, device=dev)
            cache.v_scales = torch.ones((P, BS, H), dtype=torch.float32, device=dev)
        slots = pkv.slot_mapping(bt, req.to(dev), pos.to(dev), BS)
        pkv.kv_append_scaled(kn.to(dev), vn.to(dev), kt.to(dev), vt.to(dev), slots, cache)
        outs.append(pkv.paged_decode(w.q.to(dev), cache, bt, w.context_lens.to(dev),
                                     sm_scale=w.sm_scale))
    torch.cuda.synchronize()
    a, b = PL.out_f64(outs[0]), PL.out_f64(outs[1])
    assert np.max(np.abs(a - b)) <= PL.tolerance(w)


@pytest.mark.parametrize("scales", ["token", "block"])
def test_full_fp8_long_granular(pkv, orc, scales):
    """The long-context shape with per-token (each row's amax / 448) or
    per-block scales, through the persistent kernel: every cache byte and
    every output row against the oracle (per-token scales through the
    separate calls, which carry them; per-block through pkv_decode_step)."""
    from tests.test_gpu_decode import _full_size
    name = "fp8_long_%s_scales" % scales
    w = W.fp8_long(seed=W.SEEDS[name], scales=scales)
    _full_size(w, pkv, orc, paths=("calls",) if scales == "token" else ("step",))
