"""The x-vectorised paged layout [num_blocks, num_kv_heads, head_dim // x,
block_size, x] (x = 16 bytes / element size; "Write Triton Kv Cache Append
Kernel", "Inputs the agent should gather first" item 1): append bit-exact
with the oracle's scatter laid out by oracle.to_xvec, decode within the
output tolerance of the fp64 oracle, through the persistent kernel (its XV
instances) and the general one."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import pipeline as PL
from tests.test_gpu_decode import _check, _sample_pairs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_num_gb300 as P
    P.lib()
    return P


def _x(kind):
    return 8 if kind in ("f16", "bf16") else 16


def _same_storage(w, orc, cache, oc):
    got = PL.gpu_cache_host(cache)
    x = _x(w.cache_kind)
    for n in ("k_cache", "v_cache"):
        want = orc.to_xvec(oc[n], x)
        assert got[n].shape == want.shape
        assert np.array_equal(got[n], want), n


def _as_f16(w):
    w.dtype = torch.float16
    w.cache_kind = "f16"
    for name in ("q", "k_cache0", "v_cache0", "k_new", "v_new"):
        setattr(w, name, getattr(w, name).to(torch.float16))
    return w


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("bs,d,kind", [(16, 128, "bf16"), (32, 128, "bf16"), (64, 128, "bf16"),
                                       (16, 64, "f16"), (32, 64, "bf16")])
def test_xvec_16bit(pkv, orc, bs, d, kind, splits):
    w = W.gqa_bf16(batch=5, ctx_lo=1, ctx_hi=11 * bs + 3, num_heads=16, num_kv_heads=4, head_dim=d,
                   block_size=bs, seed=200 + bs + d, layout="xvec")
    if kind == "f16":
        w = _as_f16(w)
    cache, out = PL.gpu_run(w, pkv, num_splits=splits)
    oc = PL.oracle_caches(w, orc)
    _same_storage(w, orc, cache, oc)
    _check(w, out, PL.oracle_decode(w, orc, oc))


@pytest.mark.parametrize("splits", [0, 2])
@pytest.mark.parametrize("kind,bs", [("e4m3", 32), ("e4m3", 16), ("e5m2", 64), ("i8", 32)])
def test_xvec_one_byte(pkv, orc, kind, bs, splits):
    w = W.fp8_long(batch=4, ctx_lo=20, ctx_hi=900, calib_tokens=64, block_size=bs,
                   seed=210 + bs + len(kind), fp8=kind, layout="xvec")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache, out = PL.gpu_run(w, pkv, num_splits=splits, err_flag=err)
    assert int(err.item()) == 0
    oc = PL.oracle_caches(w, orc)
    _same_storage(w, orc, cache, oc)
    _check(w, out, PL.oracle_decode(w, orc, oc))


@pytest.mark.parametrize("scales", ["block", "token"])
def test_xvec_granular_scales(pkv, orc, scales):
    """Per-block / per-token scales on an x-vectorised cache (general kernel)."""
    w = W.fp8_long(batch=3, ctx_lo=20, ctx_hi=500, calib_tokens=64, seed=220 + len(scales),
                   scales=scales, layout="xvec")
    cache, out = PL.gpu_run(w, pkv)
    oc = PL.oracle_caches(w, orc)
    _same_storage(w, orc, cache, oc)
    _check(w, out, PL.oracle_decode(w, orc, oc))


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_xvec_unaligned_sources(pkv, orc, kind):
    """New rows whose strides are not 16-byte multiples take the element-wise
    append kernels; the stored pieces are the same."""
    if kind == "bf16":
        w = W.gqa_bf16(batch=4, ctx_lo=30, ctx_hi=300, seed=230, layout="xvec")
    else:
        w = W.fp8_long(batch=3, ctx_lo=30, ctx_hi=300, calib_tokens=64, seed=231, layout="xvec")
    T, H, D = w.k_new.shape
    for name in ("k_new", "v_new") + (("k_fill", "v_fill") if w.k_fill is not None else ()):
        t = getattr(w, name)
        buf = torch.zeros((t.shape[0], H, D + 1), dtype=t.dtype)
        buf[:, :, 1:] = t
        setattr(w, name, buf[:, :, 1:])        # 2-byte offset, odd strides
    cache, _ = PL.gpu_run(w, pkv, decode=False)
    _same_storage(w, orc, cache, PL.oracle_caches(w, orc))


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_xvec_matches_flash_layout_bitwise(pkv, kind):
    """Same data, two storage layouts: the persistent kernel's flash and XV
    instances run the same products in the same order."""
    outs = []
    for layout in ("flash", "xvec"):
        if kind == "bf16":
            w = W.gqa_bf16(batch=6, ctx_lo=1, ctx_hi=2000, seed=240, layout=layout)
        else:
            w = W.fp8_long(batch=4, ctx_lo=100, ctx_hi=3000, calib_tokens=64, seed=241, layout=layout)
        outs.append(PL.gpu_run(w, pkv)[1].cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_full_gqa_bf16_xvec(pkv, orc):
    """Full-size Llama-3-8B-like GQA step (batch 64, contexts 512..4096) in
    the x-vectorised layout: every stored byte (storage order) and every
    output row against the oracle."""
    from tests.test_gpu_decode import _full_size
    _full_size(W.gqa_bf16(layout="xvec"), pkv, orc, paths=("step",))


def test_full_fp8_long_xvec(pkv, orc):
    """Full-size long-context e4m3 step (batch 16, contexts 16K..32K) in the
    x-vectorised layout: every stored byte and every output row."""
    from tests.test_gpu_decode import _full_size
    _full_size(W.fp8_long(layout="xvec"), pkv, orc, paths=("step",))


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_xvec_padded_pieces(pkv, orc, kind):
    """Pieces further apart than block_size * 16 bytes (slots padded): the
    persistent kernel then stages tiles with 5-D tensor copies instead of one
    bulk copy per head group; append and decode match the oracle."""
    if kind == "bf16":
        w = W.gqa_bf16(batch=4, ctx_lo=1, ctx_hi=900, seed=250, layout="xvec")
    else:
        w = W.fp8_long(batch=3, ctx_lo=50, ctx_hi=900, calib_tokens=64, seed=251, layout="xvec")
    P, BS, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    x = _x(kind)
    dt = torch.bfloat16 if kind == "bf16" else torch.uint8
    pad_k = torch.zeros((P, H, D // x, BS + 16, x), dtype=dt, device="cuda")
    pad_v = torch.zeros_like(pad_k)
    cache = pkv.KVCache(w.cache_kind, pad_k[:, :, :, :BS], pad_v[:, :, :, :BS],
                        k_scale=None if w.k_scale is None else w.k_scale.cuda(),
                        v_scale=None if w.v_scale is None else w.v_scale.cuda(), layout="xvec")
    if w.k_cache0 is not None:
        cache.k_cache.copy_(W.storage(w.k_cache0, "xvec").cuda())
        cache.v_cache.copy_(W.storage(w.v_cache0, "xvec").cuda())
    bt = w.block_tables.cuda()
    if w.fill_req is not None:
        sm = pkv.slot_mapping(bt, w.fill_req.cuda(), w.fill_pos.cuda(), BS)
        pkv.kv_append(w.k_fill.cuda(), w.v_fill.cuda(), sm, cache)
    sm = pkv.slot_mapping(bt, w.new_req.cuda(), w.new_pos.cuda(), BS)
    pkv.kv_append(w.k_new.cuda(), w.v_new.cuda(), sm, cache)
    out = pkv.paged_decode(w.q.cuda(), cache, bt, w.context_lens.cuda(), sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    oc = PL.oracle_caches(w, orc)
    _same_storage(w, orc, cache, oc)
    _check(w, out, PL.oracle_decode(w, orc, oc))
    # the padding slots were never written
    assert not pad_k[:, :, :, BS:].view(torch.uint8).any()
    _, packed = PL.gpu_run(w, pkv)
    assert torch.equal(out.cpu().view(torch.int16), packed.cpu().view(torch.int16))
