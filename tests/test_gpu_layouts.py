"""Cache layouts beyond the default paged one, through the same C ABI:
a contiguous per-request cache [batch, kv_heads, max_seq_len, D] for the
append (one block of max_seq_len slots per request), the dual-stacked paged
layout [num_blocks, 2, kv_heads, block_size, D] for append + decode, and the
MHA short-context benchmark shape of "10. Triton KV Cache and
PagedAttention" (fp16, contiguously allocated blocks)."""
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


def _contiguous_cache(pkv, kind, batch, Hkv, msl, D, k_scale=None, v_scale=None):
    """A [batch, Hkv, max_seq_len, row] buffer seen as [batch, msl, Hkv, row]."""
    dev = "cuda"
    row = 3 * D // 8 if kind == "u3" else D
    dt = {"bf16": torch.bfloat16, "f16": torch.float16, "e4m3": torch.uint8, "u3": torch.uint8}[kind]
    phys_k = torch.zeros((batch, Hkv, msl, row), dtype=dt, device=dev)
    phys_v = torch.zeros_like(phys_k)
    c = pkv.KVCache(kind, phys_k.permute(0, 2, 1, 3), phys_v.permute(0, 2, 1, 3),
                    k_scale=k_scale, v_scale=v_scale)
    if kind == "u3":
        def meta(t):
            return torch.zeros((batch, Hkv, msl), dtype=t, device=dev).permute(0, 2, 1)
        c.k_qscale, c.k_qzero = meta(torch.float16), meta(torch.uint8)
        c.v_qscale, c.v_qzero = meta(torch.float16), meta(torch.uint8)
    return c, phys_k, phys_v


@pytest.mark.parametrize("kind,msl", [("bf16", 1000), ("bf16", 512), ("e4m3", 1000), ("u3", 777)])
def test_contiguous_cache_append(pkv, orc, kind, msl):
    """slot = req * max_seq_len + pos into a contiguous per-request cache:
    bit-exact with the oracle's scatter, padding tokens write nothing."""
    g = torch.Generator().manual_seed(msl + len(kind))
    B, Hkv, D = 3, 4, 128
    req = [0] * 50 + [1] + [2] * 7 + [1, 0]
    pos = list(range(50)) + [msl - 1] + sorted(torch.randperm(msl, generator=g)[:7].tolist()) + [-1, -1]
    T = len(req)
    src_dt = torch.float16 if kind == "u3" else torch.bfloat16
    kn = torch.randn((T, Hkv, D), generator=g).to(src_dt)
    vn = torch.randn((T, Hkv, D), generator=g).to(src_dt)
    ks = vs = None
    if kind == "e4m3":
        ks = (torch.rand(Hkv, generator=g) * 0.02 + 0.005).float()
        vs = (torch.rand(Hkv, generator=g) * 0.02 + 0.005).float()
    slots = torch.tensor([r * msl + p if p >= 0 else -1 for r, p in zip(req, pos)], dtype=torch.int64)
    c, pk, pv = _contiguous_cache(pkv, kind, B, Hkv, msl, D,
                                  None if ks is None else ks.cuda(), None if vs is None else vs.cuda())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.kv_append(kn.cuda(), vn.cuda(), slots.cuda(), c, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # oracle: the same scatter into logical [batch, msl, Hkv, row] arrays
    row = 3 * D // 8 if kind == "u3" else D
    code = PL.KIND_CODE_ORACLE[kind]
    npdt = np.uint16 if kind == "bf16" else np.uint8
    ok_, ov_ = np.zeros((B, msl, Hkv, row), npdt), np.zeros((B, msl, Hkv, row), npdt)
    meta = {}
    if kind == "u3":
        meta = {n: np.zeros((B, msl, Hkv), np.uint16 if "scale" in n else np.uint8)
                for n in ("k_qscale", "k_qzero", "v_qscale", "v_qzero")}
    bad = orc.kv_append(code, 1 if src_dt == torch.float16 else 2, W.bits16(kn), W.bits16(vn),
                        slots.numpy(), ok_, ov_, None if ks is None else ks.numpy(),
                        None if vs is None else vs.numpy(), meta.get("k_qscale"), meta.get("k_qzero"),
                        meta.get("v_qscale"), meta.get("v_qzero"))
    assert bad == 0
    got = PL.gpu_cache_host(c)
    assert np.array_equal(got["k_cache"], ok_) and np.array_equal(got["v_cache"], ov_)
    for n, a in meta.items():
        assert np.array_equal(got[n], a), n
    # and the physical buffer is the [batch, Hkv, msl, row] layout
    phys = pk.cpu().contiguous()
    phys = phys.view(torch.int16).numpy().view(np.uint16) if phys.element_size() == 2 else phys.numpy()
    assert np.array_equal(phys, ok_.transpose(0, 2, 1, 3))


def test_contiguous_cache_rejected_by_decode(pkv):
    """Decode still needs a power-of-two block size: a 1000-slot request
    block is refused at the boundary, not mis-read."""
    c, _, _ = _contiguous_cache(pkv, "bf16", 2, 4, 1000, 128)
    q = torch.zeros((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.tensor([[0], [1]], dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError):
        pkv.decode_workspace_bytes(q, c, bt)


@pytest.mark.parametrize("splits", [0, 3])
def test_dual_stacked_layout(pkv, orc, splits):
    """K and V as the two halves of one [num_blocks, 2, kv_heads, block_size,
    D] buffer: append and decode through the strided views match the oracle."""
    w = W.gqa_bf16(batch=5, ctx_lo=20, ctx_hi=600, seed=96)
    P, BS, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    buf = torch.empty((P, 2, H, BS, D), dtype=torch.bfloat16, device="cuda")
    kview = buf[:, 0].permute(0, 2, 1, 3)          # [P, BS, H, D]
    vview = buf[:, 1].permute(0, 2, 1, 3)
    kview.copy_(w.k_cache0.cuda())
    vview.copy_(w.v_cache0.cuda())
    cache = pkv.KVCache("bf16", kview, vview)
    bt = w.block_tables.cuda()
    sm = pkv.slot_mapping(bt, w.new_req.cuda(), w.new_pos.cuda(), BS)
    pkv.kv_append(w.k_new.cuda(), w.v_new.cuda(), sm, cache)
    out = pkv.paged_decode(w.q.cuda(), cache, bt, w.context_lens.cuda(), sm_scale=w.sm_scale,
                           num_splits=splits)
    torch.cuda.synchronize()
    oc = PL.oracle_caches(w, orc)
    got = PL.gpu_cache_host(cache)
    assert np.array_equal(got["k_cache"], oc["k_cache"]) and np.array_equal(got["v_cache"], oc["v_cache"])
    _check(w, out, PL.oracle_decode(w, orc, oc))


def test_mha_short_small(pkv, orc):
    w = W.mha_short(batch=8, num_blocks=520, seed=97)
    for splits in (0, 2):
        _, out = PL.gpu_run(w, pkv, num_splits=splits)
        _check(w, out, PL.oracle_decode(w, orc, PL.oracle_caches(w, orc)))


def test_full_mha_short(pkv, orc):
    """The page's benchmark shape at full size (batch 32, 32 heads, a
    2048-block pool, contexts 100..999): every cache byte and every output
    row, through the three calls and through pkv_decode_step."""
    from tests.test_gpu_decode import _full_size
    _full_size(W.mha_short(), pkv, orc)
