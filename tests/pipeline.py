"""Run one workload through the CUDA path (via the C ABI binding) and through
the CPU oracle, from the same seeded host tensors.  The two sides share only
the inputs; each builds its own slot mapping, fills its own cache and runs
its own decode."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W

KIND_CODE_ORACLE = {"f16": 1, "bf16": 2, "e4m3": 3, "u3": 4, "e5m2": 9, "i8": 10}


def src_code(w):
    return 1 if w.dtype == torch.float16 else 2


# ---------------------------------------------------------------- GPU side

def gpu_run(w, pkv, num_splits=0, decode=True, err_flag=None, poison=None, stream=None,
            meta_slot_major=False, via_step=False):
    """Fill + append + decode on the GPU.  Returns (cache, out).
    meta_slot_major: store 3-bit scale/zero arrays contiguous [blocks, slots,
    heads] instead of the allocator's head-major layout.
    via_step: the step's tokens go through pkv_decode_step (slot computation
    fused into the append, decode reading its inputs before the append
    completes), the path the benchmark times, instead of the three calls."""
    dev = "cuda"
    cache = pkv.KVCache.allocate(w.cache_kind, w.num_blocks, w.block_size, w.num_kv_heads,
                                 w.head_dim, device=dev,
                                 k_scale=None if w.k_scale is None else w.k_scale.to(dev),
                                 v_scale=None if w.v_scale is None else w.v_scale.to(dev),
                                 fill=0, scale_mode=w.scale_mode,
                                 k_scales=None if w.k_block_scale is None else w.k_block_scale.to(dev),
                                 v_scales=None if w.v_block_scale is None else w.v_block_scale.to(dev),
                                 layout=w.layout)
    tok = w.scale_mode == "token"

    def append(kn, vn, sm, ks=None, vs=None):
        if tok:
            pkv.kv_append_scaled(kn, vn, ks.to(dev), vs.to(dev), sm, cache, err_flag=err_flag)
        else:
            pkv.kv_append(kn, vn, sm, cache, err_flag=err_flag)
    if meta_slot_major and w.cache_kind == "u3":
        for name in ("k_qscale", "k_qzero", "v_qscale", "v_qzero"):
            setattr(cache, name, torch.zeros_like(getattr(cache, name).contiguous()))
    if w.k_cache0 is not None:
        cache.k_cache.copy_(W.storage(w.k_cache0, w.layout).to(dev))
        cache.v_cache.copy_(W.storage(w.v_cache0, w.layout).to(dev))
    bt = w.block_tables.to(dev)
    if err_flag is None:
        err_flag = torch.zeros(1, dtype=torch.int32, device=dev)
    if w.fill_req is not None:
        chunk = 1 << 20
        for i in range(0, w.fill_req.shape[0], chunk):
            req = w.fill_req[i:i + chunk].to(dev)
            pos = w.fill_pos[i:i + chunk].to(dev)
            sm = pkv.slot_mapping(bt, req, pos, w.block_size, err_flag=err_flag)
            append(w.k_fill[i:i + chunk].to(dev), w.v_fill[i:i + chunk].to(dev), sm,
                   w.k_fill_scale[i:i + chunk] if tok else None,
                   w.v_fill_scale[i:i + chunk] if tok else None)
    if via_step:
        assert not tok and poison is None and decode and w.q is not None
        out = pkv.decode_step(w.k_new.to(dev), w.v_new.to(dev), w.new_req.to(dev),
                              w.new_pos.to(dev), w.q.to(dev), cache, bt, w.context_lens.to(dev),
                              sm_scale=w.sm_scale, num_splits=num_splits, err_flag=err_flag)
        torch.cuda.synchronize()
        return cache, out
    sm = pkv.slot_mapping(bt, w.new_req.to(dev), w.new_pos.to(dev), w.block_size,
                          err_flag=err_flag)
    append(w.k_new.to(dev), w.v_new.to(dev), sm, w.k_new_scale, w.v_new_scale)
    if poison is not None:
        poison(cache)
    out = None
    if decode and w.q is not None:
        out = pkv.paged_decode(w.q.to(dev), cache, bt, w.context_lens.to(dev),
                               sm_scale=w.sm_scale, num_splits=num_splits, err_flag=err_flag)
    torch.cuda.synchronize()
    return cache, out


def gpu_cache_host(cache):
    """Host numpy copies of every cache array (bit patterns), as stored."""
    d = {}
    for name in ("k_cache", "v_cache", "k_qscale", "k_qzero", "v_qscale", "v_qzero", "k_scales",
                 "v_scales"):
        t = getattr(cache, name)
        if t is not None:
            t = t.cpu().contiguous()
            d[name] = t.view(torch.int16).numpy().view(np.uint16) if t.element_size() == 2 \
                else t.numpy() if t.dtype in (torch.int8, torch.float32) else t.view(torch.uint8).numpy()
    return d


# ---------------------------------------------------------------- oracle side

def oracle_caches(w, orc, seqs=None):
    """The oracle's cache after the fill and the step's append.  With
    ``seqs`` only those sequences' rows are appended (the rest stays as
    initialised)."""
    P, BS, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    kind = w.cache_kind
    c = {}
    if kind in ("f16", "bf16"):
        c["k_cache"] = W.bits16(w.k_cache0).copy()
        c["v_cache"] = W.bits16(w.v_cache0).copy()
    elif kind in ("e4m3", "e5m2", "i8"):
        dt = np.int8 if kind == "i8" else np.uint8
        c["k_cache"] = np.zeros((P, BS, H, D), dt)
        c["v_cache"] = np.zeros((P, BS, H, D), dt)
    else:
        c["k_cache"] = np.zeros((P, BS, H, 3 * D // 8), np.uint8)
        c["v_cache"] = np.zeros((P, BS, H, 3 * D // 8), np.uint8)
        c["k_qscale"] = np.zeros((P, BS, H), np.uint16)
        c["v_qscale"] = np.zeros((P, BS, H), np.uint16)
        c["k_qzero"] = np.zeros((P, BS, H), np.uint8)
        c["v_qzero"] = np.zeros((P, BS, H), np.uint8)
    bt = w.block_tables.numpy()
    mode = {"head": orc.SCALE_PER_HEAD, "block": orc.SCALE_PER_BLOCK,
            "token": orc.SCALE_PER_TOKEN}[w.scale_mode]
    if w.scale_mode == "block":
        c["k_scales"] = w.k_block_scale.numpy().copy()
        c["v_scales"] = w.v_block_scale.numpy().copy()
    elif w.scale_mode == "token":
        c["k_scales"] = np.ones((P, BS, H), np.float32)
        c["v_scales"] = np.ones((P, BS, H), np.float32)
    rows = []
    if w.fill_req is not None:
        rows.append((w.fill_req.numpy(), w.fill_pos.numpy(), w.k_fill, w.v_fill, w.k_fill_scale,
                     w.v_fill_scale))
    rows.append((w.new_req.numpy(), w.new_pos.numpy(), w.k_new, w.v_new, w.k_new_scale,
                 w.v_new_scale))
    code = KIND_CODE_ORACLE[kind]
    for req, pos, kn, vn, kts, vts in rows:
        idx = None
        if seqs is not None:
            sel = np.isin(req, np.asarray(seqs)) & (pos >= 0)
            idx = np.nonzero(sel)[0]
            req, pos = req[idx], pos[idx]
            kb, vb = W.bits16(kn[torch.from_numpy(idx)]), W.bits16(vn[torch.from_numpy(idx)])
        else:
            kb, vb = W.bits16(kn), W.bits16(vn)
        if kts is not None:
            kts, vts = kts.numpy(), vts.numpy()
            if idx is not None:
                kts, vts = kts[idx], vts[idx]
        slots = orc.build_slot_mapping(bt, req, pos, BS)
        ks = None if w.k_scale is None else w.k_scale.numpy()
        vs = None if w.v_scale is None else w.v_scale.numpy()
        bad = orc.kv_append(code, src_code(w), kb, vb, slots, c["k_cache"], c["v_cache"], ks, vs,
                            c.get("k_qscale"), c.get("k_qzero"), c.get("v_qscale"),
                            c.get("v_qzero"), scale_mode=mode, k_new_scale=kts, v_new_scale=vts,
                            k_scales=c.get("k_scales"), v_scales=c.get("v_scales"))
        assert bad == 0
    return c


def oracle_decode(w, orc, c, pairs=None, nthreads=None):
    if nthreads is None:
        nthreads = orc.max_threads()
    out, bad = orc.paged_decode(
        KIND_CODE_ORACLE[w.cache_kind], src_code(w), W.bits16(w.q), c["k_cache"], c["v_cache"],
        w.block_tables.numpy(), w.context_lens.numpy(), w.block_size, w.sm_scale,
        k_scale=None if w.k_scale is None else w.k_scale.numpy(),
        v_scale=None if w.v_scale is None else w.v_scale.numpy(),
        k_qscale=c.get("k_qscale"), k_qzero=c.get("k_qzero"), v_qscale=c.get("v_qscale"),
        v_qzero=c.get("v_qzero"), pairs=pairs, nthreads=nthreads,
        scale_mode={"head": orc.SCALE_PER_HEAD, "block": orc.SCALE_PER_BLOCK,
                    "token": orc.SCALE_PER_TOKEN}[w.scale_mode],
        k_scales=c.get("k_scales"), v_scales=c.get("v_scales"))
    assert bad == 0
    return out


def tolerance(w):
    """Max-abs bound against the fp64 oracle: 4e-3 for fp16 outputs, 2e-2
    for bf16 outputs."""
    return 4e-3 if w.dtype == torch.float16 else 2e-2


def out_f64(out):
    return out.detach().cpu().to(torch.float64).numpy()
