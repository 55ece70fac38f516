"""GPU parity of paged_decode with the fp64 oracle (max-abs 4e-3 for fp16
outputs, 2e-2 for bf16 outputs), for 16-bit, fp8 and 3-bit caches, with and
without the split-K merge, on small cases that span several blocks and a
ragged tail, on the full-size workloads (every row, through the three
calls and through pkv_decode_step), and on the edge
cases: empty and one-token contexts, poisoned slots beyond the context,
permuted blocks, out-of-range table data."""
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


def _check(w, got, ref, pairs=None):
    g = PL.out_f64(got)
    if pairs is not None:
        g = g.reshape(-1, w.head_dim)[pairs]
        ref = ref.reshape(-1, w.head_dim)[pairs]
    assert np.isfinite(g).all()
    err = np.max(np.abs(g - ref))
    assert err <= PL.tolerance(w), err
    return err


@pytest.mark.parametrize("literal", [False, True])
def test_tiny_fp16(pkv, orc, literal):
    w = W.tiny(literal=literal)
    _, out = PL.gpu_run(w, pkv)
    ref = PL.oracle_decode(w, orc, PL.oracle_caches(w, orc))
    _check(w, out, ref)


@pytest.mark.parametrize("splits", [0, 1, 3, 8])
def test_gqa_bf16_small(pkv, orc, splits):
    w = W.gqa_bf16(batch=6, ctx_lo=1, ctx_hi=700, seed=31)
    _, out = PL.gpu_run(w, pkv, num_splits=splits)
    ref = PL.oracle_decode(w, orc, PL.oracle_caches(w, orc))
    _check(w, out, ref)


@pytest.mark.parametrize("G,BS,D", [(1, 16, 128), (2, 32, 64), (8, 16, 128), (16, 8, 64), (16, 16, 128),
                                    (4, 64, 128), (3, 16, 64)])
def test_group_block_dim_matrix(pkv, orc, G, BS, D):
    w = W.gqa_bf16(batch=3, ctx_lo=1, ctx_hi=9 * BS + 5, num_heads=2 * G, num_kv_heads=2,
                   head_dim=D, block_size=BS, seed=40 + G * BS + D)
    for splits in (0, 1, 4):
        _, out = PL.gpu_run(w, pkv, num_splits=splits)
        ref = PL.oracle_decode(w, orc, PL.oracle_caches(w, orc))
        _check(w, out, ref)


@pytest.mark.parametrize("splits", [0, 1, 5])
def test_fp8_small(pkv, orc, splits):
    w = W.fp8_long(batch=4, ctx_lo=100, ctx_hi=2000, calib_tokens=256, seed=32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache, out = PL.gpu_run(w, pkv, num_splits=splits, err_flag=err)
    assert int(err.item()) == 0
    oc = PL.oracle_caches(w, orc)
    gc = PL.gpu_cache_host(cache)
    for k in oc:
        assert np.array_equal(gc[k], oc[k]), k
    _check(w, out, PL.oracle_decode(w, orc, oc))


@pytest.mark.parametrize("kind", ["e5m2", "i8"])
@pytest.mark.parametrize("splits", [0, 1, 4])
def test_e5m2_i8_small(pkv, orc, splits, kind):
    """e5m2 and int8 caches: append bit exact, decode (fast path and split
    general kernel) against the fp64 oracle on the oracle's own cache."""
    w = W.fp8_long(batch=4, ctx_lo=20, ctx_hi=700, calib_tokens=64, seed=98, fp8=kind)
    cache, out = PL.gpu_run(w, pkv, num_splits=splits)
    oc = PL.oracle_caches(w, orc)
    gc = PL.gpu_cache_host(cache)
    for k in oc:
        assert np.array_equal(gc[k], oc[k]), k
    _check(w, out, PL.oracle_decode(w, orc, oc))


@pytest.mark.parametrize("splits", [0, 1, 4])
def test_u3_small(pkv, orc, splits):
    w = W.u3_mha(batch=4, ctx_lo=20, ctx_hi=900, num_heads=8, seed=33)
    cache, out = PL.gpu_run(w, pkv, num_splits=splits)
    oc = PL.oracle_caches(w, orc)
    gc = PL.gpu_cache_host(cache)
    for k in oc:
        assert np.array_equal(gc[k], oc[k]), k
    _check(w, out, PL.oracle_decode(w, orc, oc))


@pytest.mark.parametrize("BS,H,Hkv", [(32, 8, 8), (16, 16, 4), (32, 12, 4), (16, 4, 2), (16, 12, 6),
                                      (32, 6, 6), (16, 3, 1), (64, 8, 8), (64, 6, 6), (64, 3, 3),
                                      (64, 16, 4)])
def test_u3_block_and_group_variants(pkv, orc, BS, H, Hkv):
    """3-bit cache with blocks of 32 and 64 slots, and grouped q heads over a
    3-bit cache, including kv-head counts not divisible by the 4-head CTA
    (2- and 1-head CTAs, whose ring stages must still start on TMA-aligned
    addresses) and multi-head caches with 4, 2 and 1 kv heads per consumer
    warp."""
    w = W.u3_mha(batch=3, ctx_lo=1, ctx_hi=7 * BS + 3, num_heads=H, block_size=BS, seed=80 + BS + H)
    if Hkv != H:   # regroup: keep Hkv kv heads, H q heads
        w.num_kv_heads = Hkv
        g = torch.Generator().manual_seed(81)
        w.k_fill = w.k_fill[:, :Hkv].contiguous()
        w.v_fill = w.v_fill[:, :Hkv].contiguous()
        w.k_new = w.k_new[:, :Hkv].contiguous()
        w.v_new = w.v_new[:, :Hkv].contiguous()
    for splits in (0, 3):
        cache, out = PL.gpu_run(w, pkv, num_splits=splits)
        oc = PL.oracle_caches(w, orc)
        _check(w, out, PL.oracle_decode(w, orc, oc))


@pytest.mark.parametrize("fp8,scales,G,BS,layout", [
    ("e4m3", "head", 8, 32, "flash"), ("e5m2", "head", 4, 16, "flash"), ("i8", "head", 1, 64, "flash"),
    ("e4m3", "block", 8, 16, "flash"), ("e4m3", "token", 4, 32, "flash"), ("i8", "token", 2, 16, "flash"),
    ("e4m3", "head", 16, 32, "flash"), ("e5m2", "head", 12, 16, "flash"),
    ("e4m3", "head", 8, 32, "xvec"), ("i8", "head", 4, 16, "xvec")])
def test_one_byte_head_dim_64(pkv, orc, fp8, scales, G, BS, layout):
    """One-byte caches at head_dim 64 on the persistent kernel (64-byte rows
    with the 64-byte swizzle; x-vectorised tiles as stored): e4m3, e5m2 and
    int8 with per-head, per-block and per-token scales, groups of 1 to 16 q
    heads, blocks of 16, 32 and 64 slots; against the oracle, through the
    persistent kernel and the general one."""
    Hkv = 4
    w = W.fp8_long(batch=3, ctx_lo=5, ctx_hi=9 * BS + 7, num_heads=G * Hkv, num_kv_heads=Hkv,
                   head_dim=64, block_size=BS, calib_tokens=64, seed=300 + G + BS, fp8=fp8,
                   scales=scales, layout=layout)
    ref = PL.oracle_decode(w, orc, PL.oracle_caches(w, orc))
    for splits in (0, 2):
        cache, out = PL.gpu_run(w, pkv, num_splits=splits)
        _check(w, out, ref)
        if splits == 0:
            gc = PL.gpu_cache_host(cache)
            oc = PL.oracle_caches(w, orc)
            for k, arr in oc.items():
                if layout == "xvec" and k in ("k_cache", "v_cache"):
                    arr = orc.to_xvec(arr, 16)
                assert np.array_equal(gc[k], arr), k


def test_u3_poisoned_tail_metadata(pkv, orc):
    """NaN scales and garbage codes in slots beyond the contexts of a 3-bit
    cache leave the output finite and unchanged."""
    w = W.u3_mha(batch=4, ctx_lo=3, ctx_hi=300, num_heads=8, seed=88)
    live = torch.zeros((w.num_blocks, w.block_size), dtype=torch.bool)
    for b in range(w.batch):
        for t in range(int(w.context_lens[b])):
            live[int(w.block_tables[b, t // w.block_size]), t % w.block_size] = True
    dead = (~live).cuda()

    def poison(cache):
        for t in (cache.k_qscale, cache.v_qscale):
            t[dead] = float("nan")
        for t in (cache.k_cache, cache.v_cache):
            t[dead] = 0xA5
    for splits in (0, 2):
        _, clean = PL.gpu_run(w, pkv, num_splits=splits)
        _, dirty = PL.gpu_run(w, pkv, num_splits=splits, poison=poison)
        assert torch.isfinite(dirty.float()).all()
        assert torch.equal(clean, dirty)


def test_u3_slot_major_metadata(pkv, orc):
    """Scale / zero arrays stored slot-major (each CTA stages every head's
    metadata) give the same output as the head-major default, and match the
    oracle."""
    w = W.u3_mha(batch=5, ctx_lo=3, ctx_hi=700, num_heads=16, seed=91)
    c1, out_h = PL.gpu_run(w, pkv)
    c2, out_s = PL.gpu_run(w, pkv, meta_slot_major=True)
    assert c1.k_qscale.stride()[1:] == (1, w.block_size)
    assert c2.k_qscale.is_contiguous()
    assert torch.equal(out_h, out_s)
    oc = PL.oracle_caches(w, orc)
    _check(w, out_s, PL.oracle_decode(w, orc, oc))


def test_u3_head_dim_64(pkv, orc):
    w = W.u3_mha(batch=3, ctx_lo=5, ctx_hi=300, num_heads=4, head_dim=64, seed=34)
    cache, out = PL.gpu_run(w, pkv)
    oc = PL.oracle_caches(w, orc)
    _check(w, out, PL.oracle_decode(w, orc, oc))


@pytest.mark.parametrize("batch,ctx_hi", [(1, 5), (2, 40), (3, 17), (200, 64), (7, 5000)])
def test_fast_path_grid_shapes(pkv, orc, batch, ctx_hi):
    """Fewer blocks than CTAs (idle CTAs between the owners of one sequence),
    single-block sequences, many short sequences, one long sequence split
    over many CTAs."""
    w = W.gqa_bf16(batch=batch, ctx_lo=1, ctx_hi=ctx_hi, seed=60 + batch)
    _, out = PL.gpu_run(w, pkv, num_splits=0)
    _check(w, out, PL.oracle_decode(w, orc, PL.oracle_caches(w, orc)))


def test_fast_path_fp16_and_strided_q(pkv, orc):
    """fp16 cache with head_dim 64 (the tiny shape scaled up) and q / out
    views with padded row strides."""
    w = W.gqa_bf16(batch=5, ctx_lo=1, ctx_hi=900, num_heads=8, num_kv_heads=4, head_dim=64, seed=66)
    w.dtype = torch.float16
    w.cache_kind = "f16"
    for name in ("q", "k_cache0", "v_cache0", "k_new", "v_new"):
        setattr(w, name, getattr(w, name).to(torch.float16))
    cache, out = PL.gpu_run(w, pkv, num_splits=0)
    ref = PL.oracle_decode(w, orc, PL.oracle_caches(w, orc))
    _check(w, out, ref)
    qpad = torch.zeros((w.batch, w.num_heads, w.head_dim + 8), dtype=w.dtype, device="cuda")
    qpad[..., :w.head_dim] = w.q.cuda()
    opad = torch.zeros_like(qpad)
    pkv.paged_decode(qpad[..., :w.head_dim], cache, w.block_tables.cuda(), w.context_lens.cuda(),
                     sm_scale=w.sm_scale, out=opad[..., :w.head_dim])
    torch.cuda.synchronize()
    _check(w, opad[..., :w.head_dim], ref)


def test_split_count_invariance(pkv):
    w = W.gqa_bf16(batch=4, ctx_lo=50, ctx_hi=3000, seed=35)
    outs = [PL.out_f64(PL.gpu_run(w, pkv, num_splits=s)[1]) for s in (1, 0, 2, 7, 16)]
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 2e-2


def test_empty_and_single_token_contexts(pkv, orc):
    w = W.gqa_bf16(batch=4, ctx_lo=1, ctx_hi=300, seed=36)
    w.context_lens[0] = 0
    w.context_lens[1] = 1
    # keep the appended token inside the context of every sequence
    w.new_pos[:] = torch.clamp(w.context_lens - 1, min=0)
    w.new_pos[0] = -1
    for splits in (0, 1, 3):
        _, out = PL.gpu_run(w, pkv, num_splits=splits)
        ref = PL.oracle_decode(w, orc, PL.oracle_caches(w, orc))
        _check(w, out, ref)
        assert torch.all(out[0] == 0)


def test_poison_beyond_context(pkv, orc):
    """NaN in every slot outside the live contexts (the tail of the last block
    included) leaves the output finite and equal to the clean run."""
    w = W.gqa_bf16(batch=5, ctx_lo=17, ctx_hi=500, seed=37)
    live = torch.zeros((w.num_blocks, w.block_size), dtype=torch.bool)
    for b in range(w.batch):
        for t in range(int(w.context_lens[b])):
            live[int(w.block_tables[b, t // w.block_size]), t % w.block_size] = True
    dead = (~live).cuda()

    def poison(cache):
        cache.k_cache[dead] = float("nan")
        cache.v_cache[dead] = float("nan")

    for splits in (0, 1, 4):
        _, clean = PL.gpu_run(w, pkv, num_splits=splits)
        _, dirty = PL.gpu_run(w, pkv, num_splits=splits, poison=poison)
        assert torch.isfinite(dirty.float()).all()
        assert torch.equal(clean, dirty)


def test_block_permutation_invariance(pkv):
    w = W.gqa_bf16(batch=3, ctx_lo=30, ctx_hi=400, seed=38)
    _, base = PL.gpu_run(w, pkv)
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(1))
    k2 = torch.empty_like(w.k_cache0)
    v2 = torch.empty_like(w.v_cache0)
    k2[perm] = w.k_cache0
    v2[perm] = w.v_cache0
    w.k_cache0, w.v_cache0 = k2, v2
    w.block_tables = perm.to(torch.int32)[w.block_tables.long()]
    _, moved = PL.gpu_run(w, pkv)
    assert torch.equal(base, moved)


def test_bad_table_data_is_flagged_not_faulting(pkv):
    w = W.gqa_bf16(batch=3, ctx_lo=30, ctx_hi=60, seed=39)
    w.block_tables[1, 0] = w.num_blocks + 7
    w.block_tables[2, 1] = -3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    w.new_pos[1:] = -1          # no appends through the broken rows
    PL.gpu_run(w, pkv, err_flag=err)
    assert int(err.item()) & pkv.pkv.DEVERR_BLOCK_RANGE
    w2 = W.gqa_bf16(batch=2, ctx_lo=30, ctx_hi=60, seed=39)
    w2.context_lens[0] = 10 ** 6
    w2.new_pos[:] = -1
    err.zero_()
    PL.gpu_run(w2, pkv, err_flag=err)
    assert int(err.item()) & pkv.pkv.DEVERR_CONTEXT_RANGE


# ---------------------------------------------------------------- full-size

def _sample_pairs(w, seqs, heads_per_seq=None):
    pairs = []
    for b in seqs:
        hs = range(w.num_heads) if heads_per_seq is None else heads_per_seq
        pairs += [b * w.num_heads + h for h in hs]
    return np.array(pairs, np.int32)


def _full_size(w, pkv, orc, paths=("calls", "step")):
    """A full-size workload through the GPU along each path (the three calls;
    pkv_decode_step, the benchmark's path), the oracle once: every cache
    byte of the whole pool and every (sequence, head) output row compared."""
    oc = PL.oracle_caches(w, orc)
    ref = PL.oracle_decode(w, orc, oc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    worst = 0.0
    for path in paths:
        cache, out = PL.gpu_run(w, pkv, err_flag=err, via_step=path == "step")
        assert int(err.item()) == 0, path
        gc = PL.gpu_cache_host(cache)
        for k, arr in oc.items():
            if w.layout == "xvec" and k in ("k_cache", "v_cache"):
                arr = orc.to_xvec(arr, 16 // arr.dtype.itemsize)   # storage order
            assert np.array_equal(gc[k], arr), (path, k)
        del cache, gc
        worst = max(worst, _check(w, out, ref))
    return worst


def test_full_gqa_bf16(pkv, orc):
    """Full-size GQA bf16 workload (batch 64, contexts 512..4096)."""
    _full_size(W.gqa_bf16(), pkv, orc)


def test_full_fp8_long(pkv, orc):
    """Full-size long-context fp8 workload (batch 16, 64 q / 8 kv heads,
    contexts 16K..32K, e4m3 with per-head scales): the benchmark's
    headline workload."""
    _full_size(W.fp8_long(), pkv, orc)


def test_full_fp8_long_e5m2(pkv, orc):
    """The long-context shape with an e5m2 cache (scales amax/57344)."""
    _full_size(W.fp8_long(seed=W.SEEDS["fp8_long_e5m2"], fp8="e5m2"), pkv, orc, paths=("step",))


def test_full_i8_long(pkv, orc):
    """The long-context shape with an int8 cache (scales amax/127)."""
    _full_size(W.fp8_long(seed=W.SEEDS["i8_long"], fp8="i8"), pkv, orc, paths=("step",))


def test_full_u3_g16(pkv, orc):
    """Full-size grouped 3-bit step (batch 16, 128 q / 8 kv heads, contexts
    U{8192..32768}, blocks of 16): every row and the whole pool."""
    _full_size(W.u3_mha(batch=16, ctx_lo=8192, ctx_hi=32768, num_heads=128, num_kv_heads=8,
                        seed=W.SEEDS["u3_g16"]), pkv, orc)


def test_full_u3_mha(pkv, orc):
    """Full-size 3-bit MHA workload (batch 32, 32 heads, contexts
    1024..8192)."""
    _full_size(W.u3_mha(), pkv, orc)


@pytest.mark.parametrize("maker", ["gqa", "u3"])
def test_decode_step_equals_separate_calls(pkv, orc, maker):
    """pkv_decode_step (slot mapping + append + decode in one call) gives the
    same slots, cache bytes and output as the three calls."""
    if maker == "gqa":
        w = W.gqa_bf16(batch=6, ctx_lo=10, ctx_hi=400, seed=92)
    else:
        w = W.u3_mha(batch=5, ctx_lo=3, ctx_hi=500, num_heads=8, seed=93)
    cache, out_sep = PL.gpu_run(w, pkv)               # fill, append, decode: three calls
    before = PL.gpu_cache_host(cache)
    dev = "cuda"
    bt, req, pos = w.block_tables.to(dev), w.new_req.to(dev), w.new_pos.to(dev)
    slots_sep = pkv.slot_mapping(bt, req, pos, w.block_size)
    slots = torch.full_like(slots_sep, -7)
    out = pkv.decode_step(w.k_new.to(dev), w.v_new.to(dev), req, pos, w.q.to(dev), cache, bt,
                          w.context_lens.to(dev), sm_scale=w.sm_scale, slots=slots)
    torch.cuda.synchronize()
    assert torch.equal(slots, slots_sep)
    after = PL.gpu_cache_host(cache)
    for k in before:                                  # re-appending the same rows changes nothing
        assert np.array_equal(before[k], after[k]), k
    assert torch.equal(out, out_sep)
    _check(w, out, PL.oracle_decode(w, orc, PL.oracle_caches(w, orc)))


@pytest.mark.parametrize("kind", ["e4m3", "bf16"])
def test_decode_step_padding_and_bad_positions(pkv, orc, kind):
    """decode_step computes the slots inside its append kernel: padding
    tokens (pos -1, NaN rows) and a position beyond the block table give slot
    -1, write nothing and (the latter) raise PKV_DEVERR_POS_RANGE, exactly as
    pkv_slot_mapping does; the cache and the output match the separate calls."""
    if kind == "e4m3":
        w = W.fp8_long(batch=3, ctx_lo=40, ctx_hi=300, calib_tokens=64, seed=270)
    else:
        w = W.gqa_bf16(batch=3, ctx_lo=40, ctx_hi=300, seed=271)
    cache, out_sep = PL.gpu_run(w, pkv)
    before = PL.gpu_cache_host(cache)
    dev = "cuda"
    B = w.batch
    n_bad = 5
    req = torch.cat([w.new_req, torch.tensor([0, 1, 2, 0, 1], dtype=torch.int32)])
    pos = torch.cat([w.new_pos, torch.tensor([-1, -1, w.max_blocks * w.block_size + 3, -1, -1],
                                             dtype=torch.int32)])
    nan = torch.full((n_bad,) + tuple(w.k_new.shape[1:]), float("nan"), dtype=w.k_new.dtype)
    kn, vn = torch.cat([w.k_new, nan]).to(dev), torch.cat([w.v_new, nan]).to(dev)
    bt, req, pos = w.block_tables.to(dev), req.to(dev), pos.to(dev)
    err_sep = torch.zeros(1, dtype=torch.int32, device=dev)
    slots_sep = pkv.slot_mapping(bt, req, pos, w.block_size, err_flag=err_sep)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    slots = torch.full_like(slots_sep, -7)
    out = pkv.decode_step(kn, vn, req, pos, w.q.to(dev), cache, bt, w.context_lens.to(dev),
                          sm_scale=w.sm_scale, slots=slots, err_flag=err)
    torch.cuda.synchronize()
    assert torch.equal(slots, slots_sep)
    assert int(slots[-n_bad:].max()) == -1
    assert int(err.item()) == int(err_sep.item()) == pkv.pkv.DEVERR_POS_RANGE
    after = PL.gpu_cache_host(cache)
    for k in before:
        assert np.array_equal(before[k], after[k]), k
    assert torch.equal(out, out_sep)


def test_decode_step_prefill_sized_batch(pkv, orc):
    """A step whose append is prefill-sized (>= 1024 tokens, contiguous head
    rows) runs the bulk-copy append with the slots computed inside it: same
    slots, cache bytes (whole pool) and output as the separate calls."""
    w = W.mixed_append(n_prefill=4, n_decode=12, prefill_lo=300, prefill_hi=600, ctx_lo=100,
                       ctx_hi=900, block_size=16, seed=273)
    assert int((w.new_pos >= 0).sum()) >= 1024
    g = torch.Generator().manual_seed(274)
    w.num_heads = 4 * w.num_kv_heads
    w.q = torch.randn((w.batch, w.num_heads, w.head_dim), generator=g).to(w.dtype)
    # finite older rows for the decode requests (the pool is random bytes otherwise)
    w.k_cache0 = torch.randn(tuple(w.k_cache0.shape), generator=g).to(w.dtype)
    w.v_cache0 = torch.randn(tuple(w.v_cache0.shape), generator=g).to(w.dtype)
    dev = "cuda"
    cache_a, out_a = PL.gpu_run(w, pkv)                       # slot_mapping + append + decode
    cache_b = pkv.KVCache.allocate("bf16", w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    cache_b.k_cache.copy_(w.k_cache0.to(dev))
    cache_b.v_cache.copy_(w.v_cache0.to(dev))
    bt, req, pos = w.block_tables.to(dev), w.new_req.to(dev), w.new_pos.to(dev)
    slots = torch.full((req.shape[0],), -7, dtype=torch.int64, device=dev)
    out_b = pkv.decode_step(w.k_new.to(dev), w.v_new.to(dev), req, pos, w.q.to(dev), cache_b, bt,
                            w.context_lens.to(dev), sm_scale=w.sm_scale, slots=slots)
    torch.cuda.synchronize()
    assert torch.equal(slots, pkv.slot_mapping(bt, req, pos, w.block_size))
    a, b = PL.gpu_cache_host(cache_a), PL.gpu_cache_host(cache_b)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    assert torch.equal(out_a, out_b)
    oc = PL.oracle_caches(w, orc)
    assert np.array_equal(b["k_cache"], oc["k_cache"]) and np.array_equal(b["v_cache"], oc["v_cache"])
    _check(w, out_b, PL.oracle_decode(w, orc, oc))


class _Top:
    """The blocks [off, num_blocks) of a cache, under the attribute names
    PL.gpu_cache_host reads."""
    def __init__(self, cache, off):
        for name in ("k_cache", "v_cache", "k_qscale", "k_qzero", "v_qscale", "v_qzero", "k_scales",
                     "v_scales"):
            t = getattr(cache, name, None)
            setattr(self, name, None if t is None else t[off:])


@pytest.mark.parametrize("kind", ["bf16", "e4m3", "u3"])
def test_pool_beyond_4gib(pkv, orc, kind):
    """A pool whose K and V caches pass 4 GiB each, the sequences' blocks at
    its top (every byte offset above 2^32): the appends write the same bytes
    and both decode kernels give the same outputs, bit for bit, as on a pool
    of just those blocks."""
    if kind == "bf16":
        w = W.gqa_bf16(batch=3, ctx_lo=40, ctx_hi=300, seed=275)
    elif kind == "e4m3":
        w = W.fp8_long(batch=3, ctx_lo=40, ctx_hi=300, calib_tokens=64, seed=276)
    else:
        w = W.u3_mha(batch=3, ctx_lo=3, ctx_hi=500, num_heads=8, seed=277)
    dev = "cuda"
    small, out0 = PL.gpu_run(w, pkv)
    _, out3 = PL.gpu_run(w, pkv, num_splits=3)
    ref = PL.gpu_cache_host(small)
    del small
    row = {"bf16": 2 * w.head_dim, "e4m3": w.head_dim, "u3": 3 * w.head_dim // 8}[kind]
    block_bytes = w.block_size * w.num_kv_heads * row
    off = (1 << 32) // block_bytes + 17
    cache = pkv.KVCache.allocate(w.cache_kind, w.num_blocks + off, w.block_size, w.num_kv_heads,
                                 w.head_dim, device=dev,
                                 k_scale=None if w.k_scale is None else w.k_scale.to(dev),
                                 v_scale=None if w.v_scale is None else w.v_scale.to(dev))
    assert cache.k_cache[off:].data_ptr() - cache.k_cache.data_ptr() > (1 << 32)
    top = _Top(cache, off)
    for name in ("k_cache", "v_cache", "k_qscale", "k_qzero", "v_qscale", "v_qzero"):
        if getattr(top, name) is not None:     # as the small run's pool started (fill 0)
            getattr(top, name).zero_()
    if w.k_cache0 is not None:
        top.k_cache.copy_(w.k_cache0.to(dev))
        top.v_cache.copy_(w.v_cache0.to(dev))
    bt = (w.block_tables + off).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if w.fill_req is not None:
        sm = pkv.slot_mapping(bt, w.fill_req.to(dev), w.fill_pos.to(dev), w.block_size, err_flag=err)
        pkv.kv_append(w.k_fill.to(dev), w.v_fill.to(dev), sm, cache, err_flag=err)
    sm = pkv.slot_mapping(bt, w.new_req.to(dev), w.new_pos.to(dev), w.block_size, err_flag=err)
    pkv.kv_append(w.k_new.to(dev), w.v_new.to(dev), sm, cache, err_flag=err)
    outs = [pkv.paged_decode(w.q.to(dev), cache, bt, w.context_lens.to(dev), sm_scale=w.sm_scale,
                             num_splits=ns, err_flag=err) for ns in (0, 3)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = PL.gpu_cache_host(top)
    for k in ref:
        assert np.array_equal(ref[k], got[k]), k
    assert torch.equal(outs[0], out0) and torch.equal(outs[1], out3)
    del cache, top
    torch.cuda.empty_cache()
    _check(w, outs[0], PL.oracle_decode(w, orc, PL.oracle_caches(w, orc)))


def test_decode_step_without_new_tokens(pkv):
    """A step with no new tokens launches no append; its decode then waits
    for the stream's earlier work as a plain paged_decode does, and gives the
    same output (also right after another step's kernels on the stream)."""
    w = W.gqa_bf16(batch=5, ctx_lo=30, ctx_hi=900, seed=272)
    cache, out_sep = PL.gpu_run(w, pkv)
    dev = "cuda"
    bt, cl, q = w.block_tables.to(dev), w.context_lens.to(dev), w.q.to(dev)
    e16 = torch.empty((0,) + tuple(w.k_new.shape[1:]), dtype=w.k_new.dtype, device=dev)
    ei = torch.empty(0, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    for _ in range(3):
        pkv.decode_step(w.k_new.to(dev), w.v_new.to(dev), w.new_req.to(dev), w.new_pos.to(dev), q,
                        cache, bt, cl, sm_scale=w.sm_scale, out=out)
        pkv.decode_step(e16, e16, ei, ei, q, cache, bt, cl, sm_scale=w.sm_scale, out=out,
                        slots=torch.empty(0, dtype=torch.int64, device=dev))
    torch.cuda.synchronize()
    assert torch.equal(out, out_sep)


def test_u3_bad_block_ids_in_pairs(pkv, orc):
    """3-bit cache with 16-token blocks (which the persistent kernel takes two
    at a time): block ids out of range at an even and at an odd position of a
    sequence are skipped and flagged; the untouched sequences still match the
    oracle, and the broken ones match the general kernel, which leaves out the
    same blocks."""
    w = W.u3_mha(batch=4, ctx_lo=100, ctx_hi=200, num_heads=8, seed=95)
    w.block_tables[1, 2] = w.num_blocks + 5
    w.block_tables[2, 5] = -1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, fast = PL.gpu_run(w, pkv, err_flag=err)
    assert int(err.item()) & pkv.pkv.DEVERR_BLOCK_RANGE
    _, general = PL.gpu_run(w, pkv, num_splits=1)
    a, g = PL.out_f64(fast), PL.out_f64(general)
    assert np.isfinite(a).all()
    assert np.max(np.abs(a[1:3] - g[1:3])) <= PL.tolerance(w)
    seqs = [0, 3]
    oc = PL.oracle_caches(w, orc, seqs=seqs)
    pairs = _sample_pairs(w, seqs)
    _check(w, fast, PL.oracle_decode(w, orc, oc, pairs=pairs), pairs)


@pytest.mark.parametrize("kind,G,layout", [("bf16", 16, "flash"), ("bf16", 12, "flash"), ("f16", 16, "flash"),
                                           ("bf16", 16, "xvec"), ("e4m3", 16, "flash"), ("i8", 12, "flash"),
                                           ("e4m3", 16, "xvec")])
def test_large_groups_two_column_groups(pkv, orc, kind, G, layout):
    """Groups of 9..16 q heads per kv head (Llama-3.1-405B: 128 q / 8 kv):
    the persistent kernel's warp of a kv head serves them as two groups of
    8 head columns (the second with G - 8 of them), each K / V fragment
    feeding one MMA per group; parity with the oracle, on the persistent
    kernel (no explicit split) and the general one."""
    Hkv = 4
    if kind in ("bf16", "f16"):
        w = W.gqa_bf16(batch=5, ctx_lo=1, ctx_hi=1500, num_heads=G * Hkv, num_kv_heads=Hkv,
                       seed=280 + G, layout=layout)
        if kind == "f16":
            w.dtype = torch.float16
            w.cache_kind = "f16"
            for name in ("q", "k_cache0", "v_cache0", "k_new", "v_new"):
                setattr(w, name, getattr(w, name).to(torch.float16))
    else:
        w = W.fp8_long(batch=3, ctx_lo=20, ctx_hi=1200, num_heads=G * Hkv, num_kv_heads=Hkv,
                       calib_tokens=64, seed=290 + G, fp8=kind, layout=layout)
    ref = PL.oracle_decode(w, orc, PL.oracle_caches(w, orc))
    for splits in (0, 2):
        cache, out = PL.gpu_run(w, pkv, num_splits=splits)
        if splits == 0:
            assert pkv.decode_launches(w.q.cuda(), cache, w.block_tables.cuda()) == 2  # persistent
        _check(w, out, ref)


@pytest.mark.parametrize("BS,G,Hkv", [(16, 16, 4), (32, 16, 2), (16, 12, 2), (32, 9, 3), (16, 10, 1)])
def test_u3_large_groups(pkv, orc, BS, G, Hkv):
    """3-bit caches with groups of 9..16 q heads per kv head: two groups of
    head columns per consumer warp, the codes of each K / V fragment
    unpacked once for both; blocks of 16 and 32 slots, 1 to 4 kv heads;
    parity with the oracle on the persistent kernel and the general one, and
    the cache as written bit-exact."""
    w = W.u3_mha(batch=3, ctx_lo=1, ctx_hi=9 * BS + 5, num_heads=G * Hkv, num_kv_heads=Hkv, block_size=BS,
                 seed=400 + G + BS)
    oc = PL.oracle_caches(w, orc)
    ref = PL.oracle_decode(w, orc, oc)
    for splits in (0, 3):
        cache, out = PL.gpu_run(w, pkv, num_splits=splits)
        if splits == 0:
            assert pkv.decode_launches(w.q.cuda(), cache, w.block_tables.cuda()) == 2  # persistent
            gc = PL.gpu_cache_host(cache)
            for k in oc:
                assert np.array_equal(gc[k], oc[k]), k
        _check(w, out, ref)


def test_large_group_token_scales(pkv, orc):
    """Group 16 with per-token fp8 scales staged with the blocks."""
    w = W.fp8_long(batch=3, ctx_lo=20, ctx_hi=900, num_heads=64, num_kv_heads=4, calib_tokens=64,
                   seed=299, scales="token")
    _, out = PL.gpu_run(w, pkv)
    _check(w, out, PL.oracle_decode(w, orc, PL.oracle_caches(w, orc)))


def test_full_405b_like_fp8(pkv, orc):
    """Llama-3.1-405B-like long-context e4m3 step: batch 8, 128 q / 8 kv
    heads (group 16), contexts 16K..32K."""
    _full_size(W.fp8_long(batch=8, num_heads=128, seed=298), pkv, orc, paths=("step",))


def test_full_fp8_long_g16(pkv, orc):
    """The benchmark's group-16 long-context workload (batch 16, 128 q / 8
    kv heads, e4m3)."""
    _full_size(W.fp8_long(seed=W.SEEDS["fp8_long_g16"], num_heads=128), pkv, orc,
               paths=("step",))


@pytest.mark.parametrize("kind", ["bf16", "e4m3", "i8", "u3", "u3_g4"])
@pytest.mark.parametrize("sm_scale", [-0.0883883476, 0.0, 0.75])
def test_softmax_scale_sign_zero_and_sharp(pkv, orc, kind, sm_scale):
    """The softmax scale at its edges: negative (the softmax of -q.k), zero
    (uniform weights: each output row is the mean of its V rows) and large
    (a sharp softmax whose logits span hundreds of log2 units), on the
    persistent kernel and the general one, 16-bit, one-byte and 3-bit
    caches; against the oracle at the same scale."""
    if kind == "bf16":
        w = W.gqa_bf16(batch=3, ctx_lo=1, ctx_hi=300, num_heads=8, num_kv_heads=2, seed=500)
    elif kind in ("e4m3", "i8"):
        w = W.fp8_long(batch=3, ctx_lo=5, ctx_hi=400, num_heads=16, num_kv_heads=2, calib_tokens=64,
                       seed=501, fp8=kind)
    elif kind == "u3":
        w = W.u3_mha(batch=3, ctx_lo=1, ctx_hi=300, num_heads=8, seed=502)
    else:
        w = W.u3_mha(batch=3, ctx_lo=1, ctx_hi=300, num_heads=8, num_kv_heads=2, seed=503)
    w.sm_scale = sm_scale
    ref = PL.oracle_decode(w, orc, PL.oracle_caches(w, orc))
    for splits in (0, 2):
        cache, out = PL.gpu_run(w, pkv, num_splits=splits)
        _check(w, out, ref)
