"""pkv_paged_decode_noalloc: the decode entry point for callers that cannot
allocate device memory while they enqueue work (engine plugins that may not
allocate during enqueue, runtimes whose device memory belongs to their own
pool allocator, serving loops that cannot pay cudaMalloc's device-wide
synchronisation).  Its split-K scratch is a fixed array inside the library
instead of a caller workspace.

Called through the C ABI, its output must match pkv_paged_decode's (which
gets a workspace from the caller) within the decode tolerance -- and, as
both run the same plan and the same deterministic kernels, bit for bit --
on two calls in a row with different inputs, so the second call runs over
the first call's leftovers in the shared array.  This file sorts last so that a run
stopping at the first failure has run every other test first; it also
passes on its own in a fresh process."""
import ctypes

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


def _noalloc_c_abi(pkv_mod, q, cache, bt, cl, sm_scale, num_splits):
    """Direct C-ABI call of pkv_paged_decode_noalloc (no Python wrapper)."""
    m = pkv_mod.pkv
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=q.device)
    cs = cache._struct()
    rc = m.lib().pkv_paged_decode_noalloc(
        ctypes.byref(m._desc(q)), ctypes.byref(cs), ctypes.byref(m._desc(bt)),
        ctypes.byref(m._desc(cl)), ctypes.c_float(sm_scale), ctypes.byref(m._desc(out)),
        int(num_splits), ctypes.c_void_p(err.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, m.lib().pkv_last_error()
    return out, err


@pytest.mark.parametrize("num_splits", [0, 4])
def test_noalloc_matches_workspace_decode_twice(pkv, num_splits):
    cases = [W.gqa_bf16(batch=8, ctx_lo=100, ctx_hi=1500, seed=71),
             W.fp8_long(batch=4, ctx_lo=500, ctx_hi=3000, calib_tokens=128, seed=72)]
    for w in cases:                         # two calls in a row, different inputs
        cache, ref = PL.gpu_run(w, pkv, num_splits=num_splits)
        need = pkv.decode_workspace_bytes(w.q.cuda(), cache, w.block_tables.cuda(), num_splits)
        assert need <= pkv.lib().pkv_noalloc_scratch_bytes()
        out, err = _noalloc_c_abi(pkv, w.q.cuda(), cache, w.block_tables.cuda(),
                                  w.context_lens.cuda(), w.sm_scale, num_splits)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        d = np.max(np.abs(PL.out_f64(out) - PL.out_f64(ref)))
        assert d <= PL.tolerance(w), d
        assert torch.equal(out, ref)


def test_noalloc_auto_plan_falls_back_to_a_plan_that_fits(pkv):
    """With num_splits 0 and a batch whose automatic plan needs more scratch
    than the fixed array, the call takes the largest split count that fits
    (at worst one split, no scratch) instead of failing; its output matches
    the workspace decode's within the tolerance, on two calls in a row."""
    for seed in (73, 74):
        w = W.gqa_bf16(batch=512, ctx_lo=16, ctx_hi=200, seed=seed)
        cache, ref = PL.gpu_run(w, pkv, num_splits=0)
        need = pkv.decode_workspace_bytes(w.q.cuda(), cache, w.block_tables.cuda(), 0)
        assert need > pkv.lib().pkv_noalloc_scratch_bytes()
        out, err = _noalloc_c_abi(pkv, w.q.cuda(), cache, w.block_tables.cuda(),
                                  w.context_lens.cuda(), w.sm_scale, 0)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        d = np.max(np.abs(PL.out_f64(out) - PL.out_f64(ref)))
        assert d <= PL.tolerance(w), d


def test_noalloc_rejects_problems_beyond_its_scratch(pkv):
    """An explicit split count needing more scratch than the fixed array
    gets PKV_ERR_WORKSPACE and a message, before anything is launched."""
    m = pkv.pkv
    B, Hq, Hkv, D = 64, 64, 8, 128
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    cache = pkv.KVCache.allocate("bf16", 4, 16, Hkv, D)
    bt = torch.zeros((B, 256), dtype=torch.int32, device="cuda")
    cl = torch.ones(B, dtype=torch.int32, device="cuda")
    need = pkv.decode_workspace_bytes(q, cache, bt, 8)
    assert need > m.lib().pkv_noalloc_scratch_bytes()
    out = torch.empty_like(q)
    cs = cache._struct()
    rc = m.lib().pkv_paged_decode_noalloc(
        ctypes.byref(m._desc(q)), ctypes.byref(cs), ctypes.byref(m._desc(bt)),
        ctypes.byref(m._desc(cl)), ctypes.c_float(0.088), ctypes.byref(m._desc(out)), 8, None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == m.PkvError(-6, "").code
    assert b"scratch" in m.lib().pkv_last_error()
