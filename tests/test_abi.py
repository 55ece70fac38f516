"""The C-ABI library builds, loads and exports every entry point that
include/pkv.h declares; host-side argument validation rejects bad calls
before any launch.  CPU only (no kernel is launched)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_num_gb300 import build
    build.build()
    from paged_kv_cache_num_gb300 import pkv
    return pkv.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_expected_calls():
    names = _declared_functions()
    for n in ("pkv_kv_append", "pkv_paged_decode", "pkv_paged_decode_workspace", "pkv_pack3",
              "pkv_unpack3", "pkv_unpack3_words", "pkv_slot_mapping", "pkv_last_error",
              "pkv_decode_step", "pkv_paged_decode_noalloc", "pkv_kv_append_scaled",
              "pkv_paged_decode_launches"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_version(lib):
    from paged_kv_cache_num_gb300 import pkv
    assert "sm_103a" in pkv.version()
    assert lib.pkv_abi_version() == 3


def _fake(shape, dtype, strides=None, ptr=0x10000):
    from paged_kv_cache_num_gb300 import pkv
    d = pkv._Tensor()
    d.data = ptr
    d.dtype = dtype
    d.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, strides)):
        d.shape[i] = s
        d.stride[i] = st
    return d


def _cache(kind, P=4, BS=16, H=2, D=64):
    from paged_kv_cache_num_gb300 import pkv
    c = pkv._Cache()
    row = 3 * D // 8 if kind == pkv.U3 else D
    c.k_cache = _fake((P, BS, H, row), kind)
    c.v_cache = _fake((P, BS, H, row), kind, ptr=0x20000)
    return c


def test_append_validation_errors(lib):
    from paged_kv_cache_num_gb300 import pkv
    T, H, D = 3, 2, 64
    kn = _fake((T, H, D), pkv.F16)
    sm = _fake((T,), pkv.I64)
    c = _cache(pkv.F16)
    by = ctypes.byref
    # wrong slot_mapping dtype
    assert lib.pkv_kv_append(by(kn), by(kn), by(_fake((T,), pkv.I32)), by(c), None, None) == -2
    # source dtype differs from a 16-bit cache
    assert lib.pkv_kv_append(by(_fake((T, H, D), pkv.BF16)), by(_fake((T, H, D), pkv.BF16)),
                             by(sm), by(c), None, None) == -2
    # head count mismatch
    assert lib.pkv_kv_append(by(_fake((T, 3, D), pkv.F16)), by(_fake((T, 3, D), pkv.F16)),
                             by(sm), by(c), None, None) == -3
    # a block size that is not a power of two is fine for the append (a
    # contiguous per-request cache) but not for decode; checked through the
    # workspace query, which never launches (these pointers are fake)
    c2 = pkv._Cache()
    c2.k_cache = _fake((4, 12, H, D), pkv.F16)
    c2.v_cache = _fake((4, 12, H, D), pkv.F16)
    q2, bt2 = _fake((2, H, D), pkv.F16), _fake((2, 4), pkv.I32)
    n2 = ctypes.c_size_t(0)
    assert lib.pkv_paged_decode_workspace(by(q2), by(c2), by(bt2), 0, by(n2)) == -5
    # e4m3 without scales
    c3 = _cache(pkv.E4M3)
    assert lib.pkv_kv_append(by(kn), by(kn), by(sm), by(c3), None, None) == -1
    assert b"scale" in lib.pkv_last_error()
    # non-contiguous head_dim
    assert lib.pkv_kv_append(by(_fake((T, H, D), pkv.F16, (H * D * 2, D * 2, 2))),
                             by(kn), by(sm), by(c), None, None) == -4


def test_decode_validation_errors(lib):
    from paged_kv_cache_num_gb300 import pkv
    B, Hq, D = 2, 4, 64
    q = _fake((B, Hq, D), pkv.F16)
    bt = _fake((B, 5), pkv.I32)
    cl = _fake((B,), pkv.I32)
    c = _cache(pkv.F16, H=2, D=D)
    by = ctypes.byref
    n = ctypes.c_size_t(0)
    assert lib.pkv_paged_decode_workspace(by(q), by(c), by(bt), 0, by(n)) == 0
    # group not integral
    q3 = _fake((B, 3, D), pkv.F16)
    assert lib.pkv_paged_decode_workspace(by(q3), by(c), by(bt), 0, by(n)) == -3
    # unsupported head_dim
    c96 = _cache(pkv.F16, D=96)
    q96 = _fake((B, Hq, 96), pkv.F16)
    assert lib.pkv_paged_decode_workspace(by(q96), by(c96), by(bt), 0, by(n)) == -5
    nl = ctypes.c_int32(0)
    assert lib.pkv_paged_decode_launches(by(q), by(c), by(bt), 1, by(nl)) == 0 and nl.value == 1
    assert lib.pkv_paged_decode_launches(by(q), by(c), by(bt), 4, by(nl)) == 0 and nl.value == 2
    assert lib.pkv_paged_decode_launches(by(q3), by(c), by(bt), 0, by(nl)) == -3
    # explicit split needs workspace
    assert lib.pkv_paged_decode_workspace(by(q), by(c), by(bt), 4, by(n)) == 0
    assert n.value > 0
    out = _fake((B, Hq, D), pkv.F16)
    assert lib.pkv_paged_decode(by(q), by(c), by(bt), by(cl), ctypes.c_float(0.125), by(out), 4,
                                None, 0, None, None) == -6
    # output dtype mismatch
    outb = _fake((B, Hq, D), pkv.BF16)
    assert lib.pkv_paged_decode(by(q), by(c), by(bt), by(cl), ctypes.c_float(0.125), by(outb), 1,
                                None, 0, None, None) == -2


def test_xvec_cache_validation(lib):
    """chunk_stride (the x-vectorised layout) is checked before any launch:
    workspace queries only, the pointers being fake."""
    from paged_kv_cache_num_gb300 import pkv
    B, Hq, H, D, P, BS = 2, 4, 2, 64, 4, 16
    q, bt = _fake((B, Hq, D), pkv.F16), _fake((B, 5), pkv.I32)
    by = ctypes.byref
    n = ctypes.c_size_t(0)
    x = 8
    strides = (H * D * BS, x, D * BS, 1)      # [P, Hkv, D/x, BS, x] seen as [P, BS, Hkv, D]
    c = pkv._Cache()
    c.k_cache = _fake((P, BS, H, D), pkv.F16, strides)
    c.v_cache = _fake((P, BS, H, D), pkv.F16, strides, ptr=0x20000)
    c.chunk_stride = BS * x
    assert lib.pkv_paged_decode_workspace(by(q), by(c), by(bt), 0, by(n)) == 0
    c.chunk_stride = 4                         # 8 bytes: not a multiple of 16
    assert lib.pkv_paged_decode_workspace(by(q), by(c), by(bt), 0, by(n)) == -4
    c.chunk_stride = -BS * x
    assert lib.pkv_paged_decode_workspace(by(q), by(c), by(bt), 0, by(n)) == -4
    cu = _cache(pkv.U3, H=H, D=128)
    cu.chunk_stride = 16
    q128 = _fake((B, Hq, 128), pkv.F16)
    assert lib.pkv_paged_decode_workspace(by(q128), by(cu), by(bt), 0, by(n)) == -5
    # one-byte codes: x = 16 elements, head_dim 72 is not a multiple of it
    c8 = pkv._Cache()
    c8.k_cache = _fake((P, BS, H, 72), pkv.E4M3, (H * 72 * BS, 16, 72 * BS, 1))
    c8.v_cache = _fake((P, BS, H, 72), pkv.E4M3, (H * 72 * BS, 16, 72 * BS, 1), ptr=0x20000)
    c8.k_scale = c8.v_scale = 0x30000
    c8.chunk_stride = BS * 16
    q72 = _fake((B, Hq, 72), pkv.F16)
    assert lib.pkv_paged_decode_workspace(by(q72), by(c8), by(bt), 0, by(n)) == -3


def test_pack_validation(lib):
    assert lib.pkv_pack3(ctypes.c_void_p(0x10001), ctypes.c_void_p(0x20000), 4, None) == -4
    assert lib.pkv_unpack3(None, None, -1, None) == -7
    assert lib.pkv_copy_peak(ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), 15, None) == -7


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """No CPU fallback: a missing library raises at first use."""
    from paged_kv_cache_num_gb300 import pkv
    monkeypatch.setattr(pkv, "_lib", None)
    monkeypatch.setattr(pkv, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        pkv.lib()


def test_decode_step_validates_everything_before_launching(lib):
    """pkv_decode_step rejects a bad argument of any of its three parts (here
    with fake device pointers: a launch would fault, so none may happen)."""
    from paged_kv_cache_num_gb300 import pkv
    B, Hq, H, D, T = 2, 4, 2, 64, 2
    by = ctypes.byref
    c = _cache(pkv.F16, H=H, D=D)
    kn = _fake((T, H, D), pkv.F16)
    req, pos = _fake((T,), pkv.I32), _fake((T,), pkv.I32)
    sm = _fake((T,), pkv.I64)
    q, out = _fake((B, Hq, D), pkv.F16), _fake((B, Hq, D), pkv.F16)
    bt, cl = _fake((B, 5), pkv.I32), _fake((B,), pkv.I32)

    def step(**kw):
        a = dict(k=kn, v=kn, req=req, pos=pos, sm=sm, q=q, bt=bt, cl=cl, out=out)
        a.update(kw)
        return lib.pkv_decode_step(by(a["k"]), by(a["v"]), by(a["req"]), by(a["pos"]), by(a["sm"]),
                                   by(a["q"]), by(c), by(a["bt"]), by(a["cl"]), ctypes.c_float(0.125),
                                   by(a["out"]), 0, None, 0, None, None)
    # slot-mapping part: wrong slot dtype; append part: slot count != tokens;
    # decode part: out dtype, context_lens length
    assert step(sm=_fake((T,), pkv.I32)) == -2
    assert step(req=_fake((T + 1,), pkv.I32), pos=_fake((T + 1,), pkv.I32),
                sm=_fake((T + 1,), pkv.I64)) == -3
    assert step(out=_fake((B, Hq, D), pkv.BF16)) == -2
    assert step(cl=_fake((B + 1,), pkv.I32)) == -3
