"""CPU oracle for the paged KV-cache hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The library never does: the
CUDA path and this oracle share no code.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64 attention, the
quantisers in the exact fp32 operation order they are defined with).  This
module compiles it with gcc on first use and wraps it with ctypes over numpy
arrays.  Each wrapper names the passage it follows; see the C file's header
for the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

# dtype codes of the oracle's own interface
F16, BF16, E4M3, U3, E5M2, I8 = 1, 2, 3, 4, 9, 10
# scale granularity of fp8 / int8 caches
SCALE_PER_HEAD, SCALE_PER_BLOCK, SCALE_PER_TOKEN = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.pkvo_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.pkvo_f16_to_f64.restype = dbl
        lib.pkvo_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.pkvo_bf16_to_f64.restype = dbl
        lib.pkvo_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.pkvo_e4m3_to_f64.restype = dbl
        lib.pkvo_f32_to_e4m3.argtypes = [ctypes.c_float]
        lib.pkvo_f32_to_e4m3.restype = ctypes.c_uint8
        lib.pkvo_f32_to_f16_rn.argtypes = [ctypes.c_float]
        lib.pkvo_f32_to_f16_rn.restype = ctypes.c_uint16
        lib.pkvo_pack3.argtypes = [P, P, i64]
        lib.pkvo_unpack3.argtypes = [P, P, i64]
        lib.pkvo_unpack3_words.argtypes = [P, P, i64]
        lib.pkvo_u3_quantize_pack_rows.argtypes = [P, i32, i64, i32, P, P, P]
        lib.pkvo_build_slot_mapping.argtypes = [P, i32, i32, P, P, i64, P]
        lib.pkvo_kv_append.argtypes = [i32, i32, i64, i32, i32, P, P, P, i64, i32, P, P, P, P,
                                       P, P, P, P]
        lib.pkvo_kv_append.restype = i64
        lib.pkvo_paged_decode.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, P, P, i64, P,
                                          i32, P, dbl, P, P, P, P, P, P, P, i64, P, i32]
        lib.pkvo_paged_decode.restype = i64
        lib.pkvo_kv_append_scaled.argtypes = lib.pkvo_kv_append.argtypes + [i32, P, P, P, P]
        lib.pkvo_kv_append_scaled.restype = i64
        lib.pkvo_paged_decode_scaled.argtypes = lib.pkvo_paged_decode.argtypes + [i32, P, P]
        lib.pkvo_paged_decode_scaled.restype = i64
        lib.pkvo_max_threads.restype = i32
        for fn in ("pkvo_f32_to_e4m3_n", "pkvo_f32_to_f16_n", "pkvo_f16_to_f64_n",
                   "pkvo_bf16_to_f64_n", "pkvo_e4m3_to_f64_n", "pkvo_f32_to_e5m2_n",
                   "pkvo_e5m2_to_f64_n", "pkvo_f32_to_i8_n"):
            getattr(lib, fn).argtypes = [P, P, i64]
        _lib = lib
        return lib


def _ptr(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous numpy"
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().pkvo_max_threads())


# --------------------------------------------------------------------------
# scalar formats (array forms of the C conversions)
# --------------------------------------------------------------------------

def _conv(fn, x, in_dtype, out_dtype):
    a = np.ascontiguousarray(x, dtype=in_dtype)
    out = np.empty(a.shape, dtype=out_dtype)
    getattr(_load(), fn)(_ptr(a.reshape(-1)), _ptr(out.reshape(-1)), a.size)
    return out


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns -> float64."""
    return _conv("pkvo_f16_to_f64_n", bits, np.uint16, np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64."""
    return _conv("pkvo_bf16_to_f64_n", bits, np.uint16, np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP E4M3 decode of each byte."""
    return _conv("pkvo_e4m3_to_f64_n", codes, np.uint8, np.float64)


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """binary32 -> E4M3 code, RNE, saturating to +-448 (NaN -> 0x7F)."""
    return _conv("pkvo_f32_to_e4m3_n", x, np.float32, np.uint8)


def e5m2_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP E5M2 decode of each byte."""
    return _conv("pkvo_e5m2_to_f64_n", codes, np.uint8, np.float64)


def f32_to_e5m2(x: np.ndarray) -> np.ndarray:
    """binary32 -> E5M2 code, RNE, saturating to +-57344 (NaN -> 0x7F)."""
    return _conv("pkvo_f32_to_e5m2_n", x, np.float32, np.uint8)


def f32_to_i8(x: np.ndarray) -> np.ndarray:
    """binary32 (already divided by the scale) -> int8 code: nearest, half to
    even, saturated to +-127, NaN -> 0."""
    return _conv("pkvo_f32_to_i8_n", x, np.float32, np.int8)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """binary32 -> binary16 bits, RNE."""
    return _conv("pkvo_f32_to_f16_n", x, np.float32, np.uint16)


# --------------------------------------------------------------------------
# 3-bit packing ("triton-3bit-kv-cache-kernel" README, sections 1.A / 1.B)
# --------------------------------------------------------------------------

def pack3(values: np.ndarray) -> np.ndarray:
    """values uint8 [n, 8] -> packed uint8 [n, 3] (octet formulas, 1.A)."""
    v = np.ascontiguousarray(values, dtype=np.uint8).reshape(-1, 8)
    out = np.empty((v.shape[0], 3), dtype=np.uint8)
    _load().pkvo_pack3(_ptr(v), _ptr(out), v.shape[0])
    return out


def unpack3(packed: np.ndarray) -> np.ndarray:
    """packed uint8 [n, 3] -> values uint8 [n, 8] (octet formulas, 1.A)."""
    p = np.ascontiguousarray(packed, dtype=np.uint8).reshape(-1, 3)
    out = np.empty((p.shape[0], 8), dtype=np.uint8)
    _load().pkvo_unpack3(_ptr(p), _ptr(out), p.shape[0])
    return out


def unpack3_words(words: np.ndarray) -> np.ndarray:
    """words uint32 [m, 3] -> values uint8 [m, 32] (96-bit lane formula, 1.B)."""
    w = np.ascontiguousarray(words, dtype=np.uint32).reshape(-1, 3)
    out = np.empty((w.shape[0], 32), dtype=np.uint8)
    _load().pkvo_unpack3_words(_ptr(w), _ptr(out), w.shape[0])
    return out


def u3_quantize_pack(x_bits: np.ndarray, src_dtype: int):
    """Rows of 16-bit elements [n, D] -> (packed [n, 3D/8], scale fp16 bits [n], zero [n])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    n, D = x.shape
    packed = np.empty((n, 3 * D // 8), dtype=np.uint8)
    s = np.empty(n, dtype=np.uint16)
    z = np.empty(n, dtype=np.uint8)
    _load().pkvo_u3_quantize_pack_rows(_ptr(x), src_dtype, n, D, _ptr(packed), _ptr(s), _ptr(z))
    return packed, s, z


# --------------------------------------------------------------------------
# slot_mapping ("Write Triton Kv Cache Append Kernel", reasoning step 9)
# --------------------------------------------------------------------------

def build_slot_mapping(block_tables: np.ndarray, req: np.ndarray, pos: np.ndarray,
                       block_size: int) -> np.ndarray:
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    r = np.ascontiguousarray(req, dtype=np.int32)
    p = np.ascontiguousarray(pos, dtype=np.int32)
    out = np.empty(r.shape[0], dtype=np.int64)
    _load().pkvo_build_slot_mapping(_ptr(bt), bt.shape[1], block_size, _ptr(r), _ptr(p),
                                    r.shape[0], _ptr(out))
    return out


# --------------------------------------------------------------------------
# append and decode
# --------------------------------------------------------------------------

def kv_append(cache_dtype: int, src_dtype: int, k_new, v_new, slot_mapping, k_cache, v_cache,
              k_scale=None, v_scale=None, k_qscale=None, k_qzero=None, v_qscale=None,
              v_qzero=None, scale_mode: int = SCALE_PER_HEAD, k_new_scale=None, v_new_scale=None,
              k_scales=None, v_scales=None) -> int:
    """Scatter new rows into the (host, contiguous) cache arrays in place.

    k_new/v_new: uint16 bits [T, Hkv, D]; caches: [P, BS, Hkv, row] uint16 or
    uint8; 3-bit metadata: [P, BS, Hkv].  fp8 / int8 scales: per head
    (k_scale / v_scale [Hkv]), per block (k_scales / v_scales [P, Hkv]) or
    per token (k_new_scale / v_new_scale [T, Hkv], stored into k_scales /
    v_scales [P, BS, Hkv]).  Returns the count of out-of-range slots
    (skipped)."""
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = k_new.shape
    P, BS = k_cache.shape[0], k_cache.shape[1]
    for a in (k_cache, v_cache, k_qscale, k_qzero, v_qscale, v_qzero):
        assert a is None or a.flags["C_CONTIGUOUS"]
    ks = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
    kns = None if k_new_scale is None else np.ascontiguousarray(k_new_scale, dtype=np.float32)
    vns = None if v_new_scale is None else np.ascontiguousarray(v_new_scale, dtype=np.float32)
    for a in (k_scales, v_scales):
        assert a is None or (a.dtype == np.float32 and a.flags["C_CONTIGUOUS"])
    return int(_load().pkvo_kv_append_scaled(
        cache_dtype, src_dtype, T, Hkv, D, _ptr(k_new), _ptr(v_new), _ptr(sm), P, BS,
        _ptr(k_cache), _ptr(v_cache), _ptr(ks), _ptr(vs), _ptr(k_qscale), _ptr(k_qzero),
        _ptr(v_qscale), _ptr(v_qzero), int(scale_mode), _ptr(kns), _ptr(vns), _ptr(k_scales),
        _ptr(v_scales)))


def paged_decode(cache_dtype: int, q_dtype: int, q, k_cache, v_cache, block_tables,
                 context_lens, block_size: int, sm_scale: float, k_scale=None, v_scale=None,
                 k_qscale=None, k_qzero=None, v_qscale=None, v_qzero=None, pairs=None,
                 nthreads: int = 1, scale_mode: int = SCALE_PER_HEAD, k_scales=None, v_scales=None):
    """fp64 paged attention decode.  q: uint16 bits [B, Hq, D].  Returns
    (out float64 [B, Hq, D], bad_rows).  With ``pairs`` (flattened b*Hq+h)
    only those rows are computed; the others are NaN."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    pr = None if pairs is None else np.ascontiguousarray(pairs, dtype=np.int32)
    ks = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
    for a in (k_cache, v_cache):
        assert a.flags["C_CONTIGUOUS"]
    kss = None if k_scales is None else np.ascontiguousarray(k_scales, dtype=np.float32)
    vss = None if v_scales is None else np.ascontiguousarray(v_scales, dtype=np.float32)
    bad = _load().pkvo_paged_decode_scaled(
        cache_dtype, q_dtype, B, Hq, Hkv, D, block_size, _ptr(q), _ptr(k_cache), _ptr(v_cache),
        k_cache.shape[0], _ptr(bt), bt.shape[1], _ptr(cl), float(sm_scale), _ptr(ks), _ptr(vs),
        _ptr(k_qscale), _ptr(k_qzero), _ptr(v_qscale), _ptr(v_qzero), _ptr(pr),
        0 if pr is None else pr.shape[0], _ptr(out), int(nthreads), int(scale_mode), _ptr(kss),
        _ptr(vss))
    return out, int(bad)


# --------------------------------------------------------------------------
# storage layouts
# --------------------------------------------------------------------------

def xvec_elems(elem_bytes: int) -> int:
    """x of the x-vectorised layout: the elements of one 16-byte piece."""
    return 16 // elem_bytes


def to_xvec(cache: np.ndarray, x: int) -> np.ndarray:
    """The older vLLM paged layout with a vectorised inner dimension
    ("Write Triton Kv Cache Append Kernel", "Inputs the agent should gather
    first" item 1): a cache [num_blocks, block_size, num_kv_heads, head_dim]
    is stored as [num_blocks, num_kv_heads, head_dim // x, block_size, x],
    i.e. head_dim is cut into pieces of x consecutive elements and, within a
    block and head, piece c of every slot comes before piece c + 1 of any.
    Element (b, s, h, d) lands at [b, h, d // x, s, d % x]."""
    P, BS, H, D = cache.shape
    assert D % x == 0
    out = np.empty((P, H, D // x, BS, x), dtype=cache.dtype)
    for c in range(D // x):
        # piece c of every (block, slot, head) row, heads before slots
        out[:, :, c, :, :] = cache[:, :, :, c * x:(c + 1) * x].transpose(0, 2, 1, 3)
    return out


def from_xvec(phys: np.ndarray) -> np.ndarray:
    """Inverse of to_xvec: [P, Hkv, D // x, BS, x] -> [P, BS, Hkv, D]."""
    P, H, C, BS, x = phys.shape
    out = np.empty((P, BS, H, C * x), dtype=phys.dtype)
    for c in range(C):
        out[:, :, :, c * x:(c + 1) * x] = phys[:, :, c, :, :].transpose(0, 2, 1, 3)
    return out
