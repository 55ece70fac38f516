"""Python binding of the C ABI in include/pkv.h (ctypes; argument marshalling
only).  Every operation runs in the CUDA kernels of libpkv.so; there is no
fallback: if the library is not built or a call fails, an exception is
raised.  PyTorch provides the device memory and the current stream.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

# dtype codes (pkv.h)
F16, BF16, E4M3, U3, U8, I32, I64, F32, E5M2, I8 = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10
# device error bits
DEVERR_SLOT_RANGE, DEVERR_BLOCK_RANGE, DEVERR_CONTEXT_RANGE, DEVERR_POS_RANGE, DEVERR_TIMEOUT = (
    1, 2, 4, 8, 16)

_TORCH_CODES = {torch.float16: F16, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3,
                torch.float8_e5m2: E5M2, torch.int8: I8,
                torch.uint8: U8, torch.int32: I32, torch.int64: I64, torch.float32: F32}


class PkvError(RuntimeError):
    """A non-OK status from the library (message from pkv_last_error)."""

    def __init__(self, code: int, msg: str):
        super().__init__("pkv error %d: %s" % (code, msg))
        self.code = code


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class _Cache(ctypes.Structure):
    _fields_ = [("k_cache", _Tensor), ("v_cache", _Tensor), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("k_qscale", _Tensor), ("k_qzero", _Tensor),
                ("v_qscale", _Tensor), ("v_qzero", _Tensor), ("scale_mode", ctypes.c_int32),
                ("k_scales", _Tensor), ("v_scales", _Tensor), ("chunk_stride", ctypes.c_int64)]


# scale granularity of fp8 / int8 caches (pkv.h PKV_SCALE_*)
SCALE_MODES = {"head": 0, "block": 1, "token": 2}


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libpkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError("libpkv.so is not built (%s); run "
                                  "paged_kv_cache_num_gb300.build.build()" % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            P = ctypes.c_void_p
            TP = ctypes.POINTER(_Tensor)
            CP = ctypes.POINTER(_Cache)
            L.pkv_version.restype = ctypes.c_char_p
            L.pkv_last_error.restype = ctypes.c_char_p
            L.pkv_abi_version.restype = ctypes.c_int
            L.pkv_slot_mapping.argtypes = [TP, TP, TP, ctypes.c_int, TP, P, P]
            L.pkv_kv_append.argtypes = [TP, TP, TP, CP, P, P]
            L.pkv_kv_append_scaled.argtypes = [TP, TP, TP, TP, TP, CP, P, P]
            L.pkv_paged_decode_workspace.argtypes = [TP, CP, TP, ctypes.c_int,
                                                     ctypes.POINTER(ctypes.c_size_t)]
            L.pkv_paged_decode_launches.argtypes = [TP, CP, TP, ctypes.c_int,
                                                    ctypes.POINTER(ctypes.c_int32)]
            L.pkv_paged_decode.argtypes = [TP, CP, TP, TP, ctypes.c_float, TP, ctypes.c_int, P,
                                           ctypes.c_size_t, P, P]
            L.pkv_paged_decode_noalloc.argtypes = [TP, CP, TP, TP, ctypes.c_float, TP,
                                                   ctypes.c_int, P, P]
            L.pkv_decode_step.argtypes = [TP, TP, TP, TP, TP, TP, CP, TP, TP, ctypes.c_float, TP,
                                          ctypes.c_int, P, ctypes.c_size_t, P, P]
            L.pkv_noalloc_scratch_bytes.restype = ctypes.c_size_t
            L.pkv_pack3.argtypes = [P, P, ctypes.c_int64, P]
            L.pkv_unpack3.argtypes = [P, P, ctypes.c_int64, P]
            L.pkv_unpack3_words.argtypes = [P, P, ctypes.c_int64, P]
            L.pkv_copy_peak.argtypes = [P, P, ctypes.c_size_t, P]
            for fn in ("pkv_slot_mapping", "pkv_kv_append", "pkv_kv_append_scaled",
                       "pkv_paged_decode_workspace", "pkv_paged_decode_launches",
                       "pkv_paged_decode", "pkv_paged_decode_noalloc", "pkv_decode_step", "pkv_pack3",
                       "pkv_unpack3", "pkv_unpack3_words", "pkv_copy_peak"):
                getattr(L, fn).restype = ctypes.c_int
            _lib = L
    return _lib


def _check(rc: int):
    if rc != 0:
        raise PkvError(rc, lib().pkv_last_error().decode())


def _desc(t: Optional[torch.Tensor], code: Optional[int] = None) -> _Tensor:
    d = _Tensor()
    if t is None:
        return d
    if t.dim() > 4:
        raise ValueError("at most 4 dims")
    d.data = t.data_ptr() if t.numel() > 0 else 0
    d.dtype = _TORCH_CODES[t.dtype] if code is None else code
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _xvec_desc(t: torch.Tensor, code: int) -> _Tensor:
    if t.dim() != 5 or t.stride(4) != 1:
        raise ValueError("an xvec cache is [num_blocks, Hkv, head_dim // x, block_size, x], x contiguous")
    d = _Tensor()
    d.data = t.data_ptr() if t.numel() > 0 else 0
    d.dtype = code
    d.ndim = 4
    P, H, C, BS, x = t.shape
    for i, (n, st) in enumerate(((P, t.stride(0)), (BS, t.stride(3)), (H, t.stride(1)), (C * x, 1))):
        d.shape[i] = n
        d.stride[i] = st
    return d


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")


@dataclass
class KVCache:
    """A paged KV cache [num_blocks, block_size, num_kv_heads, row] in device
    memory.  kind: "f16", "bf16", "e4m3" / "e5m2" / "i8" (+ per-kv-head fp32 scales) or "u3"
    (3-bit codes, row = 3*head_dim/8 bytes, + fp16 scale / uint8 zero per
    (slot, head)).  layout "xvec" (16-bit and one-byte kinds): k_cache /
    v_cache are stored [num_blocks, num_kv_heads, head_dim // x, block_size,
    x] with x = 16 bytes / element size."""
    kind: str
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None
    k_qscale: Optional[torch.Tensor] = None
    k_qzero: Optional[torch.Tensor] = None
    v_qscale: Optional[torch.Tensor] = None
    v_qzero: Optional[torch.Tensor] = None
    # fp8 / int8 scale granularity: "head" (k_scale / v_scale [Hkv]), "block"
    # (k_scales / v_scales fp32 [num_blocks, Hkv]) or "token" (fp32
    # [num_blocks, block_size, Hkv], filled by kv_append_scaled)
    scale_mode: str = "head"
    k_scales: Optional[torch.Tensor] = None
    v_scales: Optional[torch.Tensor] = None
    layout: str = "flash"

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]

    @property
    def block_size(self):
        return self.k_cache.shape[3 if self.layout == "xvec" else 1]

    @property
    def num_kv_heads(self):
        return self.k_cache.shape[1 if self.layout == "xvec" else 2]

    @property
    def head_dim(self):
        if self.layout == "xvec":
            return self.k_cache.shape[2] * self.k_cache.shape[4]
        r = self.k_cache.shape[3]
        return r * 8 // 3 if self.kind == "u3" else r

    @staticmethod
    def allocate(kind: str, num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                 device="cuda", k_scale=None, v_scale=None, fill=None, scale_mode: str = "head",
                 k_scales=None, v_scales=None, layout: str = "flash") -> "KVCache":
        """A cache of `kind`; fp8 / int8 caches take per-head scales (k_scale,
        v_scale), per-block scales (scale_mode "block": k_scales / v_scales
        [num_blocks, Hkv]) or per-token scales (scale_mode "token": arrays
        allocated here, written by kv_append_scaled).  layout "xvec": the
        x-vectorised storage [num_blocks, Hkv, head_dim // x, block_size, x]."""
        shape = (num_blocks, block_size, num_kv_heads)
        if layout == "xvec":
            if kind not in ("f16", "bf16", "e4m3", "e5m2", "i8"):
                raise ValueError("layout xvec applies to 16-bit and one-byte caches")
            dt = {"f16": torch.float16, "bf16": torch.bfloat16, "i8": torch.int8}.get(kind, torch.uint8)
            x = 16 // torch.empty((), dtype=dt).element_size()
            if head_dim % x:
                raise ValueError("head_dim must be a multiple of x = %d" % x)
            k = torch.empty((num_blocks, num_kv_heads, head_dim // x, block_size, x), dtype=dt,
                            device=device)
            v = torch.empty_like(k)
            c = KVCache(kind, k, v, k_scale=k_scale, v_scale=v_scale, scale_mode=scale_mode,
                        layout="xvec")
            if scale_mode == "block":
                c.k_scales, c.v_scales = k_scales, v_scales
            elif scale_mode == "token":
                hm = (num_blocks, num_kv_heads, block_size)
                c.k_scales = torch.ones(hm, dtype=torch.float32, device=device).permute(0, 2, 1)
                c.v_scales = torch.ones(hm, dtype=torch.float32, device=device).permute(0, 2, 1)
            if fill is not None:
                for t in (k, v):
                    t.view(torch.uint8).fill_(fill)
            return c
        elif layout != "flash":
            raise ValueError(layout)
        if kind in ("f16", "bf16"):
            dt = torch.float16 if kind == "f16" else torch.bfloat16
            k = torch.empty(shape + (head_dim,), dtype=dt, device=device)
            v = torch.empty_like(k)
            c = KVCache(kind, k, v)
        elif kind in ("e4m3", "e5m2", "i8"):
            k = torch.empty(shape + (head_dim,), dtype=torch.int8 if kind == "i8" else torch.uint8,
                            device=device)
            v = torch.empty_like(k)
            c = KVCache(kind, k, v, k_scale=k_scale, v_scale=v_scale, scale_mode=scale_mode)
            if scale_mode == "block":
                c.k_scales, c.v_scales = k_scales, v_scales
            elif scale_mode == "token":
                # head-major storage behind a [num_blocks, block_size, Hkv] view,
                # as the 3-bit metadata: a decode CTA stages its heads' runs
                hm = (num_blocks, num_kv_heads, block_size)
                c.k_scales = torch.ones(hm, dtype=torch.float32, device=device).permute(0, 2, 1)
                c.v_scales = torch.ones(hm, dtype=torch.float32, device=device).permute(0, 2, 1)
        elif kind == "u3":
            k = torch.empty(shape + (3 * head_dim // 8,), dtype=torch.uint8, device=device)
            v = torch.empty_like(k)
            # scale / zero stored head-major ([num_blocks, num_kv_heads,
            # block_size]) and seen through a [num_blocks, block_size,
            # num_kv_heads] view: a decode CTA then stages only its own heads'
            # runs of each block
            meta = (num_blocks, num_kv_heads, block_size)
            phys = [torch.empty(meta, dtype=dt, device=device)
                    for dt in (torch.float16, torch.uint8, torch.float16, torch.uint8)]
            ks_, kz_, vs_, vz_ = (t.permute(0, 2, 1) for t in phys)
            c = KVCache(kind, k, v, k_qscale=ks_, k_qzero=kz_, v_qscale=vs_, v_qzero=vz_)
        else:
            raise ValueError(kind)
        if fill is not None:
            for t in [c.k_cache, c.v_cache] + (phys if kind == "u3" else []):
                t.view(torch.uint8).fill_(fill)
        return c

    def _struct(self) -> _Cache:
        key = tuple((t.data_ptr(), t.dtype, t.shape, t.stride()) for t in self.tensors())
        cached = self.__dict__.get("_cstruct")
        if cached is not None and cached[0] == key:
            return cached[1]
        s = self._build_struct()
        self.__dict__["_cstruct"] = (key, s)
        return s

    def _build_struct(self) -> _Cache:
        s = _Cache()
        code = {"f16": F16, "bf16": BF16, "e4m3": E4M3, "e5m2": E5M2, "i8": I8, "u3": U3}[self.kind]
        if self.layout == "xvec":
            # [P, Hkv, D/x, BS, x] described as [P, BS, Hkv, D] + the piece stride
            s.k_cache = _xvec_desc(self.k_cache, code)
            s.v_cache = _xvec_desc(self.v_cache, code)
            s.chunk_stride = self.k_cache.stride(2)
        else:
            s.k_cache = _desc(self.k_cache, code)
            s.v_cache = _desc(self.v_cache, code)
        if self.kind in ("e4m3", "e5m2", "i8") and self.scale_mode == "head":
            if self.k_scale is None or self.v_scale is None:
                raise ValueError("fp8 / int8 cache needs k_scale / v_scale")
            s.k_scale = self.k_scale.data_ptr()
            s.v_scale = self.v_scale.data_ptr()
        if self.kind == "u3":
            s.k_qscale = _desc(self.k_qscale, F16)
            s.k_qzero = _desc(self.k_qzero, U8)
            s.v_qscale = _desc(self.v_qscale, F16)
            s.v_qzero = _desc(self.v_qzero, U8)
        s.scale_mode = SCALE_MODES[self.scale_mode]
        if self.scale_mode != "head":
            s.k_scales = _desc(self.k_scales, F32)
            s.v_scales = _desc(self.v_scales, F32)
        return s

    def tensors(self):
        return [t for t in (self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.k_qscale,
                            self.k_qzero, self.v_qscale, self.v_qzero, self.k_scales,
                            self.v_scales) if t is not None]


def version() -> str:
    return lib().pkv_version().decode()


def slot_mapping(block_tables, req, pos, block_size: int, out=None, err_flag=None, stream=None):
    """slot = block_tables[req][pos // bs] * bs + pos % bs (pos < 0 -> -1), on the GPU."""
    _need_cuda(block_tables, req, pos)
    if out is None:
        out = torch.empty(req.shape[0], dtype=torch.int64, device=req.device)
    _check(lib().pkv_slot_mapping(ctypes.byref(_desc(block_tables)), ctypes.byref(_desc(req)),
                                  ctypes.byref(_desc(pos)), int(block_size),
                                  ctypes.byref(_desc(out)), _ptr(err_flag), _stream(stream)))
    return out


def kv_append(k_new, v_new, slot_mapping, cache: KVCache, err_flag=None, stream=None):
    """Scatter new K/V rows [T, Hkv, D] into the cache through slot_mapping."""
    _need_cuda(k_new, v_new, slot_mapping, *cache.tensors())
    cs = cache._struct()
    _check(lib().pkv_kv_append(ctypes.byref(_desc(k_new)), ctypes.byref(_desc(v_new)),
                               ctypes.byref(_desc(slot_mapping)), ctypes.byref(cs),
                               _ptr(err_flag), _stream(stream)))


def kv_append_scaled(k_new, v_new, k_new_scale, v_new_scale, slot_mapping, cache: KVCache,
                     err_flag=None, stream=None):
    """kv_append for a cache with per-token scales: k_new_scale / v_new_scale
    fp32 [num_tokens, Hkv] are divided out and stored at the tokens' slots."""
    _need_cuda(k_new, v_new, k_new_scale, v_new_scale, slot_mapping, *cache.tensors())
    _check(lib().pkv_kv_append_scaled(ctypes.byref(_desc(k_new)), ctypes.byref(_desc(v_new)),
                                      ctypes.byref(_desc(k_new_scale)), ctypes.byref(_desc(v_new_scale)),
                                      ctypes.byref(_desc(slot_mapping)), ctypes.byref(cache._struct()),
                                      _ptr(err_flag), _stream(stream)))


def decode_workspace_bytes(q, cache: KVCache, block_tables, num_splits: int = 0) -> int:
    n = ctypes.c_size_t(0)
    cs = cache._struct()
    _check(lib().pkv_paged_decode_workspace(ctypes.byref(_desc(q)), ctypes.byref(cs),
                                            ctypes.byref(_desc(block_tables)), int(num_splits),
                                            ctypes.byref(n)))
    return int(n.value)


def decode_launches(q, cache: KVCache, block_tables, num_splits: int = 0) -> int:
    """Kernel launches one paged_decode call with these arguments makes."""
    n = ctypes.c_int32(0)
    _check(lib().pkv_paged_decode_launches(ctypes.byref(_desc(q)), ctypes.byref(cache._struct()),
                                           ctypes.byref(_desc(block_tables)), int(num_splits),
                                           ctypes.byref(n)))
    return int(n.value)


def paged_decode(q, cache: KVCache, block_tables, context_lens, sm_scale: Optional[float] = None,
                 out=None, num_splits: int = 0, workspace=None, err_flag=None, stream=None):
    """softmax(sm_scale * q . K^T) V over each sequence's paged context."""
    _need_cuda(q, block_tables, context_lens, *cache.tensors())
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(q.shape[-1])
    if out is None:
        out = torch.empty_like(q)
    cs = cache._struct()
    if workspace is None:
        need = decode_workspace_bytes(q, cache, block_tables, num_splits)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = None if workspace is None else ctypes.c_void_p(workspace.data_ptr())
    ws_n = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pkv_paged_decode(ctypes.byref(_desc(q)), ctypes.byref(cs),
                                  ctypes.byref(_desc(block_tables)),
                                  ctypes.byref(_desc(context_lens)), float(sm_scale),
                                  ctypes.byref(_desc(out)), int(num_splits), ws_ptr, ws_n,
                                  _ptr(err_flag), _stream(stream)))
    return out


def decode_step(k_new, v_new, req, pos, q, cache: KVCache, block_tables, context_lens,
                sm_scale: Optional[float] = None, out=None, slots=None, num_splits: int = 0,
                workspace=None, err_flag=None, stream=None):
    """slot_mapping + kv_append + paged_decode in one library call (see
    pkv_decode_step in pkv.h); returns out.  `slots` (int64 [num_tokens])
    receives the slot mapping."""
    _need_cuda(k_new, v_new, req, pos, q, block_tables, context_lens, *cache.tensors())
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(q.shape[-1])
    if out is None:
        out = torch.empty_like(q)
    if slots is None:
        slots = torch.empty(req.shape[0], dtype=torch.int64, device=q.device)
    cs = cache._struct()
    if workspace is None:
        need = decode_workspace_bytes(q, cache, block_tables, num_splits)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = None if workspace is None else ctypes.c_void_p(workspace.data_ptr())
    ws_n = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pkv_decode_step(ctypes.byref(_desc(k_new)), ctypes.byref(_desc(v_new)),
                                 ctypes.byref(_desc(req)), ctypes.byref(_desc(pos)),
                                 ctypes.byref(_desc(slots)), ctypes.byref(_desc(q)), ctypes.byref(cs),
                                 ctypes.byref(_desc(block_tables)), ctypes.byref(_desc(context_lens)),
                                 float(sm_scale), ctypes.byref(_desc(out)), int(num_splits), ws_ptr,
                                 ws_n, _ptr(err_flag), _stream(stream)))
    return out


def paged_decode_noalloc(q, cache: KVCache, block_tables, context_lens,
                         sm_scale: Optional[float] = None, out=None, num_splits: int = 0,
                         err_flag=None, stream=None):
    """paged_decode without a caller workspace: the split-K scratch is the
    library's fixed device array (see pkv_paged_decode_noalloc in pkv.h)."""
    _need_cuda(q, block_tables, context_lens, *cache.tensors())
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(q.shape[-1])
    if out is None:
        out = torch.empty_like(q)
    cs = cache._struct()
    _check(lib().pkv_paged_decode_noalloc(ctypes.byref(_desc(q)), ctypes.byref(cs),
                                          ctypes.byref(_desc(block_tables)),
                                          ctypes.byref(_desc(context_lens)), float(sm_scale),
                                          ctypes.byref(_desc(out)), int(num_splits),
                                          _ptr(err_flag), _stream(stream)))
    return out


def pack3(values, packed=None, stream=None):
    """uint8 [n*8] codes -> uint8 [n*3] packed bytes."""
    _need_cuda(values)
    n = values.numel() // 8
    if packed is None:
        packed = torch.empty(n * 3, dtype=torch.uint8, device=values.device)
    _check(lib().pkv_pack3(_ptr(values), _ptr(packed), n, _stream(stream)))
    return packed


def unpack3(packed, values=None, stream=None):
    """uint8 [n*3] packed bytes -> uint8 [n*8] codes."""
    _need_cuda(packed)
    n = packed.numel() // 3
    if values is None:
        values = torch.empty(n * 8, dtype=torch.uint8, device=packed.device)
    _check(lib().pkv_unpack3(_ptr(packed), _ptr(values), n, _stream(stream)))
    return values


def unpack3_words(words, values=None, stream=None):
    """int32/uint32 words [m*3] (same bytes as packed octets) -> uint8 [m*32]."""
    _need_cuda(words)
    m = words.numel() // 3
    if values is None:
        values = torch.empty(m * 32, dtype=torch.uint8, device=words.device)
    _check(lib().pkv_unpack3_words(_ptr(words), _ptr(values), m, _stream(stream)))
    return values


def copy_peak(src, dst, stream=None):
    """16-byte vectorised copy of src's bytes into dst (bandwidth yardstick)."""
    _need_cuda(src, dst)
    nbytes = src.numel() * src.element_size()
    _check(lib().pkv_copy_peak(_ptr(src), _ptr(dst), nbytes, _stream(stream)))
