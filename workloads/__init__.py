"""Seeded synthetic inputs for the paged KV-cache hot path.

This module only draws random numbers and lays them out; it holds none of
the method's arithmetic (no slot computation, no quantisation, no attention).
Both the CUDA path and the CPU oracle are fed from the same tensors it
returns, so they see identical bytes.

Every workload is the shape and value distribution stated for it, drawn with
a torch generator seeded per workload (tiny case: 42, then 43, 44, ...).
Host generation (``device="cpu"``) is used by the parity tests; the
benchmark draws the same recipe on the GPU with torch's CUDA generator, which
gives different numbers from the same seed (parity never mixes the two).

Workloads (names used by the tests and the benchmark):
  tiny_fp16      batch 2, 4 heads (MHA), head_dim 64, block 16, 20 blocks,
                 5 blocks/seq, context [10, 25], distinct random block ids;
                 2 tokens appended at position context-1 (seed 42).
  tiny_literal   the same with the block tables [[5,0,0,0,0],[12,3,0,0,0]].
  gqa_bf16       batch 64, 32 q / 8 kv heads, head_dim 128, block 16,
                 context U{512..4096}, pool = needed blocks + 10 %, block
                 tables a random permutation of the pool; 64 appended tokens.
  mixed_append   bf16, 8 kv heads, head_dim 128, block 32: 8 prefill
                 requests U{128..2048} tokens at positions 0..len-1 plus 56
                 decode requests (context U{512..4096}, one token at
                 context-1), padded with -1 slots (NaN source rows) to a
                 multiple of 256; pool pre-filled with random bytes.
  fp8_long       batch 16, 64 q / 8 kv heads, head_dim 128, block 32, bf16 q,
                 context U{16384..32768}; e4m3 cache with per-kv-head fp32
                 scales amax/448 from a separate N(0,1) calibration tensor
                 [4096, 8, 128] (one for K, one for V); the context is filled
                 by appending N(0,1) rows, then 16 new tokens are appended.
  u3_mha         batch 32, 32 heads (MHA), head_dim 128, block 16, fp16,
                 context U{1024..8192}; 3-bit packed cache filled by
                 appending N(0,1) rows, then 32 new tokens.
  mha_short      the benchmark shape of "10. Triton KV Cache and
                 PagedAttention": batch 32, 32 heads (MHA), head_dim 128,
                 block 16, fp16, a 2048-block pool of N(0,1) K/V, context
                 U{100..999}, blocks allocated one after another (sequence
                 b's blocks follow sequence b-1's); 32 new tokens appended.

Token lists are given as (request index, position) pairs; a position of -1
marks a padding token.  The slot of a token is computed by the code under
test (or by the oracle), not here.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional

import torch

SEEDS = {"tiny_fp16": 42, "tiny_literal": 42, "gqa_bf16": 43, "mixed_append": 44,
         "fp8_long": 45, "u3_mha": 46, "mha_short": 47, "fp8_long_e5m2": 48, "i8_long": 49,
         "fp8_long_token_scales": 50, "fp8_long_block_scales": 51,
         "gqa_bf16_xvec": 43, "fp8_long_xvec": 45, "fp8_long_g16": 52,
         "gqa_bf16_g16": 53, "fp8_long_d64": 54, "u3_g16": 55, "u3_g8": 56}


@dataclass
class Workload:
    name: str
    dtype: torch.dtype              # q / new K,V / 16-bit cache dtype
    cache_kind: str                 # "f16", "bf16", "e4m3", "u3"
    batch: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: torch.Tensor      # int32 [B] (tokens attended, newest included)
    block_tables: torch.Tensor      # int32 [B, max_blocks]
    q: Optional[torch.Tensor]       # [B, Hq, D] or None (append-only workloads)
    # tokens appended in the step: request index / position, and their rows
    new_req: torch.Tensor           # int32 [T]
    new_pos: torch.Tensor           # int32 [T] (-1 = padding)
    k_new: torch.Tensor             # [T, Hkv, D]
    v_new: torch.Tensor
    # initial cache contents (16-bit caches) or None when filled by append
    k_cache0: Optional[torch.Tensor] = None
    v_cache0: Optional[torch.Tensor] = None
    # context fill by append (quantised caches): request / position / rows
    fill_req: Optional[torch.Tensor] = None
    fill_pos: Optional[torch.Tensor] = None
    k_fill: Optional[torch.Tensor] = None
    v_fill: Optional[torch.Tensor] = None
    k_scale: Optional[torch.Tensor] = None   # fp32 [Hkv] (fp8 / int8, per-head scales)
    v_scale: Optional[torch.Tensor] = None
    # fp8 / int8 scale granularity: "head" (k_scale / v_scale), "block"
    # (k_block_scale / v_block_scale [P, Hkv]) or "token" (one scale per
    # appended row: k_fill_scale [n_fill, Hkv], k_new_scale [T, Hkv], ...)
    scale_mode: str = "head"
    k_block_scale: Optional[torch.Tensor] = None
    v_block_scale: Optional[torch.Tensor] = None
    k_fill_scale: Optional[torch.Tensor] = None
    v_fill_scale: Optional[torch.Tensor] = None
    k_new_scale: Optional[torch.Tensor] = None
    v_new_scale: Optional[torch.Tensor] = None
    extra: Dict[str, object] = field(default_factory=dict)
    # cache storage: "flash" [P, BS, Hkv, D] or "xvec" [P, Hkv, D // x, BS, x]
    # (the same logical contents; only where each element is stored differs)
    layout: str = "flash"

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def sm_scale(self) -> float:
        # 1/sqrt(head_dim) unless set, rounded to fp32 (the value both sides receive)
        v = self.extra.get("sm_scale", 1.0 / math.sqrt(self.head_dim))
        return float(torch.tensor(v, dtype=torch.float32))

    @sm_scale.setter
    def sm_scale(self, v: float) -> None:
        self.extra["sm_scale"] = float(v)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, dtype, chunk_elems=1 << 26):
    """N(0,1) drawn in fp32 and cast to ``dtype``; drawn in chunks along the
    first dimension so big pools do not need a full fp32 copy."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(shape[0], -1)
    per = max(1, chunk_elems // max(1, flat.shape[1]))
    for i in range(0, shape[0], per):
        j = min(shape[0], i + per)
        flat[i:j] = torch.randn((j - i, flat.shape[1]), generator=g, device=device,
                                dtype=torch.float32).to(dtype)
    return out


def _randint(lo, hi_incl, n, g, device):
    return torch.randint(lo, hi_incl + 1, (n,), generator=g, device=device, dtype=torch.int64)


def _tables_from_permutation(nblocks_per_seq, max_blocks, pool, g, device):
    """Block tables whose used entries are the first sum(n) ids of a random
    permutation of the pool; unused entries are 0."""
    B = len(nblocks_per_seq)
    perm = torch.randperm(pool, generator=g, device=device).to(torch.int32)
    bt = torch.zeros((B, max_blocks), dtype=torch.int32, device=device)
    off = 0
    for b, n in enumerate(nblocks_per_seq):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt


def _cdiv(a, b):
    return -(-a // b)


def tiny(literal: bool = False, device="cpu") -> Workload:
    """The tiny fp16 case (seed 42)."""
    g = _gen(SEEDS["tiny_fp16"], device)
    B, H, D, BS, P, MB = 2, 4, 64, 16, 20, 5
    dt = torch.float16
    q = _randn((B, H, D), g, device, dt)
    k_cache0 = _randn((P, BS, H, D), g, device, dt)
    v_cache0 = _randn((P, BS, H, D), g, device, dt)
    ctx = torch.tensor([10, 25], dtype=torch.int32, device=device)
    if literal:
        bt = torch.tensor([[5, 0, 0, 0, 0], [12, 3, 0, 0, 0]], dtype=torch.int32, device=device)
    else:
        nb = [_cdiv(int(c), BS) for c in ctx.tolist()]
        ids = torch.randperm(P, generator=g, device=device).to(torch.int32)
        bt = torch.zeros((B, MB), dtype=torch.int32, device=device)
        off = 0
        for b, n in enumerate(nb):
            bt[b, :n] = ids[off:off + n]
            off += n
    k_new = _randn((B, H, D), g, device, dt)
    v_new = _randn((B, H, D), g, device, dt)
    new_req = torch.arange(B, dtype=torch.int32, device=device)
    new_pos = (ctx - 1).to(torch.int32)
    return Workload("tiny_literal" if literal else "tiny_fp16", dt, "f16", B, H, H, D, BS, P,
                    ctx, bt, q, new_req, new_pos, k_new, v_new, k_cache0, v_cache0)


def gqa_bf16(device="cpu", batch=64, ctx_lo=512, ctx_hi=4096, num_heads=32, num_kv_heads=8,
             head_dim=128, block_size=16, seed=None, layout="flash") -> Workload:
    """Llama-3-8B-like GQA decode step, bf16 (defaults: the full-size case).
    layout="xvec": the same data stored x-vectorised."""
    g = _gen(SEEDS["gqa_bf16"] if seed is None else seed, device)
    dt = torch.bfloat16
    B, Hq, Hkv, D, BS = batch, num_heads, num_kv_heads, head_dim, block_size
    ctx = _randint(ctx_lo, ctx_hi, B, g, device).to(torch.int32)
    nb = [_cdiv(int(c), BS) for c in ctx.tolist()]
    MB = _cdiv(ctx_hi, BS)
    P = _cdiv(11 * sum(nb), 10)
    bt = _tables_from_permutation(nb, MB, P, g, device)
    q = _randn((B, Hq, D), g, device, dt)
    k_cache0 = _randn((P, BS, Hkv, D), g, device, dt)
    v_cache0 = _randn((P, BS, Hkv, D), g, device, dt)
    k_new = _randn((B, Hkv, D), g, device, dt)
    v_new = _randn((B, Hkv, D), g, device, dt)
    new_req = torch.arange(B, dtype=torch.int32, device=device)
    new_pos = (ctx - 1).to(torch.int32)
    w = Workload("gqa_bf16", dt, "bf16", B, Hq, Hkv, D, BS, P, ctx, bt, q, new_req, new_pos,
                 k_new, v_new, k_cache0, v_cache0)
    w.extra["context"] = "U{%d..%d}" % (ctx_lo, ctx_hi)
    w.layout = layout
    return w


def mixed_append(device="cpu", n_prefill=8, n_decode=56, prefill_lo=128, prefill_hi=2048,
                 ctx_lo=512, ctx_hi=4096, num_kv_heads=8, head_dim=128, block_size=32,
                 pad_to=256, seed=None) -> Workload:
    """Mixed prefill + decode append, bf16, padded with -1 slots."""
    g = _gen(SEEDS["mixed_append"] if seed is None else seed, device)
    dt = torch.bfloat16
    Hkv, D, BS = num_kv_heads, head_dim, block_size
    plen = _randint(prefill_lo, prefill_hi, n_prefill, g, device).tolist()
    dctx = _randint(ctx_lo, ctx_hi, n_decode, g, device).tolist()
    lens = plen + dctx                      # tokens each request holds after the step
    B = len(lens)
    nb = [_cdiv(int(n), BS) for n in lens]
    MB = max(nb)
    P = _cdiv(11 * sum(nb), 10)
    bt = _tables_from_permutation(nb, MB, P, g, device)
    req, pos = [], []
    for r, n in enumerate(plen):
        req += [r] * n
        pos += list(range(n))
    for i, c in enumerate(dctx):
        req.append(n_prefill + i)
        pos.append(c - 1)
    n_real = len(req)
    T = _cdiv(n_real, pad_to) * pad_to
    req += [0] * (T - n_real)
    pos += [-1] * (T - n_real)
    new_req = torch.tensor(req, dtype=torch.int32, device=device)
    new_pos = torch.tensor(pos, dtype=torch.int32, device=device)
    k_new = _randn((T, Hkv, D), g, device, dt)
    v_new = _randn((T, Hkv, D), g, device, dt)
    k_new[n_real:] = float("nan")
    v_new[n_real:] = float("nan")
    pool_bytes = P * BS * Hkv * D * 2
    k_cache0 = torch.randint(0, 256, (pool_bytes,), generator=g, device=device,
                             dtype=torch.uint8).view(dt).view(P, BS, Hkv, D)
    v_cache0 = torch.randint(0, 256, (pool_bytes,), generator=g, device=device,
                             dtype=torch.uint8).view(dt).view(P, BS, Hkv, D)
    ctx = torch.tensor(lens, dtype=torch.int32, device=device)
    w = Workload("mixed_append", dt, "bf16", B, Hkv, Hkv, D, BS, P, ctx, bt, None, new_req,
                 new_pos, k_new, v_new, k_cache0, v_cache0)
    w.extra["n_real_tokens"] = n_real
    w.extra["context"] = "prefill U{%d..%d} + decode U{%d..%d}" % (prefill_lo, prefill_hi, ctx_lo,
                                                                   ctx_hi)
    return w


def _fill_lists(ctx_list, device):
    """(request, position) of every context token before the newest one."""
    req = torch.cat([torch.full((c - 1,), b, dtype=torch.int32) for b, c in enumerate(ctx_list)])
    pos = torch.cat([torch.arange(c - 1, dtype=torch.int32) for c in ctx_list])
    return req.to(device), pos.to(device)


def fp8_long(device="cpu", batch=16, ctx_lo=16384, ctx_hi=32768, num_heads=64, num_kv_heads=8,
             head_dim=128, block_size=32, calib_tokens=4096, seed=None,
             fp8="e4m3", scales="head", layout="flash") -> Workload:
    """Long-context quantised cache with per-kv-head scales amax / (the
    format's largest value): 448 for e4m3 (defaults: the full-size case),
    57344 for e5m2, 127 for int8 ("i8").  scales="block": each block's scale
    per head is the head's calibration scale times U[1, 1.5]; scales="token":
    each appended row's own amax / max, a caller-side dynamic calibration."""
    g = _gen(SEEDS["fp8_long"] if seed is None else seed, device)
    dt = torch.bfloat16
    B, Hq, Hkv, D, BS = batch, num_heads, num_kv_heads, head_dim, block_size
    ctx = _randint(ctx_lo, ctx_hi, B, g, device).to(torch.int32)
    ctx_list = ctx.tolist()
    nb = [_cdiv(int(c), BS) for c in ctx_list]
    MB = _cdiv(ctx_hi, BS)
    P = _cdiv(11 * sum(nb), 10)
    bt = _tables_from_permutation(nb, MB, P, g, device)
    q = _randn((B, Hq, D), g, device, dt)
    k_cal = _randn((calib_tokens, Hkv, D), g, device, dt)
    v_cal = _randn((calib_tokens, Hkv, D), g, device, dt)
    # calibration: per-kv-head amax / max-finite in fp32
    fmax = {"e4m3": 448.0, "e5m2": 57344.0, "i8": 127.0}[fp8]
    k_scale = k_cal.float().abs().amax(dim=(0, 2)) / fmax
    v_scale = v_cal.float().abs().amax(dim=(0, 2)) / fmax
    fill_req, fill_pos = _fill_lists(ctx_list, device)
    n_fill = int(fill_req.shape[0])
    k_fill = _randn((n_fill, Hkv, D), g, device, dt)
    v_fill = _randn((n_fill, Hkv, D), g, device, dt)
    k_new = _randn((B, Hkv, D), g, device, dt)
    v_new = _randn((B, Hkv, D), g, device, dt)
    new_req = torch.arange(B, dtype=torch.int32, device=device)
    new_pos = (ctx - 1).to(torch.int32)
    w = Workload("fp8_long", dt, fp8, B, Hq, Hkv, D, BS, P, ctx, bt, q, new_req, new_pos,
                 k_new, v_new, fill_req=fill_req, fill_pos=fill_pos, k_fill=k_fill,
                 v_fill=v_fill, k_scale=k_scale.contiguous(), v_scale=v_scale.contiguous())
    w.scale_mode = scales
    if scales == "block":
        w.k_block_scale = (k_scale[None, :] * (1 + 0.5 * torch.rand((P, Hkv), generator=g, device=device))).contiguous()
        w.v_block_scale = (v_scale[None, :] * (1 + 0.5 * torch.rand((P, Hkv), generator=g, device=device))).contiguous()
    elif scales == "token":
        def row_scale(x):          # per (token, head) amax / max, never 0
            return (x.float().abs().amax(dim=2) / fmax).clamp_min(2.0 ** -60).contiguous()
        w.k_fill_scale, w.v_fill_scale = row_scale(k_fill), row_scale(v_fill)
        w.k_new_scale, w.v_new_scale = row_scale(k_new), row_scale(v_new)
    w.extra["context"] = "U{%d..%d}" % (ctx_lo, ctx_hi)
    w.layout = layout
    return w


def u3_mha(device="cpu", batch=32, ctx_lo=1024, ctx_hi=8192, num_heads=32, head_dim=128,
           block_size=16, seed=None, num_kv_heads=None) -> Workload:
    """3-bit packed cache, fp16: MHA (defaults: the full-size case), or
    grouped q heads with num_kv_heads < num_heads."""
    g = _gen(SEEDS["u3_mha"] if seed is None else seed, device)
    dt = torch.float16
    B, H, D, BS = batch, num_heads, head_dim, block_size
    Hkv = H if num_kv_heads is None else num_kv_heads
    ctx = _randint(ctx_lo, ctx_hi, B, g, device).to(torch.int32)
    ctx_list = ctx.tolist()
    nb = [_cdiv(int(c), BS) for c in ctx_list]
    MB = _cdiv(ctx_hi, BS)
    P = _cdiv(11 * sum(nb), 10)
    bt = _tables_from_permutation(nb, MB, P, g, device)
    q = _randn((B, H, D), g, device, dt)
    fill_req, fill_pos = _fill_lists(ctx_list, device)
    n_fill = int(fill_req.shape[0])
    k_fill = _randn((n_fill, Hkv, D), g, device, dt)
    v_fill = _randn((n_fill, Hkv, D), g, device, dt)
    k_new = _randn((B, Hkv, D), g, device, dt)
    v_new = _randn((B, Hkv, D), g, device, dt)
    new_req = torch.arange(B, dtype=torch.int32, device=device)
    new_pos = (ctx - 1).to(torch.int32)
    w = Workload("u3_mha" if Hkv == H else "u3_gqa", dt, "u3", B, H, Hkv, D, BS, P, ctx, bt, q, new_req, new_pos,
                 k_new, v_new, fill_req=fill_req, fill_pos=fill_pos, k_fill=k_fill,
                 v_fill=v_fill)
    w.extra["context"] = "U{%d..%d}" % (ctx_lo, ctx_hi)
    return w


def mha_short(device="cpu", batch=32, num_heads=32, head_dim=128, block_size=16, num_blocks=2048,
              ctx_lo=100, ctx_hi=999, seed=None) -> Workload:
    """MHA fp16 decode over a pool of random K/V with contiguously allocated
    block tables (defaults: the page's benchmark shape)."""
    g = _gen(SEEDS["mha_short"] if seed is None else seed, device)
    dt = torch.float16
    B, H, D, BS, P = batch, num_heads, head_dim, block_size, num_blocks
    ctx = _randint(ctx_lo, ctx_hi, B, g, device).to(torch.int32)
    nb = [_cdiv(int(c), BS) for c in ctx.tolist()]
    if sum(nb) > P:
        raise ValueError("pool of %d blocks holds fewer than the %d needed" % (P, sum(nb)))
    MB = _cdiv(ctx_hi, BS)
    bt = torch.zeros((B, MB), dtype=torch.int32, device=device)
    off = 0
    for b, n in enumerate(nb):
        bt[b, :n] = torch.arange(off, off + n, dtype=torch.int32, device=device)
        off += n
    q = _randn((B, H, D), g, device, dt)
    k0 = _randn((P, BS, H, D), g, device, dt)
    v0 = _randn((P, BS, H, D), g, device, dt)
    k_new = _randn((B, H, D), g, device, dt)
    v_new = _randn((B, H, D), g, device, dt)
    w = Workload("mha_short", dt, "f16", B, H, H, D, BS, P, ctx, bt, q,
                 torch.arange(B, dtype=torch.int32, device=device), (ctx - 1).to(torch.int32),
                 k_new, v_new, k_cache0=k0, v_cache0=v0)
    w.extra["context"] = "U{%d..%d}" % (ctx_lo, ctx_hi)
    return w


def all_octets(device="cpu") -> torch.Tensor:
    """Every 24-bit octet state as 8 lane values, uint8 [2^24, 8]: state n
    has lane i = bits 3i..3i+2 of n (enumeration of the state space)."""
    n = torch.arange(1 << 24, dtype=torch.int64, device=device)
    lanes = torch.arange(8, dtype=torch.int64, device=device) * 3
    return ((n[:, None] >> lanes[None, :]) & 7).to(torch.uint8)


def storage(t: torch.Tensor, layout: str) -> torch.Tensor:
    """A logical [P, BS, Hkv, D] cache tensor arranged for the given storage
    layout: itself ("flash") or [P, Hkv, D // x, BS, x] ("xvec", x = 16 bytes
    / element size)."""
    if layout == "flash":
        return t
    P, BS, H, D = t.shape
    x = 16 // t.element_size()
    return t.reshape(P, BS, H, D // x, x).permute(0, 2, 3, 1, 4).contiguous()


def bits16(t: torch.Tensor):
    """A 16-bit float tensor's bit pattern as a host numpy uint16 array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
