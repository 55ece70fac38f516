"""Independent references the tests pin the oracle (and the kernels) against.

These use library routines (torch softmax / matmul in float64, numpy and
torch dtype casts) and a different route through the data (torch gathers)
from the oracle's scalar loops, so a mistake in one is not repeated in the
other.
"""
import math

import numpy as np
import torch


def bitstream_unpack3(packed_rows: np.ndarray, D: int) -> np.ndarray:
    """[n, 3D/8] bytes -> [n, D] values, element d = bits 3d..3d+2 of the
    row read as one little-endian bit string."""
    bits = np.unpackbits(packed_rows, axis=1, bitorder="little")   # [n, 3D]
    bits = bits[:, :3 * D].reshape(packed_rows.shape[0], D, 3).astype(np.uint8)
    return bits[:, :, 0] | (bits[:, :, 1] << 1) | (bits[:, :, 2] << 2)


def gather_attention(q, k_cache, v_cache, block_tables, context_lens, block_size, sm_scale):
    """float64 attention through the block tables, one (b, h) at a time:
    softmax((q . K^T) * sm_scale) @ V over the first context_len tokens.
    q [B,Hq,D]; caches [P,BS,Hkv,D] (any float dtype, dequantised already).
    GQA: q head h reads kv head h // (Hq // Hkv)."""
    q = torch.as_tensor(q).to(torch.float64)
    k_cache = torch.as_tensor(k_cache).to(torch.float64)
    v_cache = torch.as_tensor(v_cache).to(torch.float64)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    out = torch.zeros((B, Hq, D), dtype=torch.float64)
    for b in range(B):
        n = int(context_lens[b])
        if n == 0:
            continue
        nblk = math.ceil(n / block_size)
        ids = torch.as_tensor(np.asarray(block_tables[b][:nblk]), dtype=torch.long)
        k_seq = k_cache[ids].reshape(nblk * block_size, Hkv, D)[:n]
        v_seq = v_cache[ids].reshape(nblk * block_size, Hkv, D)[:n]
        for h in range(Hq):
            kv = h // G
            s = (k_seq[:, kv, :] @ q[b, h]) * sm_scale
            p = torch.softmax(s, dim=0)
            out[b, h] = p @ v_seq[:, kv, :]
    return out.numpy()


def bits_to_tensor(bits: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(dtype)


def e4m3_dequant(codes: np.ndarray, scale_per_head: np.ndarray) -> np.ndarray:
    """[..., Hkv, D] e4m3 codes -> float64 values times the per-head scale
    (torch's float8_e4m3fn view as the decoder)."""
    v = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)
    return (v * torch.from_numpy(scale_per_head.astype(np.float64))[:, None]).numpy()


def e5m2_dequant(codes: np.ndarray, scale_per_head: np.ndarray) -> np.ndarray:
    """[..., Hkv, D] e5m2 codes -> float64 values times the per-head scale
    (torch's float8_e5m2 view as the decoder)."""
    v = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e5m2).to(torch.float64)
    return (v * torch.from_numpy(scale_per_head.astype(np.float64))[:, None]).numpy()


def u3_dequant(packed: np.ndarray, qscale_bits: np.ndarray, qzero: np.ndarray, D: int):
    """[..., 3D/8] packed rows + fp16 scale bits + zero -> float64 (q-z)*s."""
    lead = packed.shape[:-1]
    q = bitstream_unpack3(packed.reshape(-1, packed.shape[-1]), D).astype(np.float64)
    s = np.ascontiguousarray(qscale_bits).view(np.float16).astype(np.float64).reshape(-1, 1)
    z = qzero.astype(np.float64).reshape(-1, 1)
    return ((q - z) * s).reshape(*lead, D)


def load_u3_ties(path=None):
    """Rows of tests/golden/u3_ties.txt -> list of (name, s_bits, z, x [16]
    fp16, q [16] uint8)."""
    import os
    if path is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "u3_ties.txt")
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, meta, xs, qs = (p.strip() for p in line.split("|"))
            s_hex, z = meta.split()
            x = np.array([float(v) for v in xs.split()], dtype=np.float64)
            x16 = x.astype(np.float16)
            assert np.array_equal(x16.astype(np.float64), x), name   # every x exact in fp16
            q = np.array([int(v) for v in qs.split()], dtype=np.uint8)
            assert x.shape == q.shape, name
            rows.append((name, int(s_hex, 16), int(z), x16, q))
    return rows
