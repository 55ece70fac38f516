"""Pins for the oracle's 3-bit affine quantiser: the round trip printed in the
"triton-3bit-kv-cache-kernel" README (section 2, item 3), range, the layout
of element d at bit 3d, the dequantisation error bound, and scale
invariance.  The formula itself is a reading (scale = fp16((max-min)/7),
zero = clamp(round(-min/scale)), q = clamp(round(x/scale)+zero)); these
properties are what pin it.  CPU only."""
import numpy as np
import pytest
import torch

from tests.refs import bitstream_unpack3


def _quant(orc, x_f16: np.ndarray):
    packed, s, z = orc.u3_quantize_pack(x_f16.view(np.uint16), orc.F16)
    q = bitstream_unpack3(packed, x_f16.shape[1])
    return q, s.view(np.float16).astype(np.float64), z.astype(np.int64)


def test_roundtrip_of_dequantised_rows(orc):
    """Rows that are exact dequantisations (q - z) * s with q covering 0 and
    7 quantise back to the same (q, s, z): the requant of a dequant is the
    identity for every q in 0..7 and every zero in 0..7."""
    rng = np.random.default_rng(2)
    D = 128
    # scales with at most 8 significant bits, so every (q - z) * s (3 more
    # bits) is exactly representable in the fp16 source row
    m = rng.integers(128, 256, 200)
    e = rng.integers(-16, -5, 200)
    s_vals = np.concatenate([m * 2.0 ** e, [2.0 ** -10, 0.5, 1.0, 3.0]])
    for i, s in enumerate(s_vals):
        s16 = np.float16(s)
        assert np.float64(s16) == s
        z = i % 8
        q = rng.integers(0, 8, D)
        q[rng.integers(0, D)] = 0
        q[rng.integers(0, D)] = 7
        q[0], q[1] = 0, 7
        x = ((q - z) * np.float64(s16)).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), (q - z) * np.float64(s16))  # exact
        q2, s2, z2 = _quant(orc, x[None, :])
        assert s2[0] == np.float64(s16) and z2[0] == z
        assert np.array_equal(q2[0], q)


def test_requant_identity_formula_page(orc):
    """The page's stated identity clamp(round(((q-z)*s)/s + z), 0, 7) == q for
    all q, z in 0..7 holds in fp32 for the fp16 scales the oracle emits."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((512, 128)).astype(np.float16)
    _, s, _ = _quant(orc, x)
    s32 = s.astype(np.float32)
    for q in range(8):
        for z in range(8):
            deq = (np.float32(q - z) * s32).astype(np.float32)
            back = np.clip(np.rint(deq / s32) + np.float32(z), 0, 7)
            assert np.all(back == q)


def test_range_and_error_bound(orc):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4096, 128)).astype(np.float16)
    q, s, z = _quant(orc, x)
    assert q.min() >= 0 and q.max() <= 7 and z.min() >= 0 and z.max() <= 7
    assert np.all(s > 0)
    xf = x.astype(np.float64)
    mn, mx = xf.min(axis=1), xf.max(axis=1)
    # scale is (max-min)/7 to fp16 precision
    assert np.all(np.abs(s - (mx - mn) / 7) <= 2.0 ** -10 * (mx - mn) / 7)
    deq = (q - z[:, None]) * s[:, None]
    err = np.abs(deq - xf)
    inner = (q > 0) & (q < 7)
    # interior codes: round to nearest step, so error <= s/2 (+ fp32 rounding)
    assert np.all(err[inner] <= (0.5 + 1e-5) * np.broadcast_to(s[:, None], err.shape)[inner])
    # everywhere: at most one step plus half a step
    assert np.all(err <= 1.5 * s[:, None])
    # the row minimum maps to code 0 when the zero point is not clamped
    rows = (z > 0) & (z < 7)
    amin = np.argmin(xf, axis=1)
    assert np.all(q[rows, amin[rows]] <= 1)


def test_power_of_two_scale_invariance(orc):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((256, 64)).astype(np.float16)
    q1, s1, z1 = _quant(orc, x)
    q2, s2, z2 = _quant(orc, (x.astype(np.float32) * 4).astype(np.float16))
    assert np.array_equal(q1, q2) and np.array_equal(z1, z2) and np.allclose(s2, 4 * s1, rtol=0)


def test_constant_row(orc):
    x = np.full((3, 64), 0.75, np.float16)
    x[1] = 0
    x[2] = -3
    q, s, z = _quant(orc, x)
    assert np.all(q == 0) and np.all(s == 0) and np.all(z == 0)


def test_bf16_source(orc):
    """bf16 rows go through the same fp32 formula (values decoded exactly)."""
    rng = np.random.default_rng(6)
    xb = torch.from_numpy(rng.standard_normal((64, 128)).astype(np.float32)).to(torch.bfloat16)
    packed, s, z = orc.u3_quantize_pack(xb.view(torch.int16).numpy().view(np.uint16), orc.BF16)
    xh = xb.to(torch.float32).numpy()
    q = bitstream_unpack3(packed, 128)
    deq = (q - z[:, None].astype(np.int64)) * s.view(np.float16).astype(np.float64)[:, None]
    assert np.all(np.abs(deq - xh) <= 1.5 * s.view(np.float16).astype(np.float64)[:, None])


def test_hand_worked_ties(orc):
    """Hand-worked rows (tests/golden/u3_ties.txt) whose quotients -min/s and
    x/s are exact half-integers, whose fp16 scale rounding meets a tie in
    both directions, and whose codes and zero points clamp: the oracle's
    scale bits, zero point and every code equal the hand-worked values.
    A quantiser that rounds ties away from zero, up, or toward zero fails
    here.  Each row is also tiled to D = 64 and D = 128 (min, max and so
    scale and zero unchanged; codes tiled)."""
    from tests.refs import load_u3_ties
    rows = load_u3_ties()
    assert len(rows) >= 10
    for D in (16, 64, 128):
        x = np.stack([np.tile(r[3], D // 16) for r in rows])
        q, _, z = _quant(orc, x)
        s_bits = orc.u3_quantize_pack(x.view(np.uint16), orc.F16)[1]
        for i, (name, s_exp, z_exp, _, q_exp) in enumerate(rows):
            assert int(s_bits[i]) == s_exp, (name, D, hex(int(s_bits[i])))
            assert int(z[i]) == z_exp, (name, D)
            assert np.array_equal(q[i], np.tile(q_exp, D // 16)), (name, D, q[i][:16])
