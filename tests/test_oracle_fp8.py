"""Pins for the FP8 row oracle (issue #1313, step 1.3, item 3: FP8 rows with FP32 scales).

The E4M3 encoder and decoder are held to values fixed by the format's bit fields (written out
by hand here), to a library's conversion (torch.float8_e4m3fn) where the two definitions meet,
and to the rounding and saturation rules on hand-picked ties and out-of-range values.
"""
import math

import numpy as np
import pytest

from oracle import fp8 as F


def test_decode_hand_values():
    assert F.decode(0x38) == 1.0 and F.decode(0xB8) == -1.0
    assert F.decode(0x7E) == 448.0 and F.decode(0xFE) == -448.0
    assert F.decode(0x08) == 2.0 ** -6          # smallest normal
    assert F.decode(0x01) == 2.0 ** -9          # smallest subnormal
    assert F.decode(0x07) == 7 * 2.0 ** -9
    assert F.decode(0x3C) == 1.5 and F.decode(0x40) == 2.0 and F.decode(0x30) == 0.5
    assert math.isnan(F.decode(0x7F)) and math.isnan(F.decode(0xFF))
    assert F.decode(0x00) == 0.0 and math.copysign(1.0, F.decode(0x80)) < 0


def test_every_code_round_trips():
    for c in range(256):
        v = F.decode(c)
        if math.isnan(v):
            assert F.encode(v) == F.NAN_CODE
        else:
            assert F.encode(v) == c, hex(c)


def test_ties_go_to_even_and_large_values_saturate():
    assert F.encode(1.0 + 1 / 16) == 0x38        # between 1 and 1.125: even mantissa 0
    assert F.encode(1.0 + 3 / 16) == 0x3A        # between 1.125 and 1.25: even mantissa 2
    assert F.encode(2.0 ** -10) == 0x00          # half the smallest subnormal: to zero
    assert F.encode(3 * 2.0 ** -10) == 0x02      # 1.5 steps: to 2
    assert F.encode(5 * 2.0 ** -10) == 0x02      # 2.5 steps: to 2
    assert F.encode(15 * 2.0 ** -10) == 0x08     # 7.5 steps: to the smallest normal
    assert F.encode(464.0) == 0x7E and F.encode(500.0) == 0x7E and F.encode(-1e30) == 0xFE
    assert F.encode(-0.0) == 0x80


def test_matches_torch_conversion_in_range():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(3)
    x = np.concatenate([g.uniform(-448, 448, 4000), g.uniform(-2 ** -5, 2 ** -5, 2000),
                        g.standard_normal(2000) * 10]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([F.encode(v) for v in x], np.uint8)
    assert np.array_equal(got, want)


def test_row_quantization():
    g = np.random.default_rng(5)
    x = (g.standard_normal(512) * 0.1).astype(np.float32)
    codes, scale = F.quantize_row(x)
    assert scale.dtype == np.float32 and scale == np.float32(np.max(np.abs(x)) / np.float32(448))
    k = int(np.argmax(np.abs(x)))
    assert codes[k] & 0x7F == 0x7E                 # the largest value maps to +-448
    deq = F.dequantize_row(codes, scale)
    q = np.abs(x.astype(np.float64)) / float(scale)
    err = np.abs(deq - x) / float(scale)
    # half a step: 2^-4 relative for normals, 2^-10 absolute in the subnormal range (plus the
    # fp32 rounding of x / scale)
    assert np.all(err <= np.maximum(q * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6) + q * 2.0 ** -23)
    assert np.array_equal(np.sign(deq[deq != 0]), np.sign(x[deq != 0]))


def test_zero_row_and_batched_form():
    codes, scale = F.quantize_row(np.zeros(512, np.float32))
    assert scale == 0 and not codes.any()
    g = np.random.default_rng(6)
    x = (g.standard_normal((3, 4, 512))).astype(np.float32)
    c, s = F.quantize_rows(x)
    c1, s1 = F.quantize_row(x[2, 1])
    assert np.array_equal(c[2, 1], c1) and s[2, 1] == s1
    assert np.array_equal(F.dequantize_rows(c, s)[2, 1], F.dequantize_row(c1, s1))


def test_attention_over_double_latent_is_the_same_definition():
    """The oracle's double-latent entry (used for FP8 rows) equals its bf16 entry bit for bit when
    the doubles are the bf16 values, and a single key gives its dequantized row exactly."""
    from oracle import attend as OA
    from paged_mla_kv_gb300 import synth as Y
    w = Y.custom("f64pin", 31, lens=[300], R=2, H=4)
    lat, rope = w.stream_rows(0, 0)
    q = w.q(0)[0]
    a = OA.attend_stream(q, lat, rope, w.scale, threads=2)
    b = OA.attend_stream(q, Y.bf16_bits_to_f32(lat).astype(np.float64), rope, w.scale, threads=2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    codes, scales = F.quantize_rows(Y.bf16_bits_to_f32(lat[:1]))
    deq = F.dequantize_rows(codes, scales)
    out, _ = OA.attend_stream(q[:1], deq, rope[:1], w.scale, threads=1)
    assert np.array_equal(out, np.repeat(deq, out.shape[0], axis=0))


def test_array_encoder_is_the_scalar_definition():
    g = np.random.default_rng(21)
    x = np.concatenate([g.standard_normal(20000) * 50, g.uniform(-2 ** -5, 2 ** -5, 20000),
                        g.uniform(-600, 600, 5000), [0.0, -0.0, np.nan, np.inf, -np.inf, 448.0, 464.0, 2 ** -10,
                                                     3 * 2 ** -10, 15 * 2 ** -10, 1 + 1 / 16, 1 + 3 / 16]])
    x = x.astype(np.float32)
    x = np.concatenate([x, np.array([F.decode(c) for c in range(256) if c not in (0x7F, 0xFF)], np.float32)])
    want = np.array([F.encode(v) for v in x], np.uint8)
    assert np.array_equal(F.encode_array(x), want)
    rows = (g.standard_normal((5, 512)) * 0.3).astype(np.float32)
    rows[2] = 0
    c, s_ = F.quantize_rows(rows)
    for i in range(5):
        ci, si = F.quantize_row(rows[i])
        assert np.array_equal(c[i], ci) and s_[i] == si
