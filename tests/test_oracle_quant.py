"""Pins of the oracle's int8 storage of the kept cache (reading R17: the LLM
KV-compression notes, "Quantization stacked on compression", one scale per head
from the head's largest |value|; the KV-cache tutorial page, "Quantization",
symmetric q = clip(round(x/s), q_min, q_max), x_hat = s q)."""
import numpy as np
import pytest

from conftest import golden
from oracle import oracle as O


def test_page_worked_example():
    g = golden("int8_quant_example.json")
    q = O.quant_code(g["x"], g["s"])
    assert q == g["q"]
    assert float(np.float32(g["s"]) * np.float32(q)) == pytest.approx(g["x_hat"], abs=1e-6)


def test_half_away_from_zero_and_clip():
    assert O.quant_code(5.0, 2.0) == 3 and O.quant_code(-5.0, 2.0) == -3   # 2.5 -> 3
    assert O.quant_code(3.0, 2.0) == 2 and O.quant_code(-3.0, 2.0) == -2   # 1.5 -> 2
    assert O.quant_code(2.9, 2.0) == 1
    assert O.quant_code(1000.0, 1.0) == 127 and O.quant_code(-1000.0, 1.0) == -127
    assert O.quant_code(3.0, 0.0) == 0


def test_integer_head_is_exact():
    # max |x| = 127 gives s = 1: every integer value is its own code
    rng = np.random.default_rng(0)
    x = rng.integers(-127, 128, size=(20, 2, 16)).astype(np.float32)
    x[3, 0, 5] = 127.0
    x[7, 1, 2] = -127.0
    codes, scales = O.quantize_int8(x)
    assert scales.tolist() == [1.0, 1.0]
    assert np.array_equal(codes.astype(np.float32), x)


def test_per_head_scales_and_error_bound():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((50, 3, 32)).astype(np.float32)
    x[:, 2] *= 100.0  # a head with large values does not touch the others' scales
    codes, scales = O.quantize_int8(x)
    for h in range(3):
        m = np.abs(x[:, h]).max()
        assert scales[h] == np.float32(m) / np.float32(127.0)
        assert np.abs(codes[:, h]).max() == 127
        err = np.abs(x[:, h].astype(np.float64) - scales[h] * codes[:, h].astype(np.float64))
        assert err.max() <= scales[h] / 2 * (1 + 1e-6)


def test_sign_symmetry_zero_head_and_bf16():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((10, 2, 8)).astype(np.float32)
    x[:, 1] = 0.0
    c1, s1 = O.quantize_int8(x)
    c2, s2 = O.quantize_int8(-x)
    assert np.array_equal(c1, -c2) and np.array_equal(s1, s2)
    assert s1[1] == 0.0 and not c1[:, 1].any()
    # bf16 bits decode exactly: 2.0 (0x4000) and -1.0 (0xBF80) in one head, max 2
    b = np.array([[[0x4000, 0xBF80]]], np.uint16)
    c, s = O.quantize_int8(b)
    assert s.tolist() == [np.float32(2.0) / np.float32(127.0)] and c.tolist() == [[[127, -64]]]


def test_empty_unit():
    c, s = O.quantize_int8(np.zeros((0, 2, 8), np.float32))
    assert c.shape == (0, 2, 8) and s.tolist() == [0.0, 0.0]
