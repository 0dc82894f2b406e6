"""The seeded input generators against the recipe they implement: the bf16
codecs against torch's conversion and exact rational rounding, every draw
inside its stated range, and the same seed giving the same inputs."""
from fractions import Fraction

import numpy as np
import pytest

import seeded_inputs as si


def test_f32_to_bf16_matches_torch_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]  # finite values only
    # ties: the low 16 bits exactly 0x8000, with even and odd kept halves
    ties = (rng.integers(0, 2**16, size=2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    ties = ties[(ties & 0x7F800000) != 0x7F800000]
    v = np.concatenate([bits, ties]).view(np.float32)
    want = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(si.f32_to_bf16_bits(v), want)


def _round_bf16_exact(x: float) -> float:
    """x rounded to bf16 (8 significant bits), nearest, ties to even, by exact
    rational arithmetic (normal range)."""
    if x == 0.0:
        return 0.0
    f = Fraction(x)
    sign = -1 if f < 0 else 1
    f = abs(f)
    e = 0
    while f >= 2:
        f /= 2
        e += 1
    while f < 1:
        f *= 2
        e -= 1
    scaled = f * 128  # 8 significant bits: 1.xxxxxxx
    lo = scaled.numerator // scaled.denominator
    rem = scaled - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * float(Fraction(lo, 128) * Fraction(2) ** e)


def test_f64_to_bf16_rounds_once():
    # just above a bf16 midpoint by less than half an fp32 ulp: rounding
    # through fp32 lands on the midpoint and then goes to even (down); a
    # single rounding goes up
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert si.bf16_bits_to_f64(si.f64_to_bf16_bits(np.array([x])))[0] == 1.0 + 2.0 ** -7
    assert si.bf16_bits_to_f64(si.f32_to_bf16_bits(np.array([x], dtype=np.float32)))[0] == 1.0
    rng = np.random.default_rng(12)
    v = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.uniform(-30, 30, 3000),
                        -(1.0 + 2.0 ** -8 + 2.0 ** -30) * 2.0 ** rng.integers(-100, 100, 200)])
    got = si.bf16_bits_to_f64(si.f64_to_bf16_bits(v))
    want = np.array([_round_bf16_exact(float(t)) for t in v])
    np.testing.assert_array_equal(got, want)


def test_bf16_values_round_trip_exactly():
    b = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]  # finite
    b = b[(b & 0x7F80) != 0]       # normals (f64_to_bf16_bits flushes subnormals to zero)
    f64 = si.bf16_bits_to_f64(b)
    np.testing.assert_array_equal(si.f64_to_bf16_bits(f64), b)
    np.testing.assert_array_equal(si.f32_to_bf16_bits(f64.astype(np.float32)), b)


def test_mixer_parameters_follow_the_recipe():
    d = si.REAL_SHAPE
    p = si.mixer_params(3, d)
    assert p["A_log"].shape == (d.H,) and p["conv_w"].shape == (d.CH, d.K) and p["conv_b"].shape == (d.CH,)
    for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b"):
        assert p[k].dtype == np.float32
    # softplus(dt_bias) is the log-uniform step size in [1e-3, 0.1]
    dt = np.logaddexp(0.0, p["dt_bias"].astype(np.float64))
    assert dt.min() >= 1e-3 * (1 - 1e-6) and dt.max() <= 0.1 * (1 + 1e-6)
    # -A = exp(A_log) in [1, 16]
    a = np.exp(p["A_log"].astype(np.float64))
    assert a.min() >= 1.0 - 1e-6 and a.max() <= 16.0 * (1 + 1e-6)
    assert np.abs(p["conv_w"]).max() <= 0.5 and np.abs(p["conv_b"]).max() <= 0.5
    # 128 draws of D ~ N(0, 1)
    assert abs(p["D"].mean()) < 0.4 and 0.7 < p["D"].std() < 1.3


def test_activations_follow_the_recipe():
    d = si.REAL_SHAPE
    a = si.mixer_activations(4, d, 1, 64, "f32")
    assert a["x"].shape == (1, 64, d.H, d.P) and a["B"].shape == (1, 64, d.G, d.N)
    assert a["dt_raw"].shape == (1, 64, d.H)
    for k, sigma in (("x", 1.0), ("B", 1.0), ("C", 1.0), ("dt_raw", 0.5)):
        v = a[k].astype(np.float64)
        assert abs(v.mean()) < 0.05 * sigma and abs(v.std() / sigma - 1.0) < 0.05, k
    # the bf16 form is the RNE rounding of the same draw
    b = si.mixer_activations(4, d, 1, 64, "bf16")
    for k in ("x", "B", "C", "dt_raw"):
        np.testing.assert_array_equal(b[k], si.f32_to_bf16_bits(a[k]))
    with pytest.raises(ValueError):
        si.mixer_activations(4, d, 1, 4, "f16")


def test_same_seed_same_inputs_other_seed_other_inputs():
    d = si.TINY_SHAPE
    a, b, c = si.mixer_inputs(5, d, 2, 16), si.mixer_inputs(5, d, 2, 16), si.mixer_inputs(6, d, 2, 16)
    for k in ("x", "B", "C", "dt_raw", "A_log", "D", "dt_bias", "conv_w", "conv_b"):
        np.testing.assert_array_equal(a[k], b[k])
        assert not np.array_equal(a[k], c[k]), k
    # parameters do not depend on the activations' sizes
    e = si.mixer_inputs(5, d, 1, 3)
    for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b"):
        np.testing.assert_array_equal(a[k], e[k])


def test_quantized_projection_inputs_follow_the_recipe():
    q = si.qlinear_inputs(8, 3, 4480, 256)
    assert q["wq"].shape == (256, 560) and q["wq"].dtype == np.uint32
    assert q["scales"].shape == (256, 70) and q["biases"].shape == (256, 70)
    # the 4-bit fields are uniform over 0..15
    fields = np.stack([(q["wq"] >> (4 * k)) & 0xF for k in range(8)]).ravel()
    counts = np.bincount(fields, minlength=16)
    assert counts.min() > 0.9 * fields.size / 16 and counts.max() < 1.1 * fields.size / 16
    s = si.bf16_bits_to_f64(q["scales"])
    b = si.bf16_bits_to_f64(q["biases"])
    lo, hi = 0.5 / (4 * np.sqrt(4480)), 1.5 / (4 * np.sqrt(4480))
    assert s.min() >= lo * (1 - 2 ** -7) and s.max() <= hi * (1 + 2 ** -7)
    # bias = -7.5 scale U(0.8, 1.2): the dequantized weights centre near zero
    r = -b / (7.5 * s)
    assert r.min() >= 0.8 * (1 - 2 ** -6) and r.max() <= 1.2 * (1 + 2 ** -6)


def test_language_model_pattern():
    lm = si.REAL_LM
    assert lm.kinds.count("M") == 27 and lm.kinds.count("*") == 4 and len(lm.kinds) == 31
    assert len(si.MAMBA_LAYERS) == 27
    assert lm.hidden == 4480 and (lm.n_heads, lm.n_kv_heads, lm.head_dim) == (40, 8, 128)
