"""Pins for the fp64 oracle, against facts fixed outside the oracle itself:
library routines (torch conv1d, numpy logaddexp, scipy lfilter/expit),
closed forms, dense matrix forms of the recurrence, special cases and the
invariants the VoiceChat doc states ("docs/nemotron-voicechat.md", section
Offline timeline: cached stepping and full-history recompute agree).

Each pin is chosen so that a plausible slip in the oracle (a reversed conv
tap, a wrong channel offset, a dropped D term, a wrong head-to-group map, a
sign error in the decay, an off-by-one in the chunk cumsum, a stale conv
tail) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch
from scipy.signal import lfilter
from scipy.special import expit

from seeded_inputs import (
    MAMBA_LAYERS, REAL_SHAPE, TINY_SHAPE, Dims, as_f64, conv_state_inputs, mixer_inputs,
    ssm_state_inputs,
)

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ----------------------------------------------------------- pages' shapes
def test_text_config_shape_and_layer_pattern():
    cfg = json.load(open(os.path.join(GOLDEN, "text_config.json")))
    d = REAL_SHAPE
    assert (d.H, d.P, d.N, d.G, d.K) == (cfg["mamba_num_heads"], cfg["mamba_head_dim"],
                                         cfg["ssm_state_size"], cfg["n_groups"], cfg["conv_kernel"])
    assert d.CH == 12288 and d.H * d.P == 10240
    pat = cfg["hybrid_override_pattern"]
    assert len(pat) == cfg["num_hidden_layers"]
    assert [i for i, c in enumerate(pat) if c == "*"] == cfg["attention_layers"]
    assert list(MAMBA_LAYERS) == [i for i, c in enumerate(pat) if c == "M"]
    assert len(MAMBA_LAYERS) == 27


# ----------------------------------------------------------- scalar maps
@pytest.mark.parametrize("z", [-1e4, -745.0, -60.0, -30.5, -5.0, -1e-3, 0.0, 1e-3, 0.7, 5.0, 30.5,
                               60.0, 700.0, 1e4])
def test_softplus_matches_logaddexp(oracle_lib, z):
    ref = float(np.logaddexp(0.0, z))
    got = oracle_lib.softplus(z)
    assert got == pytest.approx(ref, rel=4e-16, abs=1e-320)


def test_softplus_underflow_is_exact_zero(oracle_lib):
    # dt -> 0 special case relies on this: e^-1e4 underflows, log1p(0) = 0.
    assert oracle_lib.softplus(-1e4) == 0.0


@pytest.mark.parametrize("u", [-800.0, -40.0, -3.0, -0.25, 0.0, 0.25, 3.0, 40.0, 800.0])
def test_silu_matches_expit(oracle_lib, u):
    ref = u * float(expit(u))
    assert oracle_lib.silu(u) == pytest.approx(ref, rel=4e-16, abs=1e-300)


# ----------------------------------------------------------- conv + SiLU
def _torch_conv_silu(d, x, B, C, conv_w, conv_b, init_conv=None):
    """Depthwise causal conv1d by the library routine, then x*sigmoid(x)."""
    b, T = x.shape[:2]
    xin = np.concatenate([x.reshape(b, T, -1), B.reshape(b, T, -1), C.reshape(b, T, -1)], axis=2)
    if init_conv is None:
        pad = np.zeros((b, d.K - 1, d.CH))
    else:
        pad = init_conv
    seq = torch.from_numpy(np.concatenate([pad, xin], axis=1)).permute(0, 2, 1)  # [b, CH, K-1+T]
    w = torch.from_numpy(np.asarray(conv_w, np.float64)).reshape(d.CH, 1, d.K)
    bias = torch.from_numpy(np.asarray(conv_b, np.float64))
    u = torch.nn.functional.conv1d(seq, w, bias, groups=d.CH)  # [b, CH, T]
    return (u * torch.sigmoid(u)).permute(0, 2, 1).numpy()


@pytest.mark.parametrize("with_init", [False, True])
def test_conv_silu_matches_torch_conv1d(oracle_lib, with_init):
    d = Dims(H=4, P=8, N=8, G=2, K=4)
    inp = mixer_inputs(11, d, 2, 37, "f32")
    x, B, C = (as_f64(inp[k], "f32") for k in "xBC")
    ic = as_f64(conv_state_inputs(12, d, 2, "f32"), "f32") if with_init else None
    got = oracle_lib.conv_silu(d, x, B, C, inp["conv_w"], inp["conv_b"], ic)
    ref = _torch_conv_silu(d, x, B, C, inp["conv_w"], inp["conv_b"], ic)
    assert rel(got, ref) < 1e-14


@pytest.mark.parametrize("T", [0, 1, 2, 3, 5])
def test_conv_tail_is_last_three_inputs(oracle_lib, T):
    d = Dims(H=2, P=4, N=4, G=1, K=4)
    inp = mixer_inputs(3, d, 2, T, "bf16")
    ic = conv_state_inputs(4, d, 2, "bf16")
    r = oracle_lib.mixer_scan(d, inp, init_conv=ic)
    x, B, C = (as_f64(inp[k], "bf16") for k in "xBC")
    full = np.concatenate([as_f64(ic, "bf16"),
                           np.concatenate([x.reshape(2, T, d.H * d.P), B.reshape(2, T, d.G * d.N),
                                           C.reshape(2, T, d.G * d.N)], axis=2)], axis=1)
    np.testing.assert_array_equal(r["final_conv"], full[:, -3:, :])
    # without an initial tail the missing frames are zeros
    r0 = oracle_lib.mixer_scan(d, inp)
    full0 = full.copy()
    full0[:, :3, :] = 0.0
    np.testing.assert_array_equal(r0["final_conv"], full0[:, -3:, :])


# ----------------------------------------------------------- SSM core forms
def _post_conv_inputs(seed, d, b, T, scale_dt=1.0):
    rng = np.random.default_rng(seed)
    xt = rng.standard_normal((b, T, d.H, d.P))
    Bt = rng.standard_normal((b, T, d.G, d.N)) * 0.5
    Ct = rng.standard_normal((b, T, d.G, d.N)) * 0.5
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(0.3), (b, T, d.H))) * scale_dt
    A = -rng.uniform(1.0, 16.0, d.H)
    D = rng.standard_normal(d.H)
    return xt, Bt, Ct, dt, A, D


def _quadratic_form(d, xt, Bt, Ct, dt, A, D, h0=None):
    """Dense matrix form: y = (L o C B^T) (dt o x) + exp(S) C h0^T + D x, with
    L[i,j] = exp(S_i - S_j) for j <= i; final h = sum_j exp(S_T-S_j) dt_j x_j B_j^T
    + exp(S_T) h0. Built with numpy matrices, head-to-group map g = h // (H/G)."""
    b, T = xt.shape[:2]
    y = np.zeros_like(xt)
    hT = np.zeros((b, d.H, d.P, d.N))
    for bi in range(b):
        for h in range(d.H):
            g = h // (d.H // d.G)
            S = np.cumsum(dt[bi, :, h] * A[h])
            L = np.tril(np.exp(S[:, None] - np.where(np.tril(np.ones((T, T))) > 0, S[None, :], S[:, None])))
            CB = Ct[bi, :, g, :] @ Bt[bi, :, g, :].T
            u = dt[bi, :, h][:, None] * xt[bi, :, h, :]
            y[bi, :, h, :] = (L * CB) @ u + D[h] * xt[bi, :, h, :]
            w = np.exp(S[-1] - S) if T else np.zeros(0)
            hT[bi, h] = (u * w[:, None]).T @ Bt[bi, :, g, :]
            if h0 is not None:
                y[bi, :, h, :] += np.exp(S)[:, None] * (Ct[bi, :, g, :] @ h0[bi, h].T)
                hT[bi, h] += (np.exp(S[-1]) if T else 1.0) * h0[bi, h]
    return y, hT


@pytest.mark.parametrize("with_h0", [False, True])
def test_sequential_equals_dense_quadratic_form(oracle_lib, with_h0):
    d = Dims(H=4, P=5, N=6, G=2, K=4)
    xt, Bt, Ct, dt, A, D = _post_conv_inputs(5, d, 2, 23)
    h0 = np.random.default_rng(6).standard_normal((2, d.H, d.P, d.N)) if with_h0 else None
    y, h = oracle_lib.ssm(d, xt, Bt, Ct, dt, A, D, h0=h0)
    yq, hq = _quadratic_form(d, xt, Bt, Ct, dt, A, D, h0)
    assert rel(y, yq) < 1e-12
    assert rel(h, hq) < 1e-12


@pytest.mark.parametrize("Q", [1, 2, 3, 7, 16, 64, 70])
def test_chunked_equals_sequential(oracle_lib, Q):
    d = TINY_SHAPE
    T = 65 if Q != 70 else 65  # T = 65: ragged last chunk for most Q; Q = T+5 single chunk
    xt, Bt, Ct, dt, A, D = _post_conv_inputs(7, d, 1, T)
    h0 = np.random.default_rng(8).standard_normal((1, d.H, d.P, d.N)) * 0.1
    ys, hs = oracle_lib.ssm(d, xt, Bt, Ct, dt, A, D, h0=h0)
    yc, hc = oracle_lib.ssm(d, xt, Bt, Ct, dt, A, D, h0=h0, chunk=Q)
    assert rel(yc, ys) < 1e-12
    assert rel(hc, hs) < 1e-12


def test_chunk_equal_to_T_on_mixer_inputs(oracle_lib):
    d = TINY_SHAPE
    inp = mixer_inputs(0, d, 1, 64, "f32")
    r = oracle_lib.mixer_scan(d, inp)
    for Q in (8, 16, 64, 69):
        rc = oracle_lib.mixer_scan(d, inp, chunk=Q)
        assert rel(rc["y"], r["y"]) < 1e-12
        assert rel(rc["final_ssm"], r["final_ssm"]) < 1e-12


def test_closed_form_scalar_filter(oracle_lib):
    """H=P=N=G=1, B=C=1, constant dt: y_t = D x_t + dt sum_s a^(t-s) x_s with
    a = exp(dt A), i.e. the IIR filter dt / (1 - a z^-1) (scipy lfilter)."""
    d = Dims(H=1, P=1, N=1, G=1, K=4)
    T = 200
    rng = np.random.default_rng(9)
    x = rng.standard_normal(T)
    dtv, Av, Dv = 0.07, -2.5, 0.8
    a = np.exp(dtv * Av)
    y, h = oracle_lib.ssm(d, x.reshape(1, T, 1, 1), np.ones((1, T, 1, 1)), np.ones((1, T, 1, 1)),
                          np.full((1, T, 1), dtv), np.array([Av]), np.array([Dv]))
    ref = lfilter([dtv], [1.0, -a], x) + Dv * x
    assert rel(y.ravel(), ref) < 1e-13
    assert h.ravel()[0] == pytest.approx(ref[-1] - Dv * x[-1], rel=1e-13)
    # constant input: geometric series closed form
    xc = 1.3
    y2, _ = oracle_lib.ssm(d, np.full((1, T, 1, 1), xc), np.ones((1, T, 1, 1)), np.ones((1, T, 1, 1)),
                           np.full((1, T, 1), dtv), np.array([Av]), np.array([Dv]))
    t = np.arange(T)
    geo = dtv * xc * (1 - a ** (t + 1)) / (1 - a) + Dv * xc
    assert rel(y2.ravel(), geo) < 1e-13


def test_linearity_in_x(oracle_lib):
    d = Dims(H=4, P=5, N=6, G=2, K=4)
    xt, Bt, Ct, dt, A, D = _post_conv_inputs(10, d, 1, 30)
    x2 = np.random.default_rng(11).standard_normal(xt.shape)
    y1, h1 = oracle_lib.ssm(d, xt, Bt, Ct, dt, A, D)
    y2, h2 = oracle_lib.ssm(d, x2, Bt, Ct, dt, A, D)
    y3, h3 = oracle_lib.ssm(d, 2.0 * xt - 0.5 * x2, Bt, Ct, dt, A, D)
    assert rel(y3, 2.0 * y1 - 0.5 * y2) < 1e-12
    assert rel(h3, 2.0 * h1 - 0.5 * h2) < 1e-12


def test_group_map_is_contiguous(oracle_lib):
    """Perturbing B and C of group 1 changes heads 2,3 only (H=4, G=2)."""
    d = Dims(H=4, P=3, N=4, G=2, K=4)
    xt, Bt, Ct, dt, A, D = _post_conv_inputs(12, d, 1, 9)
    y0, _ = oracle_lib.ssm(d, xt, Bt, Ct, dt, A, D)
    B2, C2 = Bt.copy(), Ct.copy()
    B2[:, :, 1, :] += 1.0
    C2[:, :, 1, :] -= 0.5
    y1, _ = oracle_lib.ssm(d, xt, B2, C2, dt, A, D)
    assert np.array_equal(y0[:, :, :2], y1[:, :, :2])
    assert np.all(np.abs(y0[:, :, 2:] - y1[:, :, 2:]).max(axis=(0, 1, 3)) > 1e-3)


# ----------------------------------------------------------- whole mixer
def test_mixer_scan_composes_pinned_parts(oracle_lib):
    """Whole pipeline == torch conv1d + SiLU, split x|B|C, numpy softplus,
    A = -exp(A_log), dense quadratic form. Pins the channel offsets, the dt
    map, where D applies (post-conv x), and the initial-state handling."""
    d = Dims(H=4, P=6, N=5, G=2, K=4)
    b, T = 2, 19
    inp = mixer_inputs(13, d, b, T, "bf16")
    ic = conv_state_inputs(14, d, b, "bf16")
    h0 = ssm_state_inputs(15, d, b, scale=0.3).astype(np.float64)
    r = oracle_lib.mixer_scan(d, inp, init_ssm=h0, init_conv=ic)
    x, B, C, dtr = (as_f64(inp[k], "bf16") for k in ("x", "B", "C", "dt_raw"))
    u = _torch_conv_silu(d, x, B, C, inp["conv_w"], inp["conv_b"], as_f64(ic, "bf16"))
    HP, GN = d.H * d.P, d.G * d.N
    xt = u[:, :, :HP].reshape(b, T, d.H, d.P)
    Bt = u[:, :, HP:HP + GN].reshape(b, T, d.G, d.N)
    Ct = u[:, :, HP + GN:].reshape(b, T, d.G, d.N)
    dt = np.logaddexp(0.0, dtr + inp["dt_bias"].astype(np.float64))
    A = -np.exp(inp["A_log"].astype(np.float64))
    yq, hq = _quadratic_form(d, xt, Bt, Ct, dt, A, inp["D"].astype(np.float64), h0)
    assert rel(r["y"], yq) < 1e-12
    assert rel(r["final_ssm"], hq) < 1e-12


def test_magnitude_equals_y_when_every_term_is_positive(oracle_lib):
    """With every post-conv x~, B~, C~ positive (a conv bias of +4 against
    pre-activations of spread ~0.6), D = 0 and a non-negative initial state,
    no term of the recurrence is negative: the magnitude ybar equals y."""
    d = Dims(H=4, P=6, N=5, G=2, K=4)
    b, T = 2, 23
    inp = mixer_inputs(21, d, b, T, "bf16")
    inp["conv_b"] = np.full(d.CH, 4.0, np.float32)
    inp["D"] = np.zeros(d.H, np.float32)
    h0 = np.abs(ssm_state_inputs(22, d, b, scale=0.3).astype(np.float64))
    r = oracle_lib.mixer_scan(d, inp, init_ssm=h0)
    ybar = oracle_lib.mixer_scan_magnitude(d, inp, init_ssm=h0)
    assert np.all(ybar > 0)
    assert rel(ybar, r["y"]) < 1e-12


def test_magnitude_bounds_the_state_space_part(oracle_lib):
    """For signed inputs, |y - D x~| <= ybar everywhere (triangle inequality),
    with equality nowhere near in general: it is a bound, not the value."""
    d = Dims(H=4, P=6, N=5, G=2, K=4)
    b, T = 2, 31
    inp = mixer_inputs(23, d, b, T, "bf16")
    ic = conv_state_inputs(24, d, b, "bf16")
    h0 = ssm_state_inputs(25, d, b, scale=0.3).astype(np.float64)
    no_d = dict(inp, D=np.zeros(d.H, np.float32))
    ssm_part = oracle_lib.mixer_scan(d, no_d, init_ssm=h0, init_conv=ic)["y"]
    ybar = oracle_lib.mixer_scan_magnitude(d, inp, init_ssm=h0, init_conv=ic)
    assert np.all(np.abs(ssm_part) <= ybar * (1 + 1e-12))
    assert np.median(np.abs(ssm_part) / ybar) < 0.9
    # the magnitude covers the state-space terms only: D does not enter it
    np.testing.assert_array_equal(ybar, oracle_lib.mixer_scan_magnitude(d, no_d, init_ssm=h0, init_conv=ic))


@pytest.mark.parametrize("tsteps", [1, 2, 3, 4, 100])
def test_step_equals_recompute(oracle_lib, tsteps):
    """Stepping t frames from zero caches == full-history recompute of t frames."""
    d = TINY_SHAPE
    S = 3
    inp = mixer_inputs(16, d, S, tsteps, "f32")
    r = oracle_lib.mixer_scan(d, inp)
    ssm = np.zeros((S, d.H, d.P, d.N))
    conv = np.zeros((S, d.K - 1, d.CH))
    ys = []
    for t in range(tsteps):
        frame = {k: np.ascontiguousarray(inp[k][:, t]) for k in ("x", "B", "C", "dt_raw")}
        frame["act"] = "f32"
        ys.append(oracle_lib.mixer_step(d, frame, inp, ssm, conv))
    y = np.stack(ys, axis=1)
    assert rel(y, r["y"]) < 1e-12
    assert rel(ssm, r["final_ssm"]) < 1e-12
    np.testing.assert_array_equal(conv, r["final_conv"])


def test_scan_continuation_from_cached_state(oracle_lib):
    """A scan over [0, T) equals a scan over [0, t1) followed by a scan over
    [t1, T) that starts from the first part's SSM state and conv tail."""
    d = Dims(H=4, P=8, N=8, G=2, K=4)
    T, t1 = 40, 17
    inp = mixer_inputs(17, d, 2, T, "bf16")
    r = oracle_lib.mixer_scan(d, inp)
    a = dict(inp, **{k: inp[k][:, :t1] for k in ("x", "B", "C", "dt_raw")})
    bpart = dict(inp, **{k: inp[k][:, t1:] for k in ("x", "B", "C", "dt_raw")})
    ra = oracle_lib.mixer_scan(d, a)
    from seeded_inputs import f64_to_bf16_bits
    tail_bits = f64_to_bf16_bits(ra["final_conv"])  # exact: the tail holds input values
    rb = oracle_lib.mixer_scan(d, bpart, init_ssm=ra["final_ssm"], init_conv=tail_bits)
    assert rel(np.concatenate([ra["y"], rb["y"]], axis=1), r["y"]) < 1e-12
    assert rel(rb["final_ssm"], r["final_ssm"]) < 1e-12
    np.testing.assert_array_equal(rb["final_conv"], r["final_conv"])


def test_dt_to_zero_leaves_state_unchanged(oracle_lib):
    """dt_bias = -1e4 makes softplus underflow to exactly 0: the SSM state is
    bitwise unchanged and y = C.h_prev + D x (from zero state: D x)."""
    d = Dims(H=4, P=6, N=5, G=2, K=4)
    b, T = 1, 7
    inp = mixer_inputs(18, d, b, T, "f32")
    inp["dt_bias"] = np.full(d.H, -1e4, np.float32)
    h0 = ssm_state_inputs(19, d, b, scale=0.5).astype(np.float64)
    r = oracle_lib.mixer_scan(d, inp, init_ssm=h0)
    np.testing.assert_array_equal(r["final_ssm"], h0)
    x, B, C = (as_f64(inp[k], "f32") for k in "xBC")
    u = _torch_conv_silu(d, x, B, C, inp["conv_w"], inp["conv_b"])
    HP, GN = d.H * d.P, d.G * d.N
    xt = u[:, :, :HP].reshape(b, T, d.H, d.P)
    Ct = u[:, :, HP + GN:].reshape(b, T, d.G, d.N)
    g = np.arange(d.H) // (d.H // d.G)
    ref = np.einsum("bthn,bhpn->bthp", Ct[:, :, g, :], h0) + inp["D"].astype(np.float64)[None, None, :, None] * xt
    assert rel(r["y"], ref) < 1e-12
    r0 = oracle_lib.mixer_scan(d, inp)
    assert rel(r0["y"], inp["D"].astype(np.float64)[None, None, :, None] * xt) < 1e-14
    assert np.all(r0["final_ssm"] == 0.0)


def test_A_to_zero_is_prefix_sum(oracle_lib):
    """A_log = -1e4 gives A = -0 and exp(dt A) = 1 exactly: the state is the
    running sum of dt x (outer) B (numpy cumsum)."""
    d = Dims(H=4, P=6, N=5, G=2, K=4)
    b, T = 1, 11
    inp = mixer_inputs(20, d, b, T, "f32")
    inp["A_log"] = np.full(d.H, -1e4, np.float32)
    r = oracle_lib.mixer_scan(d, inp)
    x, B, C, dtr = (as_f64(inp[k], "f32") for k in ("x", "B", "C", "dt_raw"))
    u = _torch_conv_silu(d, x, B, C, inp["conv_w"], inp["conv_b"])
    HP, GN = d.H * d.P, d.G * d.N
    xt = u[:, :, :HP].reshape(b, T, d.H, d.P)
    Bt = u[:, :, HP:HP + GN].reshape(b, T, d.G, d.N)
    Ct = u[:, :, HP + GN:].reshape(b, T, d.G, d.N)
    dt = np.logaddexp(0.0, dtr + inp["dt_bias"].astype(np.float64))
    g = np.arange(d.H) // (d.H // d.G)
    incr = np.einsum("bth,bthp,bthn->bthpn", dt, xt, Bt[:, :, g, :])
    hs = np.cumsum(incr, axis=1)
    assert rel(r["final_ssm"], hs[:, -1]) < 1e-12
    yref = np.einsum("bthn,bthpn->bthp", Ct[:, :, g, :], hs) + inp["D"].astype(np.float64)[None, None, :, None] * xt
    assert rel(r["y"], yref) < 1e-12


def test_head_subset_matches_full(oracle_lib):
    d = REAL_SHAPE
    inp = mixer_inputs(21, d, 1, 12, "bf16")
    full = oracle_lib.mixer_scan(d, inp)
    part = oracle_lib.mixer_scan(d, inp, heads=(37, 41))
    np.testing.assert_array_equal(part["y"][:, :, 37:41], full["y"][:, :, 37:41])
    np.testing.assert_array_equal(part["final_ssm"][:, 37:41], full["final_ssm"][:, 37:41])


def test_bf16_codec_roundtrip():
    from seeded_inputs import bf16_bits_to_f64, f32_to_bf16_bits, f64_to_bf16_bits
    v = np.array([1.0, -2.5, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, 3.1415926, -1e-20, 0.0, 65504.0])
    b32 = f32_to_bf16_bits(v.astype(np.float32))
    b64 = f64_to_bf16_bits(v)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to even (1.0)
    assert bf16_bits_to_f64(b64)[2] == 1.0
    assert bf16_bits_to_f64(b64)[3] == 1.0 + 2 ** -7
    assert abs(bf16_bits_to_f64(b64)[4] - 3.140625) == 0.0
    np.testing.assert_array_equal(b32[[0, 1, 2, 3, 4, 6, 7]], b64[[0, 1, 2, 3, 4, 6, 7]])


# ------------------------------------------------------------ gated RMSNorm
def test_gated_norm_open_gate_is_torch_rms_norm():
    """With a wide-open gate (z = 1000: silu(z) = z exactly in fp64) the
    gated norm is the library RMSNorm of each channel group, scaled by the
    weight; the factor 1000 moves into eps (rms_norm of 1000 v with eps e is
    rms_norm of v with eps e / 1e6)."""
    import oracle
    rng = np.random.default_rng(7)
    rows, width, groups, eps = 5, 48, 3, 1e-5
    y = rng.standard_normal((rows, width))
    w = 1 + 0.1 * rng.standard_normal(width)
    out = oracle.gated_norm(y, np.full_like(y, 1000.0), w, groups, eps)
    gw = width // groups
    ref = torch.nn.functional.rms_norm(torch.from_numpy(y).reshape(rows, groups, gw), (gw,), eps=eps / 1e6)
    ref = ref.reshape(rows, width).numpy() * w
    assert np.max(np.abs(out - ref)) < 1e-12


def test_gated_norm_worked_case():
    """y = (3, 4), open gate, one group, eps 0: (3, 4) / sqrt(12.5)."""
    import oracle
    out = oracle.gated_norm(np.array([[3.0, 4.0]]), np.array([[1000.0, 1000.0]]), np.ones(2), 1, 0.0)
    np.testing.assert_allclose(out[0], [3 / np.sqrt(12.5), 4 / np.sqrt(12.5)], rtol=1e-15)


def test_gated_norm_gate_and_invariances():
    """The gate multiplies by silu(z) (library expit), the output does not
    change when y is scaled (eps 0), flips sign with y, and each channel
    group is normalised on its own."""
    import oracle
    rng = np.random.default_rng(8)
    rows, width, groups = 4, 40, 5
    y, z = rng.standard_normal((rows, width)), rng.standard_normal((rows, width))
    w = 1 + 0.1 * rng.standard_normal(width)
    out = oracle.gated_norm(y, z, w, groups, 0.0)
    # gate through the library sigmoid: gated input y * z * expit(z), open gate
    gated = y * z * expit(z)
    np.testing.assert_allclose(out, oracle.gated_norm(gated, np.full_like(y, 1000.0), w, groups, 0.0) ,
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.gated_norm(7.5 * y, z, w, groups, 0.0), out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.gated_norm(-y, z, w, groups, 0.0), -out, rtol=1e-12, atol=1e-12)
    y2 = y.copy()
    y2[:, :8] *= 3.0  # the first group only
    out2 = oracle.gated_norm(y2, z, w, groups, 0.0)
    np.testing.assert_allclose(out2[:, 8:], out[:, 8:], rtol=1e-12, atol=1e-12)
    assert np.max(np.abs(out2[:, :8] - out[:, :8])) < 1e-12  # scale-free within the group too
    # each group has mean square (weight-free) 1
    unit = oracle.gated_norm(y, z, np.ones(width), groups, 0.0).reshape(rows, groups, -1)
    np.testing.assert_allclose(np.mean(unit ** 2, axis=-1), 1.0, rtol=1e-12)


# ------------------------------------------------ quantized mixer projections
# Two output rows of 64 inputs, one group, written out by hand: row 0 holds
# q = i % 16 (words 0x76543210, 0xFEDCBA98, ...: the first input in the lowest
# four bits), row 1 holds q = 15 - i % 16.
_QL_WQ = np.array([[0x76543210, 0xFEDCBA98] * 4, [0x89ABCDEF, 0x01234567] * 4], dtype=np.uint32)
_QL_SCALE = np.array([[0.5], [2.0]])
_QL_BIAS = np.array([[-4.0], [1.0]])


def test_qlinear_worked_example():
    """W0[i] = 0.5 (i % 16) - 4 and W1[i] = 2 (15 - i % 16) + 1, so with
    x = 1: y0 = 64 (0.5 * 7.5 - 4) = -16 and y1 = 4 * sum_k (31 - 2k) = 1024;
    unit vectors read single weights (i = 13: 2.5 and 5; i = 63: 3.5 and 1)."""
    import oracle
    np.testing.assert_array_equal(oracle.qlinear(np.ones(64), _QL_WQ, _QL_SCALE, _QL_BIAS), [-16.0, 1024.0])
    for i, want in ((13, [2.5, 5.0]), (63, [3.5, 1.0]), (0, [-4.0, 31.0]), (8, [0.0, 15.0])):
        e = np.zeros(64)
        e[i] = 1.0
        np.testing.assert_array_equal(oracle.qlinear(e, _QL_WQ, _QL_SCALE, _QL_BIAS), want)


def test_qlinear_equals_dense_matmul():
    """Against a library matmul (torch, fp64) of the weights decoded
    separately with vectorised shifts, for several rows and groups."""
    import oracle
    from seeded_inputs import bf16_bits_to_f64, qlinear_inputs
    inp = qlinear_inputs(7, 3, 256, 40)
    x, s, b = (bf16_bits_to_f64(inp[k]) for k in ("x", "scales", "biases"))
    q = (inp["wq"][:, :, None].astype(np.int64) >> (4 * np.arange(8))) & 15
    w = np.repeat(s, 64, axis=1) * q.reshape(40, 256) + np.repeat(b, 64, axis=1)
    ref = (torch.from_numpy(x) @ torch.from_numpy(w).T).numpy()
    np.testing.assert_allclose(oracle.qlinear(x, inp["wq"], s, b), ref, rtol=1e-12, atol=1e-12)


def test_qlinear_bias_only_and_linearity():
    """With zero scales each output is sum_g bias[o, g] * (sum of x over
    group g); doubling scales and biases doubles y; y is linear in x."""
    import oracle
    from seeded_inputs import bf16_bits_to_f64, qlinear_inputs
    inp = qlinear_inputs(8, 2, 192, 5)
    x, s, b = (bf16_bits_to_f64(inp[k]) for k in ("x", "scales", "biases"))
    gsum = x.reshape(2, 3, 64).sum(axis=2)
    np.testing.assert_allclose(oracle.qlinear(x, inp["wq"], np.zeros_like(s), b), gsum @ b.T, rtol=1e-13)
    y = oracle.qlinear(x, inp["wq"], s, b)
    np.testing.assert_allclose(oracle.qlinear(x, inp["wq"], 2 * s, 2 * b), 2 * y, rtol=1e-14)
    np.testing.assert_allclose(oracle.qlinear(3 * x[:1] - x[1:], inp["wq"], s, b), 3 * y[:1] - y[1:],
                               rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- attention decode
def _attn_case(seed, S, Hq, Hkv, D, Tmax, lengths):
    from seeded_inputs import attn_inputs
    inp = attn_inputs(seed, S, Hq, Hkv, D, Tmax, lengths, act="f32")
    return {k: (v.astype(np.float64) if k not in ("lengths", "act") else v) for k, v in inp.items()}


def test_attn_single_position_returns_the_new_value():
    """With nothing cached the softmax has one term: every query head of a
    group returns its kv head's new value exactly, whatever q and scale."""
    import oracle
    c = _attn_case(21, 2, 6, 2, 8, 4, [0, 0])
    out = oracle.attn_decode(c["q"], c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], [0, 0], 0.7)
    np.testing.assert_array_equal(out, np.repeat(c["v_new"], 3, axis=1))


def test_attn_equal_keys_average_the_values():
    """Identical keys at every position give uniform weights: the output is
    the plain mean of the values over positions 0..len."""
    import oracle
    c = _attn_case(22, 1, 2, 1, 8, 6, [4])
    k = c["k_cache"]
    k[0, 0, :4] = c["k_new"][0, 0]
    out = oracle.attn_decode(c["q"], c["k_new"], c["v_new"], k, c["v_cache"], [4], 0.3)
    want = np.concatenate([c["v_cache"][0, 0, :4], c["v_new"][0, 0][None]]).mean(axis=0)
    np.testing.assert_allclose(out[0], np.stack([want, want]), rtol=1e-13, atol=1e-15)


def test_attn_two_positions_logistic_form():
    """Two positions: out = v0 + sigmoid(a1 - a0) (v1 - v0), a_t = scale q.k_t."""
    import oracle
    from scipy.special import expit
    c = _attn_case(23, 1, 1, 1, 16, 3, [1])
    q, k0, k1 = c["q"][0, 0], c["k_cache"][0, 0, 0], c["k_new"][0, 0]
    v0, v1 = c["v_cache"][0, 0, 0].copy(), c["v_new"][0, 0]
    sc = 0.25
    a0 = sc * sum(q[i] * k0[i] for i in range(16))
    a1 = sc * sum(q[i] * k1[i] for i in range(16))
    out = oracle.attn_decode(c["q"], c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], [1], sc)
    np.testing.assert_allclose(out[0, 0], v0 + expit(a1 - a0) * (v1 - v0), rtol=1e-12, atol=1e-14)


def test_attn_query_heads_read_contiguous_kv_groups():
    """Hq = 6 query heads over Hkv = 2 kv heads: heads 0-2 read kv head 0 and
    heads 3-5 kv head 1 (values constant per kv head give exactly that)."""
    import oracle
    c = _attn_case(24, 1, 6, 2, 8, 5, [3])
    for g in range(2):
        c["v_cache"][0, g] = g + 1.0
        c["v_new"][0, g] = g + 1.0
    out = oracle.attn_decode(c["q"], c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], [3], 0.5)
    np.testing.assert_array_equal(out[0, :, 0], [1, 1, 1, 2, 2, 2])


def test_attn_shift_and_scale_invariances():
    """Adding alpha q_h to every key of head h (Hq = Hkv) shifts all its
    scores equally and leaves its output unchanged; the scale multiplies the
    scores, so (scale, q) and (1, scale q) agree."""
    import oracle
    c = _attn_case(25, 2, 3, 3, 16, 9, [8, 5])
    ref = oracle.attn_decode(c["q"], c["k_new"], c["v_new"], c["k_cache"].copy(), c["v_cache"].copy(),
                             c["lengths"], 0.4)
    shifted_k = c["k_cache"] + 0.7 * c["q"][:, :, None, :]
    shifted_new = c["k_new"] + 0.7 * c["q"]
    out = oracle.attn_decode(c["q"], shifted_new, c["v_new"], shifted_k, c["v_cache"].copy(), c["lengths"], 0.4)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)
    out2 = oracle.attn_decode(0.4 * c["q"], c["k_new"], c["v_new"], c["k_cache"].copy(), c["v_cache"].copy(),
                              c["lengths"], 1.0)
    np.testing.assert_allclose(out2, ref, rtol=1e-12, atol=1e-14)


def test_attn_dominant_key_selects_its_value():
    """A key at position 2 equal to 50 q (score 50 |q|^2 scale) dominates
    every other position: the output is that position's value."""
    import oracle
    c = _attn_case(26, 1, 1, 1, 16, 8, [6])
    c["k_cache"][0, 0, 2] = 50.0 * c["q"][0, 0]
    out = oracle.attn_decode(c["q"], c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], [6], 1.0)
    np.testing.assert_allclose(out[0, 0], c["v_cache"][0, 0, 2], rtol=1e-12, atol=1e-14)


def test_attn_appends_and_touches_nothing_else():
    """Position len[s] receives the new key and value; every other slot keeps
    its bits; a length outside [0, Tmax) is refused."""
    import oracle
    c = _attn_case(27, 3, 4, 2, 8, 6, [0, 2, 5])
    k0, v0 = c["k_cache"].copy(), c["v_cache"].copy()
    oracle.attn_decode(c["q"], c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], c["lengths"], 0.35)
    for s, L in enumerate(c["lengths"]):
        k0[s, :, L], v0[s, :, L] = c["k_new"][s], c["v_new"][s]
    np.testing.assert_array_equal(c["k_cache"], k0)
    np.testing.assert_array_equal(c["v_cache"], v0)
    with pytest.raises(RuntimeError):
        oracle.attn_decode(c["q"], c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], [0, 2, 6], 0.35)


# ------------------------------------------------ hybrid model blocks (NEXT-4)
def test_rmsnorm_is_torch_rms_norm():
    import oracle
    rng = np.random.default_rng(40)
    x = rng.standard_normal((5, 96))
    w = 1 + 0.1 * rng.standard_normal(96)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (96,), torch.tensor(w), eps=1e-5).numpy()
    assert rel(oracle.rmsnorm(x, w, 1e-5), ref) < 1e-14


def test_rmsnorm_worked_case():
    """x = (3, 4): mean of squares 12.5, so x / sqrt(12.5) = (0.8485.., 1.1313..)."""
    import oracle
    out = oracle.rmsnorm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    np.testing.assert_allclose(out, [[3 / np.sqrt(12.5), 8 / np.sqrt(12.5)]], rtol=1e-15)


def _tiny_lm(S=2, max_len=16, seed=41):
    from oracle.lm import LMOracle
    from seeded_inputs import TINY_LM, lm_weights
    return LMOracle(TINY_LM, lm_weights(seed, TINY_LM), S, max_len)


def test_lm_stepping_equals_recompute():
    """The cached position stepped T times == the full-history recompute of
    the T positions (scan form of every Mamba block, attention over the
    positions in order): the model-level form of the Offline-timeline
    statement that both modes give the same tokens."""
    from seeded_inputs import TINY_LM, lm_hidden
    S, T = 2, 7
    H = lm_hidden(42, TINY_LM, S, T)
    a, b = _tiny_lm(S), _tiny_lm(S)
    stepped = np.stack([a.step(H[:, t]) for t in range(T)], axis=1)
    recomputed = b.prefill(H)
    assert rel(stepped, recomputed) < 1e-12
    for i in a.ssm:
        assert rel(a.ssm[i], b.ssm[i]) < 1e-12
        np.testing.assert_array_equal(a.conv[i], b.conv[i])
    for i in a.kc:
        np.testing.assert_array_equal(a.kc[i], b.kc[i])
    np.testing.assert_array_equal(a.lengths, b.lengths)


def test_lm_recompute_continues_from_its_caches():
    """Prefill of T1 positions, then of T2 more from the caches it left ==
    prefill of all T1 + T2 positions at once."""
    from seeded_inputs import TINY_LM, lm_hidden
    S, T1, T2 = 2, 3, 5
    H = lm_hidden(43, TINY_LM, S, T1 + T2)
    a, b = _tiny_lm(S), _tiny_lm(S)
    two = np.concatenate([a.prefill(H[:, :T1]), a.prefill(H[:, T1:])], axis=1)
    assert rel(two, b.prefill(H)) < 1e-12


def test_lm_blocks_with_zero_output_weights_pass_h_through():
    """With out_proj and Wo zero every block adds exactly zero: the residual
    stream leaves the last block as it entered (bf16 values stay exact)."""
    from seeded_inputs import TINY_LM, lm_hidden
    from oracle.lm import rb
    lm = _tiny_lm(2)
    for L in lm.w:
        if "out_scales" in L:
            L["out_scales"] = np.zeros_like(L["out_scales"])
            L["out_biases"] = np.zeros_like(L["out_biases"])
        else:
            L["wo"] = np.zeros_like(L["wo"])
    H = lm_hidden(44, TINY_LM, 2, 1)
    h0 = rb(as_f64(H[:, 0], "bf16"))
    np.testing.assert_array_equal(lm.step(H[:, 0]), h0)
    assert np.any(lm.ssm[0] != 0)  # the blocks did run


def test_lm_first_position_attention_returns_its_value():
    """At the first position each attention block attends only to the new
    key, so its output is the new value: o = v exactly (softmax of one
    score), which pins the q|k|v split of the projection."""
    from seeded_inputs import TINY_LM, lm_hidden
    lm = _tiny_lm(1)
    i = TINY_LM.kinds.index("*")
    H = lm_hidden(45, TINY_LM, 1, 1)
    h = as_f64(H[:, 0], "bf16")
    # run the blocks before the first attention block, then its projections
    for j in range(i):
        L = lm.w[j]
        proj = lm._mamba_in(L, h)
        z, x, B, C, dt = lm._split(proj)
        d = TINY_LM.mixer
        frame = dict(x=x.reshape(1, d.H, d.P), B=B.reshape(1, d.G, d.N), C=C.reshape(1, d.G, d.N), dt_raw=dt,
                     act="f32")
        from oracle import mixer_step
        y = np.asarray(mixer_step(d, frame, L, lm.ssm[j], lm.conv[j])).reshape(1, -1)
        from oracle.lm import rb
        h = lm._mamba_out(L, h, rb(y), z)
    q, k, v = lm._qkv(lm.w[i], h)
    o = lm._attend(i, q, k, v, 0)
    R = TINY_LM.n_heads // TINY_LM.n_kv_heads
    np.testing.assert_array_equal(o.reshape(TINY_LM.n_heads, -1),
                                  np.repeat(v.reshape(TINY_LM.n_kv_heads, -1), R, axis=0))


def test_lm_drift_gate_catches_a_missing_block():
    """The end-to-end gate has the power it claims: the oracle's position
    with one block left out lies beyond it."""
    from oracle.lm import LMOracle
    from seeded_inputs import TINY_LM, LMConfig, lm_hidden, lm_weights
    from m2_testlib import BF16_U
    cfg = TINY_LM
    w = lm_weights(562, cfg)
    H = lm_hidden(563, cfg, 2, 1)
    full = LMOracle(cfg, w, 2, 4).step(H[:, 0])
    for drop in range(len(cfg.kinds)):
        keep = [i for i in range(len(cfg.kinds)) if i != drop]
        sub = LMConfig(cfg.hidden, cfg.mixer, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                       "".join(cfg.kinds[i] for i in keep), cfg.eps)
        part = LMOracle(sub, [w[i] for i in keep], 2, 4).step(H[:, 0])
        err = np.linalg.norm(part - full) / np.linalg.norm(full)
        assert err > 2.0 * BF16_U * np.sqrt(len(cfg.kinds)), drop
