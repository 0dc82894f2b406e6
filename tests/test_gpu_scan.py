"""GPU parity of the chunked scan (mamba2_conv_scan) against the fp64 oracle,
through the C ABI: the tiny fp32 mixer, the real Nemotron-H mixer shape
(H=128, P=80, N=128, G=8; issue "feat(nemotron_voicechat): ...", section
config.json / text_config), ragged and empty sequences, continuation from a
cached state, and agreement with the cached step ("docs/nemotron-voicechat.md",
section Offline timeline: recompute and cached mode agree)."""
import numpy as np
import pytest

from m2_testlib import act_empty, bits_of, check_scan_y, check_state, check_y, from_dev_act, to_dev
from seeded_inputs import (REAL_SHAPE, TINY_SHAPE, Dims, conv_state_inputs, mixer_inputs,
                           ssm_state_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m2():
    import full_duplex_speech_gb300 as m2
    m2.load()
    return m2


def gpu_scan(m2, d, inp, chunk, batch, T, init_ssm=None, init_conv=None, in_place=False):
    """Runs mamba2_conv_scan; returns (y, final_ssm, final_conv) device tensors."""
    import torch
    act = inp["act"]
    dims = m2.dims(batch, T, d.H, d.P, d.N, d.G, d.K, act)
    dev = {k: to_dev(inp[k]) for k in ("x", "B", "C", "dt_raw", "A_log", "D", "dt_bias", "conv_w", "conv_b")}
    y = act_empty((batch, T, d.H, d.P), act)
    iss = None if init_ssm is None else to_dev(init_ssm)
    ic = None if init_conv is None else to_dev(init_conv)
    if in_place:
        fs, fc = iss, ic
    else:
        fs = torch.empty((batch, d.H, d.P, d.N), dtype=torch.float32, device="cuda")
        fc = act_empty((batch, d.K - 1, d.CH), act)
    nbytes = m2.mamba2_scan_workspace_bytes(dims, chunk)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    m2.mamba2_conv_scan(dims, dev["x"], dev["B"], dev["C"], dev["dt_raw"], dev["A_log"], dev["D"],
                        dev["dt_bias"], dev["conv_w"], dev["conv_b"], chunk, iss, ic, y, fs, fc, ws)
    torch.cuda.synchronize()
    assert m2.mamba2_device_error() == 0
    return y, fs, fc


def expected_tail_bits(inp, d, init_conv=None):
    b, T = inp["x"].shape[:2]
    full = np.concatenate([inp["x"].reshape(b, T, d.H * d.P), inp["B"].reshape(b, T, d.G * d.N),
                           inp["C"].reshape(b, T, d.G * d.N)], axis=2)
    pre = init_conv if init_conv is not None else np.zeros((b, d.K - 1, d.CH), full.dtype)
    return np.ascontiguousarray(np.concatenate([pre, full], axis=1)[:, -(d.K - 1):])


def check(m2, d, inp, chunk, batch, T, init_ssm=None, init_conv=None, in_place=False, heads=None):
    import oracle
    act = inp["act"]
    y, fs, fc = gpu_scan(m2, d, inp, chunk, batch, T, init_ssm, init_conv, in_place)
    ref = oracle.mixer_scan(d, inp, init_ssm=init_ssm, init_conv=init_conv, heads=heads)
    hs = slice(None) if heads is None else slice(*heads)
    if T > 0:
        ybar = oracle.mixer_scan_magnitude(d, inp, init_ssm=init_ssm, init_conv=init_conv, heads=heads)
        check_scan_y(from_dev_act(y, act)[:, :, hs], ref["y"][:, :, hs], ybar[:, :, hs], act)
    check_state(fs.cpu().numpy()[:, hs], ref["final_ssm"][:, hs])
    np.testing.assert_array_equal(bits_of(fc), expected_tail_bits(inp, d, init_conv).view(np.uint8).reshape(-1))
    return y, fs, fc


@pytest.mark.parametrize("chunk", [8, 16, 64, 128])
def test_tiny_fp32_mixer(m2, chunk):
    d = TINY_SHAPE
    inp = mixer_inputs(0, d, 1, 64, "f32")
    check(m2, d, inp, chunk, 1, 64)


@pytest.mark.parametrize("chunk", [64, 128])
def test_real_shape_one_layer_T300(m2, chunk):
    d = REAL_SHAPE
    inp = mixer_inputs(1, d, 1, 300, "bf16")
    check(m2, d, inp, chunk, 1, 300)


@pytest.mark.parametrize("T,chunk", [(1, 128), (2, 16), (3, 7), (15, 16), (17, 16), (129, 128), (200, 48),
                                     (77, 1)])
def test_ragged_lengths(m2, T, chunk):
    d = Dims(H=8, P=32, N=64, G=2)
    inp = mixer_inputs(2 + T, d, 2, T, "bf16")
    check(m2, d, inp, chunk, 2, T)


@pytest.mark.parametrize("shape", [Dims(H=6, P=48, N=32, G=3), Dims(H=4, P=80, N=128, G=1),
                                   Dims(H=16, P=16, N=16, G=16)])
def test_other_shapes(m2, shape):
    inp = mixer_inputs(31, shape, 3, 90, "f32")
    check(m2, shape, inp, 32, 3, 90)


def _prefix_state(d, seed, batch, T0, act):
    """A cached state as it arises in use: the oracle's final SSM state
    (rounded to fp32) and conv tail after a T0-frame prefix."""
    import oracle
    pre = mixer_inputs(seed, d, batch, T0, act)
    r = oracle.mixer_scan(d, pre)
    tail = expected_tail_bits(pre, d)
    return r["final_ssm"].astype(np.float32), tail


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("T", [0, 2, 45])
def test_continuation_from_cached_state(m2, T, in_place):
    d = Dims(H=8, P=80, N=128, G=2)
    inp = mixer_inputs(40, d, 2, T, "bf16")
    iss, ic = _prefix_state(d, 41, 2, 60, "bf16")
    check(m2, d, inp, 16, 2, T, init_ssm=iss, init_conv=ic, in_place=in_place)


def test_chunk_choice_does_not_change_result(m2):
    d = REAL_SHAPE
    inp = mixer_inputs(50, d, 1, 160, "bf16")
    ys = [from_dev_act(gpu_scan(m2, d, inp, q, 1, 160)[0], "bf16") for q in (32, 80, 128)]
    for y in ys[1:]:
        assert np.linalg.norm(y - ys[0]) / np.linalg.norm(ys[0]) < 2e-3


def test_scan_then_step_equals_longer_scan(m2):
    """Prefill T frames with the scan, then one cached step == a scan of T+1."""
    import torch
    d, T, S = REAL_SHAPE, 37, 2
    inp = mixer_inputs(60, d, S, T + 1, "bf16")
    pre = dict(inp, **{k: np.ascontiguousarray(inp[k][:, :T]) for k in ("x", "B", "C", "dt_raw")})
    _, fs, fc = gpu_scan(m2, d, pre, 16, S, T)
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, "bf16")
    ws = torch.empty(m2.mamba2_step_workspace_bytes(dims, S), dtype=torch.uint8, device="cuda")
    y1 = act_empty((S, d.H, d.P), "bf16")
    fr = {k: to_dev(np.ascontiguousarray(inp[k][:, T])) for k in ("x", "B", "C", "dt_raw")}
    pd = {k: to_dev(inp[k]) for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b")}
    m2.mamba2_step(dims, S, fr["x"], fr["B"], fr["C"], fr["dt_raw"], pd["A_log"], pd["D"], pd["dt_bias"],
                   pd["conv_w"], pd["conv_b"], fs, fc, y1, ws)
    torch.cuda.synchronize()
    import oracle
    ref = oracle.mixer_scan(d, inp)
    check_y(from_dev_act(y1, "bf16"), ref["y"][:, T], "bf16")
    check_state(fs.cpu().numpy(), ref["final_ssm"])
    np.testing.assert_array_equal(bits_of(fc), expected_tail_bits(inp, d).view(np.uint8).reshape(-1))


def test_zero_batch_is_a_noop(m2):
    d = TINY_SHAPE
    dims = m2.dims(0, 64, d.H, d.P, d.N, d.G, d.K, "f32")
    assert m2.mamba2_scan_workspace_bytes(dims, 16) == 0
    import torch
    z = torch.zeros(64, device="cuda")
    rc = m2.mamba2_conv_scan(dims, z, z, z, z, z, z, z, z, z, 16, None, None, z, z, z, None)
    assert rc == 0


@pytest.mark.slow
def test_long_prefill_sampled_heads(m2):
    """b=4, T=4096 at the real shape (one layer of the long-prefill workload):
    y and final state of sampled heads against the oracle."""
    d = REAL_SHAPE
    inp = mixer_inputs(400, d, 4, 4096, "bf16")
    check(m2, d, inp, 128, 4, 4096, heads=(77, 79))


# ------------------------------------------------------ variable-length batches
SENTINEL = 0x5A5A  # bit pattern left in y rows a call must not write


def gpu_scan_varlen(m2, d, inp, chunk, lengths, init_ssm=None, init_conv=None):
    """Runs mamba2_conv_scan_varlen; returns (y, final_ssm, final_conv) device tensors."""
    import torch
    act = inp["act"]
    batch, T = inp["x"].shape[:2]
    dims = m2.dims(batch, T, d.H, d.P, d.N, d.G, d.K, act)
    dev = {k: to_dev(inp[k]) for k in ("x", "B", "C", "dt_raw", "A_log", "D", "dt_bias", "conv_w", "conv_b")}
    lens = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    y = act_empty((batch, T, d.H, d.P), act)
    y.view(torch.int16 if act == "bf16" else torch.int32).fill_(SENTINEL)
    fs = torch.empty((batch, d.H, d.P, d.N), dtype=torch.float32, device="cuda")
    fc = act_empty((batch, d.K - 1, d.CH), act)
    ws = torch.empty(max(m2.mamba2_scan_workspace_bytes(dims, chunk), 16), dtype=torch.uint8, device="cuda")
    m2.mamba2_conv_scan_varlen(dims, lens, dev["x"], dev["B"], dev["C"], dev["dt_raw"], dev["A_log"], dev["D"],
                               dev["dt_bias"], dev["conv_w"], dev["conv_b"], chunk,
                               None if init_ssm is None else to_dev(init_ssm),
                               None if init_conv is None else to_dev(init_conv), y, fs, fc, ws)
    torch.cuda.synchronize()
    assert m2.mamba2_device_error() == 0
    return y, fs, fc


def check_varlen(m2, d, inp, chunk, lengths, init_ssm=None, init_conv=None):
    """Every sequence against the oracle run on its own frames only."""
    import oracle
    act = inp["act"]
    y, fs, fc = gpu_scan_varlen(m2, d, inp, chunk, lengths, init_ssm, init_conv)
    y_bits = bits_of(y).view(np.uint16 if act == "bf16" else np.uint32).reshape(y.shape)
    y_all = from_dev_act(y, act)
    fs_all, fc_bits = fs.cpu().numpy(), bits_of(fc).reshape(len(lengths), -1)
    for b, L in enumerate(lengths):
        sub = dict(inp, **{k: np.ascontiguousarray(inp[k][b:b + 1, :L]) for k in ("x", "B", "C", "dt_raw")})
        iss = None if init_ssm is None else init_ssm[b:b + 1]
        ic = None if init_conv is None else init_conv[b:b + 1]
        ref = oracle.mixer_scan(d, sub, init_ssm=iss, init_conv=ic)
        if L > 0:
            ybar = oracle.mixer_scan_magnitude(d, sub, init_ssm=iss, init_conv=ic)
            check_scan_y(y_all[b:b + 1, :L], ref["y"], ybar, act, tag=f"y[{b}]")
        assert np.all(y_bits[b, L:] == SENTINEL), b  # rows past the length are left alone
        if L == 0:  # the initial state passes through unchanged
            want = np.zeros_like(fs_all[b]) if iss is None else iss[0]
            np.testing.assert_array_equal(fs_all[b], want)
        else:
            check_state(fs_all[b:b + 1], ref["final_ssm"], tag=f"state[{b}]")
        np.testing.assert_array_equal(fc_bits[b], expected_tail_bits(sub, d, ic).view(np.uint8).reshape(-1))


@pytest.mark.parametrize("chunk", [16, 32])
def test_varlen_ragged_batch(m2, chunk):
    d = Dims(H=8, P=32, N=64, G=2)
    lengths = [100, 0, 1, 2, chunk - 1, chunk, chunk + 1, 77]
    inp = mixer_inputs(70 + chunk, d, len(lengths), 100, "bf16")
    check_varlen(m2, d, inp, chunk, lengths)


def test_varlen_continuing_sessions(m2):
    """Sessions catching up from their own cached states, different lengths."""
    d = Dims(H=8, P=80, N=128, G=2)
    lengths = [45, 0, 3, 16, 17, 2]
    inp = mixer_inputs(80, d, len(lengths), 45, "bf16")
    iss, ic = _prefix_state(d, 81, len(lengths), 60, "bf16")
    check_varlen(m2, d, inp, 16, lengths, init_ssm=iss, init_conv=ic)


def test_varlen_real_shape(m2):
    d = REAL_SHAPE
    lengths = [300, 128, 129, 7]
    inp = mixer_inputs(90, d, len(lengths), 300, "bf16")
    check_varlen(m2, d, inp, 128, lengths)


def test_varlen_full_lengths_equal_the_plain_scan(m2):
    """All lengths = T: bit-identical to mamba2_conv_scan."""
    d = Dims(H=8, P=32, N=64, G=2)
    inp = mixer_inputs(95, d, 3, 70, "bf16")
    y0, fs0, fc0 = gpu_scan(m2, d, inp, 32, 3, 70)
    y1, fs1, fc1 = gpu_scan_varlen(m2, d, inp, 32, [70, 70, 70])
    for a_, b_ in ((y0, y1), (fs0, fs1), (fc0, fc1)):
        np.testing.assert_array_equal(bits_of(a_), bits_of(b_))


def test_varlen_lengths_are_clamped(m2):
    """Lengths below 0 act as 0, above T as T."""
    d = Dims(H=4, P=16, N=16, G=1)
    inp = mixer_inputs(96, d, 2, 40, "f32")
    y, fs, fc = gpu_scan_varlen(m2, d, inp, 16, [-5, 1000])
    y1, fs1, fc1 = gpu_scan_varlen(m2, d, inp, 16, [0, 40])
    for a_, b_ in ((y, y1), (fs, fs1), (fc, fc1)):
        np.testing.assert_array_equal(bits_of(a_), bits_of(b_))


@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_saturated_silu_channels(m2, act):
    """Conv pre-activations far below zero (a bias of -300 on every other
    channel of x, B and C) saturate SiLU to zero, as the oracle's exact
    u / (1 + e^-u) does: no NaN or infinity from the overflowing exponential."""
    d = Dims(H=8, P=32, N=64, G=2)
    inp = mixer_inputs(900, d, 2, 150, act)
    inp["conv_b"] = inp["conv_b"].copy()
    inp["conv_b"][::2] = -300.0
    y, fs, _ = check(m2, d, inp, 64, 2, 150)
    assert np.isfinite(from_dev_act(y, act)).all() and np.isfinite(fs.cpu().numpy()).all()
