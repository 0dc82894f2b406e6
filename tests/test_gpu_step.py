"""GPU parity of the single-frame cached step (mamba2_step) against the fp64
oracle, through the C ABI. The step is the per-position update of the
persistent Mamba2 state ("docs/nemotron-voicechat.md", section Online
session) and must reproduce full-history recompute (same doc, Offline
timeline)."""
import numpy as np
import pytest

from m2_testlib import act_empty, bits_of, check_state, check_y, from_dev_act, to_dev
from seeded_inputs import (REAL_SHAPE, TINY_SHAPE, Dims, as_f64, conv_state_inputs, mixer_inputs,
                           ssm_state_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m2():
    import full_duplex_speech_gb300 as m2
    m2.load()
    return m2


def _params_dev(inp):
    return {k: to_dev(inp[k]) for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b")}


def _frame(inp, t):
    f = {k: np.ascontiguousarray(inp[k][:, t]) for k in ("x", "B", "C", "dt_raw")}
    f["act"] = inp["act"]
    return f


def _gpu_step(m2, d, S, frame, pdev, ssm_dev, conv_dev, act):
    import torch
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, act)
    ws = torch.zeros(m2.mamba2_step_workspace_bytes(dims, S), dtype=torch.uint8, device="cuda")
    y = act_empty((S, d.H, d.P), act)
    fd = {k: to_dev(frame[k]) for k in ("x", "B", "C", "dt_raw")}
    m2.mamba2_step(dims, S, fd["x"], fd["B"], fd["C"], fd["dt_raw"], pdev["A_log"], pdev["D"],
                   pdev["dt_bias"], pdev["conv_w"], pdev["conv_b"], ssm_dev, conv_dev, y, ws)
    torch.cuda.synchronize()
    return y


def _tail_bits(conv_init, frame, d):
    """Expected conv tail after one frame: [init[1], init[2], this frame]."""
    S = frame["x"].shape[0]
    cur = np.concatenate([frame["x"].reshape(S, -1), frame["B"].reshape(S, -1),
                          frame["C"].reshape(S, -1)], axis=1)
    return np.concatenate([conv_init[:, 1:], cur[:, None, :]], axis=1)


# group sizes H/G: 4 (tiny), 16 (real), 4, 2, 1 (one head per group) and 32
# (B and C tails read by 32 heads)
WIDE_GROUP = Dims(H=32, P=16, N=16, G=1)


@pytest.mark.parametrize("shape,act,S", [(TINY_SHAPE, "f32", 3), (REAL_SHAPE, "bf16", 4),
                                         (Dims(H=8, P=32, N=64, G=2), "bf16", 5),
                                         (Dims(H=6, P=48, N=32, G=3), "f32", 2),
                                         (Dims(H=4, P=16, N=16, G=4), "f32", 2),
                                         (WIDE_GROUP, "bf16", 3)])
def test_step_one_frame_from_random_state(m2, shape, act, S):
    d = shape
    inp = mixer_inputs(101, d, S, 1, act)
    ssm0 = ssm_state_inputs(102, d, S, scale=0.2)
    conv0 = conv_state_inputs(103, d, S, act)
    ssm_dev, conv_dev = to_dev(ssm0), to_dev(conv0)
    y = _gpu_step(m2, d, S, _frame(inp, 0), _params_dev(inp), ssm_dev, conv_dev, act)

    ssm_ref = ssm0.astype(np.float64).copy()
    conv_ref = as_f64(conv0, act).copy()
    import oracle
    y_ref = oracle.mixer_step(d, _frame(inp, 0), inp, ssm_ref, conv_ref)

    check_y(from_dev_act(y, act), y_ref, act)
    check_state(ssm_dev.cpu().numpy(), ssm_ref)
    exp_tail = _tail_bits(conv0, _frame(inp, 0), d)
    np.testing.assert_array_equal(bits_of(conv_dev), np.ascontiguousarray(exp_tail).view(np.uint8).reshape(-1))


@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_step_sequence_equals_recompute(m2, act):
    """20 cached steps from zero state == the oracle's full-history scan."""
    import torch
    import oracle
    d = REAL_SHAPE if act == "bf16" else TINY_SHAPE
    S, T = 2, 20
    inp = mixer_inputs(104, d, S, T, act)
    pdev = _params_dev(inp)
    ssm_dev = torch.zeros((S, d.H, d.P, d.N), dtype=torch.float32, device="cuda")
    conv_dev = act_empty((S, d.K - 1, d.CH), act).zero_()
    ys = [from_dev_act(_gpu_step(m2, d, S, _frame(inp, t), pdev, ssm_dev, conv_dev, act), act)
          for t in range(T)]
    y = np.stack(ys, axis=1)
    ref = oracle.mixer_scan(d, inp)
    check_y(y, ref["y"], act)
    check_state(ssm_dev.cpu().numpy(), ref["final_ssm"])
    x, B, C = (inp[k] for k in "xBC")
    full = np.concatenate([x.reshape(S, T, -1), B.reshape(S, T, -1), C.reshape(S, T, -1)], axis=2)
    np.testing.assert_array_equal(bits_of(conv_dev), np.ascontiguousarray(full[:, -3:]).view(np.uint8).reshape(-1))


def test_step_sequence_equals_recompute_wide_group(m2):
    """8 cached steps from zero state with 32 heads sharing one group's B and C
    == the oracle's full-history scan, conv tail included."""
    import torch
    import oracle
    d, act, S, T = WIDE_GROUP, "bf16", 2, 8
    inp = mixer_inputs(108, d, S, T, act)
    pdev = _params_dev(inp)
    ssm_dev = torch.zeros((S, d.H, d.P, d.N), dtype=torch.float32, device="cuda")
    conv_dev = act_empty((S, d.K - 1, d.CH), act).zero_()
    ys = [from_dev_act(_gpu_step(m2, d, S, _frame(inp, t), pdev, ssm_dev, conv_dev, act), act)
          for t in range(T)]
    ref = oracle.mixer_scan(d, inp)
    check_y(np.stack(ys, axis=1), ref["y"], act)
    check_state(ssm_dev.cpu().numpy(), ref["final_ssm"])
    x, B, C = (inp[k] for k in "xBC")
    full = np.concatenate([x.reshape(S, T, -1), B.reshape(S, T, -1), C.reshape(S, T, -1)], axis=2)
    np.testing.assert_array_equal(bits_of(conv_dev), np.ascontiguousarray(full[:, -3:]).view(np.uint8).reshape(-1))


def test_step_many_sessions_real_shape(m2):
    """64 sessions at the real shape, each from its own random state."""
    import oracle
    d, S, act = REAL_SHAPE, 64, "bf16"
    inp = mixer_inputs(105, d, S, 1, act)
    ssm0 = ssm_state_inputs(106, d, S, scale=0.3)
    conv0 = conv_state_inputs(107, d, S, act)
    ssm_dev, conv_dev = to_dev(ssm0), to_dev(conv0)
    y = _gpu_step(m2, d, S, _frame(inp, 0), _params_dev(inp), ssm_dev, conv_dev, act)
    ssm_ref = ssm0.astype(np.float64).copy()
    conv_ref = as_f64(conv0, act).copy()
    y_ref = oracle.mixer_step(d, _frame(inp, 0), inp, ssm_ref, conv_ref, nthreads=0)
    check_y(from_dev_act(y, act), y_ref, act)
    check_state(ssm_dev.cpu().numpy(), ssm_ref)


def test_step_zero_sessions_is_a_noop(m2):
    import torch
    d = TINY_SHAPE
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, "f32")
    one = torch.zeros(16, device="cuda")
    rc = m2.mamba2_step(dims, 0, one, one, one, one, one, one, one, one, one, one, one, one, one,
                        workspace_bytes=0)
    assert rc == 0


def test_step_rejects_bad_arguments_on_gpu(m2):
    import torch
    d = TINY_SHAPE
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, "f32")
    buf = torch.zeros(1 << 16, device="cuda")
    ws = torch.zeros(m2.mamba2_step_workspace_bytes(dims, 1), dtype=torch.uint8, device="cuda")
    args = [buf] * 12
    assert m2.mamba2_step(dims, 1, *args, ws, check=False) == 0
    torch.cuda.synchronize()
    # misaligned y
    assert m2.mamba2_step(dims, 1, *args[:11], buf.data_ptr() + 4, ws, workspace_bytes=ws.numel(),
                          check=False) == 3
    # workspace too small
    assert m2.mamba2_step(dims, 1, *args, ws, workspace_bytes=16, check=False) == 6


@pytest.mark.parametrize("S", [1, 8, 15, 16])
def test_step_session_counts_real_shape(m2, S):
    """1 to 16 sessions at the real shape, each from its own random state,
    against the oracle, conv tail included."""
    import oracle
    d, act = REAL_SHAPE, "bf16"
    inp = mixer_inputs(110 + S, d, S, 1, act)
    ssm0 = ssm_state_inputs(111, d, S, scale=0.2)
    conv0 = conv_state_inputs(112, d, S, act)
    ssm_dev, conv_dev = to_dev(ssm0), to_dev(conv0)
    y = _gpu_step(m2, d, S, _frame(inp, 0), _params_dev(inp), ssm_dev, conv_dev, act)
    ssm_ref = ssm0.astype(np.float64).copy()
    conv_ref = as_f64(conv0, act).copy()
    y_ref = oracle.mixer_step(d, _frame(inp, 0), inp, ssm_ref, conv_ref, nthreads=0)
    check_y(from_dev_act(y, act), y_ref, act)
    check_state(ssm_dev.cpu().numpy(), ssm_ref)
    exp_tail = _tail_bits(conv0, _frame(inp, 0), d)
    np.testing.assert_array_equal(bits_of(conv_dev), np.ascontiguousarray(exp_tail).view(np.uint8).reshape(-1))


def test_step_saturated_silu_channels(m2):
    """The step's conv + SiLU with pre-activations far below zero (bias -300 on
    every other channel): SiLU saturates to zero as in the oracle."""
    d, S, act = Dims(H=8, P=32, N=64, G=2), 3, "bf16"
    inp = mixer_inputs(910, d, S, 1, act)
    inp["conv_b"] = inp["conv_b"].copy()
    inp["conv_b"][::2] = -300.0
    ssm0 = ssm_state_inputs(911, d, S, scale=0.2)
    conv0 = conv_state_inputs(912, d, S, act)
    ssm_dev, conv_dev = to_dev(ssm0), to_dev(conv0)
    y = _gpu_step(m2, d, S, _frame(inp, 0), _params_dev(inp), ssm_dev, conv_dev, act)
    ssm_ref = ssm0.astype(np.float64).copy()
    conv_ref = as_f64(conv0, act).copy()
    import oracle
    y_ref = oracle.mixer_step(d, _frame(inp, 0), inp, ssm_ref, conv_ref)
    assert np.isfinite(from_dev_act(y, act)).all()
    check_y(from_dev_act(y, act), y_ref, act)
    check_state(ssm_dev.cpu().numpy(), ssm_ref)
