"""mamba2_step_noalloc: the cached step for callers that cannot allocate
device memory (a real-time frame loop that must not call cudaMalloc, a host
that only hands over tensors it already owns, a binding without a device
allocator). It runs the step on a fixed scratch array inside the library
instead of a caller workspace.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test. It passes alone in a fresh process
(the first call on the device does the one-time set-up) and after the others.
"""
import numpy as np
import pytest

from m2_testlib import STATE_TOL, Y_TOL, act_empty, bits_of, from_dev_act, state_error, to_dev, y_error
from seeded_inputs import REAL_SHAPE, conv_state_inputs, mixer_inputs, ssm_state_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m2():
    import full_duplex_speech_gb300 as m2
    m2.load()
    return m2


def test_noalloc_step_matches_workspace_step_two_calls(m2):
    import torch
    d, S, act = REAL_SHAPE, 8, "bf16"
    inp = mixer_inputs(900, d, S, 2, act)
    pd = {k: to_dev(inp[k]) for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b")}
    ssm0 = to_dev(ssm_state_inputs(901, d, S, scale=0.05))
    conv0 = to_dev(conv_state_inputs(902, d, S, act))
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, act)

    # reference path: the existing entry point with a caller workspace
    ssm_a, conv_a = ssm0.clone(), conv0.clone()
    ws = torch.empty(m2.mamba2_step_workspace_bytes(dims, S), dtype=torch.uint8, device="cuda")
    # path under test: the fixed library scratch, no workspace argument
    ssm_b, conv_b = ssm0.clone(), conv0.clone()
    for t in range(2):  # two calls in a row, each continuing from the last
        fr = {k: to_dev(np.ascontiguousarray(inp[k][:, t])) for k in ("x", "B", "C", "dt_raw")}
        ya = act_empty((S, d.H, d.P), act)
        yb = act_empty((S, d.H, d.P), act)
        m2.mamba2_step(dims, S, fr["x"], fr["B"], fr["C"], fr["dt_raw"], pd["A_log"], pd["D"], pd["dt_bias"],
                       pd["conv_w"], pd["conv_b"], ssm_a, conv_a, ya, ws)
        m2.mamba2_step_noalloc(dims, S, fr["x"], fr["B"], fr["C"], fr["dt_raw"], pd["A_log"], pd["D"],
                               pd["dt_bias"], pd["conv_w"], pd["conv_b"], ssm_b, conv_b, yb)
        torch.cuda.synchronize()
        assert y_error(from_dev_act(yb, act), from_dev_act(ya, act).astype(np.float64), act) <= Y_TOL
        assert state_error(ssm_b.cpu().numpy(), ssm_a.cpu().numpy().astype(np.float64)) <= STATE_TOL
        np.testing.assert_array_equal(bits_of(conv_b), bits_of(conv_a))


def test_noalloc_rejects_requests_beyond_its_scratch(m2):
    import torch
    d, act = REAL_SHAPE, "bf16"
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, act)
    cap = m2.mamba2_step_noalloc_max_bytes()
    assert cap == 1 << 20
    fits = max(s for s in range(1, 64) if m2.mamba2_step_workspace_bytes(dims, s) <= cap)
    assert fits == 21
    buf = torch.zeros(1 << 20, device="cuda")
    rc = m2.mamba2_step_noalloc(dims, fits + 1, *([buf] * 12), check=False)
    assert rc == 6  # M2_EWORKSPACE: nothing was launched
