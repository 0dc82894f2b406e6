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

from m2_testlib import act_empty, bits_of, to_dev
from seeded_inputs import REAL_SHAPE, conv_state_inputs, mixer_inputs, ssm_state_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m2():
    import full_duplex_speech_gb300 as m2
    m2.load()
    return m2


def _run_pair(m2, S, seed):
    """Two calls in a row of mamba2_step (caller workspace) and of
    mamba2_step_noalloc (library scratch) on the same inputs and states, each
    continuing from its own last call; after each pair y, the SSM state and
    the conv tail must be bit-identical (the same kernels on the same inputs)."""
    import torch
    d, act = REAL_SHAPE, "bf16"
    inp = mixer_inputs(seed, d, S, 2, act)
    pd = {k: to_dev(inp[k]) for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b")}
    ssm0 = to_dev(ssm_state_inputs(seed + 1, d, S, scale=0.05))
    conv0 = to_dev(conv_state_inputs(seed + 2, d, S, act))
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, act)

    # reference path: the existing entry point with a caller workspace
    ssm_a, conv_a = ssm0.clone(), conv0.clone()
    ws = torch.empty(m2.mamba2_step_workspace_bytes(dims, S), dtype=torch.uint8, device="cuda")
    # path under test: the fixed library scratch, no workspace argument
    ssm_b, conv_b = ssm0.clone(), conv0.clone()
    for t in range(2):
        fr = {k: to_dev(np.ascontiguousarray(inp[k][:, t])) for k in ("x", "B", "C", "dt_raw")}
        ya = act_empty((S, d.H, d.P), act)
        yb = act_empty((S, d.H, d.P), act)
        m2.mamba2_step(dims, S, fr["x"], fr["B"], fr["C"], fr["dt_raw"], pd["A_log"], pd["D"], pd["dt_bias"],
                       pd["conv_w"], pd["conv_b"], ssm_a, conv_a, ya, ws)
        m2.mamba2_step_noalloc(dims, S, fr["x"], fr["B"], fr["C"], fr["dt_raw"], pd["A_log"], pd["D"],
                               pd["dt_bias"], pd["conv_w"], pd["conv_b"], ssm_b, conv_b, yb)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits_of(yb), bits_of(ya))
        np.testing.assert_array_equal(bits_of(ssm_b), bits_of(ssm_a))
        np.testing.assert_array_equal(bits_of(conv_b), bits_of(conv_a))


def test_noalloc_step_matches_workspace_step_two_calls(m2):
    _run_pair(m2, 8, 900)


def test_noalloc_step_at_the_largest_size_that_fits(m2):
    """21 sessions at the Nemotron-H shape: the step sizes end a few KB short
    of the end of the 1 MiB scratch, where an offset error would write past it."""
    d = REAL_SHAPE
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, "bf16")
    fits = max(s for s in range(1, 64) if m2.mamba2_step_workspace_bytes(dims, s) <= m2.mamba2_step_noalloc_max_bytes())
    assert fits == 21
    _run_pair(m2, fits, 930)


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
