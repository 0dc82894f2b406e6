"""GPU parity of the gated RMSNorm of the mixer output (mamba2_gated_norm)
against the fp64 oracle, through the C ABI. The norm follows the mixer core
in each Mamba layer (the VoiceChat issue, section config.json /
text_config: rms_norm_eps 1e-5, n_groups 8)."""
import numpy as np
import pytest

from m2_testlib import act_empty, bits_of, check_y, from_dev_act, to_dev
from seeded_inputs import REAL_SHAPE, TINY_SHAPE, Dims, as_f64, norm_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m2():
    import full_duplex_speech_gb300 as m2
    m2.load()
    return m2


def gpu_norm(m2, d, inp, rows, eps=1e-5, in_place=False):
    import torch
    act = inp["act"]
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, act)
    y, z, w = to_dev(inp["y"]), to_dev(inp["z"]), to_dev(inp["weight"])
    out = y if in_place else act_empty((rows, d.H * d.P), act)
    m2.mamba2_gated_norm(dims, rows, y, z, w, eps, out)
    torch.cuda.synchronize()
    return out


def oracle_norm(d, inp, eps=1e-5):
    import oracle
    return oracle.gated_norm(as_f64(inp["y"], inp["act"]), as_f64(inp["z"], inp["act"]),
                             inp["weight"].astype(np.float64), d.G, eps)


@pytest.mark.parametrize("rows", [1, 300])
def test_gated_norm_real_shape(m2, rows):
    d = REAL_SHAPE
    inp = norm_inputs(200 + rows, d, rows, "bf16")
    out = gpu_norm(m2, d, inp, rows)
    check_y(from_dev_act(out, "bf16"), oracle_norm(d, inp), "bf16")


@pytest.mark.parametrize("shape,act", [(TINY_SHAPE, "f32"), (Dims(H=6, P=48, N=32, G=3), "bf16"),
                                       (Dims(H=16, P=16, N=16, G=16), "f32"),
                                       (Dims(H=64, P=48, N=16, G=1), "bf16"),
                                       (Dims(H=128, P=80, N=16, G=1), "bf16")])
def test_gated_norm_other_shapes(m2, shape, act):
    """Groups of 16 to 10240 channels (one to four 16-byte vectors per thread)."""
    inp = norm_inputs(210, shape, 7, act)
    out = gpu_norm(m2, shape, inp, 7)
    # fp32 results: fp32 arithmetic throughout, so 1e-5 normwise and elementwise
    check_y(from_dev_act(out, act), oracle_norm(shape, inp), act, l2_tol=2e-3 if act == "bf16" else 1e-5,
            f32_maxnorm=1e-5)


def test_gated_norm_in_place_and_eps(m2):
    d = Dims(H=8, P=32, N=64, G=2)
    inp = norm_inputs(220, d, 5, "bf16")
    a = from_dev_act(gpu_norm(m2, d, inp, 5, eps=0.5), "bf16")
    b = from_dev_act(gpu_norm(m2, d, inp, 5, eps=0.5, in_place=True), "bf16")
    np.testing.assert_array_equal(a, b)
    check_y(a, oracle_norm(d, inp, eps=0.5), "bf16")


def test_gated_norm_zero_rows_is_a_noop(m2):
    import torch
    d = TINY_SHAPE
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, "f32")
    buf = torch.zeros(64, device="cuda")
    assert m2.mamba2_gated_norm(dims, 0, buf, buf, buf, 1e-5, buf) == 0
