"""GPU parity of the 4-bit affine group-quantized linear layer (mamba2_qlinear:
the Mamba layer's in/out projections as the VoiceChat 4-bit checkpoint stores
them, Nemotron VoiceChat page, config.json `quantization`: group_size 64,
bits 4) against the fp64 oracle, through the C ABI. Sizes cover every
rows-per-pass form (1, 2 and 4 rows of x per pass over the weights), ragged
passes, the smallest and largest input widths, and the real projection shapes
(in_proj 4480 -> 22656, out_proj 10240 -> 4480)."""
import numpy as np
import pytest

from m2_testlib import check_y, from_dev_act, to_dev
from seeded_inputs import bf16_bits_to_f64, qlinear_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m2():
    import full_duplex_speech_gb300 as m2
    m2.load()
    return m2


def gpu_qlinear(m2, inp, rows, n_in, n_out):
    import torch
    x = to_dev(inp["x"])
    wq = torch.from_numpy(inp["wq"].view(np.int32)).cuda()
    s, b = to_dev(inp["scales"]), to_dev(inp["biases"])
    y = torch.full((rows, n_out), float("nan"), dtype=torch.bfloat16, device="cuda")
    m2.mamba2_qlinear(rows, n_in, n_out, x, wq, s, b, y)
    torch.cuda.synchronize()
    return y


def oracle_qlinear(inp):
    import oracle
    return oracle.qlinear(bf16_bits_to_f64(inp["x"]), inp["wq"], bf16_bits_to_f64(inp["scales"]),
                          bf16_bits_to_f64(inp["biases"]))


@pytest.mark.parametrize("rows,n_in,n_out", [
    (1, 64, 8), (1, 16384, 33),                                               # 1 row per pass
    (2, 10240, 100), (2, 14208, 17), (3, 16384, 65),                          # 2 rows per pass
    (3, 256, 40), (4, 512, 129), (5, 4480, 300), (9, 2048, 77), (6, 12480, 9),  # 4 rows per pass
])
def test_qlinear_shapes(m2, rows, n_in, n_out):
    inp = qlinear_inputs(rows * 1000 + n_in + n_out, rows, n_in, n_out)
    y = gpu_qlinear(m2, inp, rows, n_in, n_out)
    check_y(from_dev_act(y, "bf16"), oracle_qlinear(inp), "bf16")


@pytest.mark.parametrize("rows,n_in,n_out", [(1, 4480, 22656), (4, 4480, 22656), (1, 10240, 4480),
                                             (3, 10240, 4480)])
def test_qlinear_nemotron_projections(m2, rows, n_in, n_out):
    inp = qlinear_inputs(77 + rows, rows, n_in, n_out)
    y = gpu_qlinear(m2, inp, rows, n_in, n_out)
    check_y(from_dev_act(y, "bf16"), oracle_qlinear(inp), "bf16")


def test_qlinear_worked_example(m2):
    """The oracle pins' hand-written two-row weights (q = i % 16 with scale
    0.5, bias -4; q = 15 - i % 16 with scale 2, bias 1) read by unit vectors
    and by an all-ones x: every result is exact in bf16."""
    import torch
    from seeded_inputs import f32_to_bf16_bits
    wq = np.array([[0x76543210, 0xFEDCBA98] * 4, [0x89ABCDEF, 0x01234567] * 4], dtype=np.uint32)
    xs = np.zeros((5, 64), dtype=np.float32)
    xs[0] = 1.0
    for r, i in enumerate((13, 63, 0, 8)):
        xs[r + 1, i] = 1.0
    inp = dict(x=f32_to_bf16_bits(xs), wq=wq, scales=f32_to_bf16_bits(np.array([[0.5], [2.0]], np.float32)),
               biases=f32_to_bf16_bits(np.array([[-4.0], [1.0]], np.float32)))
    y = gpu_qlinear(m2, inp, 5, 64, 2).float().cpu().numpy()
    np.testing.assert_array_equal(y, [[-16, 1024], [2.5, 5], [3.5, 1], [-4, 31], [0, 15]])


def test_qlinear_zero_rows_is_a_noop(m2):
    import torch
    inp = qlinear_inputs(5, 1, 128, 16)
    x = to_dev(inp["x"])
    wq = torch.from_numpy(inp["wq"].view(np.int32)).cuda()
    y = torch.full((1, 16), 3.0, dtype=torch.bfloat16, device="cuda")
    m2.mamba2_qlinear(0, 128, 16, x, wq, to_dev(inp["scales"]), to_dev(inp["biases"]), y)
    torch.cuda.synchronize()
    assert (y == 3.0).all()


# ------------------------------------------------ many rows: the tensor-core GEMM
# From 40 rows of x without a fused norm the layer runs as a tcgen05 GEMM over
# tiles of 128 rows x 64 outputs, one 64-input group per accumulation.
@pytest.mark.parametrize("rows,n_in,n_out", [
    (40, 64, 136),        # the fewest rows and one group; 8 outputs past two tiles (enough
                          # elements for the 0.1% share gate to allow a miss near zero)
    (129, 128, 65),       # one row and one output past a tile
    (200, 4480, 100),     # in_proj's input width
    (300, 4480, 22656),   # in_proj over a 300-position prefill
    (300, 10240, 4480),   # out_proj over a 300-position prefill
])
def test_qlinear_gemm_shapes(m2, rows, n_in, n_out):
    inp = qlinear_inputs(rows * 7 + n_in + n_out, rows, n_in, n_out)
    y = gpu_qlinear(m2, inp, rows, n_in, n_out)
    assert m2.mamba2_device_error() == 0
    check_y(from_dev_act(y, "bf16"), oracle_qlinear(inp), "bf16")


def test_qlinear_gemm_worked_example(m2):
    """The hand-written two-row weights of the worked example, read by 40 rows
    of x (the GEMM): unit vectors at each of the 8 field positions of a word
    and at both ends of the group pin the nibble order; every result is
    exact in bf16."""
    from seeded_inputs import f32_to_bf16_bits
    wq = np.array([[0x76543210, 0xFEDCBA98] * 4, [0x89ABCDEF, 0x01234567] * 4], dtype=np.uint32)
    cols = [13, 63, 0, 8, 1, 2, 3, 4, 5, 6, 7, 9, 33, 62, 31, 32, 47, 48, 15] * 2 + [40]
    xs = np.zeros((len(cols) + 1, 64), dtype=np.float32)
    xs[0] = 1.0
    for r, i in enumerate(cols):
        xs[r + 1, i] = 1.0
    inp = dict(x=f32_to_bf16_bits(xs), wq=wq, scales=f32_to_bf16_bits(np.array([[0.5], [2.0]], np.float32)),
               biases=f32_to_bf16_bits(np.array([[-4.0], [1.0]], np.float32)))
    y = gpu_qlinear(m2, inp, xs.shape[0], 64, 2).float().cpu().numpy()
    q0 = np.array([i % 16 for i in range(64)], np.float64)
    q1 = 15 - q0
    ref = np.stack([xs @ (0.5 * q0 - 4.0), xs @ (2.0 * q1 + 1.0)], axis=1)
    np.testing.assert_array_equal(y, ref)


def test_qlinear_gemm_residual_and_row_stride(m2):
    """The GEMM with x read as a slice of wider rows and a residual added
    before the one rounding (mamba2_qlinear_fused without a norm)."""
    import torch
    rows, n_in, n_out, pitch = 96, 256, 136, 320
    inp = qlinear_inputs(4321, rows, n_in, n_out)
    xw = torch.zeros((rows, pitch), dtype=torch.bfloat16, device="cuda")
    xw[:, 32:32 + n_in] = to_dev(inp["x"])
    res = torch.randn((rows, n_out), device="cuda").to(torch.bfloat16)
    y = torch.full((rows, n_out), float("nan"), dtype=torch.bfloat16, device="cuda")
    wq = torch.from_numpy(inp["wq"].view(np.int32)).cuda()
    m2.mamba2_qlinear_fused(rows, n_in, n_out, xw[:, 32:], pitch, None, wq, to_dev(inp["scales"]),
                            to_dev(inp["biases"]), res, y)
    torch.cuda.synchronize()
    assert m2.mamba2_device_error() == 0
    ref = oracle_qlinear(inp) + from_dev_act(res, "bf16")
    check_y(from_dev_act(y, "bf16"), ref, "bf16")
