"""CPU-side checks of the C ABI: the library loads, exports every function
include/mamba2.h declares, and rejects bad arguments before touching the
GPU (these run without a GPU)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m2():
    from full_duplex_speech_gb300 import build
    build.build()
    import full_duplex_speech_gb300 as m2
    m2.load()
    return m2


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "mamba2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mamba2_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("mamba2_conv_scan", "mamba2_step", "mamba2_scan_workspace_bytes",
              "mamba2_step_workspace_bytes", "mamba2_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(m2):
    import ctypes
    lib = ctypes.CDLL(m2.library_path())
    for n in _declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(m2):
    for s in range(7):
        assert m2.mamba2_status_string(s)
    assert m2.mamba2_status_string(99) == "unknown status"


def _fake_ptrs(n, base=1 << 20):
    return [base + 256 * i for i in range(n)]


def test_step_validation_without_gpu(m2):
    d = m2.dims(0, 0, 4, 16, 16, 1, 4, "f32")
    p = _fake_ptrs(12)
    ws = m2.mamba2_step_workspace_bytes(d, 3)
    assert ws > 0
    ok = dict(workspace=1 << 30, workspace_bytes=ws, stream=0, check=False)
    # a NULL input
    assert m2.mamba2_step(d, 3, None, *p[1:], **ok) == 1
    # negative session count
    assert m2.mamba2_step(d, -1, *p, **ok) == 1
    # misaligned pointer
    assert m2.mamba2_step(d, 3, p[0] + 2, *p[1:], **ok) == 3
    # workspace too small
    assert m2.mamba2_step(d, 3, *p, workspace=1 << 30, workspace_bytes=ws - 1, stream=0, check=False) == 6
    # unsupported dims: K != 4, N = 24, P = 20, H not a multiple of G
    for bad in (m2.dims(0, 0, 4, 16, 16, 1, 3, "f32"), m2.dims(0, 0, 4, 16, 24, 1, 4, "f32"),
                m2.dims(0, 0, 4, 20, 16, 1, 4, "f32"), m2.dims(0, 0, 6, 16, 16, 4, 4, "f32")):
        assert m2.mamba2_step(bad, 3, *p, **ok) == 2
    # zero heads is an invalid argument
    assert m2.mamba2_step(m2.dims(0, 0, 0, 16, 16, 1, 4, "f32"), 3, *p, **ok) == 1


def test_scan_validation_without_gpu(m2):
    d = m2.dims(1, 64, 4, 16, 16, 1, 4, "f32")
    p = _fake_ptrs(9)
    outs = _fake_ptrs(3, base=1 << 24)
    ok = dict(workspace=1 << 30, workspace_bytes=1 << 40, stream=0, check=False)
    args = lambda chunk=16, ptrs=p: (d, *ptrs, chunk, None, None, *outs)  # noqa: E731
    assert m2.mamba2_conv_scan(*args(0), **ok) == 1          # chunk < 1
    assert m2.mamba2_conv_scan(*args(129), **ok) == 1        # chunk > 128
    assert m2.mamba2_conv_scan(*args(16, [None] + p[1:]), **ok) == 1
    assert m2.mamba2_conv_scan(*args(16, [p[0] + 8] + p[1:]), **ok) == 3
    bad = m2.dims(1, 64, 4, 16, 16, 1, 5, "f32")
    assert m2.mamba2_conv_scan(bad, *p, 16, None, None, *outs, **ok) == 2
    neg = m2.dims(1, -1, 4, 16, 16, 1, 4, "f32")
    assert m2.mamba2_conv_scan(neg, *p, 16, None, None, *outs, **ok) == 1


def test_varlen_scan_validation_without_gpu(m2):
    d = m2.dims(2, 64, 4, 16, 16, 1, 4, "f32")
    p = _fake_ptrs(9)
    outs = _fake_ptrs(3, base=1 << 24)
    ok = dict(workspace=1 << 30, workspace_bytes=1 << 40, stream=0, check=False)
    lens = 1 << 28
    assert m2.mamba2_conv_scan_varlen(d, None, *p, 16, None, None, *outs, **ok) == 1      # no lengths
    assert m2.mamba2_conv_scan_varlen(d, lens + 2, *p, 16, None, None, *outs, **ok) == 3  # misaligned
    assert m2.mamba2_conv_scan_varlen(d, lens, *p, 0, None, None, *outs, **ok) == 1       # chunk < 1
    bad = m2.dims(2, 64, 4, 16, 16, 1, 5, "f32")
    assert m2.mamba2_conv_scan_varlen(bad, lens, *p, 16, None, None, *outs, **ok) == 2


def test_workspace_queries(m2):
    d = m2.dims(4, 4096, 128, 80, 128, 8, 4, "bf16")
    assert m2.mamba2_step_workspace_bytes(d, 64) >= 64 * (12288 + 128) * 4
    assert m2.mamba2_step_workspace_bytes(d, -1) == 0
    assert m2.mamba2_scan_workspace_bytes(d, 0) == 0
    assert m2.mamba2_scan_workspace_bytes(m2.dims(1, 8, 4, 16, 16, 1, 3, "f32"), 8) == 0


def test_gated_norm_validation_without_gpu(m2):
    d = m2.dims(0, 0, 4, 16, 16, 2, 4, "bf16")
    p = _fake_ptrs(4)
    assert m2.mamba2_gated_norm(d, 3, None, p[1], p[2], 1e-5, p[3], stream=0, check=False) == 1  # NULL y
    assert m2.mamba2_gated_norm(d, -1, *p[:3], 1e-5, p[3], stream=0, check=False) == 1       # rows < 0
    assert m2.mamba2_gated_norm(d, 3, *p[:3], -1.0, p[3], stream=0, check=False) == 1        # eps < 0
    assert m2.mamba2_gated_norm(d, 3, *p[:3], float("inf"), p[3], stream=0, check=False) == 1
    assert m2.mamba2_gated_norm(d, 3, p[0] + 4, *p[1:3], 1e-5, p[3], stream=0, check=False) == 3  # misaligned
    bad = m2.dims(0, 0, 6, 16, 16, 4, 4, "bf16")  # H not a multiple of G
    assert m2.mamba2_gated_norm(bad, 3, *p[:3], 1e-5, p[3], stream=0, check=False) == 2
    wide = m2.dims(0, 0, 512, 80, 16, 1, 4, "bf16")  # a 40960-channel group
    assert m2.mamba2_gated_norm(wide, 3, *p[:3], 1e-5, p[3], stream=0, check=False) == 4


def test_qlinear_validation_without_gpu(m2):
    p = _fake_ptrs(5)
    q = lambda rows, i, o, *ptrs, g=64, b=4: m2.mamba2_qlinear(rows, i, o, *ptrs, group_size=g, bits=b,  # noqa: E731
                                                              stream=0, check=False)
    assert q(2, 128, 8, None, *p[1:5]) == 1            # NULL x
    assert q(2, 128, 8, *p[:4], None) == 1             # NULL y
    assert q(-1, 128, 8, *p) == 1                      # rows < 0
    assert q(2, 0, 8, *p) == 1 and q(2, 128, 0, *p) == 1
    assert q(2, 128, 8, *p, g=32) == 4                 # only group 64 ...
    assert q(2, 128, 8, *p, b=8) == 4                  # ... and 4 bits are built
    assert q(2, 96, 8, *p) == 2                        # in not a multiple of 64
    assert q(2, 16384 + 64, 8, *p) == 2                # in above 16384
    assert q(2, 128, 8, p[0] + 8, *p[1:]) == 3         # x not 16-byte aligned
    assert q(2, 128, 8, p[0], p[1] + 4, *p[2:]) == 3   # wq not 16-byte aligned
    assert q(2, 128, 8, *p[:2], p[2] + 1, *p[3:]) == 3  # scales odd


def test_attn_decode_validation_without_gpu(m2):
    """Every host-side check of mamba2_attn_decode, before any device call."""
    p = _fake_ptrs(8)
    lens, q, kn, vn, kc, vc, out, ws = p
    big = 1 << 30

    def call(S=2, Hq=40, Hkv=8, D=128, T=100, act="bf16", scale=0.088, ptrs=None, wsb=big):
        pt = ptrs or [lens, q, kn, vn, kc, vc]
        return m2.mamba2_attn_decode(S, Hq, Hkv, D, T, act, *pt, scale, out, ws, workspace_bytes=wsb,
                                     stream=0, check=False)

    assert call(S=-1) == 1 and call(Hq=0) == 1 and call(Hkv=0) == 1 and call(T=0) == 1
    assert call(D=64) == 2                      # head_dim 128 only
    assert call(Hq=40, Hkv=6) == 2              # heads not a multiple of kv heads
    assert call(Hq=72, Hkv=8) == 2              # more than 8 query heads per kv head
    assert call(S=65536) == 2                   # grid limit
    assert call(scale=float("inf")) == 1 and call(scale=float("nan")) == 1
    assert call(ptrs=[None, q, kn, vn, kc, vc]) == 1
    assert call(ptrs=[lens, q, kn, vn, None, vc]) == 1
    assert call(ptrs=[lens + 2, q, kn, vn, kc, vc]) == 3    # lengths not 4-byte aligned
    assert call(ptrs=[lens, q + 8, kn, vn, kc, vc]) == 3    # q not 16-byte aligned
    # bf16: none; the walkers of a (session, kv head) merge in shared memory
    assert m2.mamba2_attn_decode_workspace_bytes(2, 40, 8, 128, 100) == 0
    assert m2.mamba2_attn_decode_workspace_bytes(64, 40, 8, 128, 750) == 0
    assert m2.mamba2_attn_decode_workspace_bytes(1, 40, 8, 128, 7501) == 0
    # fp32: one partial result per chunk; chunks shrink to 32 positions (4 a
    # pair) so that the grid is not smaller than it must be
    need = m2.mamba2_attn_decode_workspace_bytes(2, 40, 8, 128, 100, "f32")
    assert need == 2 * 8 * 4 * 5 * 130 * 4
    # 64 sessions over 750 positions: 64-position chunks fill the GPU
    assert m2.mamba2_attn_decode_workspace_bytes(64, 40, 8, 128, 750, "f32") == 64 * 8 * 12 * 5 * 130 * 4
    assert call(wsb=need - 1, act="f32") == 6
    # bf16 takes no workspace at all: past the host checks (the device check
    # is what stops it here, with no GPU)
    assert m2.mamba2_attn_decode(2, 40, 8, 128, 100, "bf16", lens, q, kn, vn, kc, vc, 0.088, out, None,
                                 workspace_bytes=0, stream=0, check=False) not in (1, 2, 3, 6)
    assert m2.mamba2_attn_decode_workspace_bytes(2, 40, 8, 64, 100) == 0


def test_noalloc_step_validation_without_gpu(m2):
    """mamba2_step_noalloc checks its arguments as mamba2_step does, before the
    size of its scratch and before any device set-up: a NULL pointer is
    M2_EINVAL and a misaligned one M2_EALIGN even with no GPU, and a request
    beyond the scratch is M2_EWORKSPACE."""
    d = m2.dims(0, 0, 128, 80, 128, 8, 4, "bf16")
    p = _fake_ptrs(12)
    assert m2.mamba2_step_noalloc(d, 2, None, *p[1:], stream=0, check=False) == 1
    assert m2.mamba2_step_noalloc(d, -1, *p, stream=0, check=False) == 1
    assert m2.mamba2_step_noalloc(d, 2, p[0] + 8, *p[1:], stream=0, check=False) == 3
    assert m2.mamba2_step_noalloc(m2.dims(0, 0, 4, 16, 24, 1, 4, "f32"), 2, *p, stream=0, check=False) == 2
    assert m2.mamba2_step_noalloc(d, 22, *p, stream=0, check=False) == 6
