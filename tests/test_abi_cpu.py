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


def test_binding_has_every_declared_function(m2):
    """The Python binding carries the header's names one for one."""
    missing = [n for n in _declared_functions() if not callable(getattr(m2, n, None))]
    assert not missing, missing
    assert all(n in m2.__all__ for n in _declared_functions())


def test_status_strings(m2):
    for s in range(7):
        assert m2.mamba2_status_string(s)
    assert m2.mamba2_status_string(99) == "unknown status"


def _fake_ptrs(n, base=1 << 20):
    return [base + 256 * i for i in range(n)]


def _gpu_present():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # noqa: BLE001
        return False


# The calls below that pass every host check use fake device addresses. With
# a GPU present such a call would launch kernels on them, so a call of
# nonzero size is made only on a host without one (where the device check
# stops it with M2_ECUDA); a call of zero size launches nothing anywhere.
NO_GPU = not _gpu_present()


def _past_host_checks(rc):
    # M2_OK (an sm_103 GPU, nothing to do), M2_EUNSUPPORTED (another GPU),
    # M2_ECUDA (no GPU): each only after every argument check passed
    return rc in (0, 4, 5)


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
    # bf16 takes no workspace at all: past the host checks
    for S in (0, 2) if NO_GPU else (0,):
        assert _past_host_checks(m2.mamba2_attn_decode(S, 40, 8, 128, 100, "bf16", lens, q, kn, vn, kc, vc, 0.088,
                                                       out, None, workspace_bytes=0, stream=0, check=False))
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


def test_strided_and_split_scan_validation_without_gpu(m2):
    """The strided step and scan add one check each (the row stride: positive,
    and a multiple of 16 bytes), then are mamba2_step's and mamba2_conv_scan's;
    the scan's two halves validate as the whole scan does."""
    d = m2.dims(0, 0, 128, 80, 128, 8, 4, "bf16")
    p = _fake_ptrs(12)
    ws = m2.mamba2_step_workspace_bytes(d, 2)
    ok = dict(workspace=1 << 30, workspace_bytes=ws, stream=0, check=False)
    st = lambda stride, ptrs=p: m2.mamba2_step_strided(d, 2, *ptrs[:4], stride, *ptrs[4:], **ok)  # noqa: E731
    assert st(0) == 1 and st(-22656) == 1          # stride not positive
    assert st(22657) == 3 and st(22652) == 3        # 2 * stride not a multiple of 16 bytes
    assert st(22656, [None] + p[1:]) == 1           # then mamba2_step's own checks
    assert st(22656, [p[0] + 8] + p[1:]) == 3
    assert m2.mamba2_step_strided(d, 2, *p[:4], 22656, *p[4:], workspace=1 << 30, workspace_bytes=ws - 1,
                                  stream=0, check=False) == 6
    ds = m2.dims(1, 300, 128, 80, 128, 8, 4, "bf16")
    q = _fake_ptrs(9)
    outs = _fake_ptrs(3, base=1 << 24)
    big = dict(workspace=1 << 30, workspace_bytes=1 << 40, stream=0, check=False)
    sc = lambda stride, chunk=128, ptrs=q: m2.mamba2_conv_scan_strided(  # noqa: E731
        ds, *ptrs[:4], stride, *ptrs[4:], chunk, None, None, *outs, **big)
    assert sc(0) == 1 and sc(22657) == 3
    assert sc(22656, chunk=0) == 1 and sc(22656, chunk=129) == 1
    assert sc(22656, ptrs=[q[0]] + [None] + q[2:]) == 1
    assert m2.mamba2_conv_scan_strided(ds, *q[:4], 22656, *q[4:], 128, None, None, *outs, workspace=1 << 30,
                                       workspace_bytes=1, stream=0, check=False) == 6
    for half in (m2.mamba2_scan_prepare_bc, m2.mamba2_scan_chunks):
        assert half(ds, *q, 0, None, None, *outs, **big) == 1
        assert half(ds, *q, 129, None, None, *outs, **big) == 1
        assert half(ds, None, *q[1:], 128, None, None, *outs, **big) == 1
        assert half(ds, q[0] + 8, *q[1:], 128, None, None, *outs, **big) == 3
        assert half(m2.dims(1, 300, 128, 80, 128, 8, 5, "bf16"), *q, 128, None, None, *outs, **big) == 2
        need = m2.mamba2_scan_workspace_bytes(ds, 128)
        assert half(ds, *q, 128, None, None, *outs, workspace=1 << 30, workspace_bytes=need - 1,
                    stream=0, check=False) == 6


def test_fused_projection_validation_without_gpu(m2):
    """mamba2_qlinear_fused: the row stride and the fused norm are checked on
    the host, before any device call."""
    x, wq, s, b, y, w, g = _fake_ptrs(7)

    def q(rows=300, i=4480, o=22656, xs=4480, norm=None, res=None, xp=x, wqp=wq, yp=y):
        return m2.mamba2_qlinear_fused(rows, i, o, xp, xs, norm, wqp, s, b, res, yp, stream=0, check=False)

    assert q(xs=4479) == 1                          # rows overlap
    assert q(xs=4484) == 3                          # row pitch not a multiple of 16 bytes
    assert q(xp=x + 2) == 3 and q(wqp=wq + 4) == 3 and q(yp=y + 1) == 3
    assert q(res=y + 1) == 3                        # residual: bf16 alignment
    assert q(rows=-1) == 1 and q(o=0) == 1
    assert m2.mamba2_qlinear_fused(2, 4480, 8, x, 4480, None, wq, s, b, None, y, group_size=128,
                                   stream=0, check=False) == 4
    rms = lambda **k: m2.row_norm(m2.NORM_RMS, **k)  # noqa: E731
    assert q(norm=rms(weight=None)) == 1            # a norm needs its weight
    assert q(norm=rms(weight=w, eps=-1.0)) == 1
    assert q(norm=rms(weight=w, eps=float("nan"))) == 1
    assert q(norm=rms(weight=w + 4)) == 3
    bad_kind = m2.row_norm(7, weight=w)
    assert q(norm=bad_kind) == 1
    gated = lambda **k: m2.row_norm(m2.NORM_GATED, weight=w, **k)  # noqa: E731
    # the gated output norm before out_proj: 10240 inputs in 8 groups of 1280
    oq = lambda norm: q(rows=300, i=10240, o=4480, xs=10240, norm=norm)  # noqa: E731
    assert oq(gated(groups=8, gate=None, gate_stride=22656)) == 1       # no gate
    assert oq(gated(groups=0, gate=g, gate_stride=22656)) == 1          # no groups
    assert oq(gated(groups=8, gate=g, gate_stride=10239)) == 1          # gate rows overlap
    assert oq(gated(groups=3, gate=g, gate_stride=22656)) == 2          # groups do not divide the row
    assert oq(gated(groups=65, gate=g, gate_stride=22656)) == 2         # more groups than the kernel takes
    assert oq(gated(groups=8, gate=g + 2, gate_stride=22656)) == 3      # gate not 16-byte aligned
    assert oq(gated(groups=8, gate=g, gate_stride=22657)) == 3          # gate pitch not 16 bytes
    # with valid arguments the host checks pass
    for rows in (0, 300) if NO_GPU else (0,):
        assert _past_host_checks(m2.mamba2_qlinear_fused(rows, 10240, 4480, x, 10240,
                                                         gated(groups=8, gate=g, gate_stride=22656), wq, s, b, y,
                                                         y, stream=0, check=False))
        assert _past_host_checks(q(rows=rows, norm=rms(weight=w)))


def test_linear_bf16_validation_without_gpu(m2):
    """mamba2_linear_bf16 (the attention blocks' projections): sizes, strides and
    alignment are checked on the host."""
    x, w, y, r = _fake_ptrs(4)

    def lin(rows=1, i=4480, o=7168, xs=4480, ys=7168, xp=x, wp=w, yp=y, res=None, norm=None):
        return m2.mamba2_linear_bf16(rows, i, o, xp, xs, norm, wp, res, yp, ys, stream=0, check=False)

    assert lin(rows=-1) == 1 and lin(i=0) == 1 and lin(o=0) == 1
    assert lin(i=4464 + 8, xs=4472) == 2            # in_features not a multiple of 32
    assert lin(i=16384 + 32, xs=16416) == 2         # above 16384
    assert lin(xs=4479) == 1 and lin(ys=7167) == 1  # rows overlap
    assert lin(xs=4484) == 3                        # x pitch not a multiple of 16 bytes
    assert lin(xp=x + 8) == 3 and lin(wp=w + 8) == 3 and lin(yp=y + 1) == 3 and lin(res=r + 1) == 3
    assert lin(xp=None) == 1 and lin(wp=None) == 1 and lin(yp=None) == 1
    for rows in (0, 1) if NO_GPU else (0,):
        assert _past_host_checks(lin(rows=rows, res=r, ys=7168 + 5))  # an odd y pitch is fine (bf16 stores)


def _lm_layers(m2, kinds, base=1 << 20):
    """Distinct, 16-byte aligned fake device addresses for every field of every block."""
    from full_duplex_speech_gb300._binding import _LM_LAYER_FIELDS
    layers, a = [], base
    for _ in kinds:
        L = {}
        for n in _LM_LAYER_FIELDS:
            L[n] = a
            a += 1 << 12
        layers.append(L)
    return layers


def test_lm_validation_without_gpu(m2):
    """mamba2_lm_step / mamba2_lm_prefill check the model description, every
    block's pointers, the residual stream, the lengths and the workspace
    before anything is launched."""
    mixer = m2.dims(0, 0, 128, 80, 128, 8, 4, "bf16")
    kinds = "MM*M"
    hidden, lens, ws = _fake_ptrs(3, base=1 << 30)

    def model(kinds=kinds, layers=None, hid=4480, mix=mixer, **kw):
        args = dict(n_heads=40, n_kv_heads=8, head_dim=128, max_len=1000)
        args.update(kw)
        return m2.lm_model(kinds, layers if layers is not None else _lm_layers(m2, kinds), hid, mix, **args)

    m = model()
    need = m2.mamba2_lm_workspace_bytes(m, 2, 1)
    assert need > 0
    step = lambda mm, S=2, h=hidden, ln=lens, wsb=need: m2.mamba2_lm_step(  # noqa: E731
        mm, S, h, ln, ws, workspace_bytes=wsb, stream=0, check=False)
    assert step(m, S=-1) == 1
    assert step(m, h=None) == 1 and step(m, h=hidden + 8) == 3
    assert step(m, ln=None) == 1 and step(m, ln=lens + 2) == 3     # attention blocks need the lengths
    assert step(model(kinds="MMXM")) == 1                            # unknown block kind
    assert step(model(mix=m2.dims(0, 0, 128, 80, 128, 8, 4, "f32"))) == 4
    assert step(model(hid=4480 + 32)) == 2                           # hidden not a multiple of 64
    assert step(model(head_dim=64)) == 2
    assert step(model(n_heads=40, n_kv_heads=6)) == 2
    assert step(model(norm_eps=-1.0)) == 1
    for field, code in (("in_wq", 1), ("ssm_state", 1), ("wqkv", 1), ("norm_w", 1)):
        layers = _lm_layers(m2, kinds)
        layers[2 if field == "wqkv" else 0][field] = None
        assert step(model(layers=layers)) == code, field
    for field in ("in_wq", "conv_state", "k_cache"):
        layers = _lm_layers(m2, kinds)
        layers[2 if field == "k_cache" else 1][field] += 8
        assert step(model(layers=layers)) == 3, field
    # (for T = 1 the query covers both a step and a one-position prefill, so
    # it may be above what the step itself checks for)
    assert step(m, wsb=1) == 6 and m2.mamba2_lm_step(m, 2, hidden, lens, None, workspace_bytes=0, stream=0,
                                                     check=False) == 6
    sizes = (0, 2) if NO_GPU else (0,)
    for S in sizes:
        assert _past_host_checks(step(m, S=S, wsb=m2.mamba2_lm_workspace_bytes(m, S, 1)))
    # a model without attention blocks needs no lengths
    mm = model(kinds="MMM")
    for S in sizes:
        assert _past_host_checks(m2.mamba2_lm_step(mm, S, hidden, None, ws,
                                                   workspace_bytes=m2.mamba2_lm_workspace_bytes(mm, S, 1),
                                                   stream=0, check=False))
    pre = lambda chunk, S=1, T=300: m2.mamba2_lm_prefill(  # noqa: E731
        m, S, T, hidden, lens, chunk, ws, workspace_bytes=m2.mamba2_lm_workspace_bytes(m, S, T, 128),
        stream=0, check=False)
    assert pre(0) == 1 and pre(129) == 1
    for S in sizes:
        assert _past_host_checks(pre(128, S=S))
    assert m2.mamba2_lm_prefill(m, 1, 300, hidden, lens, 128, ws, workspace_bytes=m2.mamba2_lm_workspace_bytes(
        m, 1, 300, 128) - 1, stream=0, check=False) == 6


def test_lm_workspace_plan(m2):
    """The scratch of a position or a prefill covers the in_proj rows, the
    mixer output, the mixer core's own workspace and, for a prefill of 40 rows
    or more, the normalised input rows that let the projections run as GEMMs."""
    mixer = m2.dims(0, 0, 128, 80, 128, 8, 4, "bf16")
    H, P, N, G, hid = 128, 80, 128, 8, 4480
    HP, GN = H * P, G * N
    W = 2 * HP + 2 * GN + H
    assert W == 22656
    m = m2.lm_model("MMM", _lm_layers(m2, "MMM"), hid, mixer)
    # invalid descriptions ask for nothing
    assert m2.mamba2_lm_workspace_bytes(m, -1, 1) == 0
    assert m2.mamba2_lm_workspace_bytes(m2.lm_model("MQM", _lm_layers(m2, "MQM"), hid, mixer), 1, 1) == 0
    assert m2.mamba2_lm_workspace_bytes(m2.lm_model("M", _lm_layers(m2, "M"), hid + 16, mixer), 1, 1) == 0
    # one cached position of S sessions
    for S in (1, 64):
        step_ws = m2.mamba2_step_workspace_bytes(m2.dims(S, 1, H, P, N, G, 4, "bf16"), S)
        assert m2.mamba2_lm_workspace_bytes(m, S, 1) >= S * W * 2 + S * HP * 2 + step_ws
    # a prefill of T positions
    for T in (39, 40, 300):
        scan_ws = m2.mamba2_scan_workspace_bytes(m2.dims(1, T, H, P, N, G, 4, "bf16"), 128)
        floor = T * W * 2 + T * HP * 2 + scan_ws + (T * max(hid, HP) * 2 if T >= 40 else 0)
        got = m2.mamba2_lm_workspace_bytes(m, 1, T, 128)
        assert floor <= got <= floor + 16 * 256, (T, got, floor)
    # from 40 rows the normalised rows are part of it
    assert m2.mamba2_lm_workspace_bytes(m, 1, 40, 128) - m2.mamba2_lm_workspace_bytes(m, 1, 39, 128) >= 40 * HP * 2


@pytest.mark.skipif(not NO_GPU, reason="host tensors would reach a launch where a GPU is present")
def test_readme_example_passes_the_host_checks(m2):
    """The README's Python example, run on host tensors: every call gets past
    all of its argument checks and stops only at the device check."""
    src = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```python\n(.*?)```", src, re.S).group(1)
    code = code.replace('dev, bf = "cuda", torch.bfloat16', 'dev, bf = "cpu", torch.bfloat16')
    code = code.split("torch.cuda.synchronize()")[0]
    code = re.sub(r"^(m2\.mamba2_\w+\()", r"_rc.append(\1", code, flags=re.M)
    code = re.sub(r"(ws|wss)\)\n", r"\1, stream=0, check=False))\n", code)
    rcs = []
    exec(compile(code, "README.md", "exec"), {"_rc": rcs})
    assert len(rcs) == 2 and all(rc == 5 for rc in rcs), rcs   # M2_ECUDA: no device here
