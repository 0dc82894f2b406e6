"""ctypes binding of libmamba2.so: the same names as the C ABI, argument
marshalling only. Tensor arguments may be torch tensors (their data_ptr()
is passed), plain ints (device addresses) or None (NULL)."""
from __future__ import annotations

__all__ = ["M2Error", "M2Dims", "M2RowNorm", "M2Lm", "M2LmLayer", "BF16", "F32", "NORM_NONE", "NORM_RMS",
           "NORM_GATED", "library_path", "load", "dims", "row_norm", "lm_model"]

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libmamba2.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
F32 = 1

STATUS = {0: "M2_OK", 1: "M2_EINVAL", 2: "M2_ESHAPE", 3: "M2_EALIGN", 4: "M2_EUNSUPPORTED",
          5: "M2_ECUDA", 6: "M2_EWORKSPACE"}


class M2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)} ({mamba2_status_string(status)})"
        if status == 5:
            msg += f", cudaError {mamba2_last_cuda_error()}"
        super().__init__(msg)


class M2Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("T", ctypes.c_int), ("nheads", ctypes.c_int),
                ("headdim", ctypes.c_int), ("dstate", ctypes.c_int), ("ngroups", ctypes.c_int),
                ("dconv", ctypes.c_int), ("act", ctypes.c_int)]


class M2RowNorm(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("weight", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("groups", ctypes.c_int), ("gate", ctypes.c_void_p), ("gate_stride", ctypes.c_long)]


NORM_NONE, NORM_RMS, NORM_GATED = 0, 1, 2


def row_norm(kind, weight=None, eps=1e-5, groups=1, gate=None, gate_stride=0) -> M2RowNorm:
    """The m2_row_norm of the fused linear layers (kind: NORM_RMS or NORM_GATED).
    The structure holds raw device addresses; it keeps references to the
    tensors it was given so that they outlive it."""
    n = M2RowNorm(int(kind), _p(weight), float(eps), int(groups), _p(gate), int(gate_stride))
    n._keep = (weight, gate)
    return n


_LM_LAYER_FIELDS = ("norm_w", "in_wq", "in_scales", "in_biases", "A_log", "D", "dt_bias", "conv_w", "conv_b",
                    "gnorm_w", "out_wq", "out_scales", "out_biases", "ssm_state", "conv_state", "wqkv", "wo",
                    "k_cache", "v_cache")


class M2LmLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _LM_LAYER_FIELDS]


class M2Lm(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("kinds", ctypes.c_char_p), ("layers", ctypes.POINTER(M2LmLayer)),
                ("hidden", ctypes.c_int), ("mixer", M2Dims), ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("max_len", ctypes.c_int), ("norm_eps", ctypes.c_float),
                ("attn_scale", ctypes.c_float)]


def lm_model(kinds: str, layers, hidden, mixer: M2Dims, n_heads=0, n_kv_heads=0, head_dim=128, max_len=1,
             norm_eps=1e-5, attn_scale=None) -> M2Lm:
    """The m2_lm description: `layers` is a list of dicts of tensors keyed by
    the m2_lm_layer field names (absent fields are NULL). The returned
    structure keeps its arrays and the layers' tensors alive."""
    arr = (M2LmLayer * max(1, len(layers)))()
    for i, L in enumerate(layers):
        for n in _LM_LAYER_FIELDS:
            setattr(arr[i], n, _p(L.get(n)))
    kb = kinds.encode()
    m = M2Lm(len(layers), kb, arr, int(hidden), mixer, int(n_heads), int(n_kv_heads), int(head_dim), int(max_len),
             float(norm_eps), float(head_dim ** -0.5 if attn_scale is None else attn_scale))
    m._keep = (arr, kb, [dict(L) for L in layers])  # the tensors behind the raw addresses
    return m


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libmamba2.so (built by full_duplex_speech_gb300.build). Raises
    if it is missing: there is no other implementation to fall back to."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libmamba2.so not found at {_LIB_PATH}; run "
                               "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, sz, ip = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        dp = ctypes.POINTER(M2Dims)
        lib.mamba2_scan_workspace_bytes.argtypes = [dp, ip]
        lib.mamba2_scan_workspace_bytes.restype = sz
        for f in ("mamba2_conv_scan", "mamba2_scan_prepare_bc", "mamba2_scan_chunks"):
            getattr(lib, f).argtypes = [dp] + [vp] * 9 + [ip] + [vp] * 6 + [sz, vp]
            getattr(lib, f).restype = ip
        lib.mamba2_conv_scan_varlen.argtypes = [dp] + [vp] * 10 + [ip] + [vp] * 6 + [sz, vp]
        lib.mamba2_conv_scan_varlen.restype = ip
        lib.mamba2_gated_norm.argtypes = [dp, ip, vp, vp, vp, ctypes.c_float, vp, vp]
        lib.mamba2_gated_norm.restype = ip
        lib.mamba2_qlinear.argtypes = [ip] * 5 + [vp] * 6
        lib.mamba2_qlinear.restype = ip
        lib.mamba2_attn_decode.argtypes = [ip] * 6 + [vp] * 6 + [ctypes.c_float, vp, vp, sz, vp]
        lib.mamba2_attn_decode.restype = ip
        lib.mamba2_attn_decode_workspace_bytes.argtypes = [ip] * 6
        lib.mamba2_attn_decode_workspace_bytes.restype = sz
        lib.mamba2_step_workspace_bytes.argtypes = [dp, ip]
        lib.mamba2_step_workspace_bytes.restype = sz
        lib.mamba2_step.argtypes = [dp, ip] + [vp] * 13 + [sz, vp]
        lib.mamba2_step.restype = ip
        lib.mamba2_step_noalloc.argtypes = [dp, ip] + [vp] * 12 + [vp]
        lib.mamba2_step_noalloc.restype = ip
        lib.mamba2_step_noalloc_max_bytes.argtypes = []
        lib.mamba2_step_noalloc_max_bytes.restype = sz
        lp, np_ = ctypes.c_long, ctypes.POINTER(M2RowNorm)
        lib.mamba2_step_strided.argtypes = [dp, ip] + [vp] * 4 + [lp] + [vp] * 9 + [sz, vp]
        lib.mamba2_step_strided.restype = ip
        lib.mamba2_conv_scan_strided.argtypes = [dp] + [vp] * 4 + [lp] + [vp] * 5 + [ip] + [vp] * 6 + [sz, vp]
        lib.mamba2_conv_scan_strided.restype = ip
        lib.mamba2_qlinear_fused.argtypes = [ip] * 5 + [vp, lp, np_] + [vp] * 5 + [vp]
        lib.mamba2_qlinear_fused.restype = ip
        lib.mamba2_linear_bf16.argtypes = [ip] * 3 + [vp, lp, np_, vp, vp, vp, lp, vp]
        lib.mamba2_linear_bf16.restype = ip
        mp = ctypes.POINTER(M2Lm)
        lib.mamba2_lm_workspace_bytes.argtypes = [mp, ip, ip, ip]
        lib.mamba2_lm_workspace_bytes.restype = sz
        lib.mamba2_lm_step.argtypes = [mp, ip, vp, vp, vp, sz, vp]
        lib.mamba2_lm_step.restype = ip
        lib.mamba2_lm_prefill.argtypes = [mp, ip, ip, vp, vp, ip, vp, sz, vp]
        lib.mamba2_lm_prefill.restype = ip
        lib.mamba2_status_string.argtypes = [ip]
        lib.mamba2_status_string.restype = ctypes.c_char_p
        lib.mamba2_last_cuda_error.argtypes = []
        lib.mamba2_last_cuda_error.restype = ip
        lib.mamba2_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
        lib.mamba2_device_error.restype = ip
        _lib = lib
        return lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dims(batch, T, H, P, N, G, K=4, act=BF16) -> M2Dims:
    if isinstance(act, str):
        act = {"bf16": BF16, "f32": F32}[act]
    return M2Dims(batch, T, H, P, N, G, K, act)


def mamba2_status_string(status: int) -> str:
    return load().mamba2_status_string(status).decode()


def mamba2_last_cuda_error() -> int:
    return load().mamba2_last_cuda_error()


def mamba2_device_error(stream=None) -> int:
    code = ctypes.c_uint(0)
    rc = load().mamba2_device_error(_stream(stream), ctypes.byref(code))
    if rc:
        raise M2Error(rc, "mamba2_device_error")
    return code.value


def mamba2_scan_workspace_bytes(d: M2Dims, chunk: int) -> int:
    return load().mamba2_scan_workspace_bytes(ctypes.byref(d), chunk)


def mamba2_step_workspace_bytes(d: M2Dims, n_sessions: int) -> int:
    return load().mamba2_step_workspace_bytes(ctypes.byref(d), n_sessions)


def _scan_call(fname, d, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, chunk, init_ssm, init_conv,
               y, final_ssm, final_conv, workspace, workspace_bytes, stream, check):
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    rc = getattr(load(), fname)(
        ctypes.byref(d), _p(x), _p(B), _p(C), _p(dt_raw), _p(A_log), _p(D), _p(dt_bias), _p(conv_w),
        _p(conv_b), int(chunk), _p(init_ssm), _p(init_conv), _p(y), _p(final_ssm), _p(final_conv),
        _p(workspace), int(workspace_bytes), _stream(stream))
    if check and rc:
        raise M2Error(rc, fname)
    return rc


def mamba2_conv_scan(d: M2Dims, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, chunk,
                     init_ssm, init_conv, y, final_ssm, final_conv, workspace, workspace_bytes=None,
                     stream=None, check=True) -> int:
    return _scan_call("mamba2_conv_scan", d, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, chunk,
                      init_ssm, init_conv, y, final_ssm, final_conv, workspace, workspace_bytes, stream, check)


def mamba2_conv_scan_varlen(d: M2Dims, lengths, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, chunk,
                            init_ssm, init_conv, y, final_ssm, final_conv, workspace, workspace_bytes=None,
                            stream=None, check=True) -> int:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    rc = load().mamba2_conv_scan_varlen(
        ctypes.byref(d), _p(lengths), _p(x), _p(B), _p(C), _p(dt_raw), _p(A_log), _p(D), _p(dt_bias),
        _p(conv_w), _p(conv_b), int(chunk), _p(init_ssm), _p(init_conv), _p(y), _p(final_ssm), _p(final_conv),
        _p(workspace), int(workspace_bytes), _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_conv_scan_varlen")
    return rc


def mamba2_scan_prepare_bc(d: M2Dims, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, chunk,
                           init_ssm, init_conv, y, final_ssm, final_conv, workspace, workspace_bytes=None,
                           stream=None, check=True) -> int:
    return _scan_call("mamba2_scan_prepare_bc", d, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b,
                      chunk, init_ssm, init_conv, y, final_ssm, final_conv, workspace, workspace_bytes, stream,
                      check)


def mamba2_scan_chunks(d: M2Dims, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, chunk,
                       init_ssm, init_conv, y, final_ssm, final_conv, workspace, workspace_bytes=None,
                       stream=None, check=True) -> int:
    return _scan_call("mamba2_scan_chunks", d, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, chunk,
                      init_ssm, init_conv, y, final_ssm, final_conv, workspace, workspace_bytes, stream, check)


def mamba2_gated_norm(d: M2Dims, rows, y, z, weight, eps, out, stream=None, check=True) -> int:
    rc = load().mamba2_gated_norm(ctypes.byref(d), int(rows), _p(y), _p(z), _p(weight), float(eps), _p(out),
                                  _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_gated_norm")
    return rc


def mamba2_qlinear(rows, in_features, out_features, x, wq, scales, biases, y, group_size=64, bits=4,
                   stream=None, check=True) -> int:
    rc = load().mamba2_qlinear(int(rows), int(in_features), int(out_features), int(group_size), int(bits), _p(x),
                               _p(wq), _p(scales), _p(biases), _p(y), _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_qlinear")
    return rc


def _act_code(act) -> int:
    if act in ("bf16", 0):
        return 0
    if act in ("f32", 1):
        return 1
    raise ValueError(f"act must be 'bf16' or 'f32', got {act!r}")


def mamba2_attn_decode_workspace_bytes(n_sessions, n_heads, n_kv_heads, head_dim, max_len, act="bf16") -> int:
    return load().mamba2_attn_decode_workspace_bytes(int(n_sessions), int(n_heads), int(n_kv_heads), int(head_dim),
                                                     int(max_len), _act_code(act))


def mamba2_attn_decode(n_sessions, n_heads, n_kv_heads, head_dim, max_len, act, lengths, q, k_new, v_new, k_cache,
                       v_cache, scale, out, workspace, workspace_bytes=None, stream=None, check=True) -> int:
    """One cached decode position of grouped-query attention with the KV-cache
    append (see mamba2_attn_decode in include/mamba2.h)."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    rc = load().mamba2_attn_decode(int(n_sessions), int(n_heads), int(n_kv_heads), int(head_dim), int(max_len),
                                   _act_code(act), _p(lengths), _p(q), _p(k_new), _p(v_new), _p(k_cache),
                                   _p(v_cache), float(scale), _p(out), _p(workspace), int(workspace_bytes),
                                   _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_attn_decode")
    return rc


def mamba2_step(d: M2Dims, n_sessions, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, ssm_state,
                conv_state, y, workspace, workspace_bytes=None, stream=None, check=True) -> int:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    rc = load().mamba2_step(
        ctypes.byref(d), int(n_sessions), _p(x), _p(B), _p(C), _p(dt_raw), _p(A_log), _p(D),
        _p(dt_bias), _p(conv_w), _p(conv_b), _p(ssm_state), _p(conv_state), _p(y), _p(workspace),
        int(workspace_bytes), _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_step")
    return rc


def mamba2_step_noalloc_max_bytes() -> int:
    return load().mamba2_step_noalloc_max_bytes()


def mamba2_step_noalloc(d: M2Dims, n_sessions, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, ssm_state,
                        conv_state, y, stream=None, check=True) -> int:
    """mamba2_step with the library's fixed device scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    rc = load().mamba2_step_noalloc(
        ctypes.byref(d), int(n_sessions), _p(x), _p(B), _p(C), _p(dt_raw), _p(A_log), _p(D),
        _p(dt_bias), _p(conv_w), _p(conv_b), _p(ssm_state), _p(conv_state), _p(y), _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_step_noalloc")
    return rc


def _ws_bytes(workspace, workspace_bytes):
    if workspace_bytes is not None:
        return int(workspace_bytes)
    return 0 if workspace is None or isinstance(workspace, int) else workspace.numel() * workspace.element_size()


def mamba2_step_strided(d: M2Dims, n_sessions, x, B, C, dt_raw, in_row_stride, A_log, D, dt_bias, conv_w, conv_b,
                        ssm_state, conv_state, y, workspace, workspace_bytes=None, stream=None, check=True) -> int:
    """mamba2_step on column slices of wider rows (one row per session)."""
    rc = load().mamba2_step_strided(
        ctypes.byref(d), int(n_sessions), _p(x), _p(B), _p(C), _p(dt_raw), int(in_row_stride), _p(A_log), _p(D),
        _p(dt_bias), _p(conv_w), _p(conv_b), _p(ssm_state), _p(conv_state), _p(y), _p(workspace),
        _ws_bytes(workspace, workspace_bytes), _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_step_strided")
    return rc


def mamba2_conv_scan_strided(d: M2Dims, x, B, C, dt_raw, in_row_stride, A_log, D, dt_bias, conv_w, conv_b, chunk,
                             init_ssm, init_conv, y, final_ssm, final_conv, workspace, workspace_bytes=None,
                             stream=None, check=True) -> int:
    """mamba2_conv_scan on column slices of wider rows (one row per frame)."""
    rc = load().mamba2_conv_scan_strided(
        ctypes.byref(d), _p(x), _p(B), _p(C), _p(dt_raw), int(in_row_stride), _p(A_log), _p(D), _p(dt_bias),
        _p(conv_w), _p(conv_b), int(chunk), _p(init_ssm), _p(init_conv), _p(y), _p(final_ssm), _p(final_conv),
        _p(workspace), _ws_bytes(workspace, workspace_bytes), _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_conv_scan_strided")
    return rc


def mamba2_qlinear_fused(rows, in_features, out_features, x, x_stride, norm, wq, scales, biases, residual, y,
                         group_size=64, bits=4, stream=None, check=True) -> int:
    """mamba2_qlinear with a fused row norm (M2RowNorm or None) and residual."""
    rc = load().mamba2_qlinear_fused(
        int(rows), int(in_features), int(out_features), int(group_size), int(bits), _p(x), int(x_stride),
        None if norm is None else ctypes.byref(norm), _p(wq), _p(scales), _p(biases), _p(residual), _p(y),
        _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_qlinear_fused")
    return rc


def mamba2_linear_bf16(rows, in_features, out_features, x, x_stride, norm, w, residual, y, y_stride, stream=None,
                       check=True) -> int:
    """Dense bf16 linear layer for a few rows, with a fused row norm and residual."""
    rc = load().mamba2_linear_bf16(
        int(rows), int(in_features), int(out_features), _p(x), int(x_stride),
        None if norm is None else ctypes.byref(norm), _p(w), _p(residual), _p(y), int(y_stride), _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_linear_bf16")
    return rc



def mamba2_lm_workspace_bytes(m: M2Lm, n_sessions, T, chunk=128) -> int:
    return load().mamba2_lm_workspace_bytes(ctypes.byref(m), int(n_sessions), int(T), int(chunk))


def mamba2_lm_step(m: M2Lm, n_sessions, hidden, lengths, workspace, workspace_bytes=None, stream=None,
                   check=True) -> int:
    """One cached position of the hybrid model for n_sessions sessions."""
    rc = load().mamba2_lm_step(ctypes.byref(m), int(n_sessions), _p(hidden), _p(lengths), _p(workspace),
                               _ws_bytes(workspace, workspace_bytes), _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_lm_step")
    return rc


def mamba2_lm_prefill(m: M2Lm, n_sessions, T, hidden, lengths, chunk, workspace, workspace_bytes=None, stream=None,
                      check=True) -> int:
    """T positions of the hybrid model at once (full-history recompute)."""
    rc = load().mamba2_lm_prefill(ctypes.byref(m), int(n_sessions), int(T), _p(hidden), _p(lengths), int(chunk),
                                  _p(workspace), _ws_bytes(workspace, workspace_bytes), _stream(stream))
    if check and rc:
        raise M2Error(rc, "mamba2_lm_prefill")
    return rc

__all__ += [n for n in list(globals()) if n.startswith("mamba2_")]
