"""fp64 CPU oracle of the Mamba2 mixer core (conv + SiLU, softplus dt,
selective-SSM recurrence; sequential, chunked and one-step forms).

TEST INFRASTRUCTURE. Only tests/, the smoke check in __graft_entry__.py and
the cpu_baseline / reference leg of bench.py may import this package. The
CUDA library (full_duplex_speech_gb300) never imports it, and it never
imports the CUDA library: the two share no code. Inputs reach both from the
seeded_inputs module, which holds none of the mixer's arithmetic.

The arithmetic lives in mamba2_oracle.c (plain C, fp64, optional OpenMP over
(batch, head) units). This module compiles it with gcc, loads it with
ctypes, and converts numpy arrays to fp64 on the way in.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from seeded_inputs import Dims, as_f64

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mamba2_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libm2oracle.so")
_lock = threading.Lock()
_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("batch", "T", "H", "P", "N", "G", "K")]


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/libm2oracle.so (gcc, -O2, no
    fast-math: IEEE fp64 semantics are kept)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.c_int
            lib.m2o_softplus.restype = ctypes.c_double
            lib.m2o_softplus.argtypes = [ctypes.c_double]
            lib.m2o_silu.restype = ctypes.c_double
            lib.m2o_silu.argtypes = [ctypes.c_double]
            lib.m2o_max_threads.restype = ip
            lib.m2o_ssm.argtypes = [ctypes.POINTER(_Dims)] + [dp] * 8 + [ip] * 4
            lib.m2o_conv_silu.argtypes = [ctypes.POINTER(_Dims)] + [dp] * 7 + [ip]
            lib.m2o_conv_tail.argtypes = [ctypes.POINTER(_Dims)] + [dp] * 5
            lib.m2o_mixer_scan.argtypes = [ctypes.POINTER(_Dims)] + [dp] * 14 + [ip] * 4
            lib.m2o_mixer_step.argtypes = [ctypes.POINTER(_Dims), ip] + [dp] * 12 + [ip]
            lib.m2o_gated_norm.argtypes = [ip, ip, ip, dp, dp, dp, ctypes.c_double, dp]
            lib.m2o_rmsnorm.argtypes = [ip, ip, dp, dp, ctypes.c_double, dp]
            lib.m2o_qlinear.argtypes = [ip, ip, ip, ip, ctypes.POINTER(ctypes.c_uint32), dp, dp, dp, dp]
            lib.m2o_attn_decode.argtypes = [ip] * 5 + [ctypes.POINTER(ctypes.c_int)] + [dp] * 5 + \
                [ctypes.c_double, dp]
            for f in ("m2o_ssm", "m2o_conv_silu", "m2o_conv_tail", "m2o_mixer_scan", "m2o_mixer_step",
                      "m2o_gated_norm", "m2o_qlinear", "m2o_attn_decode"):
                getattr(lib, f).restype = ip
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(d: Dims, batch: int, T: int) -> _Dims:
    return _Dims(batch, T, d.H, d.P, d.N, d.G, d.K)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with status {rc}")


def max_threads() -> int:
    return int(_load().m2o_max_threads())


def softplus(z: float) -> float:
    return float(_load().m2o_softplus(float(z)))


def silu(u: float) -> float:
    return float(_load().m2o_silu(float(u)))


def conv_silu(d: Dims, x, B, C, conv_w, conv_b, init_conv=None, nthreads: int = 0) -> np.ndarray:
    """Post-conv, post-SiLU activations [b,T,CH] from fp64 pre-conv inputs."""
    x, B, C = _f64(x), _f64(B), _f64(C)
    b, T = x.shape[0], x.shape[1]
    out = np.empty((b, T, d.CH), dtype=np.float64)
    ic = None if init_conv is None else _f64(init_conv)
    rc = _load().m2o_conv_silu(ctypes.byref(_dims(d, b, T)), _ptr(x), _ptr(B), _ptr(C),
                               _ptr(_f64(conv_w)), _ptr(_f64(conv_b)), _ptr(ic), _ptr(out), nthreads)
    _check(rc, "conv_silu")
    return out


def conv_tail(d: Dims, x, B, C, init_conv=None) -> np.ndarray:
    """The last K-1 pre-conv frames [b,K-1,CH] (oldest first)."""
    x, B, C = _f64(x), _f64(B), _f64(C)
    b, T = x.shape[0], x.shape[1]
    out = np.empty((b, d.K - 1, d.CH), dtype=np.float64)
    ic = None if init_conv is None else _f64(init_conv)
    rc = _load().m2o_conv_tail(ctypes.byref(_dims(d, b, T)), _ptr(x), _ptr(B), _ptr(C), _ptr(ic), _ptr(out))
    _check(rc, "conv_tail")
    return out


def ssm(d: Dims, xt, Bt, Ct, dt, A, D, h0=None, chunk: int = 0, heads=None, nthreads: int = 0):
    """SSM core on post-conv inputs. xt [b,T,H,P], Bt/Ct [b,T,G,N], dt [b,T,H]
    (after softplus), A, D [H]. chunk <= 0: sequential; else chunked with
    that chunk length. Returns (y [b,T,H,P], h [b,H,P,N])."""
    xt, Bt, Ct, dt = _f64(xt), _f64(Bt), _f64(Ct), _f64(dt)
    b, T = xt.shape[0], xt.shape[1]
    lo, hi = (0, d.H) if heads is None else heads
    h = np.zeros((b, d.H, d.P, d.N)) if h0 is None else _f64(h0).copy()
    y = np.zeros((b, T, d.H, d.P))
    rc = _load().m2o_ssm(ctypes.byref(_dims(d, b, T)), _ptr(xt), _ptr(Bt), _ptr(Ct), _ptr(dt),
                         _ptr(_f64(A)), _ptr(_f64(D)), _ptr(h), _ptr(y), lo, hi, chunk, nthreads)
    _check(rc, "ssm")
    return y, h


def mixer_scan(d: Dims, inp: dict, init_ssm=None, init_conv=None, chunk: int = 0, heads=None,
               nthreads: int = 0):
    """Whole mixer core over a sequence from seeded_inputs-style arrays
    (bf16 bits or fp32 activations, fp32 parameters).

    Returns dict(y [b,T,H,P] fp64, final_ssm [b,H,P,N] fp64,
    final_conv [b,K-1,CH] fp64). With heads=(lo, hi) only those heads of y
    and final_ssm are computed (the rest stay zero)."""
    act = inp["act"]
    x, B, C, dtr = (as_f64(inp[k], act) for k in ("x", "B", "C", "dt_raw"))
    b, T = x.shape[0], x.shape[1]
    lo, hi = (0, d.H) if heads is None else heads
    ic = None if init_conv is None else as_f64(init_conv, act)
    iss = None if init_ssm is None else _f64(init_ssm)
    y = np.zeros((b, T, d.H, d.P))
    fs = np.zeros((b, d.H, d.P, d.N))
    fc = np.zeros((b, d.K - 1, d.CH))
    rc = _load().m2o_mixer_scan(
        ctypes.byref(_dims(d, b, T)), _ptr(x), _ptr(B), _ptr(C), _ptr(dtr),
        _ptr(_f64(inp["A_log"])), _ptr(_f64(inp["D"])), _ptr(_f64(inp["dt_bias"])),
        _ptr(_f64(inp["conv_w"])), _ptr(_f64(inp["conv_b"])), _ptr(iss), _ptr(ic),
        _ptr(y), _ptr(fs), _ptr(fc), lo, hi, chunk, nthreads)
    _check(rc, "mixer_scan")
    return dict(y=y, final_ssm=fs, final_conv=fc)


def mixer_scan_magnitude(d: Dims, inp: dict, init_ssm=None, init_conv=None, heads=None, nthreads: int = 0):
    """Magnitude of each y element's state-space terms: the recurrence run on
    the absolute values of the post-conv x~, B~, C~ and of the initial state,
    with D = 0:
        hbar_t = exp(dt A) hbar_{t-1} + dt |x~_t| (outer) |B~_t|,   ybar_t = |C~_t| . hbar_t
    so ybar_t = sum over every term of y_t's state-space part of its absolute
    value. A contraction whose operands are each rounded with relative error
    at most u (bf16: u = 2^-8) is off from the exact value by at most about
    (number of roundings per term) * u * ybar_t: the elementwise forward error
    bound of the bf16-operand chunked scan. Composed of this module's own conv,
    softplus and recurrence. Returns ybar [b,T,H,P] (heads outside `heads`
    stay zero)."""
    act = inp["act"]
    x, B, C, dtr = (as_f64(inp[k], act) for k in ("x", "B", "C", "dt_raw"))
    b, T = x.shape[0], x.shape[1]
    ic = None if init_conv is None else as_f64(init_conv, act)
    u = conv_silu(d, x, B, C, inp["conv_w"], inp["conv_b"], init_conv=ic, nthreads=nthreads)
    HP, GN = d.H * d.P, d.G * d.N
    xt = np.abs(u[:, :, :HP]).reshape(b, T, d.H, d.P)
    Bt = np.abs(u[:, :, HP:HP + GN]).reshape(b, T, d.G, d.N)
    Ct = np.abs(u[:, :, HP + GN:]).reshape(b, T, d.G, d.N)
    sp = np.vectorize(softplus, otypes=[np.float64])
    dt = sp(dtr + _f64(inp["dt_bias"])[None, None, :]) if dtr.size else np.zeros_like(dtr)
    A = -np.exp(_f64(inp["A_log"]))
    h0 = None if init_ssm is None else np.abs(_f64(init_ssm))
    ybar, _ = ssm(d, xt, Bt, Ct, dt, A, np.zeros(d.H), h0=h0, heads=heads, nthreads=nthreads)
    return ybar


def mixer_step(d: Dims, frame: dict, params: dict, ssm_state, conv_state, nthreads: int = 0):
    """One cached frame for S sessions. frame holds x [S,H,P], B/C [S,G,N],
    dt_raw [S,H] (bf16 bits or fp32, with 'act'); ssm_state [S,H,P,N] and
    conv_state [S,K-1,CH] are fp64 arrays updated in place. Returns y [S,H,P]."""
    act = frame["act"]
    x, B, C, dtr = (as_f64(frame[k], act) for k in ("x", "B", "C", "dt_raw"))
    S = x.shape[0]
    assert ssm_state.dtype == np.float64 and ssm_state.flags.c_contiguous
    assert conv_state.dtype == np.float64 and conv_state.flags.c_contiguous
    y = np.zeros((S, d.H, d.P))
    rc = _load().m2o_mixer_step(
        ctypes.byref(_dims(d, 1, 1)), S, _ptr(x), _ptr(B), _ptr(C), _ptr(dtr),
        _ptr(_f64(params["A_log"])), _ptr(_f64(params["D"])), _ptr(_f64(params["dt_bias"])),
        _ptr(_f64(params["conv_w"])), _ptr(_f64(params["conv_b"])), _ptr(ssm_state),
        _ptr(conv_state), _ptr(y), nthreads)
    _check(rc, "mixer_step")
    return y


def gated_norm(y, z, weight, groups: int, eps: float = 1e-5) -> np.ndarray:
    """Gated RMSNorm: y, z [..., width] (fp64 values), weight [width]; the
    last axis is split into `groups` contiguous blocks. Returns fp64."""
    y, z = _f64(y), _f64(z)
    width = y.shape[-1]
    rows = int(np.prod(y.shape[:-1])) if y.ndim > 1 else 1
    out = np.empty_like(y)
    rc = _load().m2o_gated_norm(rows, width, int(groups), _ptr(y), _ptr(z), _ptr(_f64(weight)), float(eps),
                                _ptr(out))
    _check(rc, "gated_norm")
    return out


def qlinear(x, wq, scales, biases, group: int = 64) -> np.ndarray:
    """Affine group-quantized linear layer. x [..., in] (values as fp64);
    wq [out, in/8] uint32 (eight 4-bit fields per word, the first input in
    the lowest bits); scales, biases [out, in/group]. Returns y [..., out]
    in fp64 (W[o][i] = scale * q + bias per group of `group` inputs)."""
    x = _f64(x)
    wq = np.ascontiguousarray(wq, dtype=np.uint32)
    n_out, in_features = wq.shape[0], wq.shape[1] * 8
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    y = np.empty(x.shape[:-1] + (n_out,), dtype=np.float64)
    rc = _load().m2o_qlinear(rows, in_features, n_out, int(group),
                             wq.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)), _ptr(_f64(scales)),
                             _ptr(_f64(biases)), _ptr(x), _ptr(y))
    _check(rc, "qlinear")
    return y


def attn_decode(q, k_new, v_new, k_cache, v_cache, lengths, scale: float) -> np.ndarray:
    """One cached decode position of grouped-query attention. q [S,Hq,D];
    k_new, v_new [S,Hkv,D]; k_cache, v_cache [S,Hkv,Tmax,D] fp64 arrays,
    UPDATED IN PLACE (the new key and value land at position lengths[s]);
    lengths [S] ints (positions already cached). Query head h reads kv head
    h // (Hq // Hkv) over positions 0..lengths[s]. Returns out [S,Hq,D] fp64."""
    q = _f64(q)
    k_new, v_new = _f64(k_new), _f64(v_new)
    for c in (k_cache, v_cache):
        if not (isinstance(c, np.ndarray) and c.dtype == np.float64 and c.flags.c_contiguous):
            raise TypeError("k_cache and v_cache must be C-contiguous float64 arrays (updated in place)")
    S, Hq, D = q.shape
    Hkv, Tmax = k_cache.shape[1], k_cache.shape[2]
    lens = np.ascontiguousarray(lengths, dtype=np.int32)
    out = np.empty((S, Hq, D), dtype=np.float64)
    rc = _load().m2o_attn_decode(S, Hq, Hkv, D, Tmax, lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                 _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                 float(scale), _ptr(out))
    _check(rc, "attn_decode")
    return out


def rmsnorm(x, weight, eps: float = 1e-5) -> np.ndarray:
    """RMSNorm over the last axis: weight * x / sqrt(mean(x^2) + eps), fp64."""
    x = _f64(x)
    width = x.shape[-1]
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    out = np.empty_like(x)
    rc = _load().m2o_rmsnorm(rows, width, _ptr(x), _ptr(_f64(weight)), float(eps), _ptr(out))
    _check(rc, "rmsnorm")
    return out


def linear(x, w) -> np.ndarray:
    """Dense linear layer without bias, y = x W^T (W [out, in]), fp64: a
    library matrix product on the exact values."""
    return _f64(x) @ _f64(w).T
