"""Helpers shared by the parity tests: moving seeded inputs to the device,
reading results back, and the acceptance gates.

Gates on a bf16 result (y of the scan and the step, the gated norm, the
projections, attention), against the fp64 oracle rounded to bf16 (RNE):
  * normwise   ||y_gpu - bf16(y_ref)||_2 / ||bf16(y_ref)||_2 <= 2e-3  (the
    library's bar for bf16 results);
  * elementwise, two parts:
      - at most 0.1% of the elements lie more than one bf16 ulp from
        bf16(y_ref) (the ulp of the rounded reference value);
      - no element lies further than 4 ulp + 1e-3 * max|y_ref| from it.
    The normwise gate alone would let a handful of elements of a large
    output be wrong by their own magnitude; these two do not.
Gates on y of the chunked scan, whose intra-chunk contractions take bf16
operands (C~, B~, the masked G, x~ and the carried state h rounded to bf16,
fp32 accumulation): normwise 2e-3 as above, and elementwise the forward error
bound of that arithmetic,
      |y_gpu - bf16(y_ref)| <= ulp(bf16(y_ref)) + 4 u ybar + 1e-6 (|y_ref| + ybar)
  for every element, with u = 2^-8 the bf16 unit roundoff and ybar the
  oracle's magnitude of the element's state-space terms (the recurrence on
  absolute values): a term of Y_diag carries four roundings (C~, B~, the mask
  M, x~), a term of Y_off two (C~, h); the last part covers the fp32 math
  (exponentials, accumulation, D x~). For fp32 y the ulp term becomes 2^-126,
  the least normal fp32 number (the GPU's fp32 math flushes smaller values).
  The share of elements more than 1 ulp off is reported, not gated: bf16
  operands put several percent of the elements there even in an exact
  implementation of this arithmetic.
Gates on an fp32 result:
  * y (the tiny fp32 mixer, the fp32 norm and attention): normwise
    ||y_gpu - y_ref|| / ||y_ref|| <= 2e-3 (tighter per test where the
    arithmetic is fp32 throughout) and max-normwise max|e| / max|y_ref|
    within the test's elementwise bound;
  * SSM state: max|e| / max|ref| <= 1e-4.
Conv tail and cache slots: bitwise.

Every gate call can append its figures to a JSON-lines file named by the
environment variable M2_GATE_LOG (the measured error figures of each case).
"""
from __future__ import annotations

import json
import os

import numpy as np

from seeded_inputs import bf16_bits_to_f64, f64_to_bf16_bits

Y_TOL = 2e-3          # normwise, bf16 or fp32 y
STATE_TOL = 1e-4      # max-normwise, fp32 state
ULP_SHARE_TOL = 1e-3  # share of bf16 elements more than 1 ulp off
ULP_MAX = 4.0         # ... and no element beyond ULP_MAX ulp + ABS_FLOOR * max|ref|
ABS_FLOOR = 1e-3
F32_MAXNORM_TOL = 1e-4  # default elementwise bound of an fp32 y (max-normwise)
BF16_U = 2.0 ** -8    # bf16 unit roundoff
SCAN_ROUNDINGS = 4    # operand roundings per term of the scan's bf16 contractions
F32_SLACK = 1e-6      # fp32 math of the scan, relative to |y_ref| + ybar


def to_dev(a, act=None):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def act_empty(shape, act):
    import torch
    dt = torch.bfloat16 if act == "bf16" else torch.float32
    return torch.empty(shape, dtype=dt, device="cuda")


def from_dev_act(t, act):
    """Device activation tensor -> fp64 numpy (exact)."""
    import torch
    if act == "bf16":
        bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return bf16_bits_to_f64(bits)
    return t.detach().double().cpu().numpy()


def bits_of(t):
    """Raw bytes of a device tensor as a numpy uint8 array."""
    import torch
    return t.detach().contiguous().view(torch.uint8).cpu().numpy().reshape(-1)


def bf16_ulp(v):
    """Spacing of bf16 numbers at each (bf16-representable) value of v: for
    |v| in [2^e, 2^(e+1)) it is 2^(e-7); at and below the smallest normal,
    the subnormal spacing 2^-133."""
    a = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(np.maximum(a, 2.0 ** -126))  # a = m * 2^e, m in [0.5, 1)
    return np.ldexp(1.0, e - 1 - 7)


def y_error(y_gpu_f64, y_ref_f64, act):
    """Normwise error of y as defined in the module docstring."""
    if act == "bf16":
        ref = bf16_bits_to_f64(f64_to_bf16_bits(y_ref_f64))
    else:
        ref = y_ref_f64
    den = np.linalg.norm(ref)
    if den == 0.0:
        return float(np.linalg.norm(y_gpu_f64))
    return float(np.linalg.norm(y_gpu_f64 - ref) / den)


def state_error(s_gpu, s_ref):
    den = float(np.max(np.abs(s_ref))) if s_ref.size else 0.0
    num = float(np.max(np.abs(np.asarray(s_gpu, np.float64) - s_ref))) if s_ref.size else 0.0
    return num / den if den > 0 else num


def y_report(y_gpu_f64, y_ref_f64, act):
    """The figures the gates read: normwise error against the rounded and the
    unrounded oracle, max-normwise error, and for bf16 the share of elements
    more than 1 ulp off and the worst element in ulp and against the
    elementwise bound."""
    y = np.asarray(y_gpu_f64, np.float64).reshape(-1)
    r = np.asarray(y_ref_f64, np.float64).reshape(-1)
    rmax = float(np.max(np.abs(r))) if r.size else 0.0
    out = {"n": int(r.size), "l2_vs_rounded": y_error(y, r, act),
           "l2_vs_fp64": float(np.linalg.norm(y - r) / max(np.linalg.norm(r), 1e-300)),
           "maxnorm": float(np.max(np.abs(y - r)) / max(rmax, 1e-300)) if r.size else 0.0}
    if act == "bf16" and r.size:
        rr = bf16_bits_to_f64(f64_to_bf16_bits(r))
        ulp = bf16_ulp(rr)
        e = np.abs(y - rr)
        out["share_gt_1ulp"] = float(np.mean(e > ulp))
        out["max_ulp"] = float(np.max(e / ulp))
        bound = ULP_MAX * ulp + ABS_FLOOR * rmax
        out["max_over_bound"] = float(np.max(e / bound)) if rmax > 0 else float(np.max(e))
    return out


def _log(tag, fig):
    path = os.environ.get("M2_GATE_LOG")
    if not path:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    with open(path, "a") as f:
        f.write(json.dumps(dict(test=test, tag=tag, **fig)) + "\n")


def check_y(y_gpu_f64, y_ref_f64, act, tag="y", l2_tol=Y_TOL, f32_maxnorm=F32_MAXNORM_TOL):
    """Applies every gate of the module docstring to one result; returns its figures."""
    fig = y_report(y_gpu_f64, y_ref_f64, act)
    _log(tag, fig)
    assert fig["l2_vs_rounded"] <= l2_tol, (tag, fig)
    if act == "bf16":
        if fig["n"]:
            assert fig["share_gt_1ulp"] <= ULP_SHARE_TOL, (tag, fig)
            assert fig["max_over_bound"] <= 1.0, (tag, fig)
    else:
        assert fig["maxnorm"] <= f32_maxnorm, (tag, fig)
    return fig


def check_state(s_gpu, s_ref, tag="state", tol=STATE_TOL):
    err = state_error(s_gpu, s_ref)
    _log(tag, {"maxnorm": err})
    assert err <= tol, (tag, err)
    return err


def check_scan_y(y_gpu_f64, y_ref_f64, ybar, act, tag="y", l2_tol=Y_TOL):
    """The chunked scan's gates (module docstring): normwise, and every element
    within the forward error bound of its bf16-operand arithmetic."""
    fig = y_report(y_gpu_f64, y_ref_f64, act)
    y = np.asarray(y_gpu_f64, np.float64).reshape(-1)
    r = np.asarray(y_ref_f64, np.float64).reshape(-1)
    m = np.asarray(ybar, np.float64).reshape(-1)
    if act == "bf16":
        rr = bf16_bits_to_f64(f64_to_bf16_bits(r))
        slack = bf16_ulp(rr)
    else:
        rr, slack = r, 2.0 ** -126  # fp32 values below the least normal are flushed by the GPU's fp32 math
    bound = slack + SCAN_ROUNDINGS * BF16_U * m + F32_SLACK * (np.abs(r) + m)
    e = np.abs(y - rr)
    fig["max_over_scan_bound"] = float(np.max(e / bound)) if r.size else 0.0
    fig["share_pass_if_zero"] = float(np.mean(np.abs(rr) <= bound)) if r.size else 0.0
    _log(tag, fig)
    assert fig["l2_vs_rounded"] <= l2_tol, (tag, fig)
    assert fig["max_over_scan_bound"] <= 1.0, (tag, fig)
    return fig


def check_y_rounded_inside(y_gpu_f64, y_ref_f64, tag="y", l2_tol=Y_TOL):
    """Gates on a bf16 result whose computation stores an intermediate in
    bf16 (a normalised row staged for a projection, the in_proj rows a block
    reads back): normwise 2e-3 and no element beyond 4 ulp + 1e-3 max|ref|.
    The GPU rounds its fp32 intermediate and the oracle its exact one, so an
    intermediate whose exact value lies within fp32 error of a rounding
    boundary comes out one ulp apart; that moves every output it feeds by a
    little, which the share gate of check_y would count for outputs near
    zero. The share is logged, not gated."""
    fig = y_report(y_gpu_f64, y_ref_f64, "bf16")
    _log(tag, fig)
    assert fig["l2_vs_rounded"] <= l2_tol, (tag, fig)
    if fig["n"]:
        assert fig["max_over_bound"] <= 1.0, (tag, fig)
    return fig


def check_drift(y_gpu_f64, y_ref_f64, n_blocks, tag="h"):
    """Gate on the residual stream after n_blocks blocks evaluated twice with
    different roundings of their bf16 activations (GPU against oracle, or
    cached steps against the chunked recompute): once two evaluations differ
    by one ulp anywhere, each later rounding point turns the difference into
    ulp-sized differences of its own, so they drift apart by bf16 rounding
    noise accumulated over the blocks. Gate: normwise <= 2 u sqrt(n_blocks),
    u = 2^-8 (4.3e-2 for the 31 blocks of Nemotron-H, whose single block
    adds ~0.2 of the stream's norm: dropping or repeating one fails it)."""
    fig = y_report(y_gpu_f64, y_ref_f64, "bf16")
    tol = 2.0 * BF16_U * float(np.sqrt(n_blocks))
    fig["drift_tol"] = tol
    _log(tag, fig)
    assert fig["l2_vs_rounded"] <= tol, (tag, fig)
    return fig
