"""Helpers shared by the parity tests: moving seeded inputs to the device,
reading results back, and the tolerance measures.

Tolerances (the mixer core's acceptance bar):
  * y, bf16 output: normwise  ||y_gpu - bf16_rne(y_oracle)||_2 / ||bf16_rne(y_oracle)||_2 <= 2e-3.
    (Elementwise relative error is not used: a perfectly rounded fp64 result
    already differs from itself by up to 2^-8 elementwise, and entries near
    zero have unbounded relative error.)
  * y, fp32 output: normwise ||y_gpu - y_oracle|| / ||y_oracle|| <= 2e-3.
  * fp32 SSM state: max|e| / max|ref| <= 1e-4.
  * conv tail: bitwise equal to the last K-1 input frames.
"""
from __future__ import annotations

import numpy as np

from seeded_inputs import bf16_bits_to_f64, f64_to_bf16_bits

Y_TOL = 2e-3
STATE_TOL = 1e-4


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
    """Extra, ungated figures: error against the unrounded oracle,
    max-normwise error, and the share of elements more than 1 bf16 ulp off."""
    out = {"l2_vs_rounded": y_error(y_gpu_f64, y_ref_f64, act),
           "l2_vs_fp64": float(np.linalg.norm(y_gpu_f64 - y_ref_f64) / max(np.linalg.norm(y_ref_f64), 1e-300)),
           "maxnorm": float(np.max(np.abs(y_gpu_f64 - y_ref_f64)) / max(np.max(np.abs(y_ref_f64)), 1e-300))}
    if act == "bf16":
        ref = bf16_bits_to_f64(f64_to_bf16_bits(y_ref_f64))
        ulp = np.maximum(np.abs(ref), 2.0 ** -126) * 2.0 ** -7
        out["frac_gt_1ulp"] = float(np.mean(np.abs(y_gpu_f64 - ref) > 1.0001 * ulp))
    return out
