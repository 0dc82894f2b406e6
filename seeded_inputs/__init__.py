"""Seeded synthetic inputs for the Mamba2 mixer core, shared by the oracle's
tests, the CUDA parity tests and bench.py.

This module draws random numbers and converts between storage formats. It
holds none of the mixer's arithmetic (no conv, SiLU, softplus, exp or scan):
that lives, independently, in the oracle and in the CUDA library.

Shapes and distributions follow the Nemotron-H text_config of the VoiceChat
checkpoint (issue "feat(nemotron_voicechat): load the VoiceChat checkpoint and
run offline duplex inference", section config.json / text_config:
mamba_num_heads 128, mamba_head_dim 80, ssm_state_size 128, n_groups 8,
conv_kernel 4, use_conv_bias true). No checkpoint or dataset is involved; the
activations and weights are drawn from these distributions:

  x, B, C (pre-conv)  ~ N(0, 1)
  dt_raw              ~ N(0, 0.5)            (sigma 0.5)
  dt_bias             = inverse softplus of a log-uniform draw in [1e-3, 0.1]
  A_log               = log U[1, 16]
  D                   ~ N(0, 1)
  conv_w, conv_b      ~ U(-0.5, 0.5)          (conv weight stored [CH, K])

Activations are stored as bf16 (as uint16 bit patterns, round-to-nearest-even
from fp32) or as fp32; parameters are fp32.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "Dims",
    "REAL_SHAPE",
    "TINY_SHAPE",
    "MAMBA_LAYERS",
    "mixer_params",
    "mixer_activations",
    "mixer_inputs",
    "f32_to_bf16_bits",
    "f64_to_bf16_bits",
    "bf16_bits_to_f64",
    "bf16_bits_to_f32",
    "as_f64",
    "conv_state_inputs",
    "ssm_state_inputs",
    "norm_inputs",
    "qlinear_inputs",
    "attn_inputs",
    "device_mixer_inputs",
    "LMConfig",
    "REAL_LM",
    "TINY_LM",
    "lm_weights",
    "lm_hidden",
    "device_lm_weights",
]


@dataclass(frozen=True)
class Dims:
    """Mixer dimensions. CH = H*P + 2*G*N conv channels (x | B | C)."""

    H: int  # mamba_num_heads
    P: int  # mamba_head_dim
    N: int  # ssm_state_size
    G: int  # n_groups
    K: int = 4  # conv_kernel

    @property
    def CH(self) -> int:
        return self.H * self.P + 2 * self.G * self.N

    @property
    def R(self) -> int:
        """Heads per group."""
        return self.H // self.G


# Nemotron-H mixer shape from the VoiceChat text_config.
REAL_SHAPE = Dims(H=128, P=80, N=128, G=8, K=4)
# The tiny fp32 mixer used for brute-force checks: 4 heads x 16, state 16, 1 group.
TINY_SHAPE = Dims(H=4, P=16, N=16, G=1, K=4)

# Layer indices of the Mamba ('M') entries of hybrid_override_pattern
# "M-M-M-MM-M-M-M*-M-M-M*-M-M-M-M*-M-M-M-M*-M-MM-M-M-M-M-M-" (27 of 56 layers).
_PATTERN = "M-M-M-MM-M-M-M*-M-M-M*-M-M-M-M*-M-M-M-M*-M-MM-M-M-M-M-M-"
MAMBA_LAYERS = tuple(i for i, ch in enumerate(_PATTERN) if ch == "M")


# ---------------------------------------------------------------- bf16 codec
def f32_to_bf16_bits(a) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even.
    Inputs are finite (no NaN handling needed for these distributions)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def f64_to_bf16_bits(a) -> np.ndarray:
    """fp64 -> bf16 bit patterns with a single round-to-nearest-even step
    (no double rounding through fp32). Valid for finite values in the
    normal bf16 range and for exact zeros; values below 2**-126 in magnitude
    are flushed to signed zero."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    bits = a.view(np.uint64)
    sign = (bits >> np.uint64(63)).astype(np.uint64)
    mag = bits & np.uint64(0x7FFFFFFFFFFFFFFF)
    # bf16 keeps 7 explicit mantissa bits; fp64 has 52 -> drop 45 bits.
    drop = np.uint64(45)
    half = np.uint64(1) << (drop - np.uint64(1))
    lsb = (mag >> drop) & np.uint64(1)
    rounded = (mag + half - np.uint64(1) + lsb) >> drop << drop
    r64 = rounded.view(np.float64)
    tiny = r64 < 2.0 ** -126
    r32 = r64.astype(np.float32)  # exact: at most 8 significant bits
    out = (r32.view(np.uint32) >> 16).astype(np.uint16)
    out = np.where(tiny, np.uint16(0), out)
    out = out | (sign.astype(np.uint16) << np.uint16(15))
    return out.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b) -> np.ndarray:
    """bf16 bit patterns -> fp64 (exact)."""
    return bf16_bits_to_f32(b).astype(np.float64)


# ---------------------------------------------------------------- generators
def mixer_params(seed: int, d: Dims) -> dict:
    """Per-layer parameters (fp32): A_log, D, dt_bias [H]; conv_w [CH, K];
    conv_b [CH]."""
    rng = np.random.default_rng([seed, 0x5EED, 1])
    dt_target = np.exp(rng.uniform(np.log(1e-3), np.log(0.1), size=d.H))
    # inverse softplus of the target step size: the draw is specified as such
    dt_bias = np.log(np.expm1(dt_target))
    A_log = np.log(rng.uniform(1.0, 16.0, size=d.H))
    D = rng.standard_normal(d.H)
    conv_w = rng.uniform(-0.5, 0.5, size=(d.CH, d.K))
    conv_b = rng.uniform(-0.5, 0.5, size=d.CH)
    f = lambda v: np.ascontiguousarray(v, dtype=np.float32)  # noqa: E731
    return dict(A_log=f(A_log), D=f(D), dt_bias=f(dt_bias), conv_w=f(conv_w), conv_b=f(conv_b))


def mixer_activations(seed: int, d: Dims, batch: int, T: int, act: str = "bf16") -> dict:
    """Pre-conv activations x [b,T,H,P], B [b,T,G,N], C [b,T,G,N],
    dt_raw [b,T,H]. act='bf16' -> uint16 bit patterns; act='f32' -> float32."""
    rng = np.random.default_rng([seed, 0x5EED, 2])
    x = rng.standard_normal((batch, T, d.H, d.P), dtype=np.float32)
    B = rng.standard_normal((batch, T, d.G, d.N), dtype=np.float32)
    C = rng.standard_normal((batch, T, d.G, d.N), dtype=np.float32)
    dt_raw = (0.5 * rng.standard_normal((batch, T, d.H), dtype=np.float32)).astype(np.float32)
    out = dict(x=x, B=B, C=C, dt_raw=dt_raw)
    if act == "bf16":
        out = {k: f32_to_bf16_bits(v) for k, v in out.items()}
    elif act != "f32":
        raise ValueError(f"act must be 'bf16' or 'f32', got {act!r}")
    return out


def mixer_inputs(seed: int, d: Dims, batch: int, T: int, act: str = "bf16") -> dict:
    """Parameters and activations of one mixer layer, both from `seed`."""
    p = mixer_params(seed, d)
    p.update(mixer_activations(seed, d, batch, T, act))
    p["act"] = act
    return p


def as_f64(a, act: str) -> np.ndarray:
    """Exact fp64 view of a stored activation (bf16 bits or fp32)."""
    if act == "bf16":
        return bf16_bits_to_f64(a)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def conv_state_inputs(seed: int, d: Dims, batch: int, act: str = "bf16") -> np.ndarray:
    """A random pre-conv conv tail [b, K-1, CH] (x|B|C channel order), used as
    an initial conv state in continuation tests."""
    rng = np.random.default_rng([seed, 0x5EED, 3])
    v = rng.standard_normal((batch, d.K - 1, d.CH), dtype=np.float32)
    return f32_to_bf16_bits(v) if act == "bf16" else v


def ssm_state_inputs(seed: int, d: Dims, batch: int, scale: float = 0.05) -> np.ndarray:
    """A random fp32 SSM state [b, H, P, N] for continuation tests."""
    rng = np.random.default_rng([seed, 0x5EED, 4])
    return (scale * rng.standard_normal((batch, d.H, d.P, d.N))).astype(np.float32)


def device_mixer_inputs(seed: int, d: Dims, batch: int, T: int, device, act: str = "bf16") -> dict:
    """The same distributions drawn on a device with torch's generator, for
    workloads too large to draw on the host (the long-prefill run: 27 layers
    x 4 x 4096 frames). Returns torch tensors (activations in the act dtype,
    parameters fp32). Consumers that need host copies slice and copy them."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 17)
    dt = torch.bfloat16 if act == "bf16" else torch.float32

    def normal(shape, sigma=1.0):
        return (torch.randn(shape, generator=g, device=device) * sigma).to(dt)

    def uniform(shape, lo, hi):
        return torch.rand(shape, generator=g, device=device, dtype=torch.float64) * (hi - lo) + lo

    out = dict(x=normal((batch, T, d.H, d.P)), B=normal((batch, T, d.G, d.N)), C=normal((batch, T, d.G, d.N)),
               dt_raw=normal((batch, T, d.H), 0.5))
    dt_target = torch.exp(uniform((d.H,), np.log(1e-3), np.log(0.1)))
    out["dt_bias"] = torch.log(torch.expm1(dt_target)).float()
    out["A_log"] = torch.log(uniform((d.H,), 1.0, 16.0)).float()
    out["D"] = torch.randn((d.H,), generator=g, device=device, dtype=torch.float64).float()
    out["conv_w"] = uniform((d.CH, d.K), -0.5, 0.5).float().contiguous()
    out["conv_b"] = uniform((d.CH,), -0.5, 0.5).float()
    out["act"] = act
    return out


def norm_inputs(seed: int, d: Dims, rows: int, act: str = "bf16") -> dict:
    """Inputs of the gated output norm: y, z [rows, H*P] ~ N(0, 1) (act dtype
    bit patterns for bf16), weight [H*P] ~ 1 + N(0, 0.1) fp32."""
    rng = np.random.default_rng([seed, 0x5EED, 5])
    y = rng.standard_normal((rows, d.H * d.P), dtype=np.float32)
    z = rng.standard_normal((rows, d.H * d.P), dtype=np.float32)
    w = (1.0 + 0.1 * rng.standard_normal(d.H * d.P)).astype(np.float32)
    if act == "bf16":
        y, z = f32_to_bf16_bits(y), f32_to_bf16_bits(z)
    return dict(y=y, z=z, weight=w, act=act)


def qlinear_inputs(seed: int, rows: int, in_features: int, out_features: int, group: int = 64) -> dict:
    """Inputs of a 4-bit affine group-quantized linear layer: x [rows, in]
    ~ N(0, 1) as bf16 bit patterns; wq [out, in/8] uint32 of uniformly drawn
    4-bit fields; scales ~ U(0.5, 1.5) / (4 sqrt(in)) and biases
    ~ -7.5 scale U(0.8, 1.2) [out, in/group] as bf16 bit patterns, so the
    weights are centred near zero with a spread like a trained layer's."""
    rng = np.random.default_rng([seed, 0x5EED, 6])
    x = rng.standard_normal((rows, in_features), dtype=np.float32)
    wq = rng.integers(0, 2**32, size=(out_features, in_features // 8), dtype=np.uint64).astype(np.uint32)
    ng = in_features // group
    scales = rng.uniform(0.5, 1.5, size=(out_features, ng)) / (4.0 * np.sqrt(in_features))
    biases = -7.5 * scales * rng.uniform(0.8, 1.2, size=(out_features, ng))
    return dict(x=f32_to_bf16_bits(x), wq=wq, scales=f32_to_bf16_bits(scales.astype(np.float32)),
                biases=f32_to_bf16_bits(biases.astype(np.float32)), group=group)


def attn_inputs(seed: int, S: int, Hq: int, Hkv: int, D: int, Tmax: int, lengths, act: str = "bf16") -> dict:
    """One cached decode position of grouped-query attention: q [S,Hq,D],
    k_new, v_new [S,Hkv,D] and the caches k_cache, v_cache [S,Hkv,Tmax,D],
    all ~ N(0, 1) (the cache slots past each session's length hold values
    too, which the position must neither read nor change); lengths [S]
    int32. act='bf16' -> uint16 bit patterns; act='f32' -> float32."""
    rng = np.random.default_rng([seed, 0x5EED, 7])
    out = dict(q=rng.standard_normal((S, Hq, D), dtype=np.float32),
               k_new=rng.standard_normal((S, Hkv, D), dtype=np.float32),
               v_new=rng.standard_normal((S, Hkv, D), dtype=np.float32),
               k_cache=rng.standard_normal((S, Hkv, Tmax, D), dtype=np.float32),
               v_cache=rng.standard_normal((S, Hkv, Tmax, D), dtype=np.float32))
    if act == "bf16":
        out = {k: f32_to_bf16_bits(v) for k, v in out.items()}
    elif act != "f32":
        raise ValueError(f"act must be 'bf16' or 'f32', got {act!r}")
    out["lengths"] = np.ascontiguousarray(lengths, dtype=np.int32)
    out["act"] = act
    return out


# ------------------------------------------------------- hybrid language model
@dataclass(frozen=True)
class LMConfig:
    """The blocks of the hybrid language model that the library runs: the
    'M' (Mamba) and '*' (attention) entries of the layer pattern, in order."""

    hidden: int
    mixer: Dims
    n_heads: int
    n_kv_heads: int
    head_dim: int
    kinds: str
    eps: float = 1e-5


# Nemotron-H (VoiceChat issue, section config.json / text_config): hidden
# 4480, the 27 'M' and 4 '*' entries of hybrid_override_pattern, attention
# 40 / 8 heads of 128.
REAL_LM = LMConfig(4480, REAL_SHAPE, 40, 8, 128, "".join(c for c in _PATTERN if c != "-"))
# A small model of the same structure for brute-force and long-sequence checks.
TINY_LM = LMConfig(256, Dims(H=8, P=16, N=16, G=2), 4, 2, 128, "MM*M*M")


def _qweights(rng, n_out: int, n_in: int, group: int = 64):
    """4-bit affine group-quantized weights drawn as qlinear_inputs draws them."""
    wq = rng.integers(0, 2**32, size=(n_out, n_in // 8), dtype=np.uint64).astype(np.uint32)
    ng = n_in // group
    scales = rng.uniform(0.5, 1.5, size=(n_out, ng)) / (4.0 * np.sqrt(n_in))
    biases = -7.5 * scales * rng.uniform(0.8, 1.2, size=(n_out, ng))
    return wq, f32_to_bf16_bits(scales.astype(np.float32)), f32_to_bf16_bits(biases.astype(np.float32))


def lm_weights(seed: int, cfg: LMConfig) -> list:
    """Synthetic weights of every block (no checkpoint is involved), one dict
    per block: norm weights ~ 1 + N(0, 0.1) fp32; 4-bit in_proj [2HP+2GN+H,
    hidden] and out_proj [hidden, HP] drawn as qlinear_inputs draws them; the
    mixer parameters of mixer_params; bf16 q|k|v [(Hq+2Hkv)D, hidden] and
    output [hidden, Hq D] projections ~ N(0, 1/in)."""
    d = cfg.mixer
    W = 2 * d.H * d.P + 2 * d.G * d.N + d.H
    out = []
    for i, kind in enumerate(cfg.kinds):
        rng = np.random.default_rng([seed, 0x5EED, 8, i])
        L = {"norm_w": (1.0 + 0.1 * rng.standard_normal(cfg.hidden)).astype(np.float32)}
        if kind == "M":
            L["in_wq"], L["in_scales"], L["in_biases"] = _qweights(rng, W, cfg.hidden)
            L.update(mixer_params(seed * 131 + i, d))
            L["gnorm_w"] = (1.0 + 0.1 * rng.standard_normal(d.H * d.P)).astype(np.float32)
            L["out_wq"], L["out_scales"], L["out_biases"] = _qweights(rng, cfg.hidden, d.H * d.P)
        else:
            nq = (cfg.n_heads + 2 * cfg.n_kv_heads) * cfg.head_dim
            ao = cfg.n_heads * cfg.head_dim
            L["wqkv"] = f32_to_bf16_bits(rng.standard_normal((nq, cfg.hidden), dtype=np.float32) / np.sqrt(cfg.hidden))
            L["wo"] = f32_to_bf16_bits(rng.standard_normal((cfg.hidden, ao), dtype=np.float32) / np.sqrt(ao))
        out.append(L)
    return out


def lm_hidden(seed: int, cfg: LMConfig, S: int, T: int) -> np.ndarray:
    """Inputs of T positions of S sessions (the fused embeddings): [S, T,
    hidden] ~ N(0, 1) as bf16 bit patterns."""
    rng = np.random.default_rng([seed, 0x5EED, 9])
    return f32_to_bf16_bits(rng.standard_normal((S, T, cfg.hidden), dtype=np.float32))


def device_lm_weights(seed: int, cfg: LMConfig, device) -> list:
    """lm_weights' distributions drawn on a device with torch's generator, for
    the full-size model (1.5 GB of 4-bit and bf16 weights): torch tensors with
    the same layouts and dtypes (bf16 fields as torch.bfloat16, packed 4-bit
    words as int32)."""
    import torch
    d = cfg.mixer
    W = 2 * d.H * d.P + 2 * d.G * d.N + d.H
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 29)

    def uni(shape, lo, hi):
        return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo

    def qw(n_out, n_in):
        wq = torch.randint(-2**31, 2**31 - 1, (n_out, n_in // 8), generator=g, device=device, dtype=torch.int32)
        sc = uni((n_out, n_in // 64), 0.5, 1.5) / (4.0 * float(np.sqrt(n_in)))
        bi = -7.5 * sc * uni((n_out, n_in // 64), 0.8, 1.2)
        return wq, sc.to(torch.bfloat16), bi.to(torch.bfloat16)

    out = []
    for i, kind in enumerate(cfg.kinds):
        L = {"norm_w": 1.0 + 0.1 * torch.randn(cfg.hidden, generator=g, device=device)}
        if kind == "M":
            L["in_wq"], L["in_scales"], L["in_biases"] = qw(W, cfg.hidden)
            dt_target = torch.exp(uni((d.H,), float(np.log(1e-3)), float(np.log(0.1))).double())
            L["dt_bias"] = torch.log(torch.expm1(dt_target)).float()
            L["A_log"] = torch.log(uni((d.H,), 1.0, 16.0))
            L["D"] = torch.randn(d.H, generator=g, device=device)
            L["conv_w"] = uni((d.CH, d.K), -0.5, 0.5).contiguous()
            L["conv_b"] = uni((d.CH,), -0.5, 0.5)
            L["gnorm_w"] = 1.0 + 0.1 * torch.randn(d.H * d.P, generator=g, device=device)
            L["out_wq"], L["out_scales"], L["out_biases"] = qw(cfg.hidden, d.H * d.P)
        else:
            nq = (cfg.n_heads + 2 * cfg.n_kv_heads) * cfg.head_dim
            ao = cfg.n_heads * cfg.head_dim
            L["wqkv"] = (torch.randn((nq, cfg.hidden), generator=g, device=device) / float(np.sqrt(cfg.hidden))
                         ).to(torch.bfloat16)
            L["wo"] = (torch.randn((cfg.hidden, ao), generator=g, device=device) / float(np.sqrt(ao))).to(torch.bfloat16)
        out.append(L)
    return out
