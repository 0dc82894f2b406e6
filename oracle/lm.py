"""fp64 oracle of the hybrid language model's blocks that the library runs:
one cached position (step) and a full-history recompute (prefill) of the
Nemotron-H 'M' (Mamba) and '*' (attention) blocks (VoiceChat issue, section
config.json / text_config: hybrid_override_pattern, hidden_size 4480,
40 / 8 attention heads of 128, layer_norm_epsilon 1e-5; the session keeps
"Mamba2 state and attention KV caches", "docs/nemotron-voicechat.md",
section Online session; stepping and recompute give the same tokens, same
doc, section Offline timeline).

TEST INFRASTRUCTURE, like the rest of this package. It composes the
package's pinned functions (rmsnorm, qlinear, mixer_step / mixer_scan,
gated_norm, linear, attn_decode) in the block order the pages give; the
only arithmetic of its own is the residual add.

Per block, on the residual stream h:
  'M': proj = in_proj(rmsnorm(h)) = z | x | B | C | dt;  y = mixer core;
       h = h + out_proj(gated_norm(y, z))
  '*': q | k | v = Wqkv rmsnorm(h);  o = attention with the KV-cache append;
       h = h + Wo o
Reading of the pages' bf16 model: every activation that passes between
operations (proj, y, the normalised rows, q|k|v, o and h itself) is stored
in bf16, so the oracle rounds each one once to bf16 (nearest even) from its
exact fp64 value; the SSM state, conv tail and KV caches hold exact values
(the conv tail and the caches hold bf16 inputs, hence exact). Everything
else is fp64.
"""
from __future__ import annotations

import numpy as np

from seeded_inputs import LMConfig, bf16_bits_to_f64, f64_to_bf16_bits

from . import attn_decode, gated_norm, linear, mixer_scan, mixer_step, qlinear, rmsnorm


def rb(a) -> np.ndarray:
    """Round fp64 values to bf16 (nearest even), returned as fp64."""
    return bf16_bits_to_f64(f64_to_bf16_bits(np.asarray(a, np.float64)))


def _f(a):
    """Stored bf16 bit patterns -> fp64 values (other arrays: as fp64)."""
    a = np.asarray(a)
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


class LMOracle:
    """Caches of S sessions and the blocks' weights (seeded_inputs.lm_weights
    layout: numpy arrays, bf16 fields as bit patterns)."""

    def __init__(self, cfg: LMConfig, weights: list, S: int, max_len: int):
        self.cfg, self.w, self.S, self.max_len = cfg, weights, S, max_len
        d = cfg.mixer
        self.ssm = {}
        self.conv = {}
        self.kc = {}
        self.vc = {}
        for i, kind in enumerate(cfg.kinds):
            if kind == "M":
                self.ssm[i] = np.zeros((S, d.H, d.P, d.N))
                self.conv[i] = np.zeros((S, d.K - 1, d.CH))
            else:
                self.kc[i] = np.zeros((S, cfg.n_kv_heads, max_len, cfg.head_dim))
                self.vc[i] = np.zeros((S, cfg.n_kv_heads, max_len, cfg.head_dim))
        self.lengths = np.zeros(S, np.int32)

    # ------------------------------------------------------------ pieces
    def _split(self, proj):
        """z | x | B | C | dt of in_proj rows [..., W]."""
        d = self.cfg.mixer
        HP, GN = d.H * d.P, d.G * d.N
        z = proj[..., :HP]
        x = proj[..., HP:2 * HP]
        B = proj[..., 2 * HP:2 * HP + GN]
        C = proj[..., 2 * HP + GN:2 * HP + 2 * GN]
        dt = proj[..., 2 * HP + 2 * GN:]
        return z, x, B, C, dt

    def _mamba_in(self, L, h):
        x = rb(rmsnorm(h, L["norm_w"], self.cfg.eps))
        return rb(qlinear(x, L["in_wq"], _f(L["in_scales"]), _f(L["in_biases"])))

    def _mamba_out(self, L, h, y, z):
        d = self.cfg.mixer
        yn = rb(gated_norm(y, z, L["gnorm_w"], d.G, self.cfg.eps))
        return rb(h + qlinear(yn, L["out_wq"], _f(L["out_scales"]), _f(L["out_biases"])))

    def _qkv(self, L, h):
        c = self.cfg
        x = rb(rmsnorm(h, L["norm_w"], c.eps))
        qkv = rb(linear(x, _f(L["wqkv"])))
        nq, nk = c.n_heads * c.head_dim, c.n_kv_heads * c.head_dim
        return qkv[..., :nq], qkv[..., nq:nq + nk], qkv[..., nq + nk:]

    def _attend(self, i, q, k, v, extra):
        """One position of every session: q [S, Hq*D], k, v [S, Hkv*D]."""
        c, S = self.cfg, self.S
        o = attn_decode(q.reshape(S, c.n_heads, c.head_dim), k.reshape(S, c.n_kv_heads, c.head_dim),
                        v.reshape(S, c.n_kv_heads, c.head_dim), self.kc[i], self.vc[i], self.lengths + extra,
                        c.head_dim ** -0.5)
        return rb(o.reshape(S, -1))

    # ------------------------------------------------------------ positions
    def step_block(self, i, h):
        """Block i of one cached position: h [S, hidden] (bf16 values) -> the
        residual stream after it; the block's caches are updated (the
        attention blocks write slot `lengths`, which step() advances after
        the last block)."""
        d = self.cfg.mixer
        L = self.w[i]
        if self.cfg.kinds[i] == "M":
            proj = self._mamba_in(L, h)
            z, x, B, C, dt = self._split(proj)
            frame = dict(x=x.reshape(self.S, d.H, d.P), B=B.reshape(self.S, d.G, d.N),
                         C=C.reshape(self.S, d.G, d.N), dt_raw=dt, act="f32")
            y = rb(mixer_step(d, frame, L, self.ssm[i], self.conv[i])).reshape(self.S, -1)
            return self._mamba_out(L, h, y, z)
        q, k, v = self._qkv(L, h)
        o = self._attend(i, q, k, v, 0)
        return rb(h + linear(o, _f(L["wo"])))

    def step(self, h):
        """One cached position: h [S, hidden] (fp64 values or bf16 bits) ->
        the residual stream after the last block [S, hidden] (bf16 values)."""
        h = _f(h)
        for i in range(len(self.cfg.kinds)):
            h = self.step_block(i, h)
        self.lengths += 1
        return h

    def prefill(self, H):
        """T positions at once from the current caches: H [S, T, hidden] ->
        [S, T, hidden]; the Mamba blocks run the chunked-scan form of the
        mixer (mixer_scan), the attention blocks the positions in order."""
        d, S = self.cfg.mixer, self.S
        h = _f(H)
        T = h.shape[1]
        for i, kind in enumerate(self.cfg.kinds):
            L = self.w[i]
            if kind == "M":
                proj = self._mamba_in(L, h)
                z, x, B, C, dt = self._split(proj)
                inp = dict(L, x=x.reshape(S, T, d.H, d.P), B=B.reshape(S, T, d.G, d.N),
                           C=C.reshape(S, T, d.G, d.N), dt_raw=dt, act="f32")
                r = mixer_scan(d, inp, init_ssm=self.ssm[i], init_conv=self.conv[i])
                self.ssm[i], self.conv[i] = r["final_ssm"], r["final_conv"]
                y = rb(r["y"]).reshape(S, T, -1)
                h = self._mamba_out(L, h, y, z)
            else:
                q, k, v = self._qkv(L, h)
                o = np.stack([self._attend(i, q[:, t], k[:, t], v[:, t], t) for t in range(T)], axis=1)
                h = rb(h + linear(o, _f(L["wo"])))
        self.lengths += T
        return h
