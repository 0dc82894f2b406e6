"""GPU parity of the hybrid model's blocks around the mixer core, through the
C ABI: the fused 4-bit projections (block pre-norm before in_proj, gated
output norm and residual around out_proj), the dense bf16 attention
projections, the strided mixer calls that read in_proj's z | x | B | C | dt
rows in place, and one cached position of the 27 Mamba + 4 attention blocks
of Nemotron-H (VoiceChat issue, section config.json / text_config) against
the oracle's composition of the same blocks and against the library's own
full-history recompute ("docs/nemotron-voicechat.md", section Offline
timeline: both modes give the same tokens)."""
import numpy as np
import pytest

from m2_testlib import act_empty, bits_of, check_y, check_y_rounded_inside, from_dev_act, to_dev
from seeded_inputs import (REAL_LM, REAL_SHAPE, TINY_LM, Dims, bf16_bits_to_f64, device_lm_weights, f32_to_bf16_bits,
                           lm_hidden, lm_weights, mixer_inputs, qlinear_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m2():
    import full_duplex_speech_gb300 as m2
    m2.load()
    return m2


def _bf16(rng, shape, scale=1.0):
    return f32_to_bf16_bits((scale * rng.standard_normal(shape)).astype(np.float32))


# ------------------------------------------------------------- linear layers
@pytest.mark.parametrize("rows,n_in,n_out", [(1, 4480, 300), (3, 4480, 129), (5, 512, 77), (1, 4480, 22656)])
def test_qlinear_with_fused_rmsnorm_and_residual(m2, rows, n_in, n_out):
    import oracle
    from oracle.lm import rb
    import torch
    inp = qlinear_inputs(500 + rows + n_out, rows, n_in, n_out)
    rng = np.random.default_rng(501)
    w = (1 + 0.1 * rng.standard_normal(n_in)).astype(np.float32)
    res = _bf16(rng, (rows, n_out))
    x = to_dev(inp["x"])
    y = act_empty((rows, n_out), "bf16")
    r = to_dev(res)
    m2.mamba2_qlinear_fused(rows, n_in, n_out, x, n_in, m2.row_norm(m2.NORM_RMS, to_dev(w), 1e-5),
                            torch.from_numpy(inp["wq"].view(np.int32)).cuda(), to_dev(inp["scales"]),
                            to_dev(inp["biases"]), r, y)
    torch.cuda.synchronize()
    xn = rb(oracle.rmsnorm(bf16_bits_to_f64(inp["x"]), w, 1e-5))
    ref = bf16_bits_to_f64(res) + oracle.qlinear(xn, inp["wq"], bf16_bits_to_f64(inp["scales"]),
                                                bf16_bits_to_f64(inp["biases"]))
    check_y_rounded_inside(from_dev_act(y, "bf16"), ref)


@pytest.mark.parametrize("rows,G", [(1, 8), (2, 8), (4, 8), (3, 1)])
def test_qlinear_with_fused_gated_norm_strided_gate_and_residual_in_place(m2, rows, G):
    """out_proj as a Mamba block runs it: x = y [rows, 10240], z read from
    the first 10240 columns of rows 22656 wide, the residual stream updated
    in place."""
    import oracle
    from oracle.lm import rb
    import torch
    n_in, n_out, width = 10240, 4480, 22656
    inp = qlinear_inputs(510 + rows, rows, n_in, n_out)
    rng = np.random.default_rng(511)
    zrows = _bf16(rng, (rows, width))
    w = (1 + 0.1 * rng.standard_normal(n_in)).astype(np.float32)
    h0 = _bf16(rng, (rows, n_out))
    h = to_dev(h0)
    nm = m2.row_norm(m2.NORM_GATED, to_dev(w), 1e-5, groups=G, gate=to_dev(zrows), gate_stride=width)
    m2.mamba2_qlinear_fused(rows, n_in, n_out, to_dev(inp["x"]), n_in, nm,
                            torch.from_numpy(inp["wq"].view(np.int32)).cuda(), to_dev(inp["scales"]),
                            to_dev(inp["biases"]), h, h)
    torch.cuda.synchronize()
    yn = rb(oracle.gated_norm(bf16_bits_to_f64(inp["x"]), bf16_bits_to_f64(zrows[:, :n_in]), w, G, 1e-5))
    ref = bf16_bits_to_f64(h0) + oracle.qlinear(yn, inp["wq"], bf16_bits_to_f64(inp["scales"]),
                                               bf16_bits_to_f64(inp["biases"]))
    check_y_rounded_inside(from_dev_act(h, "bf16"), ref)


@pytest.mark.parametrize("rows,n_in,n_out,norm,res", [(1, 4480, 7168, True, False), (3, 4480, 7168, True, False),
                                                      (1, 5120, 4480, False, True), (9, 5120, 4480, False, True),
                                                      (2, 256, 1024, True, True), (16, 512, 96, False, False)])
def test_linear_bf16(m2, rows, n_in, n_out, norm, res):
    """The attention projections: q|k|v (with the block's pre-norm) and the
    output projection (with the residual add), 1 to 16 rows (1 to 8 per pass),
    output rows wider than the layer (y_stride)."""
    import oracle
    from oracle.lm import rb
    import torch
    rng = np.random.default_rng(520 + rows + n_in)
    x = _bf16(rng, (rows, n_in))
    W = _bf16(rng, (n_out, n_in), n_in ** -0.5)
    g = (1 + 0.1 * rng.standard_normal(n_in)).astype(np.float32)
    ys = n_out + 24
    y0 = _bf16(rng, (rows, ys))
    y = to_dev(y0)
    nm = m2.row_norm(m2.NORM_RMS, to_dev(g), 1e-5) if norm else None
    m2.mamba2_linear_bf16(rows, n_in, n_out, to_dev(x), n_in, nm, to_dev(W), y if res else None, y, ys)
    torch.cuda.synchronize()
    xv = bf16_bits_to_f64(x)
    if norm:
        xv = rb(oracle.rmsnorm(xv, g, 1e-5))
    ref = oracle.linear(xv, bf16_bits_to_f64(W))
    if res:
        ref = ref + bf16_bits_to_f64(y0[:, :n_out])
    out = from_dev_act(y, "bf16")
    if norm:  # the normalised row is stored in bf16 before the product
        check_y_rounded_inside(out[:, :n_out], ref)
    else:
        check_y(out[:, :n_out], ref, "bf16")
    # the columns past the layer's outputs are left alone
    np.testing.assert_array_equal(bits_of(y).view(np.uint16).reshape(rows, ys)[:, n_out:], y0[:, n_out:])


# ------------------------------------------------------- strided mixer calls
def _wide_rows(d, inp, S, T):
    """x, B, C, dt_raw of seeded mixer inputs placed in rows z | x | B | C | dt
    of width 2HP + 2GN + H (z random), as the in_proj output holds them."""
    HP, GN = d.H * d.P, d.G * d.N
    W = 2 * HP + 2 * GN + d.H
    rows = np.zeros((S, T, W), np.uint16)
    rows[..., :HP] = f32_to_bf16_bits(np.random.default_rng(530).standard_normal((S, T, HP)).astype(np.float32))
    rows[..., HP:2 * HP] = inp["x"].reshape(S, T, HP)
    rows[..., 2 * HP:2 * HP + GN] = inp["B"].reshape(S, T, GN)
    rows[..., 2 * HP + GN:2 * HP + 2 * GN] = inp["C"].reshape(S, T, GN)
    rows[..., 2 * HP + 2 * GN:] = inp["dt_raw"].reshape(S, T, d.H)
    return rows, W


@pytest.mark.parametrize("d,S", [(REAL_SHAPE, 3), (Dims(H=8, P=16, N=16, G=2), 5)])
def test_step_strided_equals_dense_step(m2, d, S):
    import torch
    inp = mixer_inputs(540, d, S, 1, "bf16")
    rows, W = _wide_rows(d, inp, S, 1)
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, "bf16")
    p = {k: to_dev(inp[k]) for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b")}
    ws = torch.empty(m2.mamba2_step_workspace_bytes(dims, S), dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(541)
    s0 = (0.1 * rng.standard_normal((S, d.H, d.P, d.N))).astype(np.float32)
    c0 = _bf16(rng, (S, d.K - 1, d.CH))
    outs = []
    for strided in (False, True):
        ssm, conv, y = to_dev(s0), to_dev(c0), act_empty((S, d.H, d.P), "bf16")
        if strided:
            r = to_dev(rows.reshape(S, W))
            HP, GN = d.H * d.P, d.G * d.N
            m2.mamba2_step_strided(dims, S, r[:, HP:], r[:, 2 * HP:], r[:, 2 * HP + GN:], r[:, 2 * HP + 2 * GN:], W,
                                   p["A_log"], p["D"], p["dt_bias"], p["conv_w"], p["conv_b"], ssm, conv, y, ws)
        else:
            f = {k: to_dev(np.ascontiguousarray(inp[k][:, 0])) for k in ("x", "B", "C", "dt_raw")}
            m2.mamba2_step(dims, S, f["x"], f["B"], f["C"], f["dt_raw"], p["A_log"], p["D"], p["dt_bias"],
                           p["conv_w"], p["conv_b"], ssm, conv, y, ws)
        torch.cuda.synchronize()
        outs.append([bits_of(t) for t in (y, ssm, conv)])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("d,S,T,chunk", [(REAL_SHAPE, 2, 150, 128), (Dims(H=8, P=16, N=16, G=2), 3, 70, 32)])
def test_conv_scan_strided_equals_dense_scan(m2, d, S, T, chunk):
    import torch
    inp = mixer_inputs(550, d, S, T, "bf16")
    rows, W = _wide_rows(d, inp, S, T)
    dims = m2.dims(S, T, d.H, d.P, d.N, d.G, d.K, "bf16")
    p = {k: to_dev(inp[k]) for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b")}
    ws = torch.empty(m2.mamba2_scan_workspace_bytes(dims, chunk), dtype=torch.uint8, device="cuda")
    outs = []
    for strided in (False, True):
        y = act_empty((S, T, d.H, d.P), "bf16")
        fs = torch.empty((S, d.H, d.P, d.N), dtype=torch.float32, device="cuda")
        fc = act_empty((S, d.K - 1, d.CH), "bf16")
        if strided:
            r = to_dev(rows.reshape(S * T, W))
            HP, GN = d.H * d.P, d.G * d.N
            m2.mamba2_conv_scan_strided(dims, r[:, HP:], r[:, 2 * HP:], r[:, 2 * HP + GN:], r[:, 2 * HP + 2 * GN:],
                                        W, p["A_log"], p["D"], p["dt_bias"], p["conv_w"], p["conv_b"], chunk, None,
                                        None, y, fs, fc, ws)
        else:
            f = {k: to_dev(inp[k]) for k in ("x", "B", "C", "dt_raw")}
            m2.mamba2_conv_scan(dims, f["x"], f["B"], f["C"], f["dt_raw"], p["A_log"], p["D"], p["dt_bias"],
                                p["conv_w"], p["conv_b"], chunk, None, None, y, fs, fc, ws)
        torch.cuda.synchronize()
        assert m2.mamba2_device_error() == 0
        outs.append([bits_of(t) for t in (y, fs, fc)])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------ model positions
def _dev(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).cuda()
    return to_dev(a)


def _host(t):
    """A device weight as the oracle's numpy layout (bf16 as bit patterns)."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.int32:
        return t.cpu().numpy().view(np.uint32)
    return t.cpu().numpy()


def _gpu_lm(m2, cfg, wdev, S, max_len):
    """The m2_lm of the blocks with zeroed caches for S sessions."""
    import torch
    d = cfg.mixer
    layers = []
    for i, kind in enumerate(cfg.kinds):
        L = dict(wdev[i])
        if kind == "M":
            L["ssm_state"] = torch.zeros((S, d.H, d.P, d.N), dtype=torch.float32, device="cuda")
            L["conv_state"] = torch.zeros((S, d.K - 1, d.CH), dtype=torch.bfloat16, device="cuda")
        else:
            shape = (S, cfg.n_kv_heads, max_len, cfg.head_dim)
            L["k_cache"] = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
            L["v_cache"] = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        layers.append(L)
    mixer = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, "bf16")
    model = m2.lm_model(cfg.kinds, layers, cfg.hidden, mixer, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, max_len,
                        cfg.eps)
    return model, layers


def _run_steps(m2, model, H, S, T, max_len, cfg):
    """Positions one at a time through mamba2_lm_step; returns [S, T, hidden]."""
    import torch
    ws = torch.empty(max(16, m2.mamba2_lm_workspace_bytes(model, S, 1, 1)), dtype=torch.uint8, device="cuda")
    lens = torch.zeros(S, dtype=torch.int32, device="cuda")
    outs = []
    for t in range(T):
        h = to_dev(np.ascontiguousarray(H[:, t]))
        m2.mamba2_lm_step(model, S, h, lens, ws)
        lens += 1
        outs.append(from_dev_act(h, "bf16"))
    torch.cuda.synchronize()
    assert m2.mamba2_device_error() == 0
    return np.stack(outs, axis=1)


def _run_prefill(m2, model, H, S, T, chunk):
    import torch
    ws = torch.empty(max(16, m2.mamba2_lm_workspace_bytes(model, S, T, chunk)), dtype=torch.uint8, device="cuda")
    lens = torch.zeros(S, dtype=torch.int32, device="cuda")
    h = to_dev(np.ascontiguousarray(H))
    m2.mamba2_lm_prefill(model, S, T, h, lens, chunk, ws)
    torch.cuda.synchronize()
    assert m2.mamba2_device_error() == 0
    return from_dev_act(h, "bf16")


def _gpu_block(m2, cfg, i, wdev_i, orc, h_in, max_len):
    """Block i alone on the GPU through mamba2_lm_step, started from the
    oracle's caches and the oracle's input h_in (teacher forcing). Returns
    (h out fp64, the block's device caches)."""
    import torch
    from seeded_inputs import f64_to_bf16_bits
    d, S = cfg.mixer, orc.S
    L = dict(wdev_i)
    if cfg.kinds[i] == "M":
        L["ssm_state"] = torch.from_numpy(orc.ssm[i].astype(np.float32)).cuda()
        L["conv_state"] = to_dev(f64_to_bf16_bits(orc.conv[i]))
    else:
        L["k_cache"] = to_dev(f64_to_bf16_bits(orc.kc[i]))
        L["v_cache"] = to_dev(f64_to_bf16_bits(orc.vc[i]))
    model = m2.lm_model(cfg.kinds[i], [L], cfg.hidden, m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, "bf16"), cfg.n_heads,
                        cfg.n_kv_heads, cfg.head_dim, max_len, cfg.eps)
    ws = torch.empty(max(16, m2.mamba2_lm_workspace_bytes(model, S, 1, 1)), dtype=torch.uint8, device="cuda")
    lens = torch.from_numpy(orc.lengths.copy()).cuda()
    h = to_dev(f64_to_bf16_bits(h_in))
    m2.mamba2_lm_step(model, S, h, lens, ws)
    torch.cuda.synchronize()
    assert m2.mamba2_device_error() == 0
    return from_dev_act(h, "bf16"), L


def _teacher_forced(m2, cfg, w_host, wdev, H, T, max_len, tag):
    """Every block of every position on the GPU from the oracle's own input
    and caches, against the oracle's block: the residual stream leaving the
    block and the caches it updated."""
    from m2_testlib import check_state, check_y_rounded_inside
    from oracle.lm import LMOracle
    S = H.shape[0]
    orc = LMOracle(cfg, w_host, S, max_len)
    for t in range(T):
        h = bf16_bits_to_f64(H[:, t])
        for i, kind in enumerate(cfg.kinds):
            got, L = _gpu_block(m2, cfg, i, wdev[i], orc, h, max_len)
            before = orc.ssm[i].copy() if kind == "M" else None
            h = orc.step_block(i, h)
            check_y_rounded_inside(got, h, tag=f"{tag} t{t} block{i}{kind}")
            if kind == "M":
                # The state gate of the mixer core (1e-4 of max|state|) plus the
                # in_proj rows' own rounding: a row element the GPU rounds one
                # ulp away from the oracle (2^-7 relative at most) moves this
                # step's increment dt x~ (outer) B~ by about as much; allow
                # 2^-6 of the largest change of the state over the step.
                ref = orc.ssm[i]
                gs = L["ssm_state"].cpu().numpy().astype(np.float64)
                step_change = float(np.max(np.abs(ref - before)))
                tol = 1e-4 + 2.0 ** -6 * step_change / float(np.max(np.abs(ref)))
                check_state(gs, ref, tag=f"{tag} t{t} block{i} state", tol=tol)
                check_y_rounded_inside(from_dev_act(L["conv_state"], "bf16"), orc.conv[i],
                                       tag=f"{tag} t{t} block{i} conv tail")
            else:
                slot = orc.lengths
                for c_dev, c_ref in ((L["k_cache"], orc.kc[i]), (L["v_cache"], orc.vc[i])):
                    got_c = from_dev_act(c_dev, "bf16")
                    for s in range(S):
                        check_y_rounded_inside(got_c[s, :, slot[s]], c_ref[s, :, slot[s]],
                                               tag=f"{tag} t{t} block{i} kv slot")
                        untouched = np.arange(max_len) != slot[s]
                        np.testing.assert_array_equal(got_c[s][:, untouched], c_ref[s][:, untouched])
        orc.lengths += 1


def test_lm_tiny_blocks_match_the_oracle(m2):
    """Six positions of two sessions through a small model of the same block
    structure (Mamba, Mamba, attention, ...): every block against the
    oracle's from identical inputs and caches, then whole positions (cached
    steps and the recompute) against the oracle's."""
    from m2_testlib import check_drift
    from oracle.lm import LMOracle
    cfg, S, T, max_len = TINY_LM, 2, 6, 16
    w = lm_weights(560, cfg)
    H = lm_hidden(561, cfg, S, T)
    wdev = [{k: _dev(v) for k, v in L.items()} for L in w]
    _teacher_forced(m2, cfg, w, wdev, H, T, max_len, "tiny")
    model, _ = _gpu_lm(m2, cfg, wdev, S, max_len)
    got = _run_steps(m2, model, H, S, T, max_len, cfg)
    orc = LMOracle(cfg, w, S, max_len)
    n = len(cfg.kinds)
    for t in range(T):
        check_drift(got[:, t], orc.step(H[:, t]), n, f"tiny step t{t}")
    model2, _ = _gpu_lm(m2, cfg, wdev, S, max_len)
    rec = _run_prefill(m2, model2, H, S, T, 4)
    check_drift(rec, LMOracle(cfg, w, S, max_len).prefill(H), n, "tiny prefill vs oracle")
    check_drift(got, rec, n, "tiny step vs prefill")


def test_lm_tiny_100_positions_stepping_equals_recompute(m2):
    """100 positions: the cached positions against the full-history
    recompute (chunked scan in every Mamba block), both on the GPU, and the
    recompute against the oracle's."""
    from m2_testlib import check_drift
    from oracle.lm import LMOracle
    cfg, S, T, max_len = TINY_LM, 2, 100, 128
    w = lm_weights(570, cfg)
    H = lm_hidden(571, cfg, S, T)
    wdev = [{k: _dev(v) for k, v in L.items()} for L in w]
    model, _ = _gpu_lm(m2, cfg, wdev, S, max_len)
    got = _run_steps(m2, model, H, S, T, max_len, cfg)
    model2, _ = _gpu_lm(m2, cfg, wdev, S, max_len)
    rec = _run_prefill(m2, model2, H, S, T, 32)
    n = len(cfg.kinds)
    for t in (0, 9, 99):
        check_drift(got[:, t], rec[:, t], n, f"tiny100 step vs prefill t{t}")
    ref = LMOracle(cfg, w, S, max_len).prefill(H)
    for t in (0, 9, 99):
        check_drift(rec[:, t], ref[:, t], n, f"tiny100 prefill vs oracle t{t}")


@pytest.mark.slow
def test_lm_real_shape_positions(m2):
    """The 27 Mamba + 4 attention blocks of Nemotron-H at full size, one
    session: every block of two positions against the oracle's from
    identical inputs and caches; whole positions against the oracle's; and
    100 positions of cached steps against the library's own full-history
    recompute."""
    import torch
    from m2_testlib import check_drift
    from oracle.lm import LMOracle
    cfg, S, max_len = REAL_LM, 1, 128
    n = len(cfg.kinds)
    wdev = device_lm_weights(580, cfg, "cuda")
    H = lm_hidden(581, cfg, S, 100)
    whost = [{k: _host(v) for k, v in L.items()} for L in wdev]
    _teacher_forced(m2, cfg, whost, wdev, H, 2, max_len, "real")
    model, _ = _gpu_lm(m2, cfg, wdev, S, max_len)
    got = _run_steps(m2, model, H, S, 100, max_len, cfg)
    orc = LMOracle(cfg, whost, S, max_len)
    for t in range(2):
        check_drift(got[:, t], orc.step(H[:, t]), n, f"real step t{t}")
    del whost, orc
    model2, _ = _gpu_lm(m2, cfg, wdev, S, max_len)
    rec = _run_prefill(m2, model2, H, S, 100, 128)
    for t in (0, 1, 49, 99):
        check_drift(got[:, t], rec[:, t], n, f"real step vs prefill t{t}")
    torch.cuda.synchronize()
