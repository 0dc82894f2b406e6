"""Parity at the full workload sizes of the mixer core, in the launch
configurations the benchmark uses, against the fp64 oracle:

* cached decode: one frame at a time through all 27 Mamba layers of the
  Nemotron-H pattern for 750 frames (60 s at 12.5 frames/s), batch 1, from
  zero state; at frames 1, 100 and 750 the step is compared with a chunked
  scan over the same frames and with the oracle ("docs/nemotron-voicechat.md",
  section Offline timeline: cached stepping and full-history recompute agree);
* 64 sessions, each carried to a random length of 50-500 frames by a GPU scan
  (checked against the oracle), then one cached step for all 64 at once;
* long prefill: batch 4, T=4096, all 27 layers back to back: every layer's
  conv tail bit for bit and its whole final state against a recompute of the
  same layer with chunks of 64; on layers 0, 13 and 26 two heads' y and final
  state against the oracle.
"""
import numpy as np
import pytest

from m2_testlib import Y_TOL, act_empty, bits_of, check_scan_y, check_state, check_y, from_dev_act, to_dev
from seeded_inputs import MAMBA_LAYERS, REAL_SHAPE, device_mixer_inputs, mixer_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def m2():
    import full_duplex_speech_gb300 as m2
    m2.load()
    return m2


def _dev_inputs(inp):
    return {k: to_dev(inp[k]) for k in ("x", "B", "C", "dt_raw", "A_log", "D", "dt_bias", "conv_w", "conv_b")}


def _scan(m2, d, dv, b, T, chunk=128):
    import torch
    dims = m2.dims(b, T, d.H, d.P, d.N, d.G, d.K, "bf16")
    y = act_empty((b, T, d.H, d.P), "bf16")
    fs = torch.empty((b, d.H, d.P, d.N), dtype=torch.float32, device="cuda")
    fc = act_empty((b, d.K - 1, d.CH), "bf16")
    ws = torch.empty(max(m2.mamba2_scan_workspace_bytes(dims, chunk), 16), dtype=torch.uint8, device="cuda")
    m2.mamba2_conv_scan(dims, dv["x"], dv["B"], dv["C"], dv["dt_raw"], dv["A_log"], dv["D"], dv["dt_bias"],
                        dv["conv_w"], dv["conv_b"], chunk, None, None, y, fs, fc, ws)
    return y, fs, fc


def test_cached_decode_27_layers_750_frames(m2):
    import torch
    import oracle
    d, T = REAL_SHAPE, 750
    checks = (1, 100, 750)
    dims = m2.dims(1, T, d.H, d.P, d.N, d.G, d.K, "bf16")
    ws = torch.empty(m2.mamba2_step_workspace_bytes(dims, 1), dtype=torch.uint8, device="cuda")
    for li, layer in enumerate(MAMBA_LAYERS):
        inp = mixer_inputs(2000 + layer, d, 1, T, "bf16")
        dv = _dev_inputs(inp)
        ssm = torch.zeros((1, d.H, d.P, d.N), dtype=torch.float32, device="cuda")
        conv = act_empty((1, d.K - 1, d.CH), "bf16").zero_()
        ys, states = {}, {}
        y1 = act_empty((1, d.H, d.P), "bf16")
        for t in range(T):
            m2.mamba2_step(dims, 1, dv["x"][:, t], dv["B"][:, t], dv["C"][:, t], dv["dt_raw"][:, t],
                           dv["A_log"], dv["D"], dv["dt_bias"], dv["conv_w"], dv["conv_b"], ssm, conv, y1, ws)
            if t + 1 in checks:
                ys[t + 1] = from_dev_act(y1, "bf16")
                states[t + 1] = ssm.cpu().numpy().copy()
        torch.cuda.synchronize()
        ref = oracle.mixer_scan(d, inp)
        ybar = oracle.mixer_scan_magnitude(d, inp)  # row n-1 is also that of a scan over n frames
        for n in checks:
            # the step against the oracle's recompute of the first n frames
            check_y(ys[n], ref["y"][:, n - 1], "bf16", tag=f"step L{layer} n{n}")
            if n == T:
                check_state(states[n], ref["final_ssm"], tag=f"step state L{layer}")
            # the step against the GPU's own chunked recompute of the first n frames
            sub = {k: v[:, :n].contiguous() if k in ("x", "B", "C", "dt_raw") else v for k, v in dv.items()}
            ysc, fs, _ = _scan(m2, d, sub, 1, n)
            torch.cuda.synchronize()
            ylast = from_dev_act(ysc[:, n - 1], "bf16")
            check_scan_y(ylast, ref["y"][:, n - 1], ybar[:, n - 1], "bf16", tag=f"scan L{layer} n{n}")
            assert np.linalg.norm(ys[n] - ylast) / np.linalg.norm(ylast) <= Y_TOL, (layer, n)
            check_state(states[n], fs.cpu().numpy().astype(np.float64), tag=f"step vs scan state L{layer} n{n}")
        np.testing.assert_array_equal(
            bits_of(conv), np.ascontiguousarray(np.concatenate(
                [inp["x"].reshape(1, T, -1), inp["B"].reshape(1, T, -1), inp["C"].reshape(1, T, -1)],
                axis=2)[:, -3:]).view(np.uint8).reshape(-1))


def test_64_sessions_from_scanned_states(m2):
    import torch
    import oracle
    d, S = REAL_SHAPE, 64
    lengths = np.random.default_rng(3).integers(50, 501, size=S)
    params_seed = 3000
    base = mixer_inputs(params_seed, d, 1, 1, "bf16")  # the layer's weights (shared by the sessions)
    pd = {k: to_dev(base[k]) for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b")}
    ssm = torch.empty((S, d.H, d.P, d.N), dtype=torch.float32, device="cuda")
    conv = act_empty((S, d.K - 1, d.CH), "bf16")
    ref_ssm = np.zeros((S, d.H, d.P, d.N))
    ref_conv = np.zeros((S, d.K - 1, d.CH))
    frames = []
    for s in range(S):
        T = int(lengths[s])
        act = mixer_inputs(3100 + s, d, 1, T + 1, "bf16")
        seq = dict(base, **{k: np.ascontiguousarray(act[k][:, :T]) for k in ("x", "B", "C", "dt_raw")})
        frames.append({k: np.ascontiguousarray(act[k][:, T]) for k in ("x", "B", "C", "dt_raw")})
        dv = dict(pd, **{k: to_dev(seq[k]) for k in ("x", "B", "C", "dt_raw")})
        y, fs, fc = _scan(m2, d, dv, 1, T)
        ssm[s].copy_(fs[0])
        conv[s].copy_(fc[0])
        r = oracle.mixer_scan(d, seq)
        ref_ssm[s], ref_conv[s] = r["final_ssm"][0], r["final_conv"][0]
        if s % 16 == 0:  # the prefix scans themselves, on a sample of sessions
            check_scan_y(from_dev_act(y, "bf16"), r["y"], oracle.mixer_scan_magnitude(d, seq), "bf16",
                         tag=f"prefix scan {s}")
            check_state(fs.cpu().numpy(), r["final_ssm"], tag=f"prefix state {s}")
    torch.cuda.synchronize()
    check_state(ssm.cpu().numpy(), ref_ssm, tag="scanned states")
    fr = {k: np.concatenate([f[k] for f in frames], axis=0) for k in ("x", "B", "C", "dt_raw")}
    fd = {k: to_dev(v) for k, v in fr.items()}
    dims = m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, "bf16")
    ws = torch.empty(m2.mamba2_step_workspace_bytes(dims, S), dtype=torch.uint8, device="cuda")
    y1 = act_empty((S, d.H, d.P), "bf16")
    m2.mamba2_step(dims, S, fd["x"], fd["B"], fd["C"], fd["dt_raw"], pd["A_log"], pd["D"], pd["dt_bias"],
                   pd["conv_w"], pd["conv_b"], ssm, conv, y1, ws)
    torch.cuda.synchronize()
    # the oracle's step continues from the oracle's own scanned states
    fr["act"] = "bf16"
    y_ref = oracle.mixer_step(d, fr, base, ref_ssm, ref_conv)
    check_y(from_dev_act(y1, "bf16"), y_ref, "bf16", tag="64-session step")
    check_state(ssm.cpu().numpy(), ref_ssm, tag="64-session state")


def test_long_prefill_27_layers_b4_T4096(m2):
    import torch
    import oracle
    from seeded_inputs import bf16_bits_to_f64
    d, b, T = REAL_SHAPE, 4, 4096
    sample_layers = {0, 13, 26}
    for li in range(len(MAMBA_LAYERS)):
        dv = device_mixer_inputs(4000 + li, d, b, T, "cuda")
        y, fs, fc = _scan(m2, d, dv, b, T)
        torch.cuda.synchronize()
        # conv tail: the last three input frames, bit for bit (every layer)
        tail = torch.cat([dv["x"][:, -3:].reshape(b, 3, -1), dv["B"][:, -3:].reshape(b, 3, -1),
                          dv["C"][:, -3:].reshape(b, 3, -1)], dim=2)
        assert torch.equal(fc.view(torch.int16), tail.contiguous().view(torch.int16))
        # every head's final state against the GPU's own recompute with chunks
        # of 64 (the chunked form does not depend on the chunk length)
        _, fs64, _ = _scan(m2, d, dv, b, T, chunk=64)
        torch.cuda.synchronize()
        check_state(fs.cpu().numpy(), fs64.cpu().numpy().astype(np.float64), tag=f"prefill Q128 vs Q64 L{li}")
        del fs64
        if li not in sample_layers:
            continue
        heads = (16 * (li % 8) + 3, 16 * (li % 8) + 5)  # two heads of one group
        g = heads[0] // (d.H // d.G)

        def host(t):
            t = t.contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).cpu().numpy().view(np.uint16)
            return t.cpu().numpy()

        # the oracle needs only these heads' x channels and their group's B, C
        inp = {k: host(dv[k]) for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b")}
        xs = torch.zeros_like(dv["x"])
        xs[:, :, heads[0]:heads[1]] = dv["x"][:, :, heads[0]:heads[1]]
        inp["x"] = host(xs)
        bs = torch.zeros_like(dv["B"])
        cs = torch.zeros_like(dv["C"])
        bs[:, :, g] = dv["B"][:, :, g]
        cs[:, :, g] = dv["C"][:, :, g]
        inp["B"], inp["C"], inp["dt_raw"] = host(bs), host(cs), host(dv["dt_raw"])
        inp["act"] = "bf16"
        del xs, bs, cs
        ref = oracle.mixer_scan(d, inp, heads=heads)
        yh = y[:, :, heads[0]:heads[1]].contiguous()
        yg = bf16_bits_to_f64(host(yh))
        ybar = oracle.mixer_scan_magnitude(d, inp, heads=heads)
        check_scan_y(yg, ref["y"][:, :, heads[0]:heads[1]], ybar[:, :, heads[0]:heads[1]], "bf16",
                     tag=f"prefill y L{li}")
        check_state(fs[:, heads[0]:heads[1]].cpu().numpy(), ref["final_ssm"][:, heads[0]:heads[1]],
                    tag=f"prefill state L{li}")
        del dv, y, fs, fc
        torch.cuda.empty_cache()
