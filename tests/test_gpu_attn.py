"""GPU parity of the cached decode position of the hybrid model's
grouped-query attention layers (mamba2_attn_decode) against the fp64 oracle,
through the C ABI: the Nemotron-H attention layers (40 query heads, 8 kv
heads, head_dim 128; VoiceChat issue, section config.json / text_config) and
their KV caches ("docs/nemotron-voicechat.md", section Online session).

Tolerances: a bf16 output is held to the library's gates for bf16 results
(normwise 2e-3 against the oracle rounded to bf16, at most 0.1% of its
elements more than one bf16 ulp from it, none beyond 4 ulp + 1e-3 max|ref|);
an fp32 output to normwise and max-normwise 1e-5 (fp32 dot products of 128
terms and sums over at most a few thousand positions: about 1e-6). The caches must change in exactly
one slot per session and kv head, to the new key's and value's bits."""
import math

import numpy as np
import pytest

from m2_testlib import act_empty, bits_of, check_y, from_dev_act, to_dev
from seeded_inputs import attn_inputs, bf16_bits_to_f64

pytestmark = pytest.mark.gpu

HQ, HKV, D = 40, 8, 128
F32_TOL = 1e-5


@pytest.fixture(scope="module")
def m2():
    import full_duplex_speech_gb300 as m2
    m2.load()
    return m2


def _f64(a, act):
    return bf16_bits_to_f64(a) if act == "bf16" else np.asarray(a, np.float64)


def _run(m2, inp, Hq, Hkv, Tmax, scale, dev=None):
    """One position on the GPU; returns (out fp64, k_cache, v_cache device tensors)."""
    import torch
    act, S = inp["act"], inp["q"].shape[0]
    dev = dev or {k: to_dev(inp[k]) for k in ("q", "k_new", "v_new", "k_cache", "v_cache")}
    lens = torch.from_numpy(inp["lengths"]).cuda()
    out = act_empty((S, Hq, D), act)
    ws = torch.empty(max(1, m2.mamba2_attn_decode_workspace_bytes(S, Hq, Hkv, D, Tmax, act)), dtype=torch.uint8,
                     device="cuda")
    m2.mamba2_attn_decode(S, Hq, Hkv, D, Tmax, act, lens, dev["q"], dev["k_new"], dev["v_new"], dev["k_cache"],
                          dev["v_cache"], scale, out, ws)
    torch.cuda.synchronize()
    return from_dev_act(out, act), dev


def _oracle(inp, scale):
    import oracle
    act = inp["act"]
    kc, vc = _f64(inp["k_cache"], act).copy(), _f64(inp["v_cache"], act).copy()
    out = oracle.attn_decode(_f64(inp["q"], act), _f64(inp["k_new"], act), _f64(inp["v_new"], act), kc, vc,
                             inp["lengths"], scale)
    return out, kc, vc


def _check(out, ref, act):
    if act == "bf16":
        check_y(out, ref, act)
    else:
        check_y(out, ref, act, l2_tol=F32_TOL, f32_maxnorm=F32_TOL)


def _expected_cache_bits(cache, new, lengths):
    c = np.array(cache, copy=True)
    for s, L in enumerate(lengths):
        c[s, :, L] = new[s]
    return np.ascontiguousarray(c).view(np.uint8).reshape(-1)


@pytest.mark.parametrize("act,lengths", [
    ("bf16", [0, 1, 63, 64, 65, 127, 128, 299]),  # chunk edges (64 positions here), ragged tails
    ("f32", [0, 31, 32, 33, 200, 299]),           # chunks of 32 here in fp32
])
def test_attn_decode_chunk_edges_real_heads(m2, act, lengths):
    S, Tmax = len(lengths), 300
    inp = attn_inputs(301, S, HQ, HKV, D, Tmax, lengths, act)
    scale = 1.0 / math.sqrt(D)
    out, dev = _run(m2, inp, HQ, HKV, Tmax, scale)
    ref, _, _ = _oracle(inp, scale)
    _check(out, ref, act)
    np.testing.assert_array_equal(bits_of(dev["k_cache"]), _expected_cache_bits(inp["k_cache"], inp["k_new"], lengths))
    np.testing.assert_array_equal(bits_of(dev["v_cache"]), _expected_cache_bits(inp["v_cache"], inp["v_new"], lengths))


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (4, 2), (16, 2), (6, 3)])
def test_attn_decode_group_sizes(m2, Hq, Hkv):
    """1, 2, 8 and 2 query heads per kv head (the model has 5)."""
    lengths = [40, 130, 0]
    inp = attn_inputs(302, 3, Hq, Hkv, D, 160, lengths, "bf16")
    out, _ = _run(m2, inp, Hq, Hkv, 160, 0.09)
    ref, _, _ = _oracle(inp, 0.09)
    _check(out, ref, "bf16")


def test_attn_decode_longest_cache(m2):
    """One session at the 600 s session limit: 7500 frames, the last slot."""
    Tmax = 7500
    inp = attn_inputs(303, 1, HQ, HKV, D, Tmax, [Tmax - 1], "bf16")
    scale = 1.0 / math.sqrt(D)
    out, _ = _run(m2, inp, HQ, HKV, Tmax, scale)
    ref, _, _ = _oracle(inp, scale)
    _check(out, ref, "bf16")


@pytest.mark.parametrize("Hq,Hkv,Tmax,length", [
    (40, 8, 750, 749),    # one session at 60 s: clusters of 8 walkers, 2 chunks each
    (16, 2, 2000, 1999),  # 8 query heads per kv head, clusters of 16 walkers: every walker owns a head
    (40, 8, 1500, 700),   # a length well inside the cache: the walkers past it hold no positions
])
def test_attn_decode_one_session_clusters(m2, Hq, Hkv, Tmax, length):
    """One session, where the walkers of a kv head form a thread-block cluster
    and merge through distributed shared memory."""
    inp = attn_inputs(308, 1, Hq, Hkv, D, Tmax, [length], "bf16")
    scale = 1.0 / math.sqrt(D)
    out, dev = _run(m2, inp, Hq, Hkv, Tmax, scale)
    ref, _, _ = _oracle(inp, scale)
    _check(out, ref, "bf16")
    np.testing.assert_array_equal(bits_of(dev["k_cache"]), _expected_cache_bits(inp["k_cache"], inp["k_new"], [length]))


def test_attn_decode_many_sessions(m2):
    """64 sessions with lengths drawn in [0, 750) (60 s of frames)."""
    S, Tmax = 64, 750
    lengths = np.random.default_rng(304).integers(0, Tmax, size=S)
    inp = attn_inputs(305, S, HQ, HKV, D, Tmax, lengths, "bf16")
    scale = 1.0 / math.sqrt(D)
    out, _ = _run(m2, inp, HQ, HKV, Tmax, scale)
    ref, _, _ = _oracle(inp, scale)
    _check(out, ref, "bf16")


def test_attn_decode_consecutive_positions(m2):
    """Six positions in a row from an empty cache, the lengths advanced by
    the caller: each output and the final caches against the oracle run the
    same way."""
    import oracle
    S, Tmax, scale = 2, 16, 0.1
    base = attn_inputs(306, S, HQ, HKV, D, Tmax, [0, 0], "bf16")
    dev = {k: to_dev(base[k]) for k in ("k_cache", "v_cache")}
    kc, vc = _f64(base["k_cache"], "bf16").copy(), _f64(base["v_cache"], "bf16").copy()
    for t in range(6):
        step = attn_inputs(400 + t, S, HQ, HKV, D, 1, [t, t], "bf16")
        inp = dict(step, k_cache=base["k_cache"], v_cache=base["v_cache"], lengths=np.array([t, t], np.int32))
        d = dict(dev, **{k: to_dev(step[k]) for k in ("q", "k_new", "v_new")})
        out, _ = _run(m2, inp, HQ, HKV, Tmax, scale, dev=d)
        ref = oracle.attn_decode(_f64(step["q"], "bf16"), _f64(step["k_new"], "bf16"), _f64(step["v_new"], "bf16"),
                                 kc, vc, [t, t], scale)
        _check(out, ref, "bf16")
    got_k = from_dev_act(dev["k_cache"], "bf16")
    np.testing.assert_array_equal(got_k, kc)
    np.testing.assert_array_equal(from_dev_act(dev["v_cache"], "bf16"), vc)


@pytest.mark.parametrize("Tmax", [64, 300])
def test_attn_decode_refuses_a_length_past_the_cache(m2, Tmax):
    """A length the host cannot see is checked on the device: that session
    gets zeros and untouched caches, the error word reads 0x104, and the
    other sessions are computed as usual (one walker per session and kv head
    at 64 positions; a cluster of 4 walkers at 300)."""
    m2.mamba2_device_error(None)  # start from a clear error word
    inp = attn_inputs(307, 2, HQ, HKV, D, Tmax, [10, Tmax], "bf16")
    out, dev = _run(m2, inp, HQ, HKV, Tmax, 0.1)
    code = m2.mamba2_device_error(None)
    assert code == 0x104
    assert np.all(out[1] == 0.0)
    k_bits = bits_of(dev["k_cache"]).reshape(2, -1)
    np.testing.assert_array_equal(k_bits[1], np.ascontiguousarray(inp["k_cache"][1]).view(np.uint8).reshape(-1))
    ok = dict(inp, q=inp["q"][:1], k_new=inp["k_new"][:1], v_new=inp["v_new"][:1], k_cache=inp["k_cache"][:1],
              v_cache=inp["v_cache"][:1], lengths=inp["lengths"][:1])
    ref, _, _ = _oracle(ok, 0.1)
    _check(out[:1], ref, "bf16")
    assert m2.mamba2_device_error(None) == 0
