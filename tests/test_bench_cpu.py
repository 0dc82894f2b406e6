"""The reference arm of bench.py (the fp64 oracle on the host cores) keeps
the JSON contract: one line with the metric, the throughput, the timing
fields, a cpu_baseline describing the run and an e2e block without copies."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config"):
        assert k in d, k
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def _bench():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    return bench


def test_scan_unit_counts():
    """The scan's algorithmic units per token at the real shape (H=128, P=80,
    N=128, G=8, K=4): bytes read x|B|C (12,288 bf16 channels) and dt (128 bf16)
    and written y (10,240 bf16); MMA flops of the chunked form with the two
    chunk x chunk products counted over their causal half."""
    b = _bench()
    assert b.SCAN_BYTES_PER_TOKEN == 12288 * 2 + 128 * 2 + 10240 * 2 == 45312
    # per token, chunk Q: C.B^T 2*Q*N per group and M.x 2*Q*P per head, halved
    # (causal); the chunk state B^T(w x) and C.h_prev 2*N*P per head each, in full
    for q, want in ((128, 6684672), (64, 5963776)):
        cb = 2 * q * 128 * 8 // 2
        mx = 2 * q * 80 * 128 // 2
        state = 2 * 128 * 80 * 128
        ch = 2 * 128 * 80 * 128
        assert cb + mx + state + ch == want
        assert b.scan_flops_per_token(q) == want
    # one launch of the 300-frame scan
    assert b.SCAN_FLOPS_PER_TOKEN * b.T_FRAMES == 2005401600
    assert b.STATE_BYTES == 5242880 and b.TAIL_BYTES == 73728


def test_step_unit_counts():
    """One cached frame of one session and layer: the fp32 state read and
    written (2 x 5,242,880 B), the conv tail read and written (2 x 3 x 12,288
    bf16), the frame's x|B|C|dt in (12,416 bf16) and y out (10,240 bf16)."""
    b = _bench()
    assert b.STEP_BYTES_PER_SESSION == 2 * 5242880 + 2 * 73728 + 12416 * 2 + 10240 * 2 == 10678528


def test_lm_position_unit_count():
    """The cached position of the 27 Mamba and 4 attention blocks at 750 cached
    positions, summed here block by block from the layer sizes."""
    b = _bench()
    from seeded_inputs import REAL_LM
    assert REAL_LM.kinds.count("M") == 27 and REAL_LM.kinds.count("*") == 4
    mamba = (22656 * 4480 // 2 + 22656 * 70 * 2 * 2      # in_proj: 4-bit fields, bf16 scale and bias per group
             + 4480 * 10240 // 2 + 4480 * 160 * 2 * 2     # out_proj
             + 2 * 5242880 + 2 * 3 * 12288 * 2)           # state and conv tail, read and written
    attn = ((40 + 2 * 8) * 128 * 4480 * 2 + 4480 * 40 * 128 * 2   # bf16 q|k|v and output projections
            + 750 * 8 * 128 * 2 * 2 + 8 * 128 * 2 * 2)            # cached keys and values read, new ones written
    residual = 31 * 4480 * 2 * 2
    assert b.lm_position_bytes(REAL_LM, 1, 750) == 27 * mamba + 4 * attn + residual == 2978602496


def test_reference_arm_under_two_ranks():
    """Launched as the driver launches it for N > 1 (torchrun, one process per
    rank; gloo on a host without GPUs): rank 0 alone runs the oracle and
    prints the one JSON line, the other rank exits 0 without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.lstrip().startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
