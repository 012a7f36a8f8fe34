"""bench.py without a GPU: the reference arm's JSON line (the oracle timed on the host cores) and
the algorithmic byte and FLOP counts the roofline fractions divide by."""
import json
import os
import subprocess
import sys

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["unit"] == "Mtok/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] >= 3 and d["ms_per_step"] > 0
    assert d["vs_baseline"] is None and d["data"] == "synthetic" and d["dtype"] == "f64"
    assert d["config"]["workload"].startswith("prefill B=1 H=8 T=1048576")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "Mtok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_algorithmic_counts():
    # per token-head at d = 128, bf16: q, k, z, v read, beta read, out written; the chunk form's FLOPs
    assert bench.prefill_bytes_per_token_head(128, 128, 2) == 1284
    assert bench.prefill_flops_per_token_head(128, 128) == 118784
    assert bench.prefill_flops_per_token_head(32, 32) == 11264
    # decode: the fp32 state read and written, one token's inputs and output
    assert bench.decode_bytes_per_head(128, 128, 2) == 132356
    # replay round on 256 sequences x 32 heads with a 7-token window
    N, H, d, L = 256, 32, 128, 7
    verify = bench.replay_bytes(N, H, d, d, N * L, N * L, 0)
    assert verify == N * H * d * d * 4 + N * L * H * (4 * d * 2 + 4) + N * L * H * d * 2 + N * 4 == 610501632
    commit = bench.replay_bytes(N, H, d, d, 1000, 0, N)
    assert commit == 2 * N * H * d * d * 4 + 1000 * H * (4 * d * 2 + 4) + N * 4


def test_ncu_traffic_follows_the_source_hash():
    """A committed DRAM-traffic figure is reported only while its kernel source is unchanged."""
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        recorded = json.load(f)
    for kernel, entry in recorded.items():
        if bench.src_sha(kernel) == entry["source_sha"]:
            assert bench.ncu_traffic(kernel) == entry["dram_bytes_per_launch"]
        else:
            assert bench.ncu_traffic(kernel) is None
    assert bench.ncu_traffic("no_such_kernel") is None


def test_oracle_sample_layout_gives_every_thread_the_same_units():
    """The oracle sampler's (heads, value-column block) choice makes the parallel units a whole
    multiple of the threads, so the reference arm and the cpu_baseline leg time the same work."""
    for H, dv, nt in ((8, 128, 16), (16, 128, 16), (8, 128, 1), (32, 128, 72), (2, 32, 16), (8, 128, 12)):
        h, cb = bench.oracle_layout(H, dv, nt)
        assert 1 <= h <= H and 1 <= cb <= dv and dv % cb == 0
        assert (h * (dv // cb)) % nt == 0, (H, dv, nt, h, cb)
    assert bench.oracle_layout(8, 128, 16) == (8, 64)
    assert bench.oracle_layout(8, 128, 1) == (1, 128)


def test_backward_bytes():
    # read q, k, z, v, beta, dO; write dq, dk, dz, dv, dbeta (bf16 tensors, fp32 beta)
    assert bench.backward_bytes_per_token_head(128, 128, 2) == 2 * (4 * 128 * 2 + 4) + 128 * 2 == 2312
