"""Benchmark: KDA chunked prefill (B=1, H=16, T=4096, d_k=d_v=128, bf16 inputs, fp32 state) and
the decode step (256 sequences x 32 heads, d=128, 512 MiB fp32 state), on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line.  `value` is prefill throughput in million tokens per second (tokens of all
16 heads) with inputs resident in HBM, timed with CUDA events on the launching stream; L2 is
flushed (a 512 MiB write) before every timed step because the workload's 86 MB fit in L2.
`decode` reports the decode step's state bandwidth, and under `replay` the speculative-decode round
(verify a 7-token drafted window from the snapshot, then commit the accepted prefix in place);
`layer` times the layer prologue and epilogue kernels at the prefill shape.  `e2e` repeats the prefill through the same
public call with pinned host buffers, host<->device copies inside the timed region.  `roofline`
is for the kernel with the largest device time, measured live with per-launch CUDA events.
`cpu_baseline` times the fp64 oracle on the host cores on a bounded sample of the same workload.

Under torchrun (N > 1) every rank runs its own copy of the workload (weak scaling, no collective
on the data path); the step time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill Mtok/s & % BF16 tensor peak; decode-step state GB/s & % HBM"
WORKLOAD = 1        # B=1, H=16, T=4096, d=128 bf16 prefill
DECODE_WORKLOAD = 4  # 256 x 32 heads decode
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def prefill_bytes_per_token_head(dk, dv, io_bytes):
    """Minimum HBM bytes per token-head: read q, k, z (d_k each), v (d_v), beta (fp32); write out."""
    return (3 * dk + dv) * io_bytes + 4 + dv * io_bytes


def prefill_flops_per_token_head(dk, dv, C=16):
    """Dense matmul FLOPs per token-head of the chunk form (W S, Q S, K^T U at d_k x d_v, and the
    C x C tiles A = K K^T, P = Q K^T, T applied to K and V, P U)."""
    return 6 * dk * dv + 2 * C * (3 * dk + 2 * dv)


def decode_bytes_per_head(dk, dv, io_bytes):
    return 2 * dk * dv * 4 + (3 * dk + dv) * io_bytes + 4 + dv * io_bytes


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if gpu_id is not None:
            cmd += ["-i", str(gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.split(",") for r in f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.file.name)
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def src_sha(kernel):
    name = {"kda_gate": "kda_gate.cu", "kda_ut_wy": "kda_ut_wy.cu", "kda_chunk_fwd": "kda_chunk_fwd.cu",
            "kda_decode_step": "kda_decode.cu", "kda_decode_replay_verify": "kda_replay.cu",
            "kda_decode_replay_commit": "kda_replay.cu", "kda_prologue": "kda_layer.cu",
            "kda_epilogue": "kda_layer.cu",
            "kda_chunk_fwd_tc": "kda_chunk_tc.cu",
            "kda_seg_summary_tc": "kda_chunk_tc.cu", "kda_seg_scan": "kda_segment_scan.cu",
            "kda_chunk_prep_tc": "kda_prep_tc.cu", "kda_state_summary_tc": "kda_state_tc.cu",
            "kda_chunk_state_tc": "kda_state_tc.cu"}.get(kernel)
    if name is None:
        return None
    p = os.path.join(ROOT, "linear_attention_recurrence_kda_gb300", "csrc", name)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16] if os.path.exists(p) else None


def ncu_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("source_sha") != src_sha(kernel):
        return None
    return d.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- CPU oracle leg

def oracle_rate(inp, target_s=10.0, threads=0):
    """fp64 oracle throughput on a bounded prefix sample of the workload: heads [0, h) over the
    first t tokens, sized from a short calibration run to take about `target_s` seconds."""
    import numpy as np  # noqa: F401
    import oracle
    T = inp["q"].shape[0]
    H = inp["q"].shape[1]

    def run(h, t):
        sl = lambda x: x[:t, :h]
        t0 = time.perf_counter()
        oracle.forward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["z"]), inp["A"][:h], sl(inp["beta"]),
                       S0=None if inp["S0"] is None else inp["S0"][:, :h], threads=threads)
        return time.perf_counter() - t0

    cal_t = min(T, 256)
    dt = run(1, cal_t)
    per_th = dt / cal_t
    budget = max(1, int(target_s / per_th))
    h = max(1, min(H, budget // T))
    t = T if budget >= T else max(16, budget)
    el = run(h, t)
    reps = 1
    if h == H and t == T and el < target_s:
        # the whole workload is quicker than the target: repeat it for a stable time
        reps = max(1, min(200, int(target_s / max(el, 1e-3))))
        el = sum(run(h, t) for _ in range(reps))
    th_per_s = reps * h * t / el
    return {"token_heads_per_s": th_per_s, "tok_per_s": th_per_s / H, "heads": h, "tokens": t, "seconds": el,
            "reps": reps}


def reference_arm(args):
    """The fp64 oracle as the reference implementation, on the host cores, same metric/config."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import torch
    from linear_attention_recurrence_kda_gb300 import inputs as I
    import oracle
    oracle.build()
    inp = I.make_inputs(WORKLOAD)
    H = inp["q"].shape[1]
    T = inp["q"].shape[0]
    cores = oracle.max_threads()
    # per step: a prefix of head 0 sized to ~0.25 s so that warm-up + steps stay within minutes
    cal = oracle_rate(inp, target_s=0.25)
    h, t = cal["heads"], cal["tokens"]
    sl = lambda x: x[:t, :h]

    def step():
        oracle.forward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["z"]), inp["A"][:h], sl(inp["beta"]),
                       S0=inp["S0"][:, :h])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    mtok = h * t / (el / args.steps) / H / 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": mtok, "unit": "Mtok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": I.WORKLOADS[WORKLOAD].name, "B": 1, "H": H, "T": T, "d_k": 128, "d_v": 128},
        "cpu_baseline": {"value": mtok, "unit": "Mtok/s", "cores": cores, "kind": "oracle",
                         "sample": f"heads [0,{h}) x first {t} tokens of the workload per step (fp64, OpenMP)"},
        "e2e": {"value": mtok, "unit": "Mtok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-steps", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-replay", action="store_true", help="skip the speculative-decode replay leg")
    ap.add_argument("--no-layer", action="store_true", help="skip the layer prologue / epilogue leg")
    ap.add_argument("--no-shapes", action="store_true", help="skip the varlen and long-context prefill shapes")
    args = ap.parse_args()
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import torch.distributed as dist
    import __graft_entry__
    __graft_entry__.build()
    from linear_attention_recurrence_kda_gb300 import binding as B
    from linear_attention_recurrence_kda_gb300 import inputs as I
    from linear_attention_recurrence_kda_gb300 import sharding

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(x):
        return sharding.max_over_ranks(x, device=dev)

    # ---- CPU oracle baseline first (rank 0 only, before any timed GPU work)
    cpu = None
    inp = I.make_inputs(WORKLOAD, seed=I.WORKLOADS[WORKLOAD].seed + rank)
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        r = oracle_rate(inp, target_s=12.0)
        cpu = {"value": r["tok_per_s"] / 1e6, "unit": "Mtok/s", "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"heads [0,{r['heads']}) x first {r['tokens']} tokens of the workload"
                         f"{' x ' + str(r['reps']) + ' repetitions' if r['reps'] > 1 else ''}, fp64, "
                         f"{r['seconds']:.1f} s; scaled to tokens of all {inp['q'].shape[1]} heads"}

    T, H, dk = inp["k"].shape
    dv = inp["v"].shape[2]
    io_bytes = inp["k"].element_size()
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}
    out = torch.empty(T, H, dv, dtype=inp["k"].dtype, device=dev)
    fin = torch.empty(1, H, dk, dv, dtype=torch.float32, device=dev)
    prob = B.make_problem(1, T, T, H, dk, dv, inp["k"].dtype)
    ws = torch.empty(B.kda_forward_workspace_bytes(prob), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def fwd():
        B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"], out=out,
                      final_state=fin, workspace=ws)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        fwd()
    torch.cuda.synchronize()

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_id) if rank == 0 else None
    time.sleep(0.3)

    # ---- timed prefill: K steps, L2 flushed before each, per-step events on the launching stream
    barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        fwd()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms = max_over_ranks(sum(step_ms) / len(step_ms))
    srt = sorted(step_ms)
    step_stats = {"median_ms": max_over_ranks(srt[len(srt) // 2]),
                  "p90_ms": max_over_ranks(srt[min(len(srt) - 1, int(0.9 * len(srt)))])}
    # the same steps with the inputs left in L2 (no flush between steps)
    barrier()
    torch.cuda.synchronize()
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(args.steps):
        fwd()
    w1.record(stream)
    torch.cuda.synchronize()
    warm_ms = max_over_ranks(w0.elapsed_time(w1) / args.steps)
    step_stats.update({"warm_l2_ms_per_step": warm_ms, "warm_l2_value": T * world / (warm_ms * 1e-3) / 1e6})
    tokens = T * world
    value = tokens / (ms * 1e-3) / 1e6

    # ---- the same K steps again with the library's per-kernel event hooks on (they sit between the
    # kernels of a step and stop one kernel's launch from overlapping the previous one's tail, so the
    # step time above is taken without them)
    B.kda_profile_enable(True)
    for i in range(args.steps):
        flush.zero_()
        fwd()
    torch.cuda.synchronize()
    prof = B.kda_profile_read()
    B.kda_profile_enable(False)
    launches = sum(n for n, _ in prof.values())

    # roofline of the kernel with the largest device time, each kernel against the bytes its design
    # must move: the fused / output pass reads q, k, v, z, beta and writes o for every token-head
    # (plus the states); the chunk preparation reads the same inputs and writes one operand block
    # per 32-token step and head; the state passes read those blocks (the summary pass twice: S~ and
    # M chains) and write states; the scan reads (M, S~) and writes S_in per segment step.
    pk, pk_src = peaks()
    th = T * H
    plan = B.kda_forward_plan(prob, ws.numel())
    n_seg = plan["num_segments"]
    seg_tokens = 16 * plan["seg_chunks"] * (n_seg - 1) if n_seg > 1 else 0  # tokens of all but the last segment
    state_bytes = H * dk * dv * 4
    blk = 53760  # operand block of one 32-token step and head
    chunk_heads = -(-T // 32) * H  # step-heads
    seg_chunk_heads = (seg_tokens // 32) * H
    in_bytes = th * ((2 * dk + dv + dk) * io_bytes + 4)
    alg = {
        "kda_chunk_fwd_tc": th * prefill_bytes_per_token_head(dk, dv, io_bytes) + 2 * state_bytes,
        "kda_chunk_fwd": th * prefill_bytes_per_token_head(dk, dv, io_bytes) + 2 * state_bytes,
        "kda_seg_summary_tc": seg_tokens * H * ((2 * dk + dv) * io_bytes + 4) + 2 * (n_seg - 1) * state_bytes,
        "kda_seg_scan": 3 * (n_seg - 1) * state_bytes,
        "kda_chunk_prep_tc": in_bytes + chunk_heads * blk,
        "kda_state_summary_tc": 2 * seg_chunk_heads * blk + 2 * (n_seg - 1) * state_bytes,
        "kda_chunk_state_tc": chunk_heads * blk + th * dv * io_bytes + 2 * state_bytes,
    }
    kernels = {}
    for name, (cnt, tot_ms) in prof.items():
        avg = tot_ms / cnt
        ab = alg.get(name)
        gbs = ab / (avg * 1e-3) / 1e9 if ab else None
        kernels[name] = {"launches_per_step": cnt / args.steps, "avg_ms": avg, "algorithmic_bytes": ab,
                         "achieved_gbs": gbs, "frac_of_hbm": gbs / pk["hbm_gbs"] if gbs else None}
    top_name = max(prof.items(), key=lambda kv: kv[1][1])[0]
    top = kernels[top_name]
    traffic = ncu_traffic(top_name)
    roofline = {"bound": "hbm", "kernel": top_name, "achieved": top["achieved_gbs"], "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": top["frac_of_hbm"], "traffic": traffic, "peak_source": pk_src,
                "algorithmic_bytes_per_launch": top["algorithmic_bytes"], "avg_launch_ms": top["avg_ms"],
                "path_achieved_gbs": (th * prefill_bytes_per_token_head(dk, dv, io_bytes) + 2 * state_bytes)
                / (ms * 1e-3) / 1e9, "kernels": kernels}
    roofline["path_frac"] = roofline["path_achieved_gbs"] / pk["hbm_gbs"]
    # the path's own roofline: min(tensor peak, arithmetic intensity x HBM); at d = 128 and 16-token
    # chunks the intensity is below the ridge point, so the bound is HBM
    ai = prefill_flops_per_token_head(dk, dv) / prefill_bytes_per_token_head(dk, dv, io_bytes)
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    path_bytes = th * prefill_bytes_per_token_head(dk, dv, io_bytes) + 2 * state_bytes
    roofline["path_roofline"] = {"bound": "hbm" if ai < ridge else "tensor", "flop_per_byte": ai,
                                 "ridge_flop_per_byte": ridge,
                                 "floor_ms": path_bytes / (pk["hbm_gbs"] * 1e9) * 1e3 if ai < ridge
                                 else th * prefill_flops_per_token_head(dk, dv) / (pk["bf16_tflops"] * 1e12) * 1e3,
                                 "frac": roofline["path_frac"]}
    flops = th * prefill_flops_per_token_head(dk, dv)
    tensor = {"achieved_tflops": flops / (ms * 1e-3) / 1e12,
              "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"],
              "flops_per_step": flops, "peak_tflops": pk["bf16_tflops"], "peak_source": pk_src}

    # ---- decode step (config: 256 sequences x 32 heads, d = 128)
    decode = None
    if not args.no_decode:
        decode = bench_decode(args, B, I, dev, stream, max_over_ranks, barrier, pk, pk_src)

    # ---- layer prologue / epilogue around the recurrence (same shape, L2 flushed before each launch)
    layer = None if args.no_layer else bench_layer(B, dev, stream, flush, T, H, dk, dv, max_over_ranks, barrier, pk,
                                                   pk_src)

    # ---- e2e through the public call with pinned host buffers
    e2e = bench_e2e(args, B, inp, dev, stream, max_over_ranks, barrier, world)

    # ---- the other prefill shapes of the pages' workloads (varlen batch, 1M-token context)
    shapes = None if args.no_shapes else bench_shapes(B, I, dev, stream, max_over_ranks, barrier, world)

    clk = clocks.stop() if clocks else None
    line = {
        "metric": METRIC, "value": value, "unit": "Mtok/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": I.WORKLOADS[WORKLOAD].name, "B": 1, "H": H, "T": T, "d_k": dk, "d_v": dv,
                   "chunk": 16, "io_dtype": "bf16", "state_dtype": "f32",
                   "arithmetic": "bf16 tensor-core products (split hi/lo where precision needs it) with fp32 "
                                 "accumulation; fp32 state",
                   "l2": "flushed by a 512 MiB write before every timed step"},
        "step_stats": step_stats, "roofline": roofline, "tensor": tensor, "decode": decode, "layer": layer,
        "cpu_baseline": cpu, "e2e": e2e, "shapes": shapes, "gpu_launches": launches, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def bench_shapes(B, I, dev, stream, max_over_ranks, barrier, world, ids_reps=((2, 10), (3, 4))):
    """Prefill throughput at the varlen (8 sequences x 32 heads) and long-context (1,048,576 tokens x
    8 heads) shapes: inputs drawn on the device with the workloads' distributions (larger than L2,
    so no flush), two warm-up calls, then `reps` calls timed one by one with CUDA events."""
    import torch
    res = []
    for wid, reps in ids_reps:
        w = I.WORKLOADS[wid]
        if w.varlen_range is not None:
            lo, hi = w.varlen_range
            lengths = torch.randint(lo, hi + 1, (w.num_varlen,), generator=torch.Generator().manual_seed(w.seed)).tolist()
        else:
            lengths = list(w.lengths)
        N, T, H, d = len(lengths), int(sum(lengths)), w.num_heads, w.d
        gen = torch.Generator(device=dev).manual_seed(w.seed)

        def tok(normalise):
            x = torch.randn(T, H, d, generator=gen, device=dev)
            if normalise:
                x = x / torch.sqrt((x * x).sum(dim=-1, keepdim=True) + I.L2_EPS)
            return x.to(torch.bfloat16)
        q, k, v, z = tok(True), tok(True), tok(False), tok(False)
        A = torch.randn(H, generator=gen, device=dev) * I.A_STD
        beta = torch.sigmoid(torch.randn(T, H, generator=gen, device=dev))
        S0 = torch.randn(N, H, d, d, generator=gen, device=dev) * I.S0_STD
        cu = torch.zeros(N + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
        cu = cu.to(dev)
        out = torch.empty(T, H, d, dtype=torch.bfloat16, device=dev)
        fin = torch.empty(N, H, d, d, dtype=torch.float32, device=dev)
        prob = B.make_problem(N, T, max(lengths), H, d, d, torch.bfloat16)
        ws = torch.empty(B.kda_forward_workspace_bytes(prob), dtype=torch.uint8, device=dev)

        def fwd():
            B.kda_forward(q, k, v, z, A, beta, initial_state=S0, cu_seqlens=cu, out=out, final_state=fin,
                          max_seqlen=max(lengths), workspace=ws)
        for _ in range(2):
            fwd()
        torch.cuda.synchronize()
        barrier()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for e0, e1 in evs:
            e0.record(stream)
            fwd()
            e1.record(stream)
        torch.cuda.synchronize()
        ms_list = sorted(e0.elapsed_time(e1) for e0, e1 in evs)
        ms = max_over_ranks(sum(ms_list) / len(ms_list))
        res.append({"workload": w.name, "sequences": N, "tokens": T, "token_heads": T * H, "reps": reps,
                    "ms_per_step": ms, "median_ms": max_over_ranks(ms_list[len(ms_list) // 2]),
                    "value": T * world / (ms * 1e-3) / 1e6, "unit": "Mtok/s",
                    "plan": B.kda_forward_plan(prob, ws.numel()), "l2": "inputs larger than L2"})
        del q, k, v, z, A, beta, S0, cu, out, fin, ws
        torch.cuda.empty_cache()
    return res


def bench_decode(args, B, I, dev, stream, max_over_ranks, barrier, pk, pk_src):
    import torch
    w = I.WORKLOADS[DECODE_WORKLOAD]
    N, H, dd = len(w.lengths), w.num_heads, w.d
    L = w.lengths[0]
    steps = args.decode_steps
    g = torch.Generator(device=dev).manual_seed(w.seed)

    def toks(*shape):
        q = torch.randn(*shape, dd, generator=g, device=dev)
        k = torch.randn(*shape, dd, generator=g, device=dev)
        v = torch.randn(*shape, dd, generator=g, device=dev)
        z = torch.randn(*shape, dd, generator=g, device=dev)
        n = lambda x: x / torch.sqrt((x * x).sum(-1, keepdim=True) + I.L2_EPS)
        return [t.to(w.io_dtype).contiguous() for t in (n(q), n(k), v, z)]

    A = (torch.randn(H, generator=g, device=dev) * I.A_STD).float()
    # the state comes from a 512-token varlen prefill from a random initial state
    pq, pk_, pv, pz = toks(N * L, H)
    pb = torch.sigmoid(torch.randn(N * L, H, generator=g, device=dev)).float()
    s0 = (torch.randn(N, H, dd, dd, generator=g, device=dev) * I.S0_STD).float()
    cu = (torch.arange(N + 1, device=dev, dtype=torch.int32) * L)
    _, state = B.kda_forward(pq, pk_, pv, pz, A, pb, initial_state=s0, cu_seqlens=cu, max_seqlen=L)
    del pq, pk_, pv, pz, pb
    dq, dk_, dv_, dz = toks(steps, N, H)
    db = torch.sigmoid(torch.randn(steps, N, H, generator=g, device=dev)).float()
    outs = torch.empty(steps, N, H, dd, dtype=w.io_dtype, device=dev)
    for s in range(3):
        B.kda_decode_step(dq[s], dk_[s], dv_[s], dz[s], A, db[s], state, out=outs[s])
    torch.cuda.synchronize()
    B.kda_profile_enable(True)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(steps):
        B.kda_decode_step(dq[s], dk_[s], dv_[s], dz[s], A, db[s], state, out=outs[s])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    prof = B.kda_profile_read()
    B.kda_profile_enable(False)
    ms = max_over_ranks(e0.elapsed_time(e1) / steps)
    nbytes = N * H * decode_bytes_per_head(dd, dd, 2)
    kn, kms = prof.get("kda_decode_step", (steps, ms * steps))
    kavg = kms / kn
    gbs = nbytes / (kavg * 1e-3) / 1e9
    del dq, dk_, dv_, dz, db, outs
    replay = None if args.no_replay else bench_replay(B, dev, g, toks, A, state, ms, max_over_ranks, barrier, pk,
                                                      pk_src)
    return {"workload": w.name, "ms_per_step": ms, "tokens_per_s": N / (ms * 1e-3),
            "state_gbs": nbytes / (ms * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "kernel": "kda_decode_step", "achieved": gbs, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / pk["hbm_gbs"], "frac_of_8tbs": gbs / 8000.0,
                         "traffic": ncu_traffic("kda_decode_step"), "peak_source": pk_src,
                         "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": kavg},
            "gpu_launches": kn, "replay": replay}


def bench_layer(B, dev, stream, flush, T, H, dk, dv, max_over_ranks, barrier, pk, pk_src, reps=20, conv_width=4):
    """The KDA layer's prologue (short convolution, Swish, q/k L2 norm of the three projections) and
    epilogue (head-wise RMSNorm and sigmoid output gate) at the prefill workload's shape, bf16, each
    launch timed with CUDA events after an L2 flush."""
    import torch
    g = torch.Generator(device=dev).manual_seed(6)
    x = [torch.randn(T, H, d, generator=g, device=dev).to(torch.bfloat16) for d in (dk, dk, dv)]
    w = [(torch.randn(H, d, conv_width, generator=g, device=dev) * 0.5).float() for d in (dk, dk, dv)]
    outs = [torch.empty_like(t) for t in x]
    o = torch.randn(T, H, dv, generator=g, device=dev).to(torch.bfloat16)
    gate = torch.randn(T, H, dv, generator=g, device=dev).to(torch.bfloat16)
    wt = torch.randn(dv, generator=g, device=dev).float()
    y = torch.empty_like(o)

    def pro():
        B.kda_prologue(*x, *w, q=outs[0], k=outs[1], v=outs[2])

    def epi():
        B.kda_epilogue(o, gate, wt, eps=1e-5, y=y)

    res = {}
    for name, fn, nbytes in (("prologue", pro, 2 * T * H * (2 * dk + dv) * 2 + H * (2 * dk + dv) * conv_width * 4),
                             ("epilogue", epi, 3 * T * H * dv * 2 + dv * 4)):
        for _ in range(3):
            fn()
        barrier()
        torch.cuda.synchronize()
        times = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        barrier()
        ms = max_over_ranks(sum(times) / reps)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "median_ms": statistics.median(times), "algorithmic_bytes": nbytes, "gbs": gbs,
                     "frac": gbs / pk["hbm_gbs"], "traffic": ncu_traffic(f"kda_{name}")}
    return {"workload": f"T={T} H={H} d_k={dk} d_v={dv} bf16, short convolution width {conv_width}",
            **res, "peak": pk["hbm_gbs"], "peak_source": pk_src, "gpu_launches": 2 * (reps + 3),
            "l2": "flushed by a 512 MiB write before every timed launch"}


REPLAY_WINDOW = 7  # drafted tokens per sequence and speculation round


def replay_bytes(N, H, dk, dv, tokens_read, tokens_out, state_writes, io_bytes=2):
    """Minimum HBM bytes of one kda_decode_replay launch: the snapshot read once, the drafted
    tokens' q, k, z, v (io dtype) and beta (fp32) read, outputs and accepted states written."""
    return (N * H * dk * dv * 4 + tokens_read * H * ((3 * dk + dv) * io_bytes + 4)
            + tokens_out * H * dv * io_bytes + state_writes * H * dk * dv * 4 + N * 4)


def bench_replay(B, dev, g, toks, A, state, decode_ms, max_over_ranks, barrier, pk, pk_src, reps=20):
    """Speculative-decode rounds on the decode workload's state (256 sequences x 32 heads, d=128):
    verify a 7-token window per sequence from the snapshot (outputs only), then commit the accepted
    prefix in place (state only); accepted counts uniform in [0, 7].  The state (512 MiB) exceeds
    L2, so no flush is needed between launches."""
    import torch
    N, H, dd = state.shape[0], state.shape[1], state.shape[2]
    L = REPLAY_WINDOW
    rq, rk, rv, rz = toks(reps, N * L, H)
    rb = torch.sigmoid(torch.randn(reps, N * L, H, generator=g, device=dev)).float()
    acc = torch.randint(0, L + 1, (reps, N), generator=g, device=dev, dtype=torch.int32)
    out = torch.empty(N * L, H, dd, dtype=rq.dtype, device=dev)
    stream = torch.cuda.current_stream()

    def verify(r):
        B.kda_decode_replay(rq[r], rk[r], rv[r], rz[r], A, rb[r], state, out=out, want_state=False)

    def commit(r):
        B.kda_decode_replay(rq[r], rk[r], rv[r], rz[r], A, rb[r], state, accepted=acc[r], state_out=state,
                            want_out=False)

    for r in range(3):
        verify(r)
        commit(r)
    torch.cuda.synchronize()
    res = {}
    for name, fn in (("verify", verify), ("commit", commit)):
        barrier()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        ev[0].record(stream)
        for r in range(reps):
            fn(r)
            ev[r + 1].record(stream)
        torch.cuda.synchronize()
        barrier()
        times = [ev[r].elapsed_time(ev[r + 1]) for r in range(reps)]
        ms = max_over_ranks(sum(times) / reps)
        if name == "verify":
            nbytes = replay_bytes(N, H, dd, dd, N * L, N * L, 0)
        else:
            nbytes = replay_bytes(N, H, dd, dd, int(acc.sum().item()) / reps, 0, N)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "median_ms": statistics.median(times), "algorithmic_bytes": nbytes, "gbs": gbs,
                     "frac": gbs / pk["hbm_gbs"], "traffic": ncu_traffic(f"kda_decode_replay_{name}")}
    round_ms = res["verify"]["ms"] + res["commit"]["ms"]
    return {"workload": f"{N} sequences x {H} heads, d={dd}, {L}-token drafted window, bf16 inputs, fp32 state",
            "kernel": "kda_decode_replay", **res, "round_ms": round_ms,
            "drafted_tokens_per_s": N * L / (round_ms * 1e-3),
            "accepted_tokens_per_s": float(acc.sum().item()) / reps / (round_ms * 1e-3),
            "vs_decode_steps": (L * decode_ms) / round_ms,
            "peak": pk["hbm_gbs"], "peak_source": pk_src,
            "gpu_launches": 2 * reps}


def bench_e2e(args, B, inp, dev, stream, max_over_ranks, barrier, world, depth=2):
    """The prefill end to end through kda_forward with host buffers: every step copies its inputs
    from pinned host memory to the device, runs the prefill and copies the outputs and final state
    back to pinned host memory.  Steps stream through three CUDA streams with `depth` sets of device
    buffers, so step i+1's inputs travel while step i computes and step i-1's outputs travel back
    (a stream of independent prefill requests); the time per step is the steady-state spacing."""
    import torch
    keys = ("q", "k", "v", "z", "A", "beta", "S0")
    T, H, dk = inp["k"].shape
    dv = inp["v"].shape[2]
    # a step's inputs live back to back in one pinned host buffer and travel as one copy into one
    # device buffer; the call gets views of it (256-byte aligned)
    offs, total = {}, 0
    for k in keys:
        offs[k] = total
        total += (inp[k].numel() * inp[k].element_size() + 255) // 256 * 256
    h_all = torch.empty(total, dtype=torch.uint8).pin_memory()

    def views(buf):
        return {k: buf[offs[k]:offs[k] + inp[k].numel() * inp[k].element_size()].view(inp[k].dtype).view(inp[k].shape)
                for k in keys}
    host = views(h_all)
    for k in keys:
        host[k].copy_(inp[k])
    d_all = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(depth)]
    dbuf = [views(b) for b in d_all]
    # outputs and final state likewise in one buffer each side: one D2H copy per step
    o_bytes = T * H * dv * inp["k"].element_size()
    f_off = (o_bytes + 255) // 256 * 256
    o_total = f_off + H * dk * dv * 4

    def out_views(buf):
        return (buf[:o_bytes].view(inp["k"].dtype).view(T, H, dv), buf[f_off:o_total].view(torch.float32).view(1, H, dk, dv))
    d_out_all = [torch.empty(o_total, dtype=torch.uint8, device=dev) for _ in range(depth)]
    dout = [out_views(b) for b in d_out_all]
    h_out_all = torch.empty(o_total, dtype=torch.uint8).pin_memory()
    h_out, h_fin = out_views(h_out_all)
    prob = B.make_problem(1, T, T, H, dk, dv, inp["k"].dtype)
    ws = torch.empty(B.kda_forward_workspace_bytes(prob), dtype=torch.uint8, device=dev)
    h2d = total
    d2h = o_total
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(depth)]
    ev_cmp = [torch.cuda.Event() for _ in range(depth)]
    ev_out = [torch.cuda.Event() for _ in range(depth)]
    count = [0]

    def step():
        i = count[0]
        b = i % depth
        with torch.cuda.stream(s_in):
            if i >= depth:
                s_in.wait_event(ev_cmp[b])   # the compute of step i - depth has read these inputs
            d_all[b].copy_(h_all, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[b])
            if i >= depth:
                s_cmp.wait_event(ev_out[b])  # the outputs of step i - depth have left
            d = dbuf[b]
            B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                          out=dout[b][0], final_state=dout[b][1], workspace=ws, stream=s_cmp)
            ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[b])
            h_out_all.copy_(d_out_all[b], non_blocking=True)
            ev_out[b].record(s_out)
        count[0] += 1

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(args.steps):
        step()
    e1.record(s_out)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)
    return {"value": T * world / (ms * 1e-3) / 1e6, "unit": "Mtok/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "pipeline": f"{depth} device buffer sets over H2D / compute / D2H streams; one copy each way per step"}


if __name__ == "__main__":
    sys.exit(main())
