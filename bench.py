"""Benchmark: KDA chunked prefill of the 1,048,576-token context (B=1, H=8, d_k=d_v=128, bf16 inputs,
fp32 state) on one GB300 per rank, with the other workloads of the pages beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --case prefill-tc|prefill-simt|decode|replay|layer|backward [--tokens T] [--heads H]
                    [--seqs N] [--reps R] [--window L]      (one small invocation for a profiler)

Prints ONE JSON line.  `value` is prefill throughput in million tokens per second with inputs
resident in HBM (10.8 GB per step, larger than L2), timed with CUDA events on the launching stream.
`roofline` takes the kernel with the largest device time in that step: the path's algorithmic bytes
(1,284 B per token-head plus the states) over its average launch time, against the measured HBM
copy bandwidth.  `shapes` holds the 4096-token x 16-head prefill (L2 flushed by a 512 MiB write before
every step) and the varlen batch (8 sequences x 32 heads); `decode` the decode step's state
bandwidth (256 sequences x 32 heads) and, under `replay`, the speculative-decode round; `layer` the
layer prologue and epilogue; `backward` the gradients at the 4096-token shape.  `e2e` repeats the
headline prefill through the same public call with pinned host buffers, host<->device copies inside
the timed region.  `cpu_baseline` times the fp64 oracle on the host cores (all and one) on a bounded
sample of the headline workload, with the same sampler as `--impl reference`.

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
WORKLOAD = 3        # B=1, H=8, T=1,048,576, d=128 bf16 prefill (the largest workload)
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
            "kda_chunk_state_tc": "kda_state_tc.cu", "kda_bwd_gram": "kda_backward.cu",
            "kda_bwd_states": "kda_backward.cu", "kda_bwd_dstates": "kda_backward.cu",
            "kda_bwd_chunk": "kda_backward.cu", "kda_bwd_da": "kda_backward.cu"}.get(kernel)
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

def cpu_model() -> str:
    """Host CPU model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_layout(H, dv, threads):
    """Heads and value columns per unit of an oracle sample so that the (head, column block) units
    are a whole multiple of the threads (every thread gets the same number of units): the widest
    column block (least repeated gate work) for which some head count works, then the most heads."""
    cb = dv
    while cb >= 1:
        if dv % cb == 0:
            for h in range(min(H, threads * dv // cb), 0, -1):
                if (h * (dv // cb)) % threads == 0:
                    return h, cb
        cb //= 2
    return min(H, threads), dv


def oracle_rate(workload, target_s=10.0, threads=0):
    """fp64 oracle throughput on a bounded sample of a workload: the first t tokens of heads [0, h),
    drawn with the workload's own recipe (seeded), sized from a short calibration run to take about
    `target_s` seconds.  Value columns are split so that the parallel units are a whole multiple of
    the threads.  Returns token-heads/s and the sample."""
    import oracle
    from linear_attention_recurrence_kda_gb300 import inputs as I
    w = I.WORKLOADS[workload]
    nt = threads if threads > 0 else oracle.max_threads()
    h, cb = oracle_layout(w.num_heads, w.d, nt)
    cal_t = 256
    inp = I.make_inputs(workload, lengths=[cal_t], num_heads=h, seed=w.seed)

    def run(t, reps=1):
        sl = lambda x: x[:t]
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle.forward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["z"]), inp["A"], sl(inp["beta"]),
                           S0=inp["S0"], col_block=cb, threads=nt)
        return time.perf_counter() - t0

    run(16)
    per_tok = run(cal_t) / cal_t
    t = int(max(16, min(1 << 16, target_s / per_tok)))
    if t > cal_t:
        inp = I.make_inputs(workload, lengths=[t], num_heads=h, seed=w.seed)
    reps = max(1, int(target_s / (per_tok * t)))
    el = run(t, reps)
    th_per_s = reps * h * t / el
    return {"token_heads_per_s": th_per_s, "tok_per_s": th_per_s / w.num_heads, "heads": h, "tokens": t,
            "reps": reps, "seconds": el, "threads": nt, "col_block": cb}


def cpu_baseline_leg(workload, target_s=12.0):
    """The oracle on all host cores and on one core, same sampler as the reference arm."""
    import oracle
    oracle.build()
    from linear_attention_recurrence_kda_gb300 import inputs as I
    H = I.WORKLOADS[workload].num_heads
    r = oracle_rate(workload, target_s=target_s)
    r1 = oracle_rate(workload, target_s=target_s / 3, threads=1)
    return {"value": r["tok_per_s"] / 1e6, "unit": "Mtok/s", "cores": r["threads"], "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"first {r['tokens']} tokens of heads [0,{r['heads']}) of the workload's recipe, "
                      f"{r['reps']} repetition(s), value columns in blocks of {r['col_block']}, fp64, "
                      f"{r['seconds']:.1f} s; scaled to tokens of all {H} heads",
            "token_heads_per_s": r["token_heads_per_s"],
            "one_core": {"value": r1["tok_per_s"] / 1e6, "unit": "Mtok/s", "cores": 1,
                         "token_heads_per_s": r1["token_heads_per_s"],
                         "sample": f"first {r1['tokens']} tokens of head 0, {r1['reps']} repetition(s), "
                                   f"{r1['seconds']:.1f} s"}}


def reference_arm(args):
    """The fp64 oracle as the reference implementation, on the host cores, on the GPU arm's
    workload, metric and unit; each step is a bounded sample of that workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    from linear_attention_recurrence_kda_gb300 import inputs as I
    w = I.WORKLOADS[WORKLOAD]
    nt = oracle.max_threads()
    # the same sampler as the GPU arm's cpu_baseline, each step sized to ~0.25 s
    cal = oracle_rate(WORKLOAD, target_s=0.25, threads=nt)
    h, t, cb = cal["heads"], cal["tokens"], cal["col_block"]
    inp = I.make_inputs(WORKLOAD, lengths=[t], num_heads=h, seed=w.seed)

    def step():
        oracle.forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], S0=inp["S0"], col_block=cb,
                       threads=nt)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    mtok = h * t / (el / args.steps) / w.num_heads / 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": mtok, "unit": "Mtok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": 1, "H": w.num_heads, "T": sum(w.lengths), "d_k": w.d, "d_v": w.d},
        "cpu_baseline": {"value": mtok, "unit": "Mtok/s", "cores": nt, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": f"first {t} tokens of heads [0,{h}) of the workload's recipe per step, value "
                                   f"columns in blocks of {cb} (fp64, OpenMP); scaled to tokens of all "
                                   f"{w.num_heads} heads"},
        "e2e": {"value": mtok, "unit": "Mtok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- small invocations for profilers

def run_case(args):
    """One small, self-contained invocation of a kernel family (seeded inputs on the device, one
    warm-up call and `--reps` calls through the C ABI), sized for profiler captures."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from linear_attention_recurrence_kda_gb300 import binding as B
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(1)
    d = 128

    def toks(*shape, dtype=torch.bfloat16):
        x = [torch.randn(*shape, d, generator=g, device=dev) for _ in range(4)]
        n = lambda t: t / torch.sqrt((t * t).sum(-1, keepdim=True) + 1e-6)
        return [t.to(dtype).contiguous() for t in (n(x[0]), n(x[1]), x[2], x[3])]

    if args.case in ("prefill-tc", "prefill-simt", "backward"):
        dt = torch.float32 if args.case == "prefill-simt" else torch.bfloat16
        T, H, N = args.tokens * args.seqs, args.heads, args.seqs
        q, k, v, z = toks(T, H, dtype=dt)
        A = (torch.randn(H, generator=g, device=dev) * 0.5).float()
        beta = torch.sigmoid(torch.randn(T, H, generator=g, device=dev)).float()
        s0 = (torch.randn(N, H, d, d, generator=g, device=dev) * 0.02).float()
        if args.case == "backward":
            do = torch.randn(T, H, d, generator=g, device=dev).to(dt)
            dsf = torch.randn(N, H, d, d, generator=g, device=dev) * 0.1
            for _ in range(args.reps + 1):
                B.kda_backward(q, k, v, z, A, beta, do, dsf, initial_state=s0)
        else:
            out = torch.empty(T, H, d, dtype=dt, device=dev)
            fin = torch.empty_like(s0)
            for _ in range(args.reps + 1):
                B.kda_forward(q, k, v, z, A, beta, initial_state=s0, out=out, final_state=fin)
    elif args.case == "decode":
        N, H = args.seqs if args.seqs > 1 else 128, args.heads if args.heads != 16 else 32
        q, k, v, z = toks(N, H)
        A = (torch.randn(H, generator=g, device=dev) * 0.5).float()
        beta = torch.sigmoid(torch.randn(N, H, generator=g, device=dev)).float()
        state = (torch.randn(N, H, d, d, generator=g, device=dev) * 0.1).float()
        out = torch.empty(N, H, d, dtype=torch.bfloat16, device=dev)
        for _ in range(args.reps + 1):
            B.kda_decode_step(q, k, v, z, A, beta, state, out=out)
    elif args.case == "replay":
        N, H, L = args.seqs if args.seqs > 1 else 256, args.heads if args.heads != 16 else 32, args.window
        q, k, v, z = toks(N * L, H)
        A = (torch.randn(H, generator=g, device=dev) * 0.5).float()
        beta = torch.sigmoid(torch.randn(N * L, H, generator=g, device=dev)).float()
        state = (torch.randn(N, H, d, d, generator=g, device=dev) * 0.1).float()
        acc = torch.randint(0, L + 1, (N,), generator=g, device=dev, dtype=torch.int32)
        out = torch.empty(N * L, H, d, dtype=torch.bfloat16, device=dev)
        for _ in range(args.reps + 1):
            B.kda_decode_replay(q, k, v, z, A, beta, state, out=out, want_state=False)
            B.kda_decode_replay(q, k, v, z, A, beta, state, accepted=acc, state_out=state, want_out=False)
    elif args.case == "layer":
        T, H, K = args.tokens, args.heads, 4
        x = [torch.randn(T, H, d, generator=g, device=dev).to(torch.bfloat16) for _ in range(3)]
        w = [(torch.randn(H, d, K, generator=g, device=dev) * 0.5).float() for _ in range(3)]
        o = torch.randn(T, H, d, generator=g, device=dev).to(torch.bfloat16)
        gate = torch.randn(T, H, d, generator=g, device=dev).to(torch.bfloat16)
        wt = torch.randn(d, generator=g, device=dev).float()
        for _ in range(args.reps + 1):
            B.kda_prologue(*x, *w)
            B.kda_epilogue(o, gate, wt)
    torch.cuda.synchronize()
    return 0


# ---------------------------------------------------------------- GPU arm

def prefill_roofline(prof, steps, lengths, H, dk, dv, io_bytes, plan, pk, pk_src, ms):
    """Roofline of the kernel with the largest device time in a prefill step.  `achieved` is the
    path's algorithmic bytes -- the per-token-head minimum (1,284 B at d = 128) times the token-heads
    one launch processes, plus reading the initial and writing the final states -- over that
    kernel's average launch time.  `kernels` lists every kernel's share of the step with the bytes
    its own design moves (the split plan's operand blocks included); `traffic` is the committed ncu
    DRAM bytes per token-head of a smaller capture of the same source, scaled to this workload."""
    T = int(sum(lengths))
    N = len(lengths)
    th = T * H
    state_bytes = dk * dv * 4
    path_bytes = th * prefill_bytes_per_token_head(dk, dv, io_bytes) + 2 * N * H * state_bytes
    seg_len = 16 * plan["seg_chunks"] if plan["num_segments"] > 1 else 0
    nseg = [max(1, -(-L // seg_len)) if seg_len else 1 for L in lengths]
    summarised = [min(L, (ns - 1) * seg_len) for L, ns in zip(lengths, nseg)]
    n_sum = sum(ns - 1 for ns in nseg)
    blk = 53760
    step_heads = sum(-(-L // 32) for L in lengths) * H
    sum_step_heads = sum(-(-x // 32) for x in summarised) * H
    in_bytes = th * ((3 * dk + dv) * io_bytes + 4)
    own = {
        "kda_chunk_fwd_tc": path_bytes, "kda_chunk_fwd": path_bytes,
        "kda_seg_summary_tc": sum(summarised) * H * ((3 * dk + dv) * io_bytes + 4) + 2 * n_sum * H * state_bytes,
        "kda_seg_scan": 3 * n_sum * H * state_bytes,
        "kda_chunk_prep_tc": in_bytes + step_heads * blk,
        "kda_state_summary_tc": 2 * sum_step_heads * blk + 2 * n_sum * H * state_bytes,
        "kda_chunk_state_tc": step_heads * blk + th * dv * io_bytes + 2 * N * H * state_bytes,
    }
    total_ms = sum(v[1] for v in prof.values())
    kernels = {}
    traffic_step, traffic_known = 0.0, True
    for name, (cnt, tot_ms) in prof.items():
        avg = tot_ms / cnt
        ob = own.get(name)
        tr = ncu_traffic_per_token_head(name)
        if tr is None:
            traffic_known = False
        else:
            traffic_step += tr * th * cnt / steps
        kernels[name] = {"launches_per_step": cnt / steps, "avg_ms": avg, "share": tot_ms / total_ms,
                         "own_bytes": ob, "own_gbs": ob / (avg * 1e-3) / 1e9 if ob else None,
                         "traffic": tr * th if tr is not None else None}
    top_name = max(prof.items(), key=lambda kv: kv[1][1])[0]
    top = kernels[top_name]
    achieved = path_bytes / (top["avg_ms"] * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": top_name, "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": top["traffic"], "peak_source": pk_src,
            "algorithmic_bytes_per_launch": path_bytes, "avg_launch_ms": top["avg_ms"],
            "units_per_launch": th, "bytes_per_unit": prefill_bytes_per_token_head(dk, dv, io_bytes),
            "path_achieved_gbs": path_bytes / (ms * 1e-3) / 1e9,
            "path_frac": path_bytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "traffic_per_step": traffic_step if traffic_known else None,
            "traffic_ratio": traffic_step / path_bytes if traffic_known else None,
            "traffic_note": "ncu DRAM bytes per token-head of a 4096-token x 16-head capture of the same source, "
                            "scaled by token-heads (null when the source changed since the capture)",
            "kernels": kernels}


def tensor_figures(th, dk, dv, ms, pk, pk_src):
    flops = th * prefill_flops_per_token_head(dk, dv)
    io_bytes = 2
    ai = prefill_flops_per_token_head(dk, dv) / prefill_bytes_per_token_head(dk, dv, io_bytes)
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    return {"achieved_tflops": flops / (ms * 1e-3) / 1e12, "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"],
            "flops_per_step": flops, "peak_tflops": pk["bf16_tflops"], "peak_source": pk_src,
            "flop_per_byte": ai, "ridge_flop_per_byte": ridge, "path_bound": "hbm" if ai < ridge else "tensor"}


def device_workload(I, wid, dev, lengths=None):
    """A workload's inputs drawn on the device with its distributions (seeded)."""
    import torch
    w = I.WORKLOADS[wid]
    if lengths is None:
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
        return x.to(w.io_dtype)
    q, k, v, z = tok(True), tok(True), tok(False), tok(False)
    A = torch.randn(H, generator=gen, device=dev) * I.A_STD
    beta = torch.sigmoid(torch.randn(T, H, generator=gen, device=dev))
    S0 = torch.randn(N, H, d, d, generator=gen, device=dev) * I.S0_STD
    cu = torch.zeros(N + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return {"q": q, "k": k, "v": v, "z": z, "A": A, "beta": beta, "S0": S0, "cu_seqlens": cu.to(dev),
            "lengths": lengths, "name": w.name}


def bench_prefill(B, d, dev, stream, steps, warmup, max_over_ranks, barrier, world, pk, pk_src, flush=None):
    """K timed prefill steps of one workload (inputs resident in HBM), per-step CUDA events on the
    launching stream, optionally an L2 flush before every step; then the same steps with the
    library's per-kernel event hooks for the roofline."""
    import torch
    lengths = d["lengths"]
    T, H, dk = d["k"].shape
    dv = d["v"].shape[2]
    N = len(lengths)
    io_bytes = d["k"].element_size()
    out = torch.empty(T, H, dv, dtype=d["k"].dtype, device=dev)
    fin = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    ml = max(lengths)
    prob = B.make_problem(N, T, ml, H, dk, dv, d["k"].dtype)
    ws = torch.empty(B.kda_forward_workspace_bytes(prob), dtype=torch.uint8, device=dev)

    def fwd():
        B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                      cu_seqlens=d["cu_seqlens"], out=out, final_state=fin, max_seqlen=ml, workspace=ws)

    for _ in range(max(3, warmup)):
        if flush is not None:
            flush.zero_()
        fwd()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        evs[i][0].record(stream)
        fwd()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms = max_over_ranks(sum(step_ms) / len(step_ms))
    srt = sorted(step_ms)
    res = {"workload": d["name"], "sequences": N, "tokens": T, "token_heads": T * H, "ms_per_step": ms,
           "median_ms": max_over_ranks(srt[len(srt) // 2]),
           "p90_ms": max_over_ranks(srt[min(len(srt) - 1, int(0.9 * len(srt)))]),
           "value": T * world / (ms * 1e-3) / 1e6, "unit": "Mtok/s",
           "plan": B.kda_forward_plan(prob, ws.numel()),
           "l2": "flushed by a 512 MiB write before every timed step" if flush is not None else "inputs larger than L2"}
    if flush is not None:
        barrier()
        torch.cuda.synchronize()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for _ in range(steps):
            fwd()
        w1.record(stream)
        torch.cuda.synchronize()
        warm = max_over_ranks(w0.elapsed_time(w1) / steps)
        res.update({"warm_l2_ms_per_step": warm, "warm_l2_value": T * world / (warm * 1e-3) / 1e6})
    # per-kernel device times (the hooks sit between kernels and stop one kernel's launch from
    # overlapping the previous one's tail, so the step time above is taken without them)
    B.kda_profile_enable(True)
    for _ in range(steps):
        if flush is not None:
            flush.zero_()
        fwd()
    torch.cuda.synchronize()
    prof = B.kda_profile_read()
    B.kda_profile_enable(False)
    res["gpu_launches"] = sum(n for n, _ in prof.values())
    res["launches_per_step"] = res["gpu_launches"] / steps
    res["roofline"] = prefill_roofline(prof, steps, lengths, H, dk, dv, io_bytes, res["plan"], pk, pk_src, ms)
    res["tensor"] = tensor_figures(T * H, dk, dv, ms, pk, pk_src)
    del out, fin, ws
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-steps", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-replay", action="store_true", help="skip the speculative-decode replay leg")
    ap.add_argument("--no-layer", action="store_true", help="skip the layer prologue / epilogue leg")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward leg")
    ap.add_argument("--no-shapes", action="store_true", help="skip the 4096-token and varlen prefill legs")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--no-kcp", action="store_true", help="skip the context-parallel leg (N > 1 only)")
    ap.add_argument("--case", choices=["prefill-tc", "prefill-simt", "decode", "replay", "layer", "backward"],
                    help="run one small invocation for a profiler capture instead of the benchmark")
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--heads", type=int, default=16)
    ap.add_argument("--seqs", type=int, default=1)
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--window", type=int, default=7)
    args = ap.parse_args()
    if args.case:
        return run_case(args)
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

    pk, pk_src = peaks()
    # ---- CPU oracle baseline first (rank 0 only, before any timed GPU work)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(WORKLOAD)

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_id) if rank == 0 else None
    time.sleep(0.3)

    # ---- the headline: the 1,048,576-token, 8-head prefill (inputs larger than L2)
    d3 = device_workload(I, WORKLOAD, dev)
    head = bench_prefill(B, d3, dev, stream, args.steps, args.warmup, max_over_ranks, barrier, world, pk, pk_src)
    e2e = None if args.no_e2e else bench_e2e(args, B, d3, dev, max_over_ranks, barrier, world)
    T3, H3 = d3["k"].shape[0], d3["k"].shape[1]
    del d3
    torch.cuda.empty_cache()

    # ---- the 4096-token, 16-head prefill (86 MB: L2 flushed before every step) and the varlen batch
    shapes = None
    if not args.no_shapes:
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        d1 = device_workload(I, 1, dev)
        shapes = {"prefill_4096": bench_prefill(B, d1, dev, stream, 50, 5, max_over_ranks, barrier, world, pk, pk_src,
                                                flush=flush)}
        del d1
        d2 = device_workload(I, 2, dev)
        shapes["varlen"] = bench_prefill(B, d2, dev, stream, 10, 2, max_over_ranks, barrier, world, pk, pk_src)
        del d2, flush
        torch.cuda.empty_cache()

    # ---- decode step (256 sequences x 32 heads, d = 128) and the speculative-decode round
    decode = None
    if not args.no_decode:
        decode = bench_decode(args, B, I, dev, stream, max_over_ranks, barrier, pk, pk_src)

    # ---- layer prologue / epilogue and the backward at the 4096-token shape
    layer = backward = None
    if not args.no_layer or not args.no_backward:
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        if not args.no_layer:
            layer = bench_layer(B, dev, stream, flush, 4096, 16, 128, 128, max_over_ranks, barrier, pk, pk_src)
            # and at the headline context's shape, where the tensors are far larger than L2 and a
            # launch's fixed cost is a small part of its time
            layer["headline_shape"] = bench_layer(B, dev, stream, flush, T3, H3, 128, 128, max_over_ranks, barrier,
                                                  pk, pk_src, reps=5)
        if not args.no_backward:
            backward = bench_backward(B, I, dev, stream, max_over_ranks, barrier, pk, pk_src)
        del flush

    # ---- context-parallel prefill of the long context across the ranks (one exchange per call)
    kcp = None
    if world > 1 and not args.no_kcp:
        kcp = bench_kcp(B, I, dev, stream, world, rank, max_over_ranks, barrier)

    clk = clocks.stop() if clocks else None
    launches = head["gpu_launches"]
    line = {
        "metric": METRIC, "value": head["value"], "unit": "Mtok/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": I.WORKLOADS[WORKLOAD].name, "B": 1, "H": H3, "T": T3, "d_k": 128, "d_v": 128,
                   "chunk": 16, "io_dtype": "bf16", "state_dtype": "f32",
                   "arithmetic": "bf16 tensor-core products (split hi/lo where precision needs it) with fp32 "
                                 "accumulation; fp32 state",
                   "l2": "inputs larger than L2 (10.8 GB per step), no flush"},
        "step_stats": {k: head[k] for k in ("median_ms", "p90_ms", "plan", "launches_per_step")},
        "roofline": head["roofline"], "tensor": head["tensor"], "shapes": shapes, "decode": decode, "layer": layer,
        "backward": backward, "kcp": kcp, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def bench_kcp(B, I, dev, stream, world, rank, max_over_ranks, barrier, reps=5):
    """Context-parallel prefill of the 1,048,576-token, 8-head sequence split by tokens over the
    ranks: every rank summarises its range, one all-gather of the summaries (NCCL), the prefix scan
    and the re-run from the scanned state.  The sequence's total work is fixed as ranks are added
    (strong scaling); the time is the slowest rank's."""
    import torch
    from linear_attention_recurrence_kda_gb300 import context_parallel as CP
    w = I.WORKLOADS[WORKLOAD]
    T, H, d = sum(w.lengths), w.num_heads, w.d
    Tr = T // world
    gen = torch.Generator(device=dev).manual_seed(w.seed * 1000 + rank)

    def tok(normalise):
        x = torch.randn(Tr, H, d, generator=gen, device=dev)
        if normalise:
            x = x / torch.sqrt((x * x).sum(dim=-1, keepdim=True) + I.L2_EPS)
        return x.to(w.io_dtype)
    q, k, v, z = tok(True), tok(True), tok(False), tok(False)
    A = torch.randn(H, generator=torch.Generator(device=dev).manual_seed(w.seed), device=dev) * I.A_STD
    beta = torch.sigmoid(torch.randn(Tr, H, generator=gen, device=dev))
    S0 = torch.randn(1, H, d, d, generator=torch.Generator(device=dev).manual_seed(w.seed), device=dev) * I.S0_STD

    def run():
        return CP.kcp_forward(q, k, v, z, A, beta, initial_state=S0, num_seqs=1)
    for _ in range(2):
        run()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / reps)
    return {"workload": f"{w.name}, tokens split over {world} ranks", "ms_per_step": ms,
            "value": T / (ms * 1e-3) / 1e6, "unit": "Mtok/s", "scaling": "strong",
            "exchange_bytes_per_rank": 4 * H * d * (d + d),
            "flow": "kda_forward_summary, one all-gather, kda_state_scan, kda_forward from the scanned state"}


def ncu_traffic_per_token_head(kernel):
    """ncu DRAM bytes per token-head of a committed capture of this source (prefill kernels)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("source_sha") != src_sha(kernel) or not d.get("token_heads"):
        return None
    return d["dram_bytes_per_launch"] / d["token_heads"]


def layer_traffic(kernel, token_heads):
    """ncu DRAM bytes of one layer-kernel launch, from the committed capture of this source taken at
    this size (null at another size: at the capture's size the outputs stay in L2, so the traffic
    does not grow in proportion)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("source_sha") != src_sha(kernel) or d.get("token_heads") != token_heads:
        return None
    return d["dram_bytes_per_launch"]


def backward_bytes_per_token_head(dk, dv, io_bytes):
    """Minimum HBM bytes of the backward per token-head: read q, k, z, v, beta and dO; write dq, dk,
    dz, dv and dbeta."""
    return 2 * ((3 * dk + dv) * io_bytes + 4) + dv * io_bytes


def bench_backward(B, I, dev, stream, max_over_ranks, barrier, pk, pk_src, reps=10):
    """kda_backward at the 4096-token, 16-head, d = 128 bf16 shape (its workspace of per-chunk states
    is ~0.7 GB, larger than L2, so no flush is needed)."""
    import torch
    d = device_workload(I, 1, dev)
    T, H, dk = d["k"].shape
    dv = d["v"].shape[2]
    g = torch.Generator(device=dev).manual_seed(11)
    do = torch.randn(T, H, dv, generator=g, device=dev).to(d["k"].dtype)
    dsf = torch.randn(1, H, dk, dv, generator=g, device=dev) * 0.1
    prob = B.make_problem(1, T, T, H, dk, dv, d["k"].dtype)
    ws = torch.empty(B.kda_backward_workspace_bytes(prob), dtype=torch.uint8, device=dev)

    def bwd():
        B.kda_backward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], do, dsf, initial_state=d["S0"],
                       workspace=ws)
    for _ in range(3):
        bwd()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        bwd()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / reps)
    B.kda_profile_enable(True)
    for _ in range(reps):
        bwd()
    torch.cuda.synchronize()
    prof = B.kda_profile_read()
    B.kda_profile_enable(False)
    th = T * H
    nbytes = th * backward_bytes_per_token_head(dk, dv, 2) + 3 * H * dk * dv * 4
    kernels = {n: {"launches_per_step": c / reps, "avg_ms": t / c} for n, (c, t) in prof.items()}
    top = max(prof.items(), key=lambda kv: kv[1][1])[0]
    achieved = nbytes / (kernels[top]["avg_ms"] * 1e-3) / 1e9
    return {"workload": d["name"] + ", gradients of every input", "ms_per_step": ms,
            "value": T / (ms * 1e-3) / 1e6, "unit": "Mtok/s", "workspace_bytes": ws.numel(),
            "roofline": {"bound": "hbm", "kernel": top, "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / pk["hbm_gbs"], "algorithmic_bytes_per_launch": nbytes,
                         "bytes_per_unit": backward_bytes_per_token_head(dk, dv, 2), "units_per_launch": th,
                         "peak_source": pk_src, "path_frac": nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                         "kernels": kernels},
            "gpu_launches": sum(c for c, _ in prof.values()) // reps}


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
                     "frac": gbs / pk["hbm_gbs"], "traffic": layer_traffic(f"kda_{name}", T * H)}
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


class E2EPipeline:
    """Prefill requests from pinned host memory through kda_forward and back: every step copies its
    inputs from one pinned host buffer to one of `depth` device buffer sets, runs the prefill and
    copies the outputs and final states back to pinned host memory, over three CUDA streams (step
    i+1's inputs travel while step i computes and step i-1's outputs travel back).  Inputs are
    packed back to back in the host buffer (256-byte aligned) and the call gets views of the device
    copy.  `outputs()` are views of the pinned output buffer (valid after a synchronize)."""

    KEYS = ("q", "k", "v", "z", "A", "beta", "S0")

    def __init__(self, B, d, dev, depth=2):
        import torch
        self.B, self.depth, self.dev = B, depth, dev
        T, H, dk = d["k"].shape
        dv = d["v"].shape[2]
        N = len(d["lengths"])
        io = d["k"].dtype
        shapes = {k: (d[k].dtype, d[k].shape, d[k].numel() * d[k].element_size()) for k in self.KEYS}
        offs, total = {}, 0
        for k in self.KEYS:
            offs[k] = total
            total += (shapes[k][2] + 255) // 256 * 256

        def views(buf):
            return {k: buf[offs[k]:offs[k] + shapes[k][2]].view(shapes[k][0]).view(shapes[k][1]) for k in self.KEYS}
        self.h_all = torch.empty(total, dtype=torch.uint8).pin_memory()
        host = views(self.h_all)
        for k in self.KEYS:
            host[k].copy_(d[k])
        self.d_all = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(depth)]
        self.dbuf = [views(x) for x in self.d_all]
        o_bytes = T * H * dv * d["k"].element_size()
        f_off = (o_bytes + 255) // 256 * 256
        o_total = f_off + N * H * dk * dv * 4

        def out_views(buf):
            return (buf[:o_bytes].view(io).view(T, H, dv), buf[f_off:o_total].view(torch.float32).view(N, H, dk, dv))
        self.d_out_all = [torch.empty(o_total, dtype=torch.uint8, device=dev) for _ in range(depth)]
        self.dout = [out_views(x) for x in self.d_out_all]
        self.h_out_all = torch.empty(o_total, dtype=torch.uint8).pin_memory()
        self.host_out = out_views(self.h_out_all)
        self.h2d_bytes, self.d2h_bytes = total, o_total
        self.ml = max(d["lengths"])
        prob = B.make_problem(N, T, self.ml, H, dk, dv, io)
        self.ws = torch.empty(B.kda_forward_workspace_bytes(prob), dtype=torch.uint8, device=dev)
        self.cu = d["cu_seqlens"]
        self.s_in, self.s_cmp, self.s_out = (torch.cuda.Stream(dev) for _ in range(3))
        self.ev_in = [torch.cuda.Event() for _ in range(depth)]
        self.ev_cmp = [torch.cuda.Event() for _ in range(depth)]
        self.ev_out = [torch.cuda.Event() for _ in range(depth)]
        self.count = 0

    def step(self):
        import torch
        i, depth = self.count, self.depth
        b = i % depth
        with torch.cuda.stream(self.s_in):
            if i >= depth:
                self.s_in.wait_event(self.ev_cmp[b])   # the compute of step i - depth has read these inputs
            self.d_all[b].copy_(self.h_all, non_blocking=True)
            self.ev_in[b].record(self.s_in)
        with torch.cuda.stream(self.s_cmp):
            self.s_cmp.wait_event(self.ev_in[b])
            if i >= depth:
                self.s_cmp.wait_event(self.ev_out[b])  # the outputs of step i - depth have left
            x = self.dbuf[b]
            self.B.kda_forward(x["q"], x["k"], x["v"], x["z"], x["A"], x["beta"], initial_state=x["S0"],
                               cu_seqlens=self.cu, out=self.dout[b][0], final_state=self.dout[b][1],
                               max_seqlen=self.ml, workspace=self.ws, stream=self.s_cmp)
            self.ev_cmp[b].record(self.s_cmp)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.ev_cmp[b])
            self.h_out_all.copy_(self.d_out_all[b], non_blocking=True)
            self.ev_out[b].record(self.s_out)
        self.count += 1

    def outputs(self):
        return self.host_out


def bench_e2e(args, B, d, dev, max_over_ranks, barrier, world, depth=2):
    """The prefill end to end through kda_forward with host buffers (E2EPipeline: inputs uploaded,
    outputs and final states downloaded every step); the time per step is the steady-state spacing."""
    import torch
    T = d["k"].shape[0]
    pipe = E2EPipeline(B, d, dev, depth)
    for _ in range(3):
        pipe.step()
    torch.cuda.synchronize()
    barrier()
    steps = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.s_in)
    # each step's upload end: the uploads are the pipeline's bottleneck and run back to back, so the
    # spacing between consecutive ends is the step time in the steady state
    ends = []
    for _ in range(steps):
        pipe.step()
        ends.append(torch.cuda.Event(enable_timing=True))
        ends[-1].record(pipe.s_in)
    e1.record(pipe.s_out)
    torch.cuda.synchronize()
    barrier()
    mean_ms = max_over_ranks(e0.elapsed_time(e1) / steps)
    spacing = [e0.elapsed_time(ends[0])] + [ends[i - 1].elapsed_time(ends[i]) for i in range(1, steps)]
    ms = max_over_ranks(statistics.median(spacing))
    res = {"value": T * world / (ms * 1e-3) / 1e6, "unit": "Mtok/s", "h2d_bytes_per_step": pipe.h2d_bytes,
           "d2h_bytes_per_step": pipe.d2h_bytes, "ms_per_step": ms, "steps": steps,
           "statistic": "median of the per-step spacings (upload end to upload end); the mean over the "
                        "window, last step's compute and download included, is beside it",
           "mean_ms_per_step": mean_ms, "mean_value": T * world / (mean_ms * 1e-3) / 1e6,
           "step_spacing_ms": [round(x, 2) for x in spacing],
           "pipeline": f"{depth} device buffer sets over H2D / compute / D2H streams; one copy each way per step"}
    del pipe
    return res


if __name__ == "__main__":
    sys.exit(main())
