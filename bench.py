"""Benchmark: Llama-3-8B-shaped tensor-parallel MLP layer, decode, t=8 logical shards on one GPU.

One step = one SwiGLU MLP forward (column-parallel gate/up + SwiGLU, row-parallel down +
fixed-order shard fold + residual) through tp_mlp_forward for each decode batch M in
{1, 8, 32, 64}: 105 tokens.  By default each forward is one fused block launch.
Weights are 352 MB (> 129 MB L2), read once per forward, so no L2 flush is needed between
forwards.  Prints one JSON line (see the fields below).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tpx|reference]

--impl reference times the float64 CPU oracle on this host on a bounded sample of the same
workload (there is no reference GPU implementation to run).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

D, FFN, T = 4096, 14336, 8
MS = (1, 8, 32, 64)
METRIC = "decode tokens/s and HBM GB/s (% peak); prefill TFLOP/s (% peak) per TP layer"
WORKLOAD = "llama3-8b MLP layer decode (d 4096, ffn 14336, t 8 logical shards), M in {1,8,32,64}"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j["hbm_gbs"], "measured"
    return 6800.0, "fallback"


def weight_bytes():
    return 3 * D * FFN * 2


def block_bytes(M):      # all three weights + x in + residual in + y out (h stays on chip/L2)
    return 3 * D * FFN * 2 + 3 * M * D * 2


class Clocks:
    """nvidia-smi samples during the timed region."""

    def __init__(self, path):
        self.path, self.p = path, None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                       "-i", os.environ.get("LOCAL_RANK", "0"), "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        t0 = time.time()          # wait for the first sample so the timed region is covered
        while self.p and time.time() - t0 < 3.0:
            if os.path.exists(self.path) and os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)
        return self

    def __exit__(self, *a):
        if self.p:
            self.p.terminate()
            self.p.wait()
            self.f.close()

    def summary(self):
        try:
            rows = [l.split(",") for l in open(self.path).read().splitlines() if l.strip()]
        except OSError:
            rows = []
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) >= 9 for i in range(4)
                          if "Active" in r[5 + i] and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("BENCH_BACKEND") != "gloo" else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, dev):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def traffic_record():
    """Per-launch DRAM traffic of the dominant kernel from the committed ncu summary, if the
    kernel's source file is unchanged since the counters were taken (else None)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    src = os.path.join(ROOT, "megatron_tensor_transformer_gb300", "csrc", rec.get("source", ""))
    if not os.path.isfile(src):
        return None
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    return rec if rec.get("sha256") == h else None


def oracle_sample(wg, wu, wd, seconds=10.0):
    """CPU oracle on this host: the same four decode batches, repeated for about `seconds`."""
    import numpy as np
    from megatron_tensor_transformer_gb300 import inputs
    from oracle import tp_oracle as O
    xs = [O.as_f64(inputs.normal_bf16((M, D), 1.0, 0, inputs.STREAM_X, "cpu").view(
        __import__("torch").int16).numpy().view(np.uint16)) for M in MS]
    toks, t0, reps = 0, time.perf_counter(), 0
    while True:
        for x in xs:
            O.mlp(x, wg, wu, wd, residual=x)
            toks += x.shape[0]
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return toks / el, reps, el


def host_weights():
    """The benchmark's weights, drawn on the device, as float64 arrays for the oracle."""
    import numpy as np
    import torch
    from megatron_tensor_transformer_gb300 import inputs
    from oracle import tp_oracle as O
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    _, wg, wu, wd = inputs.mlp_inputs(D, FFN, 1, seed=0, device=dev)
    f = lambda w: O.as_f64(w.cpu().view(torch.int16).numpy().view(np.uint16))
    return f(wg), f(wu), f(wd)


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, rank, world):
    if rank != 0:
        return
    wg, wu, wd = host_weights()
    for _ in range(args.warmup):
        oracle_sample(wg, wu, wd, seconds=0.0)
    t0 = time.perf_counter()
    toks = 0
    for _ in range(args.steps):
        v, reps, el = oracle_sample(wg, wu, wd, seconds=0.0)
        toks += sum(MS) * reps
    el = time.perf_counter() - t0
    value = toks / el
    sample = "one step = the four decode batches M=1,8,32,64 of the 8B MLP, float64, unsharded"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "tokens_per_step": sum(MS)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_tpx(args, rank, world, local):
    import torch
    from megatron_tensor_transformer_gb300 import inputs, tpx

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    tpx.lib()
    _, wg, wu, wd = inputs.mlp_inputs(D, FFN, 1, seed=0, device=dev)
    sh = tpx.make_shape(D, ffn=FFN, t=T)
    stream = torch.cuda.Stream(device=dev)
    gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu, stream=stream)
    dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd, stream=stream)
    stream.synchronize()
    del wg, wu, wd
    xs = {M: inputs.normal_bf16((M, D), 1.0, 0, inputs.STREAM_X, dev) for M in MS}
    hs = {M: torch.empty((M, FFN), dtype=torch.bfloat16, device=dev) for M in MS}
    ys = {M: torch.empty((M, D), dtype=torch.bfloat16, device=dev) for M in MS}
    ws = tpx.new_workspace(sh, max(MS), dev)
    kf = {"auto": 0, "tc": tpx.TP_F_KERNEL_TC, "skinny": tpx.TP_F_KERNEL_SKINNY,
          "split": tpx.TP_F_SPLIT_BLOCK, "hilo": tpx.TP_F_FP8_HILO}[args.kernel]
    K = args.steps
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in MS] for _ in range(K)]

    def step(i=None):
        for j, M in enumerate(MS):
            if i is not None:
                ev[i][j][0].record(stream)
            tpx.tp_mlp_forward(gu, gu_w, dn, dn_w, xs[M], xs[M], ys[M], hs[M], ws, flags=kf, stream=stream)
            if i is not None:
                ev[i][j][1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = tpx.tp_launch_count()
        with Clocks(os.path.join(ROOT, "gpurun_out", f"clocks_rank{rank}.csv") if os.path.isdir(
                os.path.join(ROOT, "gpurun_out")) else f"/tmp/tpx_clocks_{os.getpid()}.csv") as clk:
            t_start.record(stream)
            for i in range(K):
                step()          # no events between kernels: consecutive kernels may overlap
            t_end.record(stream)
            t_end.synchronize()
        launches = tpx.tp_launch_count() - n0
        torch.cuda.synchronize()
        barrier(world)
        # second pass, same work, with an event around every forward: per-forward durations
        for i in range(K):
            step(i)
        torch.cuda.synchronize()
    ms = t_start.elapsed_time(t_end)
    ms_max = max_over_ranks(ms, world, dev)
    per_M = {}
    blk_t = blk_b = 0.0
    for j, M in enumerate(MS):
        c = sum(ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(K)) / K
        blk_t += c
        blk_b += block_bytes(M)
        per_M[str(M)] = {"tokens_per_s": M / (c * 1e-3), "block_us": 1e3 * c,
                         "block_gbs": block_bytes(M) / (c * 1e-3) / 1e9}
    peak, peak_kind = peaks()
    achieved = blk_b / (blk_t * 1e-3) / 1e9
    tr = traffic_record()
    e2e = run_e2e(args, gu, gu_w, dn, dn_w, sh, dev)
    cpu = None  # after every timed region: the oracle's host threads must not share the CPU with them
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        wg, wu, wd = host_weights()
        v, reps, el = oracle_sample(wg, wu, wd, seconds=args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
               "sample": f"{reps} repetitions of the four decode batches M=1,8,32,64 (float64, unsharded "
                         f"8B MLP incl. residual) in {el:.1f} s"}
        del wg, wu, wd
    tokens = sum(MS) * K * world
    step_bytes = sum(block_bytes(M) for M in MS)
    kname = {"auto": "fused_kernel (whole MLP block, one launch per forward)", "tc": "fused_kernel",
             "skinny": "colpar/rowpar mma.sync kernels + fold", "split": "tc_kernel x2 + fold"}[args.kernel]
    out = {
        "metric": METRIC, "value": tokens / (ms_max * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "d": D, "ffn": FFN, "t": T, "M": list(MS),
                   "tokens_per_step": sum(MS), "parallelism": "replicas" if world > 1 else "single",
                   "l2": "weights 352 MB per forward > 129 MB L2; no flush", "kernel": args.kernel},
        "hbm_gbs_step": step_bytes / (ms_max / K * 1e-3) / 1e9,
        "hbm_frac_step": step_bytes / (ms_max / K * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved,
                     "peak": peak, "peak_kind": peak_kind + " (hbm_gbs, burst)", "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": None if tr is None else tr.get("bytes_per_launch")},
        "per_M": per_M,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


LAYERS = {
    # name: (d, ffn, n_q, n_kv, hd, t, M, weights: 0 bf16, 1 e4m3, 2 e4m3 with e4m3 activations)
    "70b-layer-decode": (8192, 28672, 64, 8, 128, 8, 32, 0),
    "70b-layer-prefill": (8192, 28672, 64, 8, 128, 8, 4096, 0),
    "70b-fp8-decode": (8192, 28672, 64, 8, 128, 8, 16, 1),
    "70b-fp8-prefill": (8192, 28672, 64, 8, 128, 8, 8192, 1),
    "70b-fp8x-decode": (8192, 28672, 64, 8, 128, 8, 16, 2),
    "70b-fp8x-prefill": (8192, 28672, 64, 8, 128, 8, 8192, 2),
    "405b-layer-decode": (16384, 53248, 128, 8, 128, 8, 16, 0),
}


def layer_params(d, ffn, n_q, n_kv, hd):
    return d * (n_q + 2 * n_kv) * hd + n_q * hd * d + 3 * d * ffn


def run_layer(args, rank, world, local):
    """One 70B-shaped layer's linear parts: y1 = x + o_proj(attn(qkv(x))); y = y1 + MLP(y1),
    t logical shards, bf16, through tp_proj_forward and tp_mlp_forward.  Decode is reported in
    tokens/s and HBM GB/s, prefill in TFLOP/s (2 flops per weight per token)."""
    import torch
    from megatron_tensor_transformer_gb300 import inputs, tpx

    d, ffn, n_q, n_kv, hd, t, M, wkind = LAYERS[args.workload]
    fp8, x8 = wkind >= 1, wkind == 2
    if args.t:
        t = args.t
    prefill = "prefill" in args.workload
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    sh = tpx.make_shape(d, ffn=ffn, n_q=n_q, n_kv=n_kv, hd=hd, t=t,
                        wtype=tpx.TP_FP8_E4M3 if fp8 else tpx.TP_BF16)
    _, wg, wu, wd = inputs.mlp_inputs(d, ffn, 1, seed=0, device=dev)
    gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu, stream=stream)
    dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd, stream=stream)
    del wg, wu, wd
    _, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, 1, seed=0, device=dev)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv, stream=stream)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo, stream=stream)
    del wqkv, wo
    Q = (n_q + 2 * n_kv) * hd
    x = inputs.normal_bf16((M, d), 1.0, 0, inputs.STREAM_X, dev)
    y1, y = torch.empty_like(x), torch.empty_like(x)
    qkv = torch.empty((M, Q), dtype=torch.bfloat16, device=dev)
    o_in = torch.empty((M, n_q * hd), dtype=torch.bfloat16, device=dev)
    h = torch.empty((M, ffn), dtype=torch.bfloat16, device=dev)
    K = args.steps
    kf = {"auto": 0, "tc": tpx.TP_F_KERNEL_TC, "skinny": tpx.TP_F_KERNEL_SKINNY,
          "split": tpx.TP_F_SPLIT_BLOCK, "hilo": tpx.TP_F_FP8_HILO}[args.kernel] | (tpx.TP_F_FP8_ACT if x8 else 0)
    ws = tpx.new_workspace(sh, M, dev, flags=kf)

    def step():
        tpx.tp_proj_forward(q, q_w, o, o_w, x, x, y1, qkv, o_in, ws, flags=kf, stream=stream)
        tpx.tp_mlp_forward(gu, gu_w, dn, dn_w, y1, y1, y, h, ws, flags=kf, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = tpx.tp_launch_count()
        with Clocks(f"/tmp/tpx_clocks_{os.getpid()}.csv") as clk:
            a.record(stream)
            for _ in range(K):
                step()
            b.record(stream)
            b.synchronize()
        launches = tpx.tp_launch_count() - n0
        # dominant kernel alone: decode, the MLP block (one fused launch for bf16 weights);
        # prefill, the MLP's column-parallel gate/up + SwiGLU
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(K):
            if prefill:
                tpx.tp_colpar_forward(gu, gu_w, y1, h, flags=kf & ~tpx.TP_F_SPLIT_BLOCK, stream=stream, ws=ws)
            else:
                tpx.tp_mlp_forward(gu, gu_w, dn, dn_w, y1, y1, y, h, ws, flags=kf, stream=stream)
        c1.record(stream)
        c1.synchronize()
    ms = a.elapsed_time(b) / K
    col_ms = c0.elapsed_time(c1) / K
    params = layer_params(d, ffn, n_q, n_kv, hd)
    flops = 2.0 * params * M
    wb = 1.0 if fp8 else 2.0          # bytes per weight
    wbytes = wb * params
    col_flops = 2.0 * 2 * d * ffn * M
    col_bytes = wb * 3 * d * ffn + 2.0 * 3 * M * d     # decode: the whole MLP block
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        pk = json.load(f)
    # the contraction's own peak: e4m3 x e4m3 runs at twice the bf16 rate (nominal 4.5 / 2.25
    # PFLOP/s), so its denominator is the measured bf16 peak times two
    tpeak = pk["bf16_tflops"] * (2.0 if x8 else 1.0)
    dtype = "e4m3 weights x e4m3 activations (per token)" if x8 else ("e4m3 weights, bf16 math" if fp8 else "bf16")
    out = {"metric": METRIC, "workload": args.workload, "n_gpus": 1, "steps": K, "warmup": args.warmup,
           "ms_per_step": ms, "dtype": dtype, "data": "synthetic",
           "config": {"workload": args.workload, "d": d, "ffn": ffn, "n_q": n_q, "n_kv": n_kv,
                      "head_dim": hd, "t": t, "M": M, "kernel": args.kernel},
           "gpu_launches": launches, "clocks": clk.summary()}
    if prefill:
        out.update({"value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "higher_is_better": True,
                    "tflop_per_step": flops / 1e12,
                    "roofline": {"bound": "tensor", "kernel": "tc_kernel (gate/up + SwiGLU)",
                                 "achieved": col_flops / (col_ms * 1e-3) / 1e12, "peak": tpeak,
                                 "peak_kind": "measured bf16 x 2 (e4m3)" if x8 else "measured bf16",
                                 "unit": "TFLOP/s", "frac": col_flops / (col_ms * 1e-3) / 1e12 / tpeak,
                                 "layer_frac": flops / (ms * 1e-3) / 1e12 / tpeak}})
    else:
        out.update({"value": M / (ms * 1e-3), "unit": "tokens/s", "higher_is_better": True,
                    "hbm_gbs_step": wbytes / (ms * 1e-3) / 1e9,
                    "roofline": {"bound": "hbm", "kernel": "MLP block (tp_mlp_forward)",
                                 "achieved": col_bytes / (col_ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"],
                                 "unit": "GB/s", "frac": col_bytes / (col_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                                 "layer_frac": wbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]}})
    print(json.dumps(out), flush=True)


def run_stack(args, rank, world, local):
    """Pipeline-stage stack: 10 consecutive 405B-shaped layers (d 16384, ffn 53248, 128 q / 8 kv
    heads of 128), linear parts + RMSNorm + residual, t=8, bf16, decode M=16, through
    tp_layer_forward.  63.75 GB of weights, read once per step."""
    import torch
    from megatron_tensor_transformer_gb300 import inputs, tpx

    d, ffn, n_q, n_kv, hd, t, M, nl = 16384, 53248, 128, 8, 128, args.t or 8, 16, 10
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    sh = tpx.make_shape(d, ffn=ffn, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    layers = []
    for L in range(nl):
        _, wg, wu, wd = inputs.mlp_inputs(d, ffn, 1, seed=0, device=dev, layer=L)
        gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu, stream=stream)
        dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd, stream=stream)
        del wg, wu, wd
        _, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, 1, seed=0, device=dev, layer=L)
        q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv, stream=stream)
        o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo, stream=stream)
        del wqkv, wo
        layers.append((q, q_w, o, o_w, gu, gu_w, dn, dn_w))
        torch.cuda.empty_cache()
    x0 = inputs.normal_bf16((M, d), 1.0, 0, inputs.STREAM_X, dev)
    xa, xb = x0.clone(), torch.empty_like(x0)
    scratch = torch.empty(tpx.tp_layer_scratch_bytes(sh, M), dtype=torch.uint8, device=dev)
    ws = tpx.new_workspace(sh, M, dev)
    K = args.steps

    def step():
        cur, nxt = xa, xb
        for lay in layers:
            tpx.tp_layer_forward(*lay, cur, nxt, scratch, ws, stream=stream)
            cur, nxt = nxt, cur

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            xa.copy_(x0)
            step()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = tpx.tp_launch_count()
        with Clocks(f"/tmp/tpx_clocks_{os.getpid()}.csv") as clk:
            a.record(stream)
            for _ in range(K):
                step()
            b.record(stream)
            b.synchronize()
        launches = tpx.tp_launch_count() - n0
    ms = a.elapsed_time(b) / K
    wbytes = 2.0 * nl * layer_params(d, ffn, n_q, n_kv, hd)
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        pk = json.load(f)
    print(json.dumps({
        "metric": METRIC, "workload": "405b-stack-decode", "value": M / (ms * 1e-3), "unit": "tokens/s",
        "higher_is_better": True, "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "405b-stack-decode", "layers": nl, "d": d, "ffn": ffn, "n_q": n_q, "n_kv": n_kv,
                   "head_dim": hd, "t": t, "M": M},
        "weight_gb": wbytes / 1e9, "hbm_gbs_step": wbytes / (ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "whole stack", "achieved": wbytes / (ms * 1e-3) / 1e9,
                     "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": wbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
        "gpu_launches": launches, "clocks": clk.summary()}), flush=True)


def run_lm_head(args, rank, world, local):
    """Llama-3 70B output layer: the vocabulary-parallel lm_head (d 8192, 128256 ids over t=8
    shards, padded to 16128 per shard), decode M=32, fp32 logits, through tp_lm_head_forward;
    plus the vocabulary-parallel embedding lookup of the same tokens."""
    import torch
    from megatron_tensor_transformer_gb300 import inputs, tpx

    d, V, t, M = 8192, 128256, args.t or 8, 32
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    sh = tpx.make_shape(d, t=t, vocab=V)
    w = inputs.normal_bf16((d, V), 0.02, 0, 70, dev)
    w_p, wd = tpx.tp_partition_weights(sh, tpx.TP_W_VOCAB, w, stream=stream)
    del w
    e = inputs.normal_bf16((V, d), 1.0, 0, 71, dev)
    e_p, ed = tpx.tp_partition_weights(sh, tpx.TP_W_EMBED, e, stream=stream)
    del e
    torch.cuda.empty_cache()
    ids = torch.randint(0, V, (M,), generator=torch.Generator(device=dev).manual_seed(0), device=dev,
                        dtype=torch.int32)
    x = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
    logits = torch.empty((M, V), dtype=torch.float32, device=dev)
    ws = tpx.new_workspace(sh, M, dev)
    K = args.steps

    def step():
        tpx.tp_embed_lookup(ed, e_p, ids, x, stream=stream)
        tpx.tp_lm_head_forward(wd, w_p, x, logits, ws=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = tpx.tp_launch_count()
        with Clocks(f"/tmp/tpx_clocks_{os.getpid()}.csv") as clk:
            a.record(stream)
            for _ in range(K):
                step()
            b.record(stream)
            b.synchronize()
        launches = tpx.tp_launch_count() - n0
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(K):
            tpx.tp_lm_head_forward(wd, w_p, x, logits, ws=ws, stream=stream)
        c1.record(stream)
        c1.synchronize()
    ms, head_ms = a.elapsed_time(b) / K, c0.elapsed_time(c1) / K
    wbytes = 2.0 * d * V                         # the lm_head weights, read once
    head_bytes = wbytes + 2.0 * M * d + 4.0 * M * V
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        pk = json.load(f)
    print(json.dumps({
        "metric": METRIC, "workload": "70b-lm-head-decode", "value": M / (ms * 1e-3), "unit": "tokens/s",
        "higher_is_better": True, "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "70b-lm-head-decode", "d": d, "vocab": V, "t": t, "M": M},
        "hbm_gbs_step": wbytes / (ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "tc_kernel (vocabulary-parallel lm_head)",
                     "achieved": head_bytes / (head_ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": head_bytes / (head_ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
        "gpu_launches": launches, "clocks": clk.summary()}), flush=True)


def run_attn(args, rank, world, local):
    """Llama-3.1 70B attention block with a real KV cache: 32 sequences, each with 4095 cached
    positions (4096 with the new token), t=8.  One step = one tp_attn_block_forward: QKV
    (column-parallel) + the head-sharded decode attention over the cache + o_proj (row-parallel,
    shard fold, residual).  The roofline kernel is the attention (cache reads: M x n_kv x 4096 x
    hd x 2 x 2 bytes)."""
    import torch
    from megatron_tensor_transformer_gb300 import inputs, tpx

    d, n_q, n_kv, hd, t, M, L = 8192, 64, 8, 128, args.t or 8, 32, 4096
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    x, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, M, seed=0, device=dev)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv, stream=stream)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo, stream=stream)
    del wqkv, wo
    kc = inputs.normal_bf16((t, M, n_kv // t, L, hd), 1.0, 0, 90, dev)
    vc = inputs.normal_bf16((t, M, n_kv // t, L, hd), 1.0, 0, 91, dev)
    lens = torch.full((M,), L - 1, dtype=torch.int32, device=dev)
    qkv = torch.empty((M, (n_q + 2 * n_kv) * hd), dtype=torch.bfloat16, device=dev)
    o_in = torch.empty((M, n_q * hd), dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(x)
    bws = tpx.new_attn_block_workspace(sh, M, L, dev)
    aws = torch.empty(tpx.tp_attn_workspace_bytes(sh, M, L), dtype=torch.uint8, device=dev)
    K = args.steps

    def step():
        tpx.tp_attn_block_forward(q, q_w, o, o_w, x, x, kc, vc, lens, y, qkv, o_in, bws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = tpx.tp_launch_count()
        with Clocks(f"/tmp/tpx_clocks_{os.getpid()}.csv") as clk:
            a.record(stream)
            for _ in range(K):
                step()
            b.record(stream)
            b.synchronize()
        launches = tpx.tp_launch_count() - n0
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(K):
            tpx.tp_attn_decode(sh, qkv, kc, vc, lens, o_in, aws, stream=stream)
        c1.record(stream)
        c1.synchronize()
    ms, attn_ms = a.elapsed_time(b) / K, c0.elapsed_time(c1) / K
    cache_bytes = 2.0 * M * n_kv * L * hd * 2
    w_bytes = 2.0 * ((n_q + 2 * n_kv) * hd * d + n_q * hd * d)
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        pk = json.load(f)
    print(json.dumps({
        "metric": METRIC, "workload": "70b-attn-decode", "value": M / (ms * 1e-3), "unit": "tokens/s",
        "higher_is_better": True, "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "70b-attn-decode", "d": d, "n_q": n_q, "n_kv": n_kv, "head_dim": hd, "t": t,
                   "M": M, "context": L},
        "hbm_gbs_step": (cache_bytes + w_bytes) / (ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "decode attention (append + attention pass)",
                     "achieved": cache_bytes / (attn_ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": cache_bytes / (attn_ms * 1e-3) / 1e9 / pk["hbm_gbs"], "attn_us": 1e3 * attn_ms},
        "gpu_launches": launches, "clocks": clk.summary()}), flush=True)


def run_e2e(args, gu, gu_w, dn, dn_w, sh, dev):
    """Through the public C-ABI call tp_mlp_forward with HOST buffers: every step copies each
    batch's x from pinned host memory, runs the block, and copies y back."""
    import torch
    from megatron_tensor_transformer_gb300 import inputs, tpx
    stream = torch.cuda.Stream(device=dev)
    hx = {M: inputs.normal_bf16((M, D), 1.0, 0, inputs.STREAM_X, "cpu").pin_memory() for M in MS}
    hy = {M: torch.empty((M, D), dtype=torch.bfloat16).pin_memory() for M in MS}
    dx = {M: torch.empty((M, D), dtype=torch.bfloat16, device=dev) for M in MS}
    dy = {M: torch.empty((M, D), dtype=torch.bfloat16, device=dev) for M in MS}
    dh = {M: torch.empty((M, FFN), dtype=torch.bfloat16, device=dev) for M in MS}
    ws = tpx.new_workspace(sh, max(MS), dev)

    def step():
        for M in MS:
            dx[M].copy_(hx[M], non_blocking=True)
            tpx.tp_mlp_forward(gu, gu_w, dn, dn_w, dx[M], dx[M], dy[M], dh[M], ws, stream=stream)
            hy[M].copy_(dy[M], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        b.synchronize()
    ms = a.elapsed_time(b)
    nbytes = sum(M * D * 2 for M in MS)
    return {"value": sum(MS) * args.steps / (ms * 1e-3), "unit": "tokens/s",
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="tpx", choices=["tpx", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="8b-mlp-decode",
                    choices=["8b-mlp-decode", "405b-stack-decode", "70b-lm-head-decode", "70b-attn-decode"] +
                    sorted(LAYERS),
                    help="the headline 8B MLP decode, or a 70B-shaped layer (QKV/o_proj/MLP)")
    ap.add_argument("--t", type=int, default=0, help="shard count for the layer workloads (default: 8)")
    ap.add_argument("--kernel", default="auto", choices=["auto", "tc", "skinny", "split", "hilo"],
                    help="force the tcgen05 or the mma.sync decode kernels, or separate launches for the "
                         "two halves of a block (default: library policy, one fused launch per block)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_setup()
    if args.workload == "405b-stack-decode":
        run_stack(args, rank, world, local)
    elif args.workload == "70b-lm-head-decode":
        run_lm_head(args, rank, world, local)
    elif args.workload == "70b-attn-decode":
        run_attn(args, rank, world, local)
    elif args.workload != "8b-mlp-decode":
        run_layer(args, rank, world, local)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_tpx(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
