"""Benchmark: Megatron-style tensor-parallel layers of Llama-shaped models, t logical shards on one GPU.

Default run: every configuration of the workload set, each timed on the device, through the
public C ABI with host buffers (e2e), against its dominant kernel's roofline, and beside the
float64 CPU oracle on this host's cores (all of them, and one):

  8b-mlp-decode       Llama-3-8B MLP (d 4096, ffn 14336, t 8), decode M in {1, 8, 32, 64}
  70b-layer-decode    Llama-3.1-70B layer (GQA QKV + o_proj + MLP, ffn 28672, t 8), M = 32, bf16
  70b-layer-prefill   the same layer, M = 4096
  70b-fp8-decode      the same layer with e4m3 weights (per-output-channel scales), M = 16
  70b-fp8-prefill     the e4m3 layer, M = 8192
  405b-stack-decode   10 consecutive 405B-shaped layers (d 16384, ffn 53248, 128 q / 8 kv heads),
                      RMSNorm + residual, t 8, M = 16 (63.75 GB of weights per step)

The JSON line's headline (value, steps, roofline, e2e, cpu_baseline, clocks) is the largest
configuration that fits one GPU, the 405B stack, timed for exactly --steps steps after --warmup;
"configs" holds one sub-record per configuration in the same form.  Decode is reported in
tokens/s and HBM GB/s, prefill in TFLOP/s (2 flops per weight per token).  Every configuration
streams more than the 129 MB L2 per step, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tpx|reference] [--workload NAME]

--workload runs one configuration (or one of the extra ones: 70b-fp8x-*, 405b-layer-decode,
70b-prenorm-prefill, 70b-lm-head-decode, 70b-attn-decode) and prints its record as the line.  --impl reference times
the float64 CPU oracle on a bounded sample of the headline workload (there is no reference GPU
implementation to run).
"""
import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s and HBM GB/s (% peak); prefill TFLOP/s (% peak) per TP layer"
HEADLINE = "405b-stack-decode"
DEFAULT_SET = ["8b-mlp-decode", "70b-layer-decode", "70b-layer-prefill", "70b-fp8-decode",
               "70b-fp8-prefill", "405b-stack-decode"]

# name: (d, ffn, n_q, n_kv, hd, t, M, weights: 0 bf16, 1 e4m3, 2 e4m3 with e4m3 activations, layers)
LAYERS = {
    "70b-layer-decode": (8192, 28672, 64, 8, 128, 8, 32, 0, 1),
    "70b-layer-prefill": (8192, 28672, 64, 8, 128, 8, 4096, 0, 1),
    "70b-fp8-decode": (8192, 28672, 64, 8, 128, 8, 16, 1, 1),
    "70b-fp8-prefill": (8192, 28672, 64, 8, 128, 8, 8192, 1, 1),
    "70b-fp8x-decode": (8192, 28672, 64, 8, 128, 8, 16, 2, 1),
    "70b-fp8x-prefill": (8192, 28672, 64, 8, 128, 8, 8192, 2, 1),
    "405b-layer-decode": (16384, 53248, 128, 8, 128, 8, 16, 0, 1),
    "405b-stack-decode": (16384, 53248, 128, 8, 128, 8, 16, 0, 10),
    "70b-prenorm-prefill": (8192, 28672, 64, 8, 128, 8, 4096, 0, 1),
}
# run through tp_layer_forward (pre-norm layers: RMSNorm + residual around both blocks)
PRENORM = {"405b-stack-decode", "70b-prenorm-prefill"}
MLP8B = (4096, 14336, 8, (1, 8, 32, 64))
EXTRA = ["70b-lm-head-decode", "70b-attn-decode"]


# ------------------------------------------------------------------------------------------ host


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm": j["hbm_gbs"], "bf16": j["bf16_tflops"], "bf16_sustained": j.get("bf16_tflops_sustained"),
                "kind": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "kind": "fallback"}


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


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


class Clocks:
    """SM clocks and throttle reasons sampled while the timed region runs: NVML (read-only
    queries, through ctypes) every 20 ms on a thread, or nvidia-smi every 100 ms where NVML
    cannot be loaded.  The device is found by its PCI bus id."""

    # clock-event reason bits of NVML
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev):
        self.dev, self.rows, self.stop, self.th, self.proc, self.path = dev, [], threading.Event(), None, None, None

    def _bus_id(self):
        import torch
        p = torch.cuda.get_device_properties(self.dev)
        try:
            return "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except AttributeError:
            return None

    def _nvml(self):
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if nv.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        bus = self._bus_id()
        ok = bus is not None and nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(int(os.environ.get("LOCAL_RANK", "0")), ctypes.byref(h)) != 0:
            return None
        reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return nv, h, reasons

    def _loop(self, nv, h, reasons):
        sm, mx, r = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        while not self.stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and reasons(h, ctypes.byref(r)) == 0:
                self.rows.append((float(sm.value), float(mx.value), int(r.value)))
            self.stop.wait(0.02)

    def __enter__(self):
        got = self._nvml()
        if got:
            self.th = threading.Thread(target=self._loop, args=got, daemon=True)
            self.th.start()
            t0 = time.time()
            while not self.rows and time.time() - t0 < 1.0:
                time.sleep(0.005)
            return self
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="tpx_clocks_", suffix=".csv")
        self.f = os.fdopen(fd, "w")
        sel = self._bus_id() or os.environ.get("LOCAL_RANK", "0")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-i",
                                          sel, "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        t0 = time.time()
        while self.proc and time.time() - t0 < 3.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.05)
        return self

    def __exit__(self, *a):
        if self.th:
            self.stop.set()
            self.th.join()
        if self.proc:
            self.proc.terminate()
            self.proc.wait()
        if self.path:
            self.f.close()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            bits = [0x8, 0x40, 0x20, 0x4]
            for line in open(self.path).read().splitlines():
                c = [x.strip() for x in line.split(",")]
                if len(c) >= 6 and c[0].replace(".", "").isdigit():
                    r = sum(b for b, v in zip(bits, c[2:6]) if v == "Active")
                    self.rows.append((float(c[0]), float(c[1]), r))
            os.unlink(self.path)

    def summary(self):
        sm = [r[0] for r in self.rows]
        reasons = sorted({n for r in self.rows for b, n in self.REASONS.items() if r[2] & b})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[1] for r in self.rows) if self.rows else None,
                "reasons": reasons, "samples": len(sm), "source": "nvml" if self.th else "nvidia-smi"}


def traffic_record(name):
    """Per-launch DRAM bytes of a configuration's dominant kernel from the committed ncu
    summary, if that kernel's source file is unchanged since the counters were taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get("records", {}).get(name)
    if not rec:
        return None
    src = os.path.join(ROOT, "megatron_tensor_transformer_gb300", "csrc", rec.get("source", ""))
    if not os.path.isfile(src):
        return None
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    return rec.get("bytes_per_launch") if rec.get("sha256") == h else None


def layer_params(d, ffn, n_q, n_kv, hd):
    return d * (n_q + 2 * n_kv) * hd + n_q * hd * d + 3 * d * ffn


# ------------------------------------------------------------------------------- device harness


class Harness:
    """Device, stream and the timing helpers every configuration uses."""

    def __init__(self, local, world):
        import torch
        from megatron_tensor_transformer_gb300 import tpx
        self.torch, self.tpx, self.world = torch, tpx, world
        self.dev = torch.device("cuda", local)
        torch.cuda.set_device(self.dev)
        tpx.lib()
        self.stream = torch.cuda.Stream(device=self.dev)

    def ev(self):
        return self.torch.cuda.Event(enable_timing=True)

    def timed(self, K, W, step, before=None):
        """W untimed steps, then exactly K steps between two events with nothing else in between
        (consecutive kernels may overlap as they do in use); barrier + synchronize on both sides."""
        torch, tpx, s = self.torch, self.tpx, self.stream
        with torch.cuda.stream(s):
            for _ in range(W):
                if before:
                    before()
                step()
            s.synchronize()
            barrier(self.world)
            torch.cuda.synchronize()
            if before:
                before()
            a, b = self.ev(), self.ev()
            n0 = tpx.tp_launch_count()
            with Clocks(self.dev) as clk:
                a.record(s)
                for _ in range(K):
                    step()
                b.record(s)
                b.synchronize()
            launches = tpx.tp_launch_count() - n0
            torch.cuda.synchronize()
            barrier(self.world)
        ms = max_over_ranks(a.elapsed_time(b), self.world, self.dev)
        return ms, launches, clk.summary()

    def per_call_ms(self, K, call):
        """Mean duration of one call, with an event on each side of every call (no overlap
        between calls), on the stream the kernels are launched on."""
        torch, s = self.torch, self.stream
        evs = [(self.ev(), self.ev()) for _ in range(K)]
        with torch.cuda.stream(s):
            call()
            for e0, e1 in evs:
                e0.record(s)
                call()
                e1.record(s)
            s.synchronize()
        return sum(e0.elapsed_time(e1) for e0, e1 in evs) / K

    def e2e(self, K, W, batches, forward, unit_per_step, unit):
        """The same workload through the public C-ABI calls with HOST buffers: every step copies
        each batch's input from pinned host memory to the device, runs the forward, and copies
        the output back to pinned host memory, all inside the timed region."""
        torch, s = self.torch, self.stream
        hx = [x.cpu().pin_memory() for x, _ in batches]
        hy = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _, y in batches]

        def step():
            for j, (dx, dy) in enumerate(batches):
                dx.copy_(hx[j], non_blocking=True)
                forward(j)
                hy[j].copy_(dy, non_blocking=True)

        with torch.cuda.stream(s):
            for _ in range(W):
                step()
            s.synchronize()
            a, b = self.ev(), self.ev()
            a.record(s)
            for _ in range(K):
                step()
            b.record(s)
            b.synchronize()
        ms = max_over_ranks(a.elapsed_time(b), self.world, self.dev)
        nbx = sum(x.numel() * x.element_size() for x in hx)
        nby = sum(y.numel() * y.element_size() for y in hy)
        return {"value": unit_per_step * K * self.world / (ms * 1e-3), "unit": unit,
                "h2d_bytes_per_step": nbx, "d2h_bytes_per_step": nby, "ms_per_step": ms / K}

    def pack_layer(self, d, ffn, n_q, n_kv, hd, t, wtype, layer=0):
        tpx, dev, s = self.tpx, self.dev, self.stream
        from megatron_tensor_transformer_gb300 import inputs
        sh = tpx.make_shape(d, ffn=ffn, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=wtype)
        _, wg, wu, wd = inputs.mlp_inputs(d, ffn, 1, seed=0, device=dev, layer=layer)
        gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu, stream=s)
        dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd, stream=s)
        del wg, wu, wd
        _, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, 1, seed=0, device=dev, layer=layer)
        q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv, stream=s)
        o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo, stream=s)
        del wqkv, wo
        self.torch.cuda.empty_cache()
        return sh, (q, q_w, o, o_w, gu, gu_w, dn, dn_w)


# ------------------------------------------------------------------------------ configurations


def run_8b(hx, K, W, kernel_flags=0):
    """One step = one MLP forward (one fused launch) for each decode batch M in {1, 8, 32, 64}."""
    torch, tpx = hx.torch, hx.tpx
    from megatron_tensor_transformer_gb300 import inputs
    D, FFN, T, MS = MLP8B
    sh = tpx.make_shape(D, ffn=FFN, t=T)
    _, wg, wu, wd = inputs.mlp_inputs(D, FFN, 1, seed=0, device=hx.dev)
    gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu, stream=hx.stream)
    dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd, stream=hx.stream)
    del wg, wu, wd
    xs = {M: inputs.normal_bf16((M, D), 1.0, 0, inputs.STREAM_X, hx.dev) for M in MS}
    hs = {M: torch.empty((M, FFN), dtype=torch.bfloat16, device=hx.dev) for M in MS}
    ys = {M: torch.empty((M, D), dtype=torch.bfloat16, device=hx.dev) for M in MS}
    ws = tpx.new_workspace(sh, max(MS), hx.dev)
    fwd = lambda M: tpx.tp_mlp_forward(gu, gu_w, dn, dn_w, xs[M], xs[M], ys[M], hs[M], ws, flags=kernel_flags,
                                       stream=hx.stream)

    def step():
        for M in MS:
            fwd(M)

    ms, launches, clk = hx.timed(K, W, step)
    wbytes = 3.0 * D * FFN * 2
    blk_bytes = lambda M: wbytes + 3.0 * M * D * 2      # weights once + x, residual in, y out
    per_M, tot_t, tot_b = {}, 0.0, 0.0
    for M in MS:
        c = hx.per_call_ms(max(K, 10), lambda: fwd(M))
        tot_t, tot_b = tot_t + c, tot_b + blk_bytes(M)
        per_M[str(M)] = {"tokens_per_s": M / (c * 1e-3), "block_us": 1e3 * c,
                         "block_gbs": blk_bytes(M) / (c * 1e-3) / 1e9}
    pk = peaks()
    ach = tot_b / (tot_t * 1e-3) / 1e9
    e2e = hx.e2e(K, W, [(xs[M], ys[M]) for M in MS], lambda j: fwd(MS[j]), sum(MS), "tokens/s")
    step_bytes = sum(blk_bytes(M) for M in MS)
    return {
        "workload": "8b-mlp-decode", "value": sum(MS) * K * hx.world / (ms * 1e-3), "unit": "tokens/s",
        "steps": K, "warmup": W, "ms_per_step": ms / K, "dtype": "bf16",
        "config": {"workload": "8b-mlp-decode", "d": D, "ffn": FFN, "t": T, "M": list(MS),
                   "tokens_per_step": sum(MS), "l2": "weights 352 MB per forward > 129 MB L2; no flush"},
        "hbm_gbs_step": step_bytes / (ms / K * 1e-3) / 1e9,
        "hbm_frac_step": step_bytes / (ms / K * 1e-3) / 1e9 / pk["hbm"],
        "roofline": {"bound": "hbm", "kernel": "fused_kernel (the whole MLP block, one launch per forward)",
                     "achieved": ach, "peak": pk["hbm"], "peak_kind": pk["kind"] + " hbm_gbs (burst)", "unit": "GB/s",
                     "frac": ach / pk["hbm"], "traffic": traffic_record("8b-mlp-decode"),
                     "bytes_per_launch": tot_b / len(MS), "launch_us": 1e3 * tot_t / len(MS)},
        "per_M": per_M, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
    }


def run_layer(hx, name, K, W, kernel_flags=0, t_override=0):
    """A 70B- or 405B-shaped layer's linear parts, t logical shards:
    y1 = x + o_proj(attn(qkv(x))); y = y1 + MLP(y1), through tp_proj_forward and tp_mlp_forward;
    or, for the stack, `layers` pre-norm layers through tp_layer_forward."""
    torch, tpx = hx.torch, hx.tpx
    from megatron_tensor_transformer_gb300 import inputs
    d, ffn, n_q, n_kv, hd, t, M, wkind, nl = LAYERS[name]
    t = t_override or t
    fp8, x8 = wkind >= 1, wkind == 2
    prefill = "prefill" in name
    wtype = tpx.TP_FP8_E4M3 if fp8 else tpx.TP_BF16
    kf = kernel_flags | (tpx.TP_F_FP8_ACT if x8 else 0)
    layers = []
    for L in range(nl):
        sh, w = hx.pack_layer(d, ffn, n_q, n_kv, hd, t, wtype, layer=L)
        layers.append(w)
    Q = (n_q + 2 * n_kv) * hd
    x = inputs.normal_bf16((M, d), 1.0, 0, inputs.STREAM_X, hx.dev)
    y1, y = x.clone(), torch.empty_like(x)
    qkv = torch.empty((M, Q), dtype=torch.bfloat16, device=hx.dev)
    o_in = torch.empty((M, n_q * hd), dtype=torch.bfloat16, device=hx.dev)
    h = torch.empty((M, ffn), dtype=torch.bfloat16, device=hx.dev)
    ws = tpx.new_workspace(sh, M, hx.dev, flags=kf)
    s = hx.stream
    if name in PRENORM:
        scratch = torch.empty(tpx.tp_layer_scratch_bytes(sh, M), dtype=torch.uint8, device=hx.dev)
        xa, xb = torch.empty_like(x), torch.empty_like(x)

        def forward(src, dst):
            cur, nxt = src, xa
            for i, lay in enumerate(layers):
                out = dst if i == nl - 1 else (xa if i % 2 == 0 else xb)
                tpx.tp_layer_forward(*lay, cur, out, scratch, ws, flags=kf, stream=s)
                cur = out

        step = lambda: forward(x, y)
    else:
        q, q_w, o, o_w, gu, gu_w, dn, dn_w = layers[0]

        def forward(src, dst):
            tpx.tp_proj_forward(q, q_w, o, o_w, src, src, y1, qkv, o_in, ws, flags=kf, stream=s)
            tpx.tp_mlp_forward(gu, gu_w, dn, dn_w, y1, y1, dst, h, ws, flags=kf, stream=s)

        step = lambda: forward(x, y)
    ms, launches, clk = hx.timed(K, W, step)
    q, q_w, o, o_w, gu, gu_w, dn, dn_w = layers[0]
    pk = peaks()
    params = layer_params(d, ffn, n_q, n_kv, hd) * nl
    wb = 1.0 if fp8 else 2.0
    if prefill:
        # the dominant kernel: the MLP's column-parallel gate/up GEMM with SwiGLU (for e4m3 weights
        # the call also widens the weights into the workspace first)
        c = hx.per_call_ms(max(3, min(K, 10)), lambda: tpx.tp_colpar_forward(
            gu, gu_w, y1, h, flags=kf & ~tpx.TP_F_SPLIT_BLOCK, stream=s, ws=ws))
        kflops = 2.0 * 2 * d * ffn * M
        tpeak = pk["bf16"] * (2.0 if x8 else 1.0)
        kname = ("tc_kernel e4m3 x e4m3 (gate/up + SwiGLU)" if x8 else
                 "widen_e4m3 + tc_kernel (gate/up + SwiGLU)" if fp8 else "tc_kernel (gate/up + SwiGLU)")
        roof = {"bound": "tensor", "kernel": kname, "achieved": kflops / (c * 1e-3) / 1e12, "peak": tpeak,
                "peak_kind": pk["kind"] + (" bf16 x 2 (e4m3 rate)" if x8 else " bf16 (burst)"), "unit": "TFLOP/s",
                "frac": kflops / (c * 1e-3) / 1e12 / tpeak, "traffic": traffic_record(name),
                "flops_per_launch": kflops, "launch_us": 1e3 * c}
        flops = 2.0 * params * M
        value, unit = flops / (ms / K * 1e-3) / 1e12, "TFLOP/s"
        extra = {"tflop_per_step": flops / 1e12, "layer_frac": value / tpeak}
        unit_per_step = flops / 1e12
    else:
        # the dominant kernel: the MLP block, one fused launch (for the stack: timed with
        # tp_mlp_forward on the first layer's weights, the same kernel without the norm factor)
        c = hx.per_call_ms(max(10, min(K, 50)), lambda: tpx.tp_mlp_forward(
            gu, gu_w, dn, dn_w, y1, y1, y, h, ws, flags=kf, stream=s))
        kbytes = wb * 3 * d * ffn + 2.0 * 3 * M * d
        roof = {"bound": "hbm", "kernel": "fused_kernel (the whole MLP block, one launch)",
                "achieved": kbytes / (c * 1e-3) / 1e9, "peak": pk["hbm"], "peak_kind": pk["kind"] + " hbm_gbs (burst)",
                "unit": "GB/s", "frac": kbytes / (c * 1e-3) / 1e9 / pk["hbm"], "traffic": traffic_record(name),
                "bytes_per_launch": kbytes, "launch_us": 1e3 * c}
        wbytes = wb * params
        value, unit = M * K * hx.world / (ms * 1e-3), "tokens/s"
        extra = {"weight_gb": wbytes / 1e9, "hbm_gbs_step": wbytes / (ms / K * 1e-3) / 1e9,
                 "layer_frac": wbytes / (ms / K * 1e-3) / 1e9 / pk["hbm"]}
        unit_per_step = M
    e2e = hx.e2e(K, W, [(x, y)], lambda j: forward(x, y), unit_per_step, unit)
    dtype = "e4m3 weights x e4m3 activations (per token)" if x8 else ("e4m3 weights, bf16 activations" if fp8
                                                                       else "bf16")
    rec = {"workload": name, "value": value, "unit": unit, "steps": K, "warmup": W, "ms_per_step": ms / K,
           "dtype": dtype,
           "config": {"workload": name, "layers": nl, "d": d, "ffn": ffn, "n_q": n_q, "n_kv": n_kv, "head_dim": hd,
                      "t": t, "M": M, "weights_gb_per_step": wb * params / 1e9,
                      "l2": "weights per step > 129 MB L2; no flush"},
           "roofline": roof, "e2e": e2e, "gpu_launches": launches, "clocks": clk}
    rec.update(extra)
    return rec


def run_lm_head(hx, K, W, t_override=0):
    """Llama-3 70B output layer: the vocabulary-parallel lm_head (d 8192, 128256 ids over t=8
    shards, padded to 16128 per shard), decode M=32, fp32 logits, through tp_lm_head_forward;
    plus the vocabulary-parallel embedding lookup of the same tokens."""
    torch, tpx = hx.torch, hx.tpx
    from megatron_tensor_transformer_gb300 import inputs
    d, V, t, M = 8192, 128256, t_override or 8, 32
    sh = tpx.make_shape(d, t=t, vocab=V)
    w = inputs.normal_bf16((d, V), 0.02, 0, 70, hx.dev)
    w_p, wd = tpx.tp_partition_weights(sh, tpx.TP_W_VOCAB, w, stream=hx.stream)
    del w
    e = inputs.normal_bf16((V, d), 1.0, 0, 71, hx.dev)
    e_p, ed = tpx.tp_partition_weights(sh, tpx.TP_W_EMBED, e, stream=hx.stream)
    del e
    torch.cuda.empty_cache()
    ids = torch.randint(0, V, (M,), generator=torch.Generator(device=hx.dev).manual_seed(0), device=hx.dev,
                        dtype=torch.int32)
    x = torch.empty((M, d), dtype=torch.bfloat16, device=hx.dev)
    logits = torch.empty((M, V), dtype=torch.float32, device=hx.dev)
    ws = tpx.new_workspace(sh, M, hx.dev)

    def step():
        tpx.tp_embed_lookup(ed, e_p, ids, x, stream=hx.stream)
        tpx.tp_lm_head_forward(wd, w_p, x, logits, ws=ws, stream=hx.stream)

    ms, launches, clk = hx.timed(K, W, step)
    c = hx.per_call_ms(max(10, K), lambda: tpx.tp_lm_head_forward(wd, w_p, x, logits, ws=ws, stream=hx.stream))
    # e2e: the token ids in from host memory, the fp32 logits back, every step
    e2e = hx.e2e(K, W, [(ids, logits)], lambda j: step(), M, "tokens/s")
    head_bytes = 2.0 * d * V + 2.0 * M * d + 4.0 * M * V
    pk = peaks()
    return {"workload": "70b-lm-head-decode", "value": M * K / (ms * 1e-3), "unit": "tokens/s", "steps": K,
            "warmup": W, "ms_per_step": ms / K, "dtype": "bf16",
            "config": {"workload": "70b-lm-head-decode", "d": d, "vocab": V, "t": t, "M": M},
            "roofline": {"bound": "hbm", "kernel": "tc_kernel (vocabulary-parallel lm_head)",
                         "achieved": head_bytes / (c * 1e-3) / 1e9, "peak": pk["hbm"], "unit": "GB/s",
                         "frac": head_bytes / (c * 1e-3) / 1e9 / pk["hbm"], "traffic": None},
            "e2e": e2e, "gpu_launches": launches, "clocks": clk}


def run_attn(hx, K, W, t_override=0):
    """Llama-3.1 70B attention block with a real KV cache: 32 sequences, each with 4095 cached
    positions (4096 with the new token), t=8.  One step = one tp_attn_block_forward: QKV
    (column-parallel) + the head-sharded decode attention over the cache + o_proj (row-parallel,
    shard fold, residual).  The roofline kernel is the attention (cache reads: M x n_kv x 4096 x
    hd x 2 x 2 bytes)."""
    torch, tpx = hx.torch, hx.tpx
    from megatron_tensor_transformer_gb300 import inputs
    d, n_q, n_kv, hd, t, M, L = 8192, 64, 8, 128, t_override or 8, 32, 4096
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    x, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, M, seed=0, device=hx.dev)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv, stream=hx.stream)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo, stream=hx.stream)
    del wqkv, wo
    kc = inputs.normal_bf16((t, M, n_kv // t, L, hd), 1.0, 0, 90, hx.dev)
    vc = inputs.normal_bf16((t, M, n_kv // t, L, hd), 1.0, 0, 91, hx.dev)
    lens = torch.full((M,), L - 1, dtype=torch.int32, device=hx.dev)
    qkv = torch.empty((M, (n_q + 2 * n_kv) * hd), dtype=torch.bfloat16, device=hx.dev)
    o_in = torch.empty((M, n_q * hd), dtype=torch.bfloat16, device=hx.dev)
    y = torch.empty_like(x)
    bws = tpx.new_attn_block_workspace(sh, M, L, hx.dev)
    aws = torch.empty(tpx.tp_attn_workspace_bytes(sh, M, L), dtype=torch.uint8, device=hx.dev)
    step = lambda: tpx.tp_attn_block_forward(q, q_w, o, o_w, x, x, kc, vc, lens, y, qkv, o_in, bws, stream=hx.stream)
    ms, launches, clk = hx.timed(K, W, step)
    c = hx.per_call_ms(max(10, K), lambda: tpx.tp_attn_decode(sh, qkv, kc, vc, lens, o_in, aws, stream=hx.stream))
    # e2e: x in from host memory and y back every step (the KV cache stays resident)
    e2e = hx.e2e(K, W, [(x, y)], lambda j: step(), M, "tokens/s")
    cache_bytes = 2.0 * M * n_kv * L * hd * 2
    w_bytes = 2.0 * ((n_q + 2 * n_kv) * hd * d + n_q * hd * d)
    pk = peaks()
    return {"workload": "70b-attn-decode", "value": M * K / (ms * 1e-3), "unit": "tokens/s", "steps": K, "warmup": W,
            "ms_per_step": ms / K, "dtype": "bf16",
            "config": {"workload": "70b-attn-decode", "d": d, "n_q": n_q, "n_kv": n_kv, "head_dim": hd, "t": t,
                       "M": M, "context": L},
            "hbm_gbs_step": (cache_bytes + w_bytes) / (ms / K * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "kernel": "decode attention (append + attention pass)",
                         "achieved": cache_bytes / (c * 1e-3) / 1e9, "peak": pk["hbm"], "unit": "GB/s",
                         "frac": cache_bytes / (c * 1e-3) / 1e9 / pk["hbm"], "attn_us": 1e3 * c, "traffic": None},
            "e2e": e2e, "gpu_launches": launches, "clocks": clk}


# ----------------------------------------------------------------------- CPU oracle on the host


def cpu_setup(name):
    """A bounded sample of one configuration for the float64 oracle (as it stands).  Returns
    (rep, units per rep, unit, scale, description): one call of rep() is one sample step, and a
    full step of the configuration costs `scale` samples.  Decode samples run every token through
    shard 0 of t = 8 (1/8 of each weight: the first t-th of the column-parallel outputs and the
    matching rows of the row-parallel weights, which is exactly one term of the tensor-parallel
    sum), so a full step costs 8 samples (80 for the 10-layer stack, one layer sampled).  Prefill samples run 256 token rows through shard 0 and report the
    oracle's own TFLOP/s.  e4m3 configurations time the same float64 arithmetic: the oracle
    evaluates them on the dequantised weights, float64 arrays of the same shapes."""
    import numpy as np
    import torch
    from megatron_tensor_transformer_gb300 import inputs
    from oracle import tp_oracle as O
    torch.set_num_threads(cores())        # weight generation only; the oracle's BLAS threads are set by env
    f64 = lambda a: O.as_f64(a.view(torch.int16).numpy().view(np.uint16))
    gen = lambda shape, std, stream: f64(inputs.normal_bf16(shape, std, 0, stream, "cpu"))
    if name == "8b-mlp-decode":
        D, FFN, _, MS = MLP8B
        F = FFN // 8
        wg, wu, wd = gen((D, F), 0.02, 11), gen((D, F), 0.02, 12), gen((F, D), 0.02, 13)
        xs = [gen((M, D), 1.0, 1) for M in MS]

        def rep():
            for x in xs:
                O.mlp(x, wg, wu, wd, residual=x)
        return rep, float(sum(MS)), "tokens/s", 8.0, \
            "the four decode batches M=1,8,32,64 through shard 0 of 8 of the 8B MLP; a full step costs 8 samples"
    d, ffn, n_q, n_kv, hd, t, M, wkind, nl = LAYERS[name]
    ts = 8
    F, nq, nkv = ffn // ts, n_q // ts, n_kv // ts
    wqkv, wo = gen((d, (nq + 2 * nkv) * hd), 0.02, 14), gen((nq * hd, d), 0.02, 15)
    wg, wu, wd = gen((d, F), 0.02, 11), gen((d, F), 0.02, 12), gen((F, d), 0.02, 13)
    prefill = "prefill" in name
    rows = 256 if prefill else M
    x = gen((rows, d), 1.0, 1)

    def rep():
        if nl > 1:
            O.layer(x, wqkv, wo, wg, wu, wd, nq, nkv, hd)
        else:
            y1, _ = O.proj(x, wqkv, wo, nq, nkv, hd, residual=x)
            O.mlp(y1, wg, wu, wd, residual=y1)
    sample_params = d * (nq + 2 * nkv) * hd + nq * hd * d + 3 * d * F
    if prefill:
        return rep, 2.0 * rows * sample_params / 1e12, "TFLOP/s", 1.0, \
            f"{rows} token rows through shard 0 of {ts} of the layer (2 flops per weight per token)"
    return rep, float(M), "tokens/s", float(ts * nl), \
        (f"all {M} tokens through shard 0 of {ts} of " + ("one of the ten layers" if nl > 1 else "the layer")
         + f"; a full step costs {ts * nl} samples")


def cpu_sample(name, seconds):
    """Time the oracle on the sample of cpu_setup for about `seconds` and return the
    configuration's metric.  The first repetition is a warm-up, unless it alone takes `seconds`."""
    rep, per_rep, unit, scale, what = cpu_setup(name)
    c0, t0 = time.process_time(), time.perf_counter()
    rep()                                  # warm-up (page-in, BLAS start-up), kept if it alone is long
    n, el = 1, time.perf_counter() - t0
    if el < seconds:
        c0, t0, n = time.process_time(), time.perf_counter(), 0
        while True:
            rep()
            n += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
    used = (time.process_time() - c0) / el
    return {"value": per_rep * n / (el * scale), "unit": unit, "reps": n, "seconds": el,
            "cores_used": used, "sample": f"{n} repetitions of {what} in {el:.1f} s"}


def cpu_baseline(name, seconds):
    """The oracle's sample of one configuration in fresh processes: with every allowed core,
    then with one thread (BLAS thread counts are fixed when numpy loads, hence the processes)."""
    out = {}
    for key, nthreads in (("all", cores()), ("one", 1)):
        env = dict(os.environ)
        for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            env[v] = str(nthreads)
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", name,
                            "--cpu-seconds", str(seconds)], capture_output=True, text=True, env=env, timeout=900)
        line = [l for l in r.stdout.splitlines() if l.startswith("{")]
        if r.returncode != 0 or not line:
            return {"value": None, "kind": "oracle", "error": (r.stderr or r.stdout)[-300:]}
        out[key] = json.loads(line[-1])
        out[key]["threads"] = nthreads
    a, o = out["all"], out["one"]
    return {"value": a["value"], "unit": a["unit"], "cores": a["threads"], "cores_used": round(a["cores_used"], 2),
            "kind": "oracle", "sample": a["sample"],
            "one_thread": {"value": o["value"], "cores": 1, "cores_used": round(o["cores_used"], 2),
                           "sample": o["sample"]}}


def workload_config(name):
    """The configuration record of a workload, as the GPU arm prints it."""
    if name == "8b-mlp-decode":
        D, FFN, T, MS = MLP8B
        return {"workload": name, "d": D, "ffn": FFN, "t": T, "M": list(MS), "tokens_per_step": sum(MS)}
    d, ffn, n_q, n_kv, hd, t, M, wkind, nl = LAYERS[name]
    return {"workload": name, "layers": nl, "d": d, "ffn": ffn, "n_q": n_q, "n_kv": n_kv, "head_dim": hd, "t": t,
            "M": M, "weights_gb_per_step": (1.0 if wkind else 2.0) * layer_params(d, ffn, n_q, n_kv, hd) * nl / 1e9}


def run_reference(args, rank, world):
    """The reference arm: the float64 oracle on this host's cores, one bounded sample of the
    headline workload per step (cpu_setup), in the headline's metric and unit."""
    if rank != 0:
        return
    name = getattr(args, "workload", None) or HEADLINE
    if name == "all":
        name = HEADLINE
    if name != "8b-mlp-decode" and name not in LAYERS:
        print(json.dumps({"impl": "reference", "unavailable": f"no oracle sample is defined for {name}"}), flush=True)
        return
    rep, per_rep, unit, scale, what = cpu_setup(name)
    for _ in range(args.warmup):
        rep()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        rep()
    el = time.perf_counter() - t0
    value = per_rep * args.steps / (el * scale)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(name),
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores(), "kind": "oracle",
                         "sample": f"each step: {what}"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------------------------------ main


KERNEL_FLAGS = {"auto": 0, "tc": "TP_F_KERNEL_TC", "skinny": "TP_F_KERNEL_SKINNY", "split": "TP_F_SPLIT_BLOCK",
                "hilo": "TP_F_FP8_HILO", "foldnorm": "TP_F_FOLD_NORM"}


def run_one(hx, name, K, W, args):
    kf = KERNEL_FLAGS[args.kernel]
    kf = getattr(hx.tpx, kf) if kf else 0
    if name == "8b-mlp-decode":
        rec = run_8b(hx, K, W, kf)
    elif name == "70b-lm-head-decode":
        rec = run_lm_head(hx, K, W, args.t)
    elif name == "70b-attn-decode":
        rec = run_attn(hx, K, W, args.t)
    else:
        rec = run_layer(hx, name, K, W, kf, args.t)
    hx.torch.cuda.synchronize()
    hx.torch.cuda.empty_cache()
    return rec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tpx", choices=["tpx", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=3.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="all", choices=["all"] + ["8b-mlp-decode"] + sorted(LAYERS) + EXTRA)
    ap.add_argument("--t", type=int, default=0, help="shard count for the layer workloads (default: 8)")
    ap.add_argument("--kernel", default="auto", choices=sorted(KERNEL_FLAGS),
                    help="force the tcgen05 or the mma.sync decode kernels, or separate launches for the "
                         "two halves of a block, or (foldnorm) prefill layers with their RMSNorms folded into "
                         "the GEMMs (default: library policy, one fused launch per decode block)")
    ap.add_argument("--cpu-sample", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_sample:                     # child process of cpu_baseline
        print(json.dumps(cpu_sample(args.cpu_sample, args.cpu_seconds)), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        hx = Harness(local, world)
        K, W = args.steps, args.warmup
        names = DEFAULT_SET if args.workload == "all" else [args.workload]
        recs = {n: run_one(hx, n, K, W, args) for n in names}
        cpu_ok = rank == 0 and world == 1 and not args.no_cpu_baseline
        for n, r in recs.items():         # after every timed region: the oracle must not share the CPU
            r["cpu_baseline"] = cpu_baseline(n, args.cpu_seconds) if cpu_ok and n in DEFAULT_SET else None
        head = recs[HEADLINE if args.workload == "all" else args.workload]
        out = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": K,
               "warmup": W, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic (seeded normals, random-init weights)",
               "config": dict(head["config"], parallelism="replicas" if world > 1 else "single"),
               "roofline": head["roofline"], "e2e": head.get("e2e"), "cpu_baseline": head["cpu_baseline"],
               "gpu_launches": head["gpu_launches"], "clocks": head["clocks"]}
        for k in ("weight_gb", "hbm_gbs_step", "layer_frac", "tflop_per_step", "per_M", "hbm_frac_step"):
            if k in head:
                out[k] = head[k]
        if args.workload == "all":
            out["configs"] = recs
        if rank == 0:
            print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
