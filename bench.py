"""Benchmark of the fused ONNX Conv path on GB300.

A step is one pass of the ResNet-50 (v2) conv stack at batch 32: all 53 conv layers (7x7/2
stem, 1x1 and 3x3 bottleneck convs, strided projections) with folded BN + ReLU, bf16 inputs,
fp32 accumulation and output, each layer on its own resident input/output buffers (about
2.2 GB per step, far larger than L2, so every layer reads its input from HBM).  The step runs
as two launches: the stem (window-mode tcgen05 kernel, with its channel-padding pre-pass) and
one conv-chain launch holding the 52 other layers (conv_fused_chain_*).  `value` is the
whole-job TFLOP/s (2*N*K*Ho*Wo*C*R*S per layer, padded taps included).  The same run reports
the step as 53 per-layer launches, ResNet-50's own dataflow as one dependent chain (bf16
activations and residuals), the MobileNetV2 depthwise layers at batch 64 (GB/s against HBM),
the static int8 ResNet 3x3 layers at batch 64 (TOP/s) and the other configurations.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--layers-out F]

For N > 1 it runs under torchrun as independent replicas (one per GPU, weak scaling); the
only collectives are the timing barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused conv TFLOP/s (ResNet-50 bs32, % bf16 peak); depthwise GB/s (% HBM)"
WORKLOAD = ("ResNet-50 v2 conv stack, 53 layers (7x7/2 stem, 1x1 and 3x3 bottlenecks, strided "
            "projections) at batch 32, 224x224 input, bf16 x/W, fp32 accumulate and output, "
            "folded BN + ReLU epilogue, channels-last")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of one tc_chain_kernel launch (the 52-step chain of the step), captured with
#   python bench.py --profile chain:0
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,lts__t_sectors_srcunit_tex_op_write.sum,
#       gpu__time_duration.sum --clock-control none -k regex:tc_chain -s 2 -c 1 --csv
#       python bench.py --profile chain:0
# traffic = dram__bytes_read.sum plus the bytes the SMs wrote into L2 (lts__t_sectors_srcunit_tex_op_write
# x 32: every one of them reaches DRAM, but ncu flushes the caches around each kernel and
# dram__bytes_write.sum counts only what was evicted while the kernel ran).  It describes the
# kernel sources it was taken on (SHA-256 prefix of their code with comments and blank space
# removed) and is reported as null for any other sources.
CHAIN_TRAFFIC = {"bytes_per_launch": 1.9770e9, "read_per_launch": 657.1e6, "write_per_launch": 1319.8e6,
                 "dram_write_during_launch": 1281.1e6, "sources_sha256_16": "12a87a18773bd2ab"}
CHAIN_SOURCES = ("tc_chain.cu", "chain.cu", "ptx.cuh", "convf_internal.h", "api_internal.h")


def sources_digest():
    """SHA-256 prefix of the chain kernel's sources, comments and blank space removed."""
    import re
    h = hashlib.sha256()
    for f in CHAIN_SOURCES:
        with open(os.path.join(ROOT, "convolution_onnx_conv_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def chain_traffic():
    if CHAIN_TRAFFIC is None or sources_digest() != CHAIN_TRAFFIC["sources_sha256_16"]:
        return None
    return CHAIN_TRAFFIC["bytes_per_launch"]


def max_over_ranks(x, world, device):
    """The largest of every rank's x (each replica's measured time), so the job is timed by its
    slowest replica; x itself on one rank."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flops_per_step, steps, ms):
    """Replicas (weak scaling): every rank runs the whole step on its own GPU, so the job does
    world x the work of one step per step in `ms` milliseconds."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        hbm = float(d.get("hbm_gbs") or d.get("hbm_GBs") or d["hbm"])
        bf16 = float(d.get("bf16_tflops") or d["bf16"])
        sus = float(d.get("bf16_tflops_sustained") or bf16)
        return {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_tflops_sustained": sus}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            sel = str(device_index)
        self.sel = sel

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in self.samples:
            try:
                sm.append(float(p[0]))
                mx.append(float(p[1]))
            except ValueError:
                continue
            for name, v in zip(names, p[3:7]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ workloads
def build_layers(specs, seed_base, torch, cf, synthetic, s8=False):
    """FusedConv handles + resident device inputs/outputs for each spec (plus host copies)."""
    out = []
    for i, spec in enumerate(specs):
        seed = synthetic.seed_for(seed_base, i)
        if s8:
            inp = synthetic.int8_inputs(spec, seed)
            conv = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                                stride=spec.stride, pads=spec.pads, act=spec.act, requant_mult=inp["mult"],
                                requant_shift=inp["shift"])
        else:
            inp = synthetic.conv_inputs(spec, seed)
            scale, shift = cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5) \
                if inp["bn"] is not None else (None, None)
            conv = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                                scale, shift, stride=spec.stride, pads=spec.pads, group=spec.group,
                                act=spec.act)
        x_host = inp["x"].contiguous(memory_format=torch.channels_last)
        x = x_host.cuda()
        y = conv.new_output()
        out.append({"spec": spec, "conv": conv, "x": x, "y": y, "x_host": x_host, "inp": inp})
    return out


def build_ext_layers(specs, layers, torch, cf):
    """The ResNet-50 step with bf16 outputs (a bf16 network's activations) and the bottleneck
    shortcut added in each block's last 1x1 conv (a bf16 residual of y's shape): the extended
    epilogue.  The residual is the block's shortcut tensor, as in the network's dataflow: the
    block input (the input buffer of the block's first 1x1 conv), or in a stage's first block the
    projection conv's output.  A layer the extended epilogue cannot serve (the 3-channel stem)
    keeps its fp32 handle."""
    out = []
    for i, (spec, L) in enumerate(zip(specs, layers)):
        inp = L["inp"]
        scale, shift = cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5) \
            if inp["bn"] is not None else (None, None)
        res = "1x1b" in spec.name
        try:
            conv = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                                scale, shift, stride=spec.stride, pads=spec.pads, group=spec.group,
                                act=spec.act, out_bf16=True, residual=res)
        except cf.ConvFusedError:
            out.append(L)
            continue
        out.append({"spec": spec, "conv": conv, "x": L["x"], "y": conv.new_output(), "r": None})
    by_name = {E["spec"].name.split("_", 2)[2].split("@")[0]: E for E in out}   # "s0b0_1x1a" -> layer
    for E in out:
        name = E["spec"].name.split("_", 2)[2].split("@")[0]
        if not name.endswith("1x1b"):
            continue
        block = name[: -len("_1x1b")]
        src = by_name[block + "_proj"]["y"] if block + "_proj" in by_name else \
            by_name[block + "_1x1a"]["x"] if block + "_1x1a" in by_name else None
        if src is None:   # a subset of the layers without the block's first conv: a seeded tensor
            g = torch.Generator().manual_seed(9000 + out.index(E))
            src = torch.randn(tuple(E["y"].shape), generator=g).to(torch.bfloat16).contiguous(
                memory_format=torch.channels_last).cuda()
        assert tuple(src.shape) == tuple(E["y"].shape) and src.dtype == E["y"].dtype, (name, src.shape)
        E["r"] = src
    return out


def chain_conv(spec, inp, cf, out_bf16=False, residual=False):
    """A handle of a kind the conv chain runs: the 1x1-GEMM variant for plain 1x1 convs, the
    im2col implicit GEMM for every other shape."""
    scale, shift = cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5) \
        if inp["bn"] is not None else (None, None)
    plain = spec.R == 1 and spec.S == 1 and tuple(spec.stride) == (1, 1) and tuple(spec.pads) == (0, 0, 0, 0)
    return cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"], scale, shift,
                        stride=spec.stride, pads=spec.pads, group=spec.group, act=spec.act,
                        variant=cf.CONVF_VARIANT_GEMM_1X1 if plain else cf.CONVF_VARIANT_IMPLICIT_GEMM,
                        out_bf16=out_bf16, residual=residual)


def build_chain(layers, cf, convs=None, xs=None, ys=None):
    """The layers as one chain of independent steps (each on its own input and output buffers:
    no step reads another's output), with the layers' own buffers unless others are given."""
    convs = convs or [chain_conv(L["spec"], L["inp"], cf) for L in layers]
    xs = xs or [L["x"] for L in layers]
    ys = ys or [L["y"] for L in layers]
    return cf.ConvChain(list(zip(convs, xs, ys))), convs


def build_network_chain(specs, layers, torch, cf, workloads, synthetic):
    """ResNet-50's own dataflow as one chain: the 52 bottleneck layers in workloads.resnet50_dataflow
    order, bf16 outputs, each layer reading the output of the layer before it and each block's
    last 1x1 conv adding the block's shortcut; the input is a seeded N(0,1) bf16 tensor of the
    stem's pooled output shape (32 x 64 x 56 x 56).  Weights and BN are the step's, with each
    block's last BN damped (synthetic.residual_branch_inputs)."""
    g = torch.Generator().manual_seed(7001)
    x0 = torch.randn((specs[1].N, 64, 56, 56), generator=g).to(torch.bfloat16).contiguous(
        memory_format=torch.channels_last).cuda()
    ys, steps, convs = [], [], []
    for li, src, rsrc in workloads.resnet50_dataflow():
        # a block's last conv with the damped residual-branch BN (synthetic.residual_branch_inputs)
        inp = synthetic.residual_branch_inputs(specs[li], synthetic.seed_for(3, li)) if rsrc is not None \
            else layers[li]["inp"]
        c = chain_conv(specs[li], inp, cf, out_bf16=True, residual=rsrc is not None)
        y = c.new_output()
        x = x0 if src < 0 else ys[src]
        steps.append((c, x, y) if rsrc is None else (c, x, y, x0 if rsrc < 0 else ys[rsrc]))
        ys.append(y)
        convs.append(c)
    return cf.ConvChain(steps), convs


def build_ext_chain(specs, layers, cf, workloads):
    """The bf16-output + residual step (build_ext_layers) as one chain: the 52 non-stem layers,
    each on its own input, in workloads.resnet50_dataflow order (a block's projection before the
    1x1 conv that adds it); each block's last 1x1 conv adds the block's shortcut tensor -- the
    projection's output (a dependency inside the chain) or the block's input buffer (the input of
    its first 1x1 conv)."""
    flow = workloads.resnet50_dataflow()
    name = [s.name.split("_", 2)[2].split("@")[0] for s in specs]
    pos = {name[li]: k for k, (li, _, _) in enumerate(flow)}
    ys, steps = [], []
    for li, src, rsrc in flow:
        c = chain_conv(specs[li], layers[li]["inp"], cf, out_bf16=True, residual=rsrc is not None)
        y = c.new_output()
        if rsrc is None:
            steps.append((c, layers[li]["x"], y))
        else:
            block = name[li][: -len("_1x1b")]
            r = ys[pos[block + "_proj"]] if block + "_proj" in pos else layers[name.index(block + "_1x1a")]["x"]
            steps.append((c, layers[li]["x"], y, r))
        ys.append(y)
    return cf.ConvChain(steps)


def capture_fn(fn, torch):
    """One CUDA graph of whatever `fn` launches on the current stream."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def capture_graph(layers, torch, reps=1):
    """One CUDA graph that launches every layer of the sequence `reps` times, in order."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            for L in layers:
                L["conv"](L["x"], L["y"], r=L.get("r"))
    return g


def time_graph(g, steps, torch):
    """Device time of `steps` back-to-back replays (ms), events on the replay stream."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def time_launches(layers, steps, torch):
    """Per-launch device durations: every launch of the sequence bracketed by CUDA events on
    its stream; the stream is held by a sleep kernel while the host enqueues a step, so the
    launches run back to back and the events time the kernels, not the host.  Returns the
    summed ms per layer over `steps` passes."""
    n = len(layers)
    per = [0.0] * n
    for _ in range(steps):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda._sleep(int(4e6 + 1e5 * n))
        for i, L in enumerate(layers):
            ev[i][0].record()
            L["conv"](L["x"], L["y"])
            ev[i][1].record()
        torch.cuda.synchronize()
        for i in range(n):
            per[i] += ev[i][0].elapsed_time(ev[i][1])
    return per


def scale_to(per, steps, total_ms):
    """Per-launch event durations (summed over `steps` passes) rescaled so that one pass adds up
    to `total_ms` (the graph-timed step): the events serialise launches and add a little each."""
    per = [p / steps for p in per]
    tot = sum(per)
    return [p * total_ms / tot for p in per] if tot > 0 else per


def attainable_ms(spec, peaks):
    """Roofline time of one layer: FLOPs at the bf16 burst peak or algorithmic bytes at HBM."""
    return max(spec.flops / (peaks["bf16_tflops"] * 1e12), spec.algorithmic_bytes / (peaks["hbm_gbs"] * 1e9)) * 1e3


def layer_bound(spec, peaks):
    t = spec.flops / (peaks["bf16_tflops"] * 1e12)
    b = spec.algorithmic_bytes / (peaks["hbm_gbs"] * 1e9)
    return "tensor" if t >= b else "hbm"


def other_configs(args, torch, cf, synthetic, workloads, peaks):
    """The other workloads, each one CUDA-graph replay per pass: the single conv (batch 1), the
    whole MobileNetV2 conv stack at batch 64 (with its 1x1 expand/project layers alone as well)
    and the batch-1 latency of the ResNet-50 and MobileNetV2 stacks."""
    out = {}
    steps = max(5, args.steps // 2)

    def timed(specs, base, reps=1):
        Ls = build_layers(specs, base, torch, cf, synthetic)
        for _ in range(args.warmup):
            for L in Ls:
                L["conv"](L["x"], L["y"])
        g = capture_graph(Ls, torch)
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        ms = time_graph(g, steps, torch) / steps
        if any(L["conv"].status() != 0 for L in Ls):
            raise SystemExit("device status error in " + specs[0].name)
        return ms, Ls

    one = workloads.single_conv_relu()
    ms, _ = timed([one], 1)
    out["single_conv"] = {"workload": "Conv 3x3 + bias + ReLU, N=1, C=16, 32x32, K=32 (fp32 out)",
                          "us": ms * 1e3, "tflops": one.flops / (ms * 1e-3) / 1e12}
    mv = workloads.mobilenetv2_layers(64)
    ms, Ls = timed(mv, 4)
    pw = [s for s in mv if s.R == 1]
    ms_pw, Lpw = timed(pw, 6)
    pw_bytes = sum(s.algorithmic_bytes for s in pw)
    # the same 1x1 layers as one conv-chain launch (independent steps)
    ch_pw, _ = build_chain(Lpw, cf)
    ch_pw()
    g_pw = capture_fn(lambda: ch_pw(), torch)
    for _ in range(args.warmup):
        g_pw.replay()
    torch.cuda.synchronize()
    ms_pwc = time_graph(g_pw, steps, torch) / steps
    if ch_pw.status() != 0:
        raise SystemExit("device status error in the MobileNetV2 1x1 chain")
    # the whole stack with its 1x1 layers as one chain launch and the 17 depthwise layers as
    # their own launches (every layer on its own input, as above)
    ch_all, _ = build_chain([L for L, sp in zip(Ls, mv) if sp.R == 1], cf)
    dwL = [L for L, sp in zip(Ls, mv) if sp.R != 1]

    def mv_step():
        ch_all()
        for L in dwL:
            L["conv"](L["x"], L["y"])

    mv_step()
    g_mv = capture_fn(mv_step, torch)
    for _ in range(args.warmup):
        g_mv.replay()
    torch.cuda.synchronize()
    ms_mvc = time_graph(g_mv, steps, torch) / steps
    if ch_all.status() != 0:
        raise SystemExit("device status error in the MobileNetV2 chain")
    out["mobilenetv2_b64"] = {
        "workload": "MobileNetV2 conv stack (17 blocks: 1x1 expand + ReLU6, depthwise 3x3 + ReLU6, 1x1 "
                    "project) at batch 64, bf16 in, fp32 out",
        "ms_per_step": ms, "tflops": sum(s.flops for s in mv) / (ms * 1e-3) / 1e12,
        "gb_s": sum(s.algorithmic_bytes for s in mv) / (ms * 1e-3) / 1e9,
        "execution": "one launch per layer",
        "with_1x1_chain": {"ms_per_step": ms_mvc, "tflops": sum(s.flops for s in mv) / (ms_mvc * 1e-3) / 1e12,
                           "gb_s": sum(s.algorithmic_bytes for s in mv) / (ms_mvc * 1e-3) / 1e9,
                           "execution": "the 33 1x1 layers as one conv-chain launch + the 17 depthwise "
                                        "launches"},
        "expand_project_1x1": {"layers": len(pw), "ms": ms_pw, "gb_s": pw_bytes / (ms_pw * 1e-3) / 1e9,
                               "pct_hbm": pw_bytes / (ms_pw * 1e-3) / 1e9 / peaks["hbm_gbs"],
                               "tflops": sum(s.flops for s in pw) / (ms_pw * 1e-3) / 1e12,
                               "execution": "one launch per layer",
                               "chain": {"ms": ms_pwc, "gb_s": pw_bytes / (ms_pwc * 1e-3) / 1e9,
                                         "pct_hbm": pw_bytes / (ms_pwc * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                         "tflops": sum(s.flops for s in pw) / (ms_pwc * 1e-3) / 1e12,
                                         "execution": "the same layers as one conv-chain launch"}}}
    # the same stack as 17 fused inverted-residual blocks (one kernel per block: the expanded
    # tensor never goes to HBM); GB/s against each block's own algorithmic bytes (input, output,
    # weights)
    blocks = workloads.mobilenetv2_blocks(64)
    BL = []
    for i, (name, N, cin, h, ch, cout, st, ex, res) in enumerate(blocks):
        inp = synthetic.block_inputs(N, cin, h, ch, cout, ex, synthetic.seed_for(11, i))
        aff = lambda bn: cf.conv_bn_scale_shift(*[t.numpy() for t in bn], 1e-5)
        blk = cf.InvertedResidualBlock(N, cin, h, h, ch, cout, st, inp["we"], aff(inp["bn_e"]) if ex else None,
                                       inp["wd"], aff(inp["bn_d"]), inp["wp"], aff(inp["bn_p"]), residual=res)
        x = inp["x"].contiguous(memory_format=torch.channels_last).cuda()
        BL.append({"conv": blk, "x": x, "y": blk.new_output()})
    for _ in range(args.warmup):
        for L in BL:
            L["conv"](L["x"], L["y"])
    gb = capture_graph(BL, torch)
    for _ in range(args.warmup):
        gb.replay()
    torch.cuda.synchronize()
    ms_b = time_graph(gb, steps, torch) / steps
    if any(L["conv"].status() != 0 for L in BL):
        raise SystemExit("device status error in the fused MobileNetV2 blocks")
    blk_bytes = 0
    for (name, N, cin, h, ch, cout, st, ex, res) in blocks:
        ho = (h + 2 - 3) // st + 1
        blk_bytes += N * cin * h * h * 2 + N * cout * ho * ho * 4 + 2 * (ch * cin * ex + ch * 9 + cout * ch)
    out["mobilenetv2_b64"]["fused_blocks"] = {
        "workload": "the same 17 blocks, each one fused kernel (expand + depthwise + project + skip)",
        "ms_per_step": ms_b, "tflops": sum(s.flops for s in mv) / (ms_b * 1e-3) / 1e12,
        "gb_s": blk_bytes / (ms_b * 1e-3) / 1e9, "pct_hbm": blk_bytes / (ms_b * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "speedup_vs_per_layer": ms / ms_b}
    r1 = workloads.resnet50_layers(1)
    ms_r1, _ = timed(r1, 7)
    m1 = workloads.mobilenetv2_layers(1)
    ms_m1, _ = timed(m1, 8)
    out["latency_b1"] = {"note": "batch 1, one CUDA-graph replay of the whole conv stack (working set in L2)",
                         "resnet50_us": ms_r1 * 1e3, "mobilenetv2_us": ms_m1 * 1e3}
    return out


def qlinear_config(args, torch, cf, synthetic, workloads, peaks):
    """ONNX QLinearConv on the seven ResNet-50 3x3 shapes at batch 64: uint8 x with a zero point,
    int8 w with per-channel zero points, uint8 y with a fused Relu; one graph replay per pass."""
    specs = workloads.int8_layers(64)
    Ls = []
    for i, spec in enumerate(specs):
        inp = synthetic.qlinear_inputs(spec, synthetic.seed_for(9, i), False, True, False)
        conv = cf.QLinearConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                              x_scale=inp["x_scale"], x_zero_point=inp["x_zp"], w_scale=inp["w_scale"].numpy(),
                              w_zero_point=inp["w_zp"].numpy(), y_scale=inp["y_scale"], y_zero_point=inp["y_zp"],
                              relu=True, stride=spec.stride, pads=spec.pads)
        x = inp["x"].contiguous(memory_format=torch.channels_last).cuda()
        Ls.append({"conv": conv, "x": x, "y": conv.new_output()})
    for _ in range(args.warmup):
        for L in Ls:
            L["conv"](L["x"], L["y"])
    g = capture_graph(Ls, torch)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    steps = max(3, args.steps // 5)
    ms = time_graph(g, steps, torch) / steps
    if any(L["conv"].status() != 0 for L in Ls):
        raise SystemExit("device status error in the QLinearConv layers")
    ops = sum(s.flops for s in specs)
    return {"workload": "QLinearConv, ResNet-50 3x3 shapes (7) at batch 64: uint8 x and y with zero points, int8 "
                        "w with per-channel zero points and scales, float32 requantisation, fused Relu",
            "tops": ops / (ms * 1e-3) / 1e12, "ms": ms, "pct_bf16_peak": ops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]}


# ------------------------------------------------------------------------------ CPU oracle
_ORACLE_CACHE = {}


def _oracle_layer_inputs(spec, seed, synthetic):
    """float64 inputs of one image of the layer (the sample's points all lie in image 0)."""
    key = (spec.name, seed)
    if key not in _ORACLE_CACHE:
        one = spec.with_batch(1)
        inp = synthetic.conv_inputs(one, seed)
        bn = tuple(t.numpy() for t in inp["bn"]) if inp["bn"] is not None else None
        _ORACLE_CACHE[key] = (one, inp["x"].double().numpy(), inp["w"].double().numpy(), bn)
    return _ORACLE_CACHE[key]


def _oracle_pass(specs, frac, seed_base, synthetic, min_points=16):
    import oracle
    done_flops, secs, npts = 0, 0.0, 0
    for i, spec in enumerate(specs):
        ho, wo = spec.out_hw
        count = max(min_points, int(spec.N * spec.K * ho * wo * frac))
        one, x64, w64, bn = _oracle_layer_inputs(spec, synthetic.seed_for(seed_base, i), synthetic)
        pts = synthetic.sample_points(one, count, i).numpy()
        t0 = time.perf_counter()
        oracle.conv_bn_act_points(x64, w64, None, bn, spec.act, spec.stride, spec.pads, spec.dilation,
                                  spec.group, pts)
        secs += time.perf_counter() - t0
        done_flops += pts.shape[0] * 2 * (spec.C // spec.group) * spec.R * spec.S
        npts += pts.shape[0]
    return done_flops, secs, npts


def oracle_sample(specs, budget_s, seed_base, synthetic):
    """Times the CPU oracle (conv points -> BN -> activation, float64) on a bounded random
    sample of output points of every layer (points of the first image; the per-point work is
    the layer's C*R*S multiply-adds, as in the full batch), sized by a short calibration pass to
    take about `budget_s` seconds.  Returns (flop/s, seconds, points, threads, sampled fraction)."""
    import oracle
    f0 = 2e-3
    _, s0, _ = _oracle_pass(specs, f0, seed_base, synthetic)
    frac = min(1.0, f0 * budget_s / max(s0, 1e-3))
    flops, secs, npts = _oracle_pass(specs, frac, seed_base, synthetic)
    return flops / secs, secs, npts, oracle.num_threads(), frac


def reference_arm(args):
    """--impl reference: the CPU oracle as it stands, timed on this host's cores on bounded
    samples of the same workload, reported in the same metric and unit."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from convolution_onnx_conv_gb300 import synthetic, workloads
    import oracle
    specs = workloads.resnet50_layers(32)
    per_step = 1.0      # seconds of oracle work per step
    for _ in range(args.warmup):
        oracle_sample(specs, per_step * 0.3, 3, synthetic)
    rates, secs, flops_total, pts_total = [], 0.0, 0.0, 0
    for _ in range(args.steps):
        r, s, n, threads, frac = oracle_sample(specs, per_step, 3, synthetic)
        rates.append(r)
        secs += s
        flops_total += r * s
        pts_total += n
    value = flops_total / secs / 1e12
    sample = (f"random output points of all 53 layers (fraction {frac:.2e} of each layer's outputs, "
              f"{pts_total} points over {args.steps} steps, drawn from one image per layer), float64 "
              f"seven-loop oracle + BN + ReLU")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "global_batch": 32, "sampled": True},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def profile_layers(which):
    import torch
    import convolution_onnx_conv_gb300 as cf
    from convolution_onnx_conv_gb300 import synthetic, workloads
    cf.load_library(build_if_missing=True)
    kind, idx = which.split(":")
    idx = [int(i) for i in idx.split(",")]
    if kind in ("chain", "chainrep"):
        # chain:0 the step's 52-layer chain, chain:1 ResNet-50's dataflow as one dependent chain,
        # chainrep:I six independent copies of ResNet-50 layer I (the kernel's steady state on one
        # shape): three launches, the third the profiled one
        specs = workloads.resnet50_layers(32)
        if kind == "chainrep":
            layers = build_layers([specs[idx[0]]], 3, torch, cf, synthetic)
            conv = chain_conv(layers[0]["spec"], layers[0]["inp"], cf)
            ch = cf.ConvChain([(conv, layers[0]["x"], conv.new_output()) for _ in range(6)])
        else:
            layers = build_layers(specs, 3, torch, cf, synthetic)
            ch = build_chain(layers[1:], cf)[0] if idx[0] == 0 else \
                build_network_chain(specs, layers, torch, cf, workloads, synthetic)[0]
        for _ in range(3):
            ch()
        torch.cuda.synchronize()
        print(ch.describe().split(" |")[0], "status", ch.status())
        return
    if kind == "mb":
        # fused MobileNetV2 blocks at batch 64
        blocks = workloads.mobilenetv2_blocks(64)
        layers = []
        for i in idx:
            name, N, cin, h, ch, cout, st, ex, res = blocks[i]
            inp = synthetic.block_inputs(N, cin, h, ch, cout, ex, synthetic.seed_for(11, i))
            aff = lambda bn: cf.conv_bn_scale_shift(*[t.numpy() for t in bn], 1e-5)
            blk = cf.InvertedResidualBlock(N, cin, h, h, ch, cout, st, inp["we"], aff(inp["bn_e"]) if ex else None,
                                           inp["wd"], aff(inp["bn_d"]), inp["wp"], aff(inp["bn_p"]), residual=res)
            x = inp["x"].contiguous(memory_format=torch.channels_last).cuda()
            layers.append({"spec": type("B", (), {"name": name})(), "conv": blk, "x": x, "y": blk.new_output()})
    elif kind == "q8":
        # QLinearConv on the ResNet-50 3x3 shapes at batch 64
        specs = workloads.int8_layers(64)
        layers = []
        for i in idx:
            spec = specs[i]
            inp = synthetic.qlinear_inputs(spec, synthetic.seed_for(9, i), False, True, False)
            conv = cf.QLinearConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                                  x_scale=inp["x_scale"], x_zero_point=inp["x_zp"], w_scale=inp["w_scale"].numpy(),
                                  w_zero_point=inp["w_zp"].numpy(), y_scale=inp["y_scale"],
                                  y_zero_point=inp["y_zp"], relu=True, stride=spec.stride, pads=spec.pads)
            x = inp["x"].contiguous(memory_format=torch.channels_last).cuda()
            layers.append({"spec": spec, "conv": conv, "x": x, "y": conv.new_output()})
    elif kind == "ext":
        # ResNet-50 b32 layers with bf16 output (and, on a bottleneck's last 1x1 conv, a bf16
        # residual: the staged-residual epilogue)
        specs = workloads.resnet50_layers(32)
        sel = [specs[i] for i in idx]
        layers = build_ext_layers(sel, build_layers(sel, 3, torch, cf, synthetic), torch, cf)
    else:
        table = {"r50": (workloads.resnet50_layers(32), 3, False), "dw": (workloads.depthwise_layers(64), 4, False),
                 "s8": (workloads.int8_layers(64), 5, True)}
        specs, base, s8 = table[kind]
        layers = build_layers([specs[i] for i in idx], base, torch, cf, synthetic, s8=s8)
    for _ in range(2):
        for L in layers:
            L["conv"](L["x"], L["y"], r=L.get("r"))
    torch.cuda.synchronize()
    for L in layers:
        L["conv"](L["x"], L["y"], r=L.get("r"))
        torch.cuda.synchronize()
        print(L["spec"].name, L["conv"].describe())


# ------------------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers-out", default=None, help="write per-layer results (JSONL) here")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--profile", default=None,
                    help="profiling target instead of the benchmark: 'chain:0' (the step's 52-layer chain), "
                         "'chain:1' (ResNet-50's dataflow as one chain), 'chainrep:I' (six copies of layer I as one "
                         "chain), 'r50:I,J', 'dw:I', 's8:I', 'q8:I' (QLinearConv), "
                         "'ext:I' (ResNet-50 layer with bf16 output and, on a block's last 1x1 conv, a bf16 "
                         "residual) or 'mb:I' (fused MobileNetV2 block) runs those layers twice (warm-up) and "
                         "then once more each, printing their kernel descriptions")
    args = ap.parse_args()
    if args.impl == "reference":
        return reference_arm(args)
    if args.profile:
        return profile_layers(args.profile)
    args.warmup = max(args.warmup, 3)

    import torch
    import torch.distributed as dist
    import convolution_onnx_conv_gb300 as cf
    from convolution_onnx_conv_gb300 import synthetic, workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    cf.load_library(build_if_missing=True)

    def barrier():
        if world > 1:
            dist.barrier()

    peaks, peak_src = load_peaks()
    specs = workloads.resnet50_layers(32)
    layers = build_layers(specs, 3, torch, cf, synthetic)
    stem = layers[0]
    chain, chain_convs = build_chain(layers[1:], cf)
    dw_specs = workloads.depthwise_layers(64)
    dw_layers = build_layers(dw_specs, 4, torch, cf, synthetic)
    s8_specs = workloads.int8_layers(64)
    s8_layers = build_layers(s8_specs, 5, torch, cf, synthetic, s8=True)

    def step():
        stem["conv"](stem["x"], stem["y"])
        chain()

    for _ in range(args.warmup):
        step()
        for L in layers + dw_layers + s8_layers:
            L["conv"](L["x"], L["y"])
    torch.cuda.synchronize()
    g_step = capture_fn(step, torch)            # the step: stem + the 52-layer chain
    g_r50 = capture_graph(layers, torch)        # the same 53 layers as per-layer launches
    g_chain = capture_fn(lambda: chain(), torch)  # the dominant kernel alone
    g_dw = capture_graph(dw_layers, torch)
    g_s8 = capture_graph(s8_layers, torch)
    for g in (g_step, g_r50, g_chain, g_dw, g_s8):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.1)
    barrier()
    torch.cuda.synchronize()
    total_ms = time_graph(g_step, args.steps, torch)           # the timed region: K steps
    torch.cuda.synchronize()
    barrier()
    sub_steps = max(3, args.steps // 2)
    chain_ms = time_graph(g_chain, sub_steps, torch) / sub_steps
    r50_ms = time_graph(g_r50, sub_steps, torch) / sub_steps
    lsteps = max(3, args.steps // 5)
    per_layer = time_launches(layers, lsteps, torch)
    dw_steps = max(3, args.steps // 2)
    dw_total = time_graph(g_dw, dw_steps, torch)
    dw_per = time_launches(dw_layers, lsteps, torch)
    s8_steps = max(3, args.steps // 5)
    s8_total = time_graph(g_s8, s8_steps, torch)
    s8_per = time_launches(s8_layers, lsteps, torch)
    clocks = sampler.stop()

    statuses = [L["conv"].status() for L in layers + dw_layers + s8_layers] + [chain.status()]
    if any(s != 0 for s in statuses):
        raise SystemExit(f"device status error: {statuses}")

    total_ms = max_over_ranks(total_ms, world, "cuda")
    flops_step = sum(s.flops for s in specs)
    value = whole_job_tflops(world, flops_step, args.steps, total_ms)
    ms_per_step = total_ms / args.steps

    # per-layer times of the per-layer launch path: event pairs around each launch (serialised,
    # no dependent-launch overlap) rescaled so that they add up to its graph-timed pass
    per_layer = scale_to(per_layer, lsteps, r50_ms)
    dw_per = scale_to(dw_per, lsteps, dw_total / dw_steps)
    s8_per = scale_to(s8_per, lsteps, s8_total / s8_steps)

    chain_specs = specs[1:]
    chain_flops = sum(s.flops for s in chain_specs)
    achieved = chain_flops / (chain_ms * 1e-3) / 1e12
    # attainable time of each step: its FLOPs at the tensor peak or its algorithmic bytes at the
    # HBM bandwidth, whichever is longer (the bound of that layer)
    att_ms = [attainable_ms(s, peaks) for s in chain_specs]
    tensor_layers = [s for s in chain_specs if layer_bound(s, peaks) == "tensor"]
    att_tensor_ms = sum(attainable_ms(s, peaks) for s in tensor_layers)
    chain_bytes = sum(s.algorithmic_bytes for s in chain_specs)
    achieved_gbs = chain_bytes / (chain_ms * 1e-3) / 1e9
    cd = chain.describe()
    # The launch's bound is the one that holds for most of its attainable time: with fp32 outputs
    # 38 of the 52 layers are HBM-bound and make up ~84% of the attainable time, so the roofline
    # is algorithmic bytes against the measured HBM bandwidth; the tensor view is kept beside it.
    roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": chain_traffic(),
            "traffic_note": "per launch: DRAM reads + bytes written into L2 (all of which reach DRAM), ncu; "
                            "against per_launch_algorithmic_bytes",
            "kernel": "tc_chain_kernel (tcgen05 implicit GEMM, the 52 non-stem layers as one persistent launch: "
                      + cd.split(" |")[0] + ")",
            "peak_source": f"{peak_src} HBM copy bandwidth (the kernel timed alone as one graph replay)",
            "kernel_ms_per_step": chain_ms, "launches_per_step": 1,
            "per_launch_flops": chain_flops, "launch_ms": chain_ms,
            "per_launch_algorithmic_bytes": chain_bytes,
            "tensor_view": {"achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": achieved / peaks["bf16_tflops"],
                            "peak_source": f"{peak_src} bf16 dense, burst"},
            "layer_bounds": {"tensor": len(tensor_layers), "hbm": len(chain_specs) - len(tensor_layers),
                             "attainable_ms_tensor_bound": att_tensor_ms,
                             "attainable_ms_hbm_bound": sum(att_ms) - att_tensor_ms},
            "attainable_frac": sum(att_ms) / chain_ms,
            "attainable_note": "sum over the chain's layers of max(FLOPs / bf16 burst peak, algorithmic "
                               "bytes / HBM peak), divided by the measured time of the launch"}

    # the 17 implicit-GEMM layers (stem + 16 3x3): the stem launch, a chain of the seven 3x3
    # layers with fewer than 256 channels on single CTAs and a chain of the nine wider ones on CTA
    # pairs (the tile shape each runs fastest on), one graph replay
    idx3 = [i for i, sp in enumerate(specs) if sp.R > 1 and i > 0]
    narrow3 = [i for i in idx3 if specs[i].C < 256]
    wide3 = [i for i in idx3 if specs[i].C >= 256]
    chain3 = cf.ConvChain([(chain_convs[i - 1], layers[i]["x"], layers[i]["y"]) for i in narrow3], cta_pairs=1)
    chain3w = cf.ConvChain([(chain_convs[i - 1], layers[i]["x"], layers[i]["y"]) for i in wide3], cta_pairs=2)

    def step17():
        stem["conv"](stem["x"], stem["y"])
        chain3()
        chain3w()

    step17()
    g17 = capture_fn(step17, torch)
    for _ in range(args.warmup):
        g17.replay()
    torch.cuda.synchronize()
    t17 = time_graph(g17, sub_steps, torch) / sub_steps
    f17 = specs[0].flops + sum(specs[i].flops for i in idx3)
    tf17 = f17 / (t17 * 1e-3) / 1e12
    dw_bytes = sum(s.algorithmic_bytes for s in dw_specs)
    dw_ms = dw_total / dw_steps
    dw_gbs = dw_bytes / (dw_ms * 1e-3) / 1e9
    s8_ops = sum(s.flops for s in s8_specs)
    s8_ms = s8_total / s8_steps
    s8_tops = s8_ops / (s8_ms * 1e-3) / 1e12
    s8_peak = cf.conv_fused_measure_int8_mma_rate()

    extra = other_configs(args, torch, cf, synthetic, workloads, peaks)
    extra["qlinear"] = qlinear_config(args, torch, cf, synthetic, workloads, peaks)

    # the same step with bf16 outputs and the bottleneck shortcuts (extended epilogue), per-layer
    # launches
    ext_layers = build_ext_layers(specs, layers, torch, cf)
    for _ in range(args.warmup):
        for L in ext_layers:
            L["conv"](L["x"], L["y"], r=L.get("r"))
    g_ext = capture_graph(ext_layers, torch)
    for _ in range(args.warmup):
        g_ext.replay()
    torch.cuda.synchronize()
    ext_ms = time_graph(g_ext, sub_steps, torch) / sub_steps
    ext_bf16 = sum(1 for L in ext_layers if getattr(L["conv"], "out_bf16", False))
    ext_res = sum(1 for L in ext_layers if L.get("r") is not None)
    if any(L["conv"].status() != 0 for L in ext_layers):
        raise SystemExit("device status error in the bf16-output / residual step")
    # the same bf16-output + residual step as the stem launch and one chain
    ext_chain = build_ext_chain(specs, layers, cf, workloads)

    def ext_step():
        stem["conv"](stem["x"], stem["y"])
        ext_chain()

    ext_step()
    g_extc = capture_fn(ext_step, torch)
    for _ in range(args.warmup):
        g_extc.replay()
    torch.cuda.synchronize()
    extc_ms = time_graph(g_extc, sub_steps, torch) / sub_steps
    if ext_chain.status() != 0:
        raise SystemExit("device status error in the bf16-output / residual chain")

    # ResNet-50's dataflow as one dependent chain (bf16 activations, residuals), with the stem
    net, _ = build_network_chain(specs, layers, torch, cf, workloads, synthetic)

    def net_step():
        stem["conv"](stem["x"], stem["y"])
        net()

    net_step()
    g_net = capture_fn(net_step, torch)
    for _ in range(args.warmup):
        g_net.replay()
    torch.cuda.synchronize()
    net_ms = time_graph(g_net, sub_steps, torch) / sub_steps
    if net.status() != 0 or chain3.status() != 0 or chain3w.status() != 0:
        raise SystemExit("device status error in a chain")

    # end to end through the public API with host buffers (pinned), copies inside the timing.
    # Two device buffer sets alternate between steps: while the chain of step i runs on one set,
    # step i+1's inputs go up into the other on a copy stream and step i-1's outputs come back
    # on a second one.
    e2e_steps = max(3, min(6, args.steps))
    for L in layers:
        L["x_pin"] = L["x_host"].pin_memory()
        L["y_pin"] = torch.empty_strided(L["y"].shape, L["y"].stride(), dtype=L["y"].dtype, pin_memory=True)
    h2d = sum(L["x"].numel() * L["x"].element_size() for L in layers)
    d2h = sum(L["y"].numel() * L["y"].element_size() for L in layers)
    xs2 = [torch.empty_like(L["x"]) for L in layers]
    ys2 = [torch.empty_like(L["y"]) for L in layers]
    chain2, _ = build_chain(layers[1:], cf, convs=chain_convs, xs=xs2[1:], ys=ys2[1:])
    sets = [{"x": [L["x"] for L in layers], "y": [L["y"] for L in layers], "chain": chain},
            {"x": xs2, "y": ys2, "chain": chain2}]
    s_comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    for S in sets:
        for k in ("ev_comp", "ev_out"):
            S[k] = torch.cuda.Event()
            S[k].record(s_comp)

    def e2e_step(i):
        S = sets[i % 2]
        s_in.wait_event(S["ev_comp"])        # the set's previous chain has read its inputs
        with torch.cuda.stream(s_in):
            for L, x in zip(layers, S["x"]):
                x.copy_(L["x_pin"], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
        s_comp.wait_event(ev_in)
        s_comp.wait_event(S["ev_out"])       # the set's previous outputs have been read back
        stem["conv"](S["x"][0], S["y"][0])
        S["chain"]()
        S["ev_comp"] = torch.cuda.Event()
        S["ev_comp"].record(s_comp)
        s_out.wait_event(S["ev_comp"])
        with torch.cuda.stream(s_out):
            for L, y in zip(layers, S["y"]):
                L["y_pin"].copy_(y, non_blocking=True)
            S["ev_out"] = torch.cuda.Event()
            S["ev_out"].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_comp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    for S in sets:
        s_comp.wait_event(S["ev_out"])
    e1.record(s_comp)
    torch.cuda.synchronize()
    if chain2.status() != 0:
        raise SystemExit("device status error in the end-to-end chain")
    e2e_val = whole_job_tflops(world, flops_step, e2e_steps, max_over_ranks(e0.elapsed_time(e1), world, "cuda"))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, secs, npts, threads, frac = oracle_sample(specs, args.cpu_budget, 3, synthetic)
        cpu = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{npts} random output points over all 53 layers (fraction {frac:.2e} of the "
                         f"outputs, drawn from one image per layer), float64 seven-loop conv + BN + ReLU, "
                         f"{secs:.1f} s"}

    if args.layers_out and rank == 0:
        with open(args.layers_out, "w") as f:
            for s, L, ms in zip(specs, layers, per_layer):
                ai = s.flops / s.algorithmic_bytes
                # attainable: the tensor peak or the HBM bandwidth times the layer's intensity
                att = min(peaks["bf16_tflops"], ai * peaks["hbm_gbs"] / 1e3)
                tf = s.flops / (ms * 1e-3) / 1e12
                f.write(json.dumps({"layer": s.name, "path": "per-layer launch", "kernel": L["conv"].describe(),
                                    "ms": ms, "tflops": tf, "gbs": s.algorithmic_bytes / (ms * 1e-3) / 1e9,
                                    "ai": ai, "attainable_tflops": att, "pct_attainable": tf / att}) + "\n")
            for s, L, ms in zip(dw_specs, dw_layers, dw_per):
                gbs = s.algorithmic_bytes / (ms * 1e-3) / 1e9
                f.write(json.dumps({"layer": s.name, "kernel": L["conv"].describe(), "ms": ms, "gbs": gbs,
                                    "pct_hbm": gbs / peaks["hbm_gbs"]}) + "\n")
            for s, L, ms in zip(s8_specs, s8_layers, s8_per):
                f.write(json.dumps({"layer": s.name, "kernel": L["conv"].describe(), "ms": ms,
                                    "tops": s.flops / (ms * 1e-3) / 1e12}) + "\n")

    # the stem (its channel/column pre-pass and the window kernel) and the chain
    stem_launches = 1 + ("implicit_gemm_window" in stem["conv"].describe() or
                         ("tap_channels=0" not in stem["conv"].describe() and
                          "implicit_gemm_gather" in stem["conv"].describe()))
    launches_per_step = stem_launches + 1
    per_layer_launches = sum(1 + (("tap_channels=0" not in L["conv"].describe() and
                                   "implicit_gemm_gather" in L["conv"].describe()) or
                                  "implicit_gemm_window" in L["conv"].describe()) for L in layers)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 32 * world, "parallelism": f"replicas{world}",
                       "execution": "stem launch + one conv-chain launch of the 52 other layers (independent "
                                    "steps, each on its own input)",
                       "l2": "inputs larger than L2: 53 distinct resident input/output buffer pairs, "
                             f"{(h2d + d2h) / 1e9:.2f} GB per step"},
            "pct_bf16_peak": value / peaks["bf16_tflops"],
            "implicit_gemm_3x3_7x7": {"layers": 1 + len(idx3), "tflops": tf17, "pct_bf16_peak": tf17 / peaks["bf16_tflops"],
                                      "ms": t17, "execution": "stem launch + a single-CTA chain of the seven 3x3 "
                                                              "layers with C < 256 + a CTA-pair chain of the nine "
                                                              "with C >= 256"},
            "per_layer_launches": {"workload": "the same 53 layers, one launch each (the shape-keyed selector's "
                                               "kernels), one CUDA-graph replay",
                                   "ms_per_step": r50_ms, "tflops": flops_step / (r50_ms * 1e-3) / 1e12,
                                   "launches": per_layer_launches},
            "network_chain": {"workload": "ResNet-50's own dataflow: the 52 bottleneck layers as one dependent "
                                          "chain (each layer reads the previous one's bf16 output, each block's "
                                          "last 1x1 conv adds the block's shortcut), plus the stem launch; bf16 "
                                          "activations, fp32 accumulation",
                              "ms_per_step": net_ms, "tflops": flops_step / (net_ms * 1e-3) / 1e12,
                              "pct_bf16_peak": flops_step / (net_ms * 1e-3) / 1e12 / peaks["bf16_tflops"]},
            "depthwise": {"workload": "MobileNetV2 depthwise 3x3 layers (17) at batch 64, bf16 in, fp32 out",
                          "gb_s": dw_gbs, "pct_hbm": dw_gbs / peaks["hbm_gbs"], "ms": dw_ms},
            "int8": {"workload": "ResNet-50 3x3 shapes (7) at batch 64, int8 in/out, exact int32 sums, "
                                 "fixed-point requantisation (pre-pass to exact bf16 + tcgen05 kernel per layer)",
                     "tops": s8_tops, "ms": s8_ms, "kernel": s8_layers[0]["conv"].describe().split()[0],
                     "pct_bf16_peak": s8_tops / peaks["bf16_tflops"],
                     "peak_source": "the ops run as bf16 tcgen05 MMAs (sm_103a has no tcgen05 int8 kind): "
                                    "measured bf16 dense burst peak",
                     "mma_sync_s8_rate_tops": s8_peak,
                     "vs_mma_sync_rate": s8_tops / s8_peak},
            "bf16_out_residual": {"workload": "the same 53 layers with bf16 outputs (fp32 stem) and a bf16 "
                                              "residual added in each bottleneck's last 1x1 conv: the block's "
                                              "shortcut tensor (its input, or the projection's output)",
                                  "ms_per_step": extc_ms, "tflops": flops_step / (extc_ms * 1e-3) / 1e12,
                                  "execution": "stem launch + one chain launch (the projections' outputs are "
                                               "dependencies inside the chain)",
                                  "per_layer_launches_ms": ext_ms,
                                  "bf16_layers": ext_bf16, "residual_layers": ext_res},
            **extra,
            "peaks": {**peaks, "source": peak_src},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "copies": "pinned host buffers; per step the stem + chain launches on "
                                                   "the compute stream, H2D of the inputs and D2H of the outputs "
                                                   "on two copy streams, two device buffer sets alternating so "
                                                   "that copies of neighbouring steps overlap the kernels"},
            "gpu_launches": launches_per_step * args.steps,
            "timing": "step = one CUDA-graph replay of the stem launch and the chain launch; the dominant kernel "
                      "= one graph replay of the chain launch alone; per-layer times (layer log) belong to the "
                      "per-layer launch path (event pairs around each launch, rescaled to its graph-timed pass)",
            "clocks": clocks,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
