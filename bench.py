#!/usr/bin/env python
"""Decode-step weight-stream benchmark.

Default workload: one decode step's weight stream of a 28-layer, 1536-wide
fp16 decoder (Qwen2.5-1.5B shape: q/k/v/o/gate/up/down, 196 matrices,
2,620,391,424 weight bytes), M = 1, all inputs resident in HBM.  A step is one
dg_decode_step_weights pass, replayed from a CUDA graph.  Metric: weight bytes
streamed per second (GB/s, 1e9), with microseconds per step alongside.

Prints ONE JSON line on rank 0.  Other workloads (--workload) print the same
line for their own unit of work (one call or one step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dg|reference]
                  [--workload NAME]

--impl reference times the CPU oracle (fp64 / exact-integer C, all host cores)
on a bounded sample of the same workload: the deliberately slow checker, not a
tuned CPU GEMV.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 126 * 1024 * 1024   # GB300 L2 (nvidia reports ~126 MiB usable)
FALLBACK_HBM_GBS = 6800.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---- environment facts --------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def csrc_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "quantized_skinny_gemm_gb300", "csrc")
    for n in sorted(os.listdir(d)):
        with open(os.path.join(d, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from a committed ncu capture, only if the kernel
    sources are unchanged since it was taken; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(kernel)
    if not e or e.get("csrc_hash") != csrc_hash():
        return None
    return e.get("bytes_per_launch")


def floor_seconds(bytes_per_unit, gbs):
    """Bandwidth floor: the time to move `bytes_per_unit` at `gbs` GB/s (the
    weight-read roofline of the Orange Pi AIPro post's closing paragraph)."""
    return bytes_per_unit / (gbs * 1e9)


def job_throughput_gbs(unit_bytes, steps, world, secs):
    """Whole-job weight bytes per second over all ranks, in GB/s."""
    return unit_bytes * steps * world / secs / 1e9


def max_over_ranks(secs, dist, device):
    """The slowest rank's time (every rank gets it)."""
    import torch
    t = torch.tensor([float(secs)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


CLOCK_REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def parse_clock_samples(text):
    """nvidia-smi csv rows (sm, max sm, power, 4 throttle reasons) ->
    {sm_mhz: median, sm_max_mhz, samples, reasons: [active ones]}."""
    sm, smax, reasons = [], [], set()
    for line in text.strip().splitlines():
        f = [x.strip() for x in line.split(",")]
        if len(f) < 7:
            continue
        try:
            sm.append(float(f[0]))
            smax.append(float(f[1]))
        except ValueError:
            continue
        for n, v in zip(CLOCK_REASONS, f[3:7]):
            if v.lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "samples": len(sm), "reasons": sorted(reasons)}


class ClockSampler:
    """nvidia-smi samples every 200 ms while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self):
        if not self.p:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        return parse_clock_samples(out)


# ---- workloads ----------------------------------------------------------------

class Workload:
    """Device state for one workload: step() enqueues one unit of work."""
    name = ""
    unit_bytes = 0          # algorithmic weight bytes per unit
    launches = 0            # kernels per unit
    dtype = "f16"
    config = {}


_INT4_DATA = {}


def int4_decoder_data(synth):
    """The 32-layer int4 decoder's host data (seed 0), drawn once per process:
    its W4A16, W4A8 and fp16-head variants stream the same layers."""
    if "d" not in _INT4_DATA:
        _INT4_DATA["d"] = synth.decode_int4_workload(seed=0)
    return _INT4_DATA["d"]


def build_workload(name, dev, torch):
    import quantized_skinny_gemm_gb300 as dg
    from quantized_skinny_gemm_gb300 import plans, synth

    w = Workload()
    w.name = name
    s = torch.cuda.Stream(device=dev)
    w.stream = s
    if name == "decode_fp16":
        layers = synth.decode_fp16_workload(seed=0)
        st = plans.fp16_decode_step(layers, dev)
        w.host = layers
        w.in_arena, w.out_arena = st.in_arena, st.out_arena
        w.unit_bytes = st.weight_bytes
        w.launches = st.n_launches
        w.run = lambda: dg.decode_step_weights(st.plan, st.ws, stream=s)
        w.config = workload_config(name)
        assert w.config["weight_bytes_per_step"] == st.weight_bytes
        # the step runs as one persistent kernel launch: that launch dominates
        w.dominant = ("k_step<fp16> (persistent decode-step kernel, 28 layers)", w.run, 1,
                      st.weight_bytes)
        w.cpu_sample = ("fp", layers)
        w.dtype = "f16"
    elif name in ("decode_int4_a16", "decode_int4_a8", "decode_int4_4l_a16", "decode_int4_4l_a8"):
        act = name[-3:]
        small = "_4l_" in name
        layers, head, xh = (synth.decode_int4_workload(seed=0, layers=4, vocab=0) if small
                            else int4_decoder_data(synth))
        st = plans.int4_decode_step(layers, head, xh, dev, act=act)
        w.host = (layers, head, xh)
        w.in_arena, w.out_arena = st.in_arena, st.out_arena
        w.unit_bytes = st.weight_bytes
        w.launches = st.n_launches
        w.run = lambda: dg.decode_step_weights(st.plan, st.ws, stream=s)
        w.config = workload_config(name)
        assert w.config["weight_bytes_per_step"] == st.weight_bytes
        w.dominant = ("k_step<int4 %s> (persistent decode-step kernel, 32 layers + lm_head)"
                      % act, w.run, 1, st.weight_bytes)
        w.cpu_sample = ("w4" + act, (layers, head, xh))
        w.dtype = "int4xf16" if act == "a16" else "int4xi8"
    elif name == "lm_head":
        W, x = synth.lm_head_workload(seed=0)
        ain, aout = plans.Arena(), plans.Arena()
        ix = ain.reserve(x.shape, torch.float16)
        il, it = aout.reserve((W.shape[0],), torch.float32), aout.reserve((1,), torch.int32)
        xin, outs = ain.build(dev), aout.build(dev)
        xd = xin[ix]
        xd.copy_(x)
        logits, token = outs[il], outs[it]
        Wd = W.to(dev)
        head = dg.linear(dg.LINEAR_F16, Wd, 1, W.shape[0], W.shape[1], x=xd, logits=logits,
                         token=token)
        plan = dg.StepPlan([head], [Wd, ain.buf, aout.buf])
        ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
        w.host = (W, x)
        w.in_arena, w.out_arena = ain.buf, aout.buf
        w.unit_bytes = W.numel() * 2
        w.launches = 2
        w.run = lambda: dg.decode_step_weights(plan, ws, stream=s)
        w.config = workload_config(name)
        assert w.config["weight_bytes_per_call"] == w.unit_bytes
        w.dominant = ("lm_head 248320x2048 fp16", w.run, 1, w.unit_bytes)
        w.cpu_sample = ("head", (W, x))
    elif name == "gateup_fp16":
        # the dominant launch of the fp16 decoder alone: 4 distinct gate|up pairs
        # (220 MB, larger than L2), one fused launch each
        g = synth.generator(0)
        pairs = [(synth.normal((8960, 1536), synth.W_STD, g), synth.normal((8960, 1536), synth.W_STD, g))
                 for _ in range(4)]
        x = synth.normal((1, 1536), 1.0, g)
        ain, aout = plans.Arena(), plans.Arena()
        ix = ain.reserve(x.shape, torch.float16)
        iy = [aout.reserve((1, 8960), torch.float16) for _ in range(8)]
        xin, outs = ain.build(dev), aout.build(dev)
        xd = xin[ix]
        xd.copy_(x)
        keep, ops = [ain.buf, aout.buf], []
        for i, (Wg, Wu) in enumerate(pairs):
            for j, Wh in enumerate((Wg, Wu)):
                Wd = Wh.to(dev)
                keep.append(Wd)
                ops.append(dg.linear(dg.LINEAR_F16, Wd, 1, 8960, 1536, x=xd, y=outs[iy[2 * i + j]]))
        plan = dg.StepPlan(ops, keep)
        gws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
        w.host = (pairs, x)
        w.in_arena, w.out_arena = ain.buf, aout.buf
        w.unit_bytes = 4 * 2 * 8960 * 1536 * 2
        w.launches = plans.count_launches(list(plan.array))
        w.run = lambda: dg.decode_step_weights(plan, gws, stream=s)
        w.config = workload_config(name)
        assert w.config["weight_bytes_per_step"] == w.unit_bytes
        w.dominant = ("gate|up 17920x1536 fp16", w.run, 4, 2 * 8960 * 1536 * 2)
        w.cpu_sample = ("pairs", (pairs, x))
    elif name in ("gateup_w4a16", "gateup_w4a8"):
        # the dominant launch of the int4 decoder alone: 2 layers' fused gate|up
        # (2 x 66 MB, larger than L2)
        act = name[-3:]
        layers, _, _ = synth.decode_int4_workload(seed=0, layers=2, vocab=0)
        sub = []
        for L in layers:
            L.linears = [l for l in L.linears if l.name in ("gate", "up")]
            sub.append(L)
        st = plans.int4_decode_step(sub, None, None, dev, act=act)
        w.host = sub
        w.in_arena, w.out_arena = st.in_arena, st.out_arena
        w.unit_bytes = st.weight_bytes
        w.launches = st.n_launches
        w.run = lambda: dg.decode_step_weights(st.plan, st.ws, stream=s)
        w.config = workload_config(name)
        assert w.config["weight_bytes_per_step"] == st.weight_bytes
        w.dominant = ("gate|up 28672x4096 int4", w.run, 2, st.weight_bytes // 2)
        w.cpu_sample = ("w4" + act, (sub, None, None))
        w.dtype = "int4xf16" if act == "a16" else "int4xi8"
    elif name == "decode_fp16_4l":
        # small case of the fp16 decode step (4 layers, 374 MB > L2) for ncu captures
        layers = synth.decode_fp16_workload(seed=0, layers=4)
        st = plans.fp16_decode_step(layers, dev)
        w.host = layers
        w.in_arena, w.out_arena = st.in_arena, st.out_arena
        w.unit_bytes = st.weight_bytes
        w.launches = st.n_launches
        w.run = lambda: dg.decode_step_weights(st.plan, st.ws, stream=s)
        w.config = workload_config(name)
        assert w.config["weight_bytes_per_step"] == st.weight_bytes
        w.dominant = ("decode step (persistent kernel)", w.run, 1, st.weight_bytes)
        w.cpu_sample = ("fp", layers)
    elif name in ("block_fp16_fused", "block_fp16_unfused"):
        # the 28-layer 1536-wide decoder as decoder blocks with their epilogues
        layers = synth.decode_fp16_workload(seed=0)
        hs = synth.residual_stream(len(layers), 1536, seed=0)
        st = plans.fp16_block_step(layers, hs, dev, fused=name.endswith("_fused"))
        w.host = (layers, hs)
        w.in_arena, w.out_arena = st.in_arena, st.out_arena
        w.unit_bytes = st.weight_bytes
        w.launches = st.n_launches
        w.run = lambda: st.run(stream=s)
        w.config = workload_config(name)
        assert w.config["weight_bytes_per_step"] == st.weight_bytes
        w.dominant = ("decoder-block step (%s)" % name[10:], w.run, 1, st.weight_bytes)
        w.cpu_sample = ("fp", layers)
        w.keep = st
    elif name == "decode_int4_a16_f16head":
        layers, _, xh = int4_decoder_data(synth)
        head = synth.fp16_head(128256, 4096, seed=0)
        st = plans.int4_decode_step(layers, head, xh, dev, act="a16")
        w.host = (layers, head, xh)
        w.in_arena, w.out_arena = st.in_arena, st.out_arena
        w.unit_bytes = st.weight_bytes
        w.launches = st.n_launches
        w.run = lambda: dg.decode_step_weights(st.plan, st.ws, stream=s)
        w.config = workload_config(name)
        assert w.config["weight_bytes_per_step"] == st.weight_bytes
        w.dominant = ("int4 decode step + fp16 lm_head (two persistent launches)", w.run, 1,
                      st.weight_bytes)
        w.cpu_sample = ("w4a16", (layers, None, None))
        w.dtype = "int4xf16"
    elif name == "conv1d":
        # one decode step of 24 depthwise causal-conv1d layers, 8192 channels,
        # 4 taps, SiLU (one launch per layer, in layer order)
        L, C, Wd = 24, 8192, 4
        g = synth.generator(0)
        xs = [synth.normal((1, C), 1.0, g).to(dev) for _ in range(L)]
        sts = [synth.normal((1, C, Wd - 1), 1.0, g).to(dev) for _ in range(L)]
        wts = [synth.normal((C, Wd), 0.5, g).to(dev) for _ in range(L)]
        bs = [synth.normal((C,), 0.1, g).to(dev) for _ in range(L)]
        ys = [torch.empty(1, C, dtype=torch.float16, device=dev) for _ in range(L)]
        w.host = None
        w.in_arena = torch.cat([t.view(-1) for t in xs]).view(torch.uint8)
        w.out_arena = torch.cat([t.view(-1) for t in ys]).view(torch.uint8)
        per = C * (2 * Wd + 2 * 2 * (Wd - 1) + 2 + 2 + 2)   # taps, window in+out, x, y, bias
        w.unit_bytes = L * per
        w.launches = L
        w.run = lambda: [dg.causal_conv1d_update(xs[i], sts[i], wts[i], ys[i], bias=bs[i], stream=s)
                         for i in range(L)]
        w.config = workload_config(name)
        w.dominant = ("causal-conv1d step, 8192 channels, 4 taps", w.run, L, per)
        w.cpu_sample = ("conv", (C, Wd))
        w.keep = (xs, sts, wts, bs, ys)
    elif name in ("quant_w4", "quant_w8"):
        # the load-time packers on a 14336x4096 fp16 matrix (rotating copies > 2x L2)
        N, K = 14336, 4096
        per = N * K * 2
        C = -(-2 * L2_BYTES // per)
        Ws = [synth.normal((N, K), synth.W_STD, synth.generator(i)).to(dev) for i in range(C)]
        if name == "quant_w4":
            outs = [(torch.empty(N, K // 2, dtype=torch.uint8, device=dev),
                     torch.empty(N, K // 32, dtype=torch.float16, device=dev)) for _ in range(C)]
            calls = [lambda Wd=Wd, o=o: dg.quantize_weights_w4(Wd, o[0], o[1], stream=s)
                     for Wd, o in zip(Ws, outs)]
        else:
            outs = [(torch.empty(N, K, dtype=torch.int8, device=dev),
                     torch.empty(N, dtype=torch.float32, device=dev)) for _ in range(C)]
            calls = [lambda Wd=Wd, o=o: dg.quantize_weights_i8(Wd, o[0], o[1], stream=s)
                     for Wd, o in zip(Ws, outs)]
        w.host = None
        w.in_arena = w.out_arena = None
        w.unit_bytes = C * per
        w.launches = C
        w.run = lambda: [c() for c in calls]
        w.config = workload_config(name)
        w.dominant = ("%s packer, 14336x4096 fp16 in" % name[-2:], w.run, C, per)
        w.cpu_sample = None
        w.keep = (Ws, outs)
        w.dtype = "f16->" + ("int4" if name == "quant_w4" else "i8")
    elif name in ("int4_m8", "int4_m16", "int4_a8_m16", "int4_down_m8"):
        # one int4 matrix at 8 / 16 tokens (verify block), rotating copies > 2x L2:
        # the 14336x4096 up projection, or the 4096x14336 down projection
        M = int(name.split("_m")[1])
        NW, KW = (4096, 14336) if "down" in name else (14336, 4096)
        Wq, sc, x = synth.w4_case(NW, KW, M, seed=0)
        per = Wq.numel() + sc.numel() * 2
        C = -(-2 * L2_BYTES // per)
        xd = x.to(dev)
        copies = [(Wq.to(dev), sc.to(dev)) for _ in range(C)]
        ys = [torch.empty(M, NW, dtype=torch.float16, device=dev) for _ in range(C)]
        if name == "int4_a8_m16":
            xq = torch.empty(M, KW, dtype=torch.int8, device=dev)
            xs_ = torch.empty(M, dtype=torch.float32, device=dev)
            dg.quantize_act_i8(xd, xq, xs_, stream=s)
            calls = [lambda c=c, y=y: dg.gemv_w4(c[0], c[1], y, x_i8=xq, x_scale=xs_, stream=s)
                     for c, y in zip(copies, ys)]
            w.dtype = "int4xi8"
        else:
            calls = [lambda c=c, y=y: dg.gemv_w4(c[0], c[1], y, x_f16=xd, stream=s)
                     for c, y in zip(copies, ys)]
            w.dtype = "int4xf16"
        w.host = (Wq, x)
        w.in_arena = xd.view(torch.uint8).view(-1)
        w.out_arena = torch.cat([y.view(-1) for y in ys]).view(torch.uint8)
        w.unit_bytes = C * per
        w.launches = C
        w.run = lambda: [c() for c in calls]
        w.config = workload_config(name)
        w.dominant = ("int4 %dx%d verify tile, M=%d" % (NW, KW, M), w.run, C, per)
        w.cpu_sample = ("w4a16", ([synth.Layer([synth.Linear("m", NW, KW, Wq, sc, "x")],
                                               {"x": x})], None, None))
        w.keep = (copies, ys)
    elif name == "gemv_f16_2048" or name.startswith("w8a8_m") or name.startswith("fp16_m"):
        # one matrix called repeatedly; C rotating copies (> 2x L2 in total) keep
        # every call cold.  A step is one call on each copy.
        if name == "gemv_f16_2048":
            W, x = synth.gemv_f16_workload(seed=0)
            per = W.numel() * 2
        elif name.startswith("fp16_m"):
            M = int(name[len("fp16_m"):])
            W, x = synth.fp_case(14336, 4096, M, seed=0)
            per = W.numel() * 2
        else:
            M = int(name[len("w8a8_m"):])
            W, s_w, x = synth.w8a8_workload(M=M, seed=0)
            per = W.numel() + s_w.numel() * 4
        C = -(-2 * L2_BYTES // per)
        ain, aout = plans.Arena(), plans.Arena()
        ix = ain.reserve(x.shape, torch.float16)
        iys = [aout.reserve((x.shape[0], W.shape[0]), torch.float16) for _ in range(C)]
        xin, outs = ain.build(dev), aout.build(dev)
        xd = xin[ix]
        xd.copy_(x)
        copies = [W.to(dev) for _ in range(C)]
        if name == "gemv_f16_2048" or name.startswith("fp16_m"):
            calls = [lambda Wd=Wd, y=outs[iy]: dg.gemv_f16(Wd, xd, y, stream=s)
                     for Wd, iy in zip(copies, iys)]
            w.dtype = "f16"
            desc = workload_config(name)["workload"]
            w.cpu_sample = ("pairs", ([(W, W)], x))
        else:
            swd = s_w.to(dev)
            xq = torch.empty(x.shape, dtype=torch.int8, device=dev)
            xs = torch.empty(x.shape[0], dtype=torch.float32, device=dev)
            dg.quantize_act_i8(xd, xq, xs, stream=s)
            calls = [lambda Wd=Wd, y=outs[iy]: dg.gemv_w8a8(Wd, swd, xq, xs, y=y, stream=s)
                     for Wd, iy in zip(copies, iys)]
            w.dtype = "i8"
            desc = "W8A8 14336x4096 int8 GEMV, M=%d" % M
            w.cpu_sample = ("w8", (W, s_w, x))
        w.host = (W, x)
        w.in_arena, w.out_arena = ain.buf, aout.buf
        w.unit_bytes = C * per
        w.launches = C
        w.calls = calls
        w.run = lambda: [c() for c in calls]
        w.config = workload_config(name)
        assert (w.config["bytes_per_call"], w.config["calls_per_step"]) == (per, C)
        w.dominant = (desc, w.run, C, per)
        w.keep = copies
    else:
        raise SystemExit("unknown workload %s" % name)
    return w


def workload_config(name):
    """The `config` object of a workload's JSON line, from its shapes alone
    (no device work): both arms report the same one."""
    fp16_layer = 1536 * (1536 + 256 + 256 + 1536 + 3 * 8960) * 2
    int4_layer = 4096 * (4096 + 1024 + 1024 + 4096 + 3 * 14336)
    int4_bytes = lambda n: n // 2 + n // 32 * 2  # packed codes + fp16 scales, group 32
    if name == "decode_fp16":
        return {"workload": "decode-step weight stream, 28-layer 1536-wide fp16 decoder "
                            "(Qwen2.5-1.5B shape), 196 matrices, M=1",
                "weight_bytes_per_step": 28 * fp16_layer,
                "l2": "inputs 2.62 GB > 126 MB L2 (no flush)"}
    if name == "decode_fp16_4l":
        return {"workload": "decode-step weight stream, 4 layers of the 1536-wide fp16 "
                            "decoder, 28 matrices, M=1",
                "weight_bytes_per_step": 4 * fp16_layer,
                "l2": "inputs 374 MB > 126 MB L2 (no flush)"}
    if name == "decode_int4_a16_f16head":
        nbytes = int4_bytes(32 * int4_layer) + 128256 * 4096 * 2
        return {"workload": "decode-step weight stream, 32-layer 4096-wide int4 g32 decoder "
                            "(Llama-3.1-8B shape) + fp16 128256-row lm_head with argmax, W4A16, M=1",
                "weight_bytes_per_step": nbytes,
                "l2": "inputs %.2f GB > 126 MB L2 (no flush)" % (nbytes / 1e9)}
    if name.startswith("decode_int4"):
        act = name[-3:]
        small = "_4l_" in name
        nbytes = int4_bytes(4 * int4_layer) if small else \
            int4_bytes(32 * int4_layer + 128256 * 4096)
        return {"workload": ("decode-step weight stream, 4 layers of the 4096-wide int4 g32 "
                             "decoder, W4%s, M=1" if small else
                             "decode-step weight stream, 32-layer 4096-wide int4 g32 decoder "
                             "(Llama-3.1-8B shape) + 128256-row lm_head with argmax, W4%s, M=1")
                            % act[1:].upper(),
                "weight_bytes_per_step": nbytes,
                "l2": "inputs %.2f GB > 126 MB L2 (no flush)" % (nbytes / 1e9)}
    if name == "lm_head":
        return {"workload": "lm_head 248320x2048 fp16 with fused greedy argmax, M=1",
                "weight_bytes_per_call": 248320 * 2048 * 2,
                "l2": "inputs 1.02 GB > 126 MB L2 (no flush)"}
    if name == "gateup_fp16":
        return {"workload": "fused gate|up 17920x1536 fp16 (4 distinct pairs per step), M=1",
                "weight_bytes_per_step": 4 * 17920 * 1536 * 2,
                "l2": "inputs 220 MB > 126 MB L2 (no flush)"}
    if name in ("gateup_w4a16", "gateup_w4a8"):
        return {"workload": "fused gate|up 28672x4096 int4 g32 (2 layers per step), W4%s, M=1"
                            % name[-3:][1:].upper(),
                "weight_bytes_per_step": int4_bytes(2 * 28672 * 4096),
                "l2": "inputs 132 MB > 126 MB L2 (no flush)"}
    if name in ("block_fp16_fused", "block_fp16_unfused"):
        return {"workload": "decoder-block step of the 28-layer 1536-wide fp16 decoder: "
                            "q/k/v, o + residual, gate|up -> SwiGLU, down + residual, M=1, %s"
                            % ("epilogues fused into one persistent launch" if name.endswith("_fused")
                               else "epilogues as separate launches"),
                "weight_bytes_per_step": 28 * fp16_layer,
                "l2": "inputs 2.62 GB > 126 MB L2 (no flush)"}
    if name == "conv1d":
        return {"workload": "causal-conv1d decode step, 24 layers x 8192 channels x 4 taps, "
                            "SiLU, M=1 (one launch per layer)",
                "bytes_per_step": 24 * 8192 * (8 + 12 + 6),
                "l2": "5.0 MB per step: L2-resident (the op is launch-bound)"}
    if name in ("quant_w4", "quant_w8"):
        per = 14336 * 4096 * 2
        C = -(-2 * L2_BYTES // per)
        return {"workload": "load-time %s packer, 14336x4096 fp16 weights" %
                            ("int4 g32" if name == "quant_w4" else "int8 per-channel"),
                "bytes_per_call": per, "calls_per_step": C,
                "l2": "%d rotating copies, %.0f MB > 2x L2" % (C, C * per / 1e6)}
    if name in ("int4_m8", "int4_m16", "int4_a8_m16", "int4_down_m8"):
        per = int4_bytes(14336 * 4096)
        C = -(-2 * L2_BYTES // per)
        M = int(name.split("_m")[1])
        return {"workload": "int4 g32 %s verify tile, W4%s, M=%d"
                            % ("4096x14336" if "down" in name else "14336x4096",
                               "A8" if "a8" in name else "A16", M),
                "bytes_per_call": per, "calls_per_step": C,
                "l2": "%d rotating weight copies, %.0f MB > 2x L2" % (C, C * per / 1e6)}
    if name == "gemv_f16_2048" or name.startswith("w8a8_m") or name.startswith("fp16_m"):
        if name == "gemv_f16_2048":
            per, desc = 2048 * 2048 * 2, "fp16 GEMV 2048x2048, M=1"
        elif name.startswith("fp16_m"):
            per = 14336 * 4096 * 2
            desc = "fp16 14336x4096 verify tile, M=%d" % int(name[len("fp16_m"):])
        else:
            per = 14336 * 4096 + 14336 * 4
            desc = "W8A8 14336x4096 int8 GEMV, M=%d" % int(name[len("w8a8_m"):])
        C = -(-2 * L2_BYTES // per)
        return {"workload": desc, "bytes_per_call": per, "calls_per_step": C,
                "l2": "%d rotating weight copies, %.0f MB > 2x L2" % (C, C * per / 1e6)}
    raise SystemExit("unknown workload %s" % name)


def graph_of(fn, stream, torch):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # first launch outside capture (one-time setup)
    stream.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_graph(g, stream, n, torch):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3  # seconds


def step_percentiles(g, stream, n, torch):
    """Per-step device time of n graph replays, each between its own pair of
    events on the launching stream: (median, p10, p90) in microseconds."""
    import statistics
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            g.replay()
            b.record(stream)
    torch.cuda.synchronize()
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    q = statistics.quantiles(us, n=10, method="inclusive")
    return {"median": round(statistics.median(us), 3), "p10": round(q[0], 3),
            "p90": round(q[-1], 3), "samples": n}


# ---- CPU oracle (baseline / reference arm) ------------------------------------------

def oracle_sample(w, budget_s, nthreads=0):
    """Times the oracle on whole matrices of the workload until budget_s has
    passed, on nthreads host threads (0: all cores).  Returns (weight bytes
    done, seconds, description)."""
    import numpy as np
    import oracle
    kind, data = w.cpu_sample
    done, t0 = 0, time.perf_counter()
    mats = 0

    def bits(t):
        return t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)

    if kind == "fp":
        for L in data:
            for lin in L.linears:
                oracle.gemv_fp(bits(lin.W), bits(L.inputs[lin.x_name]), nthreads=nthreads)
                done += lin.W.numel() * 2
                mats += 1
                if time.perf_counter() - t0 > budget_s:
                    break
            if time.perf_counter() - t0 > budget_s:
                break
        desc = "%d whole fp16 matrices of the decoder in layer order" % mats
    elif kind.startswith("w4"):
        layers, head, xh = data
        for L in layers:
            for lin in L.linears:
                x = L.inputs[lin.x_name]
                if kind == "w4a16":
                    oracle.gemv_w4a16(lin.W.numpy(), bits(lin.scales), bits(x), nthreads=nthreads)
                else:
                    q, s = oracle.quant_act(bits(x))
                    oracle.gemv_w4a8(lin.W.numpy(), bits(lin.scales), q, s, nthreads=nthreads)
                done += lin.W.numel() + lin.scales.numel() * 2
                mats += 1
                if time.perf_counter() - t0 > budget_s:
                    break
            if time.perf_counter() - t0 > budget_s:
                break
        desc = "%d whole int4 matrices of the decoder in layer order" % mats
    elif kind == "conv":
        C, Wd = data
        g = __import__("torch").Generator().manual_seed(0)
        T = __import__("torch")
        x = (T.randn(1, C, generator=g)).half().numpy()
        st = (T.randn(1, C, Wd - 1, generator=g)).half().numpy()
        wt = (T.randn(C, Wd, generator=g) * 0.5).half().numpy()
        b = (T.randn(C, generator=g) * 0.1).half().numpy()
        per = C * (2 * Wd + 2 * 2 * (Wd - 1) + 2 + 2 + 2)
        while True:
            oracle.causal_conv1d_update(x, st, wt, b)
            done += per
            mats += 1
            if time.perf_counter() - t0 > budget_s:
                break
        desc = "%d causal-conv1d steps of 8192 channels" % mats
    elif kind == "w8":
        import oracle as orc
        W, s_w, x = data
        q, sx = orc.quant_act(bits(x))
        while True:
            orc.gemv_w8a8(W.numpy(), s_w.numpy(), q, sx, nthreads=nthreads)
            done += W.numel() + s_w.numel() * 4
            mats += 1
            if time.perf_counter() - t0 > budget_s:
                break
        desc = "%d whole W8A8 calls" % mats
    elif kind == "pairs":
        pairs, x = data
        while True:
            for Wg, Wu in pairs:
                for Wh in (Wg, Wu):
                    oracle.gemv_fp(bits(Wh), bits(x))
                    done += Wh.numel() * 2
                    mats += 1
            if time.perf_counter() - t0 > budget_s:
                break
        desc = "%d whole %dx%d fp16 matrices" % (mats, pairs[0][0].shape[0], pairs[0][0].shape[1])
    else:
        W, x = data
        rows = W.shape[0]
        step = 15520
        for lo in range(0, rows, step):
            oracle.gemv_fp(bits(W[lo:lo + step]), bits(x))
            done += step * W.shape[1] * 2
            mats += 1
            if time.perf_counter() - t0 > budget_s:
                break
        desc = "%d 15520-row slices of the lm_head" % mats
    return done, time.perf_counter() - t0, desc


# ---- main ----------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="dg", choices=["dg", "reference"])
    ap.add_argument("--workload", default="decode_fp16",
                    choices=["decode_fp16", "decode_int4_a16", "decode_int4_a8",
                             "decode_int4_4l_a16", "decode_int4_4l_a8", "lm_head",
                             "gateup_fp16", "gateup_w4a16", "gateup_w4a8", "decode_fp16_4l",
                             "gemv_f16_2048", "w8a8_m1",
                             "w8a8_m4", "w8a8_m8", "w8a8_m16", "fp16_m8", "fp16_m16", "block_fp16_fused",
                             "block_fp16_unfused", "decode_int4_a16_f16head", "conv1d",
                             "quant_w4", "quant_w8", "int4_m8", "int4_m16", "int4_a8_m16",
                             "int4_down_m8"])
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the per-configuration measurements (the `configs` object)")
    ap.add_argument("--config-cpu-budget", type=float, default=2.0,
                    help="seconds of oracle time per configuration's cpu_baseline")
    ap.add_argument("--quick", action="store_true",
                    help="time the step only (no dominant-kernel, e2e, probe or CPU legs); "
                         "for configuration sweeps")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, world)

    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=dev)

    import quantized_skinny_gemm_gb300 as dg
    dg.load()
    log("building workload", args.workload)
    w = build_workload(args.workload, dev, torch)
    s = w.stream
    g = graph_of(w.run, s, torch)
    for _ in range(args.warmup):
        with torch.cuda.stream(s):
            g.replay()
    torch.cuda.synchronize()

    peak, peak_src = measured_peaks()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    secs = time_graph(g, s, args.steps, torch)
    torch.cuda.synchronize()
    if dist:
        secs = max_over_ranks(secs, dist, dev)
        dist.barrier()

    if args.quick:
        clk = clocks.stop()
        if rank == 0:
            print(json.dumps({"workload": args.workload, "us_per_step": secs / args.steps * 1e6,
                              "value": w.unit_bytes * args.steps * world / secs / 1e9,
                              "tune": os.environ.get("DG_TUNE", ""), "clocks": clk}), flush=True)
        return 0

    # dominant kernel alone: its launches for every layer, replayed
    dname, dfn, dlaunch, dbytes = w.dominant
    gd = graph_of(dfn, s, torch)
    nrep = max(20, args.steps // 10)
    dsecs = time_graph(gd, s, nrep, torch)
    d_launch_s = dsecs / (nrep * dlaunch)
    pct = step_percentiles(g, s, min(200, max(args.steps, 10)), torch)
    clk = clocks.stop()

    # end to end through the public API with host buffers
    e2e = measure_e2e(w, args, torch, dg, g)

    value = job_throughput_gbs(w.unit_bytes, args.steps, world, secs)
    out = {
        "metric": "decode weight-stream GB/s",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 6),
        "us_per_step": round(secs / args.steps * 1e6, 3),
        "frac_of_hbm_peak": round(value / world / peak, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded, torch.Generator seed 0)",
        "config": dict(w.config, parallelism="replicas" if world > 1 else "single GPU",
                       graph="CUDA graph replay of the step", pdl=True),
        "gpu_launches": w.launches * args.steps,
        "roofline": {"bound": "hbm", "kernel": dname, "achieved": round(dbytes / d_launch_s / 1e9, 1),
                     "peak": peak, "peak_source": peak_src + " (MEASURED_PEAKS hbm_gbs, copy)",
                     "unit": "GB/s", "frac": round(dbytes / d_launch_s / 1e9 / peak, 4),
                     "us_per_launch": round(d_launch_s * 1e6, 3),
                     "bytes_per_launch": dbytes,
                     "traffic": recorded_traffic(dname)},
        "step_us": pct,
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0:
        out["hbm_probe"] = probe_hbm(torch, dg, s)
        if world == 1 or rank == 0:
            done, cs, desc = oracle_sample(w, args.cpu_budget)
            out["cpu_baseline"] = {"value": round(done / cs / 1e9, 4), "unit": "GB/s",
                                   "cores": os.cpu_count(), "kind": "oracle",
                                   "sample": desc + " (%.1f s)" % cs}
            if args.cpu_budget > 0:  # the same oracle on one core
                d1, c1, desc1 = oracle_sample(w, args.cpu_budget / 3, nthreads=1)
                out["cpu_baseline"]["one_core"] = {"value": round(d1 / c1 / 1e9, 4),
                                                   "sample": desc1 + " (%.1f s)" % c1}
        if world == 1 and args.configs:
            out["configs"] = measure_configs(args, torch, dg, dev, peak, local)
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


# Every configuration the library is measured on, beside the headline step:
# (row of the hot-path table it exercises, workload).
CONFIG_WORKLOADS = [
    ("config 1", "gemv_f16_2048"), ("config 3", "lm_head"), ("config 4", "w8a8_m1"),
    ("config 4", "w8a8_m4"), ("config 4", "w8a8_m16"), ("config 5", "decode_int4_a16"),
    ("config 5", "decode_int4_a8"), ("NEXT-1", "int4_m16"), ("NEXT-1", "int4_a8_m16"),
    ("NEXT-1", "int4_down_m8"),
    ("NEXT-1", "fp16_m16"), ("NEXT-2", "block_fp16_fused"), ("NEXT-2", "block_fp16_unfused"),
    ("NEXT-3", "decode_int4_a16_f16head"), ("NEXT-3", "quant_w4"), ("NEXT-4", "conv1d"),
]


def measure_config(name, row, torch, dg, dev, peak, local, cpu_budget):
    """One configuration: its step replayed from a CUDA graph for about half a
    second (inputs already resident), with the clocks sampled meanwhile, the
    per-launch time of its dominant kernel, and the oracle on a bounded sample."""
    t_build = time.perf_counter()
    w = build_workload(name, dev, torch)
    t_build = time.perf_counter() - t_build
    s = w.stream
    g = graph_of(w.run, s, torch)
    for _ in range(3):
        with torch.cuda.stream(s):
            g.replay()
    torch.cuda.synchronize()
    est = time_graph(g, s, 3, torch) / 3
    steps = int(max(10, min(3000, 0.5 / max(est, 1e-7))))
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    secs = time_graph(g, s, steps, torch)
    clk = clocks.stop()
    dname, _, dlaunch, dbytes = w.dominant
    gbs = w.unit_bytes * steps / secs / 1e9
    d_launch_s = secs / steps / dlaunch
    res = {"row": row, "workload": w.config.get("workload", name),
           "us_per_step": round(secs / steps * 1e6, 3), "steps": steps,
           "value": round(gbs, 1), "unit": "GB/s", "frac": round(gbs / peak, 4),
           "launches_per_step": w.launches,
           "kernel": {"name": dname, "us_per_launch": round(d_launch_s * 1e6, 3),
                      "bytes_per_launch": dbytes,
                      "frac": round(dbytes / d_launch_s / 1e9 / peak, 4)},
           "clocks": clk, "dtype": w.dtype, "build_s": round(t_build, 1)}
    if getattr(w, "calls", None):
        # one call per replay, rotating over the copies: the cold single-launch
        # time (graph launch included) beside the graph-amortised one above
        gs = [graph_of(c, s, torch) for c in w.calls]
        n = 40 * len(gs)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for i in range(n):
                gs[i % len(gs)].replay()
            e1.record(s)
        e1.synchronize()
        res["single_launch_us"] = round(e0.elapsed_time(e1) * 1e3 / n, 3)
        res["graph_amortised_us_per_call"] = round(d_launch_s * 1e6, 3)
    if w.cpu_sample and cpu_budget > 0:
        done, cs, desc = oracle_sample(w, cpu_budget)
        res["cpu_baseline"] = {"value": round(done / cs / 1e9, 4), "unit": "GB/s",
                               "cores": os.cpu_count(), "kind": "oracle",
                               "sample": desc + " (%.1f s)" % cs}
    del w, g
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def measure_configs(args, torch, dg, dev, peak, local):
    out = {}
    t0 = time.perf_counter()
    for row, name in CONFIG_WORKLOADS:
        log("config", row, name)
        try:
            out[name] = measure_config(name, row, torch, dg, dev, peak, local, args.config_cpu_budget)
        except Exception as e:  # report, and go on with the others
            out[name] = {"row": row, "error": repr(e)[:300]}
    fu, un = out.get("block_fp16_fused"), out.get("block_fp16_unfused")
    if fu and un and "us_per_step" in fu and "us_per_step" in un:
        out["epilogue_fusion_saves_us_per_step"] = round(un["us_per_step"] - fu["us_per_step"], 3)
    out["total_s"] = round(time.perf_counter() - t0, 1)
    return out


def measure_e2e(w, args, torch, dg, g):
    """Per step, through the public API: the step's inputs from pinned host
    memory into the device input arena, the step (its CUDA graph, as captured
    from dg_decode_step_weights), and its results back into pinned host
    memory; one copy each way on the step's stream."""
    s = w.stream
    h_in = w.in_arena.detach().cpu().pin_memory()
    h_out = torch.empty(w.out_arena.shape, dtype=w.out_arena.dtype).pin_memory()
    n = max(10, min(args.steps // 5, 1000))

    def one(replay):
        with torch.cuda.stream(s):
            w.in_arena.copy_(h_in, non_blocking=True)
            if replay:
                g.replay()
            else:
                w.run()
            h_out.copy_(w.out_arena, non_blocking=True)

    res = {}
    for mode in ("graph", "eager"):
        for _ in range(3):
            one(mode == "graph")
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(s)
        for _ in range(n):
            one(mode == "graph")
        e1.record(s)
        s.synchronize()
        res[mode] = max(time.perf_counter() - t0, e0.elapsed_time(e1) / 1e3)
    secs = res["graph"]
    return {"value": round(w.unit_bytes * n / secs / 1e9, 1), "unit": "GB/s",
            "us_per_step": round(secs / n * 1e6, 2), "h2d_bytes_per_step": h_in.numel(),
            "d2h_bytes_per_step": h_out.numel(), "steps": n,
            "eager_us_per_step": round(res["eager"] / n * 1e6, 2),
            "path": "pinned host inputs -> device arena, graph of dg_decode_step_weights, "
                    "device results -> pinned host (one copy each way, wall clock)"}


def probe_hbm(torch, dg, s):
    n = 2 * 1024 ** 3
    a = torch.empty(n, dtype=torch.uint8, device=s.device)
    b = torch.empty(n, dtype=torch.uint8, device=s.device)
    sink = torch.zeros(1024, dtype=torch.int32, device=s.device)
    res = {}
    for name, fn, nbytes in (("copy", lambda: dg.probe_copy(a, b, stream=s), 2 * n),
                             ("read", lambda: dg.probe_read(a, sink, stream=s), n)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = 1e9
        for _ in range(10):
            e0.record(s)
            fn()
            e1.record(s)
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3)
        res[name + "_gbs"] = round(nbytes / best / 1e9, 1)
    del a, b
    return res


def run_reference(args, world):
    """The oracle on the host cores, same workload / metric / unit."""
    import torch  # noqa: F401  (synthetic inputs)
    from quantized_skinny_gemm_gb300 import synth

    class W:
        pass

    w = W()
    wl = args.workload
    if wl in ("decode_fp16", "decode_fp16_4l"):
        w.cpu_sample = ("fp", synth.decode_fp16_workload(seed=0, layers=1))
        cfg = "decode-step weight stream, 1536-wide fp16 decoder (Qwen2.5-1.5B shape), M=1"
    elif wl.startswith("decode_int4"):
        act = wl[-3:]
        layers, head, xh = synth.decode_int4_workload(seed=0, layers=1, vocab=0)
        w.cpu_sample = ("w4" + act, (layers, head, xh))
        cfg = ("decode-step weight stream, 4096-wide int4 g32 decoder (Llama-3.1-8B shape), "
               "W4%s, M=1" % act[1:].upper())
    elif wl == "lm_head":
        W_, x_ = synth.fp_case(15520, 2048, 1, seed=0)
        w.cpu_sample = ("head", (W_, x_))
        cfg = "lm_head 248320x2048 fp16 with fused greedy argmax, M=1"
    elif wl == "gateup_fp16":
        g = synth.generator(0)
        pair = (synth.normal((8960, 1536), synth.W_STD, g), synth.normal((8960, 1536), synth.W_STD, g))
        w.cpu_sample = ("pairs", ([pair], synth.normal((1, 1536), 1.0, g)))
        cfg = "fused gate|up 17920x1536 fp16, M=1"
    elif wl == "gemv_f16_2048":
        W_, x_ = synth.gemv_f16_workload(seed=0)
        w.cpu_sample = ("pairs", ([(W_, W_)], x_))
        cfg = "fp16 GEMV 2048x2048, M=1"
    elif wl.startswith("fp16_m"):
        W_, x_ = synth.fp_case(14336, 4096, int(wl[len("fp16_m"):]), seed=0)
        w.cpu_sample = ("pairs", ([(W_, W_)], x_))
        cfg = "fp16 14336x4096 verify tile, M=%s" % wl[len("fp16_m"):]
    else:
        M = int(wl[len("w8a8_m"):])
        W_, s_w, x_ = synth.w8a8_workload(M=M, seed=0)
        w.cpu_sample = ("w8", (W_, s_w, x_))
        cfg = "W8A8 14336x4096 int8 GEMV, M=%d" % M
    # each step: one bounded sample (~1 s of oracle work)
    main_cfg = workload_config(wl)
    for _ in range(args.warmup):
        oracle_sample(w, 0.0)
    done = secs = 0.0
    desc = ""
    for _ in range(args.steps if args.steps <= 50 else 50):
        d, s, desc = oracle_sample(w, 1.0)
        done += d
        secs += s
    v = done / secs / 1e9
    out = {"impl": "reference", "metric": "decode weight-stream GB/s", "value": round(v, 4),
           "unit": "GB/s", "n_gpus": world, "steps": min(args.steps, 50), "warmup": args.warmup,
           "ms_per_step": round(secs / min(args.steps, 50) * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": dict(main_cfg, parallelism="single GPU box, host cores",
                          sample=("each step: about 1 s of whole-matrix oracle calls over the "
                                  "same sample (%s): %s; the sample's weights are re-read every "
                                  "step, so the host caches may hold part of them, unlike the "
                                  "GPU arm's full workload" % (cfg, desc))),
           "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": os.cpu_count(),
                            "kind": "oracle", "sample": desc},
           "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
