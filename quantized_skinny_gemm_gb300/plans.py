"""Decode-step plans: a decoder's weights, inputs and outputs on the device,
marshalled once into the dg_linear array that dg_decode_step_weights runs.

The op order is the decoder's: per layer q, k, v (sharing x_attn), o, gate, up
(sharing x_mlp), down, then the lm_head.  The library fuses each run of ops
that share an input into one launch (q|k|v, gate|up).

Memory layout: weights (and scales) are separate, resident tensors, loaded
once; every activation a step reads lives in one input arena and every result
it writes in one output arena (256-byte aligned views), so moving a step's
inputs in and its results out is one copy each way.
"""
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

from . import (EPI_RESIDUAL, EPI_SWIGLU, LINEAR_F16, LINEAR_W4A16, LINEAR_W4A8, LINEAR_W8A8,
               StepPlan, decode_step_weights, linear, residual_add, swiglu)


class Arena:
    """One device buffer carved into aligned views: reserve(), then build()."""

    def __init__(self, align=256):
        self.align = align
        self.specs = []
        self.size = 0
        self.buf = None

    def reserve(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        off = self.size
        self.size = (off + nbytes + self.align - 1) // self.align * self.align
        self.specs.append((off, tuple(shape), dtype, nbytes))
        return len(self.specs) - 1

    def build(self, device):
        self.buf = torch.zeros(max(self.size, self.align), dtype=torch.uint8, device=device)
        return [self.buf[o:o + nb].view(dt).view(shape) for o, shape, dt, nb in self.specs]


@dataclass
class DeviceStep:
    plan: StepPlan
    ws: Optional[torch.Tensor]
    inputs: List[Dict[str, torch.Tensor]]      # per layer: name -> device fp16 [M][K]
    outputs: List[Dict[str, torch.Tensor]]     # per layer: matrix name -> device y [M][N]
    in_arena: torch.Tensor                     # every input of the step (uint8 bytes)
    out_arena: torch.Tensor                    # every result of the step (uint8 bytes)
    weight_bytes: int                          # weights + scales streamed per step
    n_launches: int                            # kernel launches per step
    head_logits: Optional[torch.Tensor] = None
    head_token: Optional[torch.Tensor] = None
    head_input: Optional[torch.Tensor] = None
    keep: list = field(default_factory=list)
    # W4A8: per layer, input name -> (int8 codes [M][K], fp32 scale [M]) that
    # the step writes when it quantizes that input (empty for W4A16)
    act_codes: List[Dict[str, tuple]] = field(default_factory=list)
    head_codes: Optional[tuple] = None


def _nbytes(t):
    return t.numel() * t.element_size()


def count_launches(ops, persistent=True):
    """Kernel launches (memsets excluded) dg_decode_step_weights issues for
    these ops: with the persistent kernel, one per run of single-token ops of
    one kind (per 144 fused groups); otherwise one per fused group (same kind,
    no epilogue,
    M, K, group and activation pointers, up to 4 ops, an lm_head alone), plus
    the lm_head's argmax pass and one quantization launch per fused group with
    fp16 inputs to an int8-activation kind."""
    def groups(lo, hi):
        out, i = [], lo
        while i < hi:
            a = ops[i]
            j = i + 1
            if not a.token and not a.epilogue:
                while j < hi and j - i < 4:
                    b = ops[j]
                    if (b.token or b.epilogue or b.kind != a.kind or b.M != a.M or b.K != a.K
                            or b.x != a.x
                            or b.x_i8 != a.x_i8 or b.x_scale != a.x_scale
                            or b.group_size != a.group_size):
                        break
                    j += 1
            out.append((i, j))
            i = j
        return out

    n, i = 0, 0
    while i < len(ops):
        j = i
        while persistent and j < len(ops) and ops[j].kind == ops[i].kind and ops[j].M == 1 \
                and not ops[j].acc_out:
            j += 1
        if j > i:
            g = len(groups(i, j))
            n += (g + 143) // 144
            i = j
            continue
        a, b = groups(i, len(ops))[0]
        op = ops[a]
        int8_act = op.kind in (LINEAR_W4A8, LINEAR_W8A8)
        n += 1 + (1 if op.token else 0) + (1 if int8_act and op.x else 0)
        i = b
    return n


def fp16_decode_step(layers, device, M=1) -> DeviceStep:
    """layers: synth.decode_fp16_workload(...) output (host tensors)."""
    ain, aout = Arena(), Arena()
    in_ids = [{k: ain.reserve(v.shape, torch.float16) for k, v in L.inputs.items()}
              for L in layers]
    out_ids = [{lin.name: aout.reserve((M, lin.N), torch.float16) for lin in L.linears}
               for L in layers]
    in_views, out_views = ain.build(device), aout.build(device)
    ops, keep, ins, outs = [], [], [], []
    wbytes = 0
    for L, iid, oid in zip(layers, in_ids, out_ids):
        xin = {}
        for k, v in L.inputs.items():
            xin[k] = in_views[iid[k]]
            xin[k].copy_(v)
        ys = {}
        for lin in L.linears:
            W = lin.W.to(device)
            y = out_views[oid[lin.name]]
            ops.append(linear(LINEAR_F16, W, M, lin.N, lin.K, x=xin[lin.x_name], y=y))
            keep.append(W)
            ys[lin.name] = y
            wbytes += _nbytes(W)
        ins.append(xin)
        outs.append(ys)
    keep += [ain.buf, aout.buf]
    plan = StepPlan(ops, keep)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=device)
    return DeviceStep(plan, ws, ins, outs, ain.buf, aout.buf, wbytes, count_launches(ops),
                      keep=keep)


def int4_decode_step(layers, head, x_head, device, act="a16", M=1, group=32) -> DeviceStep:
    """layers/head/x_head: synth.decode_int4_workload(...) output (host tensors).
    act="a16": fp16 activations; act="a8": per-token int8 activations, quantized
    inside the step from the fp16 inputs (scratch codes live in the workspace
    tensors kept by the plan)."""
    kind = LINEAR_W4A16 if act == "a16" else LINEAR_W4A8
    ain, aout = Arena(), Arena()
    in_ids = [{k: ain.reserve(v.shape, torch.float16) for k, v in L.inputs.items()}
              for L in layers]
    out_ids = [{lin.name: aout.reserve((M, lin.N), torch.float16) for lin in L.linears}
               for L in layers]
    head_ids = None
    if head is not None:
        head_ids = (ain.reserve(x_head.shape, torch.float16),
                    aout.reserve((head.N,), torch.float32), aout.reserve((1,), torch.int32))
    in_views, out_views = ain.build(device), aout.build(device)
    ops, keep, ins, outs = [], [], [], []
    codes = []
    wbytes = 0

    def qbufs(x):
        if act == "a16":
            return None, None
        xq = torch.empty(x.shape, dtype=torch.int8, device=device)
        xs = torch.empty(x.shape[0], dtype=torch.float32, device=device)
        keep.extend([xq, xs])
        return xq, xs

    for L, iid, oid in zip(layers, in_ids, out_ids):
        xin = {}
        for k, v in L.inputs.items():
            xin[k] = in_views[iid[k]]
            xin[k].copy_(v)
        qin = {k: qbufs(v) for k, v in xin.items()}
        codes.append({k: v for k, v in qin.items() if v[0] is not None})
        ys = {}
        for lin in L.linears:
            W, S = lin.W.to(device), lin.scales.to(device)
            y = out_views[oid[lin.name]]
            xq, xs = qin[lin.x_name]
            ops.append(linear(kind, W, M, lin.N, lin.K, w_scale=S, x=xin[lin.x_name], x_i8=xq,
                              x_scale=xs, y=y, group_size=group))
            keep += [W, S]
            ys[lin.name] = y
            wbytes += _nbytes(W) + _nbytes(S)
        ins.append(xin)
        outs.append(ys)
    logits = token = xh = None
    hcodes = None
    if head is not None and head.scales is None:
        # an fp16 lm_head after the int4 layers (a second persistent launch)
        W = head.W.to(device)
        xh = in_views[head_ids[0]]
        xh.copy_(x_head)
        logits, token = out_views[head_ids[1]], out_views[head_ids[2]]
        ops.append(linear(LINEAR_F16, W, 1, head.N, head.K, x=xh, logits=logits, token=token))
        keep.append(W)
        wbytes += _nbytes(W)
    elif head is not None:
        W, S = head.W.to(device), head.scales.to(device)
        xh = in_views[head_ids[0]]
        xh.copy_(x_head)
        logits, token = out_views[head_ids[1]], out_views[head_ids[2]]
        xq, xs = qbufs(xh)
        hcodes = (xq, xs) if xq is not None else None
        ops.append(linear(kind, W, 1, head.N, head.K, w_scale=S, x=xh, x_i8=xq, x_scale=xs,
                          logits=logits, token=token, group_size=group))
        keep += [W, S]
        wbytes += _nbytes(W) + _nbytes(S)
    keep += [ain.buf, aout.buf]
    plan = StepPlan(ops, keep)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=device)
    return DeviceStep(plan, ws, ins, outs, ain.buf, aout.buf, wbytes, count_launches(ops),
                      logits, token, xh, keep=keep, act_codes=codes, head_codes=hcodes)


@dataclass
class BlockStep:
    """A decoder-block step with its epilogues: fused (one dg_decode_step_weights
    call, residual and SwiGLU in the stream's epilogues) or unfused (the
    GEMVs, then separate elementwise launches).  run() enqueues one step."""
    run: object
    inputs: List[Dict[str, torch.Tensor]]      # per layer: x_attn, x_o, x_mlp, h
    outputs: List[Dict[str, torch.Tensor]]     # per layer: q, k, v, h1, act, h2
    in_arena: torch.Tensor
    out_arena: torch.Tensor
    weight_bytes: int
    n_launches: int
    plan: Optional[StepPlan] = None
    ws: Optional[torch.Tensor] = None
    keep: list = field(default_factory=list)


def fp16_block_step(layers, hs, device, fused=True) -> BlockStep:
    """The 1536-wide fp16 decoder as decoder blocks (synth.decode_fp16_workload
    layers, synth.residual_stream inputs hs).  Per layer: q, k, v = W x_attn;
    h1 = h + W_o x_o; act = silu(W_gate x_mlp) * (W_up x_mlp); h2 = h1 +
    W_down act.  The attention and the norms between them are not part of the
    weight stream: x_attn, x_o and x_mlp are synthetic inputs.  Fused: the
    residual adds and SwiGLU are epilogues of one persistent launch (down
    waits for act and h1 inside it).  Unfused: per layer the GEMVs of q, k, v,
    o, gate and up in one launch, then h1 = h + o, act = swiglu(gate, up),
    the down GEMV and h2 = h1 + down as launches of their own."""
    ain, aout = Arena(), Arena()
    M = 1
    names_in = ("x_attn", "x_o", "x_mlp")
    in_ids, out_ids = [], []
    for L, h in zip(layers, hs):
        hidden = h.shape[1]
        inter = next(l.N for l in L.linears if l.name == "gate")
        ids = {k: ain.reserve(L.inputs[k].shape, torch.float16) for k in names_in}
        ids["h"] = ain.reserve(h.shape, torch.float16)
        in_ids.append(ids)
        o = {n: aout.reserve((M, l.N), torch.float16) for l in L.linears for n in (l.name,)
             if n in ("q", "k", "v")}
        o["h1"] = aout.reserve((M, hidden), torch.float16)
        o["act"] = aout.reserve((M, inter), torch.float16)
        o["h2"] = aout.reserve((M, hidden), torch.float16)
        if not fused:  # the unfused GEMV outputs
            for n, width in (("o", hidden), ("gate", inter), ("up", inter), ("down", hidden)):
                o["y_" + n] = aout.reserve((M, width), torch.float16)
        out_ids.append(o)
    in_views, out_views = ain.build(device), aout.build(device)
    keep, ins, outs, wbytes = [ain.buf, aout.buf], [], [], 0
    fused_ops, per_layer = [], []
    for L, h, iid, oid in zip(layers, hs, in_ids, out_ids):
        xin = {k: in_views[iid[k]] for k in iid}
        for k in names_in:
            xin[k].copy_(L.inputs[k])
        xin["h"].copy_(h)
        ys = {k: out_views[oid[k]] for k in oid}
        W = {l.name: l.W.to(device) for l in L.linears}
        keep += list(W.values())
        wbytes += sum(_nbytes(w) for w in W.values())
        lin = {l.name: l for l in L.linears}
        mk = lambda n, x, y, **kw: linear(LINEAR_F16, W[n], M, lin[n].N, lin[n].K, x=x, y=y, **kw)
        qkv = [mk(n, xin["x_attn"], ys[n]) for n in ("q", "k", "v")]
        if fused:
            fused_ops += qkv + [
                mk("o", xin["x_o"], ys["h1"], epilogue=EPI_RESIDUAL, residual=xin["h"]),
                mk("gate", xin["x_mlp"], ys["act"], epilogue=EPI_SWIGLU, W2=W["up"]),
                mk("down", ys["act"], ys["h2"], epilogue=EPI_RESIDUAL, residual=ys["h1"])]
        else:
            head = qkv + [mk("o", xin["x_o"], ys["y_o"]), mk("gate", xin["x_mlp"], ys["y_gate"]),
                          mk("up", xin["x_mlp"], ys["y_up"])]
            down = [mk("down", ys["act"], ys["y_down"])]
            per_layer.append((StepPlan(head), StepPlan(down), xin, ys))
        ins.append(xin)
        outs.append(ys)
    if fused:
        plan = StepPlan(fused_ops, keep)
        ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=device)
        run = lambda stream=None: decode_step_weights(plan, ws, stream=stream)
        return BlockStep(run, ins, outs, ain.buf, aout.buf, wbytes, 1, plan, ws, keep)
    wsb = max(max(a.workspace_bytes(), b.workspace_bytes()) for a, b, _, _ in per_layer)
    ws = torch.empty(wsb, dtype=torch.uint8, device=device)

    def run(stream=None):
        for head, down, xin, ys in per_layer:
            decode_step_weights(head, ws, stream=stream)
            residual_add(xin["h"], ys["y_o"], ys["h1"], stream=stream)
            swiglu(ys["y_gate"], ys["y_up"], ys["act"], stream=stream)
            decode_step_weights(down, ws, stream=stream)
            residual_add(ys["h1"], ys["y_down"], ys["h2"], stream=stream)
    keep.append(per_layer)
    return BlockStep(run, ins, outs, ain.buf, aout.buf, wbytes, 5 * len(per_layer), None, ws, keep)
