"""Seeded synthetic inputs for the decode-step skinny GEMV workloads.

This module only draws random numbers: it holds none of the method's
arithmetic (no products, sums, scales applied, quantization or argmax) and
serves both the CUDA path and the CPU oracle, which each consume the same host
arrays.  Everything is drawn on the CPU with a ``torch.Generator`` seeded per
workload, in a fixed order, so a workload is reproducible bit for bit on any
host.  fp16 values are drawn as fp32 normals and cast with round-to-nearest-even.

INT4 weights are drawn as codes in [-7, 7] and written in the library's input
layout (row-major [N][K/2] bytes, byte j holding k = 2j in bits 0-3 and
k = 2j+1 in bits 4-7, 4-bit two's complement) -- an input format, decoded
independently by the oracle and by the kernels.

Workloads (the shapes of the decoders the pages run single-request decode on):

* ``gemv_f16``     -- W [2048 x 2048] ~N(0, 0.02), x [2048] ~N(0, 1), seed 0.
* ``decode_fp16``  -- 28-layer, 1536-wide decoder (Qwen2.5-1.5B shape): per layer
  q 1536x1536, k 256x1536, v 256x1536, o 1536x1536, gate 8960x1536,
  up 8960x1536, down 1536x8960, fp16 ~N(0, 0.02); then per layer four inputs
  x_attn, x_o, x_mlp [1536] and x_down [8960] ~N(0, 1).
* ``lm_head``      -- W [248320 x 2048] ~N(0, 0.02), x [2048] ~N(0, 1).
* ``w8a8``         -- W int8 [14336 x 4096] uniform in [-127, 127], per-channel
  fp32 scale ~U(1e-3, 1e-2), activations x [M x 4096] fp16 ~N(0, 1) (quantized
  per token by the path under test).
* ``decode_int4``  -- 32-layer, 4096-wide decoder (Llama-3.1-8B shape): q 4096x4096,
  k 1024x4096, v 1024x4096, o 4096x4096, gate 14336x4096, up 14336x4096,
  down 4096x14336, plus lm_head 128256x4096; int4 codes uniform in [-7, 7],
  group 32 along K, fp16 scales ~U(1e-3, 1e-2); per layer x_attn, x_o, x_mlp
  [4096], x_down [14336] and the lm_head input [4096], fp16 ~N(0, 1).
"""
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

W_STD = 0.02


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def normal(shape, std, g, dtype=torch.float16):
    """fp32 normal draws cast (round to nearest even) to ``dtype``."""
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(dtype)


def uniform(shape, lo, hi, g, dtype=torch.float32):
    return (torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo).to(dtype)


def int8_codes(shape, g, lo=-127, hi=127):
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int8)


def int4_packed(N, K, g, lo=-7, hi=7):
    """Codes uniform in [lo, hi] written as [N][K/2] bytes (see module doc)."""
    codes = torch.randint(lo, hi + 1, (N, K), generator=g, dtype=torch.int16)
    nib = codes & 0xF
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).to(torch.uint8)


# ---- single matrices -------------------------------------------------------

def fp_case(N, K, M=1, seed=0, dtype=torch.float16, w_std=W_STD):
    g = generator(seed)
    W = normal((N, K), w_std, g, dtype)
    x = normal((M, K), 1.0, g, dtype)
    return W, x


def w8_case(N, K, M=1, seed=0):
    g = generator(seed)
    W = int8_codes((N, K), g)
    s_w = uniform((N,), 1e-3, 1e-2, g)
    x = normal((M, K), 1.0, g)
    return W, s_w, x


def w4_case(N, K, M=1, seed=0, group=32):
    g = generator(seed)
    Wq = int4_packed(N, K, g)
    scales = uniform((N, K // group), 1e-3, 1e-2, g, torch.float16)
    x = normal((M, K), 1.0, g)
    return Wq, scales, x


# ---- the named workloads ---------------------------------------------------

def gemv_f16_workload(seed=0):
    return fp_case(2048, 2048, 1, seed)


def lm_head_workload(seed=0, N=248320, K=2048):
    return fp_case(N, K, 1, seed)


def w8a8_workload(M=1, seed=0, N=14336, K=4096):
    return w8_case(N, K, M, seed)


@dataclass
class Linear:
    """One matrix of a decoder layer, in the library's input layout."""
    name: str
    N: int
    K: int
    W: torch.Tensor                       # fp16 [N][K] or packed int4 uint8 [N][K/2]
    scales: Optional[torch.Tensor] = None  # fp16 [N][K/32] for int4
    x_name: str = ""                       # which layer input feeds it


@dataclass
class Layer:
    linears: List[Linear] = field(default_factory=list)
    inputs: Dict[str, torch.Tensor] = field(default_factory=dict)


# Decoder layer order: attention inputs feed q, k, v; o; the MLP input feeds
# gate and up; down reads the MLP's inner activation.
def _layer_shapes(hidden, kv, inter):
    return [("q", hidden, hidden, "x_attn"), ("k", kv, hidden, "x_attn"),
            ("v", kv, hidden, "x_attn"), ("o", hidden, hidden, "x_o"),
            ("gate", inter, hidden, "x_mlp"), ("up", inter, hidden, "x_mlp"),
            ("down", hidden, inter, "x_down")]


def _input_shapes(hidden, inter):
    return [("x_attn", hidden), ("x_o", hidden), ("x_mlp", hidden), ("x_down", inter)]


QWEN25_15B = dict(layers=28, hidden=1536, kv=256, inter=8960)
LLAMA31_8B = dict(layers=32, hidden=4096, kv=1024, inter=14336, vocab=128256)


def decode_fp16_workload(seed=0, layers=28, hidden=1536, kv=256, inter=8960, M=1):
    """All weights first (layer by layer, in decoder order), then the inputs."""
    g = generator(seed)
    out = []
    for _ in range(layers):
        L = Layer()
        for name, N, K, xn in _layer_shapes(hidden, kv, inter):
            L.linears.append(Linear(name, N, K, normal((N, K), W_STD, g), None, xn))
        out.append(L)
    for L in out:
        for xn, K in _input_shapes(hidden, inter):
            L.inputs[xn] = normal((M, K), 1.0, g)
    return out


def decode_int4_workload(seed=0, layers=32, hidden=4096, kv=1024, inter=14336,
                         vocab=128256, group=32, M=1):
    """Layers' weights and scales (decoder order), the lm_head, then inputs.
    Returns (layers, lm_head Linear, lm_head input)."""
    g = generator(seed)
    out = []
    for _ in range(layers):
        L = Layer()
        for name, N, K, xn in _layer_shapes(hidden, kv, inter):
            Wq = int4_packed(N, K, g)
            sc = uniform((N, K // group), 1e-3, 1e-2, g, torch.float16)
            L.linears.append(Linear(name, N, K, Wq, sc, xn))
        out.append(L)
    head = None
    if vocab:
        Wq = int4_packed(vocab, hidden, g)
        sc = uniform((vocab, hidden // group), 1e-3, 1e-2, g, torch.float16)
        head = Linear("lm_head", vocab, hidden, Wq, sc, "x_head")
    for L in out:
        for xn, K in _input_shapes(hidden, inter):
            L.inputs[xn] = normal((M, K), 1.0, g)
    x_head = normal((M, hidden), 1.0, g) if vocab else None
    return out, head, x_head


def weight_bytes(linears) -> int:
    """Bytes of weights (and scales) a list of Linear holds."""
    tot = 0
    for l in linears:
        tot += l.W.numel() * l.W.element_size()
        if l.scales is not None:
            tot += l.scales.numel() * l.scales.element_size()
    return tot


def residual_stream(layers, hidden, seed=0, M=1):
    """Per layer, the residual-stream input h [M][hidden] ~N(0, 1) of a decoder
    block whose o and down projections add into it (drawn from their own
    generator, so the decoder workloads above are unchanged)."""
    g = generator(seed + 7919)
    return [normal((M, hidden), 1.0, g) for _ in range(layers)]


def fp16_head(vocab, hidden, seed=0):
    """An fp16 lm_head [vocab][hidden] ~N(0, 0.02) for the int4 decoder (its own
    generator, so the int4 workload's draws are unchanged)."""
    g = generator(seed + 104729)
    return Linear("lm_head", vocab, hidden, normal((vocab, hidden), W_STD, g), None, "x_head")
