"""Epilogues fused into the weight stream (dg_linear_forward, per op): the
residual add y = r + W x and SwiGLU y = silu(W x) * (W2 x), for fp16, bf16,
W4A16, W4A8 and (residual only) W8A8, at one token and at several tokens,
ragged N; checked against the oracle's definitions within the bounds derived
for them (oracle/tolerance.py)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, host, need_gpu, sync

pytestmark = pytest.mark.gpu


def _fp(N, K, M, seed, dtype=torch.float16):
    W, x = synth.fp_case(N, K, M, seed=seed, dtype=dtype)
    g = synth.generator(seed + 100)
    W2 = synth.normal((N, K), synth.W_STD, g, dtype)
    r = synth.normal((M, N), 1.0, g, dtype)
    return W, W2, x, r


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("N,K,M", [(333, 512, 1), (1000, 1536, 1), (257, 1024, 3), (129, 2048, 16)])
def test_residual_fp(fmt, N, K, M):
    need_gpu()
    dt = torch.float16 if fmt == "f16" else torch.bfloat16
    W, _, x, r = _fp(N, K, M, seed=N + K + M, dtype=dt)
    Wd, xd, rd = W.to(DEV), x.to(DEV), r.to(DEV)
    y = torch.empty(M, N, dtype=dt, device=DEV)
    kind = dg.LINEAR_F16 if fmt == "f16" else dg.LINEAR_BF16
    dg.linear_forward(dg.linear(kind, Wd, M, N, K, x=xd, y=y, epilogue=dg.EPI_RESIDUAL,
                                residual=rd))
    sync()
    yr, A = oracle.gemv_residual_fp(bits(W), bits(x), bits(r), fmt)
    tol.assert_close(host(y).astype(np.float64) if fmt == "f16" else
                     oracle.decode_bf16(host(y)).reshape(M, N), yr, A, fmt, "residual %s" % fmt)


def test_residual_in_place_equals_out_of_place():
    need_gpu()
    N, K, M = 777, 1024, 2
    W, _, x, r = _fp(N, K, M, seed=3)
    Wd, xd = W.to(DEV), x.to(DEV)
    out = torch.empty(M, N, dtype=torch.float16, device=DEV)
    rd = r.to(DEV)
    dg.linear_forward(dg.linear(dg.LINEAR_F16, Wd, M, N, K, x=xd, y=out,
                                epilogue=dg.EPI_RESIDUAL, residual=rd))
    inplace = r.to(DEV)
    dg.linear_forward(dg.linear(dg.LINEAR_F16, Wd, M, N, K, x=xd, y=inplace,
                                epilogue=dg.EPI_RESIDUAL, residual=inplace))
    sync()
    assert torch.equal(out, inplace)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("N,K,M", [(333, 512, 1), (2001, 1536, 1), (64, 1024, 4), (97, 1024, 16)])
def test_swiglu_fp(fmt, N, K, M):
    need_gpu()
    dt = torch.float16 if fmt == "f16" else torch.bfloat16
    W, W2, x, _ = _fp(N, K, M, seed=2 * N + K + M, dtype=dt)
    y = torch.empty(M, N, dtype=dt, device=DEV)
    kind = dg.LINEAR_F16 if fmt == "f16" else dg.LINEAR_BF16
    dg.linear_forward(dg.linear(kind, W.to(DEV), M, N, K, x=x.to(DEV), y=y,
                                epilogue=dg.EPI_SWIGLU, W2=W2.to(DEV)))
    sync()
    h, g, u, Ag, Au = oracle.gemv_swiglu_fp(bits(W), bits(W2), bits(x), fmt)
    got = host(y).astype(np.float64) if fmt == "f16" else oracle.decode_bf16(host(y)).reshape(M, N)
    tol.assert_within(got, h, tol.bound_swiglu(g, u, Ag, Au, fmt), "swiglu %s" % fmt)


def _w4(N, K, M, seed, group=32):
    Wq, sc, x = synth.w4_case(N, K, M, seed=seed, group=group)
    Wq2, sc2, _ = synth.w4_case(N, K, M, seed=seed + 7, group=group)
    r = synth.normal((M, N), 1.0, synth.generator(seed + 9))
    return Wq, sc, Wq2, sc2, x, r


@pytest.mark.parametrize("act", ["a16", "a8"])
@pytest.mark.parametrize("N,K,M,group", [(999, 4096, 1, 32), (14336 // 8, 4096, 1, 128),
                                         (300, 1024, 2, 32), (45, 512, 16, 64)])
def test_swiglu_and_residual_int4(act, N, K, M, group):
    need_gpu()
    Wq, sc, Wq2, sc2, x, r = _w4(N, K, M, seed=N + K + M + group, group=group)
    xd = x.to(DEV)
    kind = dg.LINEAR_W4A16 if act == "a16" else dg.LINEAR_W4A8
    kw = {}
    q = s = None
    if act == "a8":
        xq = torch.empty(M, K, dtype=torch.int8, device=DEV)
        xs = torch.empty(M, dtype=torch.float32, device=DEV)
        dg.quantize_act_i8(xd, xq, xs)
        kw = dict(x_i8=xq, x_scale=xs)
        q, s = oracle.quant_act(bits(x))
    else:
        kw = dict(x=xd)
    y = torch.empty(M, N, dtype=torch.float16, device=DEV)
    dg.linear_forward(dg.linear(kind, Wq.to(DEV), M, N, K, w_scale=sc.to(DEV), y=y,
                                group_size=group, epilogue=dg.EPI_SWIGLU, W2=Wq2.to(DEV),
                                w2_scale=sc2.to(DEV), **kw))
    yr = torch.empty(M, N, dtype=torch.float16, device=DEV)
    dg.linear_forward(dg.linear(kind, Wq.to(DEV), M, N, K, w_scale=sc.to(DEV), y=yr,
                                group_size=group, epilogue=dg.EPI_RESIDUAL,
                                residual=r.to(DEV), **kw))
    sync()
    if act == "a16":
        h, g, u, Ag, Au = oracle.gemv_swiglu_w4a16(Wq.numpy(), bits(sc), Wq2.numpy(), bits(sc2),
                                                   bits(x), group)
        ref, A = oracle.gemv_residual_w4a16(Wq.numpy(), bits(sc), bits(x), bits(r), group)
    else:
        h, g, u, Ag, Au = oracle.gemv_swiglu_w4a8(Wq.numpy(), bits(sc), Wq2.numpy(), bits(sc2),
                                                  q, s, group)
        z, A, _ = oracle.gemv_w4a8(Wq.numpy(), bits(sc), q, s, group)
        ref = oracle.decode_f16(bits(r)).reshape(M, N) + z
    tol.assert_within(host(y).astype(np.float64), h, tol.bound_swiglu(g, u, Ag, Au),
                      "int4 %s swiglu" % act)
    tol.assert_close(host(yr).astype(np.float64), ref, A, "f16", "int4 %s residual" % act)


def test_residual_w8a8_per_channel_scales():
    need_gpu()
    N, K, M = 1111, 4096, 4
    W, s_w, x = synth.w8_case(N, K, M, seed=21)
    r = synth.normal((M, N), 1.0, synth.generator(22))
    xd = x.to(DEV)
    xq = torch.empty(M, K, dtype=torch.int8, device=DEV)
    xs = torch.empty(M, dtype=torch.float32, device=DEV)
    dg.quantize_act_i8(xd, xq, xs)
    y = torch.empty(M, N, dtype=torch.float16, device=DEV)
    dg.linear_forward(dg.linear(dg.LINEAR_W8A8, W.to(DEV), M, N, K, w_scale=s_w.to(DEV),
                                x_i8=xq, x_scale=xs, y=y, epilogue=dg.EPI_RESIDUAL,
                                residual=r.to(DEV)))
    sync()
    q, s = oracle.quant_act(bits(x))
    _, z, A = oracle.gemv_w8a8(W.numpy(), s_w.numpy(), q, s)
    ref = oracle.decode_f16(bits(r)).reshape(M, N) + z
    tol.assert_close(host(y).astype(np.float64), ref, A, "f16", "w8a8 residual")


def test_elementwise_swiglu_and_residual_kernels():
    need_gpu()
    g = synth.generator(31)
    n = 8960 * 3
    a = synth.normal((n,), 3.0, g)
    b = synth.normal((n,), 3.0, g)
    a[:8] = torch.tensor([0, -0.0, 100, -100, 20, -20, 1e-4, 60000], dtype=torch.float16)
    b[:8] = 0.5
    h = torch.empty(n, dtype=torch.float16, device=DEV)
    o = torch.empty(n, dtype=torch.float16, device=DEV)
    dg.swiglu(a.to(DEV), b.to(DEV), h)
    dg.residual_add(a.to(DEV), b.to(DEV), o)
    sync()
    av, bv = a.double().numpy(), b.double().numpy()
    # inputs are exact (errors e = 0): only the fp32 evaluation and the rounding remain
    tol.assert_within(host(h).astype(np.float64), oracle.silu(av) * bv,
                      tol.bound_swiglu(av, bv, np.zeros(n), np.zeros(n)), "swiglu kernel")
    tol.assert_close(host(o).astype(np.float64), av + bv, np.zeros(n), "f16", "residual kernel")
