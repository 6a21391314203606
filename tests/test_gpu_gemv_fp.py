"""fp16 / bf16 weight-streaming GEMV against the oracle (C ABI dg_gemv_f16)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, as_f64, bits, need_gpu, sync

pytestmark = pytest.mark.gpu


def run(W, x, dtype):
    N, K = W.shape
    M = x.shape[0]
    y = torch.empty(M, N, dtype=W.dtype, device=DEV)
    dg.gemv_f16(W.to(DEV), x.to(DEV), y, dtype)
    sync()
    return y


def check(W, x, y, dtype, what):
    fmt = "f16" if dtype == dg.F16 else "bf16"
    yr, A = oracle.gemv_fp(bits(W), bits(x), fmt)
    tol.assert_close(as_f64(y), yr, A, fmt, what)


def test_gemv_2048_square_seed0():
    need_gpu()
    W, x = synth.gemv_f16_workload(seed=0)
    check(W, x, run(W, x, dg.F16), dg.F16, "2048x2048 fp16 M=1")


@pytest.mark.parametrize("dtype", [dg.F16, dg.BF16])
@pytest.mark.parametrize("N,K,M", [(1, 8, 1), (7, 8, 1), (33, 24, 1), (1000, 520, 1),
                                   (4097, 1536, 1), (257, 8960, 1), (300, 2048, 2),
                                   (129, 1536, 3), (64, 4096, 4), (515, 1024, 8),
                                   (99, 1536, 16), (17, 17920, 1), (1536, 8960, 1)])
def test_gemv_shapes(dtype, N, K, M):
    need_gpu()
    tdt = torch.float16 if dtype == dg.F16 else torch.bfloat16
    W, x = synth.fp_case(N, K, M, seed=N + K + M, dtype=tdt)
    check(W, x, run(W, x, dtype), dtype, "N=%d K=%d M=%d" % (N, K, M))


def test_bf16_lm_head_shape():
    need_gpu()
    W, x = synth.fp_case(248320, 2048, 1, seed=3, dtype=torch.bfloat16)
    y = run(W, x, dg.BF16)
    rows = np.random.default_rng(0).integers(0, 248320, 4096)
    yr, A = oracle.gemv_fp(bits(W), bits(x), "bf16", rows=rows)
    tol.assert_close(as_f64(y)[:, rows], yr, A, "bf16", "bf16 248320x2048 sampled")


def test_identity_one_hot_and_ones_are_exact():
    need_gpu()
    K = 1024
    x = synth.normal((1, K), 1.0, synth.generator(5))
    y = run(torch.eye(K, dtype=torch.float16), x, dg.F16)
    assert torch.equal(y.cpu(), x)  # every row selects one element: exact
    cols = torch.randint(0, K, (300,), generator=synth.generator(6))
    Wh = torch.zeros(300, K, dtype=torch.float16)
    Wh[torch.arange(300), cols] = 1
    y = run(Wh, x, dg.F16)
    assert torch.equal(y.cpu()[0], x[0, cols])
    y = run(torch.ones(2, K, dtype=torch.float16), x, dg.F16)
    ref = np.float16(np.sum(x.double().numpy()))
    assert abs(float(y[0, 0]) - float(ref)) <= float(tol.ulp_f16(float(ref)))


def test_repeated_calls_are_bitwise_identical():
    need_gpu()
    W, x = synth.fp_case(8960, 1536, 1, seed=7)
    Wd, xd = W.to(DEV), x.to(DEV)
    y0 = torch.empty(1, 8960, dtype=torch.float16, device=DEV)
    dg.gemv_f16(Wd, xd, y0)
    for _ in range(10):
        y = torch.empty_like(y0)
        dg.gemv_f16(Wd, xd, y)
        sync()
        assert torch.equal(y, y0)


def test_row_slices_reproduce_full_rows_bitwise():
    need_gpu()
    W, x = synth.fp_case(4000, 3072, 1, seed=8)
    Wd, xd = W.to(DEV), x.to(DEV)
    full = torch.empty(1, 4000, dtype=torch.float16, device=DEV)
    dg.gemv_f16(Wd, xd, full)
    for lo, hi in [(0, 1), (1, 250), (250, 2017), (2017, 4000)]:
        part = torch.empty(1, hi - lo, dtype=torch.float16, device=DEV)
        dg.gemv_f16(Wd[lo:hi], xd, part)
        sync()
        assert torch.equal(part, full[:, lo:hi])
