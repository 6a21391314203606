"""fp16 / bf16 weights for 8..16 tokens on the tensor cores (k_fp_mma):
against the oracle's bound for ragged rows and tokens, repeated calls
bitwise identical, and a row slice of W bitwise equal to the same rows of the
whole matrix (the K split follows K alone)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, need_gpu, sync

pytestmark = pytest.mark.gpu


def _run(W, x, dtype):
    t = dg.F16 if dtype == torch.float16 else dg.BF16
    y = torch.empty(x.shape[0], W.shape[0], dtype=dtype, device=DEV)
    dg.gemv_f16(W, x, y, dtype=t)
    sync()
    return y


@pytest.mark.parametrize("N,K,M", [(1000, 1536, 16), (4097, 4096, 8), (17, 2048, 9),
                                   (16, 32, 16), (1, 1024, 12), (333, 6144, 16)])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_fp_mma_against_the_oracle(N, K, M, dtype):
    need_gpu()
    W, x = synth.fp_case(N, K, M, seed=N + K + M, dtype=dtype)
    Wd, xd = W.to(DEV), x.to(DEV)
    y = _run(Wd, xd, dtype)
    assert torch.equal(y, _run(Wd, xd, dtype))  # the same order on every call
    fmt = "f16" if dtype == torch.float16 else "bf16"
    yr, A = oracle.gemv_fp(bits(W), bits(x), fmt)
    tol.assert_close(y.float().cpu().double().numpy(), yr, A, fmt, "mma %dx%d M=%d" % (N, K, M))


def test_fp_mma_row_slice_equals_the_whole_matrix():
    need_gpu()
    N, K, M = 4096, 4096, 16
    W, x = synth.fp_case(N, K, M, seed=7)
    Wd, xd = W.to(DEV), x.to(DEV)
    full = _run(Wd, xd, torch.float16)
    for r0, r1 in ((0, 1000), (1000, 1003), (1003, 4096), (2048, 2064)):
        part = _run(Wd[r0:r1].contiguous(), xd, torch.float16)
        assert torch.equal(part, full[:, r0:r1]), (r0, r1)


def test_fp_mma_one_hot_rows_select_the_activation():
    """W[i] = e_j: y[m][i] = x[m][j] exactly (fp16 in, fp32 sum, fp16 out)."""
    need_gpu()
    N, K, M = 64, 2048, 16
    g = synth.generator(11)
    x = synth.normal((M, K), 1.0, g)
    cols = torch.randint(0, K, (N,), generator=g)
    W = torch.zeros(N, K, dtype=torch.float16)
    W[torch.arange(N), cols] = 1.0
    y = _run(W.to(DEV), x.to(DEV), torch.float16)
    assert torch.equal(y.cpu(), x[:, cols])
