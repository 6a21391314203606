"""Cases run by test_gpu_tc_grid.py in child processes whose DG_TUNE forces
the fp16 / bf16 tcgen05 tile's grid (TG=g) to a size other than the SM count
(named without the test_ prefix so the main session does not collect it with
its own settings).

The stream-K split hands each CTA an equal contiguous range of (row tile,
64-k block) pairs; a CTA whose range ends inside a tile processes that tile
first, and the CTA holding a tile's last k block finishes the tile, either
after one acquire load finds every other piece there or through the
publish / atomic protocol.  Forcing grids of 5, 37, 151 and 256 CTAs (more
CTAs than SMs, and ranges shorter and longer than a tile) puts every piece
shape through both finishing paths: results against the oracle's bound,
repeated calls bitwise identical, untouched memory past y."""
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, need_gpu, sync

pytestmark = pytest.mark.gpu


def _fmt(dtype):
    return "f16" if dtype == torch.float16 else "bf16"


@pytest.mark.parametrize("N,K,M", [(1000, 1536, 16), (4097, 4096, 8), (300, 8, 8), (129, 4104, 11),
                                   (5, 65600, 10), (2000, 520, 13), (6144, 2048, 16), (256, 14336, 9)])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_forced_grid_against_the_oracle(N, K, M, dtype):
    need_gpu()
    W, x = synth.fp_case(N, K, M, seed=3 * N + K + M, dtype=dtype)
    Wd, xd = W.to(DEV), x.to(DEV)
    t = dg.F16 if dtype == torch.float16 else dg.BF16
    buf = torch.full((M + 1, N), 3.0, dtype=dtype, device=DEV)
    y = buf[:M]
    dg.gemv_f16(Wd, xd, y, dtype=t)
    y2 = torch.empty_like(y)
    dg.gemv_f16(Wd, xd, y2, dtype=t)
    sync()
    assert torch.equal(y, y2)  # the same order on every call
    assert torch.all(buf[M] == 3.0)
    yr, A = oracle.gemv_fp(bits(W), bits(x), _fmt(dtype))
    tol.assert_close(y.float().cpu().double().numpy(), yr, A, _fmt(dtype), "grid %dx%d M=%d" % (N, K, M))


@pytest.mark.parametrize("M", [8, 16])
def test_forced_grid_fused_segments(M):
    """q|k|v as one launch of three matrices (tiles never straddle two) under
    the forced grid, through the per-group path of dg_decode_step_weights."""
    need_gpu()
    K = 2048
    Ns = (2048, 256, 384)
    g = synth.generator(90 + M)
    Ws = [synth.normal((n, K), synth.W_STD, g) for n in Ns]
    x = synth.normal((M, K), 1.0, g)
    xd = x.to(DEV)
    ys = [torch.empty(M, n, dtype=torch.float16, device=DEV) for n in Ns]
    Wd = [W.to(DEV) for W in Ws]
    ops = [dg.linear(dg.LINEAR_F16, W, M, n, K, x=xd, y=y) for W, n, y in zip(Wd, Ns, ys)]
    plan = dg.StepPlan(ops, Wd + ys + [xd])
    ws = torch.empty(max(plan.workspace_bytes(), 16), dtype=torch.uint8, device=DEV)
    dg.decode_step_weights(plan, ws)
    sync()
    first = [y.clone() for y in ys]
    dg.decode_step_weights(plan, ws)
    sync()
    for W, y, y0, n in zip(Ws, ys, first, Ns):
        assert torch.equal(y, y0)
        yr, A = oracle.gemv_fp(bits(W), bits(x), "f16")
        tol.assert_close(y.float().cpu().double().numpy(), yr, A, "f16", "segment N=%d M=%d" % (n, M))
