"""Split-K across CTAs for per-op calls with few rows: when a dg_gemv_* call
gets a workspace and its row groups would fill fewer than half of the SMs, K
is cut into S ranges, CTAs write partial sums [S][M][N] to the workspace and a
second kernel adds them in range order.  Checked against the oracle's bound,
for determinism, for the pass-2 sum (the workspace planes added in order on
the host give y), and, for W8A8, bitwise against the unsplit call (integer
sums are exact)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, need_gpu, sync

pytestmark = pytest.mark.gpu


def _ws(kind, M, N, K, **kw):
    op = dg.Linear(kind=kind, M=M, N=N, K=K, W=16, x=16, y=16, **kw)
    return torch.zeros(dg.workspace_bytes([op]), dtype=torch.uint8, device=DEV)


def _planes(ws, M, N):
    """The workspace's partial planes that the split wrote (fp32 view)."""
    f = ws.view(torch.float32)[: 8 * M * N].view(8, M, N).cpu()
    used = [s for s in range(8) if torch.count_nonzero(f[s].view(torch.int32)) > 0]
    assert used == list(range(len(used))) and len(used) >= 2, used
    return f[: len(used)]


@pytest.mark.parametrize("N,K,M,dtype", [(256, 1536, 1, torch.float16),
                                         (257, 2048, 1, torch.float16),
                                         (300, 1024, 4, torch.float16),
                                         (256, 2048, 1, torch.bfloat16)])
def test_fp_split_k(N, K, M, dtype):
    need_gpu()
    W, x = synth.fp_case(N, K, M, seed=N + K, dtype=dtype)
    Wd, xd = W.to(DEV), x.to(DEV)
    t = dg.F16 if dtype == torch.float16 else dg.BF16
    ws = _ws(dg.LINEAR_F16 if t == dg.F16 else dg.LINEAR_BF16, M, N, K)
    y1 = torch.empty(M, N, dtype=dtype, device=DEV)
    y2 = torch.empty_like(y1)
    dg.gemv_f16(Wd, xd, y1, dtype=t, ws=ws)
    sync()
    planes = _planes(ws, M, N)
    dg.gemv_f16(Wd, xd, y2, dtype=t, ws=ws)
    sync()
    assert torch.equal(y1, y2)  # the same order on every call
    acc = planes[0].clone()
    for s in range(1, planes.shape[0]):
        acc += planes[s]
    assert torch.equal(y1.cpu(), acc.to(dtype))  # pass 2: the planes in range order
    fmt = "f16" if dtype == torch.float16 else "bf16"
    yr, A = oracle.gemv_fp(bits(W), bits(x), fmt)
    tol.assert_close(y1.float().cpu().double().numpy(), yr, A, fmt, "split-K %dx%d M=%d" % (N, K, M))


@pytest.mark.parametrize("M", [1, 4])
def test_w8a8_split_k_is_bitwise_the_unsplit_call(M):
    need_gpu()
    N, K = 200, 4096
    W, s_w, xf = synth.w8_case(N, K, M, seed=5)
    q, sx = oracle.quant_act(bits(xf.half()))
    Wd, swd = W.to(DEV), s_w.to(DEV)
    qd, sxd = torch.from_numpy(q).to(DEV), torch.from_numpy(sx).to(DEV)
    ws = _ws(dg.LINEAR_W8A8, M, N, K)
    ya, yb = (torch.empty(M, N, dtype=torch.float16, device=DEV) for _ in range(2))
    aa, ab = (torch.empty(M, N, dtype=torch.int32, device=DEV) for _ in range(2))
    dg.gemv_w8a8(Wd, swd, qd, sxd, y=ya, acc_out=aa, ws=ws)
    dg.gemv_w8a8(Wd, swd, qd, sxd, y=yb, acc_out=ab)
    sync()
    planes = ws.view(torch.int32)[: 8 * M * N].view(8, M, N).cpu()
    assert torch.count_nonzero(planes[1]) > 0  # the split path ran
    assert torch.equal(aa, ab) and torch.equal(ya, yb)
    acc_ref = W.numpy().astype(np.int64) @ q.astype(np.int64).T
    assert np.array_equal(aa.cpu().numpy(), acc_ref.T)


@pytest.mark.parametrize("act", ["a16", "a8"])
def test_w4_split_k(act):
    need_gpu()
    N, K, grp = 128, 4096, 32
    Wq, sc, x = synth.w4_case(N, K, 1, seed=9, group=grp)
    Wd, scd = Wq.to(DEV), sc.to(DEV)
    kind = dg.LINEAR_W4A16 if act == "a16" else dg.LINEAR_W4A8
    ws = _ws(kind, 1, N, K, group_size=grp)
    y1 = torch.empty(1, N, dtype=torch.float16, device=DEV)
    y2 = torch.empty_like(y1)
    if act == "a16":
        xd = x.half().to(DEV)
        for y in (y1, y2):
            dg.gemv_w4(Wd, scd, y, x_f16=xd, group_size=grp, ws=ws)
        yr, A = oracle.gemv_w4a16(Wq.numpy(), bits(sc), bits(x.half()), group=grp)
    else:
        q, s = oracle.quant_act(bits(x.half()))
        qd, sd = torch.from_numpy(q).to(DEV), torch.from_numpy(s).to(DEV)
        for y in (y1, y2):
            dg.gemv_w4(Wd, scd, y, x_i8=qd, x_scale=sd, group_size=grp, ws=ws)
        yr, A, _ = oracle.gemv_w4a8(Wq.numpy(), bits(sc), q, s, group=grp)
    sync()
    _planes(ws, 1, N)
    assert torch.equal(y1, y2)
    tol.assert_close(y1.cpu().double().numpy(), yr, A, "f16", "split-K int4 " + act)


def test_large_calls_do_not_split():
    """Enough rows to fill the GPU: no split even with a large workspace."""
    need_gpu()
    N, K = 14336, 1024
    W, x = synth.fp_case(N, K, 1, seed=3)
    ws = torch.zeros(8 * N * 4, dtype=torch.uint8, device=DEV)
    y = torch.empty(1, N, dtype=torch.float16, device=DEV)
    dg.gemv_f16(W.to(DEV), x.to(DEV), y, ws=ws)
    sync()
    assert torch.count_nonzero(ws) == 0
