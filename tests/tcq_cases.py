"""Cases run by test_gpu_tcq.py in a child process whose DG_TUNE sends every
int8 / int4 launch of 8+ tokens to the tcgen05 tile (named without the test_
prefix so the main session does not collect it with its own settings).

int8 and int4 weights for 8..16 tokens on the tcgen05 tile (codes widened
to fp16 in tensor memory, one accumulator per int4 group / per 1024-k run of
W8A8, stream-K over all SMs): against the oracle at the run and group edges,
every group size the tile takes, 128-row tile edges cut between CTAs, the
full 14336x4096 / 4096x14336 shapes on sampled rows, extreme codes; W8A8
int32 sums bit-exact whatever the split (so a row slice equals the whole
matrix bitwise); fused q|k|v segments; two streams at once; a stream first
used inside graph capture (mma.sync fallback)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, host, need_gpu, sync

pytestmark = pytest.mark.gpu


def _quant(xd):
    M, K = xd.shape
    xq = torch.empty(M, K, dtype=torch.int8, device=DEV)
    xs = torch.empty(M, dtype=torch.float32, device=DEV)
    dg.quantize_act_i8(xd, xq, xs)
    return xq, xs


def _w8(Wd, swd, xq, xs, stream=None):
    M, N = xq.shape[0], Wd.shape[0]
    y = torch.empty(M, N, dtype=torch.float16, device=DEV)
    acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
    dg.gemv_w8a8(Wd, swd, xq, xs, y, acc, stream=stream)
    return y, acc


@pytest.mark.parametrize("N,K,M", [(300, 128, 16), (1000, 1024, 8), (129, 1152, 9), (777, 2176, 16),
                                   (4111, 4096, 12), (64, 9216, 16), (3, 14336, 8)])
def test_w8a8_exact_sums(N, K, M):
    """Runs of 1024 k, pieces cut at any 128-k box: int32 sums bit-exact."""
    need_gpu()
    W, s_w, x = synth.w8_case(N, K, M, seed=N + K + M)
    xq, xs = _quant(x.to(DEV))
    y, acc = _w8(W.to(DEV), s_w.to(DEV), xq, xs)
    sync()
    q, s = oracle.quant_act(bits(x))
    acc_ref, y_ref, A = oracle.gemv_w8a8(W.numpy(), s_w.numpy(), q, s)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acc_ref)
    tol.assert_close(y.cpu().double().numpy(), y_ref, A, "f16", "w8a8 tc %dx%d M=%d" % (N, K, M))


def test_w8a8_extreme_codes_and_row_slices_exact():
    """All codes -128 against x codes of +-127 / -128: the largest run sums
    (2^24 in magnitude) stay exact; row slices give bitwise the same sums."""
    need_gpu()
    N, K, M = 600, 4096, 16
    W = torch.full((N, K), -128, dtype=torch.int8)
    W[1::2] = 127
    xq = torch.full((M, K), -128, dtype=torch.int8)
    xq[1::3] = 127
    s_w = torch.full((N,), 1e-3, dtype=torch.float32)
    xs = torch.full((M,), 1e-2, dtype=torch.float32)
    Wd, swd, xqd, xsd = W.to(DEV), s_w.to(DEV), xq.to(DEV), xs.to(DEV)
    y, acc = _w8(Wd, swd, xqd, xsd)
    sync()
    ref = xq.long() @ W.long().T
    assert torch.equal(acc.cpu().long(), ref)
    for r0, r1 in ((0, 128), (5, 300), (511, 600)):
        _, a2 = _w8(Wd[r0:r1].contiguous(), swd[r0:r1].contiguous(), xqd, xsd)
        sync()
        assert torch.equal(a2, acc[:, r0:r1])


def _w4(Wq, sc, x, act, group, stream=None):
    M, K = x.shape
    y = torch.empty(M, Wq.shape[0], dtype=torch.float16, device=DEV)
    xd = x.to(DEV)
    if act == "a16":
        dg.gemv_w4(Wq, sc, y, x_f16=xd, group_size=group, stream=stream)
    else:
        xq, xs = _quant(xd)
        dg.gemv_w4(Wq, sc, y, x_i8=xq, x_scale=xs, group_size=group, stream=stream)
    return y


def _w4_ref(Wq, sc, x, act, group):
    if act == "a16":
        return oracle.gemv_w4a16(Wq.numpy(), bits(sc), bits(x), group)
    q, s = oracle.quant_act(bits(x))
    y, A, _ = oracle.gemv_w4a8(Wq.numpy(), bits(sc), q, s, group)
    return y, A


@pytest.mark.parametrize("act", ["a16", "a8"])
@pytest.mark.parametrize("N,K,M,group", [(300, 256, 16, 32), (1000, 768, 8, 64), (129, 4096, 11, 128),
                                         (2000, 1280, 16, 256), (130, 6144, 13, 32),
                                         (5, 2048, 10, 16 * 2)])
def test_int4_groups(act, N, K, M, group):
    need_gpu()
    Wq, sc, x = synth.w4_case(N, K, M, seed=N + K + M + group, group=group)
    y = _w4(Wq.to(DEV), sc.to(DEV), x, act, group)
    sync()
    yr, A = _w4_ref(Wq, sc, x, act, group)
    tol.assert_close(host(y).astype(np.float64), yr, A, "f16", "int4 %s tc g%d" % (act, group))


@pytest.mark.parametrize("act", ["a16", "a8"])
@pytest.mark.parametrize("N,K,M", [(14336, 4096, 16), (4096, 14336, 8)])
def test_int4_full_size_sampled_rows(act, N, K, M):
    need_gpu()
    Wq, sc, x = synth.w4_case(N, K, M, seed=N + 3, group=32)
    y = _w4(Wq.to(DEV), sc.to(DEV), x, act, 32)
    sync()
    rows = sorted(set(list(range(0, N, 1013)) + [t * 128 + o for t in range(0, N // 128, 7)
                                                   for o in (0, 127)] + [N - 1]))
    yr, A = _w4_ref(Wq[rows].contiguous(), sc[rows].contiguous(), x, act, 32)
    tol.assert_close(host(y[:, rows]).astype(np.float64), yr, A, "f16", "int4 %s full" % act)


def test_w8a8_full_size_sampled_rows():
    need_gpu()
    N, K, M = 14336, 4096, 16
    W, s_w, x = synth.w8a8_workload(M=M, seed=5)
    xq, xs = _quant(x.to(DEV))
    y, acc = _w8(W.to(DEV), s_w.to(DEV), xq, xs)
    sync()
    rows = list(range(0, N, 211)) + [N - 1]
    q, s = oracle.quant_act(bits(x))
    acc_ref, y_ref, A = oracle.gemv_w8a8(W[rows].numpy(), s_w[rows].numpy(), q, s)
    assert np.array_equal(acc[:, rows].cpu().numpy().astype(np.int64), acc_ref)
    tol.assert_close(y[:, rows].cpu().double().numpy(), y_ref, A, "f16", "w8a8 full")


@pytest.mark.parametrize("kind", ["a16", "a8"])
def test_int4_fused_segments_through_a_decode_step(kind):
    """q|k|v as one launch of three int4 matrices at 16 tokens."""
    need_gpu()
    K, M, group = 2048, 16, 32
    Ns = (2048, 256, 384)
    cases = [synth.w4_case(n, K, M, seed=90 + i, group=group) for i, n in enumerate(Ns)]
    x = cases[0][2]
    xd = x.to(DEV)
    Wd = [c[0].to(DEV) for c in cases]
    Sd = [c[1].to(DEV) for c in cases]
    ys = [torch.empty(M, n, dtype=torch.float16, device=DEV) for n in Ns]
    keep = Wd + Sd + ys + [xd]
    if kind == "a16":
        ops = [dg.linear(dg.LINEAR_W4A16, W, M, n, K, w_scale=S, x=xd, y=y, group_size=group)
               for W, S, n, y in zip(Wd, Sd, Ns, ys)]
    else:
        xq, xs = _quant(xd)
        keep += [xq, xs]
        ops = [dg.linear(dg.LINEAR_W4A8, W, M, n, K, w_scale=S, x_i8=xq, x_scale=xs, y=y,
                         group_size=group) for W, S, n, y in zip(Wd, Sd, Ns, ys)]
    plan = dg.StepPlan(ops, keep)
    ws = torch.empty(max(plan.workspace_bytes(), 16), dtype=torch.uint8, device=DEV)
    dg.decode_step_weights(plan, ws)
    sync()
    for (Wq, sc, _), y, n in zip(cases, ys, Ns):
        yr, A = _w4_ref(Wq, sc, x, kind, group)
        tol.assert_close(host(y).astype(np.float64), yr, A, "f16", "segment N=%d" % n)


def test_two_streams_at_once_equal_one_stream():
    need_gpu()
    N, K, M = 6144, 4096, 16
    a = synth.w4_case(N, K, M, seed=1)
    b = synth.w4_case(N, K, M, seed=2)
    Wa, Sa, Wb, Sb = a[0].to(DEV), a[1].to(DEV), b[0].to(DEV), b[1].to(DEV)
    ref_a = _w4(Wa, Sa, a[2], "a16", 32)
    ref_b = _w4(Wb, Sb, b[2], "a16", 32)
    sync()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [(_w4(Wa, Sa, a[2], "a16", 32, stream=s1), _w4(Wb, Sb, b[2], "a16", 32, stream=s2))
            for _ in range(4)]
    sync()
    for ya, yb in outs:
        assert torch.equal(ya, ref_a) and torch.equal(yb, ref_b)


def test_graph_capture_on_a_new_stream():
    """No fixup scratch can be made inside capture: the mma.sync tile runs,
    within the same bound; replays are bitwise identical."""
    need_gpu()
    N, K, M = 3000, 4096, 16
    W, s_w, x = synth.w8_case(N, K, M, seed=9)
    Wd, swd = W.to(DEV), s_w.to(DEV)
    xq, xs = _quant(x.to(DEV))
    y = torch.empty(M, N, dtype=torch.float16, device=DEV)
    acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dg.gemv_w8a8(Wd, swd, xq, xs, y, acc, stream=s)
    g.replay()
    sync()
    first = acc.clone()
    acc.zero_()
    g.replay()
    sync()
    assert torch.equal(acc, first)
    q, sq = oracle.quant_act(bits(x))
    acc_ref, y_ref, A = oracle.gemv_w8a8(W.numpy(), s_w.numpy(), q, sq)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acc_ref)
    tol.assert_close(y.cpu().double().numpy(), y_ref, A, "f16", "captured w8a8")
