"""fp16 / bf16 weights for 8..16 tokens on the tensor cores: the tcgen05 + TMA
tile (stream-K over all SMs, last-arriver fixup of the tiles cut between
CTAs) and, where that tile cannot be set up (a stream seen for the first time
inside graph capture), the mma.sync tile.  Checked against the oracle's bound
for ragged rows, ragged K (TMA zero fill), every token count, fused segments
and the full 14336x4096 / 4096x14336 shapes on sampled rows; repeated calls
bitwise identical; two streams at once equal to one stream."""
import numpy as np
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


def _run(W, x, dtype, stream=None, y=None):
    t = dg.F16 if dtype == torch.float16 else dg.BF16
    if y is None:
        y = torch.empty(x.shape[0], W.shape[0], dtype=dtype, device=DEV)
    dg.gemv_f16(W, x, y, dtype=t, stream=stream)
    return y


def _check(y, W, x, dtype, what):
    yr, A = oracle.gemv_fp(bits(W), bits(x), _fmt(dtype))
    tol.assert_close(y.float().cpu().double().numpy(), yr, A, _fmt(dtype), what)


@pytest.mark.parametrize("N,K,M", [(1000, 1536, 16), (4097, 4096, 8), (17, 2048, 9),
                                   (16, 32, 16), (1, 1024, 12), (333, 6144, 16),
                                   (1000, 1032, 16), (300, 8, 8), (129, 4104, 11),
                                   (2000, 520, 13), (5, 65600, 10)])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_fp_mma_against_the_oracle(N, K, M, dtype):
    need_gpu()
    W, x = synth.fp_case(N, K, M, seed=N + K + M, dtype=dtype)
    Wd, xd = W.to(DEV), x.to(DEV)
    y = _run(Wd, xd, dtype)
    sync()
    assert torch.equal(y, _run(Wd, xd, dtype))  # the same order on every call
    _check(y, W, x, dtype, "mma %dx%d M=%d" % (N, K, M))


@pytest.mark.parametrize("M", [8, 9, 12, 15, 16])
def test_every_token_count_and_untouched_padding(M):
    """Tokens past M are zero-filled by TMA and never stored: y has M rows,
    and memory right after y keeps its contents."""
    need_gpu()
    N, K = 777, 2048
    W, x = synth.fp_case(N, K, M, seed=100 + M)
    buf = torch.full((M + 1, N), 7.0, dtype=torch.float16, device=DEV)
    y = buf[:M]
    _run(W.to(DEV), x.to(DEV), torch.float16, y=y)
    sync()
    assert torch.all(buf[M] == 7.0)
    _check(y, W, x, torch.float16, "M=%d" % M)


@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_full_size_sampled_rows(N, K):
    """The verify-block shapes at full size (tiles cut between CTAs): every
    output of sampled rows, including the first and last row of every
    128-row tile around the stream-K cut points, against the oracle."""
    need_gpu()
    M = 16
    W, x = synth.fp_case(N, K, M, seed=N // 7 + K)
    y = _run(W.to(DEV), x.to(DEV), torch.float16)
    sync()
    rows = sorted(set(list(range(0, N, 997)) + [t * 128 + o for t in range(0, N // 128, 5)
                                                  for o in (0, 127)] + [N - 1]))
    got = y[:, rows].float().cpu().double().numpy()
    yr, A = oracle.gemv_fp(bits(W[rows]), bits(x), "f16")
    tol.assert_close(got, yr, A, "f16", "full %dx%d sampled rows" % (N, K))


def test_two_streams_at_once_equal_one_stream():
    """Each stream has its own fixup scratch: launches interleaved on two
    streams give bitwise what each gives alone."""
    need_gpu()
    N, K, M = 6144, 4096, 16
    W1, x1 = synth.fp_case(N, K, M, seed=1)
    W2, x2 = synth.fp_case(N, K, M, seed=2)
    W1d, x1d, W2d, x2d = W1.to(DEV), x1.to(DEV), W2.to(DEV), x2.to(DEV)
    ref1 = _run(W1d, x1d, torch.float16)
    ref2 = _run(W2d, x2d, torch.float16)
    sync()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(4):
        outs.append((_run(W1d, x1d, torch.float16, stream=s1), _run(W2d, x2d, torch.float16, stream=s2)))
    sync()
    for a, b in outs:
        assert torch.equal(a, ref1) and torch.equal(b, ref2)


def test_graph_capture_on_a_new_stream_and_replay():
    """A stream first seen inside graph capture cannot get fixup scratch: the
    call falls back to the mma.sync tile, within the same bound; replays are
    bitwise identical."""
    need_gpu()
    N, K, M = 3000, 4096, 16
    W, x = synth.fp_case(N, K, M, seed=5)
    Wd, xd = W.to(DEV), x.to(DEV)
    y = torch.empty(M, N, dtype=torch.float16, device=DEV)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _run(Wd, xd, torch.float16, stream=s, y=y)
    g.replay()
    sync()
    first = y.clone()
    y.zero_()
    g.replay()
    sync()
    assert torch.equal(y, first)
    _check(y, W, x, torch.float16, "captured")


def test_fused_segments_through_a_decode_step():
    """q|k|v as one launch of three matrices (tiles never straddle two) at
    16 tokens, through the per-group path of dg_decode_step_weights."""
    need_gpu()
    K, M = 2048, 16
    Ns = (2048, 256, 256)
    g = synth.generator(77)
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
    for W, y, n in zip(Ws, ys, Ns):
        _check(y, W, x, torch.float16, "segment N=%d" % n)


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
    sync()
    assert torch.equal(y.cpu(), x[:, cols])
