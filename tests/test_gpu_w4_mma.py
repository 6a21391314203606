"""W4A16 at one token: tile and segment edges and group sizes against the
oracle, row slices bitwise equal to the whole matrix, decode-step row slices
that straddle fused segments bitwise equal to the per-op calls, a ragged int4
lm_head with a tie across tiles.  The parent runs them on the default
CUDA-core path; a child process runs them, with the int4 GEMV and step tests,
on the tensor-core tile (mma.sync m16n8k16: 16 weight rows per warp tile,
each column of the B operand one 32-code chunk, the chunk's group scale
applied in fp32), which DG_TUNE=W4MMA=1 selects."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, need_gpu, sync

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TILE = "W4MMA=1" in os.environ.get("DG_TUNE", "")
parent_only = pytest.mark.skipif(TILE, reason="run by the parent pytest")


def _case(N, K, group, seed):
    g = synth.generator(seed)
    Wq = synth.int4_packed(N, K, g)
    sc = synth.uniform((N, K // group), 1e-3, 1e-2, g, torch.float16)
    x = synth.normal((1, K), 1.0, g)
    return Wq, sc, x


def _gemv(Wq, sc, x, group=32):
    y = torch.empty(1, Wq.shape[0], dtype=torch.float16, device=DEV)
    dg.gemv_w4(Wq, sc, y, x_f16=x, group_size=group)
    sync()
    return y


# one row, a full tile, a ragged tile; 1, 3 (odd: the last batch of two
# segments half full) and 5 segments; groups of 64, 128 and 256 (two to eight
# chunks per scale); a few thousand rows
@pytest.mark.parametrize("N,K,group", [(1, 256, 32), (16, 256, 32), (17, 256, 32),
                                       (7, 768, 32), (250, 1280, 32), (300, 1024, 64),
                                       (300, 1024, 128), (129, 2304, 256), (4097, 512, 32)])
def test_tile_edges_against_the_oracle(N, K, group):
    need_gpu()
    Wq, sc, x = _case(N, K, group, seed=N + K + group)
    y = _gemv(Wq.to(DEV), sc.to(DEV), x.to(DEV), group)
    yr, A = oracle.gemv_w4a16(Wq.numpy(), bits(sc), bits(x), group=group)
    tol.assert_close(y.cpu().double().numpy(), yr, A, "f16", "w4a16 %dx%d g%d" % (N, K, group))


def test_row_slices_equal_the_whole_matrix_bitwise():
    """A row's place in its row group or tile changes with the slice (row 500
    sits at position 4 of its 16-row tile in the whole matrix, 0 in the slice
    from 500): its result must not."""
    need_gpu()
    N, K = 1000, 1024
    Wq, sc, x = _case(N, K, 32, seed=5)
    Wd, sd, xd = Wq.to(DEV), sc.to(DEV), x.to(DEV)
    full = _gemv(Wd, sd, xd)
    for r0, r1 in ((3, 21), (500, 517), (993, 1000), (16, 48), (0, 1)):
        part = _gemv(Wd[r0:r1].contiguous(), sd[r0:r1].contiguous(), xd)
        assert torch.equal(part, full[:, r0:r1]), (r0, r1)


def test_step_tiles_straddling_fused_segments_equal_the_per_op_calls():
    """Three ops on one input (one fused phase of 7600 rows, about 50 per CTA):
    the step's row groups or tiles start at each CTA's slice and cross the
    segment boundaries; every row equals the per-op call bitwise and the
    oracle."""
    need_gpu()
    g = synth.generator(31)
    K = 1024
    x = synth.normal((1, K), 1.0, g).to(DEV)
    ops, keep, cases = [], [x], []
    for N in (3000, 1700, 2900):
        Wq = synth.int4_packed(N, K, g).to(DEV)
        sc = synth.uniform((N, K // 32), 1e-3, 1e-2, g, torch.float16).to(DEV)
        y = torch.empty(1, N, dtype=torch.float16, device=DEV)
        keep += [Wq, sc, y]
        ops.append(dg.linear(dg.LINEAR_W4A16, Wq, 1, N, K, w_scale=sc, x=x, y=y))
        cases.append((Wq, sc, y))
    plan = dg.StepPlan(ops, keep)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=DEV)
    dg.decode_step_weights(plan, ws)
    sync()
    dg.check_device_status()
    for Wq, sc, y in cases:
        ref = _gemv(Wq, sc, x)
        assert torch.equal(y, ref), tuple(Wq.shape)
        yr, A = oracle.gemv_w4a16(Wq.cpu().numpy(), bits(sc.cpu()), bits(x.cpu()))
        tol.assert_close(y.cpu().double().numpy(), yr, A, "f16", "fused %s" % (tuple(Wq.shape),))


def test_ragged_int4_head_and_a_tie_across_tiles():
    """1000 rows (the last tile half full); rows 5 and 17 (tiles 0 and 1)
    hold the same winning codes and scales: equal logits, the lower index
    wins; the logits match the oracle."""
    need_gpu()
    N, K = 1000, 512
    Wq, sc, x = _case(N, K, 32, seed=41)
    plant = torch.where(x[0] > 0, 7, -7).to(torch.int16) & 0xF
    row = (plant[0::2] | (plant[1::2] << 4)).to(torch.uint8)
    for r in (5, 17):
        Wq[r] = row
        sc[r] = 0.01
    Wd, sd, xd = Wq.to(DEV), sc.to(DEV), x.to(DEV)
    logits = torch.empty(N, dtype=torch.float32, device=DEV)
    token = torch.empty(1, dtype=torch.int32, device=DEV)
    head = dg.linear(dg.LINEAR_W4A16, Wd, 1, N, K, w_scale=sd, x=xd, logits=logits, token=token)
    ws = torch.empty(dg.workspace_bytes([head]), dtype=torch.uint8, device=DEV)
    dg.lm_head_argmax(head, ws)
    sync()
    lg = logits.cpu()
    assert torch.equal(lg[5], lg[17])
    assert int(token.item()) == 5
    lr, A = oracle.gemv_w4a16(Wq.numpy(), bits(sc), bits(x))
    tol.assert_close(lg.double().numpy(), lr[0], A[0], "f32", "ragged int4 head")
    assert int(np.argmax(lg.numpy())) == 5


@parent_only
def test_tensor_core_w4a16_tile_in_a_child_process():
    need_gpu()
    env = dict(os.environ, DG_TUNE="W4MMA=1")
    files = [os.path.join(ROOT, "tests", f) for f in ("test_gpu_w4.py", "test_gpu_w4_mma.py")]
    step = os.path.join(ROOT, "tests", "test_gpu_decode_step.py")
    split = os.path.join(ROOT, "tests", "test_gpu_split_k.py::test_w4_split_k")
    r = subprocess.run([sys.executable, "-m", "pytest", *files, split,
                        step + "::test_persistent_step_equals_per_op_calls_bitwise_int4",
                        step + "::test_int4_step_mixing_laid_out_and_staged_activations_matches_"
                        "sequential_calls", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    assert " passed" in r.stdout and "failed" not in r.stdout
