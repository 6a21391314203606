"""W4A16 at one token: row-group and chunk-batch edges and group sizes against
the oracle, row slices bitwise equal to the whole matrix (a row's place in its
four-row slot must not change its result), decode-step row slices that
straddle fused segments bitwise equal to the per-op calls, a ragged int4
lm_head with a tie across row groups."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, need_gpu, sync

pytestmark = pytest.mark.gpu

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


# one row, a full and a ragged row group; one to fourteen chunks per lane
# (batches of two chunks, the last one partial); groups of 64, 128 and 256
# (two to eight chunks per scale); a few thousand rows; and the general slot
# loop: a 96-code group (no power of two), rows of 16384 codes (two warps per
# row) and a 2048-code group (more than 32 chunks per scale)
@pytest.mark.parametrize("N,K,group", [(1, 256, 32), (16, 256, 32), (17, 256, 32),
                                       (7, 768, 32), (250, 1280, 32), (300, 1024, 64),
                                       (300, 1024, 128), (129, 2304, 256), (4097, 512, 32),
                                       (6, 288, 32), (5, 14336, 32), (33, 9216, 128),
                                       (40, 288, 96), (20, 16384, 32), (9, 4096, 2048)])
def test_tile_edges_against_the_oracle(N, K, group):
    need_gpu()
    Wq, sc, x = _case(N, K, group, seed=N + K + group)
    y = _gemv(Wq.to(DEV), sc.to(DEV), x.to(DEV), group)
    yr, A = oracle.gemv_w4a16(Wq.numpy(), bits(sc), bits(x), group=group)
    tol.assert_close(y.cpu().double().numpy(), yr, A, "f16", "w4a16 %dx%d g%d" % (N, K, group))


def test_row_slices_equal_the_whole_matrix_bitwise():
    """A row's place in its row group changes with the slice (row 501 sits at
    position 1 of its four-row slot in the whole matrix, 0 in the slice from
    501): its result must not."""
    need_gpu()
    N, K = 1000, 1024
    Wq, sc, x = _case(N, K, 32, seed=5)
    Wd, sd, xd = Wq.to(DEV), sc.to(DEV), x.to(DEV)
    full = _gemv(Wd, sd, xd)
    for r0, r1 in ((3, 21), (501, 517), (993, 1000), (16, 48), (0, 1), (2, 3)):
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
    """1000 rows; rows 5 and 17 (different row groups and warps) hold the same
    winning codes and scales: equal logits, the lower index wins; the logits
    match the oracle."""
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
