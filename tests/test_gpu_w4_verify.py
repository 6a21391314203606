"""Groupwise int4 for 8..16 tokens (draft / verify blocks) on the tensor
cores (the tcgen05 tile; groups of 512, which it does not take, on the
mma.sync tile): W4A16 and W4A8 against the oracle at M = 8, 9, 12 and 16,
ragged N, groups of 32, 64, 128 and 512, every code value including -8; row
slices within the bound of the whole matrix's rows and repeated calls
bitwise identical; 8 tokens of K = 14336 rows; 16 such tokens refused."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, host, need_gpu, sync

pytestmark = pytest.mark.gpu


def _case(N, K, M, group, seed):
    g = synth.generator(seed)
    codes = torch.randint(-8, 8, (N, K), generator=g, dtype=torch.int16)
    codes[0, :16] = -8                               # the code no symmetric draw gives
    codes[-1, -16:] = 7
    nib = codes & 0xF
    Wq = (nib[:, 0::2] | (nib[:, 1::2] << 4)).to(torch.uint8)
    sc = synth.uniform((N, K // group), 1e-3, 1e-2, g, torch.float16)
    x = synth.normal((M, K), 1.0, g)
    return Wq, sc, x


def _run(Wq, sc, x, act, group):
    M, K = x.shape
    y = torch.empty(M, Wq.shape[0], dtype=torch.float16, device=DEV)
    xd = x.to(DEV)
    if act == "a16":
        dg.gemv_w4(Wq.to(DEV), sc.to(DEV), y, x_f16=xd, group_size=group)
    else:
        xq = torch.empty(M, K, dtype=torch.int8, device=DEV)
        xs = torch.empty(M, dtype=torch.float32, device=DEV)
        dg.quantize_act_i8(xd, xq, xs)
        dg.gemv_w4(Wq.to(DEV), sc.to(DEV), y, x_i8=xq, x_scale=xs, group_size=group)
    sync()
    return y


def _ref(Wq, sc, x, act, group):
    if act == "a16":
        return oracle.gemv_w4a16(Wq.numpy(), bits(sc), bits(x), group)
    q, s = oracle.quant_act(bits(x))
    y, A, _ = oracle.gemv_w4a8(Wq.numpy(), bits(sc), q, s, group)
    return y, A


@pytest.mark.parametrize("act", ["a16", "a8"])
@pytest.mark.parametrize("N,K,M,group", [(17, 1024, 8, 32), (1000, 4096, 9, 32), (4095, 4096, 12, 128),
                                         (14336 // 4, 4096, 16, 32), (300, 6144, 16, 64),
                                         (33, 512, 16, 512)])
def test_tensor_core_tile_against_the_oracle(act, N, K, M, group):
    need_gpu()
    Wq, sc, x = _case(N, K, M, group, seed=N + K + M + group)
    y = _run(Wq, sc, x, act, group)
    yr, A = _ref(Wq, sc, x, act, group)
    tol.assert_close(host(y).astype(np.float64), yr, A, "f16", "w4 %s tile M=%d" % (act, M))


@pytest.mark.parametrize("act", ["a16", "a8"])
def test_row_slices_and_repeated_calls(act):
    """The stream-K split follows the launch's rows, so a slice is summed in
    another order than the whole matrix (both within the bound); the same
    call twice is bitwise the same."""
    need_gpu()
    N, K, M = 1000, 2048, 16
    Wq, sc, x = _case(N, K, M, 32, seed=77)
    full = _run(Wq, sc, x, act, 32)
    assert torch.equal(full, _run(Wq, sc, x, act, 32))
    yr, A = _ref(Wq, sc, x, act, 32)
    for r0, r1 in ((3, 21), (501, 517), (993, 1000), (16, 48)):
        part = _run(Wq[r0:r1].contiguous(), sc[r0:r1].contiguous(), x, act, 32)
        tol.assert_close(host(part).astype(np.float64), yr[:, r0:r1], A[:, r0:r1], "f16",
                         "slice %d:%d" % (r0, r1))


@pytest.mark.parametrize("act", ["a16", "a8"])
def test_eight_tokens_of_long_rows(act):
    """8 tokens of 14336-wide rows (the shapes' down projection)."""
    need_gpu()
    N, K, M = 257, 14336, 8
    Wq, sc, x = _case(N, K, M, 32, seed=78)
    y = _run(Wq, sc, x, act, 32)
    yr, A = _ref(Wq, sc, x, act, 32)
    tol.assert_close(host(y).astype(np.float64), yr, A, "f16", "w4 %s long rows" % act)


def test_sixteen_tokens_of_rows_too_long_for_any_tile_are_refused():
    """16 tokens of 14336 fp16 activations need more than a CTA's shared
    memory on the tiles a launch may fall back to: DG_ERR_UNSUPPORTED, as
    documented, nothing launched."""
    need_gpu()
    N, K, M = 64, 14336, 16
    Wq, sc, x = _case(N, K, M, 32, seed=79)
    y = torch.zeros(M, N, dtype=torch.float16, device=DEV)
    with pytest.raises(dg.DGError) as e:
        dg.gemv_w4(Wq.to(DEV), sc.to(DEV), y, x_f16=x.to(DEV))
    assert e.value.status == 2
    sync()
    assert not y.any()
