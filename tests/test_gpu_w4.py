"""Groupwise int4 weights (dg_gemv_w4: W4A16 and W4A8) and the int4 lm_head
against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, need_gpu, sync

pytestmark = pytest.mark.gpu


def run(Wq, sc, x, act, group=32):
    N = Wq.shape[0]
    M = x.shape[0]
    y = torch.empty(M, N, dtype=torch.float16, device=DEV)
    xd = x.to(DEV)
    if act == "a16":
        dg.gemv_w4(Wq.to(DEV), sc.to(DEV), y, x_f16=xd, group_size=group)
        sync()
        yr, A = oracle.gemv_w4a16(Wq.numpy(), bits(sc), bits(x), group=group)
    else:
        xq = torch.empty(x.shape, dtype=torch.int8, device=DEV)
        xs = torch.empty(M, dtype=torch.float32, device=DEV)
        dg.quantize_act_i8(xd, xq, xs)
        dg.gemv_w4(Wq.to(DEV), sc.to(DEV), y, x_i8=xq, x_scale=xs, group_size=group)
        sync()
        q_ref, s_ref = oracle.quant_act(bits(x))
        assert np.array_equal(xq.cpu().numpy(), q_ref)
        yr, A, _ = oracle.gemv_w4a8(Wq.numpy(), bits(sc), q_ref, s_ref, group=group)
    return y, yr, A


@pytest.mark.parametrize("act", ["a16", "a8"])
@pytest.mark.parametrize("N,K,M", [(1, 32, 1), (9, 64, 1), (4096, 4096, 1), (1024, 4096, 1),
                                   (4096, 14336, 1), (333, 4096, 3), (64, 1024, 16),
                                   (2000, 96, 2), (17, 4096, 8)])
def test_shapes(act, N, K, M):
    need_gpu()
    Wq, sc, x = synth.w4_case(N, K, M, seed=N + 3 * K + M)
    y, yr, A = run(Wq, sc, x, act)
    tol.assert_close(y.cpu().double().numpy(), yr, A, "f16", "w4%s %dx%d M=%d" % (act, N, K, M))


@pytest.mark.parametrize("act", ["a16", "a8"])
@pytest.mark.parametrize("group", [64, 128])
def test_larger_groups(act, group):
    need_gpu()
    g = synth.generator(11)
    N, K = 300, 1024
    Wq = synth.int4_packed(N, K, g)
    sc = synth.uniform((N, K // group), 1e-3, 1e-2, g, torch.float16)
    x = synth.normal((2, K), 1.0, g)
    y, yr, A = run(Wq, sc, x, act, group)
    tol.assert_close(y.cpu().double().numpy(), yr, A, "f16", "group %d" % group)


@pytest.mark.parametrize("act", ["a16", "a8"])
def test_code_minus_eight_and_every_nibble(act):
    need_gpu()
    N, K = 256, 512
    # row n holds byte value n in every position: all 256 (lo, hi) code pairs,
    # including -8 in both nibbles
    Wq = torch.arange(256, dtype=torch.int32).to(torch.uint8)[:, None].repeat(1, K // 2)
    sc = synth.uniform((N, K // 32), 1e-3, 1e-2, synth.generator(12), torch.float16)
    x = synth.normal((1, K), 1.0, synth.generator(13))
    y, yr, A = run(Wq, sc, x, act)
    tol.assert_close(y.cpu().double().numpy(), yr, A, "f16", "all nibbles")


def test_scaled_one_hot_is_exact():
    need_gpu()
    N, K = 40, 256
    codes = np.zeros((N, K), np.int64)
    cols = np.arange(N) * 5 % K
    vals = np.array([-8, -7, -1, 1, 7] * 8)
    codes[np.arange(N), cols] = vals
    nib = codes & 0xF
    Wq = torch.from_numpy((nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8))
    sc = torch.full((N, K // 32), 0.25, dtype=torch.float16)
    x = synth.normal((1, K), 1.0, synth.generator(14))
    y = torch.empty(1, N, dtype=torch.float16, device=DEV)
    dg.gemv_w4(Wq.to(DEV), sc.to(DEV), y, x_f16=x.to(DEV))
    sync()
    expect = (0.25 * vals * x[0, cols].double().numpy()).astype(np.float16)
    assert np.array_equal(y.cpu().numpy()[0], expect)


@pytest.mark.parametrize("act", ["a16", "a8"])
def test_int4_lm_head_argmax(act):
    need_gpu()
    N, K = 128256, 4096
    Wq, sc, x = synth.w4_case(N, K, 1, seed=21)
    Wd, sd, xd = Wq.to(DEV), sc.to(DEV), x.to(DEV)
    r = 99999
    plant = torch.where(xd[0] > 0, 7, -7).to(torch.int16).cpu() & 0xF
    Wd[r] = (plant[0::2] | (plant[1::2] << 4)).to(torch.uint8).to(DEV)
    Wq2 = Wd.cpu()
    logits = torch.empty(N, dtype=torch.float32, device=DEV)
    token = torch.empty(1, dtype=torch.int32, device=DEV)
    if act == "a16":
        head = dg.linear(dg.LINEAR_W4A16, Wd, 1, N, K, w_scale=sd, x=xd, logits=logits,
                         token=token)
    else:
        xq = torch.empty(1, K, dtype=torch.int8, device=DEV)
        xs = torch.empty(1, dtype=torch.float32, device=DEV)
        dg.quantize_act_i8(xd, xq, xs)
        head = dg.linear(dg.LINEAR_W4A8, Wd, 1, N, K, w_scale=sd, x_i8=xq, x_scale=xs,
                         logits=logits, token=token)
    ws = torch.empty(dg.workspace_bytes([head]), dtype=torch.uint8, device=DEV)
    dg.lm_head_argmax(head, ws)
    sync()
    if act == "a16":
        lr, A = oracle.gemv_w4a16(Wq2.numpy(), bits(sc), bits(x))
    else:
        q_ref, s_ref = oracle.quant_act(bits(x))
        lr, A, _ = oracle.gemv_w4a8(Wq2.numpy(), bits(sc), q_ref, s_ref)
    tol.assert_close(logits.cpu().double().numpy(), lr[0], A[0], "f32", "int4 head")
    assert int(token.item()) == r
    assert int(token.item()) == int(np.argmax(logits.cpu().numpy()))
