"""W8A8 (dg_gemv_w8a8) and per-token activation quantization
(dg_quantize_act_i8) against the oracle: int32 accumulators and int8 codes
bit-exact, fp16 outputs within tolerance."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, need_gpu, sync

pytestmark = pytest.mark.gpu


def quant_gpu(x):
    xd = x.to(DEV)
    M, K = x.shape
    xq = torch.empty(M, K, dtype=torch.int8, device=DEV)
    xs = torch.empty(M, dtype=torch.float32, device=DEV)
    dg.quantize_act_i8(xd, xq, xs)
    sync()
    return xq, xs


def run_w8(W, s_w, xq, xs):
    N, K = W.shape
    M = xq.shape[0]
    y = torch.empty(M, N, dtype=torch.float16, device=DEV)
    acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
    dg.gemv_w8a8(W.to(DEV), s_w.to(DEV), xq, xs, y, acc)
    sync()
    return y, acc


@pytest.mark.parametrize("M", [1, 4, 16])
def test_llama_mlp_shape(M):
    need_gpu()
    W, s_w, x = synth.w8a8_workload(M=M, seed=0)
    xq, xs = quant_gpu(x)
    q_ref, s_ref = oracle.quant_act(bits(x))
    assert np.array_equal(xq.cpu().numpy(), q_ref)
    assert np.array_equal(xs.cpu().numpy(), s_ref)
    y, acc = run_w8(W, s_w, xq, xs)
    acc_ref, y_ref, A = oracle.gemv_w8a8(W.numpy(), s_w.numpy(), q_ref, s_ref)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acc_ref)
    tol.assert_close(y.cpu().double().numpy(), y_ref, A, "f16", "w8a8 M=%d" % M)


@pytest.mark.parametrize("N,K,M", [(1, 16, 1), (5, 16, 3), (77, 48, 2), (1000, 4096, 8),
                                   (3, 14336, 16), (2049, 1536, 1), (129, 65536, 1)])
def test_shapes(N, K, M):
    need_gpu()
    W, s_w, x = synth.w8_case(N, K, M, seed=N * 7 + K)
    xq, xs = quant_gpu(x)
    y, acc = run_w8(W, s_w, xq, xs)
    q_ref, s_ref = oracle.quant_act(bits(x))
    acc_ref, y_ref, A = oracle.gemv_w8a8(W.numpy(), s_w.numpy(), q_ref, s_ref)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acc_ref)
    tol.assert_close(y.cpu().double().numpy(), y_ref, A, "f16", "w8a8 %dx%d M=%d" % (N, K, M))


def test_extreme_codes_exact():
    need_gpu()
    K = 4096
    W = torch.full((3, K), -127, dtype=torch.int8)
    W[1] = 127
    W[2, ::2] = 127
    xq = torch.full((2, K), 127, dtype=torch.int8, device=DEV)
    xq[1] = -127
    xs = torch.tensor([1e-3, 2e-3], dtype=torch.float32, device=DEV)
    s_w = torch.tensor([1e-3, 2e-3, 3e-3], dtype=torch.float32)
    y, acc = run_w8(W, s_w, xq, xs)
    a = acc.cpu().numpy()
    assert a[0].tolist() == [-127 * 127 * K, 127 * 127 * K, 0]
    assert a[1].tolist() == [127 * 127 * K, -127 * 127 * K, 0]


def test_quant_act_edge_tokens():
    need_gpu()
    K = 1024
    x = torch.zeros(4, K, dtype=torch.float16)
    x[1, 5] = -3.0
    x[2] = synth.normal((K,), 1.0, synth.generator(2))
    x[3, ::3] = 65504.0
    xq, xs = quant_gpu(x)
    q_ref, s_ref = oracle.quant_act(bits(x))
    assert np.array_equal(xq.cpu().numpy(), q_ref)
    assert np.array_equal(xs.cpu().numpy(), s_ref)
    assert float(xs[0]) == 1.0 and int(xq[0].abs().max()) == 0


@pytest.mark.parametrize("N,K,M", [(37, 64, 9), (100, 128, 16), (16, 4096, 12), (4111, 4096, 16),
                                   (257, 192, 8), (1, 4096, 16)])
def test_tensor_core_tile_for_8_to_16_tokens(N, K, M):
    """8..16 tokens with K a multiple of 64 run on the mma.sync s8 kernel:
    int32 accumulators still bit-exact."""
    need_gpu()
    W, s_w, x = synth.w8_case(N, K, M, seed=N + K + 100 * M)
    xq, xs = quant_gpu(x)
    y, acc = run_w8(W, s_w, xq, xs)
    q_ref, s_ref = oracle.quant_act(bits(x))
    acc_ref, y_ref, A = oracle.gemv_w8a8(W.numpy(), s_w.numpy(), q_ref, s_ref)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acc_ref)
    tol.assert_close(y.cpu().double().numpy(), y_ref, A, "f16", "w8a8 mma %dx%d M=%d" % (N, K, M))


def test_tensor_core_tile_extreme_codes_exact():
    need_gpu()
    K = 4096
    W = torch.full((32, K), 127, dtype=torch.int8)
    W[1::2] = -127
    xq = torch.full((16, K), -127, dtype=torch.int8, device=DEV)
    xq[::3] = 127
    xs = torch.full((16,), 1e-3, dtype=torch.float32, device=DEV)
    y, acc = run_w8(W, torch.full((32,), 1e-3), xq, xs)
    ref = xq.cpu().long() @ W.long().T
    assert torch.equal(acc.cpu().long(), ref)
