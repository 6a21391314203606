"""Load-time weight packers (dg_quantize_weights_i8 / _w4) against the
oracle's quantizers bit for bit (codes, packed bytes and scales), including
all-zero rows and groups, a group whose scale underflows to fp16 subnormals,
and values on rounding ties; then the packed weights through the GEMV against
the oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, host, need_gpu, sync

pytestmark = pytest.mark.gpu


def _weights(N, K, seed):
    W = synth.normal((N, K), synth.W_STD, synth.generator(seed))
    W[0] = 0                                  # all-zero row / groups
    W[1, :64] = 1e-7                          # tiny: the int4 scale rounds to a subnormal
    W[2, :32] = torch.tensor([7 * 0.5 * (2 * i + 1) / 7 for i in range(16)] * 2)  # ties at the scale
    W[3, ::5] = 0.0
    return W


@pytest.mark.parametrize("N,K", [(37, 4096), (1000, 1536)])
def test_int8_packer_matches_the_oracle_bitwise(N, K):
    need_gpu()
    W = _weights(N, K, seed=N)
    q = torch.empty(N, K, dtype=torch.int8, device=DEV)
    s = torch.empty(N, dtype=torch.float32, device=DEV)
    dg.quantize_weights_i8(W.to(DEV), q, s)
    sync()
    qr, sr = oracle.quant_w8(W.float().numpy())
    assert np.array_equal(q.cpu().numpy(), qr)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), sr.view(np.uint32))


@pytest.mark.parametrize("N,K,group", [(37, 4096, 32), (257, 1536, 128), (8, 512, 512)])
def test_int4_packer_matches_the_oracle_bitwise(N, K, group):
    need_gpu()
    W = _weights(N, K, seed=N + group)
    Wq = torch.empty(N, K // 2, dtype=torch.uint8, device=DEV)
    sc = torch.empty(N, K // group, dtype=torch.float16, device=DEV)
    dg.quantize_weights_w4(W.to(DEV), Wq, sc, group_size=group)
    sync()
    codes, s16 = oracle.quant_w4(W.float().numpy(), group)
    assert np.array_equal(Wq.cpu().numpy(), oracle.pack_w4(codes))
    assert np.array_equal(host(sc).view(np.uint16), s16.view(np.uint16))
    # and the packed result streams through the W4A16 GEMV
    x = synth.normal((1, K), 1.0, synth.generator(N + 1))
    y = torch.empty(1, N, dtype=torch.float16, device=DEV)
    dg.gemv_w4(Wq, sc, y, x_f16=x.to(DEV), group_size=group)
    sync()
    yr, A = oracle.gemv_w4a16(Wq.cpu().numpy(), bits(sc.cpu()), bits(x), group)
    tol.assert_close(host(y).astype(np.float64), yr, A, "f16", "packed w4a16")
