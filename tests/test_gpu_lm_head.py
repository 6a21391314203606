"""Wide lm_head with fused greedy argmax (C ABI dg_lm_head_argmax) against the
oracle, including the 16-slice split with a host reduce of the Orange Pi AIPro
post (paragraph on the ~248k-vocabulary lm_head)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, need_gpu, sync

pytestmark = pytest.mark.gpu

N_FULL, K_FULL = 248320, 2048


@pytest.fixture(scope="module")
def head_inputs():
    need_gpu()
    W, x = synth.lm_head_workload(seed=0)
    return W, x, W.to(DEV), x.to(DEV)


def run_head(Wd, xd, kind=dg.LINEAR_F16):
    N, K = Wd.shape
    logits = torch.empty(N, dtype=torch.float32, device=DEV)
    token = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    head = dg.linear(kind, Wd, 1, N, K, x=xd, logits=logits, token=token)
    ws = torch.empty(dg.workspace_bytes([head]), dtype=torch.uint8, device=DEV)
    dg.lm_head_argmax(head, ws)
    sync()
    return logits, int(token.item())


def first_argmax(v):
    return int(np.argmax(v))  # numpy returns the first index of the maximum


def test_full_size_logits_and_token(head_inputs):
    W, x, Wd, xd = head_inputs
    logits, tok = run_head(Wd, xd)
    lr, A, _ = oracle.lm_head(bits(W), bits(x))
    tol.assert_close(logits.cpu().numpy(), lr, A, "f32", "lm_head logits")
    ok, pinned = tol.argmax_check(tok, lr, A)
    assert ok, (tok, pinned)
    assert tok == first_argmax(logits.cpu().numpy())


def test_sixteen_slices_with_host_reduce_match_unsplit_bitwise(head_inputs):
    W, x, Wd, xd = head_inputs
    full, tok = run_head(Wd, xd)
    rows = N_FULL // 16
    best_v, best_i = None, -1
    for s in range(16):
        lg, t = run_head(Wd[s * rows:(s + 1) * rows], xd)
        assert torch.equal(lg, full[s * rows:(s + 1) * rows]), s
        v, gi = float(lg[t]), s * rows + t
        if best_i < 0 or v > best_v or (v == best_v and gi < best_i):
            best_v, best_i = v, gi
    assert best_i == tok


@pytest.mark.parametrize("where", [0, 1, 15519, 15520, 124160, 248318, 248319])
def test_planted_winner(head_inputs, where):
    W, x, Wd, xd = head_inputs
    W2 = Wd.clone()
    W2[where] = (0.05 * torch.sign(xd[0].float())).half()
    _, tok = run_head(W2, xd)
    assert tok == where


def test_planted_exact_tie_lowest_index_wins(head_inputs):
    W, x, Wd, xd = head_inputs
    W2 = Wd.clone()
    row = (0.05 * torch.sign(xd[0].float())).half()
    for r in (200000, 77777, 150001):
        W2[r] = row
    logits, tok = run_head(W2, xd)
    assert tok == 77777
    assert float(logits[77777]) == float(logits[200000]) == float(logits[150001])


def test_all_equal_logits_give_token_zero():
    need_gpu()
    Wd = torch.zeros(40000, 256, dtype=torch.float16, device=DEV)
    xd = torch.ones(1, 256, dtype=torch.float16, device=DEV)
    logits, tok = run_head(Wd, xd)
    assert tok == 0 and float(logits.abs().max()) == 0.0


@pytest.mark.parametrize("N,K", [(1, 8), (31, 64), (5000, 520), (70001, 1024)])
def test_small_and_ragged_heads(N, K):
    need_gpu()
    W, x = synth.fp_case(N, K, 1, seed=N)
    logits, tok = run_head(W.to(DEV), x.to(DEV))
    lr, A, _ = oracle.lm_head(bits(W), bits(x))
    tol.assert_close(logits.cpu().numpy(), lr, A, "f32", "head N=%d" % N)
    assert tol.argmax_check(tok, lr, A)[0]
    assert tok == first_argmax(logits.cpu().numpy())


def test_bf16_head():
    need_gpu()
    W, x = synth.fp_case(30000, 2048, 1, seed=9, dtype=torch.bfloat16)
    logits, tok = run_head(W.to(DEV), x.to(DEV), dg.LINEAR_BF16)
    lr, A, _ = oracle.lm_head(bits(W), bits(x), "bf16")
    tol.assert_close(logits.cpu().numpy(), lr, A, "f32", "bf16 head")
    assert tok == first_argmax(logits.cpu().numpy())
