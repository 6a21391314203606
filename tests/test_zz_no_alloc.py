"""The workspace-free lm_head entry point (dg_lm_head_argmax_noalloc).

Callers that cannot allocate device memory (a decode loop that must not
allocate once it runs, a plugin whose host runtime owns all device memory)
use this variant: its argmax partials live in a fixed array inside the library.
Three heads run back to back, largest grid first, so later calls start with an
earlier call's partials still in the array: the 248320-row fp16 head, the
128256x4096 int4 (W4A16) head and a small ragged fp16 head.  One call goes
through the C ABI directly (ctypes), the others through the package's wrapper.
Each result must equal dg_lm_head_argmax with a caller workspace bit for bit
(the same kernels in the same launch configuration), and logits and token are
checked against the oracle.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, need_gpu, sync

pytestmark = pytest.mark.gpu


def _head(case, logits, token):
    kind, Wd, Sd, xd = case
    N, K = Wd.shape[0], xd.shape[-1]
    return dg.linear(kind, Wd, 1, N, K, w_scale=Sd, x=xd, logits=logits, token=token)


def with_workspace(case):
    N = case[1].shape[0]
    logits = torch.empty(N, dtype=torch.float32, device=DEV)
    token = torch.empty(1, dtype=torch.int32, device=DEV)
    head = _head(case, logits, token)
    ws = torch.empty(dg.workspace_bytes([head]), dtype=torch.uint8, device=DEV)
    dg.lm_head_argmax(head, ws)
    sync()
    return logits, int(token.item())


def without_workspace(case, via_ctypes):
    N = case[1].shape[0]
    logits = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    token = torch.full((1,), -5, dtype=torch.int32, device=DEV)
    head = _head(case, logits, token)
    if via_ctypes:
        st = dg.load().dg_lm_head_argmax_noalloc(ctypes.byref(head),
                                                 torch.cuda.current_stream().cuda_stream)
        assert st == 0, dg.status_string(st)
    else:
        dg.lm_head_argmax_noalloc(head)
    sync()
    return logits, int(token.item())


def _cases():
    W1, x1 = synth.fp_case(248320, 2048, 1, seed=41)
    Wq, sc, x2 = synth.w4_case(128256, 4096, 1, seed=43)
    W3, x3 = synth.fp_case(30011, 1024, 1, seed=42)
    return [("f16", (dg.LINEAR_F16, W1.to(DEV), None, x1.to(DEV)), (W1, x1)),
            ("w4a16", (dg.LINEAR_W4A16, Wq.to(DEV), sc.to(DEV), x2.to(DEV)), (Wq, sc, x2)),
            ("f16", (dg.LINEAR_F16, W3.to(DEV), None, x3.to(DEV)), (W3, x3))]


def test_noalloc_matches_workspace_entry_point_and_oracle_back_to_back():
    need_gpu()
    for i, (fmt, case, host) in enumerate(_cases()):
        ref_logits, ref_tok = with_workspace(case)
        logits, tok = without_workspace(case, via_ctypes=(i != 1))
        N = case[1].shape[0]
        what = "noalloc %s N=%d" % (fmt, N)
        # the same kernels, grid and summation order: identical bits
        assert torch.equal(logits.view(torch.int32), ref_logits.view(torch.int32)), what
        assert tok == ref_tok, what
        # and against the oracle
        if fmt == "f16":
            lr, A, _ = oracle.lm_head(bits(host[0]), bits(host[1]))
        else:
            y, A2 = oracle.gemv_w4a16(host[0].numpy(), bits(host[1]), bits(host[2]))
            lr, A = y[0], A2[0]
        tol.assert_close(logits.cpu().double().numpy(), lr, A, "f32", what + " logits")
        ok, info = tol.argmax_check(tok, lr, A)
        assert ok, (what, info)
        assert tok == int(np.argmax(logits.cpu().numpy()))
