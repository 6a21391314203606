"""The workspace-free lm_head entry point (dg_lm_head_argmax_noalloc).

Callers that cannot allocate device memory (a decode loop that must not
allocate once it runs, a plugin whose host runtime owns all device memory)
use this variant: its argmax partials live in a fixed array inside the library.
Here it is called through the C ABI twice in a row — two different heads, so
the second call starts with the first call's partials still in the array — and
each result is checked against dg_lm_head_argmax with a caller workspace, within
the tolerance the other tests use.  This file is collected last.
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


def with_workspace(Wd, xd):
    N, K = Wd.shape
    logits = torch.empty(N, dtype=torch.float32, device=DEV)
    token = torch.empty(1, dtype=torch.int32, device=DEV)
    head = dg.linear(dg.LINEAR_F16, Wd, 1, N, K, x=xd, logits=logits, token=token)
    ws = torch.empty(dg.workspace_bytes([head]), dtype=torch.uint8, device=DEV)
    dg.lm_head_argmax(head, ws)
    sync()
    return logits, int(token.item())


def without_workspace(lib, Wd, xd):
    N, K = Wd.shape
    logits = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    token = torch.full((1,), -5, dtype=torch.int32, device=DEV)
    head = dg.linear(dg.LINEAR_F16, Wd, 1, N, K, x=xd, logits=logits, token=token)
    st = lib.dg_lm_head_argmax_noalloc(ctypes.byref(head),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0, dg.status_string(st)
    sync()
    return logits, int(token.item())


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    need_gpu()
    lib = dg.load()
    cases = [synth.fp_case(248320, 2048, 1, seed=41), synth.fp_case(30011, 1024, 1, seed=42)]
    for W, x in cases:
        Wd, xd = W.to(DEV), x.to(DEV)
        ref_logits, ref_tok = with_workspace(Wd, xd)
        logits, tok = without_workspace(lib, Wd, xd)
        _, A, _ = oracle.lm_head(bits(W), bits(x))
        tol.assert_close(logits.cpu().double().numpy(), ref_logits.cpu().double().numpy(), A,
                         "f32", "noalloc logits N=%d" % W.shape[0])
        assert tok == ref_tok
        assert tok == int(np.argmax(logits.cpu().numpy()))
