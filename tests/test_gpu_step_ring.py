"""The fp16 / bf16 decode step through the weight ring (k_step_ring): shapes
that take each of its paths (activations kept in registers or streamed with
the weights, K split over 1, 2 or 4 warps, stages grown to a row longer than
the default stage, ragged and one-chunk rows, fused matrices), lm_heads inside
a step, the fallback to the register-streaming kernel when two stages do not
fit, and a run that writes into its own weights (per-launch path).  Every
output is compared bitwise with the per-op entry points and against the
oracle's bound.

The ring is selected with DG_TUNE=RING=1, which the library reads once per
process: the in-process tests run in a child pytest started with it (and are
skipped in the parent)."""
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
RING_ON = "RING=1" in os.environ.get("DG_TUNE", "")
ring_only = pytest.mark.skipif(not RING_ON, reason="runs in the child pytest (DG_TUNE=RING=1)")
parent_only = pytest.mark.skipif(RING_ON, reason="run by the parent pytest")


@parent_only
def test_ring_kernel_suite_in_a_child_process():
    env = dict(os.environ, DG_TUNE="RING=1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.abspath(__file__), "-q", "-x",
                        "-p", "no:cacheprovider", "-m", "gpu"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    assert " passed" in r.stdout and "failed" not in r.stdout


def _ftype(dtype):
    return dg.F16 if dtype == torch.float16 else dg.BF16


def _kind(dtype):
    return dg.LINEAR_F16 if dtype == torch.float16 else dg.LINEAR_BF16


def _run_independent(shapes, dtype, seed, fuse_pairs=()):
    """One step over independent ops (N, K); ops i and i+1 listed in
    fuse_pairs share their input (one fused phase).  Returns (cases, ws)."""
    g = synth.generator(seed)
    cases, ops, keep = [], [], []
    x_prev = None
    for i, (N, K) in enumerate(shapes):
        W = synth.normal((N, K), 0.02, g, dtype).to(DEV)
        if i in fuse_pairs:
            x = x_prev
        else:
            x = synth.normal((1, K), 1.0, g, dtype).to(DEV)
        y = torch.empty(1, N, dtype=dtype, device=DEV)
        keep += [W, x, y]
        ops.append(dg.linear(_kind(dtype), W, 1, N, K, x=x, y=y))
        cases.append((W, x, y))
        x_prev = x
    plan = dg.StepPlan(ops, keep)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=DEV)
    dg.decode_step_weights(plan, ws)
    sync()
    dg.check_device_status()
    return cases


def _check_cases(cases, dtype, oracle_too=True):
    fmt = "f16" if dtype == torch.float16 else "bf16"
    for W, x, y in cases:
        ref = torch.empty_like(y)
        dg.gemv_f16(W, x, ref, dtype=_ftype(dtype))
        sync()
        assert torch.equal(y, ref), tuple(W.shape)
        if oracle_too:
            yr, A = oracle.gemv_fp(bits(W.cpu()), bits(x.cpu()), fmt)
            tol.assert_close(y.float().cpu().double().numpy(), yr, A, fmt, str(tuple(W.shape)))


# K = 3072: 12 chunks per lane (streamed); 4096: 2 warps per row, 8 chunks
# (kept); 12288: 4 warps per row, 12 chunks (streamed); 520: 65 chunks
# (lanes hold 3 or 2); 8: one chunk; 20000: a 40000-byte row, longer than the
# default 36 KB stage.
MIXED = [(1000, 3072), (777, 4096), (300, 12288), (4097, 520), (151, 8), (256, 1536),
         (1, 1536), (40, 20000)]


@ring_only
def test_ring_step_mixed_shapes_fp16():
    need_gpu()
    cases = _run_independent(MIXED, torch.float16, seed=1, fuse_pairs=(6,))
    _check_cases(cases, torch.float16)


@ring_only
def test_ring_step_mixed_shapes_bf16():
    need_gpu()
    cases = _run_independent(MIXED[:6], torch.bfloat16, seed=2)
    _check_cases(cases, torch.bfloat16)


@ring_only
def test_ring_step_with_lm_heads_between_and_at_the_end():
    """[y1 = W1 x0] -> [head 1 reads y1] -> [y3 = W3 x3] -> [head 2 reads x3]:
    grid barriers before head 1 (read after write), after it (its token),
    and a final one for head 2's token."""
    need_gpu()
    g = synth.generator(3)
    W1 = synth.normal((2048, 1024), 0.02, g).to(DEV)
    x0 = synth.normal((1, 1024), 1.0, g).to(DEV)
    Wh1 = synth.normal((32000, 2048), 0.02, g).to(DEV)
    W3 = synth.normal((512, 1024), 0.02, g).to(DEV)
    x3 = synth.normal((1, 1024), 1.0, g).to(DEV)
    Wh2 = synth.normal((5003, 1024), 0.02, g).to(DEV)
    y1 = torch.empty(1, 2048, dtype=torch.float16, device=DEV)
    y3 = torch.empty(1, 512, dtype=torch.float16, device=DEV)
    l1 = torch.empty(32000, dtype=torch.float32, device=DEV)
    l2 = torch.empty(5003, dtype=torch.float32, device=DEV)
    t1 = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    t2 = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    ops = [dg.linear(dg.LINEAR_F16, W1, 1, 2048, 1024, x=x0, y=y1),
           dg.linear(dg.LINEAR_F16, Wh1, 1, 32000, 2048, x=y1, logits=l1, token=t1),
           dg.linear(dg.LINEAR_F16, W3, 1, 512, 1024, x=x3, y=y3),
           dg.linear(dg.LINEAR_F16, Wh2, 1, 5003, 1024, x=x3, logits=l2, token=t2)]
    plan = dg.StepPlan(ops, [W1, x0, Wh1, W3, x3, Wh2, y1, y3, l1, l2, t1, t2])
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=DEV)
    dg.decode_step_weights(plan, ws)
    sync()
    dg.check_device_status()

    r1 = torch.empty_like(y1)
    dg.gemv_f16(W1, x0, r1)
    r3 = torch.empty_like(y3)
    dg.gemv_f16(W3, x3, r3)
    sync()
    assert torch.equal(y1, r1) and torch.equal(y3, r3)
    for W, x, lg, tk in ((Wh1, r1, l1, t1), (Wh2, x3, l2, t2)):
        N, K = W.shape
        rl = torch.empty_like(lg)
        rt = torch.empty_like(tk)
        head = dg.linear(dg.LINEAR_F16, W, 1, N, K, x=x, logits=rl, token=rt)
        hws = torch.empty(dg.workspace_bytes([head]), dtype=torch.uint8, device=DEV)
        dg.lm_head_argmax(head, hws)
        sync()
        assert torch.equal(lg, rl)
        assert int(tk.item()) == int(rt.item())
        lr, A = oracle.gemv_fp(bits(W.cpu()), bits(x.cpu()))
        tol.assert_close(lg.cpu().double().numpy(), lr[0], A[0], "f32", "head %d" % N)
        ok, _ = tol.argmax_check(int(tk.item()), lr[0], A[0])
        assert ok


@ring_only
def test_rows_too_long_for_two_stages_use_the_register_streaming_kernel():
    """A 65536-wide row (128 KB) leaves no room for two ring stages: the launch
    takes k_step; results still equal the per-op calls bitwise."""
    need_gpu()
    cases = _run_independent([(64, 65536), (300, 1024)], torch.float16, seed=4)
    _check_cases(cases, torch.float16, oracle_too=False)
    W, x, y = cases[0]
    yr, A = oracle.gemv_fp(bits(W.cpu()), bits(x.cpu()))
    tol.assert_close(y.cpu().double().numpy(), yr, A, "f16", "65536-wide")


@ring_only
def test_run_that_writes_into_its_own_weights_keeps_op_order():
    """Op 1 writes its output over the first 256 weights of op 2's matrix;
    the step must give what the two calls in order give."""
    need_gpu()
    g = synth.generator(5)
    W1 = synth.normal((256, 512), 0.02, g).to(DEV)
    x1 = synth.normal((1, 512), 1.0, g).to(DEV)
    W2_init = synth.normal((128, 512), 0.02, g).to(DEV)
    x2 = synth.normal((1, 512), 1.0, g).to(DEV)

    W2 = W2_init.clone()
    y1 = W2.view(-1)[:256].view(1, 256)
    y2 = torch.empty(1, 128, dtype=torch.float16, device=DEV)
    ops = [dg.linear(dg.LINEAR_F16, W1, 1, 256, 512, x=x1, y=y1),
           dg.linear(dg.LINEAR_F16, W2, 1, 128, 512, x=x2, y=y2)]
    plan = dg.StepPlan(ops, [W1, x1, W2, x2, y2])
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=DEV)
    dg.decode_step_weights(plan, ws)
    sync()

    R2 = W2_init.clone()
    r1 = R2.view(-1)[:256].view(1, 256)
    dg.gemv_f16(W1, x1, r1)
    r2 = torch.empty_like(y2)
    dg.gemv_f16(R2, x2, r2)
    sync()
    assert torch.equal(W2, R2)
    assert torch.equal(y2, r2)


@parent_only
@pytest.mark.parametrize("tune,workload", [("RING=1,TSB=4,TNS=2,TNC=8", "small"),
                                           ("RING=1,TSB=4,TNS=3", "small"),
                                           ("", "small"),
                                           ("", "splits"),
                                           ("RING=1,TNC=8", "splits"),
                                           ("RING=1", "splits")])
def test_ring_small_stages_and_consumer_counts_in_a_child_process(tune, workload):
    """4 KB stages (a few rows each, the ring wrapped hundreds of times), 8 or
    12 consumer warps, the default kernel (k_step), and phases with rows split
    over 1, 2 and 4 warps back to back."""
    need_gpu()
    env = dict(os.environ, DG_TUNE=tune)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "step_ring_child.py"),
                        workload], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "OK" in r.stdout
