"""Decoder-block steps with their epilogues fused into the weight stream:
the 1536-wide fp16 decoder as blocks (o + residual, gate|up -> SwiGLU, down
reading the SwiGLU result + residual) in ONE persistent launch, against the
oracle (each op checked on the inputs it actually read) and bitwise against
the same ops run one by one (dg_linear_forward); the unfused form of the same
step agrees with the oracle too.  And the int4 decoder with an fp16 lm_head
(two persistent launches) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import plans, synth
from gpu_util import DEV, bits, host, need_gpu, sync

pytestmark = pytest.mark.gpu


def _check_block(layers, step, what):
    for li, (L, xin, ys) in enumerate(zip(layers, step.inputs, step.outputs)):
        lin = {l.name: l for l in L.linears}
        for n in ("q", "k", "v"):
            yr, A = oracle.gemv_fp(bits(lin[n].W), bits(xin["x_attn"].cpu()))
            tol.assert_close(host(ys[n]).astype(np.float64), yr, A, "f16", "%s %d %s" % (what, li, n))
        h1r, A = oracle.gemv_residual_fp(bits(lin["o"].W), bits(xin["x_o"].cpu()), bits(xin["h"].cpu()))
        tol.assert_close(host(ys["h1"]).astype(np.float64), h1r, A, "f16", "%s %d h1" % (what, li))
        h, g, u, Ag, Au = oracle.gemv_swiglu_fp(bits(lin["gate"].W), bits(lin["up"].W),
                                                bits(xin["x_mlp"].cpu()))
        tol.assert_within(host(ys["act"]).astype(np.float64), h, tol.bound_swiglu(g, u, Ag, Au),
                          "%s %d act" % (what, li))
        # down on what it read: the step's own act and h1
        h2r, A = oracle.gemv_residual_fp(bits(lin["down"].W), bits(ys["act"].cpu()),
                                         bits(ys["h1"].cpu()))
        tol.assert_close(host(ys["h2"]).astype(np.float64), h2r, A, "f16", "%s %d h2" % (what, li))


def test_fused_block_step_one_launch_against_the_oracle_and_per_op_calls():
    need_gpu()
    layers = synth.decode_fp16_workload(seed=8, layers=3)
    hs = synth.residual_stream(3, 1536, seed=8)
    step = plans.fp16_block_step(layers, hs, DEV, fused=True)
    assert step.n_launches == 1
    step.run()
    sync()
    dg.check_device_status()
    _check_block(layers, step, "fused")
    # the same ops one at a time give the same bits
    for i, op in enumerate(step.plan.array):
        out = torch.empty(1, op.N, dtype=torch.float16, device=DEV)
        ref = dg.Linear.from_buffer_copy(op)
        ref.y = out.data_ptr()
        dg.linear_forward(ref)
        sync()
        # find the step's own output tensor by pointer
        ys = [t for d in step.outputs for t in d.values() if t.data_ptr() == op.y]
        assert len(ys) == 1
        assert torch.equal(ys[0], out), i


def test_unfused_block_step_agrees_with_the_oracle():
    need_gpu()
    layers = synth.decode_fp16_workload(seed=9, layers=2)
    hs = synth.residual_stream(2, 1536, seed=9)
    step = plans.fp16_block_step(layers, hs, DEV, fused=False)
    step.run()
    sync()
    _check_block(layers, step, "unfused")


def test_int4_decoder_with_fp16_lm_head():
    need_gpu()
    layers, _, xh = synth.decode_int4_workload(seed=10, layers=2, hidden=1024, kv=256,
                                               inter=2816, vocab=32000)
    head = synth.fp16_head(32000, 1024, seed=10)
    step = plans.int4_decode_step(layers, head, xh, DEV, act="a16")
    assert step.n_launches == 2   # the int4 layers, then the fp16 head
    dg.decode_step_weights(step.plan, step.ws)
    sync()
    lr, A, _ = oracle.lm_head(bits(head.W), bits(xh))
    logits = step.head_logits.cpu().double().numpy()
    tol.assert_close(logits, lr, A, "f32", "fp16 head")
    tok = int(step.head_token.item())
    ok, _ = tol.argmax_check(tok, lr, A)
    assert ok and tok == int(np.argmax(step.head_logits.cpu().numpy()))
    L = layers[1]
    for lin in L.linears:
        yr, A = oracle.gemv_w4a16(lin.W.numpy(), bits(lin.scales), bits(L.inputs[lin.x_name]))
        tol.assert_close(host(step.outputs[1][lin.name]).astype(np.float64), yr, A, "f16", lin.name)
