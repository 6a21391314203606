"""Decode-step weight streams (dg_decode_step_weights) in the launch
configuration the benchmark times: the 28-layer 1536-wide fp16 decoder (every
output of every matrix checked) and the 32-layer 4096-wide int4 decoder with
its 128256-row lm_head (sampled rows of every matrix, the whole lm_head)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import plans, synth
from gpu_util import DEV, bits, need_gpu, sync

pytestmark = pytest.mark.gpu


def test_fp16_decoder_step_all_outputs():
    need_gpu()
    layers = synth.decode_fp16_workload(seed=0)
    step = plans.fp16_decode_step(layers, DEV)
    assert step.weight_bytes == 2620391424
    assert step.n_launches == 1
    dg.decode_step_weights(step.plan, step.ws)
    sync()
    for li, L in enumerate(layers):
        for lin in L.linears:
            yr, A = oracle.gemv_fp(bits(lin.W), bits(L.inputs[lin.x_name]))
            y = step.outputs[li][lin.name].cpu().double().numpy()
            tol.assert_close(y, yr, A, "f16", "layer %d %s" % (li, lin.name))


def test_fp16_decoder_step_is_deterministic_and_graph_replayable():
    need_gpu()
    layers = synth.decode_fp16_workload(seed=1, layers=3)
    step = plans.fp16_decode_step(layers, DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dg.decode_step_weights(step.plan, step.ws, stream=s)
    s.synchronize()
    ref = [{k: v.clone() for k, v in o.items()} for o in step.outputs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dg.decode_step_weights(step.plan, step.ws, stream=s)
    for _ in range(3):
        for o in step.outputs:
            for v in o.values():
                v.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        for o, r in zip(step.outputs, ref):
            for k in o:
                assert torch.equal(o[k], r[k]), k


@pytest.fixture(scope="module")
def int4_workload():
    need_gpu()
    return synth.decode_int4_workload(seed=0)


def _slice_edge_rows(N, grids):
    """Rows of an N-row phase next to the persistent kernel's CTA slice
    boundaries (CTA b of G starts at floor(N b / G)), plus the first and last."""
    rows = {0, N - 1}
    for G in grids:
        for b in range(1, G):
            r = N * b // G
            rows.update((r - 1, r))
    return rows


def _phase_rows(L, grids):
    """For every matrix of a decoder layer: its rows at the slice edges of the
    fused phase it belongs to (q|k|v, o, gate|up, down), in its own numbering."""
    phases, cur, prev = [], [], None
    for lin in L.linears:
        if cur and lin.x_name != prev:
            phases.append(cur)
            cur = []
        cur.append(lin)
        prev = lin.x_name
    phases.append(cur)
    out = {}
    for ph in phases:
        N = sum(l.N for l in ph)
        edges = _slice_edge_rows(N, grids)
        base = 0
        for l in ph:
            out[l.name] = sorted({r - base for r in edges if base <= r < base + l.N} |
                                 {0, l.N - 1})
            base += l.N
    return out


def _check_codes(layers, codes, head_x=None, head_codes=None):
    """The int8 codes and fp32 scales the step's quantizer wrote equal the
    oracle's quantizer bit for bit."""
    n = 0
    for li, (L, qc) in enumerate(zip(layers, codes)):
        for name, (xq, xs) in qc.items():
            q, s = oracle.quant_act(bits(L.inputs[name]))
            assert np.array_equal(xq.cpu().numpy(), q), "codes layer %d %s" % (li, name)
            assert np.array_equal(xs.cpu().numpy().view(np.uint32), s.view(np.uint32)), \
                "scale layer %d %s" % (li, name)
            n += 1
    if head_codes is not None:
        q, s = oracle.quant_act(bits(head_x))
        assert np.array_equal(head_codes[0].cpu().numpy(), q), "lm_head codes"
        assert np.array_equal(head_codes[1].cpu().numpy().view(np.uint32), s.view(np.uint32))
        n += 1
    return n


@pytest.mark.parametrize("act", ["a16", "a8"])
def test_int4_decoder_step(int4_workload, act):
    """Every row of every matrix of one layer; in all 32 layers, the rows at
    the CTA slice boundaries of each fused phase (for one and two CTAs per SM)
    and the first and last row of every matrix; the whole lm_head; (W4A8) the
    codes and scales the step's quantizer wrote, bitwise."""
    layers, head, x_head = int4_workload
    step = plans.int4_decode_step(layers, head, x_head, DEV, act=act)
    assert step.weight_bytes == 4221370368
    dg.decode_step_weights(step.plan, step.ws)
    sync()
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    grids = (sms, 2 * sms)
    full_layer = 13
    for li, L in enumerate(layers):
        edge = _phase_rows(L, grids)
        for lin in L.linears:
            rows = None if li == full_layer else np.array(edge[lin.name], np.int64)
            x = L.inputs[lin.x_name]
            if act == "a16":
                yr, A = oracle.gemv_w4a16(lin.W.numpy(), bits(lin.scales), bits(x), rows=rows)
            else:
                q, s = oracle.quant_act(bits(x))
                yr, A, _ = oracle.gemv_w4a8(lin.W.numpy(), bits(lin.scales), q, s, rows=rows)
            y = step.outputs[li][lin.name].cpu().double().numpy()
            if rows is not None:
                y = y[:, rows]
            tol.assert_close(y, yr, A, "f16", "%s layer %d %s" % (act, li, lin.name))
    if act == "a16":
        lr, A = oracle.gemv_w4a16(head.W.numpy(), bits(head.scales), bits(x_head))
    else:
        q, s = oracle.quant_act(bits(x_head))
        lr, A, _ = oracle.gemv_w4a8(head.W.numpy(), bits(head.scales), q, s)
        assert _check_codes(layers, step.act_codes, x_head, step.head_codes) == 4 * 32 + 1
    logits = step.head_logits.cpu().double().numpy()
    tol.assert_close(logits, lr[0], A[0], "f32", "%s lm_head" % act)
    tok = int(step.head_token.item())
    ok, _ = tol.argmax_check(tok, lr[0], A[0])
    assert ok
    assert tok == int(np.argmax(step.head_logits.cpu().numpy()))


def _per_op_outputs(ops, M=1):
    """Runs every op of a plan through the per-op entry points."""
    outs = []
    for op in ops:
        N, K = op.N, op.K
        if op.token:
            continue
        y = torch.empty(M, N, dtype=torch.float16, device=DEV)
        if op.kind == dg.LINEAR_F16:
            dg.load().dg_gemv_f16(op.W, op.x, y.data_ptr(), dg.F16, M, N, K, None, 0,
                                  torch.cuda.current_stream().cuda_stream)
        else:
            x_i8 = op.x_i8 if op.kind == dg.LINEAR_W4A8 else None
            dg.load().dg_gemv_w4(op.W, op.w_scale, op.group_size, op.x, x_i8, op.x_scale,
                                 y.data_ptr(), M, N, K, None, 0,
                                 torch.cuda.current_stream().cuda_stream)
        outs.append(y)
    sync()
    return outs


def test_persistent_step_equals_per_op_calls_bitwise_fp16():
    need_gpu()
    layers = synth.decode_fp16_workload(seed=3, layers=4)
    step = plans.fp16_decode_step(layers, DEV)
    assert step.n_launches == 1
    dg.decode_step_weights(step.plan, step.ws)
    sync()
    got = [y for L in step.outputs for y in L.values()]
    ref = _per_op_outputs(list(step.plan.array))
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("act", ["a16", "a8"])
def test_persistent_step_equals_per_op_calls_bitwise_int4(act):
    need_gpu()
    layers, head, xh = synth.decode_int4_workload(seed=4, layers=2, hidden=1024, kv=256,
                                                  inter=2816, vocab=32000)
    step = plans.int4_decode_step(layers, head, xh, DEV, act=act)
    dg.decode_step_weights(step.plan, step.ws)
    sync()
    # the step wrote the int8 codes / scales it used (W4A8): the per-op calls reuse them
    got = [y for L in step.outputs for y in L.values()]
    ref = _per_op_outputs(list(step.plan.array))
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    if act == "a8":  # the codes and scales the step wrote equal the oracle's quantizer
        assert _check_codes(layers, step.act_codes, xh, step.head_codes) == 4 * 2 + 1
    # the lm_head token against the oracle
    if act == "a16":
        lr, A = oracle.gemv_w4a16(head.W.numpy(), bits(head.scales), bits(xh))
    else:
        q, s = oracle.quant_act(bits(xh))
        lr, A, _ = oracle.gemv_w4a8(head.W.numpy(), bits(head.scales), q, s)
    tol.assert_close(step.head_logits.cpu().double().numpy(), lr[0], A[0], "f32", "head")
    assert int(step.head_token.item()) == int(np.argmax(step.head_logits.cpu().numpy()))


def test_two_token_step_uses_per_group_launches_and_matches_oracle():
    need_gpu()
    layers = synth.decode_fp16_workload(seed=5, layers=2, M=2)
    step = plans.fp16_decode_step(layers, DEV, M=2)
    assert step.n_launches == 2 * 4
    dg.decode_step_weights(step.plan, step.ws)
    sync()
    for li, L in enumerate(layers):
        for lin in L.linears:
            yr, A = oracle.gemv_fp(bits(lin.W), bits(L.inputs[lin.x_name]))
            tol.assert_close(step.outputs[li][lin.name].cpu().double().numpy(), yr, A, "f16",
                             "M=2 layer %d %s" % (li, lin.name))


def test_bounded_wait_timeout_reaches_the_host_as_a_status():
    need_gpu()
    dg.check_device_status()  # clean start
    dg.selftest_wait_timeout(2000)
    with pytest.raises(dg.DGError) as e:
        dg.check_device_status()
    assert e.value.status == 6  # DG_ERR_TIMEOUT
    dg.check_device_status()  # the flag was cleared; the context is still usable
    W, x = synth.fp_case(64, 64, 1, seed=1)
    y = torch.empty(1, 64, dtype=torch.float16, device=DEV)
    dg.gemv_f16(W.to(DEV), x.to(DEV), y)
    sync()


def test_dependent_ops_in_one_step_match_sequential_calls():
    """An op that reads an earlier op's output (read after write) and an op
    that overwrites an earlier op's input (write after read) force grid
    barriers inside the persistent kernel; results equal sequential calls."""
    need_gpu()
    g = synth.generator(9)
    K0, N1, N2, N3 = 1024, 2048, 1536, 3072
    W1 = synth.normal((N1, K0), 0.02, g).to(DEV)
    W2 = synth.normal((N2, N1), 0.02, g).to(DEV)
    W3 = synth.normal((N3, N2), 0.02, g).to(DEV)
    W4 = synth.normal((K0, N2), 0.02, g).to(DEV)
    x0 = synth.normal((1, K0), 1.0, g).to(DEV)

    def run_step():
        buf = torch.zeros(1, 8192, dtype=torch.float16, device=DEV)
        xa = buf[:, :K0]
        xa.copy_(x0)
        y1 = buf[:, 1024:1024 + N1]
        y2 = buf[:, 3072:3072 + N2]
        y3 = torch.empty(1, N3, dtype=torch.float16, device=DEV)
        ops = [dg.linear(dg.LINEAR_F16, W1, 1, N1, K0, x=xa, y=y1),     # y1 = f(x)
               dg.linear(dg.LINEAR_F16, W2, 1, N2, N1, x=y1, y=y2),     # reads y1 (RAW)
               dg.linear(dg.LINEAR_F16, W3, 1, N3, N2, x=y2, y=y3),     # reads y2 (RAW)
               dg.linear(dg.LINEAR_F16, W4, 1, K0, N2, x=y2, y=xa)]     # overwrites x (WAR)
        plan = dg.StepPlan(ops, [buf, y3])
        ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=DEV)
        dg.decode_step_weights(plan, ws)
        sync()
        return y1.clone(), y2.clone(), y3.clone(), xa.clone()

    def run_sequential():
        y1 = torch.empty(1, N1, dtype=torch.float16, device=DEV)
        y2 = torch.empty(1, N2, dtype=torch.float16, device=DEV)
        y3 = torch.empty(1, N3, dtype=torch.float16, device=DEV)
        y4 = torch.empty(1, K0, dtype=torch.float16, device=DEV)
        dg.gemv_f16(W1, x0, y1)
        dg.gemv_f16(W2, y1, y2)
        dg.gemv_f16(W3, y2, y3)
        dg.gemv_f16(W4, y2, y4)
        sync()
        return y1, y2, y3, y4

    for got, ref in zip(run_step(), run_sequential()):
        assert torch.equal(got, ref)


def test_w4a8_step_with_one_shared_code_buffer_for_every_layer():
    """Callers often reuse one int8 scratch buffer for every layer's codes.
    Then no input may be quantized ahead of its phase: each phase quantizes
    its own input in place; results still match the oracle."""
    need_gpu()
    layers, _, _ = synth.decode_int4_workload(seed=6, layers=2, hidden=1024, kv=256, inter=2048,
                                              vocab=0)
    xq = torch.empty(1, 2048, dtype=torch.int8, device=DEV)     # shared scratch (max K)
    xs = torch.empty(1, dtype=torch.float32, device=DEV)
    ops, keep, outs = [], [], []
    for L in layers:
        xin = {k: v.to(DEV) for k, v in L.inputs.items()}
        keep += list(xin.values())
        for lin in L.linears:
            W, S = lin.W.to(DEV), lin.scales.to(DEV)
            y = torch.empty(1, lin.N, dtype=torch.float16, device=DEV)
            keep += [W, S, y]
            outs.append((L, lin, y))
            ops.append(dg.linear(dg.LINEAR_W4A8, W, 1, lin.N, lin.K, w_scale=S, x=xin[lin.x_name],
                                 x_i8=xq[:, :lin.K], x_scale=xs, y=y))
    plan = dg.StepPlan(ops, keep)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=DEV)
    dg.decode_step_weights(plan, ws)
    sync()
    for L, lin, y in outs:
        q, s = oracle.quant_act(bits(L.inputs[lin.x_name]))
        yr, A, _ = oracle.gemv_w4a8(lin.W.numpy(), bits(lin.scales), q, s)
        tol.assert_close(y.cpu().double().numpy(), yr, A, "f16", "shared-scratch %s" % lin.name)


def test_w4a8_step_with_given_codes_reads_the_prologue_layout():
    """W4A8 ops whose int8 codes are given (no fp16 x): the launch's prologue
    lays them out once in the workspace and every CTA reads them from there.
    Two fused ops share one code vector, a third has its own; ragged N, groups
    of 32 and 128; results equal the per-op calls bitwise and the oracle."""
    need_gpu()
    g = synth.generator(17)
    shapes = [(777, 4096, 32), (1025, 4096, 32), (333, 1024, 128)]
    xs = {}
    keep, ops, cases = [], [], []
    for i, (N, K, grp) in enumerate(shapes):
        Wq = synth.int4_packed(N, K, g).to(DEV)
        sc = synth.uniform((N, K // grp), 1e-3, 1e-2, g, torch.float16).to(DEV)
        key = 0 if i < 2 else i  # ops 0 and 1 share their codes (one fused phase)
        if key not in xs:
            xq = synth.int8_codes((1, K), g).to(DEV)
            s = synth.uniform((1,), 1e-3, 1e-1, g).to(DEV)
            xs[key] = (xq, s)
        xq, s = xs[key]
        y = torch.empty(1, N, dtype=torch.float16, device=DEV)
        keep += [Wq, sc, xq, s, y]
        ops.append(dg.linear(dg.LINEAR_W4A8, Wq, 1, N, K, w_scale=sc, x_i8=xq, x_scale=s, y=y,
                             group_size=grp))
        cases.append((Wq, sc, xq, s, y, grp))
    plan = dg.StepPlan(ops, keep)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=DEV)
    for _ in range(2):  # the workspace is reused
        dg.decode_step_weights(plan, ws)
    sync()
    dg.check_device_status()
    for Wq, sc, xq, s, y, grp in cases:
        ref = torch.empty_like(y)
        dg.gemv_w4(Wq, sc, ref, x_i8=xq, x_scale=s, group_size=grp)
        sync()
        assert torch.equal(y, ref), tuple(Wq.shape)
        yr, A, _ = oracle.gemv_w4a8(Wq.cpu().numpy(), bits(sc.cpu()), xq.cpu().numpy(),
                                    s.cpu().numpy(), group=grp)
        tol.assert_close(y.cpu().double().numpy(), yr, A, "f16", "given codes %s" % (tuple(Wq.shape),))


def test_int4_step_mixing_laid_out_and_staged_activations_matches_sequential_calls():
    """W4A16 ops: y1 = W1 x0 (x0 read-only: laid out by the prologue),
    y2 = W2 y1 (y1 written in the launch: staged in shared memory after a
    grid barrier), y3 = W3 x3 (laid out again); equal to the calls in order."""
    need_gpu()
    g = synth.generator(23)
    K0, N1, N2, N3 = 2048, 4096, 1024, 3072
    W1, W2, W3 = (synth.int4_packed(N, K, g).to(DEV) for N, K in ((N1, K0), (N2, N1), (N3, K0)))
    S1, S2, S3 = (synth.uniform((N, K // 32), 1e-3, 1e-2, g, torch.float16).to(DEV)
                  for N, K in ((N1, K0), (N2, N1), (N3, K0)))
    x0 = synth.normal((1, K0), 1.0, g).to(DEV)
    x3 = synth.normal((1, K0), 1.0, g).to(DEV)
    y1 = torch.empty(1, N1, dtype=torch.float16, device=DEV)
    y2 = torch.empty(1, N2, dtype=torch.float16, device=DEV)
    y3 = torch.empty(1, N3, dtype=torch.float16, device=DEV)
    ops = [dg.linear(dg.LINEAR_W4A16, W1, 1, N1, K0, w_scale=S1, x=x0, y=y1),
           dg.linear(dg.LINEAR_W4A16, W2, 1, N2, N1, w_scale=S2, x=y1, y=y2),
           dg.linear(dg.LINEAR_W4A16, W3, 1, N3, K0, w_scale=S3, x=x3, y=y3)]
    plan = dg.StepPlan(ops, [W1, W2, W3, S1, S2, S3, x0, x3, y1, y2, y3])
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=DEV)
    dg.decode_step_weights(plan, ws)
    sync()
    dg.check_device_status()
    r1, r2, r3 = torch.empty_like(y1), torch.empty_like(y2), torch.empty_like(y3)
    dg.gemv_w4(W1, S1, r1, x_f16=x0)
    dg.gemv_w4(W2, S2, r2, x_f16=r1)
    dg.gemv_w4(W3, S3, r3, x_f16=x3)
    sync()
    for a, b in ((y1, r1), (y2, r2), (y3, r3)):
        assert torch.equal(a, b)
    yr, A = oracle.gemv_w4a16(W2.cpu().numpy(), bits(S2.cpu()), bits(r1.cpu()))
    tol.assert_close(y2.cpu().double().numpy(), yr, A, "f16", "chained W4A16")
