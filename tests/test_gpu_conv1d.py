"""The causal-conv1d decode step (dg_causal_conv1d_update) against the
oracle's definition: every window width 2..8, with and without bias and SiLU,
one and several tokens, a wide channel count; the rolled window bitwise; and
several steps in a row matching the oracle stepped the same way."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance as tol
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import synth
from gpu_util import DEV, bits, host, need_gpu, sync

pytestmark = pytest.mark.gpu


def _case(M, C, W, seed):
    g = synth.generator(seed)
    x = synth.normal((M, C), 1.0, g)
    st = synth.normal((M, C, W - 1), 1.0, g)
    w = synth.normal((C, W), 0.5, g)
    b = synth.normal((C,), 0.1, g)
    return x, st, w, b


def _check(y, yr, v, A, silu, what):
    if silu:
        tol.assert_within(host(y).astype(np.float64), yr, tol.bound_silu(v, A), what)
    else:
        tol.assert_close(host(y).astype(np.float64), yr, A, "f16", what)


@pytest.mark.parametrize("W", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("bias,silu", [(True, True), (False, False), (True, False)])
def test_widths_bias_and_activation(W, bias, silu):
    need_gpu()
    M, C = 2, 8 * 37
    x, st, w, b = _case(M, C, W, seed=W * 10 + bias + 2 * silu)
    std = st.to(DEV)
    y = torch.empty(M, C, dtype=torch.float16, device=DEV)
    dg.causal_conv1d_update(x.to(DEV), std, w.to(DEV), y, bias=b.to(DEV) if bias else None,
                            act=dg.ACT_SILU if silu else dg.ACT_NONE)
    sync()
    yr, v, A, ns = oracle.causal_conv1d_update(bits(x), bits(st), bits(w), bits(b) if bias else None,
                                               act="silu" if silu else "none")
    _check(y, yr, v, A, silu, "conv W=%d" % W)
    assert np.array_equal(host(std).view(np.uint16), ns)


def test_several_steps_and_a_wide_layer():
    """4 steps of a 4-tap, 8192-channel layer (one token), the window carried
    by the kernel from step to step, against the oracle carried the same way."""
    need_gpu()
    M, C, W = 1, 8192, 4
    x0, st, w, b = _case(M, C, W, seed=5)
    g = synth.generator(6)
    xs = [x0] + [synth.normal((M, C), 1.0, g) for _ in range(3)]
    std, wd, bd = st.to(DEV), w.to(DEV), b.to(DEV)
    ost = bits(st)
    for t, x in enumerate(xs):
        y = torch.empty(M, C, dtype=torch.float16, device=DEV)
        dg.causal_conv1d_update(x.to(DEV), std, wd, y, bias=bd)
        sync()
        yr, v, A, ost = oracle.causal_conv1d_update(bits(x), ost, bits(w), bits(b))
        _check(y, yr, v, A, True, "step %d" % t)
        assert np.array_equal(host(std).view(np.uint16), ost)
