"""The C ABI on a host without a GPU: libdg.so loads, exports every entry point
include/dg.h declares, and rejects bad arguments on the host with the
documented status before any CUDA call (fake, never-dereferenced pointers)."""
import ctypes
import os
import re

import pytest

import quantized_skinny_gemm_gb300 as dg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA, TIMEOUT = range(7)
A = 0x100000          # a fake 16-byte-aligned device address (never dereferenced)
B = 0x200000
ODD = 0x100008        # 8-byte but not 16-byte aligned


@pytest.fixture(scope="module")
def lib():
    from quantized_skinny_gemm_gb300 import build
    build.build()
    return dg.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12, names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for i, name in enumerate(["DG_OK", "DG_ERR_INVALID_ARG", "DG_ERR_UNSUPPORTED",
                              "DG_ERR_MISALIGNED", "DG_ERR_WORKSPACE", "DG_ERR_CUDA",
                              "DG_ERR_TIMEOUT"]):
        assert dg.status_string(i) == name
    assert dg.version().startswith("dg ")


def test_linear_struct_layout_matches_header():
    # 5 int32, 4 bytes padding, 9 pointers (to 96), epilogue + reserved int32, 3 pointers
    assert ctypes.sizeof(dg.Linear) == 128
    assert dg.Linear.W.offset == 24
    assert dg.Linear.epilogue.offset == 96
    assert dg.Linear.residual.offset == 104
    assert dg.Linear.W2.offset == 112 and dg.Linear.w2_scale.offset == 120


def test_gemv_f16_validation(lib):
    f = lib.dg_gemv_f16
    assert f(None, A, B, 0, 1, 8, 8, None, 0, None) == INVALID
    assert f(A, A, B, 5, 1, 8, 8, None, 0, None) == INVALID         # bad dtype
    assert f(A, A, B, 0, 0, 8, 8, None, 0, None) == INVALID         # M = 0
    assert f(A, A, B, 0, 1, 0, 8, None, 0, None) == INVALID         # N = 0
    assert f(A, A, B, 0, 17, 8, 8, None, 0, None) == UNSUPPORTED    # M > 16
    assert f(A, A, B, 0, 1, 8, 12, None, 0, None) == MISALIGNED     # K % 8
    assert f(ODD, A, B, 0, 1, 8, 8, None, 0, None) == MISALIGNED    # W
    assert f(A, ODD, B, 0, 1, 8, 8, None, 0, None) == MISALIGNED    # x
    assert f(A, A, B + 1, 0, 1, 8, 8, None, 0, None) == MISALIGNED  # y odd


def test_gemv_w8a8_validation(lib):
    f = lib.dg_gemv_w8a8
    assert f(A, A, A, A, None, None, 1, 8, 16, None, 0, None) == INVALID    # no output
    assert f(A, None, A, A, B, None, 1, 8, 16, None, 0, None) == INVALID    # no w_scale
    assert f(A, A, A, None, B, None, 1, 8, 16, None, 0, None) == INVALID    # no x_scale
    assert f(A, A, A, A, B, None, 1, 8, 24, None, 0, None) == MISALIGNED    # K % 16
    assert f(A, A, A, A, B, None, 1, 8, 262144, None, 0, None) == UNSUPPORTED


def test_gemv_w4_validation(lib):
    f = lib.dg_gemv_w4
    assert f(A, A, 32, None, None, None, B, 1, 8, 64, None, 0, None) == INVALID  # no x
    assert f(A, A, 48, A, None, None, B, 1, 8, 96, None, 0, None) == UNSUPPORTED  # group 48
    assert f(A, A, 64, A, None, None, B, 1, 8, 96, None, 0, None) == UNSUPPORTED  # K % group
    assert f(A, A, 32, A, None, None, B, 1, 8, 48, None, 0, None) == MISALIGNED   # K % 32
    assert f(A, A, 32, None, A, None, B, 1, 8, 64, None, 0, None) == INVALID      # a8 no scale
    assert f(A, None, 32, A, None, None, B, 1, 8, 64, None, 0, None) == INVALID   # no scales


def test_quantize_validation(lib):
    f = lib.dg_quantize_act_i8
    assert f(None, A, A, 1, 8, None) == INVALID
    assert f(A, A, A, 1, 12, None) == MISALIGNED
    assert f(A, ODD, A, 1, 8, None) == MISALIGNED


def _head(**kw):
    d = dict(kind=dg.LINEAR_F16, M=1, N=100, K=64, group_size=32, W=A, x=A, logits=B,
             token=B + 64)
    d.update(kw)
    return dg.Linear(**d)


def test_lm_head_validation_and_workspace(lib):
    h = _head()
    need = dg.workspace_bytes([h])
    assert need > 0 and need % 16 == 0
    assert lib.dg_lm_head_argmax(ctypes.byref(h), None, 0, None) == WORKSPACE
    assert lib.dg_lm_head_argmax(ctypes.byref(h), A, need - 16, None) == WORKSPACE
    assert lib.dg_lm_head_argmax(ctypes.byref(_head(M=2)), A, need, None) == INVALID
    assert lib.dg_lm_head_argmax(ctypes.byref(_head(logits=None)), A, need, None) == INVALID
    assert lib.dg_lm_head_argmax(ctypes.byref(_head(kind=dg.LINEAR_W8A8, w_scale=A, x_i8=A,
                                                    x_scale=A, x=None)), A, need,
                                 None) == UNSUPPORTED
    plain = dg.Linear(kind=dg.LINEAR_F16, M=1, N=8, K=8, W=A, x=A, y=B)
    assert dg.workspace_bytes([plain]) == 256  # the persistent step's barrier words


def test_lm_head_noalloc_validation(lib):
    """The workspace-free lm_head rejects bad heads on the host before any
    CUDA call, with the statuses dg_lm_head_argmax uses."""
    f = lib.dg_lm_head_argmax_noalloc
    assert f(None, None) == INVALID
    assert f(ctypes.byref(_head(token=None)), None) == INVALID
    assert f(ctypes.byref(_head(logits=None)), None) == INVALID
    assert f(ctypes.byref(_head(M=2)), None) == INVALID
    assert f(ctypes.byref(_head(W=None)), None) == INVALID
    assert f(ctypes.byref(_head(x=None)), None) == INVALID
    assert f(ctypes.byref(_head(W=ODD)), None) == MISALIGNED
    assert f(ctypes.byref(_head(K=60)), None) == MISALIGNED
    assert f(ctypes.byref(_head(token=B + 2)), None) == MISALIGNED
    assert f(ctypes.byref(_head(kind=dg.LINEAR_W8A8, w_scale=A, x_i8=A, x_scale=A, x=None)),
             None) == UNSUPPORTED
    # the package wrapper raises the same status
    with pytest.raises(dg.DGError) as e:
        dg.lm_head_argmax_noalloc(_head(M=2), stream=0)
    assert e.value.status == INVALID


def test_workspace_covers_split_k_partials_of_small_ops():
    # a per-op call with at most 65536 outputs may split K into up to 8 ranges
    # of M x N fp32 / int32 partials; larger ones never split
    f16 = lambda N, M=1: dg.Linear(kind=dg.LINEAR_F16, M=M, N=N, K=1536, W=A, x=A, y=B)
    assert dg.workspace_bytes([f16(256)]) == 8 * 256 * 4
    assert dg.workspace_bytes([f16(1000, M=4)]) == 8 * 4000 * 4
    assert dg.workspace_bytes([f16(65536)]) == 8 * 65536 * 4
    assert dg.workspace_bytes([f16(65537)]) == 256


def test_workspace_holds_the_w4a8_activation_layouts():
    # per W4A8 op at M = 1: ceil(K/32/32)*32 chunks x 32 bytes of interleaved
    # codes + K/32 int32 chunk sums, rounded up to 256 bytes, after the
    # barrier words (and the argmax partials when an op is an lm_head)
    def w4a8(K, **kw):
        d = dict(kind=dg.LINEAR_W4A8, M=1, N=8, K=K, W=A, w_scale=A, x_i8=A, x_scale=A, y=B,
                 group_size=32)
        d.update(kw)
        return dg.Linear(**d)
    assert dg.workspace_bytes([w4a8(4096)]) == 256 + 4096 + 512
    assert dg.workspace_bytes([w4a8(1024)]) == 256 + 1024 + 128 + 128  # 1152 -> 1280
    assert dg.workspace_bytes([w4a8(14336), w4a8(4096)]) == 256 + (14336 + 1792) + 4608
    head_ws = dg.workspace_bytes([_head()])
    assert dg.workspace_bytes([w4a8(4096), _head()]) == head_ws + 4608
    # M > 1 runs per group: no layout; the split-K bound 8 x M x N x 4 = 512
    assert dg.workspace_bytes([w4a8(4096, M=2)]) == 512
    # W4A16: the fp16 interleaved activations, 64 bytes per 32-code chunk
    assert dg.workspace_bytes([w4a8(4096, kind=dg.LINEAR_W4A16, x=A, x_i8=None,
                                    x_scale=None)]) == 256 + 128 * 64
    assert dg.workspace_bytes([w4a8(14336, kind=dg.LINEAR_W4A16, x=A, x_i8=None,
                                    x_scale=None)]) == 256 + 14 * 32 * 64


def test_decode_step_validates_every_op_first(lib):
    good = [dg.Linear(kind=dg.LINEAR_F16, M=1, N=8, K=8, W=A, x=A, y=B) for _ in range(6)]
    bad = list(good)
    bad[5] = dg.Linear(kind=dg.LINEAR_F16, M=1, N=8, K=12, W=A, x=A, y=B)
    arr = (dg.Linear * 6)(*bad)
    assert lib.dg_decode_step_weights(ctypes.cast(arr, ctypes.c_void_p), 6, None, 0,
                                      None) == MISALIGNED
    assert lib.dg_decode_step_weights(None, 0, None, 0, None) == INVALID
    withhead = (dg.Linear * 2)(good[0], _head())
    assert lib.dg_decode_step_weights(ctypes.cast(withhead, ctypes.c_void_p), 2, None, 0,
                                      None) == WORKSPACE
    plain = (dg.Linear * 1)(good[0])
    assert lib.dg_decode_step_weights(ctypes.cast(plain, ctypes.c_void_p), 1, None, 0,
                                      None) == WORKSPACE
    assert lib.dg_decode_step_weights(ctypes.cast(plain, ctypes.c_void_p), 1, ODD, 256,
                                      None) == MISALIGNED


def test_selftest_validation(lib):
    assert lib.dg_selftest_wait_timeout(0, None) == INVALID
    assert lib.dg_selftest_wait_timeout(10 ** 8, None) == INVALID


def test_probe_validation(lib):
    assert lib.dg_probe_copy(A, B, 24, None) == MISALIGNED
    assert lib.dg_probe_read(None, 16, A, None) == INVALID


def _op(**kw):
    d = dict(kind=dg.LINEAR_F16, M=1, N=8, K=64, group_size=32, W=A, x=A, y=B)
    d.update(kw)
    return dg.Linear(**d)


def test_linear_forward_and_epilogue_validation(lib):
    f = lib.dg_linear_forward
    assert f(None, None, 0, None) == INVALID
    assert f(ctypes.byref(_head()), None, 0, None) == INVALID           # lm_heads go elsewhere
    assert f(ctypes.byref(_op(epilogue=7)), None, 0, None) == INVALID
    assert f(ctypes.byref(_op(reserved=1)), None, 0, None) == INVALID
    assert f(ctypes.byref(_op(epilogue=dg.EPI_RESIDUAL)), None, 0, None) == INVALID  # no residual
    assert f(ctypes.byref(_op(epilogue=dg.EPI_RESIDUAL, residual=B + 1)), None, 0,
             None) == MISALIGNED
    assert f(ctypes.byref(_op(epilogue=dg.EPI_SWIGLU)), None, 0, None) == INVALID    # no W2
    assert f(ctypes.byref(_op(epilogue=dg.EPI_SWIGLU, W2=ODD)), None, 0, None) == MISALIGNED
    assert f(ctypes.byref(_op(kind=dg.LINEAR_W4A16, w_scale=A, epilogue=dg.EPI_SWIGLU, W2=A)),
             None, 0, None) == INVALID                                    # no w2_scale
    assert f(ctypes.byref(_op(kind=dg.LINEAR_W8A8, w_scale=A, x=None, x_i8=A, x_scale=A,
                              epilogue=dg.EPI_SWIGLU, W2=A)), None, 0, None) == UNSUPPORTED
    assert f(ctypes.byref(_op(kind=dg.LINEAR_W8A8, w_scale=A, x=None, x_i8=A, x_scale=A,
                              acc_out=B, epilogue=dg.EPI_RESIDUAL, residual=A)), None, 0,
             None) == INVALID
    head = _head(epilogue=dg.EPI_RESIDUAL, residual=A)
    arr = (dg.Linear * 1)(head)
    assert lib.dg_decode_step_weights(ctypes.cast(arr, ctypes.c_void_p), 1, A, 1 << 20,
                                      None) == INVALID
    # epilogue ops never split K: no split-K workspace is asked for them
    assert dg.workspace_bytes([_op(N=256, epilogue=dg.EPI_RESIDUAL, residual=A)]) == 256


def test_elementwise_conv1d_and_packer_validation(lib):
    assert lib.dg_swiglu(None, A, B, 8, None) == INVALID
    assert lib.dg_swiglu(A, A, B, 12, None) == MISALIGNED
    assert lib.dg_residual_add(A, ODD, B, 8, None) == MISALIGNED
    c = lib.dg_causal_conv1d_update
    assert c(None, B, A, None, 0x300000, 1, 16, 4, 1, None) == INVALID
    assert c(A, B, A, None, 0x300000, 1, 16, 4, 5, None) == INVALID     # act
    assert c(A, B, A, None, 0x300000, 1, 16, 9, 1, None) == UNSUPPORTED  # width
    assert c(A, B, A, None, 0x300000, 1, 12, 4, 1, None) == MISALIGNED   # C % 8
    assert c(A, B, A, ODD, 0x300000, 1, 16, 4, 1, None) == MISALIGNED    # bias
    assert c(A, B, A, None, B + 16, 1, 16, 4, 1, None) == INVALID        # y overlaps state
    assert lib.dg_quantize_weights_i8(A, B, A, 8, 24, None) == MISALIGNED
    assert lib.dg_quantize_weights_w4(A, B, A, 8, 96, 64, None) == UNSUPPORTED
    assert lib.dg_quantize_weights_w4(A, B, A + 1, 8, 64, 32, None) == MISALIGNED
