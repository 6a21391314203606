"""Python binding of libdg.so, the sm_103a decode-step skinny GEMV library.

Argument marshalling only: every function takes torch CUDA tensors, passes
their device pointers, shapes and the current CUDA stream to the C entry point
of the same name (``dg_<name>`` in include/dg.h) and raises ``DGError`` when it
returns a status other than DG_OK.  All arithmetic runs in the library's
kernels; there is no fallback of any kind, and using a function without the
built library raises.
"""
import ctypes
import os

__all__ = [
    "DGError", "Linear", "StepPlan", "F16", "BF16", "LINEAR_F16", "LINEAR_BF16",
    "LINEAR_W8A8", "LINEAR_W4A16", "LINEAR_W4A8", "gemv_f16", "gemv_w8a8", "gemv_w4",
    "quantize_act_i8", "lm_head_argmax", "lm_head_argmax_noalloc", "decode_step_weights", "workspace_bytes",
    "EPI_NONE", "EPI_RESIDUAL", "EPI_SWIGLU", "ACT_NONE", "ACT_SILU", "linear_forward", "swiglu",
    "residual_add", "causal_conv1d_update", "quantize_weights_i8", "quantize_weights_w4",
    "check_device_status", "selftest_wait_timeout", "status_string", "probe_copy", "probe_read", "version",
    "library_path", "load",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libdg.so")

F16, BF16 = 0, 1
LINEAR_F16, LINEAR_BF16, LINEAR_W8A8, LINEAR_W4A16, LINEAR_W4A8 = range(5)
EPI_NONE, EPI_RESIDUAL, EPI_SWIGLU = range(3)
ACT_NONE, ACT_SILU = range(2)
_STATUS = ["DG_OK", "DG_ERR_INVALID_ARG", "DG_ERR_UNSUPPORTED", "DG_ERR_MISALIGNED",
           "DG_ERR_WORKSPACE", "DG_ERR_CUDA", "DG_ERR_TIMEOUT"]


class DGError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        name = _STATUS[status] if 0 <= status < len(_STATUS) else str(status)
        super().__init__("%s returned %s" % (where, name))


class Linear(ctypes.Structure):
    """Mirror of the C struct dg_linear."""
    _fields_ = [
        ("kind", ctypes.c_int32), ("M", ctypes.c_int32), ("N", ctypes.c_int32),
        ("K", ctypes.c_int32), ("group_size", ctypes.c_int32),
        ("W", ctypes.c_void_p), ("w_scale", ctypes.c_void_p), ("x", ctypes.c_void_p),
        ("x_i8", ctypes.c_void_p), ("x_scale", ctypes.c_void_p), ("y", ctypes.c_void_p),
        ("logits", ctypes.c_void_p), ("token", ctypes.c_void_p), ("acc_out", ctypes.c_void_p),
        ("epilogue", ctypes.c_int32), ("reserved", ctypes.c_int32), ("residual", ctypes.c_void_p),
        ("W2", ctypes.c_void_p), ("w2_scale", ctypes.c_void_p),
    ]


_lib = None


def library_path():
    return _LIB_PATH


def load():
    """Loads libdg.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError("libdg.so is not built (%s); run __graft_entry__.build()" % _LIB_PATH)
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "dg_gemv_f16": [P, P, P, I, I, I, I, P, Z, P],
        "dg_gemv_w8a8": [P, P, P, P, P, P, I, I, I, P, Z, P],
        "dg_gemv_w4": [P, P, I, P, P, P, P, I, I, I, P, Z, P],
        "dg_quantize_act_i8": [P, P, P, I, I, P],
        "dg_lm_head_argmax": [P, P, Z, P],
        "dg_lm_head_argmax_noalloc": [P, P],
        "dg_decode_step_weights": [P, I, P, Z, P],
        "dg_check_device_status": [P],
        "dg_selftest_wait_timeout": [ctypes.c_uint, P],
        "dg_probe_copy": [P, P, Z, P],
        "dg_linear_forward": [P, P, Z, P],
        "dg_swiglu": [P, P, P, I, P],
        "dg_residual_add": [P, P, P, I, P],
        "dg_causal_conv1d_update": [P, P, P, P, P, I, I, I, I, P],
        "dg_quantize_weights_i8": [P, P, P, I, I, P],
        "dg_quantize_weights_w4": [P, P, P, I, I, I, P],
        "dg_probe_read": [P, Z, P, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.dg_workspace_bytes.argtypes = [P, I]
    lib.dg_workspace_bytes.restype = Z
    lib.dg_status_string.argtypes = [I]
    lib.dg_status_string.restype = ctypes.c_char_p
    lib.dg_version.argtypes = []
    lib.dg_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _call(name, *args):
    st = getattr(load(), name)(*args)
    if st != 0:
        raise DGError(st, name)


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


# ---- entry points ----------------------------------------------------------------

def gemv_f16(W, x, y, dtype=F16, ws=None, stream=None):
    """y[M][N] = x[M][K] . W[N][K]^T for fp16 (dtype=F16) or bf16 (BF16) tensors."""
    N, K = W.shape
    M = x.numel() // K
    _call("dg_gemv_f16", _ptr(W), _ptr(x), _ptr(y), dtype, M, N, K, _ptr(ws), _nbytes(ws),
          _stream(stream))


def gemv_w8a8(W, w_scale, x_i8, x_scale, y=None, acc_out=None, ws=None, stream=None):
    N, K = W.shape
    M = x_i8.numel() // K
    _call("dg_gemv_w8a8", _ptr(W), _ptr(w_scale), _ptr(x_i8), _ptr(x_scale), _ptr(y),
          _ptr(acc_out), M, N, K, _ptr(ws), _nbytes(ws), _stream(stream))


def gemv_w4(Wq, scales, y, x_f16=None, x_i8=None, x_scale=None, group_size=32, ws=None,
            stream=None):
    """W4A16 when x_i8 is None, W4A8 otherwise.  Wq uint8 [N][K/2]."""
    N, K2 = Wq.shape
    K = 2 * K2
    xa = x_i8 if x_i8 is not None else x_f16
    M = xa.numel() // K
    _call("dg_gemv_w4", _ptr(Wq), _ptr(scales), group_size, _ptr(x_f16), _ptr(x_i8),
          _ptr(x_scale), _ptr(y), M, N, K, _ptr(ws), _nbytes(ws), _stream(stream))


def quantize_act_i8(x, xq, x_scale, stream=None):
    K = x.shape[-1]
    M = x.numel() // K
    _call("dg_quantize_act_i8", _ptr(x), _ptr(xq), _ptr(x_scale), M, K, _stream(stream))


def linear(kind, W, M, N, K, w_scale=None, x=None, x_i8=None, x_scale=None, y=None,
           logits=None, token=None, acc_out=None, group_size=32, epilogue=EPI_NONE,
           residual=None, W2=None, w2_scale=None):
    """Builds a Linear descriptor from tensors (pointers only; keep the tensors alive)."""
    return Linear(kind, M, N, K, group_size, _ptr(W), _ptr(w_scale), _ptr(x), _ptr(x_i8),
                  _ptr(x_scale), _ptr(y), _ptr(logits), _ptr(token), _ptr(acc_out), epilogue, 0,
                  _ptr(residual), _ptr(W2), _ptr(w2_scale))


def linear_forward(op, ws=None, stream=None):
    """Runs one op described by a Linear (any kind but an lm_head; any epilogue)."""
    _call("dg_linear_forward", ctypes.byref(op), _ptr(ws), _nbytes(ws), _stream(stream))


def swiglu(g, u, h, stream=None):
    """h = silu(g) * u elementwise (fp16)."""
    _call("dg_swiglu", _ptr(g), _ptr(u), _ptr(h), g.numel(), _stream(stream))


def residual_add(a, b, out, stream=None):
    """out = a + b elementwise (fp16)."""
    _call("dg_residual_add", _ptr(a), _ptr(b), _ptr(out), a.numel(), _stream(stream))


def causal_conv1d_update(x, state, w, y, bias=None, act=ACT_SILU, stream=None):
    """One causal-conv1d decode step: x [M][C], state [M][C][W-1] (updated in
    place), w [C][W], bias [C] or None, y [M][C]; all fp16."""
    C, width = w.shape
    M = x.numel() // C
    _call("dg_causal_conv1d_update", _ptr(x), _ptr(state), _ptr(w), _ptr(bias), _ptr(y), M, C,
          width, act, _stream(stream))


def quantize_weights_i8(W, Wq, w_scale, stream=None):
    """fp16 W [N][K] -> int8 Wq [N][K] + fp32 per-row scales (load-time packer)."""
    N, K = W.shape
    _call("dg_quantize_weights_i8", _ptr(W), _ptr(Wq), _ptr(w_scale), N, K, _stream(stream))


def quantize_weights_w4(W, Wq, scales, group_size=32, stream=None):
    """fp16 W [N][K] -> packed int4 Wq [N][K/2] + fp16 scales [N][K/group] (load-time packer)."""
    N, K = W.shape
    _call("dg_quantize_weights_w4", _ptr(W), _ptr(Wq), _ptr(scales), N, K, group_size,
          _stream(stream))


def lm_head_argmax(head, ws, stream=None):
    _call("dg_lm_head_argmax", ctypes.byref(head), _ptr(ws), _nbytes(ws), _stream(stream))


def lm_head_argmax_noalloc(head, stream=None):
    """lm_head + argmax with the library's own fixed scratch (no workspace)."""
    _call("dg_lm_head_argmax_noalloc", ctypes.byref(head), _stream(stream))


class StepPlan:
    """A decode step's ops, marshalled once into a C array of dg_linear."""

    def __init__(self, ops, keep=()):
        self.n = len(ops)
        self.array = (Linear * self.n)(*ops)
        self.keep = list(keep)  # tensors the descriptors point into

    def workspace_bytes(self):
        return int(load().dg_workspace_bytes(ctypes.cast(self.array, ctypes.c_void_p), self.n))


def decode_step_weights(plan, ws=None, stream=None):
    _call("dg_decode_step_weights", ctypes.cast(plan.array, ctypes.c_void_p), plan.n, _ptr(ws),
          _nbytes(ws), _stream(stream))


def workspace_bytes(ops):
    arr = (Linear * len(ops))(*ops)
    return int(load().dg_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), len(ops)))


def check_device_status(stream=None):
    _call("dg_check_device_status", _stream(stream))


def selftest_wait_timeout(spin_limit, stream=None):
    """Launches the bounded-wait self test (see include/dg.h)."""
    _call("dg_selftest_wait_timeout", spin_limit, _stream(stream))


def status_string(s):
    return load().dg_status_string(s).decode()


def probe_copy(src, dst, stream=None):
    _call("dg_probe_copy", _ptr(src), _ptr(dst), _nbytes(src), _stream(stream))


def probe_read(src, sink, stream=None):
    _call("dg_probe_read", _ptr(src), _nbytes(src), _ptr(sink), _stream(stream))


def version():
    return load().dg_version().decode()
