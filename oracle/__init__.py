"""CPU oracle for the decode-step skinny GEMV paths.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA library (``quantized_skinny_gemm_gb300``)
and imports nothing from it; the two meet only through the seeded input
generators, which hold none of the method's arithmetic.

Every function is the plain definition of what the path computes, in fp64 (or
exact int64 for integer accumulators), summed in ascending k:

* ``gemv_fp``   -- y[m,n] = sum_k W[n,k] x[m,k] for fp16 / bf16 W and x.  The M=1
  vector-matrix product of the custom cube matmul in "MiniCPM-V on Orange Pi
  AIPro (Ascend 310B)" (paragraph on the custom M=1 cube matmul).
* ``lm_head`` / ``lm_head_split16`` -- logits of the wide vocabulary projection
  and the greedy token (largest logit, lowest index on exact ties); the split
  form cuts W into 16 equal row slices, takes each slice's best (value, index)
  and reduces those on the host, as the same post does for its ~248k-row
  lm_head (paragraph on the 16-slice lm_head split with a host reduce).
* ``gemv_w8a8`` -- "vLLM Arm CPU optimizations", section "INT8 W8A8": exact
  integer accumulation, then per-output-channel and per-token fp32 scales.
* ``gemv_w4a16`` / ``gemv_w4a8`` -- same page, section "INT8 W4A8", and the fused
  INT4 dequantization of the Orange Pi AIPro post's closing paragraph: explicit
  two's-complement nibble unpacking, one fp16 scale per group of 32 k.
* ``quant_act`` -- per-token symmetric int8 quantization of the activations for
  W8A8 / W4A8, decided in IEEE fp32.
* ``quant_w8`` / ``quant_w4`` / ``dequant_w4`` -- weight quantizers (per-channel
  int8, groupwise int4), the definitions the load-time packers must reproduce
  bit for bit ("vLLM Arm CPU optimizations", section "Dense layer weight
  prepacking": weights are put in the kernel's format once, at warm-up).
* ``silu`` / ``gemv_swiglu_*`` / ``gemv_residual_*`` -- the epilogues a decoder
  applies right after the weight stream (SwiGLU after gate|up, a residual add
  after o and down); the pages only motivate removing the extra launches
  around the stream (EdgeFM, section 2.C, graph-accelerated decode), so the
  definitions are the plain ones: silu(v) = v / (1 + e^-v), h = silu(g) * u,
  y = r + W x.
* ``causal_conv1d_update`` -- one decode step of a depthwise causal 1-D
  convolution over a rolling window ("MiniCPM-V on Orange Pi AIPro": the scalar
  causal-conv1d baseline that became a vectorized step kernel): per channel c,
  v = b[c] + sum_j w[c][j] u[j], u = the channel's last W-1 inputs (oldest
  first) followed by the new input; y = v or silu(v); the window then drops
  its oldest input and appends the new one.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, closed forms, library special cases, invariants, hand-written
fixtures under ``tests/golden/``).  Nothing here is "parity unpinned".
"""
import ctypes
import os

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build()
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.orc_f16_to_f64.restype = ctypes.c_double
    lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_f64.restype = ctypes.c_double
    lib.orc_decode_f16.argtypes = [P, I64, P]
    lib.orc_decode_bf16.argtypes = [P, I64, P]
    lib.orc_unpack_w4.argtypes = [P, I64, P]
    lib.orc_pack_w4.argtypes = [P, I64, P]
    lib.orc_pack_w4.restype = I
    lib.orc_argmax.argtypes = [P, I64]
    lib.orc_argmax.restype = I64
    lib.orc_gemv_fp.argtypes = [P, P, I, I64, I64, I64, P, I64, P, P, I]
    lib.orc_gemv_fp.restype = I
    lib.orc_gemv_w8a8.argtypes = [P, P, P, P, I64, I64, I64, P, I64, P, P, P, I]
    lib.orc_gemv_w8a8.restype = I
    lib.orc_gemv_w4.argtypes = [P, P, I64, P, P, P, I64, I64, I64, P, I64, P, P, P, I]
    lib.orc_gemv_w4.restype = I
    lib.orc_quant_act.argtypes = [P, I64, I64, P, P]
    lib.orc_quant_act.restype = I
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _bits16(a):
    """fp16 / bf16 payload as uint16 bits.  Accepts numpy float16 or uint16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype in (np.uint16, np.int16):
        return a.view(np.uint16)
    raise TypeError("expected float16 or uint16 bits, got %s" % a.dtype)


def _rows(rows, N):
    if rows is None:
        return None, N
    r = _c(rows, np.int64).reshape(-1)
    return r, r.size


def _check(rc, what):
    if rc != 0:
        raise ValueError("oracle %s rejected its arguments (code %d)" % (what, rc))


# ---- decoding / packing ----------------------------------------------------

def decode_f16(bits):
    b = _bits16(bits).reshape(-1)
    out = np.empty(b.size, np.float64)
    _load().orc_decode_f16(_ptr(b), b.size, _ptr(out))
    return out.reshape(np.shape(bits))


def decode_bf16(bits):
    b = _bits16(bits).reshape(-1)
    out = np.empty(b.size, np.float64)
    _load().orc_decode_bf16(_ptr(b), b.size, _ptr(out))
    return out.reshape(np.shape(bits))


def unpack_w4(packed):
    """uint8 [..., K/2] -> int8 codes [..., K] (k = 2j in bits 0-3, 2j+1 in 4-7)."""
    p = _c(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.int8)
    _load().orc_unpack_w4(_ptr(p), p.size, _ptr(out))
    return out


def pack_w4(codes):
    c = _c(codes, np.int8)
    out = np.empty(c.shape[:-1] + (c.shape[-1] // 2,), np.uint8)
    _check(_load().orc_pack_w4(_ptr(c), c.size, _ptr(out)), "pack_w4")
    return out


def argmax(v):
    """Largest value, lowest index on exact ties; NaN never wins."""
    a = _c(v, np.float64).reshape(-1)
    return int(_load().orc_argmax(_ptr(a), a.size))


# ---- GEMV definitions ------------------------------------------------------

def gemv_fp(W, x, fmt="f16", rows=None, nthreads=0):
    """y[M][nrows], A[M][nrows] in fp64 for fp16/bf16 bits W [N][K], x [M][K]."""
    Wb, xb = _bits16(W), _bits16(x)
    N, K = Wb.shape
    xb = xb.reshape(-1, K)
    M = xb.shape[0]
    r, nr = _rows(rows, N)
    y = np.empty((M, nr), np.float64)
    A = np.empty((M, nr), np.float64)
    rc = _load().orc_gemv_fp(_ptr(Wb), _ptr(xb), {"f16": 0, "bf16": 1}[fmt], M, N, K,
                             _ptr(r), nr, _ptr(y), _ptr(A), nthreads)
    _check(rc, "gemv_fp")
    return y, A


def lm_head(W, x, fmt="f16", nthreads=0):
    """(logits [N] fp64, A [N], token) for M = 1."""
    y, A = gemv_fp(W, x, fmt, nthreads=nthreads)
    return y[0], A[0], argmax(y[0])


def lm_head_split16(W, x, fmt="f16", nslices=16, nthreads=0):
    """The 16-slice form: each slice of N/16 consecutive rows is an independent
    product with its own (best value, local index); the host then picks the
    best slice result, converting local to global indices, lowest global index
    on exact ties.  Returns (logits [N], token)."""
    Wb = _bits16(W)
    N = Wb.shape[0]
    if N % nslices:
        raise ValueError("N=%d is not a multiple of %d slices" % (N, nslices))
    rows_per = N // nslices
    logits = np.empty(N, np.float64)
    best_v, best_i = None, -1
    for s in range(nslices):
        lo = s * rows_per
        ys, _ = gemv_fp(Wb[lo:lo + rows_per], x, fmt, nthreads=nthreads)
        logits[lo:lo + rows_per] = ys[0]
        li = argmax(ys[0])
        if li < 0:
            continue
        v, gi = ys[0][li], lo + li
        if best_i < 0 or v > best_v or (v == best_v and gi < best_i):
            best_v, best_i = v, gi
    return logits, best_i


def gemv_w8a8(W, s_w, xq, s_x, rows=None, nthreads=0):
    """(acc int64 [M][nrows], y fp64, A fp64)."""
    Wc = _c(W, np.int8)
    N, K = Wc.shape
    xc = _c(xq, np.int8).reshape(-1, K)
    M = xc.shape[0]
    sw, sx = _c(s_w, np.float32).reshape(-1), _c(s_x, np.float32).reshape(-1)
    r, nr = _rows(rows, N)
    acc = np.empty((M, nr), np.int64)
    y = np.empty((M, nr), np.float64)
    A = np.empty((M, nr), np.float64)
    rc = _load().orc_gemv_w8a8(_ptr(Wc), _ptr(sw), _ptr(xc), _ptr(sx), M, N, K, _ptr(r), nr,
                               _ptr(acc), _ptr(y), _ptr(A), nthreads)
    _check(rc, "gemv_w8a8")
    return acc, y, A


def gemv_w4a16(Wq, scales, x, group=32, rows=None, nthreads=0):
    """(y fp64 [M][nrows], A)."""
    Wc = _c(Wq, np.uint8)
    N, K2 = Wc.shape
    K = 2 * K2
    sc = _bits16(scales).reshape(N, K // group)
    xb = _bits16(x).reshape(-1, K)
    M = xb.shape[0]
    r, nr = _rows(rows, N)
    y = np.empty((M, nr), np.float64)
    A = np.empty((M, nr), np.float64)
    rc = _load().orc_gemv_w4(_ptr(Wc), _ptr(sc), group, _ptr(xb), None, None, M, N, K,
                             _ptr(r), nr, _ptr(y), _ptr(A), None, nthreads)
    _check(rc, "gemv_w4a16")
    return y, A


def gemv_w4a8(Wq, scales, xq, s_x, group=32, rows=None, nthreads=0):
    """(y fp64 [M][nrows], A, acc_groups int64 [M][nrows][K/group])."""
    Wc = _c(Wq, np.uint8)
    N, K2 = Wc.shape
    K = 2 * K2
    sc = _bits16(scales).reshape(N, K // group)
    xc = _c(xq, np.int8).reshape(-1, K)
    M = xc.shape[0]
    sx = _c(s_x, np.float32).reshape(-1)
    r, nr = _rows(rows, N)
    y = np.empty((M, nr), np.float64)
    A = np.empty((M, nr), np.float64)
    accg = np.empty((M, nr, K // group), np.int64)
    rc = _load().orc_gemv_w4(_ptr(Wc), _ptr(sc), group, None, _ptr(xc), _ptr(sx), M, N, K,
                             _ptr(r), nr, _ptr(y), _ptr(A), _ptr(accg), nthreads)
    _check(rc, "gemv_w4a8")
    return y, A, accg


# ---- quantizers ------------------------------------------------------------

def quant_act(x):
    """Per-token int8: s = amax/127 (fp32), q = clamp(rne(x/s), -127, 127)."""
    xb = _bits16(x)
    K = xb.shape[-1]
    xb = xb.reshape(-1, K)
    M = xb.shape[0]
    q = np.empty((M, K), np.int8)
    s = np.empty(M, np.float32)
    _check(_load().orc_quant_act(_ptr(xb), M, K, _ptr(q), _ptr(s)), "quant_act")
    return q, s


def quant_w8(w):
    """Per-output-channel int8 weights, decided in fp32:
    s[n] = max_k |w[n,k]| / 127, q = clamp(rne(w/s), -127, 127); s = 1 for a zero row."""
    w32 = np.asarray(w, np.float32)
    amax = np.max(np.abs(w32), axis=1)
    s = np.where(amax > 0, amax / np.float32(127), np.float32(1)).astype(np.float32)
    q = np.clip(np.rint(w32 / s[:, None]), -127, 127).astype(np.int8)
    return q, s


def quant_w4(w, group=32):
    """Groupwise symmetric int4, decided in fp32 with an fp16 scale:
    s = fp16(max_g |w| / 7) (1 for an all-zero group, at least the smallest fp16
    subnormal otherwise), q = clamp(rne(w / s), -7, 7).  Returns (codes, scales f16)."""
    w32 = np.asarray(w, np.float32)
    N, K = w32.shape
    g = w32.reshape(N, K // group, group)
    amax = np.max(np.abs(g), axis=2)
    s16 = (amax / np.float32(7)).astype(np.float16)
    s16 = np.where(amax > 0, np.maximum(s16, np.float16(2.0 ** -24)), np.float16(1))
    s16 = s16.astype(np.float16)
    q = np.clip(np.rint(g / s16.astype(np.float32)[:, :, None]), -7, 7).astype(np.int8)
    return q.reshape(N, K), s16


def dequant_w4(codes, scales, group=32):
    """fp64 weights codes * scale of their group."""
    c = np.asarray(codes, np.float64)
    N, K = c.shape
    s = decode_f16(_bits16(scales)).reshape(N, K // group)
    return (c.reshape(N, K // group, group) * s[:, :, None]).reshape(N, K)


# ---- epilogues and the causal-conv1d decode step -----------------------------

def silu(v):
    """v / (1 + exp(-v)) in fp64 (v * sigmoid(v))."""
    v = np.asarray(v, np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def gemv_swiglu_fp(Wg, Wu, x, fmt="f16", rows=None, nthreads=0):
    """h = silu(Wg x) * (Wu x) per row, from the exact fp64 products.
    Returns (h, g, u, A_g, A_u), each [M][nrows]."""
    g, Ag = gemv_fp(Wg, x, fmt, rows=rows, nthreads=nthreads)
    u, Au = gemv_fp(Wu, x, fmt, rows=rows, nthreads=nthreads)
    return silu(g) * u, g, u, Ag, Au


def gemv_swiglu_w4a16(Wg, Sg, Wu, Su, x, group=32, rows=None, nthreads=0):
    g, Ag = gemv_w4a16(Wg, Sg, x, group, rows=rows, nthreads=nthreads)
    u, Au = gemv_w4a16(Wu, Su, x, group, rows=rows, nthreads=nthreads)
    return silu(g) * u, g, u, Ag, Au


def gemv_swiglu_w4a8(Wg, Sg, Wu, Su, xq, s_x, group=32, rows=None, nthreads=0):
    g, Ag, _ = gemv_w4a8(Wg, Sg, xq, s_x, group, rows=rows, nthreads=nthreads)
    u, Au, _ = gemv_w4a8(Wu, Su, xq, s_x, group, rows=rows, nthreads=nthreads)
    return silu(g) * u, g, u, Ag, Au


def gemv_residual_fp(W, x, r, fmt="f16", rows=None, nthreads=0):
    """y = r + W x (r fp16 / bf16 [M][N]); returns (y, A) with A = sum |w x|."""
    y, A = gemv_fp(W, x, fmt, rows=rows, nthreads=nthreads)
    rb = (decode_bf16 if fmt == "bf16" else decode_f16)(_bits16(r)).reshape(y.shape[0], -1)
    if rows is not None:
        rb = rb[:, _c(rows, np.int64)]
    return rb + y, A


def gemv_residual_w4a16(Wq, scales, x, r, group=32, rows=None, nthreads=0):
    y, A = gemv_w4a16(Wq, scales, x, group, rows=rows, nthreads=nthreads)
    rb = decode_f16(_bits16(r)).reshape(y.shape[0], -1)
    if rows is not None:
        rb = rb[:, _c(rows, np.int64)]
    return rb + y, A


def causal_conv1d_update(x, state, w, bias=None, act="silu"):
    """One decode step of a depthwise causal conv1d.

    x fp16 bits [M][C] (the new input), state fp16 bits [M][C][W-1] (each
    channel's last W-1 inputs, oldest first), w fp16 bits [C][W] (tap j
    multiplies window position j, position W-1 being the new input), bias fp16
    bits [C] or None, act "silu" or "none".
    Returns (y [M][C] fp64, v [M][C] the pre-activation sum, A [M][C] =
    |b| + sum_j |w_j u_j|, new_state fp16 bits [M][C][W-1]).  The sum runs in
    fp64 over j ascending, after the bias."""
    xb = _bits16(x)
    C = xb.shape[-1]
    xb = xb.reshape(-1, C)
    M = xb.shape[0]
    wb = _bits16(w).reshape(C, -1)
    Wd = wb.shape[1]
    sb = _bits16(state).reshape(M, C, Wd - 1)
    wv = decode_f16(wb).reshape(C, Wd)
    u = np.concatenate([decode_f16(sb).reshape(M, C, Wd - 1),
                        decode_f16(xb).reshape(M, C, 1)], axis=2)
    bv = decode_f16(_bits16(bias)).reshape(C) if bias is not None else np.zeros(C)
    v = np.empty((M, C))
    A = np.empty((M, C))
    for m in range(M):
        acc = bv.copy()
        aa = np.abs(bv)
        for j in range(Wd):
            t = wv[:, j] * u[m, :, j]
            acc = acc + t
            aa = aa + np.abs(t)
        v[m] = acc
        A[m] = aa
    y = silu(v) if act == "silu" else v
    new_state = np.concatenate([sb[:, :, 1:], xb.reshape(M, C, 1)], axis=2)
    return y, v, A, new_state
