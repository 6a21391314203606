"""Acceptance rules for comparing the CUDA library against the oracle.

TEST INFRASTRUCTURE ONLY (same import rule as the rest of ``oracle/``).

Floating-point outputs:   |y - y_ref| <= 1e-3 * A + ulp_out(y_ref)
  where A = sum_k |w_k x_k| of the dequantized operands (returned by the oracle)
  and ulp_out is the spacing of the output type at |y_ref|: fp16 2^(e-10) for
  normal values and 2^-24 below 2^-14; fp32 2^(e-23) and 2^-149.  The 1e-3
  relative budget covers fp32 accumulation of up to ~10^5 exact products
  (bounded by K * 2^-24 * A) and, for int4 x fp16, fp32 group sums; the ulp
  term covers the final rounding to the output type.
Integer outputs (int32 accumulators, int8 codes, quantization scales): exact.
Greedy argmax: with b_i = 1e-3 * A_i + ulp_f32(logit_i), the token must equal
  the oracle's when its top-1 beats top-2 by more than b_top1 + b_top2;
  otherwise it must be a near-tie candidate: ref[token] >= v1 - b_top1 - b_token.
"""
import numpy as np

REL = 1e-3


def _ulp(v, mant_bits, min_exp, sub_exp):
    a = np.abs(np.asarray(v, np.float64))
    _, E = np.frexp(a)          # a = f * 2^E, f in [0.5, 1)
    e = np.maximum(E - 1, min_exp)
    u = np.ldexp(1.0, e - mant_bits)
    return np.where(a == 0, np.ldexp(1.0, sub_exp), u)


def ulp_f16(v):
    return _ulp(v, 10, -14, -24)


def ulp_bf16(v):
    return _ulp(v, 7, -126, -133)


def ulp_f32(v):
    return _ulp(v, 23, -126, -149)


_ULP = {"f16": ulp_f16, "bf16": ulp_bf16, "f32": ulp_f32}


def bound(y_ref, A, out="f16"):
    return REL * np.asarray(A, np.float64) + _ULP[out](y_ref)


def violations(y, y_ref, A, out="f16"):
    """Boolean mask of elements outside the bound."""
    y = np.asarray(y, np.float64)
    err = np.abs(y - np.asarray(y_ref, np.float64))
    return ~(err <= bound(y_ref, A, out))


def assert_close(y, y_ref, A, out="f16", what=""):
    bad = violations(y, y_ref, A, out)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        y = np.asarray(y, np.float64)
        yr = np.asarray(y_ref, np.float64)
        det = ["%s: y=%r ref=%r bound=%r" % (tuple(i), y[tuple(i)], yr[tuple(i)],
                                              bound(yr[tuple(i)], np.asarray(A)[tuple(i)], out))
               for i in idx]
        raise AssertionError("%s: %d of %d outside tolerance; first: %s"
                             % (what, int(bad.sum()), bad.size, "; ".join(det)))


def argmax_check(token, logits_ref, A_ref):
    """Returns (ok, pinned): pinned is True when the gap rule forces equality."""
    v = np.asarray(logits_ref, np.float64)
    A = np.asarray(A_ref, np.float64)
    i1 = int(np.argmax(v))  # numpy: first index of the maximum
    rest = v.copy()
    rest[i1] = -np.inf
    i2 = int(np.argmax(rest))
    b = REL * A + ulp_f32(v)
    pinned = v[i1] - v[i2] > b[i1] + b[i2]
    if pinned:
        return token == i1, True
    if not (0 <= token < v.size):
        return False, False
    return bool(v[token] >= v[i1] - b[i1] - b[token]), False
