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
Epilogues evaluated in fp32 by the kernel after its fp32 sums (SiLU with the
  library exp, a product, a sum with the residual) carry the sums' error
  through the function: with e = 1e-3 * A + ulp_f32(v) for an fp32 sum v and
  |silu'| <= 1.1 everywhere,
    silu(v):        1.1 e + 2^-20 |silu(v)| + ulp_out
    silu(g) * u:    1.1 e_g |u| + |silu(g)| e_u + 1.1 e_g e_u + 2^-20 |h| + ulp_out
  where 2^-20 relative covers the fp32 evaluation of the function (a few
  fp32 roundings and the library exp).  A residual add y = r + W x is a sum
  with one more exact term: the plain bound with A = sum |w x|.
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


ACT_REL = 2.0 ** -20
SILU_SLOPE = 1.1   # max |d/dv (v sigmoid(v))| = 1.0998...


def _silu(v):
    v = np.asarray(v, np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def bound_silu(v_ref, A, out="f16"):
    """Bound for y = silu(v) where the kernel's fp32 sum v errs by 1e-3 A."""
    v = np.asarray(v_ref, np.float64)
    e = REL * np.asarray(A, np.float64) + ulp_f32(v)
    y = _silu(v)
    return SILU_SLOPE * e + ACT_REL * np.abs(y) + _ULP[out](y)


def bound_swiglu(g_ref, u_ref, A_g, A_u, out="f16"):
    """Bound for h = silu(g) * u from two fp32 sums g, u."""
    g = np.asarray(g_ref, np.float64)
    u = np.asarray(u_ref, np.float64)
    eg = REL * np.asarray(A_g, np.float64) + ulp_f32(g)
    eu = REL * np.asarray(A_u, np.float64) + ulp_f32(u)
    h = _silu(g) * u
    return (SILU_SLOPE * eg * np.abs(u) + np.abs(_silu(g)) * eu + SILU_SLOPE * eg * eu
            + ACT_REL * np.abs(h) + _ULP[out](h))


def assert_within(y, y_ref, bnd, what=""):
    """|y - y_ref| <= bnd elementwise (an explicit bound array)."""
    y = np.asarray(y, np.float64)
    yr = np.asarray(y_ref, np.float64)
    bad = ~(np.abs(y - yr) <= np.asarray(bnd, np.float64))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        det = ["%s: y=%r ref=%r bound=%r" % (tuple(i), y[tuple(i)], yr[tuple(i)],
                                              np.asarray(bnd)[tuple(i)]) for i in idx]
        raise AssertionError("%s: %d of %d outside tolerance; first: %s"
                             % (what, int(bad.sum()), bad.size, "; ".join(det)))
