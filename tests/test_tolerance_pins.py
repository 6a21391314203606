"""Pins for the acceptance rules (oracle/tolerance.py), which every parity
test applies: the unit-in-the-last-place helpers against the spacing of
consecutive bit patterns (brute force over every fp16 and bf16 value, and
numpy's float32 spacing), both sides of the bound's edge, and the
greedy-token rule on planted gaps and near ties."""
import numpy as np
import pytest
import torch

from oracle import tolerance as tol


def _next_up_spacing16(bits_pos, decode):
    """Distance from each positive finite 16-bit pattern to the next one up."""
    v = decode(bits_pos)
    w = decode(bits_pos + 1)
    return v, w - v


def _f16(bits):
    return bits.astype(np.uint16).view(np.float16).astype(np.float64)


def _bf16(bits):
    t = torch.from_numpy(bits.astype(np.int32).astype(np.int16)).view(torch.bfloat16)
    return t.double().numpy()


def test_ulp_f16_is_the_gap_to_the_next_value_for_every_finite_fp16():
    bits = np.arange(0, 0x7BFF, dtype=np.int64)  # +0 .. the value below the largest finite
    v, gap = _next_up_spacing16(bits, _f16)
    assert np.array_equal(tol.ulp_f16(v), gap)
    assert np.array_equal(tol.ulp_f16(-v), gap)  # symmetric in sign


def test_ulp_bf16_is_the_gap_to_the_next_value_for_every_finite_bf16():
    bits = np.arange(0, 0x7F7F, dtype=np.int64)
    v, gap = _next_up_spacing16(bits, _bf16)
    assert np.array_equal(tol.ulp_bf16(v), gap)


def test_ulp_f32_matches_numpy_spacing():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(10000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-40).astype(np.float32),  # subnormals
        np.float32([0.0, 1.0, 2.0, 0.5, 3.0, 1e-38, 1.1754944e-38, 1e30]),
    ]).astype(np.float32)
    a = np.abs(vals)
    assert np.array_equal(tol.ulp_f32(a.astype(np.float64)), np.spacing(a).astype(np.float64))


def test_bound_edge_just_inside_passes_and_just_beyond_fails():
    y_ref = np.array([1.0, -3.5, 0.0, 1000.0])
    A = np.array([10.0, 7.0, 0.0, 5000.0])
    b = tol.bound(y_ref, A, "f16")
    assert np.allclose(b, 1e-3 * A + tol.ulp_f16(y_ref))
    # (y_ref + b) - y_ref is not exactly b in fp64: probe just inside and
    # just outside the edge
    assert not tol.violations(y_ref + b * (1 - 1e-9), y_ref, A, "f16").any()
    assert not tol.violations(y_ref - b * (1 - 1e-9), y_ref, A, "f16").any()
    assert tol.violations(y_ref + b * (1 + 1e-9), y_ref, A, "f16").all()
    assert tol.violations(y_ref - b * (1 + 1e-9), y_ref, A, "f16").all()
    with pytest.raises(AssertionError):
        tol.assert_close(y_ref + 2 * b + 1e-9, y_ref, A, "f16", "edge")
    # a sign error is far outside the bound whenever |y| is well above it
    assert tol.violations(np.array([-1.0]), np.array([1.0]), np.array([10.0]), "f16").all()


def test_argmax_rule_pins_clear_winners_and_accepts_only_near_ties():
    logits = np.array([0.0, 5.0, 1.0, 4.9999, 4.0])
    A = np.full(5, 1.0)  # bound per logit about 1e-3
    ok, pinned = tol.argmax_check(1, logits, A)
    assert ok and not pinned  # 5.0 vs 4.9999: within the two bounds, a near tie
    assert tol.argmax_check(3, logits, A)[0]  # the other near-tie candidate
    assert not tol.argmax_check(4, logits, A)[0]  # 1.0 below: not a candidate
    assert not tol.argmax_check(-1, logits, A)[0]
    assert not tol.argmax_check(5, logits, A)[0]
    wide = np.array([0.0, 5.0, 1.0, 4.0])
    ok, pinned = tol.argmax_check(1, wide, np.ones(4))
    assert ok and pinned
    ok, pinned = tol.argmax_check(3, wide, np.ones(4))
    assert not ok and pinned
    # exact ties: the lowest index is the oracle's choice and is pinned only
    # by the gap rule's failure; both tied indices are accepted
    tie = np.array([2.0, 7.0, 7.0, 1.0])
    assert tol.argmax_check(1, tie, np.zeros(4))[0]
    assert tol.argmax_check(2, tie, np.zeros(4))[0]
    assert not tol.argmax_check(0, tie, np.zeros(4))[0]


def test_silu_slope_constant_bounds_the_derivative_and_is_tight():
    v = np.linspace(-30, 30, 600001)
    s = 1 / (1 + np.exp(-v))
    d = s * (1 + v * (1 - s))
    assert np.max(np.abs(d)) <= tol.SILU_SLOPE
    assert np.max(np.abs(d)) > 1.09   # 1.0998...: a looser slope would hide errors


def test_silu_and_swiglu_bounds_cover_input_errors_at_their_edge():
    """Perturb the fp32 sums by exactly their own error budget (the worst
    case): the bounds still hold, and each term of the SwiGLU bound is
    needed somewhere."""
    rng = np.random.default_rng(5)
    n = 200000
    g = rng.normal(0, 3, n)
    u = rng.normal(0, 3, n)
    Ag = np.abs(g) * rng.uniform(1, 50, n)
    Au = np.abs(u) * rng.uniform(1, 50, n)
    eg = tol.REL * Ag + tol.ulp_f32(g)
    eu = tol.REL * Au + tol.ulp_f32(u)
    sg = rng.choice([-1.0, 1.0], n)
    su = rng.choice([-1.0, 1.0], n)
    silu = lambda t: t / (1 + np.exp(-t))
    h0 = silu(g) * u
    h1 = silu(g + sg * eg) * (u + su * eu)
    b = tol.bound_swiglu(g, u, Ag, Au, "f32")
    assert np.all(np.abs(h1 - h0) <= b)
    # dropping the |silu(g)| e_u term breaks it
    part = b - np.abs(silu(g)) * eu
    assert np.any(np.abs(h1 - h0) > part)
    # the silu bound
    bs = tol.bound_silu(g, Ag, "f32")
    assert np.all(np.abs(silu(g + sg * eg) - silu(g)) <= bs)
