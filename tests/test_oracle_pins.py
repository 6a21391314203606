"""Pins for the CPU oracle, checked against things other than itself.

Each pin is one of: a hand-worked fixture under tests/golden (with its
citation), exact rational brute force on tiny shapes, a closed form (identity,
one-hot, all-ones rows), a library special case (numpy / torch decoding,
numpy int64 matmul, numpy fp64 matmul on dequantized weights), an invariant
(16-slice split with host reduce, thread-count independence, row subsets), or
a rounding bound of a quantizer.  Shapes are non-square and scales distinct per
row / group so that a transposed operand, a wrong index, a dropped term or a
wrong sign fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f16(a):
    return np.asarray(a, np.float16)


# ---- decoding ---------------------------------------------------------------

def test_f16_decode_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode_f16(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_matches_torch_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ---- int4 nibble layout -------------------------------------------------------

def test_nibble_decode_hand_fixture():
    g = golden("w4_nibble_decode.json")
    for byte, lo, hi in g["cases"]:
        codes = oracle.unpack_w4(np.array([[byte]], np.uint8))
        assert codes.tolist() == [[lo, hi]], (byte, codes)


def test_pack_unpack_roundtrip_all_bytes_and_codes():
    b = np.arange(256, dtype=np.uint8).reshape(1, 256)
    codes = oracle.unpack_w4(b)
    assert codes.min() == -8 and codes.max() == 7
    assert np.array_equal(oracle.pack_w4(codes), b)
    lo, hi = np.meshgrid(np.arange(-8, 8), np.arange(-8, 8), indexing="ij")
    c = np.stack([lo.ravel(), hi.ravel()], axis=1).reshape(1, -1).astype(np.int8)
    assert np.array_equal(oracle.unpack_w4(oracle.pack_w4(c)), c)


def test_pack_rejects_out_of_range_code():
    with pytest.raises(ValueError):
        oracle.pack_w4(np.array([[8, 0]], np.int8))


# ---- hand-worked GEMV fixtures ------------------------------------------------

def test_fp16_gemv_hand_fixture():
    g = golden("gemv_tiny.json")["fp16"]
    y, A = oracle.gemv_fp(f16(g["W"]), f16(g["x"]))
    assert y.tolist() == g["y"] and A.tolist() == g["A"]


def test_w8a8_hand_fixture():
    g = golden("gemv_tiny.json")["w8a8"]
    acc, y, A = oracle.gemv_w8a8(np.array(g["W"], np.int8), g["s_w"],
                                 np.array(g["xq"], np.int8), g["s_x"])
    assert acc.tolist() == g["acc"]
    assert y.tolist() == g["y"] and A.tolist() == g["A"]


def _w4_fixture_rows(g):
    rows = []
    for a, b in g["row_bytes"]:
        rows.append([a] * 16 + [b] * 16)
    return np.array(rows, np.uint8)


def test_w4a16_hand_fixture():
    g = golden("gemv_tiny.json")["w4"]
    Wq = _w4_fixture_rows(g)
    sc = f16(g["scales"])
    y, A = oracle.gemv_w4a16(Wq, sc, f16(np.ones((1, 64))), group=32)
    assert y.tolist() == g["x_ones"]["y"] and A.tolist() == g["x_ones"]["A"]
    y, A = oracle.gemv_w4a16(Wq, sc, f16(np.arange(64).reshape(1, 64)), group=32)
    assert y.tolist() == g["x_index"]["y"] and A.tolist() == g["x_index"]["A"]


def test_w4a8_hand_fixture():
    g = golden("gemv_tiny.json")["w4"]
    t = g["w4a8_twos"]
    y, A, accg = oracle.gemv_w4a8(_w4_fixture_rows(g), f16(g["scales"]),
                                  np.full((1, 64), 2, np.int8), [t["s_x"]], group=32)
    assert accg.tolist() == t["acc_groups"]
    assert y.tolist() == t["y"] and A.tolist() == t["A"]


# ---- quantizers -----------------------------------------------------------------

def test_quant_act_hand_fixture():
    for case in golden("quant_act_cases.json")["cases"]:
        q, s = oracle.quant_act(f16(case["x"]))
        assert q.tolist() == case["q"], case
        for got, frac in zip(s, case["s"]):
            num, den = frac.split("/")
            assert got == np.float32(num) / np.float32(den), (case, got)


def test_quant_act_rounding_bound_and_extremes():
    rng = np.random.default_rng(1)
    x = f16(rng.standard_normal((5, 4096)) * np.array([[1], [3], [0.01], [100], [1e-3]]))
    q, s = oracle.quant_act(x)
    xf = x.astype(np.float64)
    assert np.all(np.abs(q.astype(np.int64)) <= 127)
    for m in range(x.shape[0]):
        err = np.abs(q[m].astype(np.float64) * float(s[m]) - xf[m])
        assert np.all(err <= float(s[m]) * (0.5 + 1e-6)), m  # nearest code
        k = int(np.argmax(np.abs(xf[m])))
        assert abs(int(q[m, k])) == 127  # the largest magnitude maps to the end code


def test_quant_w8_roundtrip_and_bound():
    rng = np.random.default_rng(2)
    w = rng.standard_normal((37, 96)) * rng.uniform(0.01, 1, (37, 1))
    q, s = oracle.quant_w8(w)
    w32 = w.astype(np.float32).astype(np.float64)
    assert np.all(np.abs(q.astype(np.float64) * s[:, None] - w32) <= s[:, None] * (0.5 + 1e-6))
    assert np.all(np.max(np.abs(q.astype(np.int64)), axis=1) == 127)
    deq = q.astype(np.float64) * s[:, None].astype(np.float64)
    q2, s2 = oracle.quant_w8(deq)
    assert np.array_equal(q2, q)


def test_quant_w4_roundtrip_and_bound():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((19, 128)) * 0.02
    codes, s16 = oracle.quant_w4(w, group=32)
    assert codes.min() >= -7 and codes.max() <= 7
    deq = oracle.dequant_w4(codes, s16, group=32)
    sg = np.repeat(s16.astype(np.float64), 32, axis=1)
    assert np.all(np.abs(deq - w.astype(np.float32)) <= sg * 0.5 * (1 + 1e-3) + 1e-12)
    codes2, s2 = oracle.quant_w4(deq, group=32)
    assert np.array_equal(codes2, codes)
    assert np.array_equal(s2, s16)


# ---- exact rational brute force -----------------------------------------------------

def _exact_fp(Wf, xf):
    N, K = Wf.shape
    M = xf.shape[0]
    y = [[sum((Fraction(float(Wf[n, k])) * Fraction(float(xf[m, k])) for k in range(K)),
              Fraction(0)) for n in range(N)] for m in range(M)]
    return y


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(3, 5, 1), (7, 64, 2), (1, 8, 3), (5, 40, 1)])
def test_fp_gemv_brute_force(fmt, shape):
    N, K, M = shape
    rng = np.random.default_rng(N * 100 + K + M)
    Wt = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32) * 0.7)
    xt = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32))
    dt = torch.float16 if fmt == "f16" else torch.bfloat16
    Wb = Wt.to(dt).view(torch.int16).numpy().view(np.uint16)
    xb = xt.to(dt).view(torch.int16).numpy().view(np.uint16)
    Wf = Wt.to(dt).double().numpy()
    xf = xt.to(dt).double().numpy()
    y, A = oracle.gemv_fp(Wb, xb, fmt)
    ex = _exact_fp(Wf, xf)
    for m in range(M):
        for n in range(N):
            absum = sum(abs(Fraction(float(Wf[n, k])) * Fraction(float(xf[m, k]))) for k in range(K))
            assert A[m, n] == pytest.approx(float(absum), rel=K * 2.0 ** -52)
            assert abs(Fraction(y[m, n]) - ex[m][n]) <= K * Fraction(2) ** -52 * absum


@pytest.mark.parametrize("shape", [(3, 16, 1), (6, 48, 4), (2, 32, 16)])
def test_w8a8_brute_force(shape):
    N, K, M = shape
    rng = np.random.default_rng(K + N)
    W = rng.integers(-127, 128, (N, K)).astype(np.int8)
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    s_w = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    s_x = rng.uniform(1e-2, 5e-2, M).astype(np.float32)
    acc, y, A = oracle.gemv_w8a8(W, s_w, xq, s_x)
    for m in range(M):
        for n in range(N):
            ex = sum(int(W[n, k]) * int(xq[m, k]) for k in range(K))
            assert acc[m, n] == ex
            exy = Fraction(ex) * Fraction(float(s_w[n])) * Fraction(float(s_x[m]))
            assert abs(Fraction(y[m, n]) - exy) <= abs(exy) * Fraction(2) ** -51


def _random_w4(rng, N, K, G=32):
    codes = rng.integers(-8, 8, (N, K)).astype(np.int8)  # includes the code -8
    nib = codes.astype(np.int64) & 0xF
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)  # the test's own packing
    scales = f16(rng.uniform(1e-3, 1e-2, (N, K // G)))
    return codes, packed, scales


@pytest.mark.parametrize("shape", [(3, 32, 1), (5, 96, 2), (2, 64, 3)])
def test_w4a16_brute_force(shape):
    N, K, M = shape
    rng = np.random.default_rng(7 * N + K)
    codes, packed, scales = _random_w4(rng, N, K)
    x = f16(rng.standard_normal((M, K)))
    y, A = oracle.gemv_w4a16(packed, scales, x, group=32)
    for m in range(M):
        for n in range(N):
            ex = Fraction(0)
            ab = Fraction(0)
            for g in range(K // 32):
                s = Fraction(float(scales[n, g]))
                for k in range(32 * g, 32 * g + 32):
                    t = s * int(codes[n, k]) * Fraction(float(x[m, k]))
                    ex += t
                    ab += abs(t)
            assert abs(Fraction(y[m, n]) - ex) <= 2 * K * Fraction(2) ** -52 * ab
            assert A[m, n] == pytest.approx(float(ab), rel=2 * K * 2.0 ** -52)


@pytest.mark.parametrize("shape", [(3, 32, 1), (4, 128, 4)])
def test_w4a8_brute_force(shape):
    N, K, M = shape
    rng = np.random.default_rng(11 * N + K)
    codes, packed, scales = _random_w4(rng, N, K)
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    s_x = rng.uniform(1e-2, 5e-2, M).astype(np.float32)
    y, A, accg = oracle.gemv_w4a8(packed, scales, xq, s_x, group=32)
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for g in range(K // 32):
                a = sum(int(codes[n, k]) * int(xq[m, k]) for k in range(32 * g, 32 * g + 32))
                assert accg[m, n, g] == a
                tot += Fraction(float(scales[n, g])) * a
            ex = tot * Fraction(float(s_x[m]))
            assert abs(Fraction(y[m, n]) - ex) <= 2 * K * Fraction(2) ** -52 * Fraction(A[m, n])


# ---- library special cases --------------------------------------------------------------

def test_w8a8_acc_equals_numpy_int64_matmul():
    rng = np.random.default_rng(5)
    W = rng.integers(-127, 128, (300, 512)).astype(np.int8)
    xq = rng.integers(-127, 128, (3, 512)).astype(np.int8)
    acc, _, _ = oracle.gemv_w8a8(W, np.ones(300, np.float32), xq, np.ones(3, np.float32))
    assert np.array_equal(acc, xq.astype(np.int64) @ W.astype(np.int64).T)


def test_w4a8_group_acc_equals_numpy_int64():
    rng = np.random.default_rng(6)
    codes, packed, scales = _random_w4(rng, 64, 256)
    xq = rng.integers(-127, 128, (2, 256)).astype(np.int8)
    _, _, accg = oracle.gemv_w4a8(packed, scales, xq, np.ones(2, np.float32), group=32)
    ref = np.einsum("ngk,mgk->mng", codes.astype(np.int64).reshape(64, 8, 32),
                    xq.astype(np.int64).reshape(2, 8, 32))
    assert np.array_equal(accg, ref)


def test_w4a16_equals_fp64_matmul_on_dequantized_weights():
    rng = np.random.default_rng(8)
    codes, packed, scales = _random_w4(rng, 50, 256)
    x = f16(rng.standard_normal((2, 256)))
    y, A = oracle.gemv_w4a16(packed, scales, x, group=32)
    deq = codes.astype(np.float64) * np.repeat(scales.astype(np.float64), 32, axis=1)
    ref = x.astype(np.float64) @ deq.T
    assert np.all(np.abs(y - ref) <= 256 * 2.0 ** -50 * A)


def test_fp_gemv_equals_fp64_matmul():
    rng = np.random.default_rng(9)
    W = f16(rng.standard_normal((70, 300)) * 0.02)
    x = f16(rng.standard_normal((3, 300)))
    y, A = oracle.gemv_fp(W, x)
    ref = x.astype(np.float64) @ W.astype(np.float64).T
    assert np.all(np.abs(y - ref) <= 300 * 2.0 ** -50 * A)


# ---- closed forms --------------------------------------------------------------------

def test_identity_weights_return_x_exactly():
    rng = np.random.default_rng(10)
    x = f16(rng.standard_normal((2, 64)))
    y, _ = oracle.gemv_fp(np.eye(64, dtype=np.float16), x)
    assert np.array_equal(y, x.astype(np.float64))


def test_one_hot_rows_select_a_column():
    rng = np.random.default_rng(11)
    K, N = 80, 13
    cols = rng.integers(0, K, N)
    W = np.zeros((N, K), np.float16)
    W[np.arange(N), cols] = 1
    x = f16(rng.standard_normal((1, K)))
    y, _ = oracle.gemv_fp(W, x)
    assert np.array_equal(y[0], x[0, cols].astype(np.float64))


def test_all_ones_row_is_the_sum_of_x():
    rng = np.random.default_rng(12)
    x = f16(rng.standard_normal((1, 64)))
    y, _ = oracle.gemv_fp(np.ones((1, 64), np.float16), x)
    assert y[0, 0] == math.fsum(x[0].astype(np.float64))  # exact: 64 fp16 terms fit in fp64


def test_scaled_one_hot_w8a8_and_w4():
    K = 64
    W = np.zeros((3, K), np.int8)
    W[0, 5], W[1, 0], W[2, 63] = 100, -127, 1
    xq = np.arange(-32, 32, dtype=np.int8).reshape(1, K)
    s_w = np.array([0.5, 0.25, 2.0], np.float32)
    acc, y, _ = oracle.gemv_w8a8(W, s_w, xq, np.array([0.125], np.float32))
    assert acc[0].tolist() == [100 * -27, -127 * -32, 31]
    assert y[0].tolist() == [100 * -27 * 0.0625, -127 * -32 * 0.03125, 31 * 0.25]
    codes = np.zeros((2, K), np.int8)
    codes[0, 7], codes[1, 40] = -8, 7
    nib = codes.astype(np.int64) & 0xF
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    scales = f16([[0.5, 4.0], [0.25, 2.0]])
    x = f16(np.linspace(-3, 3, K).reshape(1, K))
    y, _ = oracle.gemv_w4a16(packed, scales, x, group=32)
    assert y[0].tolist() == [0.5 * -8 * float(x[0, 7]), 2.0 * 7 * float(x[0, 40])]


# ---- argmax and the 16-slice invariant ------------------------------------------------------

def test_argmax_lowest_index_on_ties_and_nan_never_wins():
    assert oracle.argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.argmax([-0.0, 0.0]) == 0
    assert oracle.argmax([np.nan, 1.0, np.nan, 1.0]) == 1
    assert oracle.argmax([-np.inf, -np.inf]) == 0
    assert oracle.argmax([np.nan]) == -1
    assert oracle.argmax([]) == -1


def test_split16_host_reduce_equals_unsplit():
    rng = np.random.default_rng(13)
    N, K = 16 * 37, 128
    W = f16(rng.standard_normal((N, K)) * 0.02)
    x = f16(rng.standard_normal((1, K)))
    logits, _, tok = oracle.lm_head(W, x)
    l16, t16 = oracle.lm_head_split16(W, x)
    assert np.array_equal(l16, logits) and t16 == tok
    # planted winner in a late slice
    W2 = W.copy()
    W2[11 * 37 + 5] = f16(0.05 * np.sign(x[0].astype(np.float64)))
    l, _, tok2 = oracle.lm_head(W2, x)
    _, t2 = oracle.lm_head_split16(W2, x)
    assert tok2 == t2 == 11 * 37 + 5
    # an exact tie across slices: the lower global index wins
    W3 = W2.copy()
    W3[3 * 37 + 36] = W2[11 * 37 + 5]
    _, _, tok3 = oracle.lm_head(W3, x)
    _, t3 = oracle.lm_head_split16(W3, x)
    assert tok3 == t3 == 3 * 37 + 36


# ---- invariants of the partitioning ---------------------------------------------------------

def test_thread_count_and_row_subset_do_not_change_results():
    rng = np.random.default_rng(14)
    W = f16(rng.standard_normal((333, 200)) * 0.02)
    x = f16(rng.standard_normal((2, 200)))
    y1, A1 = oracle.gemv_fp(W, x, nthreads=1)
    y7, A7 = oracle.gemv_fp(W, x, nthreads=7)
    assert np.array_equal(y1, y7) and np.array_equal(A1, A7)
    rows = [300, 5, 17, 5]
    ys, As = oracle.gemv_fp(W, x, rows=rows, nthreads=3)
    assert np.array_equal(ys, y1[:, rows]) and np.array_equal(As, A1[:, rows])
    codes, packed, scales = _random_w4(rng, 90, 128)
    ya, _ = oracle.gemv_w4a16(packed, scales, x[:, :128], nthreads=1)
    yb, _ = oracle.gemv_w4a16(packed, scales, x[:, :128], rows=[89, 0], nthreads=4)
    assert np.array_equal(yb, ya[:, [89, 0]])


# ---- SiLU, SwiGLU, residual, causal-conv1d step -------------------------------

def test_silu_closed_forms_and_reflection():
    assert oracle.silu(0.0) == 0.0
    # sigmoid(ln 3) = 3/4 exactly, so silu(ln 3) = 0.75 ln 3
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12             # v sigmoid(v) -> v
    assert abs(oracle.silu(-40.0) / (-40.0 * math.exp(-40.0)) - 1.0) < 1e-12  # -> v e^v
    v = np.random.default_rng(3).normal(0, 4, 1000)
    # sigmoid(-v) = 1 - sigmoid(v)  =>  silu(-v) = silu(v) - v
    assert np.allclose(oracle.silu(-v), oracle.silu(v) - v, rtol=0, atol=1e-12)
    # and torch's own fp64 silu
    ref = torch.nn.functional.silu(torch.from_numpy(v)).numpy()
    assert np.allclose(oracle.silu(v), ref, rtol=1e-15, atol=1e-300)


def _dq(bits16):
    return np.asarray(bits16, np.uint16).view(np.float16).astype(np.float64)


def test_swiglu_equals_silu_of_gate_times_up_by_fp64_matmul():
    g = torch.Generator().manual_seed(11)
    Wg = (torch.randn(37, 96, generator=g) * 0.3).half().numpy()
    Wu = (torch.randn(37, 96, generator=g) * 0.3).half().numpy()
    x = torch.randn(3, 96, generator=g).half().numpy()
    h, gg, uu, Ag, Au = oracle.gemv_swiglu_fp(Wg, Wu, x)
    G = x.astype(np.float64) @ Wg.astype(np.float64).T
    Uu = x.astype(np.float64) @ Wu.astype(np.float64).T
    assert np.allclose(gg, G, rtol=0, atol=1e-12) and np.allclose(uu, Uu, rtol=0, atol=1e-12)
    assert np.allclose(h, (G / (1 + np.exp(-G))) * Uu, rtol=1e-14, atol=1e-14)
    # gate and up are not interchangeable
    assert not np.allclose(h, (Uu / (1 + np.exp(-Uu))) * G, rtol=1e-3, atol=1e-3)
    assert np.allclose(Ag, np.abs(x.astype(np.float64)) @ np.abs(Wg.astype(np.float64)).T)


def test_swiglu_w4a16_uses_each_matrix_with_its_own_scales():
    Wq, sc, x = _w4_small(29, 128, seed=12)
    Wq2, sc2, _ = _w4_small(29, 128, seed=13)
    h, gg, uu, _, _ = oracle.gemv_swiglu_w4a16(Wq, sc, Wq2, sc2, x)
    G = x.astype(np.float64) @ oracle.dequant_w4(oracle.unpack_w4(Wq).reshape(29, 128), sc).T
    Uu = x.astype(np.float64) @ oracle.dequant_w4(oracle.unpack_w4(Wq2).reshape(29, 128), sc2).T
    assert np.allclose(h, oracle.silu(G) * Uu, rtol=1e-13, atol=1e-13)


def _w4_small(N, K, seed):
    g = torch.Generator().manual_seed(seed)
    codes = torch.randint(-8, 8, (N, K), generator=g, dtype=torch.int16)
    nib = codes & 0xF
    Wq = (nib[:, 0::2] | (nib[:, 1::2] << 4)).to(torch.uint8).numpy()
    sc = (torch.rand(N, K // 32, generator=g) * 0.01 + 0.001).half().numpy()
    x = torch.randn(1, K, generator=g).half().numpy()
    return Wq, sc, x


def test_residual_adds_r_to_the_product():
    g = torch.Generator().manual_seed(14)
    W = (torch.randn(21, 64, generator=g) * 0.1).half().numpy()
    x = torch.randn(2, 64, generator=g).half().numpy()
    r = torch.randn(2, 21, generator=g).half().numpy()
    y, A = oracle.gemv_residual_fp(W, x, r)
    ref = r.astype(np.float64) + x.astype(np.float64) @ W.astype(np.float64).T
    assert np.allclose(y, ref, rtol=0, atol=1e-12)
    rows = np.array([20, 3, 0])
    ys, _ = oracle.gemv_residual_fp(W, x, r, rows=rows)
    assert np.array_equal(ys, y[:, rows])


def _conv_case(M, C, Wd, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, C, generator=g).half().numpy()
    st = torch.randn(M, C, Wd - 1, generator=g).half().numpy()
    w = (torch.randn(C, Wd, generator=g) * 0.5).half().numpy()
    b = (torch.randn(C, generator=g) * 0.1).half().numpy()
    return x, st, w, b


def test_conv1d_step_one_hot_taps_and_all_ones():
    x, st, w, b = _conv_case(2, 9, 4, seed=15)
    e_new = np.zeros((9, 4), np.float16)
    e_new[:, 3] = 1
    y, v, _, ns = oracle.causal_conv1d_update(x, st, e_new, None, act="none")
    assert np.array_equal(y, x.astype(np.float64))            # newest tap: y = x
    e_old = np.zeros((9, 4), np.float16)
    e_old[:, 0] = 1
    y, _, _, _ = oracle.causal_conv1d_update(x, st, e_old, None, act="none")
    assert np.array_equal(y, st[:, :, 0].astype(np.float64))  # oldest tap
    ones = np.ones((9, 4), np.float16)
    y, _, A, _ = oracle.causal_conv1d_update(x, st, ones, b, act="none")
    win = np.concatenate([st.astype(np.float64), x.astype(np.float64)[:, :, None]], axis=2)
    assert np.allclose(y, b.astype(np.float64) + win.sum(axis=2), rtol=0, atol=1e-12)
    assert np.allclose(A, np.abs(b.astype(np.float64)) + np.abs(win).sum(axis=2))
    # the window drops its oldest input and appends the new one
    assert np.array_equal(ns[:, :, :2].view(np.uint16), st[:, :, 1:].view(np.uint16))
    assert np.array_equal(ns[:, :, 2].view(np.uint16), x.view(np.uint16))


def test_conv1d_steps_equal_numpy_convolve_over_a_sequence():
    """Stepping from a zero window over a sequence gives the causal
    convolution: y_t = sum_j w[j] s[t - (W-1) + j] = np.convolve(s, w[::-1])[t]."""
    g = torch.Generator().manual_seed(16)
    C, Wd, T = 5, 4, 11
    seq = torch.randn(T, C, generator=g).half().numpy()
    w = (torch.randn(C, Wd, generator=g) * 0.5).half().numpy()
    st = np.zeros((1, C, Wd - 1), np.float16)
    for t in range(T):
        y, _, _, st = oracle.causal_conv1d_update(seq[t][None], st, w, None, act="none")
        for c in range(C):
            ref = np.convolve(seq[:, c].astype(np.float64), w[c, ::-1].astype(np.float64))[t]
            assert abs(y[0, c] - ref) <= 1e-12 * (1 + abs(ref))


def test_conv1d_step_brute_force_fractions_and_silu():
    x, st, w, b = _conv_case(2, 6, 3, seed=17)
    y, v, A, _ = oracle.causal_conv1d_update(x, st, w, b, act="silu")
    for m in range(2):
        for c in range(6):
            u = [Fraction(float(q)) for q in st[m, c]] + [Fraction(float(x[m, c]))]
            ex = Fraction(float(b[c])) + sum(Fraction(float(w[c, j])) * u[j] for j in range(3))
            assert abs(Fraction(v[m, c]) - ex) <= Fraction(1, 2 ** 50) * (1 + abs(ex))
    assert np.allclose(y, v / (1 + np.exp(-v)), rtol=1e-15, atol=0)
