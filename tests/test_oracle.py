"""Pins for the CPU oracle (no GPU).

The oracle is the plain definition ref = x @ W^T summed in fp64 from the bf16
inputs.  None of these checks retypes its loop: each one compares it with
something fixed independently of it — IEEE binary32 bit patterns, closed forms
(one-hot rows, identity slices), exact rational arithmetic (``fractions``),
integer matrix products (numpy int64), invariance under permuting k, and a
float64 library matmul within the textbook summation error bound.  The last
test plants plausible mistakes in a scratch copy of the oracle's C source and
checks that these pins catch every one of them.
"""
import math
import os
import shutil
import subprocess
import ctypes
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import projection_inputs as pin

EPS64 = 2.0 ** -53


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- widening
@pytest.mark.parametrize("pattern,value", [
    (0x0000, 0.0),
    (0x3F80, 1.0),
    (0xBF80, -1.0),
    (0x4000, 2.0),
    (0xC0A0, -5.0),
    (0x3F81, 1.0 + 2.0 ** -7),          # last mantissa bit
    (0x4049, 3.140625),                 # 1.5703125 * 2
    (0x0080, 2.0 ** -126),              # smallest normal
    (0x0001, 2.0 ** -133),              # smallest subnormal
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),  # largest finite
])
def test_widening_matches_binary32_layout(pattern, value):
    got = oracle.bf16_to_f64(np.array([pattern], dtype=np.uint16))[0]
    assert got == value


def test_widening_signed_zero_and_inf():
    got = oracle.bf16_to_f64(np.array([0x8000, 0x7F80, 0xFF80], dtype=np.uint16))
    assert got[0] == 0.0 and math.copysign(1.0, got[0]) == -1.0
    assert got[1] == math.inf and got[2] == -math.inf


# ---------------------------------------------------------------- rounding
@pytest.mark.parametrize("value,pattern", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),                 # tie -> even (mantissa 0)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),             # tie -> even (mantissa 2)
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),    # just above the tie
    (-(1.0 + 2.0 ** -8 - 2.0 ** -40), 0xBF80), # just below the tie, negative
    (2.0 ** -127, 0x0040),                     # subnormal, exact
    (2.0 ** -134, 0x0000),                     # half the smallest subnormal: tie -> 0
    (3 * 2.0 ** -134, 0x0002),                 # 1.5 subnormal steps: tie -> even (2)
    ((2.0 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),  # overflow tie -> inf
    ((2.0 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),  # largest finite stays
    (65536.0 + 256.0, 0x4780),                 # 65792 is a tie between 65536 and 66048 -> even
])
def test_round_bf16_known_values(value, pattern):
    assert int(oracle.round_bf16([value])[0]) == pattern


def test_round_bf16_agrees_with_torch_cast_on_binary32_values():
    # For values already exact in binary32, rounding to bf16 is the library cast.
    g = torch.Generator().manual_seed(7)
    v = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp2(
        torch.randint(-30, 30, (20000,), generator=g).float())
    want = bits(v.to(torch.bfloat16))
    got = oracle.round_bf16(v.double().numpy())
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- closed forms
def test_one_hot_rows_select_a_weight_column():
    N, K = 37, 29
    w = pin.weight(N, K, seed=3)
    cols = [0, 5, 28, 17]
    x = pin.one_hot_rows(len(cols), K, cols)
    ref, s = oracle.projection(x, w)
    wv = w.double().numpy()
    for m, j in enumerate(cols):
        assert np.array_equal(ref[m], wv[:, j])
        assert np.array_equal(s[m], np.abs(wv[:, j]))


def test_identity_slice_returns_x_columns():
    M, K = 5, 24
    for N in (16, 24, 40):  # N < K, N == K, N > K
        x = pin.case(8, K, seed=11)[1][:M]
        w = pin.identity_slice(N, K)
        ref, s = oracle.projection(x, w)
        xv = x.double().numpy()
        d = min(N, K)
        assert np.array_equal(ref[:, :d], xv[:, :d])
        assert np.all(ref[:, d:] == 0.0)
        assert np.array_equal(s[:, :d], np.abs(xv[:, :d]))


def test_all_ones_scale_is_sqrt_k():
    M, N, K = 3, 4, 100
    ones = torch.ones
    ref, s = oracle.projection(ones(M, K, dtype=torch.bfloat16), ones(N, K, dtype=torch.bfloat16))
    assert np.all(ref == K) and np.all(s == math.sqrt(K))


# ---------------------------------------------------------------- exact brute force
def _exact(xv, wv):
    M, K = xv.shape
    N = wv.shape[0]
    fx = [[Fraction(float(v)) for v in row] for row in xv]
    fw = [[Fraction(float(v)) for v in row] for row in wv]
    out = [[sum((fx[m][k] * fw[n][k] for k in range(K)), Fraction(0)) for n in range(N)]
           for m in range(M)]
    sq = [[sum(((fx[m][k] * fw[n][k]) ** 2 for k in range(K)), Fraction(0)) for n in range(N)]
          for m in range(M)]
    return out, sq


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 3, 5), (3, 1, 7), (2, 5, 3), (8, 7, 8), (4, 6, 2)])
def test_brute_force_exact_rationals(shape):
    M, N, K = shape
    g = torch.Generator().manual_seed(M * 100 + N * 10 + K)
    x = (torch.randn(M, K, generator=g) * 3).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.3).to(torch.bfloat16)
    ref, s = oracle.projection(x, w)
    ex, sq = _exact(x.double().numpy(), w.double().numpy())
    xa, wa = x.double().abs().numpy(), w.double().abs().numpy()
    for m in range(M):
        for n in range(N):
            # recursive summation: |fl(sum) - sum| <= (K-1) u sum|p| (+ o(u))
            bound = 1.01 * max(K - 1, 0) * EPS64 * float(np.dot(xa[m], wa[n]))
            assert abs(Fraction(ref[m, n]) - ex[m][n]) <= Fraction(bound)
            exact_s = math.sqrt(float(sq[m][n]))
            assert abs(s[m, n] - exact_s) <= 4 * K * EPS64 * exact_s + 1e-300


def test_small_integers_are_exact_integer_products():
    M, N, K = 6, 33, 1000
    x = pin.small_integers(M, K, seed=1)
    w = pin.small_integers(N, K, seed=2)
    ref, s = oracle.projection(x, w)
    xi = x.float().numpy().astype(np.int64)
    wi = w.float().numpy().astype(np.int64)
    assert np.array_equal(ref, (xi @ wi.T).astype(np.float64))
    sq = ((xi[:, None, :] * wi[None, :, :]) ** 2).sum(-1)
    assert np.allclose(s, np.sqrt(sq.astype(np.float64)), rtol=1e-15, atol=0)


# ---------------------------------------------------------------- invariants
def test_order_invariance_under_k_permutation():
    M, N, K = 4, 50, 7168
    w, x = pin.case(N, K, seed=5)
    x = x[:M]
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(9))
    ref, s = oracle.projection(x, w)
    ref_p, s_p = oracle.projection(x[:, perm], w[:, perm])
    absdot = x.double().abs().numpy() @ w.double().abs().numpy().T
    assert np.all(np.abs(ref - ref_p) <= 2.02 * K * EPS64 * absdot)
    assert np.allclose(s, s_p, rtol=4 * K * EPS64, atol=0)


def test_matches_float64_library_matmul_within_summation_bound():
    M, N, K = 8, 300, 7168
    w, x = pin.case(N, K, seed=0)
    x = x[:M]
    ref, _ = oracle.projection(x, w)
    lib = x.double().numpy() @ w.double().numpy().T
    absdot = x.double().abs().numpy() @ w.double().abs().numpy().T
    assert np.all(np.abs(ref - lib) <= 2.02 * K * EPS64 * absdot)


def test_row_pitch_views_match_packed():
    M, N, K = 3, 20, 64
    w, x = pin.case(N + 4, K + 32, seed=2)
    xs, ws = x[:M, 8:8 + K], w[2:2 + N, 16:16 + K]  # strided views
    r1, s1 = oracle.projection(xs, ws)
    r2, s2 = oracle.projection(xs.contiguous(), ws.contiguous())
    assert np.array_equal(r1, r2) and np.array_equal(s1, s2)


# ---------------------------------------------------------------- tolerance rule
def test_tolerance_rule_hand_values():
    ref = np.array([1.0, -2.0, 0.0, 100.0])
    s = np.array([1.0, 1.0, 0.5, 0.0])
    # bounds: 8e-3*1+2e-3 = 0.010; 0.016+0.002 = 0.018; 0.001; 0.8
    ok = oracle.tolerance_ok(np.array([1.0099, -2.0181, 0.0011, 100.79]), ref, s)
    assert ok.tolist() == [True, False, False, True]
    assert oracle.tolerance_excess(np.array([1.005, -2.0, 0.0, 100.0]), ref, s) == pytest.approx(0.5)


# ---------------------------------------------------------------- planted mistakes
MUTATIONS = {
    "sign": ("acc += p;", "acc += (k == 0 ? -p : p);"),
    "dropped_term": ("for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 1; k < K; ++k) {"),
    "transposed_w": ("const uint16_t* wn = w + n * ldw;", "const uint16_t* wn = w + n;"),
    "wrong_x_row": ("const uint16_t* xm = x + m * ldx;", "const uint16_t* xm = x;"),
    "float_accum": ("double acc = 0.0, sq = 0.0;", "float acc = 0.0f; double sq = 0.0;"),
    "widen_shift": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
}


def _mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "ref.c")).read()
    old, new = MUTATIONS[name]
    assert old in src, f"mutation anchor for {name} not found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new, 1))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC",
                    str(path), "-o", str(so), "-lm"], check=True, capture_output=True)
    lib = ctypes.CDLL(str(so))
    p16, p64 = ctypes.POINTER(ctypes.c_uint16), ctypes.POINTER(ctypes.c_double)
    lib.oracle_projection.argtypes = [p16, ctypes.c_int64, p16, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_int64, ctypes.c_int64, p64, p64, ctypes.c_int]

    def run(x, w):
        xb, wb = np.ascontiguousarray(bits(x)), np.ascontiguousarray(bits(w))
        M, K = xb.shape
        N = wb.shape[0]
        ref = np.empty((M, N)); s = np.empty((M, N))
        lib.oracle_projection(xb.ctypes.data_as(p16), K, wb.ctypes.data_as(p16), K, M, N, K,
                              ref.ctypes.data_as(p64), s.ctypes.data_as(p64), 1)
        return ref
    return run


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc needed to build mutants")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(tmp_path, name):
    run = _mutant(tmp_path, name)
    caught = []
    # one-hot closed form
    w = pin.weight(9, 12, seed=4)
    x = pin.one_hot_rows(3, 12, [0, 4, 11])
    caught.append(not np.array_equal(run(x, w)[1], w.double().numpy()[:, 4]) or
                  not np.array_equal(run(x, w)[0], w.double().numpy()[:, 0]))
    # exact brute force (non-square, so a transposed operand cannot pass)
    g = torch.Generator().manual_seed(1)
    xs = (torch.randn(3, 7, generator=g) * 3).to(torch.bfloat16)
    ws = (torch.randn(5, 7, generator=g) * 0.3).to(torch.bfloat16)
    ex, _ = _exact(xs.double().numpy(), ws.double().numpy())
    got = run(xs, ws)
    bound = 7 * EPS64 * float(np.abs(xs.double().numpy()).sum() * np.abs(ws.double().numpy()).max())
    caught.append(any(abs(Fraction(got[m, n]) - ex[m][n]) > Fraction(bound)
                      for m in range(3) for n in range(5)))
    # exact integer products whose partial sums pass 2^24, where a binary32
    # accumulator would drop low bits
    xi = pin.small_integers(2, 4096, seed=1, lo=100, hi=255)
    wi = pin.small_integers(3, 4096, seed=2, lo=100, hi=255)
    want = (xi.double().numpy().astype(np.int64) @ wi.double().numpy().astype(np.int64).T)
    caught.append(not np.array_equal(run(xi, wi), want.astype(np.float64)))
    assert any(caught), f"mutation {name} slipped past every pin"


# ---------------------------------------------------------------- fp16 inputs
def test_fp16_widening_all_bit_patterns_match_numpy():
    """Every binary16 pattern widens exactly as numpy's float16 -> float64 does."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.fp16_to_f64(pats)
    want = pats.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


@pytest.mark.parametrize("pattern,value", [
    (0x3C00, 1.0), (0xC000, -2.0), (0x0001, 2.0 ** -24), (0x0400, 2.0 ** -14),
    (0x7BFF, 65504.0), (0x3555, 0.333251953125), (0x3C01, 1.0 + 2.0 ** -10),
])
def test_fp16_widening_known_values(pattern, value):
    assert oracle.fp16_to_f64(np.array([pattern], dtype=np.uint16))[0] == value


def test_fp16_one_hot_and_small_integers():
    N, K = 33, 40
    w = pin.weight(N, K, seed=8).to(torch.float16)
    x = pin.one_hot_rows(3, K, [0, 17, 39]).to(torch.float16)
    ref, s = oracle.projection(x, w)
    wv = w.double().numpy()
    for m, j in enumerate([0, 17, 39]):
        assert np.array_equal(ref[m], wv[:, j]) and np.array_equal(s[m], np.abs(wv[:, j]))
    xi = pin.small_integers(5, 700, seed=3, dtype=torch.float16)
    wi = pin.small_integers(9, 700, seed=4, dtype=torch.float16)
    ref, _ = oracle.projection(xi, wi)
    want = xi.numpy().astype(np.int64) @ wi.numpy().astype(np.int64).T
    assert np.array_equal(ref, want.astype(np.float64))


def test_fp16_brute_force_exact_rationals():
    g = torch.Generator().manual_seed(12)
    x = (torch.randn(3, 6, generator=g) * 5).to(torch.float16)
    w = (torch.randn(4, 6, generator=g) * 0.2).to(torch.float16)
    ref, _ = oracle.projection(x, w)
    ex, _ = _exact(x.double().numpy(), w.double().numpy())
    xa, wa = x.double().abs().numpy(), w.double().abs().numpy()
    for m in range(3):
        for n in range(4):
            bound = 1.01 * 5 * EPS64 * float(np.dot(xa[m], wa[n]))
            assert abs(Fraction(ref[m, n]) - ex[m][n]) <= Fraction(bound)


def test_bit_arrays_need_an_explicit_type():
    b = np.zeros((2, 8), dtype=np.uint16)
    r0, _ = oracle.projection(b, b, dtype="fp16")
    assert np.all(r0 == 0)
    with pytest.raises(TypeError):
        oracle.projection(torch.zeros(2, 8, dtype=torch.float16), torch.zeros(2, 8, dtype=torch.bfloat16))


# ---------------------------------------------------------------- residual
def test_residual_zero_x_returns_the_residual_exactly():
    w = pin.weight(20, 64, seed=1)
    r = (torch.randn(3, 20, generator=torch.Generator().manual_seed(2)) * 7).to(torch.bfloat16)
    ref, s = oracle.projection_residual(torch.zeros(3, 64, dtype=torch.bfloat16), w, r)
    assert np.array_equal(ref, r.double().numpy()) and np.all(s == 0)


def test_residual_small_integers_exact():
    x = pin.small_integers(4, 300, seed=5)
    w = pin.small_integers(11, 300, seed=6)
    r = pin.small_integers(4, 11, seed=7, lo=-1000, hi=1000).to(torch.float32)
    ref, _ = oracle.projection_residual(x, w, r)
    want = x.float().numpy().astype(np.int64) @ w.float().numpy().astype(np.int64).T + \
        r.numpy().astype(np.int64)
    assert np.array_equal(ref, want.astype(np.float64))


def test_residual_shape_checked():
    w = pin.weight(8, 16, seed=1)
    with pytest.raises(ValueError):
        oracle.projection_residual(torch.zeros(2, 16, dtype=torch.bfloat16), w, np.zeros((2, 9)))
