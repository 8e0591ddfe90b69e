"""Pins of the oracle's bit-level exponential forward (inference only).

FLAMIA summary, §3.7 Bit-Level Exponentials for Inference and §4.4; close
reading, 4.5: for the 8-bit P^, a Schraudolph-style approximation computes
2^z in the bf16 bit field (a fused multiply-add writes z as a fixed-point
number, the integer is shifted into the exponent field), with a shift that
makes its error zero-mean, on five of every eight pairs of exponentials; the
output's cosine similarity changes by less than 1e-4.  Reading: the cosine to
the unquantized high-precision output, with and without the approximation.
The backward cannot use it (it must rebuild the forward's P^ exactly).

* integer z gives 2^z * 249 / 256 (the fraction is 0, the shift 7 units of a
  7-bit mantissa); hand values, ties of the rounding, the clamp;
* every value is bf16-exact and the function is non-decreasing;
* the error bound of the piecewise-linear 2^floor(z) (1 + frac z) (at most
  +6.2 %) with the shift, and its mean log error near 0 (a shift of 6 or 8
  units fails it);
* with zero queries every visible key's z is an integer, so O has a closed
  form that counts the approximated keys: O_i = sum_j V_j / sum_j w_j with
  w_j = 249/256 on pairs 0-4 of every 8 in each 32-key block and 1 elsewhere;
* the cosine of O to the unquantized fp64 output drops by less than 1e-4.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def test_integer_points():
    for k in range(-120, 9):
        assert oracle.bitexp2(float(k)) == math.ldexp(249.0 / 256.0, k), k


def test_hand_values_ties_and_clamp():
    # 128 z = 64: n = 64 + 16249 = 16313, exponent 127, mantissa 57
    assert oracle.bitexp2(0.5) == 185.0 / 128.0
    # 128 z = -416: n = 15833, exponent 123, mantissa 89 -> 217 / 2048
    assert oracle.bitexp2(-3.25) == 217.0 / 2048.0
    # ties of 128 z go to the even integer: 0.5 -> 0, 1.5 -> 2
    assert oracle.bitexp2(1.0 / 256.0) == 249.0 / 256.0
    assert oracle.bitexp2(3.0 / 256.0) == 251.0 / 256.0
    # n = 0 at z_lo = -126.9453125 and below; one unit above it, the least bf16 subnormal
    z_lo = -126.9453125
    assert oracle.bitexp2(z_lo) == 0.0
    assert oracle.bitexp2(-1e6) == 0.0
    assert oracle.bitexp2(-math.inf) == 0.0
    assert oracle.bitexp2(math.nan) == 0.0
    assert oracle.bitexp2(z_lo + 1.0 / 128.0) == 2.0 ** -133
    # the largest z a P^ block can hold, log2 448: n = RNE(1127.3) + 16249 =
    # 17376, exponent 135, mantissa 96: 2^8 * 1.75 = 448, E4M3's largest value
    assert oracle.bitexp2(math.log2(448.0)) == 448.0


def test_bf16_exact_and_monotone():
    z = np.linspace(-30.0, math.log2(448.0), 20011)
    v = np.array([oracle.bitexp2(t) for t in z])
    assert all(oracle.round_bf16(t) == t for t in v)
    assert (np.diff(v) >= 0).all()
    assert (v > 0).all()


def test_error_bound_and_zero_mean():
    # z uniform over many binades, dense in the fraction
    z = (np.arange(64 * 4096) + 0.37) / 4096.0 - 40.0
    r = np.log2(np.array([oracle.bitexp2(t) for t in z])) - z
    # Mitchell: 0 <= log2((1 + f) / 2^f) <= 0.0861; rounding the fraction to
    # 7 bits moves it by at most half a unit, the shift takes 7 units away
    # (in the binade below when the rounded fraction is under 7 units)
    assert r.max() <= 0.0861 - 6.5 / 128 + 1e-9
    assert r.min() >= -7.5 / 128 - 1e-9
    # zero-mean: residual (7.33 - 7) / 128 of a unit; shift 6 gives +0.0104,
    # shift 8 gives -0.0052
    assert abs(r.mean()) < 0.004


def _closed_form_O(cu, V, causal):
    T = V.shape[0]
    O = np.zeros_like(V)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for i in range(a, b):
            js = range(a, (i + 1) if causal else b)
            w = [249.0 / 256.0 if (((j - a) % 32) // 2) % 8 < 5 else 1.0 for j in js]
            O[i] = V[list(js)].sum(axis=0) / sum(w)
    return O


@pytest.mark.parametrize("causal", [True, False])
def test_zero_queries_closed_form(causal):
    rng = np.random.default_rng(5)
    cu = np.array([0, 45, 100, 171], np.int32)
    T, H, d = int(cu[-1]), 2, 8
    Q = np.zeros((T, H, d))
    K = rng.standard_normal((T, 1, d))
    V = rng.standard_normal((T, 1, d))
    eV = rng.integers(-3, 1, (1, T)).astype(np.int32)
    r = oracle.attention(cu, Q, K, V, eV=eV, causal=causal, bitexp=True)
    want = _closed_form_O(cu, V[:, 0], causal)
    for h in range(H):
        np.testing.assert_allclose(r["O"][:, h], want, rtol=1e-13, atol=1e-13)
    # the exact exponential gives the plain mean over the visible keys
    e = oracle.attention(cu, Q, K, V, eV=eV, causal=causal)
    assert not np.allclose(e["O"], r["O"])


def _cos(x, y):
    x, y = x.ravel(), y.ravel()
    return float(x @ y / np.linalg.norm(x) / np.linalg.norm(y))


@pytest.mark.parametrize("lens,d,seed", [([700, 333, 64], 128, 41), ([1024], 64, 9)])
def test_cosine_change_below_1e_4(lens, d, seed):
    w = synth.custom(lens, H=2, Hkv=1, d=d, seed=seed)
    q, k, v = (w.tensor(n) for n in ("q", "k", "v"))
    ref = oracle.train_call(q, k, v, None, w.cu_seqlens, out_dtype="f64", quantize=False)["O"]
    a = oracle.train_call(q, k, v, None, w.cu_seqlens, out_dtype="f64")["O"]
    b = oracle.train_call(q, k, v, None, w.cu_seqlens, out_dtype="f64", bitexp=True)["O"]
    assert 0 <= _cos(a, ref) - _cos(b, ref) < 1e-4
    # the approximation does change O, by about the size of the 8-bit P^ noise
    assert 0.999 < _cos(a, b) < 1.0


def test_no_backward():
    w = synth.custom([40], H=1, d=64, seed=3)
    q, k, v, do = (w.tensor(n) for n in ("q", "k", "v", "do"))
    with pytest.raises(ValueError):
        oracle.train_call(q, k, v, do, w.cu_seqlens, bitexp=True)
