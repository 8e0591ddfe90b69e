"""Pins of the oracle's FP16 dQ partials with a power-of-two prescale.

Close reading, 四 4.4 (low-precision 2-CTA backward): dQ partials are
accumulated in FP16 by bulk reduce-adds, with a data-dependent power-of-two
prescale because a fixed one overflows on outlier K channels.  FLAMIA
summary, §4.5: an optional causal dQ scale removes the sequence-range
dependency of the FP16 accumulator.

* the FP16 rounding equals numpy's float16 conversion (a library routine);
* the prescale constant and exponent take their hand-derived values;
* on outlier workloads the FP16 result stays finite and within the FP16
  rounding bound of the fp64 sum;
* the causal dQ scale: perturbing tokens past L/2 leaves dQ of rows <= L/2
  bit-identical; the document-range prescale does not.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def test_round_f16_equals_numpy_float16():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(20000) * np.exp2(rng.integers(-30, 17, 20000)),
        # exact ties between neighbouring binary16 values, normal and subnormal
        (np.arange(1, 2048) + 0.5) * 2.0 ** -10, (np.arange(1, 1024) + 0.5) * 2.0 ** -24,
        [0.0, -0.0, 65504.0, 65519.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 6.1e-5],
    ])
    got = np.array([oracle.round_f16(v) for v in x])
    with np.errstate(over="ignore"):  # values beyond 65519 become infinity on both sides
        want = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, want)
    assert oracle.round_f16(65520.0) == math.inf


def test_prescale_hand_values():
    # d = 128, scale 1/sqrt(128): 2.5 * 128 * 448^3 / sqrt(128) = 2.54e9, in (2^31, 2^32]
    assert oracle.dq_prescale_c0(128, 128 ** -0.5) == 32
    # d = 64, scale 1/8: 2.5 * 64 * 448^3 / 8 = 1.80e9, in (2^30, 2^31]
    assert oracle.dq_prescale_c0(64, 0.125) == 31
    # exactly a power of two: 2.5 * 64 * 448^3 * s = 2^40
    s = 2.0 ** 40 / (2.5 * 64 * 448.0 ** 3)
    assert oracle.dq_prescale_c0(64, s) == 40
    # p = 15 - c0 - (edO + max eK + max eV), clamped to [-126, 127]
    assert oracle.dq_prescale(32, -7, -7, -7) == 4
    assert oracle.dq_prescale(32, -100, -100, -100) == 127
    assert oracle.dq_prescale(32, 100, 100, 100) == -126


@pytest.mark.parametrize("outliers", [0, 2])
def test_fp16_dq_within_rounding_bound(outliers):
    w = synth.custom([300, 45, 400], H=2, d=64, seed=61 + outliers, outlier_channels=outliers)
    q, k, v, do = (w.tensor(n) for n in ("q", "k", "v", "do"))
    a = oracle.train_call(q, k, v, do, w.cu_seqlens, out_dtype="f64", dq_fp16=False)
    b = oracle.train_call(q, k, v, do, w.cu_seqlens, out_dtype="f64", dq_fp16=True)
    assert np.isfinite(b["dQ"]).all()
    for n in ("O", "dK", "dV"):  # only dQ's reduction changes
        assert np.array_equal(a[n], b[n]), n
    # per row: at most one FP16 rounding of each partial and each running sum,
    # every value of the prescaled row below 2^15: the error stays below
    # (2 n_tiles) 2^-11 of the row's largest partial sum, bounded here by the
    # row max-abs of the fp64 result times the tiles' count
    err = np.abs(b["dQ"] - a["dQ"])
    rowmax = np.abs(a["dQ"]).max(axis=-1, keepdims=True)
    n_tiles = max(math.ceil(l / 128) for l in w.seqlens)
    assert (err <= 2 * n_tiles * 2.0 ** -11 * n_tiles * rowmax + 1e-12).all()
    assert err.max() > 0  # the FP16 accumulation did round
    cos = float((a["dQ"].ravel() @ b["dQ"].ravel()) / np.linalg.norm(a["dQ"]) / np.linalg.norm(b["dQ"]))
    assert cos > 0.99999


def _perturb_future(x, t0, seed):
    y = x.copy()
    rng = np.random.default_rng(seed)
    y[t0 + 1:] = rng.standard_normal(y[t0 + 1:].shape).astype(y.dtype)
    y[t0 + 1:t0 + 4] *= 1000.0
    return y


def test_causal_dq_scale_removes_the_future_dependency():
    w = synth.custom([512], H=2, d=64, seed=63)
    q, k, v, do = (w.tensor(n).astype(np.float64) for n in ("q", "k", "v", "do"))
    half = 256
    pert = [_perturb_future(x, half, 70 + i) for i, x in enumerate((q, k, v, do))]
    kw = dict(exact=True, dq_fp16=True)
    a = oracle.train_call(q, k, v, do, w.cu_seqlens, dq_causal_scale=True, **kw)
    b = oracle.train_call(*pert, w.cu_seqlens, dq_causal_scale=True, **kw)
    assert np.array_equal(a["dQ"][:half + 1], b["dQ"][:half + 1])
    # the document-range prescale sees the perturbed keys' larger exponents
    c = oracle.train_call(q, k, v, do, w.cu_seqlens, dq_causal_scale=False, **kw)
    d = oracle.train_call(*pert, w.cu_seqlens, dq_causal_scale=False, **kw)
    assert not np.array_equal(c["dQ"][:half + 1], d["dQ"][:half + 1])


def test_prescales_per_row_hand_values():
    # two documents [3, 2], one KV head, two query heads; d = 128 gives c0 = 32
    cu = np.array([0, 3, 5], np.int32)
    eK = np.array([[-5, -3, -4, -2, -6]])
    eV = np.array([[-7, -7, -1, -3, -3]])
    edO = np.array([[-8] * 5, [0] * 5])
    causal = oracle.dq_prescales(cu, eK, eV, edO, 128, causal=True, causal_scale=True)
    # p = 15 - 32 - (edO + MK + MV), MK / MV over keys j <= i of the document
    assert causal.tolist() == [[3, 1, -5, -4, -4], [-5, -7, -13, -12, -12]]
    docwide = oracle.dq_prescales(cu, eK, eV, edO, 128, causal=True, causal_scale=False)
    assert docwide.tolist() == [[-5, -5, -5, -4, -4], [-13, -13, -13, -12, -12]]
    # non-causal attention sees the whole document either way
    full = oracle.dq_prescales(cu, eK, eV, edO, 128, causal=False, causal_scale=True)
    assert np.array_equal(full, docwide)
