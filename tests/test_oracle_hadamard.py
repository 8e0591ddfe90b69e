"""Pins of the oracle's Hadamard rotation of Q and K.

FLAMIA summary, abstract and §4.3 Ablation Study: the fused quantizer applies
a Hadamard rotation; close reading, 四 4.4 (fused quantization): QuIP-style
incoherence processing mixes the head-dimension channels to spread outliers,
and the orthogonal transform keeps the dot products.

* the Sylvester matrix: hand values, entries +-1, symmetric, H H = d I;
* the fp32 fast transform: equal to x H on inputs where fp32 is exact (basis
  vectors, small integers), within the per-stage rounding bound on bf16
  data, and applied twice it returns d x;
* the rotation is invisible to the unquantized call (the 1/d in the softmax
  scale and the back-rotation of dQ, dK are right): O, dQ, dK, dV agree
  with the unrotated call to 1e-12;
* on workloads with x20 outlier channels it brings the quantized O and dV
  closer to the unquantized output (the reason the pages give for it).
"""
import numpy as np
import pytest

import oracle
import synth


def test_sylvester_hand_values_and_orthogonality():
    assert oracle.sylvester(2).tolist() == [[1, 1], [1, -1]]
    assert oracle.sylvester(4)[3].tolist() == [1, -1, -1, 1]
    assert oracle.sylvester(8)[5].tolist() == [1, -1, 1, -1, -1, 1, -1, 1]
    for d in (2, 4, 8, 16, 32, 64, 128):
        h = oracle.sylvester(d)
        assert h.shape == (d, d)
        assert set(np.unique(h)) == {-1.0, 1.0}
        assert np.array_equal(h, h.T)
        assert np.array_equal(h @ h, d * np.eye(d))


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_exact_cases(d):
    h = oracle.sylvester(d)
    # basis vectors give the rows of H
    assert np.array_equal(oracle.fwht_f32(np.eye(d)), h)
    # small integers: every partial sum is exact in fp32
    rng = np.random.default_rng(d)
    x = rng.integers(-1000, 1000, (50, d)).astype(np.float64)
    y = oracle.fwht_f32(x)
    assert np.array_equal(y, x @ h)
    assert np.array_equal(oracle.fwht_f32(y), d * x)


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_rounding_bound(d):
    x = synth.round_to_bf16(np.random.default_rng(3 + d).standard_normal((400, d)).astype(np.float32))
    x[:, 5] *= 20.0  # an outlier channel
    exact = x.astype(np.float64) @ oracle.sylvester(d)
    got = oracle.fwht_f32(x)
    # log2(d) stages, each rounding a partial sum of at most sum |x| by 2^-24
    bound = np.log2(d) * 2.0 ** -24 * np.abs(x).sum(axis=1, keepdims=True)
    assert (np.abs(got - exact) <= bound).all()
    assert np.abs(got - exact).max() > 0  # fp32 does round here
    # the values the quantizer sees are fp32 numbers
    assert np.array_equal(got.astype(np.float32).astype(np.float64), got)


@pytest.mark.parametrize("causal", [True, False])
def test_rotation_invisible_without_quantization(causal):
    w = synth.custom([300, 45, 129], H=4, Hkv=2, d=128, seed=71)
    q, k, v, do = (w.tensor(n) for n in ("q", "k", "v", "do"))
    a = oracle.train_call(q, k, v, do, w.cu_seqlens, causal=causal, quantize=False)
    b = oracle.train_call(q, k, v, do, w.cu_seqlens, causal=causal, quantize=False, hadamard=True)
    for n in ("O", "dQ", "dK", "dV"):
        assert np.abs(a[n] - b[n]).max() <= 1e-12 * np.abs(a[n]).max(), n


def _cos(x, y):
    x, y = x.ravel(), y.ravel()
    return float(x @ y / np.linalg.norm(x) / np.linalg.norm(y))


@pytest.mark.parametrize("lens,d,seed", [([300, 257], 128, 41), ([512], 64, 7)])
def test_rotation_spreads_outlier_channels(lens, d, seed):
    w = synth.custom(lens, H=2, Hkv=1, d=d, seed=seed, outlier_channels=2)
    q, k, v, do = (w.tensor(n) for n in ("q", "k", "v", "do"))
    ref = oracle.train_call(q, k, v, do, w.cu_seqlens, out_dtype="f64", quantize=False)
    a = oracle.train_call(q, k, v, do, w.cu_seqlens, out_dtype="f64")
    b = oracle.train_call(q, k, v, do, w.cu_seqlens, out_dtype="f64", hadamard=True)
    for n in ("O", "dV"):
        assert 1.0 - _cos(b[n], ref[n]) < 0.5 * (1.0 - _cos(a[n], ref[n])), n
    # the rotated operands are what was quantized: Q's codes differ
    assert not np.array_equal(a["q_codes"], b["q_codes"])


def test_rotation_not_offered_on_the_mixed_path():
    w = synth.custom([40], H=1, d=64, seed=3)
    q, k, v, do = (w.tensor(n) for n in ("q", "k", "v", "do"))
    with pytest.raises(ValueError):
        oracle.train_call(q, k, v, do, w.cu_seqlens, path=oracle.PATH_NVFP4_FP8, hadamard=True)
