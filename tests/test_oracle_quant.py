"""Pins of the oracle's quantizers: a hand-derived fixture and the invariants the
pages state for token-block scaling (transpose validity, no clamping, minimal
exponent, document locality) and for the NVFP4 operand of the mixed path."""
import json
import os

import numpy as np
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_small_fixture():
    g = json.load(open(os.path.join(GOLDEN, "quant_small.json")))
    x = np.array(g["x"], dtype=np.float64)
    codes, scales = oracle.quantize_blocks(x, g["cu_seqlens"], 32)
    assert codes.tolist() == g["codes"]
    assert scales.tolist() == g["scales"]


def _blocks(cu, block):
    for s, e in zip(cu[:-1], cu[1:]):
        for b in range(s, e, block):
            yield b, min(b + block, e)


def test_codes_equal_torch_cast_and_exponent_is_minimal():
    w = synth.custom([37, 100, 5, 64], H=3, d=128, outlier_channels=2)
    x = w.tensor("q").astype(np.float64)
    cu = w.cu_seqlens
    codes, scales = oracle.quantize_blocks(x, cu, 32)
    vals = oracle.e4m3_values()
    for s, e in _blocks(cu, 32):
        for h in range(3):
            ex = int(scales[h, s]) - 127
            assert (scales[h, s:e] == scales[h, s]).all()
            blk = x[s:e, h, :]
            scaled = np.ldexp(blk, -ex)
            amax = np.abs(scaled).max()
            assert amax <= 448.0          # nothing clamps
            assert amax > 224.0           # e is the smallest that does not clamp
            ref = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert (codes[s:e, h, :] == ref).all()
            assert np.abs(vals[codes[s:e, h, :]]).max() <= 448.0


def test_transpose_validity():
    # A 32 x 32 block read MN-major (tokens <-> channels) gives the transposed
    # codes and the same exponent: one payload serves both orientations.
    rng = np.random.default_rng(11)
    blk = np.ldexp(rng.standard_normal((32, 32)), 3)
    c1, s1 = oracle.quantize_blocks(blk[:, None, :], [0, 32], 32)
    c2, s2 = oracle.quantize_blocks(blk.T.copy()[:, None, :], [0, 32], 32)
    assert (c1[:, 0, :] == c2[:, 0, :].T).all()
    assert (s1 == s2).all()


def test_document_locality():
    w = synth.custom([45, 70, 33], H=2, d=64)
    x = w.tensor("k").astype(np.float64)
    cu = w.cu_seqlens
    c1, s1 = oracle.quantize_blocks(x, cu, 32)
    y = x.copy()
    y[45:115] *= 1000.0
    y[60, 1, 3] = 1e30
    c2, s2 = oracle.quantize_blocks(y, cu, 32)
    for sl in (slice(0, 45), slice(115, 148)):
        assert (c1[sl] == c2[sl]).all()
        assert (s1[:, sl] == s2[:, sl]).all()
    assert not (s1[:, 45:115] == s2[:, 45:115]).all()


def test_per_token_exponent():
    w = synth.custom([20, 13], H=2, d=64, seed=99)
    x = w.tensor("v").astype(np.float64)
    codes, scales = oracle.quantize_blocks(x, w.cu_seqlens, 1)
    for t in range(w.T):
        for h in range(2):
            ex = int(scales[h, t]) - 127
            a = np.abs(np.ldexp(x[t, h], -ex)).max()
            assert 224.0 < a <= 448.0


def test_block_partial_and_zero_blocks():
    x = np.zeros((40, 1, 16))
    x[33:40, 0, 0] = 3.0
    codes, scales = oracle.quantize_blocks(x, [0, 40], 32)
    assert (scales[0, :32] == 127).all()         # all-zero block: e = 0
    assert (codes[:32] == 0).all()
    assert (scales[0, 32:] == 127 - 7).all()     # 3 = 0.75 * 2^2 -> e = 2 - 9 = -7


def test_dequantize_roundtrip_error_bound():
    w = synth.custom([64, 64], H=2, d=128, seed=5)
    x = w.tensor("q").astype(np.float64)
    codes, scales = oracle.quantize_blocks(x, w.cu_seqlens, 32)
    xh = oracle.dequantize_blocks(codes, scales)
    e = (scales.T.astype(np.float64) - 127)[:, :, None]
    # RNE with 3 mantissa bits: relative error <= 2^-4 in the normal range,
    # absolute error <= 2^-10 * 2^e in the subnormal range
    bound = np.maximum(np.abs(x) * 2.0 ** -4, np.ldexp(1.0, -10) * np.exp2(e))
    assert (np.abs(xh - x) <= bound).all()


def test_nvfp4_no_clamp_minimal_scale_and_nearest_code():
    w = synth.custom([50, 30], H=2, d=128, seed=12, outlier_channels=2)
    x = w.tensor("q").astype(np.float64)
    codes, bsc, g = oracle.quantize_nvfp4(x)
    vals4 = np.array([oracle.e2m1_decode(c) for c in range(16)])
    v8 = oracle.e4m3_values()
    for t in range(w.T):
        for h in range(2):
            amax_t = np.float32(np.abs(x[t, h]).max())
            assert g[h, t] == np.float32(amax_t / np.float32(2688.0))
            for b in range(8):
                seg = x[t, h, 16 * b:16 * b + 16].astype(np.float32)
                amax_b = np.abs(seg).max()
                c = int(bsc[t, h, b])
                r = np.float32(amax_b / np.float32(np.float32(6.0) * g[h, t]))
                if r > 448.0:   # fp32 rounding of g can push r an ulp past 448: saturate
                    assert c == 0x7E and r <= 448.0 * (1 + 2.0 ** -20)
                else:
                    assert v8[c] >= r and (c == 1 or v8[c - 1] < r)  # rounded-up, minimal
                sg = np.float32(np.float32(v8[c]) * g[h, t])
                q = (seg / sg).astype(np.float32)
                # no clamp: fp32 rounding of g and s may overshoot 6 by an ulp or
                # two, which still rounds to 6 under RNE (the next midpoint is 7)
                assert np.abs(q).max() <= 6.0 * (1 + 2.0 ** -20)
                got = vals4[codes[t, h, 16 * b:16 * b + 16]]
                best = np.min(np.abs(np.abs(q)[:, None] - vals4[None, :8]), axis=1)
                assert np.allclose(np.abs(np.abs(got) - np.abs(q)), best, atol=0)
                assert (np.sign(got[got != 0]) == np.sign(q[got != 0])).all()
    xh = oracle.dequantize_nvfp4(codes, bsc, g)
    cos = (xh * x).sum() / np.sqrt((xh * xh).sum() * (x * x).sum())
    assert cos > 0.99


def test_scale_byte_clamps_at_the_bottom_of_ue8m0():
    """A block whose no-clamp exponent lies below UE8M0's range is stored with
    byte 0 (scale 2^-127, the format's smallest), and its codes are the E4M3
    roundings of x 2^127; the two format definitions alone fix the values.
    A block of fp32 inputs (the fp32 input option) of subnormal size with max
    2^-130 (no-clamp exponent -138):
    2^-130 -> 2^-3, E4M3 0x20 (exponent field 4, mantissa 0), its negative
    0xA0; 2^-136 -> 2^-9, E4M3's smallest subnormal, 0x01; 2^-137 -> 2^-10,
    half of it: a tie, to even, 0x00; 1.5 2^-137 -> 0.75 2^-9: up to 0x01.
    At the top the clamp is out of reach of finite bf16 or fp32 inputs: the
    largest bf16, (2 - 2^-7) 2^127, takes e = 120 (byte 247) and scales to
    255, which rounds to 256 (0x78); the largest fp32 takes e = 120 too."""
    assert oracle.noclamp_exponent(2.0 ** -130) == -138
    assert oracle.scale_exponent(2.0 ** -130) == -127
    assert oracle.scale_exponent(2.0 ** 200) == 127          # reachable in fp64 only
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert float(torch.tensor(big, dtype=torch.bfloat16)) == big
    assert oracle.scale_exponent(big) == 120
    assert oracle.scale_exponent(float(np.finfo(np.float32).max)) == 120

    x = np.zeros((64, 1, 64))
    small = {(0, 0): 2.0 ** -130, (1, 1): -(2.0 ** -130), (2, 2): 2.0 ** -136, (3, 3): 2.0 ** -137,
             (4, 4): 1.5 * 2.0 ** -137}
    for (t, c), v in small.items():
        assert float(np.float32(v)) == v                               # fp32 holds each value
        x[t, 0, c] = v
    x[32, 0, 0] = big
    codes, scales = oracle.quantize_blocks(x, [0, 32, 64], 32)
    assert (scales[0, :32] == 0).all() and (scales[0, 32:] == 247).all()
    want = np.zeros((64, 1, 64), np.uint8)
    for (t, c), code in zip(small, (0x20, 0xA0, 0x01, 0x00, 0x01)):
        want[t, 0, c] = code
    want[32, 0, 0] = 0x78
    assert (codes == want).all()
