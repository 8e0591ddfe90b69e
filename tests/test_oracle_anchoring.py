"""Pins of where the oracle's in-attention quantizers put their blocks.

FLAMIA (paper summary), §3.1 Token-Block Scaling and §3.6.2 Load-Balanced
Scheduling: scale blocks cover 32 consecutive positions and never cross a
document boundary; §3.3: dS takes one exponent per 32x32 block; the exact
option (§4.5) quantizes dS for dQ per query row.  So, with keys and queries
counted from their document's start:

* P^   one exponent per (query row, 32-key block);
* dS^  one exponent per 32x32 (query block, key block); exact option: per
       (query row, 32-key block) for dQ, 32x32 for dK;
* P~   (the dV operand) one exponent per 32x32 block.

Each case below is built so that the value at one position is fixed by hand
(derivation in the comments) and changes if the blocks are anchored at the
absolute token index, are 16 wide, or have the other shape.  The second
document starts at token 45, so absolute 32-token blocks cut it at local
positions 19 and 51 instead of 32 and 64.  The wrong readings are written out
below as test-local functions and shown to miss the hand values.

The last test checks the same property on the whole call: a document's
outputs, codes and scales are bit-identical whether it is packed after other
documents or run alone.
"""
import math

import numpy as np
import pytest

import oracle
import synth

LENS = [45, 70, 33]            # document 1 starts at token 45 (not 32-aligned)
S0, L1 = 45, 70
CU = np.array([0, 45, 115, 148], np.int32)
T = 148
D = 72                          # >= L1: one channel per document-1 position
LN2 = 1.0 / 1.4426950408889634  # softmax scale that makes x = S * log2(e) the dot product


# ---------------------------------------------------------------------------
# Test-local block quantizer with a chosen block map (used for the readings).
# ---------------------------------------------------------------------------
def _quantize_blocks(M, row_block, col_block):
    """E4M3 with one no-clamp exponent per group of entries that share
    (row_block(i), col_block(j)); returns the dequantized matrix."""
    n_r, n_c = M.shape
    out = np.zeros_like(M)
    groups = {}
    for i in range(n_r):
        for j in range(n_c):
            groups.setdefault((row_block(i), col_block(j)), []).append((i, j))
    for idx in groups.values():
        amax = max(abs(M[i, j]) for i, j in idx)
        e = oracle.noclamp_exponent(amax)
        for i, j in idx:
            out[i, j] = math.ldexp(oracle.e4m3_decode(oracle.e4m3_encode(math.ldexp(M[i, j], -e))), e)
    return out


LOCAL32 = lambda t: t // 32            # the pages' reading: from the document start
ABS32 = lambda t: (S0 + t) // 32       # wrong: absolute token index
LOCAL16 = lambda t: t // 16            # wrong: 16-wide blocks
ROW = lambda t: t                      # one row per block


# ---------------------------------------------------------------------------
# P^: one exponent per (query row, 32 keys), document-local.
# ---------------------------------------------------------------------------
def _phat_case():
    """Scores of document 1 (x = dot product): row 20 sees key 5 at x = 0 and
    key 20 at x = -19; row 21 sees key 55 at 0 and key 21 at -19; every other
    row sees key 69 at 0; everything else is at -60.  V_j = e_j, eV = 0, so
    O_i[j] = P^_ij / l_i."""
    qs = np.zeros((T, 1, D))
    ks = np.zeros((T, 1, D))
    for i in range(L1):
        qs[S0 + i, 0, 0 if i == 20 else 1 if i == 21 else 2] = 1.0
    ks[S0:S0 + L1, 0, :3] = -60.0
    ks[S0 + 5, 0, 0] = 0.0
    ks[S0 + 20, 0, 0] = -19.0
    ks[S0 + 55, 0, 1] = 0.0
    ks[S0 + 21, 0, 1] = -19.0
    ks[S0 + 69, 0, 2] = 0.0
    v = np.zeros((T, 1, D))
    for j in range(L1):
        v[S0 + j, 0, j] = 1.0
    x = np.full((L1, L1), -60.0)        # the designed logits, exactly
    for i in range(L1):
        x[i, 69] = 0.0
    x[20] = -60.0
    x[20, 5], x[20, 20] = 0.0, -19.0
    x[21] = -60.0
    x[21, 55], x[21, 21] = 0.0, -19.0
    return qs, ks, v, x


def _phat_hand():
    # row 20: the block of keys 0-31 holds 2^0 (key 5), so its exponent is
    # -8 (448 * 2^-8 >= 1 > 448 * 2^-9) and key 20's 2^-19 * 2^8 = 2^-11 is
    # below half the smallest E4M3 subnormal 2^-9: code 0.  l_20 = 1 + 2^-19.
    # row 21: keys 0-31 hold only 2^-19 (key 21): exponent -27, code 256,
    # P^ = 2^-19 exactly; key 55 alone in keys 32-63: P^ = 1.
    l = 1.0 + 2.0 ** -19
    return {(20, 5): 1.0 / l, (20, 20): 0.0, (21, 21): 2.0 ** -19 / l, (21, 55): 1.0 / l}


def test_phat_blocks_are_row_by_32_document_local():
    qs, ks, v, _ = _phat_case()
    r = oracle.attention(CU, qs, ks, v, None, eV=np.zeros((1, T), np.int32), causal=False, softmax_scale=LN2,
                         quant_p=True, quant_ds=False, quant_pt=False, out_round=0)
    for (i, j), want in _phat_hand().items():
        got = r["O"][S0 + i, 0, j]
        assert got == pytest.approx(want, rel=1e-14, abs=0.0), (i, j, got, want)


def _phat_reading(row_block, col_block):
    _, _, _, x = _phat_case()
    a = np.exp2(x)
    l = a.sum(axis=1)
    p = _quantize_blocks(a, row_block, col_block)
    return {k: p[k] / l[k[0]] for k in _phat_hand()}


def test_phat_wrong_readings_miss_the_hand_values():
    hand = _phat_hand()
    ok = _phat_reading(ROW, LOCAL32)
    assert all(ok[k] == pytest.approx(hand[k], rel=1e-14, abs=0.0) for k in hand)
    for wrong in ((ROW, ABS32), (ROW, LOCAL16), (LOCAL32, LOCAL32)):
        got = _phat_reading(*wrong)
        assert any(got[k] != pytest.approx(hand[k], rel=1e-9, abs=1e-30) for k in hand), wrong


# ---------------------------------------------------------------------------
# dS^: 32x32 document-local blocks (default); exact option: per (row, 32 keys)
# for dQ, 32x32 for dK.
# ---------------------------------------------------------------------------
def _ds_case():
    """Zero scores (uniform P = 1/70 over document 1, non-causal), P^ and P~
    unquantized.  V_j[0] = v_j with v_0 = 1, v_1 = -1, v_20 = 2^-14,
    v_21 = -2^-14 (sum exactly 0, so O = 0 and D = 0); dO_i[0] = g_i with
    g_0 = 1, g_20 = 2^-5.  Then dS_ij = fl(1/70) g_i v_j exactly.  K_j = e_j
    and Q_i = e_i, softmax scale 1: dQ_i[j] = dS^q_ij and dK_j[i] = dS^k_ij."""
    z = np.zeros((T, 1, D))
    v = z.copy()
    for j, val in ((0, 1.0), (1, -1.0), (20, 2.0 ** -14), (21, -(2.0 ** -14))):
        v[S0 + j, 0, 0] = val
    do = z.copy()
    do[S0 + 0, 0, 0] = 1.0
    do[S0 + 20, 0, 0] = 2.0 ** -5
    q = z.copy()
    k = z.copy()
    for t in range(L1):
        q[S0 + t, 0, t] = 1.0
        k[S0 + t, 0, t] = 1.0
    ds = np.zeros((L1, L1))
    g = {0: 1.0, 20: 2.0 ** -5}
    vv = {0: 1.0, 1: -1.0, 20: 2.0 ** -14, 21: -(2.0 ** -14)}
    for i, gi in g.items():
        for j, vj in vv.items():
            ds[i, j] = (1.0 / 70.0) * gi * vj
    return z, q, k, v, do, ds


# fl(1/70) = 0.9143 * 2^-6, so a block holding it takes exponent -6 - 8 = -14
# and fl(1/70) * 2^14 = 234.06 rounds to 240 (E4M3 step 16 in [128, 256)).
# In the same block: 2^-14 fl(1/70) 2^14 = 0.01429 = 7.31 * 2^-9 is
# subnormal and rounds to 7 * 2^-9; 2^-5 fl(1/70) 2^14 = 7.31 rounds to 7.5
# (step 0.5 in [4, 8)); 2^-19 fl(1/70) 2^14 = 4.5e-4 is below 2^-10, half the
# smallest subnormal, and becomes 0.  In a (row 20, 32 keys) block the largest
# entry is 2^-5 fl(1/70): exponent -19, (20, 0) -> 240 * 2^-19 and (20, 20)
# -> 7 * 2^-9 * 2^-19 (the same subnormal rounding as (0, 20)).  A block that
# held (20, 20) without the larger entries would round it like 234.06 -> 240.
DS_HAND = {(0, 0): 240.0 * 2 ** -14, (0, 1): -240.0 * 2 ** -14, (0, 20): 7.0 * 2 ** -23,
           (0, 21): -7.0 * 2 ** -23, (20, 0): 7.5 * 2 ** -14, (20, 1): -7.5 * 2 ** -14,
           (20, 20): 0.0, (20, 21): 0.0}
DSQ_EXACT_HAND = dict(DS_HAND)
DSQ_EXACT_HAND.update({(20, 0): 240.0 * 2 ** -19, (20, 1): -240.0 * 2 ** -19, (20, 20): 7.0 * 2 ** -28,
                       (20, 21): -7.0 * 2 ** -28})


def _run_ds(exact):
    z, q, k, v, do, _ = _ds_case()
    return oracle.attention(CU, q, k, v, do, Qs=z, Ks=z, causal=False, softmax_scale=1.0, quant_p=False,
                            quant_ds=True, quant_pt=False, exact=exact, out_round=0)


def test_ds_blocks_are_32x32_document_local():
    r = _run_ds(exact=False)
    for (i, j), want in DS_HAND.items():
        assert r["dQ"][S0 + i, 0, j] == want, ("dQ", i, j)
        assert r["dK"][S0 + j, 0, i] == want, ("dK", i, j)


def test_ds_exact_option_rows_for_dq_blocks_for_dk():
    r = _run_ds(exact=True)
    for (i, j), want in DSQ_EXACT_HAND.items():
        assert r["dQ"][S0 + i, 0, j] == want, ("dQ", i, j)
    for (i, j), want in DS_HAND.items():
        assert r["dK"][S0 + j, 0, i] == want, ("dK", i, j)


def test_ds_wrong_readings_miss_the_hand_values():
    ds = _ds_case()[-1]
    pick = lambda m, hand: {k: m[k] for k in hand}
    assert pick(_quantize_blocks(ds, LOCAL32, LOCAL32), DS_HAND) == DS_HAND
    assert pick(_quantize_blocks(ds, ROW, LOCAL32), DSQ_EXACT_HAND) == DSQ_EXACT_HAND
    for wrong in ((ABS32, ABS32), (LOCAL16, LOCAL16), (ROW, LOCAL32)):
        assert pick(_quantize_blocks(ds, *wrong), DS_HAND) != DS_HAND, wrong
    for wrong in ((LOCAL32, LOCAL32), (ROW, ABS32), (ROW, LOCAL16)):
        assert pick(_quantize_blocks(ds, *wrong), DSQ_EXACT_HAND) != DSQ_EXACT_HAND, wrong


# ---------------------------------------------------------------------------
# P~: 32x32 document-local blocks.
# ---------------------------------------------------------------------------
def _pt_case():
    """Non-causal scores of document 1 (x = dot product): row 0 sees key 0 at
    0; row 20 sees key 55 at 0 and key 20 at -19; every other row sees key
    69 at 0; everything else is at -60.  V = 0 (so dS = 0), P^ unquantized,
    dO_i = e_i: dV_j[i] = P~_ij."""
    qs = np.zeros((T, 1, D))
    ks = np.zeros((T, 1, D))
    for i in range(L1):
        qs[S0 + i, 0, 0 if i == 0 else 1 if i == 20 else 2] = 1.0
    ks[S0:S0 + L1, 0, :3] = -60.0
    ks[S0 + 0, 0, 0] = 0.0
    ks[S0 + 55, 0, 1] = 0.0
    ks[S0 + 20, 0, 1] = -19.0
    ks[S0 + 69, 0, 2] = 0.0
    do = np.zeros((T, 1, D))
    for i in range(L1):
        do[S0 + i, 0, i] = 1.0
    x = np.full((L1, L1), -60.0)
    for i in range(L1):
        x[i, 69] = 0.0
    x[0] = -60.0
    x[0, 0] = 0.0
    x[20] = -60.0
    x[20, 55], x[20, 20] = 0.0, -19.0
    return qs, ks, do, x


# Pn(0, 0) = 1 (l_0 rounds to 1): the block of rows 0-31 x keys 0-31 takes
# exponent -8, so Pn(20, 20) = 2^-19 / (1 + 2^-19) becomes 0 and Pn(0, 0)
# stays 1.  Pn(20, 55) = 1 - 2^-19 + ... is the largest of rows 0-31 x keys
# 32-63: exponent -8, code 256, P~ = 1.  Rows 1-19 see key 69 with Pn = 1.
PT_HAND = {(0, 0): 1.0, (20, 20): 0.0, (20, 55): 1.0, (7, 69): 1.0}


def test_pt_blocks_are_32x32_document_local():
    qs, ks, do, _ = _pt_case()
    z = np.zeros((T, 1, D))
    r = oracle.attention(CU, z, z, z, do, Qs=qs, Ks=ks, causal=False, softmax_scale=LN2, quant_p=False,
                         quant_ds=False, quant_pt=True, out_round=0)
    for (i, j), want in PT_HAND.items():
        assert r["dV"][S0 + j, 0, i] == want, (i, j)


def test_pt_wrong_readings_miss_the_hand_values():
    _, _, _, x = _pt_case()
    a = np.exp2(x)
    pn = a / a.sum(axis=1, keepdims=True)
    pick = lambda m: {k: m[k] for k in PT_HAND}
    assert pick(_quantize_blocks(pn, LOCAL32, LOCAL32)) == PT_HAND
    for wrong in ((ABS32, ABS32), (LOCAL16, LOCAL16), (ROW, LOCAL32)):
        assert pick(_quantize_blocks(pn, *wrong)) != PT_HAND, wrong


# ---------------------------------------------------------------------------
# The whole call: packed documents == each document alone, bit for bit.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("exact", [False, True])
def test_packed_call_equals_each_document_alone(exact):
    w = synth.custom([13] + LENS, H=2, Hkv=1, d=64, seed=91)
    q, k, v, do = (w.tensor(n) for n in ("q", "k", "v", "do"))
    full = oracle.train_call(q, k, v, do, w.cu_seqlens, exact=exact)
    per_token = ("O", "dQ", "dK", "dV", "q_codes", "k_codes", "v_codes", "do_codes")
    per_head = ("q_scales", "k_scales", "v_scales", "do_scales", "D", "lse2")
    cu = w.cu_seqlens
    for s, e in zip(cu[:-1], cu[1:]):
        sl = lambda a: np.ascontiguousarray(a[s:e])
        one = oracle.train_call(sl(q), sl(k), sl(v), sl(do), np.array([0, e - s], np.int32), exact=exact)
        for n in per_token:
            assert np.array_equal(full[n][s:e], one[n]), (n, s, e)
        for n in per_head:
            assert np.array_equal(full[n][:, s:e], one[n]), (n, s, e)
