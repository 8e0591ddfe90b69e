"""GPU quantizer parity: codes and scale bytes bit-exact against the oracle
(token-block, per-token, per-key V, the NVFP4 operand), D within fp32 rounding."""
import numpy as np
import pytest
import torch

import oracle
import precision_causal_attention_token_gb300 as fl
import synth
from gpu_helpers import np_of, to_dev

pytestmark = pytest.mark.gpu


def _quantize(w, exact=False, path=fl.PATH_MXFP8, heads_slice=None):
    dev = torch.device("cuda:0")
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    dt = fl.BF16 if w.dtype == "bf16" else fl.F32
    tc = fl.TrainCall(w.T, w.H, w.Hkv, w.d, cu, exact=exact, path=path, in_dtype=dt, out_dtype=dt)
    tc.plan()
    q, k, v = (w.tensor(n) for n in ("q", "k", "v"))
    fl.flamia_quantize(tc.prob, fl.ROLE_QKV, [to_dev(q, w.dtype), to_dev(k, w.dtype), to_dev(v, w.dtype)], None,
                       [tc.opq, tc.opk, tc.opv], None, tc.ws)
    torch.cuda.synchronize()
    assert fl.flamia_get_device_status(tc.ws) == fl.OK
    return tc, (q, k, v), cu


CASES = [
    ("ragged packed, bf16, outliers", synth.custom([37, 100, 5, 64, 1, 200, 33], H=3, d=128, outlier_channels=2)),
    ("tiny fp32 d=64 one document", synth.workload(1)),
    ("GQA with an empty document", synth.custom([129, 0, 31, 300], H=4, Hkv=2, d=128, seed=808)),
]


@pytest.mark.parametrize("exact", [False, True])
@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_codes_and_scales_bit_exact(name, w, exact):
    tc, (q, k, v), _ = _quantize(w, exact=exact)
    blk = 1 if exact else 32
    for x, codes, scales in ((q, tc.q_codes, tc.q_scales), (k, tc.k_codes, tc.k_scales)):
        rc, rs = oracle.quantize_blocks(x, w.cu_seqlens, blk)
        assert (codes.cpu().numpy() == rc).all()
        assert (scales.cpu().numpy() == rs).all()
    rc, rs = oracle.quantize_blocks(v, w.cu_seqlens, 1)  # V: one exponent per key
    assert (tc.v_codes.cpu().numpy() == rc).all()
    assert (tc.v_scales.cpu().numpy() == rs).all()


def test_nvfp4_operand_bit_exact():
    w = synth.custom([37, 100, 5, 64, 200], H=2, d=128, outlier_channels=2, seed=77)
    tc, (q, k, v), _ = _quantize(w, path=fl.PATH_NVFP4_FP8)
    for x, (c4, s4, g4) in ((q, tc.q4), (k, tc.k4)):
        rc, rb, rg = oracle.quantize_nvfp4(x)
        packed = c4.cpu().numpy()
        lo, hi = packed & 0xF, packed >> 4
        got = np.stack([lo, hi], axis=-1).reshape(rc.shape)
        assert (got == rc).all()
        assert (s4.cpu().numpy() == rb).all()
        assert (g4.cpu().numpy() == rg).all()


@pytest.mark.parametrize("exact", [False, True])
def test_dO_codes_and_D(exact):
    w = synth.custom([40, 129, 3, 250], H=2, d=128, seed=31)
    dev = torch.device("cuda:0")
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    tc = fl.TrainCall(w.T, w.H, w.Hkv, w.d, cu, exact=exact)
    tc.plan()
    do = w.tensor("do")
    O = synth.round_to_bf16(synth.normal(99, 9, w.T * w.H * w.d).astype(np.float32)).reshape(w.T, w.H, w.d)
    Od = to_dev(O, "bf16")
    fl.flamia_quantize(tc.prob, fl.ROLE_DO, [to_dev(do, "bf16")], Od, [tc.opdo], tc.D, tc.ws)
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_blocks(do, w.cu_seqlens, 1 if exact else 32)
    assert (tc.do_codes.cpu().numpy() == rc).all()
    assert (tc.do_scales.cpu().numpy() == rs).all()
    D = oracle.compute_D(oracle.dequantize_blocks(rc, rs), O.astype(np.float64))
    got = np_of(tc.D)
    scale = np.abs(oracle.dequantize_blocks(rc, rs)).sum(-1).T * np.abs(O).max()
    assert (np.abs(got - D) <= 1e-6 * scale + 1e-30).all()


def test_full_size_batched_workload_sampled_heads():
    # 4 x 4096 tokens, H = 16, d = 128 (the timed workload); oracle on two heads
    w = synth.workload(2)
    tc, (q, k, v), _ = _quantize(w)
    for h in (0, 11):
        for x, codes, scales in ((q, tc.q_codes, tc.q_scales), (k, tc.k_codes, tc.k_scales)):
            rc, rs = oracle.quantize_blocks(x[:, h:h + 1], w.cu_seqlens, 32)
            assert (codes[:, h:h + 1].cpu().numpy() == rc).all()
            assert (scales[h:h + 1].cpu().numpy() == rs).all()
        rc, rs = oracle.quantize_blocks(v[:, h:h + 1], w.cu_seqlens, 1)
        assert (tc.v_codes[:, h:h + 1].cpu().numpy() == rc).all()
        assert (tc.v_scales[h:h + 1].cpu().numpy() == rs).all()
