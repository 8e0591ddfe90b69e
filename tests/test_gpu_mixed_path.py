"""Mixed NVFP4/FP8 path on the GPU against the oracle's mixed path: QK^T from
the NVFP4 payload (E2M1 codes, E4M3 16-element block scales, fp32 per-token
scale), everything else MXFP8.  Same bar as the MXFP8 path: O, dQ, dK, dV
within 2e-2 of the row max-abs with cosine >= 0.9999 against the oracle's
result of the same quantization; the recomputed P^ equals the forward's."""
import numpy as np
import pytest
import torch

import oracle
import precision_causal_attention_token_gb300 as fl
import synth
from gpu_helpers import compare_all, cosine, np_of, o_rows_differ, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

NV = dict(path=fl.PATH_NVFP4_FP8)
NV_ORC = dict(path=oracle.PATH_NVFP4_FP8)


def _check(tc, ref, noise=None):
    names = ("O", "dQ", "dK", "dV")
    od = o_rows_differ(tc.O, ref["O"]) if noise is not None else None
    compare_all(names, {n: getattr(tc, n) for n in names}, ref, noise=noise, o_differs=od)
    lse = np_of(tc.m) + np.log2(np_of(tc.l))
    assert np.abs(lse - ref["lse2"]).max() < 1e-3


CASES = [
    ("ragged packed bf16", synth.custom([300, 45, 129, 1, 600], H=2, d=128, seed=701), {}),
    ("GQA H=4 Hkv=2", synth.custom([257, 130, 64], H=4, Hkv=2, d=128, seed=702), {}),
    ("non-causal", synth.custom([200, 77, 129], H=2, d=128, seed=703), {"causal": False}),
    ("d=64", synth.custom([190, 66, 300], H=2, d=64, seed=704), {}),
    ("tiny fp32 d=64", synth.workload(1), {}),
]


@pytest.mark.parametrize("name,w,kw", CASES, ids=[c[0] for c in CASES])
def test_mixed_parity_small(name, w, kw):
    tc = run_gpu(w, **kw, **NV)
    ref = run_oracle(w, **kw, **NV_ORC)
    # the NVFP4 payload and the MXFP8 codes both match the oracle bit for bit
    rc, rb, rg = oracle.quantize_nvfp4(w.tensor("q"))
    packed = tc.q4[0].cpu().numpy()
    got = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(rc.shape)
    assert (got == rc).all()
    assert (tc.q4[1].cpu().numpy() == rb).all()
    assert (tc.q4[2].cpu().numpy() == rg).all()
    assert (tc.q_codes.cpu().numpy() == ref["q_codes"]).all()
    _check(tc, ref)


@pytest.mark.parametrize("dq_fp16,deterministic,d", [(True, False, 128), (True, True, 128), (False, True, 128),
                                                    (True, False, 64), (True, True, 64)])
def test_mixed_fused_dq_options(dq_fp16, deterministic, d):
    # the mixed path's dQ goes through the fused backward's reduction like the
    # MXFP8 path's: FP16 or fp32 partials, unordered or in key-tile order
    w = synth.custom([300, 45, 129, 1, 600], H=4, Hkv=2, d=d, seed=708)
    tc = run_gpu(w, dq_fp16=dq_fp16, deterministic=deterministic, **NV)
    ref = run_oracle(w, dq_fp16=dq_fp16, **NV_ORC)
    _check(tc, ref)
    if deterministic:
        again = run_gpu(w, dq_fp16=dq_fp16, deterministic=deterministic, **NV)
        assert torch.equal(tc.dQ, again.dQ) and torch.equal(tc.dK, again.dK)


def test_nvfp4_payload_on_rounding_midpoints():
    # Each 16-element block holds the E2M1 rounding midpoints (0.25, 0.75,
    # ..., 5) and the largest value 6, scaled by a power of two per token, so
    # the block scale comes out at about 2^k and many quotients x / (s g) sit
    # within a few ulps of a step of the E2M1 rounding: the product with the
    # reciprocal cannot decide those and the exact quotient must.  The payload
    # still equals the oracle's byte for byte.
    T, H, d = 96, 2, 128
    mids = np.array([6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25, -5, -3.5, -2.5, -1.75, -1.25, -0.75, -0.25, 4],
                    np.float32)
    rng = np.random.default_rng(9)
    x = np.empty((T, H, d), np.float32)
    for t in range(T):
        for h in range(H):
            row = np.concatenate([rng.permutation(mids) for _ in range(d // 16)])
            x[t, h] = row * np.float32(2.0 ** int(rng.integers(-6, 7)))
    w = synth.custom([T], H=H, d=d, seed=710)
    v = w.tensor("v")
    tc = run_gpu(w, inputs=(x, x.copy(), v, w.tensor("do")), backward=False, **NV)
    rc, rb, rg = oracle.quantize_nvfp4(x)
    packed = tc.q4[0].cpu().numpy()
    got = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(rc.shape)
    assert (got == rc).all()
    assert (tc.q4[1].cpu().numpy() == rb).all()
    assert (tc.q4[2].cpu().numpy() == rg).all()


def test_mixed_outlier_channels():
    # x20 channels in Q and K: near one-hot softmax, dS cancels down to O's
    # rounding; compare against the oracle within its own O-rounding sensitivity
    w = synth.custom([180, 300], H=2, d=128, seed=705, outlier_channels=2)
    tc = run_gpu(w, **NV)
    q, k, v, do = (w.tensor(n) for n in ("q", "k", "v", "do"))
    ref = oracle.train_call(q, k, v, do, w.cu_seqlens, path=oracle.PATH_NVFP4_FP8, out_dtype="bf16")
    r64 = oracle.train_call(q, k, v, do, w.cu_seqlens, path=oracle.PATH_NVFP4_FP8, out_dtype="f64")
    _check(tc, ref, noise={n: ref[n] - r64[n] for n in ("dQ", "dK", "dV")})


def test_mixed_cosine_to_unquantized_reference():
    # the pages' band for the mixed path: O about 0.992, dQ about 0.991
    w = synth.custom([512, 300], H=2, d=128, seed=706)
    tc = run_gpu(w, **NV)
    q, k, v, do = (w.tensor(n) for n in ("q", "k", "v", "do"))
    ref = oracle.train_call(q, k, v, do, w.cu_seqlens, quantize=False)
    c = {n: cosine(np_of(getattr(tc, n)), ref[n]) for n in ("O", "dQ", "dK", "dV")}
    assert c["O"] >= 0.99 and c["dQ"] >= 0.985 and c["dK"] >= 0.985 and c["dV"] >= 0.99, c


def test_mixed_forward_and_backward_phat_bit_identical():
    """The backward rebuilds the forward's P^ codes and block exponents bit for
    bit on the mixed path too (same NVFP4 scores, same per-key factors)."""
    w = synth.custom([200, 70, 129], H=2, d=128, seed=707)
    dev = torch.device("cuda")
    q, k, v, do = (torch.from_numpy(w.tensor(n)).to(dev, torch.bfloat16) for n in ("q", "k", "v", "do"))
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    tc = fl.TrainCall(w.T, w.H, w.Hkv, w.d, cu, path=fl.PATH_NVFP4_FP8)
    tc.plan()
    buf = lambda: (torch.zeros(w.H, w.T, w.T, dtype=torch.uint8, device=dev),
                   torch.full((w.H, w.T, w.T), -7777, dtype=torch.int32, device=dev))
    cf, ef = buf()
    fl.flamia_debug_set_phat_dump(tc.ws, cf, ef)
    tc.forward(q, k, v)
    cb, eb = buf()
    fl.flamia_debug_set_phat_dump(tc.ws, cb, eb)
    tc.backward(do)
    fl.flamia_debug_set_phat_dump(tc.ws, None, None)
    torch.cuda.synchronize()
    assert fl.flamia_get_device_status(tc.ws) == fl.OK
    assert (ef != -7777).sum().item() > 0
    assert torch.equal(ef, eb)
    assert torch.equal(cf, cb)
    assert (cf != 0).float().mean().item() > 0.01


def test_mixed_full_size_sampled_against_oracle():
    """The mixed-path workload (4 x 32768 packed, log-normal documents, x20
    outlier channels) in full; the oracle recomputes one (document, head)
    slice, which equals the full call's outputs there."""
    w = synth.workload(4)
    q, k, v, do = (w.tensor(n) for n in ("q", "k", "v", "do"))
    tc = run_gpu(w, inputs=(q, k, v, do), **NV)
    lens = np.diff(w.cu_seqlens)
    doc = int(np.argsort(lens)[len(lens) // 2])
    head = 9
    s, e = int(w.cu_seqlens[doc]), int(w.cu_seqlens[doc + 1])
    sl = lambda a: np.ascontiguousarray(a[s:e, head:head + 1])
    cu1 = np.array([0, e - s], np.int32)
    ref = oracle.train_call(sl(q), sl(k), sl(v), sl(do), cu1, path=oracle.PATH_NVFP4_FP8, out_dtype="bf16")
    r64 = oracle.train_call(sl(q), sl(k), sl(v), sl(do), cu1, path=oracle.PATH_NVFP4_FP8, out_dtype="f64")
    got = {n: getattr(tc, n)[s:e, head:head + 1] for n in ("O", "dQ", "dK", "dV")}
    noise = {n: ref[n] - r64[n] for n in ("dQ", "dK", "dV")}
    compare_all(("O", "dQ", "dK", "dV"), got, ref, noise=noise, o_differs=o_rows_differ(got["O"], ref["O"]))
