"""GPU parity of the Hadamard option (FLAMIA summary §4.3 and abstract: the
fused quantizer rotates Q and K; close reading 四 4.4: the rotation spreads
outlier channels and keeps dot products) against the oracle's rotated call:
Q/K codes and scale bytes bit-exact (the rotation runs in fp32 in the same
stage order on both sides), O, dQ, dK, dV within the attention tests' per-row
bound and cosine, on every dQ path (fp32 partials, FP16 partials, the
deterministic and exact options).  On x20 outlier channels the rotated call
is closer to the unquantized output than the plain one."""
import numpy as np
import pytest

import oracle
import precision_causal_attention_token_gb300 as fl
import synth
from gpu_helpers import compare_all, cosine, np_of, o_rounding_noise, o_rows_differ, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    ("ragged packed bf16 d=128", synth.custom([300, 45, 129, 1, 600], H=2, d=128, seed=951), {}),
    ("GQA d=64 non-causal", synth.custom([257, 130, 64], H=4, Hkv=2, d=64, seed=952), {"causal": False}),
    ("exact option", synth.custom([256, 100, 33], H=2, d=128, seed=953), {"exact": True}),
    ("deterministic dQ", synth.custom([300, 129], H=2, Hkv=1, d=128, seed=954), {"deterministic": True}),
    ("FP16 dQ partials, causal scale", synth.custom([400, 77], H=2, d=128, seed=955),
     {"dq_fp16": True, "causal_dq_scale": True}),
    ("tiny fp32 d=64", synth.workload(1), {}),
    ("outlier channels", synth.custom([180, 300], H=2, d=128, seed=956, outlier_channels=2), {}),
]

_ORACLE_KW = {"causal", "exact"}


@pytest.mark.parametrize("name,w,kw", CASES, ids=[c[0] for c in CASES])
def test_hadamard_parity(name, w, kw):
    tc = run_gpu(w, hadamard=True, **kw)
    okw = {k: v for k, v in kw.items() if k in _ORACLE_KW}
    if kw.get("dq_fp16"):
        okw.update(dq_fp16=True, dq_causal_scale=kw.get("causal_dq_scale", False))
    noise = None
    if w.outlier_channels:
        ref, noise = o_rounding_noise(w, hadamard=True, **okw)
    else:
        ref = run_oracle(w, hadamard=True, **okw)
    for n in ("q", "k", "v"):
        assert (getattr(tc, f"{n}_codes").cpu().numpy() == ref[f"{n}_codes"]).all(), n
        assert (getattr(tc, f"{n}_scales").cpu().numpy() == ref[f"{n}_scales"]).all(), n
    names = ("O", "dQ", "dK", "dV")
    od = o_rows_differ(tc.O, ref["O"]) if noise is not None else None
    compare_all(names, {n: getattr(tc, n) for n in names}, ref, noise=noise, o_differs=od)
    lse = np_of(tc.m) + np.log2(np_of(tc.l))
    assert np.abs(lse - ref["lse2"]).max() < 1e-3


def test_hadamard_helps_on_outlier_channels():
    w = synth.custom([300, 257], H=2, Hkv=1, d=128, seed=41, outlier_channels=2)
    q, k, v, do = (w.tensor(n) for n in ("q", "k", "v", "do"))
    ref = oracle.train_call(q, k, v, do, w.cu_seqlens, out_dtype="f64", quantize=False)
    a = run_gpu(w)
    b = run_gpu(w, hadamard=True)
    for n in ("O", "dV"):
        ca, cb = cosine(np_of(getattr(a, n)), ref[n]), cosine(np_of(getattr(b, n)), ref[n])
        assert 1.0 - cb < 0.5 * (1.0 - ca), (n, ca, cb)
