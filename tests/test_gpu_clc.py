"""Work items handed out by cluster launch control (the `clc` option; FLAMIA
summary §3.6.2 Load-Balanced Scheduling, close reading 四 4.4 GPU-side
scheduling): the grid has one CTA per work item, and a CTA that has finished
its item cancels a CTA that has not been launched yet and takes its item.

* parity with the oracle on small ragged, GQA, non-causal, d = 64 and mixed
  path cases, with FP16 and fp32 dQ partials (the same bar as the persistent
  grid);
* against the persistent grid on the same inputs: every item is computed by
  one CTA whichever CTA it is, so O, m, l, dK, dV and the mixed path's dQ
  (its dQ kernel sums in a fixed order) are bit-identical; the default dQ
  differs only by the order of its partials' additions;
* at full size on the packed workload (ragged documents up to 8192 tokens),
  where most items are taken over by cancellation.
"""
import numpy as np
import pytest
import torch

import oracle
import precision_causal_attention_token_gb300 as fl
import synth
from gpu_helpers import compare_all, np_of, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    ("ragged packed bf16", synth.custom([300, 45, 129, 1, 600], H=2, d=128, seed=801), {}, True),
    ("GQA H=4 Hkv=2 fp32 partials", synth.custom([257, 130, 64], H=4, Hkv=2, d=128, seed=802), {}, False),
    ("non-causal", synth.custom([200, 77, 129], H=2, d=128, seed=803), {"causal": False}, True),
    ("d=64", synth.custom([190, 66, 300], H=2, Hkv=1, d=64, seed=804), {}, True),
    ("tiny fp32 d=64", synth.workload(1), {}, False),
]


@pytest.mark.parametrize("name,w,kw,dq16", CASES, ids=[c[0] for c in CASES])
def test_clc_parity_small(name, w, kw, dq16):
    tc = run_gpu(w, clc=True, dq_fp16=dq16, **kw)
    ref = run_oracle(w, dq_fp16=dq16, **kw)
    names = ("O", "dQ", "dK", "dV")
    compare_all(names, {n: getattr(tc, n) for n in names}, ref)
    lse = np_of(tc.m) + np.log2(np_of(tc.l))
    assert np.abs(lse - ref["lse2"]).max() < 1e-3


def test_clc_mixed_path_parity_and_identity():
    w = synth.custom([300, 45, 129, 1, 600], H=2, d=128, seed=805)
    a = run_gpu(w, clc=True, path=fl.PATH_NVFP4_FP8)
    ref = run_oracle(w, path=oracle.PATH_NVFP4_FP8)
    names = ("O", "dQ", "dK", "dV")
    compare_all(names, {n: getattr(a, n) for n in names}, ref)
    b = run_gpu(w, path=fl.PATH_NVFP4_FP8)
    for n in ("O", "m", "l", "dQ", "dK", "dV"):
        assert torch.equal(getattr(a, n), getattr(b, n)), n


@pytest.mark.parametrize("kw,okw", [({"hadamard": True}, {"hadamard": True}),
                                      ({"path": fl.PATH_NVFP4_FP8}, {"path": oracle.PATH_NVFP4_FP8})],
                         ids=["hadamard", "mixed d=64"])
def test_clc_with_other_options(kw, okw):
    # the scheduler under the rotated-operand option and the mixed path at d = 64
    d = 128 if "hadamard" in kw else 64
    w = synth.custom([300, 45, 129, 1, 600], H=2, d=d, seed=807)
    tc = run_gpu(w, clc=True, **kw)
    ref = run_oracle(w, **okw)
    names = ("O", "dQ", "dK", "dV")
    compare_all(names, {n: getattr(tc, n) for n in names}, ref)


def _same_up_to_dq_order(a, b, dq16):
    for n in ("O", "m", "l", "dK", "dV"):
        assert torch.equal(getattr(a, n), getattr(b, n)), n
    # dQ: the same partials added in another order; FP16 adds round at each
    # step (2^-11 of the running sum), fp32 ones far less; the stored bf16
    # values may then differ by their own rounding
    x, y = np_of(a.dQ), np_of(b.dQ)
    rowmax = np.abs(y).max(axis=-1, keepdims=True) + 1e-30
    tol = (2.0 ** -6 if dq16 else 2.0 ** -7)
    assert (np.abs(x - y) <= tol * rowmax).all()


@pytest.mark.parametrize("dq16", [True, False])
def test_clc_matches_persistent_grid(dq16):
    # more items than SMs in both kernels: 73 tiles x 4 heads
    w = synth.custom([3000, 700, 129, 5000, 64], H=4, d=128, seed=806)
    a = run_gpu(w, clc=True, dq_fp16=dq16)
    b = run_gpu(w, dq_fp16=dq16)
    _same_up_to_dq_order(a, b, dq16)


def test_clc_full_size_packed_workload():
    w = synth.workload(3)
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    inputs = [torch.randn(w.T, h, w.d, generator=g, device=dev).to(torch.bfloat16)
              for h in (w.H, w.Hkv, w.Hkv, w.H)]
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    out = []
    for clc in (True, False):
        tc = fl.TrainCall(w.T, w.H, w.Hkv, w.d, cu, clc=clc)
        tc.run(*inputs)
        torch.cuda.synchronize()
        assert fl.flamia_get_device_status(tc.ws) == fl.OK
        out.append(tc)
    _same_up_to_dq_order(out[0], out[1], True)
