"""GPU parity of the inference forward with bit-level exponentials (FLAMIA
summary, §3.7 Bit-Level Exponentials for Inference, §4.4) against the
oracle's forward of the same reading: O within the attention tests' per-row
bound and cosine, (m, l) against the oracle's base-2 log-sum-exp.  The P^
dump shows where the approximation acts: block exponents and the codes of
key pairs 5-7 of every 8 equal the default forward's, pairs 0-4 differ on a
share of the keys."""
import numpy as np
import pytest
import torch

import oracle
import precision_causal_attention_token_gb300 as fl
import synth
from gpu_helpers import compare, np_of, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    ("ragged packed bf16 d=128", synth.custom([300, 45, 129, 1, 600], H=2, d=128, seed=901), {}),
    ("GQA d=64 non-causal", synth.custom([257, 130, 64], H=4, Hkv=2, d=64, seed=902), {"causal": False}),
    ("tiny fp32 d=64", synth.workload(1), {}),
]


def _fwd(w, dumps=False, **kw):
    dev = torch.device("cuda:0")
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    dt = fl.BF16 if w.dtype == "bf16" else fl.F32
    tc = fl.TrainCall(w.T, w.H, w.Hkv, w.d, cu, in_dtype=dt, out_dtype=dt, **kw)
    tc._keep = cu
    tc.plan()
    dump = None
    if dumps:
        dump = (torch.zeros(w.H, w.T, w.T, dtype=torch.uint8, device=dev),
                torch.full((w.H, w.T, w.T), -7777, dtype=torch.int32, device=dev))
        fl.flamia_debug_set_phat_dump(tc.ws, *dump)
    tc.forward(*(to_dev(w.tensor(n), w.dtype) for n in ("q", "k", "v")))
    if dumps:
        fl.flamia_debug_set_phat_dump(tc.ws, None, None)
    torch.cuda.synchronize()
    st = fl.flamia_get_device_status(tc.ws)
    assert st == fl.OK, fl.status_string(st)
    return tc, dump


@pytest.mark.parametrize("name,w,kw", CASES, ids=[c[0] for c in CASES])
def test_bitexp_forward_parity(name, w, kw):
    tc, _ = _fwd(w, bitexp=True, **kw)
    q, k, v = (w.tensor(n) for n in ("q", "k", "v"))
    ref = oracle.train_call(q, k, v, None, w.cu_seqlens, out_dtype=w.dtype, bitexp=True, **kw)
    compare("O", tc.O, ref["O"])
    lse = np_of(tc.m) + np.log2(np_of(tc.l))
    assert np.abs(lse - ref["lse2"]).max() < 1e-3
    # the GPU follows the approximation, not the exact exponential: its mean
    # error to the bitexp oracle is well below its distance to the default one
    ex = oracle.train_call(q, k, v, None, w.cu_seqlens, out_dtype=w.dtype, **kw)
    o = np_of(tc.O)
    assert np.abs(o - ref["O"]).mean() < 0.5 * np.abs(o - ex["O"]).mean()


def test_bitexp_acts_on_pairs_0_to_4_only():
    w = synth.custom([300, 129, 64], H=2, d=128, seed=903)
    _, (cd, ed) = _fwd(w, dumps=True)
    _, (cb, eb) = _fwd(w, dumps=True, bitexp=True)
    assert torch.equal(ed, eb)
    vis = torch.zeros(w.T, w.T, dtype=torch.bool)
    approx = torch.zeros(w.T, w.T, dtype=torch.bool)
    for a, b in zip(w.cu_seqlens[:-1], w.cu_seqlens[1:]):
        for i in range(a, b):
            vis[i, a:i + 1] = True
            j = torch.arange(0, i + 1 - a)
            approx[i, a:i + 1] = ((j % 32) // 2) % 8 < 5
    cd, cb = cd.cpu(), cb.cpu()
    exact_pos = vis & ~approx
    assert torch.equal(cd[:, exact_pos], cb[:, exact_pos])
    diff = (cd[:, vis & approx] != cb[:, vis & approx]).float().mean().item()
    assert diff > 0.05, diff


def test_bitexp_backward_refused():
    w = synth.custom([64], H=1, d=128, seed=904)
    tc, _ = _fwd(w, bitexp=True)
    with pytest.raises(fl.FlamiaError):
        tc.backward(to_dev(w.tensor("do"), w.dtype))
