"""Failure detection without a GPU fault: every wait inside the attention
kernels is bounded (about 2 s).  A test hook makes each CTA's producer
withhold its first work item, so the other roles' waits for it run out.  The
kernel must then record FLAMIA_ERR_TIMEOUT in the workspace's status word and
exit cleanly (tensor memory released, nothing in flight), and the context
must stay usable: the next normal call returns OK and matches the oracle."""
import pytest
import torch

import precision_causal_attention_token_gb300 as fl
import synth
from gpu_helpers import compare, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def _call(w):
    dev = torch.device("cuda:0")
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    tc = fl.TrainCall(w.T, w.H, w.Hkv, w.d, cu)
    tc._keep = cu
    q, k, v, do = (to_dev(w.tensor(n), w.dtype) for n in ("q", "k", "v", "do"))
    return tc, (q, k, v, do)


def test_forward_wait_runs_out_and_reports_timeout():
    w = synth.custom([300, 129, 64], H=2, d=128, seed=811)
    tc, (q, k, v, do) = _call(w)
    tc.plan()
    fl.flamia_quantize(tc.prob, fl.ROLE_QKV, [q, k, v], None, [tc.opq, tc.opk, tc.opv], None, tc.ws)
    fl.flamia_debug_withhold_first_item(True)
    try:
        fl.flamia_fwd(tc.prob, tc.opq, tc.opk, tc.opv, tc.O, tc.m, tc.l, tc.ws)
        torch.cuda.synchronize()
    finally:
        fl.flamia_debug_withhold_first_item(False)
    assert fl.flamia_get_device_status(tc.ws) == fl.ERR_TIMEOUT
    # the plan clears the status word and the hook; the same workspace then works
    tc.run(q, k, v, do)
    torch.cuda.synchronize()
    assert fl.flamia_get_device_status(tc.ws) == fl.OK
    ref = run_oracle(w, dq_fp16=tc.dq_fp16)
    for name in ("O", "dQ", "dK", "dV"):
        compare(name, getattr(tc, name), ref[name])


def test_backward_wait_runs_out_and_reports_timeout():
    w = synth.custom([257, 100], H=2, Hkv=1, d=128, seed=812)
    tc, (q, k, v, do) = _call(w)
    tc.plan()
    tc.forward(q, k, v)
    fl.flamia_debug_withhold_first_item(True)
    try:
        tc.backward(do)
        torch.cuda.synchronize()
    finally:
        fl.flamia_debug_withhold_first_item(False)
    assert fl.flamia_get_device_status(tc.ws) == fl.ERR_TIMEOUT
    # a fresh workspace and call on the same context
    tc2 = run_gpu(w)
    ref = run_oracle(w)
    for name in ("O", "dQ", "dK", "dV"):
        compare(name, getattr(tc2, name), ref[name])
