"""The allocation-free work-list builder, flamia_plan_noalloc.

Some callers cannot allocate device memory (a CUDA graph being captured, an
embedding without an allocator, a framework that owns every allocation); this
entry point keeps its scratch in a library-held device array instead of a
caller workspace.  Its work lists must equal those of flamia_plan, call after
call, whether it runs alone in a fresh process or after every other test.
This file sorts last so that a run stopping at the first failure has already
run every other test."""
import numpy as np
import pytest
import torch

import precision_causal_attention_token_gb300 as fl
import synth

pytestmark = pytest.mark.gpu


def _a256(x):
    return (x + 255) // 256 * 256


def _lists_from_workspace(ws, T, n_seq):
    # flamia_plan's workspace: header (256 B), tile prefix, 32-block prefix,
    # forward items, backward items (int32 pairs)
    max_items = (T + 127) // 128 + n_seq
    o = _a256(256 + 4 * (n_seq + 1))
    o = _a256(o + 4 * (n_seq + 1))
    fwd = o
    bwd = _a256(o + 8 * max_items)
    host = ws.cpu().numpy()
    n = int(host[:16].view(np.int32)[2])
    f = host[fwd:fwd + 8 * n].view(np.int32).reshape(-1, 2)
    b = host[bwd:bwd + 8 * n].view(np.int32).reshape(-1, 2)
    return n, f, b


def _host_lists(lens, causal):
    """The longest-first order by definition: cost descending, ties in item order."""
    items = [(d, t) for d, l in enumerate(lens) for t in range((l + 127) // 128)]
    nt = {d: (l + 127) // 128 for d, l in enumerate(lens)}
    fc = lambda it: (it[1] + 1) if causal else nt[it[0]]
    bc = lambda it: (nt[it[0]] - it[1]) if causal else nt[it[0]]
    f = sorted(range(len(items)), key=lambda i: (-fc(items[i]), i))
    b = sorted(range(len(items)), key=lambda i: (-bc(items[i]), i))
    return np.array([items[i] for i in f], np.int32), np.array([items[i] for i in b], np.int32)


def _check(lens, causal, heads=(4, 2)):
    import __graft_entry__
    __graft_entry__.build()
    T = int(sum(lens))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device="cuda")
    prob = fl.make_problem(T, heads[0], heads[1], 128, cu, causal=causal)
    ws = torch.full((fl.flamia_workspace_size(prob),), 0xA5, dtype=torch.uint8, device="cuda")
    fl.flamia_plan(prob, ws)
    max_items = (T + 127) // 128 + len(lens)
    fwd = torch.full((max_items, 2), -1, dtype=torch.int32, device="cuda")
    bwd = torch.full((max_items, 2), -1, dtype=torch.int32, device="cuda")
    n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    fl.flamia_plan_noalloc(prob, fwd, bwd, n)
    torch.cuda.synchronize()
    n_ref, f_ref, b_ref = _lists_from_workspace(ws, T, len(lens))
    assert int(n.item()) == n_ref > 0
    assert np.array_equal(fwd[:n_ref].cpu().numpy(), f_ref)
    assert np.array_equal(bwd[:n_ref].cpu().numpy(), b_ref)
    hf, hb = _host_lists(lens, causal)
    assert np.array_equal(f_ref, hf) and np.array_equal(b_ref, hb)


def test_noalloc_plan_matches_workspace_plan_twice():
    # calls in a row, different problems: the shared scratch keeps no stale state
    _check(synth.workload(3).seqlens, causal=True)
    _check([1, 300, 0, 129, 128, 4000, 31] + [1] * 2000, causal=False)
    _check(synth.workload(3).seqlens, causal=True)


@pytest.mark.parametrize("causal", [True, False])
def test_noalloc_plan_multi_pass_after_larger_problem(causal):
    # several merge passes over lists that are mostly padding, right after a
    # larger problem: the shared scratch then holds that problem's keys, some
    # smaller than this problem's padding keys
    _check([128] * 9000, causal=causal, heads=(1, 1))
    _check([128] * 3837, causal=causal, heads=(1, 1))
    _check([128] * 3837, causal=not causal, heads=(1, 1))


def test_noalloc_plan_rejects_oversized_problems():
    T = 128 * 70000
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    prob = fl.make_problem(T, 1, 1, 128, cu)
    dummy = torch.empty((1, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(fl.FlamiaError) as e:
        fl.flamia_plan_noalloc(prob, dummy, dummy, dummy[0])
    assert e.value.status == fl.ERR_UNSUPPORTED
