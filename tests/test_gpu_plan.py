"""GPU work-list parity: the longest-first lists built on the GPU equal the host
sort of the same items (cost descending, ties in document/tile order)."""
import numpy as np
import pytest
import torch

import precision_causal_attention_token_gb300 as fl
import synth

pytestmark = pytest.mark.gpu


def _a256(x):
    return (x + 255) // 256 * 256


def _read_lists(tc, T, n_seq):
    # device workspace layout: header (256 B), tile prefix, 32-block prefix,
    # forward items, backward items (int32 pairs), sort keys, dQ accumulator
    max_items = (T + 127) // 128 + n_seq
    o = 256
    tile_prefix = o; o = _a256(o + 4 * (n_seq + 1))
    blk_prefix = o; o = _a256(o + 4 * (n_seq + 1))
    fwd = o; o = _a256(o + 8 * max_items)
    bwd = o
    ws = tc.ws.cpu().numpy()
    hdr = ws[:16].view(np.int32)
    n_items, n_blk = int(hdr[2]), int(hdr[3])
    f = ws[fwd:fwd + 8 * n_items].view(np.int32).reshape(-1, 2)
    b = ws[bwd:bwd + 8 * n_items].view(np.int32).reshape(-1, 2)
    tp = ws[tile_prefix:tile_prefix + 4 * (n_seq + 1)].view(np.int32)
    bp = ws[blk_prefix:blk_prefix + 4 * (n_seq + 1)].view(np.int32)
    return n_items, n_blk, f, b, tp, bp


def _host_lists(lens, causal):
    items = [(d, t) for d, l in enumerate(lens) for t in range((l + 127) // 128)]
    nt = {d: (l + 127) // 128 for d, l in enumerate(lens)}
    fc = lambda it: (it[1] + 1) if causal else nt[it[0]]
    bc = lambda it: (nt[it[0]] - it[1]) if causal else nt[it[0]]
    f = sorted(range(len(items)), key=lambda i: (-fc(items[i]), i))
    b = sorted(range(len(items)), key=lambda i: (-bc(items[i]), i))
    return [items[i] for i in f], [items[i] for i in b]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("wl", ["ragged", "packed3", "long5", "many_single"])
def test_worklist_matches_host_sort(wl, causal):
    if wl == "ragged":
        lens = [1, 300, 0, 129, 128, 4000, 31]
    elif wl == "packed3":
        lens = synth.workload(3).seqlens
    elif wl == "long5":
        lens = synth.workload(5).seqlens
    else:
        lens = [1] * 5000 + [3000]  # skew: one long document among many single tokens
    T = int(sum(lens))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device="cuda")
    prob = fl.make_problem(T, 2, 2, 128, cu, causal=causal)
    ws = torch.zeros(fl.flamia_workspace_size(prob), dtype=torch.uint8, device="cuda")

    class _TC:
        pass

    tc = _TC()
    tc.ws = ws
    fl.flamia_plan(prob, ws)
    torch.cuda.synchronize()
    n_items, n_blk, f, b, tp, bp = _read_lists(tc, T, len(lens))
    hf, hb = _host_lists(lens, causal)
    assert n_items == len(hf)
    assert n_blk == sum((l + 31) // 32 for l in lens)
    assert [tuple(x) for x in f] == hf
    assert [tuple(x) for x in b] == hb
    assert (tp == np.concatenate([[0], np.cumsum([(l + 127) // 128 for l in lens])])).all()
    assert (bp == np.concatenate([[0], np.cumsum([(l + 31) // 32 for l in lens])])).all()
    assert fl.flamia_get_device_status(ws) == fl.OK


@pytest.mark.parametrize("fill", [0x00, 0xA5])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("n_docs", [3837, 9000])
def test_worklist_multi_pass_with_padding(n_docs, causal, fill):
    """Several merge passes (sort_n = 8192 and 18432) over lists that are
    mostly padding: ceil(T/128) + n_seq bounds the item count at twice the real
    items.  The workspace starts as all 0x00 or all 0xA5 bytes, so a pass that
    left a slot unwritten would hand stale words to the next pass."""
    lens = [128] * n_docs
    T = int(sum(lens))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device="cuda")
    prob = fl.make_problem(T, 1, 1, 128, cu, causal=causal)
    ws = torch.full((fl.flamia_workspace_size(prob),), fill, dtype=torch.uint8, device="cuda")

    class _TC:
        pass

    tc = _TC()
    tc.ws = ws
    fl.flamia_plan(prob, ws)
    torch.cuda.synchronize()
    n_items, _, f, b, _, _ = _read_lists(tc, T, len(lens))
    hf, hb = _host_lists(lens, causal)
    assert n_items == len(hf) == n_docs
    assert [tuple(x) for x in f] == hf
    assert [tuple(x) for x in b] == hb
    assert fl.flamia_get_device_status(ws) == fl.OK


def test_bad_seqlens_reported_on_device():
    cu = torch.tensor([0, 50, 40, 100], dtype=torch.int32, device="cuda")  # decreasing
    prob = fl.make_problem(100, 1, 1, 128, cu)
    ws = torch.zeros(fl.flamia_workspace_size(prob), dtype=torch.uint8, device="cuda")
    fl.flamia_plan(prob, ws)
    assert fl.flamia_get_device_status(ws) == fl.ERR_BAD_SEQLENS
    fl.flamia_clear_device_status(ws)
    assert fl.flamia_get_device_status(ws) == fl.OK
