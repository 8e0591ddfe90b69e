"""C-ABI checks that need no GPU: the library loads, exports every entry point
that include/flamia.h declares, and rejects bad arguments on the host before
any launch."""
import os
import re

import pytest
import torch

import precision_causal_attention_token_gb300 as fl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "flamia.h")).read()
    return sorted(set(re.findall(r"\b(flamia_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return fl.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(fl.EXPORTED) <= set(names)


def _prob(**kw):
    cu = torch.tensor([0, 100, 228], dtype=torch.int32)
    base = dict(T=228, H=4, Hkv=2, d=128)
    base.update(kw)
    p = fl.make_problem(base["T"], base["H"], base["Hkv"], base["d"], cu)
    for k, v in kw.items():
        if k not in base or k in ("path", "in_dtype", "out_dtype"):
            setattr(p, k, v)
    return p, cu


def test_workspace_size_valid_and_invalid(lib):
    p, _ = _prob()
    n = fl.flamia_workspace_size(p)
    assert n > 228 * 4 * 128 * 2 + 228 * 4  # holds the FP16 dQ accumulator and the row prescales
    # the offsets tests read back lie inside the workspace, in layout order
    offs = [fl.flamia_debug_workspace_offset(p, r) for r in (fl.WS_FWD_ITEMS, fl.WS_BWD_ITEMS, fl.WS_DQ_PRESCALE)]
    assert 0 < offs[0] < offs[1] < offs[2] and offs[2] + 228 * 4 <= n
    assert fl.flamia_debug_workspace_offset(p, 99) == 0
    for bad in (dict(d=96), dict(H=3), dict(T=0), dict(Hkv=0)):
        q, _ = _prob(**bad)
        assert fl.flamia_workspace_size(q) == 0, bad
    q, _ = _prob()
    q.path = 7
    assert fl.flamia_workspace_size(q) == 0
    # the exact option is not offered on the mixed NVFP4/FP8 path
    q, _ = _prob()
    q.path, q.exact = fl.PATH_NVFP4_FP8, 1
    assert fl.flamia_workspace_size(q) == 0
    assert lib.flamia_plan(q, torch.empty(16, dtype=torch.uint8).data_ptr(), 1 << 30, None) == fl.ERR_UNSUPPORTED
    # the mixed path reads its score operands from the caller's NVFP4 payload:
    # no workspace of its own
    q, _ = _prob()
    q.path = fl.PATH_NVFP4_FP8
    assert fl.flamia_workspace_size(q) == n


def test_status_strings(lib):
    for s in range(7):
        assert fl.status_string(s)
    assert fl.status_string(fl.ERR_TIMEOUT) == "device wait timed out"


def test_host_validation_rejects_before_launch(lib):
    p, cu = _prob()
    ws = torch.empty(16, dtype=torch.uint8)
    # workspace too small -> reported without touching the device
    st = lib.flamia_plan(p, ws.data_ptr(), 16, None)
    assert st == fl.ERR_WORKSPACE_TOO_SMALL
    q, _ = _prob(d=80)
    assert lib.flamia_plan(q, ws.data_ptr(), 1 << 30, None) == fl.ERR_UNSUPPORTED
    q, _ = _prob(H=5)
    assert lib.flamia_plan(q, ws.data_ptr(), 1 << 30, None) == fl.ERR_INVALID_ARG
    # misaligned workspace pointer
    assert lib.flamia_plan(p, ws.data_ptr() + 1, 1 << 30, None) == fl.ERR_INVALID_ARG
    # null operands
    big = 1 << 40
    op = fl.Operand()
    assert lib.flamia_fwd(p, op, op, op, None, None, None, ws.data_ptr(), big, None) == fl.ERR_INVALID_ARG
    assert lib.flamia_get_device_status(None, None) == fl.ERR_INVALID_ARG


def test_misaligned_pointers_rejected_before_launch(lib):
    """Every device pointer must be 16-byte aligned (cu_seqlens 4-byte): the
    host rejects a misaligned scale vector, D, m or l without touching the
    device (the pointers below are never dereferenced)."""
    p, _ = _prob()
    big = 1 << 40
    ws = 1 << 20
    good = lambda: fl.Operand(0x10000, 0x20000, None, None, None)
    for field in ("codes", "scales"):
        bad = good()
        setattr(bad, field, getattr(bad, field) + 1)
        assert lib.flamia_fwd(p, bad, good(), good(), 0x30000, 0x40000, 0x50000, ws, big, None) == fl.ERR_INVALID_ARG
    for m, l in ((0x40004, 0x50000), (0x40000, 0x50008)):
        assert lib.flamia_fwd(p, good(), good(), good(), 0x30000, m, l, ws, big, None) == fl.ERR_INVALID_ARG
    ops = [good() for _ in range(4)]
    for D, m, l in ((0x60004, 0x40000, 0x50000), (0x60000, 0x40008, 0x50000), (0x60000, 0x40000, 0x5000c)):
        st = lib.flamia_bwd(p, ops[0], ops[1], ops[2], ops[3], D, m, l, 0x70000, 0x80000, 0x90000, ws, big, None)
        assert st == fl.ERR_INVALID_ARG


def test_withhold_hook_is_host_side(lib):
    # the hook only sets a host-side flag for the next launches (no device call)
    assert lib.flamia_debug_withhold_first_item(1) == fl.OK
    assert lib.flamia_debug_withhold_first_item(0) == fl.OK


def test_binding_raises_without_library(tmp_path):
    import importlib
    mod = importlib.import_module("precision_causal_attention_token_gb300")
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(RuntimeError):
            mod.load_library(str(tmp_path / "missing.so"))
    finally:
        mod._lib = saved


def test_bitexp_is_inference_only(lib):
    """The bit-level exponential forward ([SUM] §3.7) is offered on the MXFP8
    default option only, and flamia_bwd refuses it on the host (its P^ cannot
    be rebuilt by the backward).  No pointer below is dereferenced."""
    p, _ = _prob()
    p.bitexp = 1
    assert fl.flamia_workspace_size(p) > 0
    for field, val in (("exact", 1), ("path", fl.PATH_NVFP4_FP8)):
        q, _ = _prob()
        q.bitexp = 1
        setattr(q, field, val)
        assert fl.flamia_workspace_size(q) == 0, field
    good = lambda: fl.Operand(0x10000, 0x20000, None, None, None)
    ops = [good() for _ in range(4)]
    st = lib.flamia_bwd(p, ops[0], ops[1], ops[2], ops[3], 0x60000, 0x40000, 0x50000, 0x70000, 0x80000, 0x90000,
                        1 << 20, 1 << 40, None)
    assert st == fl.ERR_UNSUPPORTED


def test_hadamard_option_host_rules(lib):
    """The Hadamard option runs on the MXFP8 path only and adds the fp32 dK
    buffer of the back-rotation (4 T Hkv d bytes) to the workspace."""
    p, _ = _prob()
    n = fl.flamia_workspace_size(p)
    p.hadamard = 1
    assert fl.flamia_workspace_size(p) >= n + 4 * 228 * 2 * 128
    q, _ = _prob()
    q.hadamard, q.path = 1, fl.PATH_NVFP4_FP8
    assert fl.flamia_workspace_size(q) == 0
    # with FP16 dQ partials the dQ buffer stays fp32 (the back-rotation reads it)
    r, _ = _prob()
    r.dq_fp16 = 1
    n16 = fl.flamia_workspace_size(r)
    r.hadamard = 1
    assert fl.flamia_workspace_size(r) >= n16 + 2 * 228 * 4 * 128 + 4 * 228 * 2 * 128


def test_clc_option_host_rules(lib):
    """Cluster launch control hands out the items of every option but the two
    whose ordered dQ reduction needs them in list order (exact,
    deterministic); it changes nothing in the workspace."""
    p, _ = _prob()
    n = fl.flamia_workspace_size(p)
    p.clc = 1
    assert fl.flamia_workspace_size(p) == n
    for field in ("exact", "deterministic"):
        q, _ = _prob()
        q.clc = 1
        setattr(q, field, 1)
        assert fl.flamia_workspace_size(q) == 0, field
    r, _ = _prob()
    r.clc, r.path = 1, fl.PATH_NVFP4_FP8
    assert fl.flamia_workspace_size(r) > 0


def test_noalloc_plan_host_rules(lib):
    """flamia_plan_noalloc checks its arguments on the host before it makes
    any CUDA call: an invalid problem or a NULL output is rejected, and so is
    a problem larger than its fixed scratch (more than 65536 tiles plus
    documents).  No pointer below is dereferenced."""
    p, _ = _prob()
    a, b, n = 0x10000, 0x20000, 0x30000
    for args in ((None, b, n), (a, None, n), (a, b, None)):
        assert lib.flamia_plan_noalloc(p, *args, None) == fl.ERR_INVALID_ARG, args
    q, _ = _prob(H=3)
    assert lib.flamia_plan_noalloc(q, a, b, n, None) == fl.ERR_INVALID_ARG
    big, _ = _prob(T=128 * 70000)
    assert lib.flamia_plan_noalloc(big, a, b, n, None) == fl.ERR_UNSUPPORTED
