"""Shared helpers for the GPU parity tests: run one training call through the
C ABI on seeded inputs, run the oracle on the same inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import precision_causal_attention_token_gb300 as fl

# Tolerances for floating-point outputs against the oracle's result of the
# same quantization: max |err| <= 2e-2 of the row's max-abs, cosine >= 0.9999.
ROW_TOL = 2e-2
COS_TOL = 0.9999


def to_dev(a: np.ndarray, dtype: str, dev="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(dev, torch.bfloat16 if dtype == "bf16" else torch.float32)


def run_gpu(w, *, causal=True, exact=False, path=fl.PATH_MXFP8, deterministic=False, inputs=None,
            backward=True, causal_dq_scale=False, dq_fp16=False, hadamard=False, clc=False):
    dev = torch.device("cuda:0")
    q, k, v, do = inputs if inputs is not None else (w.tensor(n) for n in ("q", "k", "v", "do"))
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    dt = fl.BF16 if w.dtype == "bf16" else fl.F32
    tc = fl.TrainCall(w.T, w.H, w.Hkv, w.d, cu, causal=causal, exact=exact, path=path, in_dtype=dt,
                      out_dtype=dt, deterministic=deterministic, causal_dq_scale=causal_dq_scale, dq_fp16=dq_fp16,
                      hadamard=hadamard, clc=clc)
    tc.plan()
    tc.forward(to_dev(q, w.dtype), to_dev(k, w.dtype), to_dev(v, w.dtype))
    if backward:
        tc.backward(to_dev(do, w.dtype))
    torch.cuda.synchronize()
    st = fl.flamia_get_device_status(tc.ws)
    assert st == fl.OK, fl.status_string(st)
    tc._keep = cu
    return tc


def run_oracle(w, *, causal=True, exact=False, path=oracle.PATH_MXFP8, inputs=None, backward=True,
               dq_fp16=False, dq_causal_scale=False, hadamard=False):
    """The oracle's call on the same inputs (dq_fp16: FP16 dQ partials with the
    power-of-two prescale, as the GPU's dq_fp16 option)."""
    q, k, v, do = inputs if inputs is not None else (w.tensor(n) for n in ("q", "k", "v", "do"))
    return oracle.train_call(q, k, v, do if backward else None, w.cu_seqlens, causal=causal, exact=exact,
                             path=path, out_dtype=w.dtype, dq_fp16=dq_fp16, dq_causal_scale=dq_causal_scale,
                             hadamard=hadamard)


def np_of(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


# Outputs whose oracle value cancels down to the rounding of O before
# D = <dO^, O> (near one-hot softmax rows, from x20 outlier channels in Q and
# K) get, on top of ROW_TOL, NOISE_K times the row's largest oracle-only
# sensitivity to that rounding.  Why 4: the oracle's noise is the change
# between O rounded to bf16 and O kept exact, at most half a bf16 ulp per
# element; the GPU rounds an fp32 O whose last bits differ from the oracle's
# fp64 O, so an element of its stored O can sit one whole ulp from the
# oracle's stored O (twice the per-element deviation), and the row sum
# D_i = sum_k dO_ik O_ik can add those deviations with the same sign where the
# oracle's half-ulp errors partly cancel (another factor of two).
NOISE_K = 4.0


def compare_all(names, got, want, noise=None, o_differs=None, **kw):
    """compare() for several outputs; every failure is reported before the
    test fails, so one run shows all of them."""
    errors = []
    for n in names:
        try:
            compare(n, got[n], want[n], noise=None if noise is None else noise.get(n),
                    o_differs=o_differs if n == "dQ" else None, **kw)
        except AssertionError as e:
            errors.append(str(e))
    assert not errors, "; ".join(errors)


def compare(name, got, want, row_tol=ROW_TOL, cos_tol=COS_TOL, rows=None, noise=None, o_differs=None):
    """Per-row (last axis) max-error bound and whole-tensor cosine.

    noise: the oracle's own change in this output when only the rounding of
    O before D = <dO, O> changes (O stored in the output dtype vs kept in
    fp64), same shape as `want`.  When given, each row may in addition differ
    by NOISE_K times that row's largest noise, and the cosine bound becomes
    the oracle's own cosine (want - noise against want) with its deficit
    multiplied by NOISE_K, if that is lower.  All of it comes from the oracle."""
    g = np_of(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    r = np.asarray(want, np.float64)
    nz = None if noise is None else np.asarray(noise, np.float64)
    if rows is not None:
        g, r = g[rows], r[rows]
        nz = None if nz is None else nz[rows]
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    err = np.abs(g - r)
    rowmax = np.abs(r).max(axis=-1, keepdims=True)
    floor = 1e-6 * max(np.abs(r).max(), 1e-30)
    allow = row_tol * np.maximum(rowmax, floor)
    if nz is not None and np.abs(nz).max() > 0:
        allow = allow + NOISE_K * np.abs(nz).max(axis=-1, keepdims=True)
        cos_tol = min(cos_tol, 1.0 - NOISE_K * (1.0 - cosine(r - nz, r)))
    ratio = err / allow
    worst = float(ratio.max()) if err.size else 0.0
    gg, rr = g.ravel(), r.ravel()
    denom = np.sqrt((gg @ gg) * (rr @ rr))
    cos = float(gg @ rr / denom) if denom > 0 else 1.0
    row_ratio = ratio.max(axis=-1)
    over = row_ratio > 1.0
    if over.any():
        flat = np.argsort(row_ratio.ravel())[::-1][:5]
        print(f"{name}: {int(over.sum())} of {over.size} rows over the allowance; worst (flattened row, "
              f"err / allowance):", [(int(i), float(row_ratio.ravel()[i])) for i in flat])
    if o_differs is not None and nz is not None and over.any():
        # dQ rows whose stored O differs from the oracle's: there D and the
        # cancelling dS follow the GPU's own O (see NOISE_K); such rows may
        # exceed the allowance, but only those, at most 1% of the rows, and
        # by no more than 10% of the tensor's max-abs
        od = np.asarray(o_differs, bool)
        od = od[rows] if rows is not None else od
        assert od.shape == over.shape, (od.shape, over.shape)
        unexplained = over & ~od
        assert not unexplained.any(), f"{name}: {int(unexplained.sum())} rows over the allowance with O equal"
        assert over.sum() <= max(1, 0.01 * over.size), f"{name}: {int(over.sum())} rows over the allowance"
        rel = float(err[over].max() / max(np.abs(r).max(), 1e-30))
        assert rel <= 0.1, f"{name}: an excepted row is off by {rel:.3e} of the tensor's max-abs"
    else:
        assert worst <= 1.0, f"{name}: max |err| exceeds the per-row allowance by {worst:.3f}x"
    assert cos >= cos_tol, f"{name}: cosine {cos:.7f} < {cos_tol:.7f}"
    return worst, cos


def o_rows_differ(tc_O, ref_O):
    """Rows (token, head) whose stored O differs from the oracle's stored O."""
    return np.any(np_of(tc_O) != np.asarray(ref_O, np.float64), axis=-1)


def o_rounding_noise(w, *, causal=True, exact=False, inputs=None, hadamard=False):
    """Oracle-only sensitivity of dQ/dK/dV to rounding O before D."""
    a = run_oracle(w, causal=causal, exact=exact, inputs=inputs, hadamard=hadamard)
    q, k, v, do = inputs if inputs is not None else (w.tensor(n) for n in ("q", "k", "v", "do"))
    b = oracle.train_call(q, k, v, do, w.cu_seqlens, causal=causal, exact=exact, out_dtype="f64", hadamard=hadamard)
    return a, {n: a[n] - b[n] for n in ("dQ", "dK", "dV")}


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / np.sqrt((a @ a) * (b @ b)))
