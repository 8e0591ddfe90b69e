"""fp64 oracle of the FLAMIA training call — TEST INFRASTRUCTURE ONLY.

ctypes front end of ``flamia_oracle.cpp`` (plain single-threaded C++, fp64).
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package; the library path never does.  It shares no code
with the CUDA path: the two meet only in the seeded inputs of ``synth``.

Functions that have no independent pin say "parity unpinned" in their
docstring; every other one is pinned by a ``-m "not gpu"`` test.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "flamia_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PATH_MXFP8, PATH_NVFP4_FP8 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle to liboracle.so (g++, -O2, no FP contraction so x86 and Arm agree)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("Hkv", ctypes.c_int), ("d", ctypes.c_int),
                ("nseq", ctypes.c_int), ("causal", ctypes.c_int), ("softmax_scale", ctypes.c_double),
                ("quant_p", ctypes.c_int), ("quant_ds", ctypes.c_int), ("quant_pt", ctypes.c_int),
                ("exact", ctypes.c_int), ("out_round", ctypes.c_int), ("bitexp", ctypes.c_int),
                ("dq_fp16", ctypes.c_int),
                ("dq_causal_scale", ctypes.c_int)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            d, u, i, p = ctypes.c_double, ctypes.c_uint, ctypes.c_int, ctypes.c_void_p
            L.orc_e4m3_decode.restype, L.orc_e4m3_decode.argtypes = d, [u]
            L.orc_e4m3_encode.restype, L.orc_e4m3_encode.argtypes = u, [d]
            L.orc_e4m3_roundup.restype, L.orc_e4m3_roundup.argtypes = u, [d]
            L.orc_e2m1_decode.restype, L.orc_e2m1_decode.argtypes = d, [u]
            L.orc_e2m1_encode.restype, L.orc_e2m1_encode.argtypes = u, [d]
            L.orc_ue8m0_decode.restype, L.orc_ue8m0_decode.argtypes = d, [u]
            L.orc_noclamp_exponent.restype, L.orc_noclamp_exponent.argtypes = i, [d]
            L.orc_scale_exponent.restype, L.orc_scale_exponent.argtypes = i, [d]
            L.orc_round_bf16.restype, L.orc_round_bf16.argtypes = d, [d]
            L.orc_round_f16.restype, L.orc_round_f16.argtypes = d, [d]
            L.orc_bitexp2.restype, L.orc_bitexp2.argtypes = d, [d]
            L.orc_fwht_f32.restype, L.orc_fwht_f32.argtypes = None, [ctypes.c_void_p, i, i]
            L.orc_dq_prescale_c0.restype, L.orc_dq_prescale_c0.argtypes = i, [i, d]
            L.orc_dq_prescale.restype, L.orc_dq_prescale.argtypes = i, [i, i, i, i]
            L.orc_dq_prescales.restype = None
            L.orc_dq_prescales.argtypes = [i, i, i, p, i, p, p, p, i, i, i, p]
            for f in ("orc_e4m3_encode_array", "orc_e2m1_encode_array", "orc_noclamp_exponent_array"):
                getattr(L, f).restype = None
                getattr(L, f).argtypes = [p, ctypes.c_long, p]
            L.orc_quantize_blocks.restype = None
            L.orc_quantize_blocks.argtypes = [p, i, i, i, p, i, i, p, p]
            L.orc_dequantize_blocks.restype = None
            L.orc_dequantize_blocks.argtypes = [p, p, i, i, i, p]
            L.orc_quantize_nvfp4.restype = None
            L.orc_quantize_nvfp4.argtypes = [p, i, i, i, p, p, p]
            L.orc_dequantize_nvfp4.restype = None
            L.orc_dequantize_nvfp4.argtypes = [p, p, p, i, i, i, p]
            L.orc_compute_D.restype = None
            L.orc_compute_D.argtypes = [p, p, i, i, i, p]
            L.orc_attention.restype = None
            L.orc_attention.argtypes = [ctypes.POINTER(_Cfg), p] + [p] * 15
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


# --------------------------------------------------------------------------- codecs
def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    return lib().orc_e4m3_encode(float(x))


def e4m3_encode_array(x) -> np.ndarray:
    x = _f64(x)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_roundup(r: float) -> int:
    return lib().orc_e4m3_roundup(float(r))


def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e2m1_encode(x: float) -> int:
    return lib().orc_e2m1_encode(float(x))


def e2m1_encode_array(x) -> np.ndarray:
    x = _f64(x)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e2m1_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def ue8m0_decode(b: int) -> float:
    return lib().orc_ue8m0_decode(int(b))


def noclamp_exponent(amax: float) -> int:
    return lib().orc_noclamp_exponent(float(amax))


def noclamp_exponent_array(x) -> np.ndarray:
    x = _f64(x)
    out = np.empty(x.shape, np.int32)
    lib().orc_noclamp_exponent_array(_ptr(x), x.size, _ptr(out))
    return out


def scale_exponent(amax: float) -> int:
    return lib().orc_scale_exponent(float(amax))


def round_bf16(x: float) -> float:
    return lib().orc_round_bf16(float(x))


def bitexp2(z: float) -> float:
    """The bit-level approximation of 2^z (bf16 bit field, zero-mean shift)."""
    return lib().orc_bitexp2(float(z))


def fwht_f32(x) -> np.ndarray:
    """Hadamard rotation x -> x H_d of every d-vector along the last axis, in
    fp32 by the fast Walsh-Hadamard transform (unnormalised).  Returns the
    fp32 results as float64."""
    a = np.ascontiguousarray(x, dtype=np.float32).copy()
    d = a.shape[-1]
    lib().orc_fwht_f32(a.ctypes.data, int(a.size // d), int(d))
    return a.astype(np.float64)


def sylvester(d: int) -> np.ndarray:
    """The Sylvester Hadamard matrix H_d (entries +-1) from its recursion."""
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def round_f16(x: float) -> float:
    return lib().orc_round_f16(float(x))


def dq_prescale_c0(d: int, softmax_scale: float) -> int:
    return lib().orc_dq_prescale_c0(int(d), float(softmax_scale))


def dq_prescale(c0: int, edo: int, mk: int, mv: int) -> int:
    return lib().orc_dq_prescale(int(c0), int(edo), int(mk), int(mv))


def dq_prescales(cu_seqlens, eK, eV, edO, d, softmax_scale=None, causal=True, causal_scale=False) -> np.ndarray:
    """Prescale exponents p [H][T] of the FP16 dQ partials from the exponent
    arrays eK, eV [Hkv][T] and edO [H][T] (scale byte - 127)."""
    eK, eV, edO = (np.ascontiguousarray(a, dtype=np.int32) for a in (eK, eV, edO))
    Hkv, T = eK.shape
    H = edO.shape[0]
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    out = np.zeros((H, T), np.int32)
    scale = float(softmax_scale if softmax_scale is not None else 1.0 / np.sqrt(d))
    lib().orc_dq_prescales(T, H, Hkv, _ptr(cu), len(cu) - 1, _ptr(eK), _ptr(eV), _ptr(edO),
                           dq_prescale_c0(d, scale), int(causal), int(causal_scale), _ptr(out))
    return out


E4M3_TABLE = None


def e4m3_values() -> np.ndarray:
    """The 256 decoded E4M3FN values (NaN at 0x7F, 0xFF)."""
    global E4M3_TABLE
    if E4M3_TABLE is None:
        E4M3_TABLE = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return E4M3_TABLE


# --------------------------------------------------------------------------- quantizers
def quantize_blocks(x, cu_seqlens, block: int):
    """Token-block quantization: x [T][H][d] -> (codes uint8 [T][H][d], scales uint8 [H][T])."""
    x = _f64(x)
    T, H, d = x.shape
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    codes = np.empty((T, H, d), np.uint8)
    scales = np.zeros((H, T), np.uint8)
    lib().orc_quantize_blocks(_ptr(x), T, H, d, _ptr(cu), len(cu) - 1, int(block), _ptr(codes), _ptr(scales))
    return codes, scales


def dequantize_blocks(codes, scales) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    T, H, d = codes.shape
    out = np.empty((T, H, d), np.float64)
    lib().orc_dequantize_blocks(_ptr(codes), _ptr(scales), T, H, d, _ptr(out))
    return out


def quantize_nvfp4(x):
    """NVFP4 per-token quantization: -> (codes uint8 [T][H][d] one nibble each,
    block scales uint8 [T][H][d/16] E4M3, token scales fp32 [H][T])."""
    x = _f64(x)
    T, H, d = x.shape
    codes = np.empty((T, H, d), np.uint8)
    bsc = np.empty((T, H, d // 16), np.uint8)
    g = np.empty((H, T), np.float32)
    lib().orc_quantize_nvfp4(_ptr(x), T, H, d, _ptr(codes), _ptr(bsc), _ptr(g))
    return codes, bsc, g


def dequantize_nvfp4(codes, bsc, g) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    bsc = np.ascontiguousarray(bsc, dtype=np.uint8)
    g = np.ascontiguousarray(g, dtype=np.float32)
    T, H, d = codes.shape
    out = np.empty((T, H, d), np.float64)
    lib().orc_dequantize_nvfp4(_ptr(codes), _ptr(bsc), _ptr(g), T, H, d, _ptr(out))
    return out


def compute_D(dOq, O_stored) -> np.ndarray:
    dOq, O_stored = _f64(dOq), _f64(O_stored)
    T, H, d = dOq.shape
    D = np.empty((H, T), np.float64)
    lib().orc_compute_D(_ptr(dOq), _ptr(O_stored), T, H, d, _ptr(D))
    return D


# --------------------------------------------------------------------------- attention
def attention(cu_seqlens, Q, K, V, dO=None, *, Qs=None, Ks=None, eQ=None, eK=None, eV=None, edO=None,
              causal=True, softmax_scale=None, quant_p=True, quant_ds=True, quant_pt=True, exact=False,
              out_round=0, dq_fp16=False, dq_causal_scale=False, bitexp=False):
    """Attention forward (+ backward when dO is given) in fp64.

    Q [T][H][d], K/V [T][Hkv][d], dO [T][H][d] are operand values (dequantized
    payloads, or plain values for the identity reference).  Exponent arrays
    default to zero.  Returns dict(O, D, lse2, dQ, dK, dV).
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    T, H, d = Q.shape
    Hkv = K.shape[1]
    Qs = Q if Qs is None else _f64(Qs)
    Ks = K if Ks is None else _f64(Ks)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    z = lambda n: np.zeros((n, T), np.int32)
    eQ = z(H) if eQ is None else np.ascontiguousarray(eQ, dtype=np.int32)
    eK = z(Hkv) if eK is None else np.ascontiguousarray(eK, dtype=np.int32)
    eV = z(Hkv) if eV is None else np.ascontiguousarray(eV, dtype=np.int32)
    edO = z(H) if edO is None else np.ascontiguousarray(edO, dtype=np.int32)
    cfg = _Cfg(T, H, Hkv, d, len(cu) - 1, int(causal),
               float(softmax_scale if softmax_scale is not None else 1.0 / np.sqrt(d)),
               int(quant_p), int(quant_ds), int(quant_pt), int(exact), int(out_round), int(bitexp), int(dq_fp16),
               int(dq_causal_scale))
    O = np.empty((T, H, d), np.float64)
    lse2 = np.empty((H, T), np.float64)
    D = dQ = dK = dV = None
    if dO is not None:
        dO = _f64(dO)
        D = np.empty((H, T), np.float64)
        dQ = np.empty((T, H, d), np.float64)
        dK = np.empty((T, Hkv, d), np.float64)
        dV = np.empty((T, Hkv, d), np.float64)
    lib().orc_attention(ctypes.byref(cfg), _ptr(cu), _ptr(Qs), _ptr(Ks), _ptr(Q), _ptr(K), _ptr(V), _ptr(dO),
                        _ptr(eQ), _ptr(eK), _ptr(eV), _ptr(edO), _ptr(O), _ptr(D), _ptr(lse2), _ptr(dQ),
                        _ptr(dK), _ptr(dV))
    return dict(O=O, D=D, lse2=lse2, dQ=dQ, dK=dK, dV=dV)


def train_call(q, k, v, do, cu_seqlens, *, causal=True, exact=False, path=PATH_MXFP8, out_dtype="bf16",
               softmax_scale=None, quantize=True, dq_fp16=False, dq_causal_scale=False, bitexp=False,
               hadamard=False):
    """The whole training call from raw inputs: quantize Q/K/V, forward, quantize
    dO (+ D), backward.  Inputs are fp32 arrays whose values are the exact inputs
    (bf16-exact for bf16 workloads).  Returns a dict with every intermediate
    payload (codes, scale bytes), O as stored, D, lse2, dQ, dK, dV.

    quantize=False gives the unquantized fp64 reference of the same call.
    dq_fp16: dQ partials per 128-key tile in FP16 with a power-of-two row
    prescale (the pages' FP16 reduction); False sums dQ in fp64.
    dq_causal_scale: the prescale from keys j <= i only.
    bitexp: the inference forward with bit-level exponentials (no backward).
    hadamard: Q and K rotated by H_d before quantization (fwht_f32), the
    softmax scale divided by d, and dQ, dK rotated back (x H_d, fp64).
    """
    if bitexp and do is not None:
        raise ValueError("the bit-level exponential forward is for inference: no backward")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do) if do is not None else None
    out_round = {"bf16": 1, "f32": 2, "f64": 0}[out_dtype]
    res: dict = {}
    Hd = None
    if hadamard:
        if path == PATH_NVFP4_FP8:
            raise ValueError("the Hadamard rotation is offered on the MXFP8 path")
        d = q.shape[-1]
        Hd = sylvester(d)
        softmax_scale = (softmax_scale if softmax_scale else 1.0 / np.sqrt(d)) / d
        # unquantized: the plain definition in fp64; quantized: the fp32
        # rotation the codes are decided from
        q, k = (q @ Hd, k @ Hd) if not quantize else (fwht_f32(q), fwht_f32(k))
    if not quantize:
        r = attention(cu, q, k, v, do, causal=causal, softmax_scale=softmax_scale, quant_p=False,
                      quant_ds=False, quant_pt=False, exact=exact, out_round=0)
        res.update(r)
        if Hd is not None and do is not None:
            res["dQ"], res["dK"] = r["dQ"] @ Hd, r["dK"] @ Hd
        return res
    blk = 1 if exact else 32
    qc, qs = quantize_blocks(q, cu, blk)
    kc, ks = quantize_blocks(k, cu, blk)
    vc, vs = quantize_blocks(v, cu, 1)
    Qh, Kh, Vh = dequantize_blocks(qc, qs), dequantize_blocks(kc, ks), dequantize_blocks(vc, vs)
    res.update(q_codes=qc, q_scales=qs, k_codes=kc, k_scales=ks, v_codes=vc, v_scales=vs)
    Qs_, Ks_ = Qh, Kh
    if path == PATH_NVFP4_FP8:
        q4, qb, qg = quantize_nvfp4(q)
        k4, kb, kg = quantize_nvfp4(k)
        Qs_, Ks_ = dequantize_nvfp4(q4, qb, qg), dequantize_nvfp4(k4, kb, kg)
        res.update(q4_codes=q4, q4_bscales=qb, q4_gscales=qg, k4_codes=k4, k4_bscales=kb, k4_gscales=kg)
    dOh = edO = None
    if do is not None:
        dc, ds = quantize_blocks(do, cu, blk)
        dOh = dequantize_blocks(dc, ds)
        edO = ds.astype(np.int32) - 127
        res.update(do_codes=dc, do_scales=ds)
    r = attention(cu, Qh, Kh, Vh, dOh, Qs=Qs_, Ks=Ks_, eQ=qs.astype(np.int32) - 127,
                  eK=ks.astype(np.int32) - 127, eV=vs.astype(np.int32) - 127, edO=edO, causal=causal,
                  softmax_scale=softmax_scale, exact=exact, out_round=out_round,
                  dq_fp16=dq_fp16 and do is not None, dq_causal_scale=dq_causal_scale, bitexp=bitexp)
    res.update(r)
    if Hd is not None and do is not None:
        res["dQ"], res["dK"] = r["dQ"] @ Hd, r["dK"] @ Hd
    return res
