"""Python binding of libflamia (block-scaled causal attention for training on GB300).

Argument marshalling only: every step runs in the library's CUDA kernels, called
through its C ABI (include/flamia.h) with the same names.  PyTorch provides the
device memory and streams.  There is no CPU path: without the compiled library
every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libflamia.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, ERR_TIMEOUT, ERR_BAD_SEQLENS = range(7)
PATH_MXFP8, PATH_NVFP4_FP8 = 0, 1
F32, BF16 = 0, 1
ROLE_QKV, ROLE_DO = 0, 1

EXPORTED = ("flamia_workspace_size", "flamia_plan", "flamia_quantize", "flamia_fwd", "flamia_bwd",
            "flamia_get_device_status", "flamia_clear_device_status", "flamia_status_string",
            "flamia_debug_set_phat_dump", "flamia_debug_withhold_first_item", "flamia_debug_workspace_offset",
            "flamia_plan_noalloc", "flamia_debug_mma_idesc", "flamia_debug_smem_desc")
WS_FWD_ITEMS, WS_BWD_ITEMS, WS_DQ_PRESCALE = range(3)
MMA_F8F6F4, MMA_MXF8F6F4, MMA_MXF4NVF4 = range(3)
SWZ_NONE, SWZ_128B, SWZ_64B, SWZ_32B = 0, 2, 4, 6


class FlamiaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class Problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32),
                ("n_seq", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p), ("causal", ctypes.c_int32),
                ("exact", ctypes.c_int32), ("causal_dq_scale", ctypes.c_int32), ("deterministic", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("path", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("dq_fp16", ctypes.c_int32), ("bitexp", ctypes.c_int32),
                ("hadamard", ctypes.c_int32), ("clc", ctypes.c_int32)]


class Operand(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("codes4", ctypes.c_void_p),
                ("scales4", ctypes.c_void_p), ("gscale4", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libflamia.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
    L = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    P = ctypes.POINTER(Problem)
    O = ctypes.POINTER(Operand)
    L.flamia_workspace_size.restype, L.flamia_workspace_size.argtypes = sz, [P]
    L.flamia_plan.restype, L.flamia_plan.argtypes = i32, [P, vp, sz, vp]
    L.flamia_quantize.restype = i32
    L.flamia_quantize.argtypes = [P, i32, ctypes.POINTER(vp), vp, O, vp, vp, sz, vp]
    L.flamia_fwd.restype = i32
    L.flamia_fwd.argtypes = [P, O, O, O, vp, vp, vp, vp, sz, vp]
    L.flamia_bwd.restype = i32
    L.flamia_bwd.argtypes = [P, O, O, O, O, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flamia_get_device_status.restype, L.flamia_get_device_status.argtypes = i32, [vp, vp]
    L.flamia_clear_device_status.restype, L.flamia_clear_device_status.argtypes = i32, [vp, vp]
    L.flamia_status_string.restype, L.flamia_status_string.argtypes = ctypes.c_char_p, [i32]
    L.flamia_debug_set_phat_dump.restype = i32
    L.flamia_debug_set_phat_dump.argtypes = [vp, sz, vp, vp, vp]
    L.flamia_debug_workspace_offset.restype, L.flamia_debug_workspace_offset.argtypes = sz, [P, i32]
    L.flamia_debug_withhold_first_item.restype = i32
    L.flamia_debug_withhold_first_item.argtypes = [i32]
    L.flamia_debug_mma_idesc.restype = i32
    L.flamia_debug_mma_idesc.argtypes = [i32, ctypes.c_uint32, ctypes.c_uint32, i32, i32, i32, i32,
                                         ctypes.POINTER(ctypes.c_uint32)]
    L.flamia_debug_smem_desc.restype = i32
    L.flamia_debug_smem_desc.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, i32,
                                         ctypes.POINTER(ctypes.c_uint64)]
    L.flamia_plan_noalloc.restype = i32
    L.flamia_plan_noalloc.argtypes = [P, vp, vp, vp, vp]
    _lib = L
    return L


def status_string(s: int) -> str:
    return load_library().flamia_status_string(int(s)).decode()


def _check(s: int, what: str):
    if s != OK:
        raise FlamiaError(s, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def make_problem(T, H, Hkv, d, cu_seqlens, *, causal=True, exact=False, causal_dq_scale=False,
                 deterministic=False, softmax_scale=0.0, path=PATH_MXFP8, in_dtype=BF16, out_dtype=BF16,
                 dq_fp16=False, bitexp=False, hadamard=False, clc=False) -> Problem:
    """cu_seqlens: int32 device tensor [n_seq + 1] (kept referenced by the caller)."""
    return Problem(int(T), int(H), int(Hkv), int(d), int(cu_seqlens.numel() - 1), cu_seqlens.data_ptr(),
                   int(causal), int(exact), int(causal_dq_scale), int(deterministic), float(softmax_scale),
                   int(path), int(in_dtype), int(out_dtype), int(dq_fp16), int(bitexp),
                   int(hadamard), int(clc))


def operand(codes, scales, codes4=None, scales4=None, gscale4=None) -> Operand:
    return Operand(_ptr(codes), _ptr(scales), _ptr(codes4), _ptr(scales4), _ptr(gscale4))


def flamia_workspace_size(prob: Problem) -> int:
    return int(load_library().flamia_workspace_size(ctypes.byref(prob)))


def flamia_plan(prob: Problem, ws, stream=None):
    _check(load_library().flamia_plan(ctypes.byref(prob), _ptr(ws), ws.numel() * ws.element_size(),
                                      _stream(stream)), "flamia_plan")


def flamia_quantize(prob: Problem, role: int, inputs, O, outs, D, ws, stream=None):
    n = len(inputs)
    arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in inputs])
    ops = (Operand * len(outs))(*outs)
    _check(load_library().flamia_quantize(ctypes.byref(prob), int(role), arr, _ptr(O), ops, _ptr(D), _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream(stream)), "flamia_quantize")


def flamia_fwd(prob: Problem, q: Operand, k: Operand, v: Operand, O, m, l, ws, stream=None):
    _check(load_library().flamia_fwd(ctypes.byref(prob), ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                     _ptr(O), _ptr(m), _ptr(l), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)), "flamia_fwd")


def flamia_bwd(prob: Problem, q: Operand, k: Operand, v: Operand, dO: Operand, D, m, l, dQ, dK, dV, ws,
               stream=None):
    _check(load_library().flamia_bwd(ctypes.byref(prob), ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                     ctypes.byref(dO), _ptr(D), _ptr(m), _ptr(l), _ptr(dQ), _ptr(dK), _ptr(dV),
                                     _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "flamia_bwd")


def flamia_plan_noalloc(prob: Problem, fwd_items, bwd_items, n_items, stream=None):
    """Work lists without a workspace (library-held scratch; see include/flamia.h).
    fwd_items/bwd_items: int32 device tensors [ceil(T/128) + n_seq, 2]; n_items: int32 device [1]."""
    _check(load_library().flamia_plan_noalloc(ctypes.byref(prob), _ptr(fwd_items), _ptr(bwd_items), _ptr(n_items),
                                              _stream(stream)), "flamia_plan_noalloc")


def flamia_get_device_status(ws, stream=None) -> int:
    return int(load_library().flamia_get_device_status(_ptr(ws), _stream(stream)))


def flamia_debug_set_phat_dump(ws, codes, exps, stream=None):
    """Test hook: record P^ codes / block exponents of the next fwd/bwd calls (None, None: off)."""
    _check(load_library().flamia_debug_set_phat_dump(_ptr(ws), ws.numel() * ws.element_size(), _ptr(codes), _ptr(exps),
                                                     _stream(stream)), "flamia_debug_set_phat_dump")


def flamia_debug_workspace_offset(prob: Problem, region: int) -> int:
    """Byte offset of a workspace region (WS_FWD_ITEMS, WS_BWD_ITEMS, WS_DQ_PRESCALE)."""
    return int(load_library().flamia_debug_workspace_offset(ctypes.byref(prob), int(region)))


def flamia_debug_withhold_first_item(on: bool):
    """Test hook: the next attention launches withhold each CTA's first work
    item, so that their bounded waits run out (see include/flamia.h)."""
    _check(load_library().flamia_debug_withhold_first_item(int(bool(on))), "flamia_debug_withhold_first_item")


def flamia_debug_mma_idesc(kind: int, M: int, N: int, a_mn: int = 0, b_mn: int = 0, a_sf_id: int = 0,
                           b_sf_id: int = 0) -> int:
    """Test hook: the tcgen05.mma instruction descriptor the kernels encode
    for `kind` (MMA_F8F6F4, MMA_MXF8F6F4, MMA_MXF4NVF4) on an M x N tile."""
    out = ctypes.c_uint32()
    _check(load_library().flamia_debug_mma_idesc(int(kind), int(M), int(N), int(a_mn), int(b_mn), int(a_sf_id),
                                                 int(b_sf_id), ctypes.byref(out)), "flamia_debug_mma_idesc")
    return int(out.value)


def flamia_debug_smem_desc(saddr: int, lbo: int, sbo: int, swizzle: int) -> int:
    """Test hook: the shared-memory matrix descriptor the kernels encode."""
    out = ctypes.c_uint64()
    _check(load_library().flamia_debug_smem_desc(int(saddr), int(lbo), int(sbo), int(swizzle), ctypes.byref(out)),
           "flamia_debug_smem_desc")
    return int(out.value)


def flamia_clear_device_status(ws, stream=None):
    _check(load_library().flamia_clear_device_status(_ptr(ws), _stream(stream)), "flamia_clear_device_status")


@dataclass
class TrainCall:
    """Device buffers for one training call of a fixed problem, and the call itself.

    Holds the quantized payloads, O, (m, l), D and the gradients.  ``run()``
    issues plan -> quantize(QKV) -> fwd -> quantize(dO) -> bwd on the current
    stream (no host synchronisation)."""

    T: int
    H: int
    Hkv: int
    d: int
    cu_seqlens: object  # int32 device tensor
    causal: bool = True
    exact: bool = False
    deterministic: bool = False
    causal_dq_scale: bool = False
    dq_fp16: bool = True  # FP16 dQ partials with the power-of-two prescale (the pages' default)
    bitexp: bool = False  # inference forward only: backward() raises
    hadamard: bool = False  # Q and K rotated before quantization; gradients rotated back
    clc: bool = False  # work items taken over by cluster launch control (a CTA per item)
    path: int = PATH_MXFP8
    in_dtype: int = BF16
    out_dtype: int = BF16
    softmax_scale: float = 0.0

    def __post_init__(self):
        import torch
        dev = self.cu_seqlens.device
        self.prob = make_problem(self.T, self.H, self.Hkv, self.d, self.cu_seqlens, causal=self.causal,
                                 exact=self.exact, deterministic=self.deterministic,
                                 causal_dq_scale=self.causal_dq_scale, dq_fp16=self.dq_fp16, bitexp=self.bitexp,
                                 hadamard=self.hadamard, clc=self.clc,
                                 softmax_scale=self.softmax_scale, path=self.path, in_dtype=self.in_dtype,
                                 out_dtype=self.out_dtype)
        nbytes = flamia_workspace_size(self.prob)
        if nbytes == 0:
            raise FlamiaError(ERR_INVALID_ARG, "flamia_workspace_size")
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        u8 = dict(dtype=torch.uint8, device=dev)
        T, H, Hkv, d = self.T, self.H, self.Hkv, self.d
        odt = torch.bfloat16 if self.out_dtype == BF16 else torch.float32
        self.q_codes, self.k_codes, self.v_codes = (torch.empty(T, h, d, **u8) for h in (H, Hkv, Hkv))
        self.q_scales, self.k_scales, self.v_scales = (torch.empty(h, T, **u8) for h in (H, Hkv, Hkv))
        self.do_codes, self.do_scales = torch.empty(T, H, d, **u8), torch.empty(H, T, **u8)
        self.q4 = self.k4 = None
        if self.path == PATH_NVFP4_FP8:
            self.q4 = (torch.empty(T, H, d // 2, **u8), torch.empty(T, H, d // 16, **u8),
                       torch.empty(H, T, dtype=torch.float32, device=dev))
            self.k4 = (torch.empty(T, Hkv, d // 2, **u8), torch.empty(T, Hkv, d // 16, **u8),
                       torch.empty(Hkv, T, dtype=torch.float32, device=dev))
        self.O = torch.empty(T, H, d, dtype=odt, device=dev)
        self.m = torch.empty(H, T, dtype=torch.int32, device=dev)
        self.l = torch.empty(H, T, dtype=torch.float32, device=dev)
        self.D = torch.empty(H, T, dtype=torch.float32, device=dev)
        self.dQ = torch.empty(T, H, d, dtype=odt, device=dev)
        self.dK = torch.empty(T, Hkv, d, dtype=odt, device=dev)
        self.dV = torch.empty(T, Hkv, d, dtype=odt, device=dev)
        q4, k4 = self.q4 or (None,) * 3, self.k4 or (None,) * 3
        self.opq = operand(self.q_codes, self.q_scales, *q4)
        self.opk = operand(self.k_codes, self.k_scales, *k4)
        self.opv = operand(self.v_codes, self.v_scales)
        self.opdo = operand(self.do_codes, self.do_scales)

    def plan(self, stream=None):
        flamia_plan(self.prob, self.ws, stream)

    def forward(self, q, k, v, stream=None):
        flamia_quantize(self.prob, ROLE_QKV, [q, k, v], None, [self.opq, self.opk, self.opv], None, self.ws, stream)
        flamia_fwd(self.prob, self.opq, self.opk, self.opv, self.O, self.m, self.l, self.ws, stream)

    def backward(self, do, stream=None):
        flamia_quantize(self.prob, ROLE_DO, [do], self.O, [self.opdo], self.D, self.ws, stream)
        flamia_bwd(self.prob, self.opq, self.opk, self.opv, self.opdo, self.D, self.m, self.l, self.dQ, self.dK,
                   self.dV, self.ws, stream)

    def run(self, q, k, v, do, stream=None):
        self.plan(stream)
        self.forward(q, k, v, stream)
        self.backward(do, stream)
