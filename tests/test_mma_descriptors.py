"""Host checks (no GPU) of the tensor-core descriptors the kernels issue.

The library's own builders are reached through two test hooks of the C ABI
(flamia_debug_mma_idesc, flamia_debug_smem_desc).  Each encoded word is taken
apart here field by field with the field tables of the PTX ISA's tcgen05
sections ("Instruction descriptor" for kind::f16/f8f6f4 and for the
block-scaled kinds, "Shared memory descriptor"), and a few words are also
compared with values worked out by hand from those tables.  A field in the
wrong place, a reserved bit set, an MN-major flag on the wrong operand or a
wrong scale type (UE8M0 for MXFP8 against UE4M3 for NVFP4) fails here before
any GPU run.

The descriptors the kernels issue (found in the sources by the last test):
  scores S = Q K^T and dP = dO V^T   kind::f8f6f4, 128 x 128, both K-major;
  mixed-path scores                  kind::mxf4nvf4, 128 x 128, K-major;
  O += P^ V (forward)                kind::mxf8f6f4, 128 x d, B MN-major;
  dV += P~^T dO, dK += dS^T Q        kind::mxf8f6f4, 128 x d, both MN-major;
  dQ = dS K                          kind::mxf8f6f4, 128 x 64 (one half of d
                                     per MMA), B MN-major;
with the scale-factor id kk = 0..3 picking the byte of each scale word.
"""
import os
import re

import pytest

import precision_causal_attention_token_gb300 as fl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return fl.load_library()


# (name, first bit, width) of the instruction descriptor for kind::f16 and
# kind::f8f6f4 (dense, no sparsity)
DENSE_FIELDS = [
    ("sparsity_selector", 0, 2), ("sparsity", 2, 1), ("saturate", 3, 1), ("d_format", 4, 2),
    ("reserved6", 6, 1), ("a_format", 7, 3), ("b_format", 10, 3), ("negate_a", 13, 1), ("negate_b", 14, 1),
    ("transpose_a", 15, 1), ("transpose_b", 16, 1), ("n_shr3", 17, 6), ("reserved23", 23, 1),
    ("m_shr4", 24, 5), ("reserved29", 29, 1), ("max_shift", 30, 2),
]
# the same for the block-scaled kinds (kind::mxf8f6f4, kind::mxf4nvf4)
SCALED_FIELDS = [
    ("reserved0", 0, 2), ("sparsity", 2, 1), ("reserved3", 3, 1), ("b_sf_id", 4, 2), ("reserved6", 6, 1),
    ("a_format", 7, 3), ("b_format", 10, 3), ("negate_a", 13, 1), ("negate_b", 14, 1), ("transpose_a", 15, 1),
    ("transpose_b", 16, 1), ("n_shr3", 17, 6), ("scale_type", 23, 1), ("m_shr4", 24, 5), ("a_sf_id", 29, 2),
    ("reserved31", 31, 1),
]
# the shared-memory matrix descriptor
SMEM_FIELDS = [
    ("start_shr4", 0, 14), ("reserved14", 14, 2), ("lbo_shr4", 16, 14), ("reserved30", 30, 2),
    ("sbo_shr4", 32, 14), ("version", 46, 2), ("reserved48", 48, 1), ("base_offset", 49, 3),
    ("lbo_mode", 52, 1), ("reserved53", 53, 8), ("swizzle", 61, 3),
]

F32 = 1            # d_format: fp32 accumulator
E4M3 = 0           # a/b format of kind::f8f6f4 and kind::mxf8f6f4
E2M1 = 1           # a/b format of kind::mxf4nvf4
UE8M0, UE4M3 = 1, 0


def _decode(word, fields, bits):
    out, covered = {}, 0
    for name, lo, w in fields:
        out[name] = (word >> lo) & ((1 << w) - 1)
        covered |= ((1 << w) - 1) << lo
    assert covered == (1 << bits) - 1, "the field table must cover every bit"
    return out


def _reserved_clear(f):
    for name, v in f.items():
        if name.startswith("reserved"):
            assert v == 0, name


def test_tables_tile_the_words():
    for fields, bits in ((DENSE_FIELDS, 32), (SCALED_FIELDS, 32), (SMEM_FIELDS, 64)):
        ends = [lo + w for _, lo, w in fields]
        starts = [lo for _, lo, _ in fields]
        assert starts[0] == 0 and ends[-1] == bits and starts[1:] == ends[:-1]


@pytest.mark.parametrize("M,N", [(128, 128), (128, 64), (128, 256), (64, 8), (128, 16)])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
def test_f8f6f4_fields(M, N, a_mn, b_mn):
    f = _decode(fl.flamia_debug_mma_idesc(fl.MMA_F8F6F4, M, N, a_mn, b_mn), DENSE_FIELDS, 32)
    _reserved_clear(f)
    assert (f["sparsity_selector"], f["sparsity"], f["saturate"], f["max_shift"]) == (0, 0, 0, 0)
    assert f["d_format"] == F32 and f["a_format"] == E4M3 and f["b_format"] == E4M3
    assert (f["negate_a"], f["negate_b"]) == (0, 0)
    assert (f["transpose_a"], f["transpose_b"]) == (a_mn, b_mn)
    assert f["n_shr3"] << 3 == N and f["m_shr4"] << 4 == M


@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 1), (1, 1)])
@pytest.mark.parametrize("kk", range(4))
def test_mxf8f6f4_fields(N, a_mn, b_mn, kk):
    a_sf, b_sf = kk, 3 - kk      # distinct ids, so a swapped pair shows
    f = _decode(fl.flamia_debug_mma_idesc(fl.MMA_MXF8F6F4, 128, N, a_mn, b_mn, a_sf, b_sf), SCALED_FIELDS, 32)
    _reserved_clear(f)
    assert f["sparsity"] == 0 and f["scale_type"] == UE8M0
    assert f["a_format"] == E4M3 and f["b_format"] == E4M3
    assert (f["negate_a"], f["negate_b"]) == (0, 0)
    assert (f["transpose_a"], f["transpose_b"]) == (a_mn, b_mn)
    assert (f["a_sf_id"], f["b_sf_id"]) == (a_sf, b_sf)
    assert f["n_shr3"] << 3 == N and f["m_shr4"] << 4 == 128


@pytest.mark.parametrize("M,N", [(128, 128), (128, 64), (64, 128)])
def test_mxf4nvf4_fields(M, N):
    f = _decode(fl.flamia_debug_mma_idesc(fl.MMA_MXF4NVF4, M, N), SCALED_FIELDS, 32)
    _reserved_clear(f)
    assert f["sparsity"] == 0
    assert f["a_format"] == E2M1 and f["b_format"] == E2M1
    assert f["scale_type"] == UE4M3           # NVFP4: E4M3 block scales, one per 16 elements
    assert (f["transpose_a"], f["transpose_b"]) == (0, 0)   # 4-bit operands are K-major only
    assert (f["a_sf_id"], f["b_sf_id"]) == (0, 0)
    assert f["n_shr3"] << 3 == N and f["m_shr4"] << 4 == M


def test_descriptor_words_worked_by_hand():
    # kind::f8f6f4 128x128 K-major: fp32 D (bit 4), N/8 = 16 at bit 17, M/16 = 8 at bit 24
    assert fl.flamia_debug_mma_idesc(fl.MMA_F8F6F4, 128, 128) == 0x08200010
    # kind::mxf4nvf4 128x128: E2M1 at bits 7 and 10, UE4M3 (bit 23 clear)
    assert fl.flamia_debug_mma_idesc(fl.MMA_MXF4NVF4, 128, 128) == 0x08200480
    # kind::mxf8f6f4 128x128, B MN-major, ids 2/2: b id 2 at bit 4, bit 16, UE8M0 bit 23, a id 2 at bit 29
    assert fl.flamia_debug_mma_idesc(fl.MMA_MXF8F6F4, 128, 128, 0, 1, 2, 2) == 0x48A10020
    # the dQ half tile: 128x64, B MN-major, ids 3/3
    assert fl.flamia_debug_mma_idesc(fl.MMA_MXF8F6F4, 128, 64, 0, 1, 3, 3) == 0x68910030
    # a 128B-swizzled tile at 0x1C400, LBO 16, SBO 1024, version 1 at bit 46, mode 2 at bit 61
    assert fl.flamia_debug_smem_desc(0x1C400, 16, 1024, fl.SWZ_128B) == 0x4000404000011C40


@pytest.mark.parametrize("swz", [fl.SWZ_NONE, fl.SWZ_128B, fl.SWZ_64B, fl.SWZ_32B])
@pytest.mark.parametrize("saddr,lbo,sbo", [(0, 16, 1024), (0x3FFF0, 8 * 128, 512), (0x12340, 0x3FFF0, 16)])
def test_smem_desc_fields(swz, saddr, lbo, sbo):
    f = _decode(fl.flamia_debug_smem_desc(saddr, lbo, sbo, swz), SMEM_FIELDS, 64)
    _reserved_clear(f)
    assert f["start_shr4"] << 4 == saddr and f["lbo_shr4"] << 4 == lbo and f["sbo_shr4"] << 4 == sbo
    assert f["version"] == 1 and f["base_offset"] == 0 and f["lbo_mode"] == 0
    assert f["swizzle"] == swz


def test_swizzle_codes():
    # the descriptor's layout codes: 0 none, 2 128-byte, 4 64-byte, 6 32-byte
    assert (fl.SWZ_NONE, fl.SWZ_128B, fl.SWZ_64B, fl.SWZ_32B) == (0, 2, 4, 6)
    for bad in (1, 3, 5, 7, 8, -1):
        with pytest.raises(fl.FlamiaError) as e:
            fl.flamia_debug_smem_desc(0, 16, 16, bad)
        assert e.value.status == fl.ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (fl.MMA_F8F6F4, 96, 128), (fl.MMA_F8F6F4, 128, 120), (fl.MMA_F8F6F4, 128, 272), (fl.MMA_F8F6F4, 64, 4),
    (fl.MMA_F8F6F4, 128, 128, 2, 0), (fl.MMA_F8F6F4, 128, 128, 0, 0, 1, 0),
    (fl.MMA_MXF8F6F4, 128, 128, 0, 0, 4, 0), (fl.MMA_MXF4NVF4, 128, 128, 0, 1),
    (fl.MMA_MXF4NVF4, 128, 128, 0, 0, 0, 1), (3, 128, 128),
])
def test_idesc_rejects_unsupported(args):
    with pytest.raises(fl.FlamiaError) as e:
        fl.flamia_debug_mma_idesc(*args)
    assert e.value.status == fl.ERR_INVALID_ARG


def test_smem_desc_rejects_unaligned_or_wide():
    for args in ((8, 16, 16), (0, 24, 16), (0, 16, 1 << 18), (1 << 18, 16, 16)):
        with pytest.raises(fl.FlamiaError):
            fl.flamia_debug_smem_desc(*args, fl.SWZ_NONE)


def test_kernel_descriptor_uses_are_the_checked_ones():
    """Every instruction descriptor the kernels build is one of the forms the
    tests above check (a new form must be added there)."""
    allowed = {
        "idesc_f8(128, 128, 0, 0)",
        "idesc_mxf4nvf4(128, 128)",
        "idesc_mxf8(128, HD, 0, 1, kk, kk)",
        "idesc_mxf8(128, HD, 1, 1, kk, kk)",
        "idesc_mxf8(128, 64, 0, 1, kk, kk)",
    }
    csrc = os.path.join(ROOT, "precision_causal_attention_token_gb300", "csrc")
    seen = set()
    for name in os.listdir(csrc):
        if not name.endswith((".cu", ".cuh")) or name == "api.cu":   # api.cu: the hooks, which forward arguments
            continue
        for m in re.finditer(r"\bidesc_\w+\([^()]*\)", open(os.path.join(csrc, name)).read()):
            call = m.group(0)
            if "uint32_t" in call:          # the builders' own definitions
                continue
            assert call in allowed, (name, call)
            seen.add(call)
    assert seen == allowed
