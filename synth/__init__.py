"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This module holds input generation only: no step of the attention method.
Numbers come from a counter-based SplitMix64 generator (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", 2014): the i-th draw of a
stream is the SplitMix64 finaliser applied to seed + (i + 1) * golden_gamma,
with the stream folded into the seed.  Normals use the Box-Muller transform.
Values are produced in fp64, rounded to fp32 and then (for bf16 workloads)
rounded to the nearest-even bf16, so every side sees the same bit patterns.

Workloads (shapes of the causal packed-document training workloads):
  1  tiny:     T=128, H=1, d=64, fp32 N(0,1), one document
  2  batched:  4 rows x 4096 tokens, H=16, d=128, bf16 N(0,1), equal documents
  3  packed:   8 rows x 16384 tokens, H=16, d=128, bf16; log-normal document
               lengths (arithmetic mean 1500, sigma 1.0, clipped to [32, 16384]);
               Q and K carry two seed-chosen outlier channels per head x20
  4  mixed:    as 3 with 4 rows x 32768 tokens (NVFP4 scores)
  5  long GQA: 2 rows x 65536 tokens, H=32, Hkv=8, d=128, log-normal mean 6000
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20261202
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_Q, STREAM_K, STREAM_V, STREAM_DO, STREAM_DOCS, STREAM_OUTLIERS = 1, 2, 3, 4, 5, 6


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """Draws start..start+n-1 of one stream as uint64."""
    base = np.uint64((seed * 0x100000001B3 + stream * 0xD1B54A32D192ED03) & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(base + idx * _GAMMA)


def uniform(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """Uniform fp64 in [0, 1) from the top 53 bits."""
    return (raw_u64(seed, stream, start, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n standard normals; normal k uses uniforms 2k and 2k+1 (Box-Muller, cosine branch)."""
    u = uniform(seed, stream, 2 * start, 2 * n)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    return r * np.cos(2.0 * np.pi * u2)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 values rounded to the nearest-even bf16, returned as fp32."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = ((u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return u.view(np.float32)


def doc_lengths_lognormal(seed: int, row: int, row_len: int, mean: float, sigma: float = 1.0,
                          lo: int = 32, hi: int = 16384) -> list[int]:
    """Document lengths for one packed row.

    Log-normal with the given arithmetic mean (mu = ln(mean) - sigma^2 / 2),
    rounded to integers and clipped to [lo, hi]; documents are drawn until the
    row would overflow and the last one is truncated to fill the row exactly,
    so boundaries are generally not 32-aligned.
    """
    mu = math.log(mean) - 0.5 * sigma * sigma
    out: list[int] = []
    total, k = 0, 0
    while total < row_len:
        z = normal(seed, STREAM_DOCS, 1, start=row * 1_000_003 + k)[0]
        k += 1
        n = int(min(max(round(math.exp(mu + sigma * z)), lo), hi))
        n = min(n, row_len - total)
        out.append(n)
        total += n
    return out


@dataclass
class Workload:
    name: str
    T: int
    H: int
    Hkv: int
    d: int
    dtype: str  # "f32" or "bf16"
    seqlens: list[int]
    outlier_channels: int = 0
    seed: int = SEED_BASE
    meta: dict = field(default_factory=dict)

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens)]).astype(np.int32)

    @property
    def causal_pairs(self) -> int:
        return int(sum(l * (l + 1) // 2 for l in self.seqlens))

    def flops(self) -> float:
        """Algorithmic causal FLOPs of one fwd+bwd: 14 d H per unmasked pair (4d fwd, 10d bwd)."""
        return 14.0 * self.d * self.H * self.causal_pairs

    def tensor(self, which: str, heads: int | None = None) -> np.ndarray:
        """One input tensor [T][heads][d] as fp32 values (bf16-exact for bf16 workloads)."""
        stream = {"q": STREAM_Q, "k": STREAM_K, "v": STREAM_V, "do": STREAM_DO}[which]
        nh = heads if heads is not None else (self.H if which in ("q", "do") else self.Hkv)
        n = self.T * nh * self.d
        x = normal(self.seed, stream, n).astype(np.float32).reshape(self.T, nh, self.d)
        if self.outlier_channels and which in ("q", "k"):
            for h, chans in enumerate(self.outliers()[: nh] if which == "q" else self.outliers_kv()):
                x[:, h, chans] *= np.float32(20.0)
        if self.dtype == "bf16":
            x = round_to_bf16(x)
        return x

    def outliers(self) -> list[list[int]]:
        """Seed-chosen distinct outlier channels per query head (scaled x20 in Q and K)."""
        res = []
        for h in range(self.H):
            u = uniform(self.seed, STREAM_OUTLIERS, 16 * h, 16)
            chans: list[int] = []
            for v in u:
                c = int(v * self.d)
                if c not in chans:
                    chans.append(c)
                if len(chans) == self.outlier_channels:
                    break
            res.append(chans)
        return res

    def outliers_kv(self) -> list[list[int]]:
        g = self.H // self.Hkv
        return [self.outliers()[hk * g] for hk in range(self.Hkv)]


def workload(idx: int, **over) -> Workload:
    """The five workloads by index (1-based)."""
    seed = SEED_BASE + idx
    if idx == 1:
        w = Workload("tiny T=128 H=1 d=64 fp32, one document", 128, 1, 1, 64, "f32", [128], seed=seed)
    elif idx == 2:
        w = Workload("batched 4x4096 H=16 d=128 bf16", 4 * 4096, 16, 16, 128, "bf16", [4096] * 4, seed=seed)
    elif idx == 3:
        lens = [l for r in range(8) for l in doc_lengths_lognormal(seed, r, 16384, 1500.0)]
        w = Workload("packed 8x16384 H=16 d=128 bf16, log-normal(1500) docs, outliers x20", 8 * 16384, 16,
                     16, 128, "bf16", lens, outlier_channels=2, seed=seed)
    elif idx == 4:
        lens = [l for r in range(4) for l in doc_lengths_lognormal(seed, r, 32768, 1500.0)]
        w = Workload("mixed NVFP4/FP8 packed 4x32768 H=16 d=128 bf16, log-normal(1500) docs, outliers x20",
                     4 * 32768, 16, 16, 128, "bf16", lens, outlier_channels=2, seed=seed)
    elif idx == 5:
        lens = [l for r in range(2) for l in doc_lengths_lognormal(seed, r, 65536, 6000.0)]
        w = Workload("long GQA 2x65536 H=32 Hkv=8 d=128 bf16, log-normal(6000) docs", 2 * 65536, 32, 8,
                     128, "bf16", lens, seed=seed)
    else:
        raise ValueError(idx)
    for k, v in over.items():
        setattr(w, k, v)
    return w


def custom(seqlens: list[int], H: int, d: int, Hkv: int | None = None, dtype: str = "bf16",
           seed: int = SEED_BASE + 100, outlier_channels: int = 0, name: str = "custom") -> Workload:
    """A small workload of the same recipe with explicit document lengths."""
    return Workload(name, int(sum(seqlens)), H, Hkv or H, d, dtype, list(seqlens),
                    outlier_channels=outlier_channels, seed=seed)
