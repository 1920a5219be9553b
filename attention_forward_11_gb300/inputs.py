"""Seeded synthetic inputs and the workload table.

This module holds no attention arithmetic.  It draws Q, K, V as bf16 bit
patterns (numpy uint16) from numpy's PCG64 generator, the same bits on any
machine, so the CUDA path and the fp64 oracle see identical inputs.  Values are
drawn as fp32 normals N(0, sigma^2) and rounded to bf16 (round to nearest,
ties to even) -- the pages draw their benchmark inputs as normals too (the
Pallas page's ``main`` uses ``jax.random.normal``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    causal: int          # 0: no mask, 1: causal, bottom-right aligned (top-left when Sq == Skv)
    q_sigma: float = 1.0
    kv_sigma: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def as_dict(self) -> dict:
        return {"workload": self.name, "B": self.B, "Hq": self.Hq, "Hkv": self.Hkv,
                "Sq": self.Sq, "Skv": self.Skv, "D": self.D, "causal": self.causal,
                "scale": self.scale, "q_sigma": self.q_sigma, "kv_sigma": self.kv_sigma}


# The five benchmark shapes of this attention forward (D = 128, bf16).
WORKLOADS = {
    "tiny_causal": Workload("tiny_causal", 1, 2, 2, 256, 256, 128, 1),
    "tiny_noncausal": Workload("tiny_noncausal", 1, 2, 2, 256, 256, 128, 0),
    "mha_causal_4x16x4096": Workload("mha_causal_4x16x4096", 4, 16, 16, 4096, 4096, 128, 1),
    "gqa_causal_2x32x8_8192": Workload("gqa_causal_2x32x8_8192", 2, 32, 8, 8192, 8192, 128, 1),
    "long_sharp_1x16x16384": Workload("long_sharp_1x16x16384", 1, 16, 16, 16384, 16384, 128, 0,
                                      q_sigma=4.0),
    "chunked_prefill_gqa_64x8_512x32768": Workload("chunked_prefill_gqa_64x8_512x32768", 1, 64,
                                                   8, 512, 32768, 128, 1),
    # the headline shape at head sizes 64 and 256 (the Pallas page's benchmark sweeps 64, 128, 256)
    "mha_causal_4x16x4096_d64": Workload("mha_causal_4x16x4096_d64", 4, 16, 16, 4096, 4096, 64, 1),
    "mha_causal_4x16x4096_d256": Workload("mha_causal_4x16x4096_d256", 4, 16, 16, 4096, 4096, 256, 1),
    # a decode-like split-KV shape: one query row per sequence against 32K keys, GQA 8/1
    "decode_gqa_8x1_b8_1x32768": Workload("decode_gqa_8x1_b8_1x32768", 8, 8, 1, 1, 32768, 128, 1),
}

HEADLINE = "mha_causal_4x16x4096"


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def normal_bf16(shape, sigma: float, seed: int, stream: int, dtype: str = "bf16") -> np.ndarray:
    """16-bit patterns of N(0, sigma^2) draws from PCG64 seeded with (seed, stream):
    bf16 (default) or IEEE binary16 ("f16", numpy's round-to-nearest-even)."""
    rng = np.random.Generator(np.random.PCG64([seed, stream]))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    return f32_to_bf16_bits(x)


def make_qkv(B, Sq, Skv, Hq, Hkv, D, seed: int = 0, q_sigma: float = 1.0,
             kv_sigma: float = 1.0, dtype: str = "bf16"):
    """Q [B,Sq,Hq,D], K and V [B,Skv,Hkv,D] as uint16 bit patterns (streams 0, 1, 2)."""
    q = normal_bf16((B, Sq, Hq, D), q_sigma, seed, 0, dtype)
    k = normal_bf16((B, Skv, Hkv, D), kv_sigma, seed, 1, dtype)
    v = normal_bf16((B, Skv, Hkv, D), kv_sigma, seed, 2, dtype)
    return q, k, v


def make_workload(w: Workload, seed: int = 0):
    return make_qkv(w.B, w.Sq, w.Skv, w.Hq, w.Hkv, w.D, seed, w.q_sigma, w.kv_sigma)


def sample_rows(B, Hq, Sq, n: int, seed: int, extra_rows=()) -> np.ndarray:
    """(b, h, i) rows to check at full size: row 0, the last row, the rows around
    every 128-row tile edge of one head, and n uniform draws; deduplicated."""
    rng = np.random.Generator(np.random.PCG64([seed, 99]))
    rows = set()
    for b in {0, B - 1}:
        for h in {0, Hq - 1}:
            for i in (0, Sq - 1, *extra_rows):
                if 0 <= i < Sq:
                    rows.add((b, h, i))
    for edge in range(0, Sq, 128):
        for i in (edge, edge + 127):
            if i < Sq:
                rows.add((B - 1, Hq // 2, i))
    bb = rng.integers(0, B, n)
    hh = rng.integers(0, Hq, n)
    ii = rng.integers(0, Sq, n)
    rows.update(zip(bb.tolist(), hh.tolist(), ii.tolist()))
    return np.array(sorted(rows), dtype=np.int64)
