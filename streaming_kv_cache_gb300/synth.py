"""Seeded synthetic workloads for streaming view-major KV-cache attention.

This module only draws inputs: shapes, seeds, normally distributed bf16 tensors
and token ids.  It holds none of the attention, rotary or ring arithmetic, so
that both the CUDA path and the fp64 oracle can be fed the very same bits
without sharing any of the method's code.

Every tensor is drawn from numpy's PCG64 generator seeded by a stable hash of
(workload, step, cache, tensor name), as fp32 N(0, 1) (times an optional scale,
applied in fp32) and rounded to bf16 with round-to-nearest-even.  bf16 tensors
are returned as uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math

import numpy as np

VOCAB = 151936  # token-id range of the Qwen-family tokenizer the verify ids are drawn from


@dataclasses.dataclass(frozen=True)
class Workload:
    """Geometry of one streaming-attention workload.

    P prefix (system/text) tokens, V camera views, F frames per view in the
    sliding window, T tokens per frame; Hq query heads, Hkv key/value heads,
    head dimension d, rotary base theta.  C independent caches (model layers
    x batch) are processed by one call.
    """

    name: str
    P: int
    V: int
    F: int
    T: int
    Hq: int
    Hkv: int
    d: int
    theta: float
    C: int = 1
    q_scale: float = 1.0      # scale folded into Q when it is drawn
    sm_scale: float = 1.0     # softmax scale passed to the kernels
    tail_cap: int = 128       # rows reserved for reasoning tokens after the views
    steps: int = 1            # streaming steps after the initial fill
    tail_len: int = 0         # reasoning tokens already in the tail before a verify block
    blk: int = 9              # verify block: last accepted token + drafted tokens

    @property
    def n_window(self) -> int:
        """Keys in the visual window including the prefix: P + V*F*T."""
        return self.P + self.V * self.F * self.T

    @property
    def n_new(self) -> int:
        """New-frame query tokens per step: V*T."""
        return self.V * self.T

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _inv_sqrt(n: int) -> float:
    return 1.0 / math.sqrt(n)


# The five workloads: a tiny one the oracle finishes instantly, one streaming
# step of the Alpamayo-shaped 4-view x 4-frame window, 20 consecutive steps of
# it, speculative verify on that cache, and a 6-view x 8-frame scale-up over
# 36 layer caches.
WORKLOADS = {
    "tiny": Workload("tiny", P=8, V=2, F=2, T=16, Hq=4, Hkv=2, d=64, theta=1e4,
                     sm_scale=_inv_sqrt(64), tail_cap=32, steps=3),
    "alpamayo_step": Workload("alpamayo_step", P=256, V=4, F=4, T=180, Hq=32, Hkv=8, d=128,
                              theta=1e6, q_scale=_inv_sqrt(128), sm_scale=1.0, steps=1),
    "alpamayo_20steps": Workload("alpamayo_20steps", P=256, V=4, F=4, T=180, Hq=32, Hkv=8,
                                 d=128, theta=1e6, q_scale=_inv_sqrt(128), sm_scale=1.0,
                                 steps=20),
    "alpamayo_verify": Workload("alpamayo_verify", P=256, V=4, F=4, T=180, Hq=32, Hkv=8,
                                d=128, theta=1e6, q_scale=_inv_sqrt(128), sm_scale=1.0,
                                tail_len=16, blk=9, C=64),
    "scaleup_36L": Workload("scaleup_36L", P=512, V=6, F=8, T=256, Hq=32, Hkv=8, d=128,
                            theta=1e6, C=36, sm_scale=_inv_sqrt(128), steps=1),
}

VERIFY_BATCHES = (1, 8, 32, 64)


def seed_for(*parts) -> int:
    """Stable 64-bit seed from a tuple of names and numbers."""
    h = hashlib.blake2b("/".join(str(p) for p in parts).encode(), digest_size=8)
    return int.from_bytes(h.digest(), "little")


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def normal_bf16(shape, *seed_parts, scale: float = 1.0) -> np.ndarray:
    """N(0, 1) fp32 draw, times `scale` in fp32, rounded to bf16 bits."""
    rng = np.random.Generator(np.random.PCG64(seed_for(*seed_parts)))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return f32_to_bf16_bits(x)


# --- per-step tensors -------------------------------------------------------
# Token-major layouts, as a QKV projection emits them:
#   frame K/V  [C][V][T][Hkv][d]     new-frame Q  [C][V*T][Hq][d]
#   prefix K/V [C][P][Hkv][d]        tail K/V     [C][n][Hkv][d]
#   verify block Q [C][blk][Hq][d], K/V [C][blk][Hkv][d]
#   window Q [C][P+V*F*T][Hq][d]    tail-token Q [C][n][Hq][d], K/V [C][n][Hkv][d]

def prefix_kv(w: Workload, tag: str = ""):
    shp = (w.C, w.P, w.Hkv, w.d)
    return (normal_bf16(shp, w.name, tag, "prefix_k"), normal_bf16(shp, w.name, tag, "prefix_v"))


def frame_kv(w: Workload, insert_index: int, tag: str = ""):
    """K/V of the frame inserted by the `insert_index`-th insert (0-based,
    counting the initial fill)."""
    shp = (w.C, w.V, w.T, w.Hkv, w.d)
    return (normal_bf16(shp, w.name, tag, insert_index, "frame_k"),
            normal_bf16(shp, w.name, tag, insert_index, "frame_v"))


def frame_q(w: Workload, insert_index: int, tag: str = ""):
    shp = (w.C, w.n_new, w.Hq, w.d)
    return normal_bf16(shp, w.name, tag, insert_index, "frame_q", scale=w.q_scale)


def tail_kv(w: Workload, n: int, tag: str = ""):
    shp = (w.C, n, w.Hkv, w.d)
    return (normal_bf16(shp, w.name, tag, "tail_k"), normal_bf16(shp, w.name, tag, "tail_v"))


def window_q(w: Workload, tag: str = ""):
    """Queries of every window token, logical order: [C][P + V*F*T][Hq][d]."""
    return normal_bf16((w.C, w.n_window, w.Hq, w.d), w.name, tag, "window_q", scale=w.q_scale)


def tail_block(w: Workload, n: int, tag: str = ""):
    """Q, K, V of n tokens that follow the views (trajectory / text)."""
    q = normal_bf16((w.C, n, w.Hq, w.d), w.name, tag, n, "tail_q", scale=w.q_scale)
    k = normal_bf16((w.C, n, w.Hkv, w.d), w.name, tag, n, "tail_blk_k")
    v = normal_bf16((w.C, n, w.Hkv, w.d), w.name, tag, n, "tail_blk_v")
    return q, k, v


def verify_block(w: Workload, tag: str = ""):
    q = normal_bf16((w.C, w.blk, w.Hq, w.d), w.name, tag, "blk_q", scale=w.q_scale)
    k = normal_bf16((w.C, w.blk, w.Hkv, w.d), w.name, tag, "blk_k")
    v = normal_bf16((w.C, w.blk, w.Hkv, w.d), w.name, tag, "blk_v")
    return q, k, v


def planted_ids(n_batch: int, blk: int, *seed_parts):
    """Target and draft token ids [n_batch][blk] with a planted accept length.

    Slot 0 of `draft` is the last accepted token and is never compared.  For
    batch element b a prefix length k_b = b mod blk is planted:
    draft[b][i] = target[b][i-1] for 1 <= i <= k_b, and, when k_b < blk-1,
    draft[b][k_b+1] differs from target[b][k_b].  Returns (target, draft, k).
    """
    rng = np.random.Generator(np.random.PCG64(seed_for("ids", n_batch, blk, *seed_parts)))
    target = rng.integers(0, VOCAB, size=(n_batch, blk), dtype=np.int64).astype(np.int32)
    draft = rng.integers(0, VOCAB, size=(n_batch, blk), dtype=np.int64).astype(np.int32)
    k = np.arange(n_batch, dtype=np.int32) % blk
    for b in range(n_batch):
        kb = int(k[b])
        for i in range(1, kb + 1):
            draft[b, i] = target[b, i - 1]
        if kb + 1 < blk and draft[b, kb + 1] == target[b, kb]:
            draft[b, kb + 1] = (target[b, kb] + 1) % VOCAB
    return target, draft, k
