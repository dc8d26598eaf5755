"""Seeded synthetic workloads for causal attention (forward, backward, backward-over-backward).

This module holds only shapes and random-number recipes.  It contains none of
the attention arithmetic, so both the CPU oracle and the GPU tests/bench can
draw identical inputs from it without sharing any of the method's code.

Every tensor is laid out [B, H, N, d] (batch, heads, sequence, head dim), the
layout the FlashAttention tutorial page ("Flash attention for trading models",
section "Eight-line integration") gives for q, k, v.

Random streams.  Each (tensor, batch, head) slice has its own PCG64 stream,
keyed by SeedSequence(seed, spawn_key=(tensor_id, b, h)); a slice is drawn as
float32 standard normals with NumPy's float32 ziggurat.  Slices are therefore
reproducible one at a time, which lets the oracle regenerate just the heads it
checks at long sequence lengths.

bf16 configurations round the float32 draws to bfloat16 with
round-to-nearest-even and keep them as float32 holding bf16-exact values; the
GPU side converts those to bf16 losslessly and the oracle widens them to
float64 losslessly, so both sides see bit-identical inputs.
"""
from __future__ import annotations

import dataclasses
import numpy as np

# Tensor ids for the per-slice streams (order matters only for stream keys).
TENSORS = ("Q", "K", "V", "dO", "gdQ", "gdK", "gdV")
# Key-side tensors: with grouped key/value heads these have H / group heads.
KV_TENSORS = ("K", "V", "gdK", "gdV")
_TID = {name: i for i, name in enumerate(TENSORS)}
_TID_SHARED_MEAN = 100  # per-head shared key mean of the large-key workload
_TID_PERM = 101         # per-slice earlier-position draw of the large-key workload
_TID_QNOISE = 102       # per-slice query noise of the large-key workload
_TID_SEGMENTS = 103     # per-batch-row document lengths of the document-mask workloads


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str          # "f32" or "bf16": the arithmetic type of the inputs
    kind: str = "iid"   # "iid" or "large_key"
    dO_std: float = 1.0
    seed: int = 0
    group: int = 1      # query heads per key/value head: K, V, gdK, gdV have H / group heads

    @property
    def Hkv(self) -> int:
        return self.H // self.group

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    @property
    def rows(self) -> int:
        return self.B * self.H * self.N

    def with_n(self, N: int) -> "Workload":
        return dataclasses.replace(self, N=N, name=f"{self.name.split('@')[0]}@N{N}")


# The five workloads the method is checked on, plus the headline throughput shape.
TINY_F32 = Workload("tiny_f32_B1H1N256d64", 1, 1, 256, 64, "f32")
GPT2_LAYER = Workload("gpt2small_B4H12N1024d64", 4, 12, 1024, 64, "bf16")
LONG_SWEEP = tuple(Workload(f"long_B1H12d64@N{n}", 1, 12, n, 64, "bf16")
                   for n in (4096, 16384, 65536, 262144))
FULL_DAY = Workload("fullday_B2H12N23400d64", 2, 12, 23400, 64, "bf16", dO_std=0.1)
LARGE_KEY = Workload("largekey_B8H8N2048d128", 8, 8, 2048, 128, "bf16", kind="large_key")
GPT2_N8192 = Workload("gpt2small_B4H12N8192d64", 4, 12, 8192, 64, "bf16")


def _rng(seed: int, key: tuple) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=key)))


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); return float32.

    Input preparation only (finite inputs assumed)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _normal(w: Workload, name: str, b: int, h: int) -> np.ndarray:
    return _rng(w.seed, (_TID[name], b, h)).standard_normal((w.N, w.d), dtype=np.float32)


def _large_key_slice(w: Workload, b: int, h: int) -> dict:
    """Late-training large-key regime (GProj page, "How the zero sum turns into a
    false gradient"): keys share a large per-head mean of norm 40, each query is half
    of the key at a random earlier position plus N(0, 0.5^2) noise."""
    g = _rng(w.seed, (_TID_SHARED_MEAN, 0, h)).standard_normal(w.d)
    m = 40.0 * g / np.linalg.norm(g)
    K = m[None, :] + _normal(w, "K", b, h).astype(np.float64)
    r = _rng(w.seed, (_TID_PERM, b, h))
    i = np.arange(w.N)
    # pi(0) = 0; pi(i) uniform on {0, ..., i-1} for i >= 1
    pi = np.where(i == 0, 0, np.floor(r.random(w.N) * np.maximum(i, 1)).astype(np.int64))
    pi = np.minimum(pi, np.maximum(i - 1, 0))
    qn = _rng(w.seed, (_TID_QNOISE, b, h)).standard_normal((w.N, w.d))
    Q = 0.5 * K[pi] + 0.5 * qn
    return {"Q": Q.astype(np.float32), "K": K.astype(np.float32)}


def slice_inputs(w: Workload, b: int, h: int, names=TENSORS) -> dict:
    """Inputs of one (b, h) slice as float32 arrays [N, d] (bf16-exact for bf16 workloads)."""
    out = {}
    special = _large_key_slice(w, b, h) if w.kind == "large_key" else {}
    for name in names:
        if name in special:
            x = special[name]
        else:
            x = _normal(w, name, b, h)
            if name == "dO" and w.dO_std != 1.0:
                x = x * np.float32(w.dO_std)
        if w.dtype == "bf16":
            x = round_to_bf16(x)
        out[name] = x
    return out


def inputs(w: Workload, names=TENSORS, heads=None, batches=None) -> dict:
    """Full inputs [B', H', N, d] float32 for the selected batches/heads (default: all).

    With w.group > 1 the key-side tensors (KV_TENSORS) hold heads 0 .. H/group - 1 and
    are drawn from the same per-slice streams; only full inputs are offered then."""
    if w.group != 1 and (heads is not None or w.kind != "iid" or w.H % w.group):
        raise ValueError("grouped key/value heads: full iid inputs only, group dividing H")
    batches = range(w.B) if batches is None else list(batches)
    heads = range(w.H) if heads is None else list(heads)
    def nheads(n):
        return w.Hkv if (w.group != 1 and n in KV_TENSORS) else len(heads)
    out = {n: np.empty((len(batches), nheads(n), w.N, w.d), dtype=np.float32) for n in names}
    for bi, b in enumerate(batches):
        for hi, h in enumerate(heads):
            here = [n for n in names if hi < nheads(n)]
            s = slice_inputs(w, b, h, here)
            for n in here:
                out[n][bi, hi] = s[n]
    return out


def segment_ids(B: int, N: int, mean_len: int, seed: int = 0) -> np.ndarray:
    """Document ids [B, N] int32 of a packed batch: each row is cut into documents of
    random lengths drawn uniformly from 1 .. 2 mean_len - 1 (the last one clipped at N),
    numbered 0, 1, 2, ... along the row, so the ids are non-decreasing and each document
    is one run.  Only random draws: no attention arithmetic."""
    out = np.empty((B, N), dtype=np.int32)
    for b in range(B):
        r = _rng(seed, (_TID_SEGMENTS, b, 0))
        pos, doc = 0, 0
        while pos < N:
            n = int(r.integers(1, 2 * mean_len))
            out[b, pos:pos + n] = doc
            pos += n
            doc += 1
    return out
