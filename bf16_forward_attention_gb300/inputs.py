"""Seeded synthetic inputs for bf16 forward attention.

This module only draws numbers. It holds none of the attention arithmetic, so the
fp64 CPU oracle (test side) and the CUDA path (product side) can both be fed from
it without sharing any of the method.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), used counter-based: draw ``i`` of stream ``key`` is
``mix64(key + (i + 1) * GOLDEN)``. Normals come from the Box-Muller transform
(Box and Muller, 1958) on two 53-bit uniforms. Values are drawn in fp64, narrowed
to fp32, then rounded to bf16 (round to nearest, ties to even) by torch.

The workloads are the ones the attention pages describe: head_dim 128, BSHD or
BHSD, self- and cross-attention lengths, unit-normal Q/K/V; plus a stress case with
wide logits (Q, K ~ N(0, 8^2)), V ~ U(-1, 1) and one NaN in Q and one +Inf in K per
batch.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

LAYOUTS = ("bhsd", "bshd")
# Variable-length batches are packed token after token: (total tokens, heads, d),
# sequence b owning tokens cu_seqlens[b] .. cu_seqlens[b+1]-1.
ROUNDINGS = ("rtne", "rtna", "rtz")


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    """Key of an independent counter stream for (seed, stream id)."""
    with np.errstate(over="ignore"):
        base = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * GOLDEN + np.uint64(stream & 0xFFFFFFFF)
        return _mix64(np.array([base], dtype=np.uint64))[0]


def splitmix64(key: np.uint64, start: int, n: int) -> np.ndarray:
    """Draws ``start .. start+n-1`` of the counter stream ``key`` as uint64."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix64(key + idx * GOLDEN)


def _u01_open_low(bits: np.ndarray) -> np.ndarray:
    # (0, 1]: never 0, so log() below is finite.
    return ((bits >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def _u01(bits: np.ndarray) -> np.ndarray:
    # [0, 1)
    return (bits >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal_f32(seed: int, stream: int, n: int, std: float = 1.0) -> np.ndarray:
    """n draws of N(0, std^2) as float32 (Box-Muller, both outputs used)."""
    key = stream_key(seed, stream)
    out = np.empty(n, dtype=np.float32)
    pairs = (n + 1) // 2
    for p0 in range(0, pairs, _CHUNK):
        m = min(_CHUNK, pairs - p0)
        bits = splitmix64(key, 2 * p0, 2 * m)
        u1 = _u01_open_low(bits[0::2])
        u2 = _u01(bits[1::2])
        r = np.sqrt(-2.0 * np.log(u1)) * std
        th = (2.0 * math.pi) * u2
        blk = np.empty(2 * m, dtype=np.float64)
        blk[0::2] = r * np.cos(th)
        blk[1::2] = r * np.sin(th)
        lo = 2 * p0
        hi = min(n, lo + 2 * m)
        out[lo:hi] = blk[: hi - lo]
    return out


def uniform_f32(seed: int, stream: int, n: int, a: float, b: float) -> np.ndarray:
    """n draws of U(a, b) as float32."""
    key = stream_key(seed, stream)
    out = np.empty(n, dtype=np.float32)
    for s0 in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s0)
        out[s0 : s0 + m] = a + (b - a) * _u01(splitmix64(key, s0, m))
    return out


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """fp32 numpy array -> bf16 torch tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def shape_of(layout: str, B: int, H: int, S: int, D: int = 128) -> tuple:
    if layout == "bhsd":
        return (B, H, S, D)
    if layout == "bshd":
        return (B, S, H, D)
    raise ValueError(f"unknown layout {layout!r}")


def index_of(layout: str, b: int, h: int, s: int, c: int) -> tuple:
    return (b, h, s, c) if layout == "bhsd" else (b, s, h, c)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic attention problem (sizes, distributions, specials)."""

    name: str
    layout: str
    B: int
    H: int
    Sq: int
    Sk: int
    D: int = 128
    qk_std: float = 1.0
    v_dist: str = "normal"  # "normal" (N(0,1)) or "uniform" (U(-1,1))
    specials: bool = False  # one NaN in Q and one +Inf in K per batch
    roundings: tuple = ("rtne",)
    seed: int = 20260001
    splitkv: bool = False  # run with the key range split over CTAs
    causal: bool = False   # key j visible to query i iff j <= i + Sk - Sq
    hkv: int = 0           # key/value heads (grouped-query); 0 means H
    seqlens: tuple = ()    # variable-length batch: per-sequence (Sq_b, Sk_b); B, Sq, Sk
                           # then hold the count and the longest lengths

    @property
    def kv_heads(self) -> int:
        return self.hkv or self.H

    @property
    def visible_pairs(self) -> int:
        """(query, key) pairs one head computes: Sq*Sk, or under the causal mask
        sum over rows i of clamp(i + Sk - Sq + 1, 0, Sk). For a variable-length
        batch the sum over its sequences (then per head, not per batch entry)."""
        if self.seqlens:
            return sum(dataclasses.replace(self, seqlens=(), B=1, Sq=a, Sk=b).visible_pairs
                       for a, b in self.seqlens)
        if not self.causal:
            return self.Sq * self.Sk
        # Rows i < lo see no key; row i >= lo sees i + off + 1 keys (at most Sk,
        # reached by the last row).
        off = self.Sk - self.Sq
        lo = max(0, -off)
        n = self.Sq - lo
        return n * (lo + off + 1) + n * (n - 1) // 2

    @property
    def flops(self) -> int:
        """Counted work of one call: 4*D per visible (query, key) pair and head
        (QK^T and PV, 2 flops per MAC); 4*B*H*Sq*Sk*D without a mask."""
        if self.seqlens:
            return 4 * self.H * self.visible_pairs * self.D
        return 4 * self.B * self.H * self.visible_pairs * self.D

    @property
    def cu_seqlens(self) -> tuple:
        """(cu_seqlens_q, cu_seqlens_k) of a variable-length batch, as int32 arrays."""
        cq = np.concatenate([[0], np.cumsum([a for a, _ in self.seqlens])]).astype(np.int32)
        ck = np.concatenate([[0], np.cumsum([b for _, b in self.seqlens])]).astype(np.int32)
        return cq, ck

    @property
    def io_bytes(self) -> int:
        """Algorithmic bytes of one call: Q, K, V read once and O written once, bf16
        (K and V once per key/value head: the query tiles of a head share them)."""
        if self.seqlens:
            tq = sum(a for a, _ in self.seqlens)
            tk = sum(b for _, b in self.seqlens)
            return 2 * self.D * (2 * tq * self.H + 2 * tk * self.kv_heads)
        return 2 * self.D * self.B * (2 * self.Sq * self.H + 2 * self.Sk * self.kv_heads)

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def varlen_lengths(seed: int, n: int, lo: int, hi: int) -> tuple:
    """n seeded sequence lengths, uniform on the integers lo..hi."""
    r = splitmix64(stream_key(seed, 7), 0, n)
    return tuple(int(lo + int(x % np.uint64(hi - lo + 1))) for x in r)


# The five synthetic workloads: a tiny self-attention case, the 8K self-attention
# case in all three rounding modes, a 4K x 32K cross-attention case, the 128K
# long-context case and the ragged stress case.
WORKLOADS = {
    "tiny": Workload("tiny", "bhsd", 1, 2, 256, 256, roundings=("rtne",), seed=20260001),
    "self8k": Workload("self8k", "bshd", 2, 16, 8192, 8192,
                       roundings=("rtne", "rtna", "rtz"), seed=20260002),
    "cross4k32k": Workload("cross4k32k", "bhsd", 1, 32, 4096, 32768, roundings=("rtne",),
                           seed=20260003),
    "long128k": Workload("long128k", "bshd", 1, 8, 131072, 131072, roundings=("rtna",),
                         seed=20260004),
    "stress16381": Workload("stress16381", "bhsd", 4, 24, 16381, 16381, qk_std=8.0,
                            v_dist="uniform", specials=True, roundings=("rtz",),
                            seed=20260005),
    # Follow-on workloads: few query rows against long keys (split-KV path), the
    # 8K self-attention case under the causal mask, and with grouped-query heads
    # (16 query heads sharing 4 key/value heads).
    "decode32k": Workload("decode32k", "bhsd", 1, 8, 256, 32768, roundings=("rtne",),
                          seed=20260006, splitkv=True),
    "causal8k": Workload("causal8k", "bshd", 2, 16, 8192, 8192, roundings=("rtne",),
                         seed=20260007, causal=True),
    "gqa8k": Workload("gqa8k", "bshd", 2, 16, 8192, 8192, roundings=("rtne",),
                      seed=20260008, hkv=4),
    # Short key range: 16K query tokens against a 77-token context (the shape of
    # text cross-attention in image and video diffusion). Q and O dominate the
    # bytes, so the call is bound by HBM bandwidth, not by the tensor pipe.
    "short77": Workload("short77", "bshd", 2, 32, 16384, 77, roundings=("rtne",),
                        seed=20260010),
}
# Variable-length self-attention batch: 16 sequences of seeded lengths 256..16384
# (a mix around the 8K case), 16 heads, packed token after token.
_VL = varlen_lengths(20260009, 16, 256, 16384)
WORKLOADS["varlen16"] = Workload("varlen16", "thd", len(_VL), 16, max(_VL), max(_VL),
                                 roundings=("rtne",), seed=20260009,
                                 seqlens=tuple((n, n) for n in _VL))


def special_positions(w: Workload) -> list:
    """Per batch: (b, (h, i, c) of the NaN in Q, (h', j, c') of the +Inf in K)."""
    key = stream_key(w.seed, 99)
    out = []
    for b in range(w.B):
        r = splitmix64(key, 8 * b, 6)
        qpos = (int(r[0] % np.uint64(w.H)), int(r[1] % np.uint64(w.Sq)), int(r[2] % np.uint64(w.D)))
        kpos = (int(r[3] % np.uint64(w.kv_heads)), int(r[4] % np.uint64(w.Sk)), int(r[5] % np.uint64(w.D)))
        out.append((b, qpos, kpos))
    return out


def make_qkv(w: Workload) -> tuple:
    """Returns (q, k, v) as contiguous bf16 CPU tensors in the workload's layout
    (a variable-length batch: packed (total, heads, D))."""
    if w.seqlens:
        tq = sum(a for a, _ in w.seqlens)
        tk = sum(b for _, b in w.seqlens)
        q = normal_f32(w.seed, 0, tq * w.H * w.D, w.qk_std).reshape(tq, w.H, w.D)
        k = normal_f32(w.seed, 1, tk * w.kv_heads * w.D, w.qk_std).reshape(tk, w.kv_heads, w.D)
        v = normal_f32(w.seed, 2, tk * w.kv_heads * w.D, 1.0).reshape(tk, w.kv_heads, w.D)
        return to_bf16(q), to_bf16(k), to_bf16(v)
    nq = w.B * w.H * w.Sq * w.D
    nk = w.B * w.kv_heads * w.Sk * w.D
    q = normal_f32(w.seed, 0, nq, w.qk_std)
    k = normal_f32(w.seed, 1, nk, w.qk_std)
    if w.v_dist == "normal":
        v = normal_f32(w.seed, 2, nk, 1.0)
    elif w.v_dist == "uniform":
        v = uniform_f32(w.seed, 2, nk, -1.0, 1.0)
    else:
        raise ValueError(w.v_dist)
    qs = shape_of(w.layout, w.B, w.H, w.Sq, w.D)
    ks = shape_of(w.layout, w.B, w.kv_heads, w.Sk, w.D)
    q = q.reshape(qs)
    k = k.reshape(ks)
    v = v.reshape(ks)
    if w.specials:
        for b, (h, i, c), (h2, j, c2) in special_positions(w):
            q[index_of(w.layout, b, h, i, c)] = np.nan
            k[index_of(w.layout, b, h2, j, c2)] = np.inf
    return to_bf16(q), to_bf16(k), to_bf16(v)


def default_scale(D: int = 128) -> float:
    """1/sqrt(D) as the fp32 value both sides use."""
    return float(np.float32(1.0 / math.sqrt(D)))
