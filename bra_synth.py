"""Seeded synthetic inputs for the Bi-Level Routing Attention (BRA) forward.

This module only draws numbers and lays them out. It holds none of BRA's
arithmetic (no pooling, affinity, routing, attention or convolution), so both
the CPU oracle and the CUDA path may take their inputs from it.

Random numbers
--------------
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014, with the output mix constants of Vigna's public
reference version) gives a counter-based stream: output i (i = 1, 2, ...) of
seed s is mix(s + i * 0x9E3779B97F4A7C15). Uniforms take the top 53 bits. Two
uniforms make two standard normals by the Box-Muller transform
(Box and Muller, 1958): r = sqrt(-2 ln u1), n0 = r cos(2 pi u2),
n1 = r sin(2 pi u2), with u1 in (0, 1] and u2 in [0, 1).

Each array draws from its own stream, seed = 256 * seed + stream id:
q offsets 0, q noise 1, k offsets 2, k noise 3, v offsets 4, v noise 5,
LePE weights 6, LePE bias 7.

Value recipe (the workload statement: per-region offset N(0,1) plus per-token
N(0, 0.5^2); LePE weights N(0, 0.02^2))
  x[b, y, x, c] = off[b, region(y, x), c] + 0.5 * noise[b, y, x, c]
for x in {q, k, v}, with one offset per (image, region, channel) shared by the
region's tokens, regions numbered row-major on the S x S grid. LePE weights
w[c, u, v] = 0.02 * N(0,1) and bias[c] = 0.02 * N(0,1). Values are rounded to
float32 (round to nearest even) and, for bf16 workloads, then to bfloat16
(round to nearest even), so every returned float32 holds the exact value both
sides consume.
"""
from __future__ import annotations

import dataclasses

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One BRA problem: shapes, routing parameters and arithmetic type."""

    name: str
    B: int
    H: int
    W: int
    C: int
    heads: int
    S: int
    topk: int
    ks: int
    dtype: str  # "f32" or "bf16"

    @property
    def R(self) -> int:
        return self.S * self.S

    @property
    def n(self) -> int:
        return (self.H // self.S) * (self.W // self.S)

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.W

    def describe(self) -> dict:
        return dict(name=self.name, B=self.B, H=self.H, W=self.W, C=self.C,
                    heads=self.heads, d=self.C // self.heads, S=self.S,
                    tokens_per_region=self.n, topk=self.topk,
                    lepe_kernel=self.ks, dtype=self.dtype)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five BiFormer-shaped workloads: ImageNet-224 stage shapes at strides
# 4, 8 and 16 with stage top-k 1 / 4 / 16, and a 512x512 dense-prediction map
# at stride 4 with S = 16; plus a tiny float32 case.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 14, 14, 64, 2, 7, 4, 5, "f32"),
    "stage1_bf16": Workload("stage1_bf16", 64, 56, 56, 64, 2, 7, 1, 5, "bf16"),
    "stage2_bf16": Workload("stage2_bf16", 64, 28, 28, 128, 4, 7, 4, 5, "bf16"),
    "stage3_bf16": Workload("stage3_bf16", 64, 14, 14, 256, 8, 7, 16, 5, "bf16"),
    "seg512_bf16": Workload("seg512_bf16", 8, 128, 128, 64, 2, 16, 4, 5, "bf16"),
}


def rank_slice(per_rank: int, rank: int) -> slice:
    """Images of a world * per_rank batch that rank `rank` draws and runs:
    a contiguous block, so the shards of all ranks tile the batch."""
    return slice(rank * per_rank, (rank + 1) * per_rank)


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start+1 .. start+count of SplitMix64 seeded with `seed`."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def normals(seed: int, count: int) -> np.ndarray:
    """`count` standard normals (float64) from the start of one stream."""
    return normals_range(seed, 0, count)


def round_bf16(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), as float32."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    bits = x32.view(np.uint32).astype(np.uint64)
    bits = (bits + np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1)))
    bits = (bits & np.uint64(0xFFFF0000)).astype(np.uint32)
    return bits.view(np.float32).reshape(x32.shape)


def bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already exact bfloat16."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    return (x32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _region_field(off: np.ndarray, H: int, W: int, S: int) -> np.ndarray:
    """Broadcast per-region offsets [B, S*S, C] to tokens [B, H, W, C]."""
    B, _, C = off.shape
    hr, wr = H // S, W // S
    grid = off.reshape(B, S, 1, S, 1, C)
    return np.broadcast_to(grid, (B, S, hr, S, wr, C)).reshape(B, H, W, C)


@dataclasses.dataclass
class Inputs:
    """Input arrays as float32 holding exact values of the workload's type."""

    q: np.ndarray  # [B, H, W, C]
    k: np.ndarray
    v: np.ndarray
    lepe_w: np.ndarray  # [C, ks, ks]
    lepe_b: np.ndarray  # [C]


def _round(x: np.ndarray, dtype: str) -> np.ndarray:
    x32 = x.astype(np.float32)
    return round_bf16(x32) if dtype == "bf16" else x32


def make_inputs(wl: Workload, seed: int = 0, batch: slice | None = None,
                noise_std: float = 0.5) -> Inputs:
    """Draw the seeded inputs of workload `wl`.

    `batch` selects a contiguous range of images; the values of an image do not
    depend on which other images are drawn, so a slice equals the same slice of
    the full batch.
    """
    if wl.H % wl.S or wl.W % wl.S:
        raise ValueError("H and W must be multiples of S")
    b0, b1 = (0, wl.B) if batch is None else (batch.start or 0, batch.stop)
    nb = b1 - b0
    R, C, H, W = wl.R, wl.C, wl.H, wl.W
    tensors = []
    for t in range(3):
        s_off = seed * 256 + 2 * t
        s_noise = s_off + 1
        off = _slice_stream(s_off, b0, nb, R * C).reshape(nb, R, C)
        noise = _slice_stream(s_noise, b0, nb, H * W * C).reshape(nb, H, W, C)
        x = _region_field(off, H, W, wl.S) + noise_std * noise
        tensors.append(_round(x, wl.dtype))
    w = 0.02 * normals(seed * 256 + 6, C * wl.ks * wl.ks)
    bias = 0.02 * normals(seed * 256 + 7, C)
    return Inputs(tensors[0], tensors[1], tensors[2],
                  w.astype(np.float32).reshape(C, wl.ks, wl.ks),
                  bias.astype(np.float32))


def _slice_stream(seed: int, b0: int, nb: int, per_image: int) -> np.ndarray:
    """Normals for images b0 .. b0+nb-1 of a stream laid out image by image.

    Box-Muller pairs are aligned to the stream, so drawing a slice reproduces
    exactly the values a full draw puts there.
    """
    start, count = b0 * per_image, nb * per_image
    lo = start - (start % 2)
    full = normals_range(seed, lo, count + (start - lo))
    return full[start - lo:start - lo + count]


def normals_range(seed: int, first: int, count: int) -> np.ndarray:
    """Normals number first .. first+count-1 of a stream (first is even)."""
    assert first % 2 == 0
    pairs = (count + 1) // 2
    z = splitmix64(seed, first, 2 * pairs)
    scale = 2.0 ** -53
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * scale
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * scale
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * pairs, dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    return out[:count]


def make_projection_inputs(M: int, C: int, seed: int = 0):
    """Seeded inputs of the Q/K/V projection: x [M, C] (N(0,1) per element),
    w [3C, C] (N(0, 1/C), the scale of a default-initialised linear layer),
    bias [3C] (0.02 N(0,1)); x and w rounded to bfloat16, all returned as
    float32 holding the exact values both sides consume. Streams: seed * 256
    + 8 (x), + 9 (w), + 10 (bias)."""
    x = normals(seed * 256 + 8, M * C).reshape(M, C)
    w = normals(seed * 256 + 9, 3 * C * C).reshape(3 * C, C) / np.sqrt(C)
    b = 0.02 * normals(seed * 256 + 10, 3 * C)
    return (round_bf16(x.astype(np.float32)), round_bf16(w.astype(np.float32)),
            b.astype(np.float32))
