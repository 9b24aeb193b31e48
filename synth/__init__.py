"""Seeded synthetic inputs for the decode-step tests and the bench.

This module is shared by both sides of every parity check: the oracle side and the
CUDA side read the very same tensors it returns.  It therefore holds none of the
decode step's own arithmetic (no GEMV, no rotation, no softmax).  It holds:

* a counter-based random generator: SplitMix64 (Steele, Lea and Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014, with Vigna's 64-bit
  finaliser constants) evaluated at counter positions, so any element can be
  produced on its own and the result is the same on CPU and GPU;
* normal draws from it by the Box-Muller transform, in float64;
* the Q8_0 input encoding of a weight matrix (32 int8 values and one f16 scale
  per block, the scale being max|w|/127), which turns a float weight matrix into
  the block bytes the decode step consumes;
* the workload recipes: the shapes of the tiny, Llama-3.2-1B-like and
  Llama-3.2-3B-like layers, the row positions and the cache lengths.

Everything works on torch tensors on any device, so the bench can draw
gigabytes of weights straight into device memory with the same recipe the CPU
tests use.
"""

from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Dict, List, Optional, Sequence

import torch

__all__ = [
    "LayerShape", "TINY", "LLAMA_1B", "LLAMA_3B",
    "stream_id", "words", "uniform", "normal", "randint_inclusive",
    "quantize_q8_0", "q8_0_blocks_from_normal", "kv_cache_normal",
    "Q8_0_BLOCK", "Q8_0_BYTES",
]

Q8_0_BLOCK = 32          # weights per Q8_0 block
Q8_0_BYTES = 34          # bytes per block: f16 scale then 32 int8

_MASK64 = (1 << 64) - 1


def _s64(v: int) -> int:
    """Reinterpret an unsigned 64-bit constant as a signed int64 (torch has no uint64 math)."""
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


_GOLDEN = _s64(0x9E3779B97F4A7C15)
_MUL1 = _s64(0xBF58476D1CE4E5B9)
_MUL2 = _s64(0x94D049BB133111EB)


def _srl(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    """SplitMix64 output finaliser on int64 bit patterns (multiplication wraps mod 2^64)."""
    z = z ^ _srl(z, 30)
    z = z * _MUL1
    z = z ^ _srl(z, 27)
    z = z * _MUL2
    return z ^ _srl(z, 31)


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & _MASK64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_id(label: str) -> int:
    """A stable stream number for a tensor's label (CRC-32 of its UTF-8 bytes)."""
    return zlib.crc32(label.encode("utf-8"))


def _stream_key(seed: int, stream: int) -> int:
    return _mix64_int((seed & _MASK64) * 0x9E3779B97F4A7C15 + (stream & _MASK64) + 1)


def words(seed: int, stream: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """SplitMix64 words number start..start+n-1 of the generator keyed by (seed, stream).

    Word i is mix64(key + (i + 1) * golden), i.e. the i-th output of SplitMix64 started
    at state `key`; returned as int64 bit patterns.
    """
    key = _s64(_stream_key(seed, stream))
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    return _mix64(i * _GOLDEN + key)


def uniform(seed: int, stream: int, n: int, start: int = 0, device="cpu") -> torch.Tensor:
    """Doubles in the open interval (0, 1): ((word >> 11) + 0.5) * 2^-53."""
    w = _srl(words(seed, stream, start, n, device), 11)
    return (w.to(torch.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0,
           device="cpu", chunk: int = 1 << 24) -> torch.Tensor:
    """n float64 normal draws by Box-Muller: pair j uses words 2j and 2j+1.

    Output 2j is r*cos(2*pi*u2), output 2j+1 is r*sin(2*pi*u2), r = sqrt(-2 ln u1).
    Generated in chunks so large draws do not hold every intermediate at once.
    """
    out = torch.empty(n, dtype=torch.float64, device=device)
    pairs = (n + 1) // 2
    p0 = 0
    while p0 < pairs:
        pc = min(chunk, pairs - p0)
        u = uniform(seed, stream, 2 * pc, start=2 * p0, device=device).view(pc, 2)
        r = torch.sqrt(-2.0 * torch.log(u[:, 0]))
        t = (2.0 * math.pi) * u[:, 1]
        z = torch.stack((r * torch.cos(t), r * torch.sin(t)), dim=1).reshape(-1)
        e0 = 2 * p0
        e1 = min(n, e0 + 2 * pc)
        out[e0:e1] = z[: e1 - e0]
        p0 += pc
    if std != 1.0:
        out.mul_(std)
    if mean != 0.0:
        out.add_(mean)
    return out


def randint_inclusive(seed: int, stream: int, n: int, lo: int, hi: int) -> List[int]:
    """n integers uniform on [lo, hi], drawn as lo + floor(u * (hi - lo + 1))."""
    u = uniform(seed, stream, n)
    span = hi - lo + 1
    return [lo + min(span - 1, int(math.floor(float(v) * span))) for v in u]


def quantize_q8_0(w: torch.Tensor) -> torch.Tensor:
    """Encode a float32 matrix [n_out, n_in] as Q8_0 blocks, returned as uint8 [n_out, n_in/32, 34].

    Per block of 32 consecutive inputs of one output row: d32 = max|w| / 127 in float32;
    q = w / d32 rounded half away from zero and clamped to [-127, 127] (all zero when
    d32 == 0); the stored scale is d32 rounded to f16 (round to nearest even).  Bytes
    0-1 hold the f16 scale little-endian, bytes 2-33 the 32 int8 values in input order.
    This is how the test inputs are made; both sides of a parity check then read the
    same bytes.
    """
    assert w.dim() == 2 and w.shape[1] % Q8_0_BLOCK == 0
    n_out, n_in = w.shape
    nb = n_in // Q8_0_BLOCK
    wb = w.to(torch.float32).reshape(n_out, nb, Q8_0_BLOCK)
    amax = wb.abs().amax(dim=2, keepdim=True)
    d32 = amax / 127.0
    safe = torch.where(d32 > 0, d32, torch.ones_like(d32))
    t = wb / safe
    q = torch.sign(t) * torch.floor(t.abs() + 0.5)
    q = torch.where(d32 > 0, q, torch.zeros_like(q)).clamp_(-127, 127).to(torch.int8)
    d16 = d32.to(torch.float16).view(torch.int16)
    out = torch.empty(n_out, nb, Q8_0_BYTES, dtype=torch.uint8, device=w.device)
    out[:, :, 0] = (d16[:, :, 0] & 0xFF).to(torch.uint8)
    out[:, :, 1] = ((d16[:, :, 0] >> 8) & 0xFF).to(torch.uint8)
    out[:, :, 2:] = q.view(torch.uint8)
    return out


def q8_0_blocks_from_normal(seed: int, label: str, n_out: int, n_in: int, std: float = 0.02,
                            device="cpu", rows_per_chunk: int = 2048) -> torch.Tensor:
    """Q8_0 blocks of an [n_out, n_in] weight matrix drawn w ~ N(0, std^2), element
    (o, i) being normal draw o*n_in + i of stream `label`."""
    sid = stream_id(label)
    out = torch.empty(n_out, n_in // Q8_0_BLOCK, Q8_0_BYTES, dtype=torch.uint8, device=device)
    for r0 in range(0, n_out, rows_per_chunk):
        r1 = min(n_out, r0 + rows_per_chunk)
        # draw the chunk's elements at their global counter positions
        z = _normal_range(seed, sid, r0 * n_in, (r1 - r0) * n_in, device)
        w = (z * std).to(torch.float32).view(r1 - r0, n_in)
        out[r0:r1] = quantize_q8_0(w)
    return out


def f16_weights_from_normal(seed: int, label: str, n_out: int, n_in: int, std: float = 0.02,
                            device="cpu", rows_per_chunk: int = 2048) -> torch.Tensor:
    """An f16 [n_out, n_in] weight matrix drawn w ~ N(0, std^2) and rounded to f16 (RNE), element
    (o, i) being normal draw o*n_in + i of stream `label`."""
    sid = stream_id(label)
    out = torch.empty(n_out, n_in, dtype=torch.float16, device=device)
    for r0 in range(0, n_out, rows_per_chunk):
        r1 = min(n_out, r0 + rows_per_chunk)
        z = _normal_range(seed, sid, r0 * n_in, (r1 - r0) * n_in, device)
        out[r0:r1] = (z * std).to(torch.float32).view(r1 - r0, n_in).to(torch.float16)
    return out


def _normal_range(seed: int, stream: int, first: int, n: int, device) -> torch.Tensor:
    """Normal draws first..first+n-1 of a stream (Box-Muller pairs aligned to even indices)."""
    p0 = first // 2
    p1 = (first + n + 1) // 2
    u = uniform(seed, stream, 2 * (p1 - p0), start=2 * p0, device=device).view(-1, 2)
    r = torch.sqrt(-2.0 * torch.log(u[:, 0]))
    t = (2.0 * math.pi) * u[:, 1]
    z = torch.stack((r * torch.cos(t), r * torch.sin(t)), dim=1).reshape(-1)
    off = first - 2 * p0
    return z[off: off + n]


def kv_cache_normal(seed: int, label: str, n_regions: int, n_kv: int, capacity: int, head_dim: int,
                    device="cpu") -> torch.Tensor:
    """An f16 cache plane [n_regions, n_kv, capacity, head_dim] filled with N(0,1) draws (RNE to f16)."""
    n = n_regions * n_kv * capacity * head_dim
    z = _normal_range(seed, stream_id(label), 0, n, device)
    return z.to(torch.float32).to(torch.float16).view(n_regions, n_kv, capacity, head_dim)


def kv_q8_random_planes(seed: int, label: str, n_regions: int, n_kv: int, capacity: int, head_dim: int,
                        device="cpu"):
    """Random q8_0-mirror planes: int8 codes uniform in [-127, 127] and f16 scales uniform in
    [0.005, 0.015), one per 32 values (plain draws, no encoding)."""
    n = n_regions * n_kv * capacity * head_dim
    u = uniform(seed, stream_id(label + "/codes"), n, device=device)
    codes = (torch.floor(u * 255.0) - 127.0).clamp_(-127, 127).to(torch.int8)
    us = uniform(seed, stream_id(label + "/scales"), n // 32, device=device)
    scales = (0.005 + 0.01 * us).to(torch.float32).to(torch.float16)
    return (codes.view(n_regions, n_kv, capacity, head_dim),
            scales.view(n_regions, n_kv, capacity, head_dim // 32))


def normal_f32(seed: int, label: str, shape: Sequence[int], std: float = 1.0, device="cpu") -> torch.Tensor:
    """float32 N(0, std^2) draws of the given shape from stream `label`."""
    n = 1
    for s in shape:
        n *= int(s)
    z = _normal_range(seed, stream_id(label), 0, n, device)
    return (z * std).to(torch.float32).view(*shape)


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Projection and attention shape of one decoder layer."""
    name: str
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    rope_theta: float = 500000.0

    @property
    def qkv_out(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim

    @property
    def group(self) -> int:
        return self.n_q // self.n_kv

    def projections(self) -> Dict[str, tuple]:
        """(n_out, n_in) of each Q8_0 projection of the layer step (gate and up concatenated)."""
        p = {
            "wqkv": (self.qkv_out, self.hidden),
            "wo": (self.n_q * self.head_dim, self.hidden) if self.n_q * self.head_dim == self.hidden
            else (self.hidden, self.n_q * self.head_dim),
        }
        if self.ffn:
            p["wgu"] = (2 * self.ffn, self.hidden)
            p["wdown"] = (self.hidden, self.ffn)
        return p


# Tiny layer: hidden 256, 4 query / 2 KV heads of 64; Wq/Wk/Wv/Wo only (no FFN).
TINY = LayerShape("tiny", hidden=256, n_q=4, n_kv=2, head_dim=64, ffn=0)
# Llama-3.2-1B-like layer: hidden 2048, 32/8 heads of 64, FFN 8192.
LLAMA_1B = LayerShape("llama-3.2-1b", hidden=2048, n_q=32, n_kv=8, head_dim=64, ffn=8192)
# Llama-3.2-3B-like layer: hidden 3072, 24/8 heads of 128, FFN 8192.
LLAMA_3B = LayerShape("llama-3.2-3b", hidden=3072, n_q=24, n_kv=8, head_dim=128, ffn=8192)


def twelve_stream_lengths(seed: int = 0, n: int = 12, lo: int = 512, hi: int = 8192) -> List[int]:
    """Per-stream cache lengths of the twelve-stream workload, uniform on [lo, hi]."""
    return randint_inclusive(seed, stream_id("streams/lengths"), n, lo, hi)
