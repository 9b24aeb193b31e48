"""Seeded test workloads and the comparison rules of the parity tests.

Inputs come from `synth` only; expected values from `oracle` only.  The
tolerances are the decode step's stated bars:
  * GEMV outputs within 1e-3 relative error of the fp64 oracle, per element
    |y - ref| <= 1e-3 * max(|ref|, rms(ref over the row));
  * stored f16 K/V values within 1 ulp (distance of the ordered binary16
    encodings), the KV-store indexing bit-exact;
  * attention outputs within 2e-3 max abs error, LSE within 1e-4 relative.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import synth

GEMV_RTOL = 1e-3
ATTN_ATOL = 2e-3
LSE_RTOL = 1e-4
KV_ULP = 1


def gemv_err(y, ref) -> float:
    """Largest |y - ref| / max(|ref|, rms(ref row)) over all elements."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    den = np.maximum(np.abs(ref), rms)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(np.abs(y - ref) / den))


def assert_gemv_close(y, ref):
    e = gemv_err(y, ref)
    assert e <= GEMV_RTOL, "GEMV relative error %.3g > %.1g" % (e, GEMV_RTOL)
    return e


def ordered_f16(bits) -> np.ndarray:
    """binary16 bit patterns -> integers ordered like the values (+0 and -0 both 0)."""
    b = np.asarray(bits).view(np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def f16_ulp_dist(a, b) -> np.ndarray:
    return np.abs(ordered_f16(a) - ordered_f16(b))


def assert_attn_close(out, lse, ref_out, ref_lse):
    out = np.asarray(out, np.float64)
    lse = np.asarray(lse, np.float64)
    e_out = float(np.max(np.abs(out - ref_out)))
    e_lse = float(np.max(np.abs(lse - ref_lse) / np.abs(ref_lse)))
    assert e_out <= ATTN_ATOL, "attention max abs error %.3g > %.1g" % (e_out, ATTN_ATOL)
    assert e_lse <= LSE_RTOL, "LSE relative error %.3g > %.1g" % (e_lse, LSE_RTOL)
    return e_out, e_lse


@functools.lru_cache(maxsize=16)
def layer_blocks(shape_name: str, seed: int = 0, layer: int = 0):
    """Q8_0 interchange blocks (CPU uint8) of one layer's projections, w ~ N(0, 0.02^2)."""
    S = {s.name: s for s in (synth.TINY, synth.LLAMA_1B, synth.LLAMA_3B)}[shape_name]
    out = {}
    for name, (n_out, n_in) in S.projections().items():
        out[name] = synth.q8_0_blocks_from_normal(seed, "%s/L%d/%s" % (S.name, layer, name), n_out, n_in)
    return out


def kv_planes(label: str, n_regions: int, n_kv: int, capacity: int, D: int, seed: int = 0):
    """K and V f16 planes filled with N(0,1) draws (CPU tensors)."""
    k = synth.kv_cache_normal(seed, label + "/K", n_regions, n_kv, capacity, D)
    v = synth.kv_cache_normal(seed, label + "/V", n_regions, n_kv, capacity, D)
    return k, v


def as_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
