"""Pins of the CPU oracle to facts fixed outside it (CPU only).

Each test checks the oracle against something other than itself: the IEEE 754
binary16 encoding, numpy's own float16 rounding, a numpy dequantise-then-matmul
written from the Q8_0 byte layout, complex multiplication, closed forms of
softmax attention, scipy's logsumexp, and brute force over small cases.  The
negative controls at the end plant a mistake in a copy of the oracle's inputs
or results and show that the comparison notices.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ----------------------------------------------------------------- binary16

def test_half_golden_encodings():
    """Encodings fixed by IEEE 754-2008 binary16 (tests/golden/binary16.txt)."""
    for hexbits, value in _read_golden("binary16.txt"):
        h = int(hexbits, 16)
        v = float.fromhex(value) if value.startswith(("0x", "-0x")) else float(value)
        if math.isnan(v):
            assert math.isnan(oracle.half_to_double(h))
            continue
        assert oracle.half_to_double(h) == v, hexbits
        if not math.isinf(v):
            assert oracle.double_to_half(v) == h, hexbits


def test_half_roundtrip_exhaustive():
    """Every finite binary16 value survives decode then encode."""
    L = oracle.lib()
    for h in range(0x10000):
        e = (h >> 10) & 0x1F
        if e == 31 and (h & 0x3FF):
            continue
        assert L.orc_double_to_half(L.orc_half_to_double(h)) == h, hex(h)


def test_half_rounding_matches_numpy():
    """Round-to-nearest-even against numpy's float64 -> float16 conversion,
    including exact ties, subnormals and values near the overflow threshold."""
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000))
    for h in range(0, 0x7C00, 97):          # midpoints between neighbours are exact ties
        a = oracle.half_to_double(h)
        b = oracle.half_to_double(h + 1)
        vals += [(a + b) / 2, -(a + b) / 2, a + (b - a) * 0.49, a + (b - a) * 0.51]
    vals += [65504.0, 65519.99, 65520.0, 1e5, -1e5, 2.0 ** -25, 2.0 ** -24, 2.0 ** -25 * 1.5, 0.0]
    for v in vals:
        with np.errstate(over="ignore"):
            want = int(np.array([v], np.float64).astype(np.float16).view(np.uint16)[0])
        assert oracle.double_to_half(float(v)) == want, v


# ---------------------------------------------------------------- Q8_0 GEMV

def _numpy_dequant(blocks):
    """Dequantise from the byte layout with numpy views (independent of the oracle's C)."""
    b = np.ascontiguousarray(blocks.numpy() if hasattr(blocks, "numpy") else blocks)
    d = b[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    q = b[:, :, 2:].copy().view(np.int8).astype(np.float64)
    return (q * d[:, :, None]).reshape(b.shape[0], -1)


@pytest.mark.parametrize("n_out,n_in,rows", [(5, 32, 1), (37, 256, 3), (64, 512, 8)])
def test_gemv_matches_dequant_matmul(n_out, n_in, rows):
    blocks = synth.q8_0_blocks_from_normal(7, "pin/w", n_out, n_in)
    x = synth.normal_f32(7, "pin/x", (rows, n_in))
    y = oracle.gemv_q8(blocks, x)
    want = x.numpy().astype(np.float64) @ _numpy_dequant(blocks).T
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)
    # the oracle's own dequantiser agrees with the numpy one, and its matmul with numpy's
    np.testing.assert_array_equal(oracle.q8_dequant(blocks), _numpy_dequant(blocks))
    np.testing.assert_allclose(oracle.matmul(_numpy_dequant(blocks), x), want, rtol=1e-12, atol=1e-12)


def _blocks_from(q, d):
    """Q8_0 bytes from integer values q [n_out][n_in] and f16 scales d [n_out][n_in/32]."""
    n_out, n_in = q.shape
    nb = n_in // 32
    out = np.zeros((n_out, nb, 34), np.uint8)
    dh = np.asarray(d, np.float16).reshape(n_out, nb).view(np.uint16)
    out[:, :, 0] = dh & 0xFF
    out[:, :, 1] = dh >> 8
    out[:, :, 2:] = np.asarray(q, np.int8).reshape(n_out, nb, 32).view(np.uint8)
    return out


def test_gemv_all_ones_is_block_sums():
    """q = 1 and d = 1 everywhere: every output is the plain sum of x."""
    x = synth.normal_f32(3, "pin/ones", (2, 96))
    blocks = _blocks_from(np.ones((4, 96)), np.ones((4, 3)))
    y = oracle.gemv_q8(blocks, x)
    for r in range(2):
        assert np.allclose(y[r], math.fsum(float(v) for v in x[r]), rtol=0, atol=1e-12)


def test_gemv_one_hot_column():
    """A single nonzero weight q at input k of output o gives y[o] = d*q*x[k] exactly."""
    x = synth.normal_f32(3, "pin/onehot", (3, 64))
    q = np.zeros((6, 64))
    d = np.full((6, 2), 0.25)
    q[4, 45] = -113
    blocks = _blocks_from(q, d)
    y = oracle.gemv_q8(blocks, x)
    for r in range(3):
        assert y[r, 4] == 0.25 * -113 * float(x[r, 45])
        assert np.all(y[r, [0, 1, 2, 3, 5]] == 0.0)


def test_gemv_rows_independent():
    """Rows stepped together equal each row stepped alone (the column tiling's contract)."""
    blocks = synth.q8_0_blocks_from_normal(5, "pin/rows", 48, 128)
    x = synth.normal_f32(5, "pin/rows/x", (9, 128))
    y = oracle.gemv_q8(blocks, x)
    for r in range(9):
        np.testing.assert_array_equal(y[r], oracle.gemv_q8(blocks, x[r:r + 1])[0])


@pytest.mark.parametrize("n_out,n_in,rows", [(5, 32, 1), (37, 224, 3), (64, 512, 8)])
def test_gemv_f16w_matches_numpy_half_matmul(n_out, n_in, rows):
    """The f16-weight GEMV equals numpy's float16 -> float64 widening followed by a dense product."""
    w = synth.f16_weights_from_normal(7, "pin/w16", n_out, n_in)
    x = synth.normal_f32(7, "pin/x16", (rows, n_in))
    y = oracle.gemv_f16w(w, x)
    want = x.numpy().astype(np.float64) @ w.numpy().astype(np.float64).T
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-13)
    # the weight bits and the float16 values give the same result
    np.testing.assert_array_equal(oracle.gemv_f16w(w.numpy().view(np.uint16), x), y)


def test_gemv_f16w_extremes_exact():
    """Single weights at the ends of the f16 range give exact products: the largest normal
    65504, the smallest subnormal 2^-24, a negative normal and -0; all others zero."""
    x = synth.normal_f32(3, "pin/w16x", (2, 64))
    w = np.zeros((5, 64), np.uint16)
    w[0, 3] = 0x7BFF          # 65504
    w[1, 63] = 0x0001         # 2^-24
    w[2, 10] = 0xC500         # -5.0
    w[3, 20] = 0x8000         # -0.0
    y = oracle.gemv_f16w(w, x)
    for r in range(2):
        assert y[r, 0] == 65504.0 * float(x[r, 3])
        assert y[r, 1] == 2.0 ** -24 * float(x[r, 63])
        assert y[r, 2] == -5.0 * float(x[r, 10])
        assert y[r, 3] == 0.0 and y[r, 4] == 0.0


def test_gemv_f16w_ones_is_row_sum():
    """w = 1 everywhere: every output is the plain sum of its activation row."""
    x = synth.normal_f32(4, "pin/w16ones", (3, 96))
    w = np.full((4, 96), 0x3C00, np.uint16)
    y = oracle.gemv_f16w(w, x)
    for r in range(3):
        assert np.allclose(y[r], math.fsum(float(v) for v in x[r]), rtol=0, atol=1e-12)


def test_quantizer_bytes():
    """Q8_0 input encoding: scale max|w|/127 as f16, values rounded half away from zero."""
    w = torch.zeros(1, 32)
    w[0, 0] = 1.27
    w[0, 1] = -0.635          # exactly -63.5 units -> -64 (half away from zero)
    w[0, 2] = 0.005           # 0.5 units -> 1
    b = synth.quantize_q8_0(w).numpy()
    d = b[0, 0, 0:2].copy().view(np.float16)[0]
    q = b[0, 0, 2:].view(np.int8)
    assert d == np.float16(np.float32(1.27) / np.float32(127.0))
    assert q[0] == 127 and q[1] == -64 and q[2] == 1 and np.all(q[3:] == 0)


# ---------------------------------------------------------------------- RoPE

def test_rope_complex_multiplication():
    """NeoX rotation of (x_j, x_{j+rot/2}) equals multiplying x_j + i x_{j+rot/2} by e^{i a_j}."""
    rng = np.random.default_rng(2)
    D, rot, theta = 64, 64, 500000.0
    for pos in (0, 1, 7, 127, 4096, 32767):
        x = rng.standard_normal(D)
        y = oracle.rope_vec(x, rot, True, theta, pos)
        j = np.arange(rot // 2)
        a = pos * theta ** (-2.0 * j / rot)
        z = (x[:rot // 2] + 1j * x[rot // 2:rot]) * np.exp(1j * a)
        np.testing.assert_allclose(y[:rot // 2], z.real, rtol=0, atol=1e-12)
        np.testing.assert_allclose(y[rot // 2:rot], z.imag, rtol=0, atol=1e-12)


def test_rope_known_angles():
    """Pair 0 turns by exactly `pos` radians; at theta 10000, rot 4, pair 1 turns by pos/100."""
    y = oracle.rope_vec([1.0, 0.0], 2, True, 500000.0, 1.0)
    assert abs(y[0] - math.cos(1.0)) < 1e-15 and abs(y[1] - math.sin(1.0)) < 1e-15
    y = oracle.rope_vec([0.0, 1.0, 0.0, 0.0], 4, True, 10000.0, 100.0)
    # x = e_1 is pair 1's first channel; pair 1 couples channels 1 and 3, angle 100 * 10000^-0.5 = 1
    assert abs(y[1] - math.cos(1.0)) < 1e-14 and abs(y[3] - math.sin(1.0)) < 1e-14
    assert y[0] == 0.0 and y[2] == 0.0
    # interleaved pairing couples (0,1) and (2,3) instead
    y = oracle.rope_vec([0.0, 0.0, 1.0, 0.0], 4, False, 10000.0, 100.0)
    assert abs(y[2] - math.cos(1.0)) < 1e-14 and abs(y[3] - math.sin(1.0)) < 1e-14


def test_rope_invariants():
    rng = np.random.default_rng(3)
    D, theta = 128, 500000.0
    for rot in (128, 64, 32):
        x = rng.standard_normal(D)
        for neox in (True, False):
            # position 0 is the identity
            assert np.array_equal(oracle.rope_vec(x, rot, neox, theta, 0.0), x)
            y = oracle.rope_vec(x, rot, neox, theta, 5000.0)
            # channels past the rotated width pass through bit for bit
            assert np.array_equal(y[rot:], x[rot:])
            # each pair keeps its length
            if neox:
                n0 = x[:rot // 2] ** 2 + x[rot // 2:rot] ** 2
                n1 = y[:rot // 2] ** 2 + y[rot // 2:rot] ** 2
            else:
                n0 = x[0:rot:2] ** 2 + x[1:rot:2] ** 2
                n1 = y[0:rot:2] ** 2 + y[1:rot:2] ** 2
            np.testing.assert_allclose(n1, n0, rtol=1e-12)
            # rope(p1) after rope(p2) is rope(p1 + p2)
            a = oracle.rope_vec(oracle.rope_vec(x, rot, neox, theta, 1234.0), rot, neox, theta, 777.0)
            b = oracle.rope_vec(x, rot, neox, theta, 2011.0)
            np.testing.assert_allclose(a, b, rtol=0, atol=1e-9)


def _cache(n_reg, n_kv, cap, D, fill=0x7E00):
    return np.full((n_reg, n_kv, cap, D), fill, np.uint16)


def test_rope_store_writes_only_its_slots():
    """Poisoned cache: exactly rows*n_kv*D halves change in each plane, at [reg][h][pos][:]."""
    n_q, n_kv, D, cap = 4, 2, 64, 32
    rows = 3
    q = synth.normal_f32(0, "pin/q", (rows, n_q * D))
    k = synth.normal_f32(0, "pin/k", (rows, n_kv * D))
    v = synth.normal_f32(0, "pin/v", (rows, n_kv * D))
    pos = np.array([5, 31, 0], np.int32)
    reg = np.array([1, 0, 1], np.int32)
    kc, vc = _cache(2, n_kv, cap, D), _cache(2, n_kv, cap, D)
    oracle.rope_kv_store(q, k, v, pos, kc, vc, n_q=n_q, n_kv=n_kv, head_dim=D, rot_dim=D,
                         theta=500000.0, row_region=reg)
    changed = np.argwhere(kc != 0x7E00)
    assert len(changed) == rows * n_kv * D
    assert len(np.argwhere(vc != 0x7E00)) == rows * n_kv * D
    want = {(int(reg[r]), h, int(pos[r])) for r in range(rows) for h in range(n_kv)}
    assert {tuple(int(c) for c in idx[:3]) for idx in changed} == want
    # V is stored as the f16 rounding of v (library conversion), K at position 0 likewise
    vv = v.numpy().reshape(rows, n_kv, D)
    for r in range(rows):
        for h in range(n_kv):
            np.testing.assert_array_equal(vc[reg[r], h, pos[r]], vv[r, h].astype(np.float16).view(np.uint16))
    kk = k.numpy().reshape(rows, n_kv, D)
    np.testing.assert_array_equal(kc[1, :, 0], kk[2].astype(np.float16).view(np.uint16))


def test_rope_store_clamp_and_bias():
    """Values past the half range clamp to +-65504 (0x7BFF); bias rows are added before rotating."""
    n_q, n_kv, D = 2, 1, 64
    q = np.zeros((1, n_q * D), np.float32)
    k = np.zeros((1, n_kv * D), np.float32)
    v = np.zeros((1, n_kv * D), np.float32)
    k[0, 3] = 1e5
    v[0, 4] = -1e5
    kc, vc = _cache(1, n_kv, 4, D), _cache(1, n_kv, 4, D)
    oracle.rope_kv_store(q, k, v, np.array([0], np.int32), kc, vc, n_q=n_q, n_kv=n_kv,
                         head_dim=D, rot_dim=D, theta=500000.0)
    assert kc[0, 0, 0, 3] == 0x7BFF and vc[0, 0, 0, 4] == 0xFBFF
    bias = synth.normal_f32(4, "pin/bias", ((n_q + 2 * n_kv) * D,))
    qq = synth.normal_f32(4, "pin/bq", (1, n_q * D))
    kc2, vc2 = _cache(1, n_kv, 8, D), _cache(1, n_kv, 8, D)
    qo = oracle.rope_kv_store(qq, k * 0, v * 0, np.array([6], np.int32), kc2, vc2, n_q=n_q,
                              n_kv=n_kv, head_dim=D, rot_dim=D, theta=500000.0, bias=bias)
    b = bias.numpy().astype(np.float64)
    want_q0 = oracle.rope_vec(qq.numpy()[0, :D].astype(np.float64) + b[:D], D, True, 500000.0, 6.0)
    np.testing.assert_array_equal(qo[0, :D], want_q0)
    np.testing.assert_array_equal(vc2[0, 0, 6], b[(n_q + n_kv) * D:].astype(np.float16).view(np.uint16))


# ----------------------------------------------------------------- attention

def _attn_inputs(seed, rows, n_q, n_kv, D, cap, seqlen):
    kc = synth.kv_cache_normal(seed, "pin/K", 1, n_kv, cap, D).numpy().view(np.uint16)
    vc = synth.kv_cache_normal(seed, "pin/V", 1, n_kv, cap, D).numpy().view(np.uint16)
    q = synth.normal_f32(seed, "pin/aq", (rows, n_q * D)).numpy().astype(np.float64)
    return q, kc.copy(), vc.copy(), np.array(seqlen, np.int32)


def _numpy_attention(q, kc, vc, seqlen, n_q, n_kv, D, kv_of=None):
    """Softmax attention with scipy's logsumexp (independent of the oracle's C)."""
    from scipy.special import logsumexp
    G = n_q // n_kv
    kv_of = kv_of or (lambda h: h // G)
    K = kc.view(np.float16).astype(np.float64)
    V = vc.view(np.float16).astype(np.float64)
    rows = q.shape[0]
    out = np.zeros((rows, n_q * D))
    lse = np.zeros((rows, n_q))
    for r in range(rows):
        for h in range(n_q):
            s = K[0, kv_of(h), :seqlen[r]] @ q[r, h * D:(h + 1) * D] / math.sqrt(D)
            lse[r, h] = logsumexp(s)
            out[r, h * D:(h + 1) * D] = np.exp(s - lse[r, h]) @ V[0, kv_of(h), :seqlen[r]]
    return out, lse


def test_attention_full_matches_scipy():
    n_q, n_kv, D = 6, 2, 64
    q, kc, vc, sl = _attn_inputs(1, 3, n_q, n_kv, D, 200, [200, 57, 1])
    out, lse = oracle.attn_full(q, kc, vc, sl, n_q=n_q, n_kv=n_kv, head_dim=D)
    wo, wl = _numpy_attention(q, kc, vc, sl, n_q, n_kv, D)
    np.testing.assert_allclose(out, wo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, wl, rtol=1e-13)


@pytest.mark.parametrize("chunk", [1, 7, 64, 100, 200])
def test_split_merge_equals_full(chunk):
    """Any split of the keys, merged by log-sum-exp, equals one softmax over all keys."""
    n_q, n_kv, D = 4, 2, 64
    q, kc, vc, sl = _attn_inputs(2, 4, n_q, n_kv, D, 200, [200, 128, 3, 129])
    n_splits = (200 + chunk - 1) // chunk
    out, lse = oracle.attention(q, kc, vc, sl, n_q=n_q, n_kv=n_kv, head_dim=D, chunk=chunk,
                                n_splits=n_splits)
    fo, fl = oracle.attn_full(q, kc, vc, sl, n_q=n_q, n_kv=n_kv, head_dim=D)
    np.testing.assert_allclose(out, fo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, fl, rtol=1e-12)


def test_attention_closed_forms():
    n_q, n_kv, D = 2, 1, 64
    q, kc, vc, _ = _attn_inputs(3, 1, n_q, n_kv, D, 50, [50])
    V = vc.view(np.float16).astype(np.float64)
    K = kc.view(np.float16).astype(np.float64)
    # one key: out = v_0 and LSE = s_0
    out, lse = oracle.attention(q, kc, vc, np.array([1], np.int32), n_q=n_q, n_kv=n_kv, head_dim=D,
                                chunk=16, n_splits=4)
    np.testing.assert_allclose(out[0, :D], V[0, 0, 0], rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - float(K[0, 0, 0] @ q[0, :D]) / 8.0) < 1e-12
    # all keys equal: out = mean of v, LSE = s + ln n
    kc2 = kc.copy()
    kc2[0, 0, :] = kc[0, 0, 0]
    out, lse = oracle.attention(q, kc2, vc, np.array([50], np.int32), n_q=n_q, n_kv=n_kv,
                                head_dim=D, chunk=16, n_splits=4)
    np.testing.assert_allclose(out[0, :D], V[0, 0, :50].mean(axis=0), rtol=0, atol=1e-12)
    s = float(K[0, 0, 0] @ q[0, :D]) / 8.0
    assert abs(lse[0, 0] - (s + math.log(50))) < 1e-12
    # a peaked query picks out its key's value
    j = 17
    kj = K[0, 0, j]
    qp = np.zeros((1, n_q * D))
    qp[0, :D] = 30.0 * kj / np.linalg.norm(kj) * math.sqrt(D)
    out, _ = oracle.attention(qp, kc, vc, np.array([50], np.int32), n_q=n_q, n_kv=n_kv, head_dim=D,
                              chunk=16, n_splits=4)
    np.testing.assert_allclose(out[0, :D], V[0, 0, j], rtol=0, atol=1e-6)


def test_gqa_head_map_and_regions():
    """Query head h reads KV head h // (n_q/n_kv) of its row's region."""
    n_q, n_kv, D, cap = 6, 3, 64, 40
    kc = synth.kv_cache_normal(4, "pin/rK", 2, n_kv, cap, D).numpy().view(np.uint16).copy()
    vc = synth.kv_cache_normal(4, "pin/rV", 2, n_kv, cap, D).numpy().view(np.uint16).copy()
    q = synth.normal_f32(4, "pin/rq", (2, n_q * D)).numpy().astype(np.float64)
    sl = np.array([40, 33], np.int32)
    out, lse = oracle.attention(q, kc, vc, sl, n_q=n_q, n_kv=n_kv, head_dim=D, chunk=8, n_splits=5,
                                row_region=np.array([1, 0], np.int32))
    for r, reg in ((0, 1), (1, 0)):
        wo, wl = _numpy_attention(q[r:r + 1], kc[reg:reg + 1], vc[reg:reg + 1], sl[r:r + 1], n_q, n_kv, D)
        np.testing.assert_allclose(out[r], wo[0], atol=1e-12)
        np.testing.assert_allclose(lse[r], wl[0], rtol=1e-12)


def test_empty_split_weighs_nothing():
    n_q, n_kv, D = 2, 1, 64
    q, kc, vc, _ = _attn_inputs(5, 1, n_q, n_kv, D, 64, [64])
    po, pl = oracle.attn_split(q, kc, vc, np.array([10], np.int32), n_q=n_q, n_kv=n_kv, head_dim=D,
                               chunk=8, n_splits=8)
    assert np.all(np.isneginf(pl[0, :, 2:])) and np.all(po[0, :, 2:] == 0)
    assert np.all(np.isfinite(pl[0, :, :2]))


# ------------------------------------------------------------------ grouping

def test_f32_mirror_store():
    """The f32 mirror: k rotated as a complex product and rounded once to f32, v (plus bias) rounded
    once to f32, no clamp to the half range; the slot layout is the f16 mirror's."""
    n_q, n_kv, D, cap = 2, 2, 64, 16
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, n_q * D)).astype(np.float32)
    k = rng.standard_normal((1, n_kv * D)).astype(np.float32)
    v = rng.standard_normal((1, n_kv * D)).astype(np.float32)
    k[0, 3] = 1.0e5                    # past the half range: kept in the f32 mirror
    b = rng.standard_normal((n_q + 2 * n_kv) * D).astype(np.float32)
    kc = np.zeros((1, n_kv, cap, D), np.float32)
    vc = np.zeros((1, n_kv, cap, D), np.float32)
    pos = 11
    oracle.rope_kv_store(q, k, v, np.array([pos], np.int32), kc, vc, n_q=n_q, n_kv=n_kv, head_dim=D, rot_dim=D,
                         theta=500000.0, neox=True, bias=b)
    j = np.arange(D // 2)
    ang = pos * 500000.0 ** (-2.0 * j / D)
    for h in range(n_kv):
        kb = k[0, h * D:(h + 1) * D].astype(np.float64) + b[(n_q + h) * D:(n_q + h + 1) * D]
        z = (kb[:D // 2] + 1j * kb[D // 2:]) * np.exp(1j * ang)
        want = np.concatenate([z.real, z.imag]).astype(np.float32)
        got = kc[0, h, pos]
        assert np.max(np.abs(got.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))) <= 1
        vb = (v[0, h * D:(h + 1) * D].astype(np.float64) + b[(n_q + n_kv + h) * D:(n_q + n_kv + h + 1) * D])
        np.testing.assert_array_equal(vc[0, h, pos], vb.astype(np.float32))
    # the pair holding 1e5 keeps its norm: one of its two channels is past 65504 (nothing clamped)
    assert max(abs(float(kc[0, 0, pos, 3])), abs(float(kc[0, 0, pos, 3 + D // 2]))) > 65504.0
    assert np.count_nonzero(kc) == n_kv * D and np.count_nonzero(vc) == n_kv * D


def test_f32_mirror_attention():
    """Attention over f32 planes equals scipy's softmax over the same values, and f16-valued
    f32 planes give exactly the f16 mirror's result."""
    n_q, n_kv, D = 6, 2, 64
    q, kc16, vc16, sl = _attn_inputs(3, 3, n_q, n_kv, D, 200, [200, 57, 1])
    rng = np.random.default_rng(7)
    kc32 = rng.standard_normal(kc16.shape).astype(np.float32)
    vc32 = rng.standard_normal(vc16.shape).astype(np.float32)
    out, lse = oracle.attn_full(q, kc32, vc32, sl, n_q=n_q, n_kv=n_kv, head_dim=D)
    from scipy.special import logsumexp
    K, V = kc32.astype(np.float64), vc32.astype(np.float64)
    for r in range(3):
        for h in range(n_q):
            s_ = K[0, h // 3, :sl[r]] @ q[r, h * D:(h + 1) * D] / math.sqrt(D)
            assert abs(lse[r, h] - logsumexp(s_)) < 1e-12
            np.testing.assert_allclose(out[r, h * D:(h + 1) * D], np.exp(s_ - logsumexp(s_)) @ V[0, h // 3, :sl[r]],
                                       rtol=0, atol=1e-12)
    po, pl = oracle.attn_split(q, kc32, vc32, sl, n_q=n_q, n_kv=n_kv, head_dim=D, chunk=32, n_splits=7)
    mo, ml = oracle.attn_merge(po, pl)
    np.testing.assert_allclose(mo, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, lse, rtol=0, atol=1e-12)
    # the f16 values widened into an f32 mirror: identical to the f16 mirror's result
    k_w = kc16.view(np.float16).astype(np.float32)
    v_w = vc16.view(np.float16).astype(np.float32)
    o16, l16 = oracle.attn_full(q, kc16, vc16, sl, n_q=n_q, n_kv=n_kv, head_dim=D)
    o32, l32 = oracle.attn_full(q, k_w, v_w, sl, n_q=n_q, n_kv=n_kv, head_dim=D)
    np.testing.assert_array_equal(o16, o32)
    np.testing.assert_array_equal(l16, l32)


def _numpy_q8_encode(x):
    """Q8_0 encoding in numpy float32 (independent of the oracle's C)."""
    x = np.asarray(x, np.float32)
    amax = np.float32(np.max(np.abs(x)))
    d32 = np.float32(amax / np.float32(127.0))
    if d32 == 0:
        return np.zeros(32, np.int8), 0
    t = (x / d32).astype(np.float32)
    r = np.floor(np.abs(t) + np.float32(0.5)).astype(np.float32)
    q = np.clip(np.where(t < 0, -r, r), -127, 127).astype(np.int8)
    return q, int(np.array([d32], np.float32).astype(np.float16).view(np.uint16)[0])


def test_q8_encode_block():
    """The q8_0 mirror's block encoding: numpy float32 agrees; ties round away from zero; an
    all-zero block has scale 0 and codes 0; the largest magnitude takes code +-127."""
    rng = np.random.default_rng(11)
    for scale in (1e-3, 1.0, 3e4):
        x = (rng.standard_normal(32) * scale).astype(np.float32)
        q, d = oracle.q8_encode_block(x)
        wq, wd = _numpy_q8_encode(x)
        np.testing.assert_array_equal(q, wq)
        assert d == wd
        assert np.max(np.abs(q.astype(int))) == 127
    ties = np.zeros(32, np.float32)
    ties[:6] = [127.0, 2.5, -2.5, 0.5, -0.5, -126.5]      # d = 127 / 127 = 1: t = x exactly
    q, d = oracle.q8_encode_block(ties)
    assert list(q[:6]) == [127, 3, -3, 1, -1, -127] and d == 0x3C00
    q, d = oracle.q8_encode_block(np.zeros(32, np.float32))
    assert d == 0 and not q.any()


def test_q8_mirror_store_and_attention():
    """The q8_0 mirror: the stored codes and scales are numpy's rotation rounded to f32 and encoded
    per block; attention over the planes equals scipy's softmax over the decoded values."""
    n_q, n_kv, D, cap = 4, 2, 64, 40
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, n_q * D)).astype(np.float32)
    k = rng.standard_normal((1, n_kv * D)).astype(np.float32)
    v = rng.standard_normal((1, n_kv * D)).astype(np.float32)
    kp = oracle.Q8Plane(rng.integers(-127, 128, (1, n_kv, cap, D)).astype(np.int8),
                        np.full((1, n_kv, cap, D // 32), 0x2C00, np.uint16))          # scale 1/16
    vp = oracle.Q8Plane(rng.integers(-127, 128, (1, n_kv, cap, D)).astype(np.int8),
                        np.full((1, n_kv, cap, D // 32), 0x2C00, np.uint16))
    pos = 33
    qo = oracle.rope_kv_store(q, k, v, np.array([pos], np.int32), kp, vp, n_q=n_q, n_kv=n_kv, head_dim=D,
                              rot_dim=D, theta=500000.0, neox=True)
    ang = pos * 500000.0 ** (-2.0 * np.arange(D // 2) / D)
    for h in range(n_kv):
        kh = k[0, h * D:(h + 1) * D].astype(np.float64)
        z = (kh[:D // 2] + 1j * kh[D // 2:]) * np.exp(1j * ang)
        kr = np.concatenate([z.real, z.imag]).astype(np.float32)
        for b in range(D // 32):
            wq, wd = _numpy_q8_encode(kr[32 * b:32 * (b + 1)])
            np.testing.assert_array_equal(kp.codes[0, h, pos, 32 * b:32 * (b + 1)], wq)
            assert kp.scales[0, h, pos, b] == wd
            wq, wd = _numpy_q8_encode(v[0, h * D + 32 * b:h * D + 32 * (b + 1)])
            np.testing.assert_array_equal(vp.codes[0, h, pos, 32 * b:32 * (b + 1)], wq)
            assert vp.scales[0, h, pos, b] == wd
    from scipy.special import logsumexp
    sl = np.array([pos + 1], np.int32)
    out, lse = oracle.attn_full(qo, kp, vp, sl, n_q=n_q, n_kv=n_kv, head_dim=D)
    K, V = kp.values(), vp.values()
    for h in range(n_q):
        s_ = K[0, h // 2, :pos + 1] @ qo[0, h * D:(h + 1) * D] / math.sqrt(D)
        assert abs(lse[0, h] - logsumexp(s_)) < 1e-12
        np.testing.assert_allclose(out[0, h * D:(h + 1) * D], np.exp(s_ - logsumexp(s_)) @ V[0, h // 2, :pos + 1],
                                   rtol=0, atol=1e-12)
    po, pl = oracle.attn_split(qo, kp, vp, sl, n_q=n_q, n_kv=n_kv, head_dim=D, chunk=32, n_splits=2)
    mo, ml = oracle.attn_merge(po, pl)
    np.testing.assert_allclose(mo, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, lse, rtol=0, atol=1e-12)


def test_grouping_golden():
    """The pages' twelve streams run as two commands of six (tests/golden/grouping.txt)."""
    for n, sizes in _read_golden("grouping.txt"):
        assert oracle.plan_groups(int(n)) == [int(s) for s in sizes.split(",")]


def test_grouping_brute_force():
    for n in range(1, 65):
        g = oracle.plan_groups(n)
        assert sum(g) == n and max(g) <= 8 and max(g) - min(g) <= 1
        assert len(g) == -(-n // 8)
        assert g == sorted(g, reverse=True)


# ------------------------------------------------------------------ controls

def test_controls_catch_planted_mistakes():
    """Each comparison used above rejects a result with a planted mistake."""
    n_q, n_kv, D = 4, 2, 64
    q, kc, vc, sl = _attn_inputs(6, 2, n_q, n_kv, D, 64, [64, 20])
    out, lse = oracle.attn_full(q, kc, vc, sl, n_q=n_q, n_kv=n_kv, head_dim=D)
    wo, wl = _numpy_attention(q, kc, vc, sl, n_q, n_kv, D)
    np.testing.assert_allclose(out, wo, atol=1e-12)
    # an interleaved GQA map (h % n_kv instead of h // G) is caught
    bo, _ = _numpy_attention(q, kc, vc, sl, n_q, n_kv, D, kv_of=lambda h: h % n_kv)
    assert not np.allclose(out, bo, atol=1e-6)
    # a dropped scale (no 1/sqrt(D)) is caught
    assert not np.allclose(lse, wl * math.sqrt(D), rtol=1e-4)
    # a transposed weight operand is caught by the GEMV pin
    blocks = synth.q8_0_blocks_from_normal(8, "ctl/w", 64, 64)
    x = synth.normal_f32(8, "ctl/x", (1, 64))
    y = oracle.gemv_q8(blocks, x)
    assert not np.allclose(y, x.numpy().astype(np.float64) @ _numpy_dequant(blocks), rtol=1e-3)
    # the f16-weight pin catches a transposed operand and weights read as bf16 instead of f16
    w16 = synth.f16_weights_from_normal(8, "ctl/w16", 64, 64)
    y16 = oracle.gemv_f16w(w16, x)
    assert not np.allclose(y16, x.numpy().astype(np.float64) @ w16.numpy().astype(np.float64), rtol=1e-3)
    as_bf16 = (w16.numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert not np.allclose(y16, x.numpy().astype(np.float64) @ as_bf16.T, rtol=1e-3)
    # a sign flip in the rotation is caught by the complex-multiplication pin
    xr = np.random.default_rng(0).standard_normal(64)
    yr = oracle.rope_vec(xr, 64, True, 500000.0, 3.0)
    z = (xr[:32] + 1j * xr[32:]) * np.exp(-1j * 3.0 * 500000.0 ** (-2.0 * np.arange(32) / 64))
    assert not np.allclose(yr[:32], z.real, atol=1e-6)
