"""The whole layer step as one launch (dl_layer_step) against the oracle (GPU).

Each command's outputs are compared with the oracle element by element:
  * the QKV projection (q, k and v as projected) with the oracle's GEMV of the
    same input, within the GEMV bar;
  * the attention output and LSE with the oracle's attention of its own
    rotated queries over its own updated cache, within the attention bars;
  * the O, gate/up and down projections with the oracle's GEMV of the inputs
    the launch actually read (the launch's own attention output, and with
    `chain_ffn` its own O and gate/up outputs), within the GEMV bar;
  * the stored rows of the mirror within one f16 ulp plus the GEMV bar of their
    row, every other slot bit-identical.
A second call on the same inputs must give the same results within the bars
(its counters were left at zero by the first; the K-slices of a projection row
tile are added in the order they arrive, so the last bits may differ).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import assert_attn_close, assert_gemv_close, as_u16, kv_planes, layer_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _packed(dl, S):
    from row_decode_step_gb300.step import LayerWeights
    blocks = layer_blocks(S.name)
    packed = {n: dl.dl_q8_pack(b.cuda(), b.shape[0], b.shape[1] * 32) for n, b in blocks.items()}
    return blocks, LayerWeights(packed["wqkv"], packed["wo"], packed.get("wgu"), packed.get("wdown"))


def _inputs(S, label, n):
    x = synth.normal_f32(0, label + "/x", (n, S.hidden))
    xf = synth.normal_f32(0, label + "/xf", (n, S.hidden)) if S.ffn else None
    h = synth.normal_f32(0, label + "/h", (n, S.ffn)) if S.ffn else None
    return x, xf, h


def _build_step(dl, S, positions, regions, x, xf, h, **kw):
    from row_decode_step_gb300.step import LayerStep
    step = LayerStep(positions, regions, S.n_q, S.n_kv, S.head_dim, S.hidden, S.ffn, "cuda", **kw)
    r0 = 0
    for c in step.commands:
        c.x.copy_(x[r0:r0 + c.n].cuda())
        if S.ffn:
            c.x_ffn.copy_(xf[r0:r0 + c.n].cuda())
            c.h.copy_(h[r0:r0 + c.n].cuda())
        r0 += c.n
    return step


def _check(dl, S, blocks, step, positions, regions, x, k, v, kv, chain_ffn):
    D, n_q, n_kv, F = S.head_dim, S.n_q, S.n_kv, S.ffn
    kc_o = k.numpy().view(np.uint16).copy()
    vc_o = v.numpy().view(np.uint16).copy()
    r0 = 0
    for c in step.commands:
        sl = slice(r0, r0 + c.n)
        assert dl.dl_status_read(c.status) == 0
        ref = oracle.layer_step(blocks, x[sl], kc_o, vc_o, positions[sl], n_q=n_q, n_kv=n_kv, head_dim=D,
                                theta=S.rope_theta, chunk=c.plan.chunk, n_splits=c.plan.max_splits,
                                regions=regions[sl])
        assert_gemv_close(c.qkv.cpu().numpy(), ref["qkv"])
        attn = c.attn.cpu().numpy()
        assert_attn_close(attn, c.lse.cpu().numpy(), ref["attn"], ref["lse"])
        y_o = c.y_o.cpu().numpy()
        assert_gemv_close(y_o, oracle.gemv_q8(blocks["wo"], attn))
        if F:
            gu = c.gu.cpu().numpy()
            xf_used = y_o if chain_ffn else c.x_ffn.cpu().numpy()
            h_used = gu[:, :F].copy() if chain_ffn else c.h.cpu().numpy()
            assert_gemv_close(gu, oracle.gemv_q8(blocks["wgu"], xf_used))
            assert_gemv_close(c.y_down.cpu().numpy(), oracle.gemv_q8(blocks["wdown"], h_used))
        r0 += c.n
    # stored rows within one f16 ulp plus the GEMV bar of their row; everything else untouched
    for got, ref, init in ((as_u16(kv.k), kc_o, as_u16(k)), (as_u16(kv.v), vc_o, as_u16(v))):
        _cache_close(got, ref, ref != init)


def _cache_close(got, ref, written):
    """f16 cache planes (as u16): bit-identical outside `written`, within one ulp plus 1e-3 of the
    written values' rms inside (a stored row is the f16 rounding of a projected, rotated value)."""
    assert np.array_equal(got[~written], ref[~written])
    gf = got.view(np.float16).astype(np.float64)
    rf = ref.view(np.float16).astype(np.float64)
    rms = np.sqrt(np.mean(rf[written] ** 2))
    ulp = np.abs(np.spacing(rf.astype(np.float16)).astype(np.float64))
    assert np.all(np.abs(gf - rf)[written] <= ulp[written] + 1e-3 * rms)


def _case(dl, S, positions, regions, n_regions, capacity, label, chain_ffn=False, path=0, repeat=True):
    blocks, W = _packed(dl, S)
    k, v = kv_planes(label, n_regions, S.n_kv, capacity, S.head_dim)
    kv = dl.KVCache(k.cuda(), v.cuda())
    rope = dl.make_rope(S.rope_theta, S.head_dim, capacity)
    x, xf, h = _inputs(S, label, len(positions))
    step = _build_step(dl, S, positions, regions, x, xf, h, one_launch=True, chain_ffn=chain_ffn, gemv_path=path)
    assert step.launches == len(step.commands)
    step.run(W, rope, kv)
    torch.cuda.synchronize()
    _check(dl, S, blocks, step, positions, regions, x, k, v, kv, chain_ffn)
    if repeat:
        # the same call again on the same starting cache: the same bits everywhere
        first = [(c.qkv.clone(), c.attn.clone(), c.lse.clone(), c.y_o.clone(),
                  None if c.gu is None else c.gu.clone(), None if c.y_down is None else c.y_down.clone())
                 for c in step.commands]
        kv1 = (kv.k.clone(), kv.v.clone())
        kv.k.copy_(k.cuda())
        kv.v.copy_(v.cuda())
        for c in step.commands:
            for t in (c.qkv, c.attn, c.lse, c.y_o, c.gu, c.y_down):
                if t is not None:
                    t.fill_(float("nan"))
        step.run(W, rope, kv)
        torch.cuda.synchronize()
        for c, f in zip(step.commands, first):
            q1, a1, l1, o1, g1, d1 = f
            assert_gemv_close(c.qkv.cpu().numpy(), q1.cpu().numpy())
            assert_attn_close(c.attn.cpu().numpy(), c.lse.cpu().numpy(), a1.cpu().numpy(), l1.cpu().numpy())
            assert_gemv_close(c.y_o.cpu().numpy(), o1.cpu().numpy())
            if g1 is not None:
                assert_gemv_close(c.gu.cpu().numpy(), g1.cpu().numpy())
                assert_gemv_close(c.y_down.cpu().numpy(), d1.cpu().numpy())
            assert dl.dl_status_read(c.status) == 0
        for got, ref, init in ((kv.k, kv1[0], k), (kv.v, kv1[1], v)):
            _cache_close(as_u16(got), as_u16(ref), as_u16(ref) != as_u16(init))
    return step


def test_layer_step_tiny(dl):
    _case(dl, synth.TINY, [127], [0], 1, 128, "ls/tiny")


def test_layer_step_1b(dl):
    _case(dl, synth.LLAMA_1B, [4096], [0], 1, 4097, "ls/1b")


@pytest.mark.parametrize("rows", [1, 2, 4, 8])
def test_layer_step_3b(dl, rows):
    _case(dl, synth.LLAMA_3B, list(range(5120, 5120 + rows)), [0] * rows, 1, 5128, "ls/3b%d" % rows)


@pytest.mark.parametrize("rows", [1, 8])
def test_layer_step_3b_chained_ffn(dl, rows):
    """gate/up reads the O output and down the gate half of gate/up: the launch must wait for them."""
    _case(dl, synth.LLAMA_3B, list(range(5120, 5120 + rows)), [0] * rows, 1, 5128, "ls/3bc%d" % rows,
          chain_ffn=True)


@pytest.mark.parametrize("path", [1, 2])
def test_layer_step_3b_two_rows_paths(dl, path):
    """Two rows on either inner product of the projections (CUDA cores, tensor cores)."""
    _case(dl, synth.LLAMA_3B, [5120, 5121], [0, 0], 1, 5128, "ls/3b2p%d" % path, path=path)


def test_layer_step_twelve_streams(dl):
    lens = synth.twelve_stream_lengths(0)
    step = _case(dl, synth.LLAMA_3B, lens, list(range(12)), 12, max(lens) + 1, "ls/streams")
    assert step.group_sizes == [6, 6]


def test_layer_step_long_context(dl):
    _case(dl, synth.LLAMA_3B, list(range(32760, 32768)), [0] * 8, 1, 32768, "ls/32k", repeat=False)


def test_layer_step_matches_separate_launches(dl):
    """The one launch and the six-launch step give the same results within the bars."""
    S = synth.LLAMA_3B
    blocks, W = _packed(dl, S)
    pos = list(range(5120, 5128))
    k, v = kv_planes("ls/vs", 1, S.n_kv, 5128, S.head_dim)
    rope = dl.make_rope(S.rope_theta, S.head_dim, 5128)
    x, xf, h = _inputs(S, "ls/vs", 8)
    outs = []
    for one in (False, True):
        kv = dl.KVCache(k.cuda(), v.cuda())
        step = _build_step(dl, S, pos, [0] * 8, x, xf, h, one_launch=one, fused_rope=not one)
        step.run(W, rope, kv)
        torch.cuda.synchronize()
        c = step.commands[0]
        outs.append((c.qkv.cpu().numpy(), c.attn.cpu().numpy(), c.lse.cpu().numpy(), c.y_o.cpu().numpy(),
                     c.gu.cpu().numpy(), c.y_down.cpu().numpy()))
    (q0, a0, l0, o0, g0, d0), (q1, a1, l1, o1, g1, d1) = outs
    assert_gemv_close(q1, q0)
    assert_attn_close(a1, l1, a0, l0)
    assert_gemv_close(g1, g0)
    assert_gemv_close(d1, d0)


def test_layer_step_refuses_concurrent(dl):
    from row_decode_step_gb300.step import LayerStep
    S = synth.LLAMA_3B
    lens = synth.twelve_stream_lengths(0)
    with pytest.raises(ValueError):
        LayerStep(lens, list(range(12)), S.n_q, S.n_kv, S.head_dim, S.hidden, S.ffn, "cuda", one_launch=True,
                  concurrent=True)


@pytest.mark.parametrize("rows", [3, 4, 8])
def test_layer_step_3b_cuda_core_wide(dl, rows):
    """The CUDA-core projections asked for explicitly on 3 to 8 rows (the option that compares the
    two inner products on the same launch)."""
    _case(dl, synth.LLAMA_3B, list(range(5120, 5120 + rows)), [0] * rows, 1, 5128, "ls/3bcc%d" % rows, path=1)
