"""A whole decode layer step through the library against the oracle's step (GPU).

The chain feeds each call's output to the next on both sides, so the
comparison of a later call also carries the earlier calls' rounding: the
attention bars apply to the attention of the oracle's own roped q, and the O
projection is compared with the GEMV bar scaled by the attention bar's share
of its input (its input is the attention output, not a fresh draw)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import (assert_attn_close, assert_gemv_close, f16_ulp_dist, gemv_err, kv_planes,
                             layer_blocks, as_u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _step(dl, S, positions, regions, n_regions, capacity, label, fused_rope=False, cluster_merge=False,
          gemv_chain=False, l2_prefetch=False, concurrent=False, tail_merge=False):
    from row_decode_step_gb300.step import LayerStep, LayerWeights
    D, n_q, n_kv, H, F = S.head_dim, S.n_q, S.n_kv, S.hidden, S.ffn
    blocks = layer_blocks(S.name)
    if S.name == "tiny":
        blocks = dict(blocks)
    packed = {n: dl.dl_q8_pack(b.cuda(), b.shape[0], b.shape[1] * 32) for n, b in blocks.items()}
    W = LayerWeights(packed["wqkv"], packed["wo"], packed.get("wgu"), packed.get("wdown"))
    k, v = kv_planes(label, n_regions, n_kv, capacity, D)
    kv = dl.KVCache(k.cuda(), v.cuda())
    rope = dl.make_rope(S.rope_theta, D, capacity)
    n = len(positions)
    x = synth.normal_f32(0, label + "/x", (n, H))
    xf = synth.normal_f32(0, label + "/xf", (n, H)) if F else None
    h = synth.normal_f32(0, label + "/h", (n, F)) if F else None
    step = LayerStep(positions, regions, n_q, n_kv, D, H, F, "cuda", fused_rope=fused_rope,
                     cluster_merge=cluster_merge, gemv_chain=gemv_chain, l2_prefetch=l2_prefetch,
                     concurrent=concurrent, tail_merge=tail_merge)
    r0 = 0
    for c in step.commands:
        c.x.copy_(x[r0:r0 + c.n].cuda())
        if F:
            c.x_ffn.copy_(xf[r0:r0 + c.n].cuda())
            c.h.copy_(h[r0:r0 + c.n].cuda())
        r0 += c.n
    step.run(W, rope, kv)
    torch.cuda.synchronize()

    kc_o = k.numpy().view(np.uint16).copy()
    vc_o = v.numpy().view(np.uint16).copy()
    r0 = 0
    for c in step.commands:
        sl = slice(r0, r0 + c.n)
        ref = oracle.layer_step(blocks, x[sl], kc_o, vc_o, positions[sl], n_q=n_q, n_kv=n_kv, head_dim=D,
                                theta=S.rope_theta, chunk=c.plan.chunk, n_splits=c.plan.max_splits,
                                regions=regions[sl], x_ffn=None if xf is None else xf[sl],
                                h=None if h is None else h[sl])
        # q is roped in place inside qkv; its k and v parts are the GEMV's own output
        qd = n_q * D
        assert_gemv_close(c.qkv.cpu().numpy()[:, qd:], ref["qkv"][:, qd:])
        # roped q carries the GEMV's error through a rotation of channel pairs, which keeps each
        # pair's error norm: at most sqrt(2) times the GEMV bar per element
        # (the fused launch rotates its queries in shared memory and leaves q as projected)
        if not fused_rope:
            assert gemv_err(c.q.cpu().numpy(), ref["q"]) < 1e-3 * np.sqrt(2)
        assert_attn_close(c.attn.cpu().numpy(), c.lse.cpu().numpy(), ref["attn"], ref["lse"])
        # the O projection of the attention output the step actually produced, at the GEMV bar
        assert_gemv_close(c.y_o.cpu().numpy(), oracle.gemv_q8(blocks["wo"], c.attn.cpu().numpy()))
        if F:
            assert_gemv_close(c.gu.cpu().numpy(), ref["gu"])
            assert_gemv_close(c.y_down.cpu().numpy(), ref["y_down"])
        assert dl.dl_status_read(c.status) == 0
        r0 += c.n
    # the stored K/V rows carry the QKV GEMV's rounding: the unwritten slots must be identical,
    # the written ones within one f16 ulp plus the GEMV bar of their row
    kg, vg = as_u16(kv.k), as_u16(kv.v)
    k0, v0 = as_u16(k), as_u16(v)
    for got, ref, init in ((kg, kc_o, k0), (vg, vc_o, v0)):
        written = ref != init
        assert np.array_equal(got[~written], ref[~written])
        gf = got.view(np.float16).astype(np.float64)
        rf = ref.view(np.float16).astype(np.float64)
        rms = np.sqrt(np.mean(rf[written] ** 2))
        ulp = np.abs(np.spacing(rf.astype(np.float16)).astype(np.float64))
        assert np.all(np.abs(gf - rf)[written] <= ulp[written] + 1e-3 * rms)
    return step


def test_step_tiny(dl):
    _step(dl, synth.TINY, [127], [0], 1, 128, "step/tiny")


def test_step_1b(dl):
    _step(dl, synth.LLAMA_1B, [4096], [0], 1, 4097, "step/1b")


FORMS = [(False, False, False, False), (True, False, False, False), (True, True, False, False),
         (True, False, True, False), (True, False, False, True), (False, False, False, True)]


@pytest.mark.parametrize("fused,cluster,chain,prefetch", FORMS)
@pytest.mark.parametrize("rows", [1, 8])
def test_step_3b(dl, rows, fused, cluster, chain, prefetch):
    """Every form of the step (rope in the attention, cluster merge, GEMV chain, L2 prefetches)
    against the oracle's layer step."""
    _step(dl, synth.LLAMA_3B, list(range(5120, 5120 + rows)), [0] * rows, 1, 5128, "step/3b%d" % rows,
          fused_rope=fused, cluster_merge=cluster, gemv_chain=chain, l2_prefetch=prefetch)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("rows", [2, 4])
def test_step_3b_two_and_four_rows(dl, rows, fused):
    """The 2- and 4-row steps (CUDA-core and tensor-core projections) chained through the whole
    step, with the rope/store separate and inside the attention."""
    _step(dl, synth.LLAMA_3B, list(range(5120, 5120 + rows)), [0] * rows, 1, 5128, "step/3b%dc" % rows,
          fused_rope=fused)


@pytest.mark.parametrize("fused,cluster,chain,prefetch", FORMS)
def test_step_twelve_streams(dl, fused, cluster, chain, prefetch):
    lens = synth.twelve_stream_lengths(0)
    step = _step(dl, synth.LLAMA_3B, lens, list(range(12)), 12, max(lens) + 1, "step/streams", fused_rope=fused,
                 cluster_merge=cluster, gemv_chain=chain, l2_prefetch=prefetch)
    assert step.group_sizes == [6, 6]


def test_step_twelve_streams_concurrent(dl):
    """The two 6-row commands on streams of their own (forked and joined around them)."""
    lens = synth.twelve_stream_lengths(0)
    step = _step(dl, synth.LLAMA_3B, lens, list(range(12)), 12, max(lens) + 1, "step/streams", fused_rope=True,
                 concurrent=True)
    assert step.concurrent and step.group_sizes == [6, 6]


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("rows", [1, 2])
def test_step_3b_tail_merge(dl, rows, fused):
    """The attention's last piece merges (one launch fewer) at 3 and 6 queries per KV head."""
    step = _step(dl, synth.LLAMA_3B, list(range(5120, 5120 + rows)), [0] * rows, 1, 5128, "step/3b%d" % rows,
                 fused_rope=fused, tail_merge=True)
    assert step.commands[0].tail_merge


def test_step_twelve_streams_tail_merge(dl):
    lens = synth.twelve_stream_lengths(0)
    step = _step(dl, synth.LLAMA_3B, lens, list(range(12)), 12, max(lens) + 1, "step/streams", fused_rope=True,
                 tail_merge=True, concurrent=True)
    assert all(c.tail_merge for c in step.commands)


@pytest.mark.parametrize("mirror", ["f32", "q8_0"])
@pytest.mark.parametrize("rows", [1, 8])
def test_step_3b_mirrors(dl, mirror, rows):
    """The default step (rope/store inside the attention) over the f32 and the q8_0 mirrors
    against the oracle's layer step on the same planes.  Stored rows: f32 within the GEMV bar of
    their values; q8_0 codes within one and scales within two f16 steps (the stored values carry
    the QKV GEMV's rounding); unwritten slots identical."""
    from row_decode_step_gb300.step import LayerStep, LayerWeights
    S = synth.LLAMA_3B
    D, n_q, n_kv, H, F = S.head_dim, S.n_q, S.n_kv, S.hidden, S.ffn
    blocks = layer_blocks(S.name)
    packed = {n: dl.dl_q8_pack(b.cuda(), b.shape[0], b.shape[1] * 32) for n, b in blocks.items()}
    W = LayerWeights(packed["wqkv"], packed["wo"], packed.get("wgu"), packed.get("wdown"))
    cap = 5128
    positions = list(range(5120, 5120 + rows))
    regions = [0] * rows
    label = "stepm/%s/%d" % (mirror, rows)
    if mirror == "q8_0":
        kc, ks = synth.kv_q8_random_planes(0, label + "/K", 1, n_kv, cap, D)
        vc, vs = synth.kv_q8_random_planes(0, label + "/V", 1, n_kv, cap, D)
        kv = dl.KVCache.q8(kc.cuda(), ks.cuda(), vc.cuda(), vs.cuda())
        ko = oracle.Q8Plane(kc.numpy().copy(), ks.numpy().view(np.uint16).copy())
        vo = oracle.Q8Plane(vc.numpy().copy(), vs.numpy().view(np.uint16).copy())
    else:
        k = synth.normal_f32(0, label + "/K", (1, n_kv, cap, D))
        v = synth.normal_f32(0, label + "/V", (1, n_kv, cap, D))
        kv = dl.KVCache(k.cuda(), v.cuda())
        ko, vo = k.numpy().copy(), v.numpy().copy()
    rope = dl.make_rope(S.rope_theta, D, cap)
    x = synth.normal_f32(0, label + "/x", (rows, H))
    xf = synth.normal_f32(0, label + "/xf", (rows, H))
    h = synth.normal_f32(0, label + "/h", (rows, F))
    step = LayerStep(positions, regions, n_q, n_kv, D, H, F, "cuda", fused_rope=True)
    c = step.commands[0]
    c.x.copy_(x.cuda())
    c.x_ffn.copy_(xf.cuda())
    c.h.copy_(h.cuda())
    step.run(W, rope, kv)
    torch.cuda.synchronize()
    assert dl.dl_status_read(c.status) == 0
    ref = oracle.layer_step(blocks, x, ko, vo, positions, n_q=n_q, n_kv=n_kv, head_dim=D, theta=S.rope_theta,
                            chunk=c.plan.chunk, n_splits=c.plan.max_splits, regions=regions, x_ffn=xf, h=h)
    qd = n_q * D
    assert_gemv_close(c.qkv.cpu().numpy()[:, qd:], ref["qkv"][:, qd:])
    assert_attn_close(c.attn.cpu().numpy(), c.lse.cpu().numpy(), ref["attn"], ref["lse"])
    assert_gemv_close(c.y_o.cpu().numpy(), oracle.gemv_q8(blocks["wo"], c.attn.cpu().numpy()))
    assert_gemv_close(c.gu.cpu().numpy(), ref["gu"])
    assert_gemv_close(c.y_down.cpu().numpy(), ref["y_down"])
    slots = np.zeros((1, n_kv, cap), bool)
    slots[0, :, positions] = True
    if mirror == "q8_0":
        for got_c, got_s, o, (c0, s0) in ((kv.k, kv.k_scale, ko, (kc, ks)), (kv.v, kv.v_scale, vo, (vc, vs))):
            gc = got_c.cpu().numpy().astype(np.int64)
            gs = got_s.cpu().numpy().view(np.uint16).astype(np.int64)
            assert np.array_equal(gc[~slots], c0.numpy().astype(np.int64)[~slots])
            assert np.array_equal(gs[~slots], s0.numpy().view(np.uint16).astype(np.int64)[~slots])
            assert int(np.abs(gc[slots] - o.codes.astype(np.int64)[slots]).max()) <= 1
            assert int(np.abs(gs[slots] - o.scales.astype(np.int64)[slots]).max()) <= 2
    else:
        for got, o, init in ((kv.k, ko, k), (kv.v, vo, v)):
            g = got.cpu().numpy()
            assert np.array_equal(g[~slots], init.numpy()[~slots])
            ref_w = o[slots].astype(np.float64)
            rms = float(np.sqrt(np.mean(ref_w ** 2)))
            # the GEMV bar per element, times sqrt(2) for the rotation of a pair
            assert np.all(np.abs(g[slots] - ref_w) <= 1.5e-3 * np.maximum(np.abs(ref_w), rms))
