"""The q8_0 (block-codec) KV mirror: dl_rope_kv_store's encoding and the CUDA-core attention
over int8 codes and f16 scales against the oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import assert_attn_close

pytestmark = pytest.mark.gpu

POISON_CODE = -128          # never produced (codes are clamped to +-127)
POISON_SCALE = 0x7E00       # a NaN pattern


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _planes(label, n_reg, n_kv, cap, D):
    kc, ks = synth.kv_q8_random_planes(0, label + "/K", n_reg, n_kv, cap, D)
    vc, vs = synth.kv_q8_random_planes(0, label + "/V", n_reg, n_kv, cap, D)
    return kc, ks, vc, vs


def _cache(dl, kc, ks, vc, vs):
    return dl.KVCache.q8(kc.cuda(), ks.cuda(), vc.cuda(), vs.cuda())


def _oracle_planes(kc, ks, vc, vs):
    return (oracle.Q8Plane(kc.numpy().copy(), ks.numpy().view(np.uint16).copy()),
            oracle.Q8Plane(vc.numpy().copy(), vs.numpy().view(np.uint16).copy()))


@pytest.mark.parametrize("D,neox,rot,bias", [(128, True, 128, False), (64, False, 32, True)])
def test_q8_store(dl, D, neox, rot, bias):
    """Exactly the computed slots are written; v codes and scales are bit-exact (one correctly
    rounded add, the same f32 encoding); k's scales are within one f16 step and its codes within
    one of the oracle's (the rotation is f32 on the GPU, double rounded to f32 in the oracle)."""
    rows, n_q, n_kv, cap = 3, 8, 2, 300
    pos = np.array([5, 299, 100], np.int32)
    regions = np.array([0, 1, 0], np.int32)
    q = synth.normal_f32(1, "q8s/q", (rows, n_q * D))
    k = synth.normal_f32(1, "q8s/k", (rows, n_kv * D))
    v = synth.normal_f32(1, "q8s/v", (rows, n_kv * D))
    b = synth.normal_f32(1, "q8s/b", ((n_q + 2 * n_kv) * D,)) if bias else None
    shape, sshape = (2, n_kv, cap, D), (2, n_kv, cap, D // 32)
    ko = oracle.Q8Plane(np.full(shape, POISON_CODE, np.int8), np.full(sshape, POISON_SCALE, np.uint16))
    vo = oracle.Q8Plane(np.full(shape, POISON_CODE, np.int8), np.full(sshape, POISON_SCALE, np.uint16))
    oracle.rope_kv_store(q, k, v, pos, ko, vo, n_q=n_q, n_kv=n_kv, head_dim=D, rot_dim=rot, theta=500000.0,
                         neox=neox, bias=b, row_region=regions)
    kv = dl.KVCache.q8(torch.full(shape, POISON_CODE, dtype=torch.int8).cuda(),
                       torch.from_numpy(np.full(sshape, POISON_SCALE, np.uint16).view(np.float16)).cuda(),
                       torch.full(shape, POISON_CODE, dtype=torch.int8).cuda(),
                       torch.from_numpy(np.full(sshape, POISON_SCALE, np.uint16).view(np.float16)).cuda())
    rope = dl.make_rope(500000.0, rot, cap, neox=neox)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dl_rope_kv_store(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(pos).cuda(), rope, kv, n_q,
                        bias=None if b is None else b.cuda(), row_region=torch.from_numpy(regions).cuda(),
                        status=status)
    torch.cuda.synchronize()
    assert dl.dl_status_read(status) == 0
    kcg, ksg = kv.k.cpu().numpy(), kv.k_scale.cpu().numpy().view(np.uint16)
    vcg, vsg = kv.v.cpu().numpy(), kv.v_scale.cpu().numpy().view(np.uint16)
    assert np.array_equal(kcg == POISON_CODE, ko.codes == POISON_CODE)
    assert np.array_equal(ksg == POISON_SCALE, ko.scales == POISON_SCALE)
    assert np.array_equal(vcg, vo.codes) and np.array_equal(vsg, vo.scales)
    w = ko.scales != POISON_SCALE
    assert int(np.abs(ksg[w].astype(np.int64) - ko.scales[w].astype(np.int64)).max()) <= 1
    wc = ko.codes != POISON_CODE
    assert int(np.abs(kcg[wc].astype(np.int64) - ko.codes[wc].astype(np.int64)).max()) <= 1


@pytest.mark.parametrize("rows,n_q,n_kv,D,cap,first", [
    (1, 4, 2, 64, 128, 128),
    (1, 32, 8, 64, 4100, 4097),
    (1, 24, 8, 128, 5128, 5121),
    (2, 24, 8, 128, 5128, 5121),
    (8, 24, 8, 128, 5128, 5121),
    (8, 32, 8, 64, 4100, 4090),
])
@pytest.mark.parametrize("path", [0, 1, 2])
def test_q8_attention(dl, rows, n_q, n_kv, D, cap, first, path):
    """Both inner products (CUDA cores; tensor cores with the codes as exact f16 operands and
    the block scales on the score sums and the V operand) and the library's choice."""
    seqlen = list(range(first, first + rows))
    kc, ks, vc, vs = _planes("q8a/%d/%d" % (rows, D), 1, n_kv, cap, D)
    q = synth.normal_f32(2, "q8a/q/%d/%d" % (rows, D), (rows, n_q * D))
    plan = dl.dl_attn_plan_build(seqlen, n_q, n_kv, D)
    ws = dl.workspace_for(plan)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = dl.decode_attention(q.cuda(), _cache(dl, kc, ks, vc, vs),
                                   torch.tensor(seqlen, dtype=torch.int32, device="cuda"), plan, ws, status=status,
                                   path=path)
    torch.cuda.synchronize()
    assert dl.dl_status_read(status) == 0
    kp, vp = _oracle_planes(kc, ks, vc, vs)
    ref_out, ref_lse = oracle.attention(q.numpy().astype(np.float64), kp, vp, np.array(seqlen, np.int32), n_q=n_q,
                                        n_kv=n_kv, head_dim=D, chunk=plan.chunk, n_splits=plan.max_splits)
    assert_attn_close(out.cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse)


@pytest.mark.parametrize("path", [0, 2])
def test_q8_sessions_and_cluster(dl, path):
    """Six sessions of different lengths in their own regions, through the partials path and the
    cluster merge, on the library's choice (CUDA cores for one-row sessions) and tensor cores."""
    lens = [513, 4000, 1500, 64, 2049, 2900]
    n_q, n_kv, D, cap = 24, 8, 128, 4000
    kc, ks, vc, vs = _planes("q8a/sess", 6, n_kv, cap, D)
    q = synth.normal_f32(3, "q8a/sess/q", (6, n_q * D))
    kv = _cache(dl, kc, ks, vc, vs)
    kp, vp = _oracle_planes(kc, ks, vc, vs)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for cluster in (False, True):
        if cluster:
            plan = dl.dl_attn_plan_build_cluster(lens, n_q, n_kv, D, regions=list(range(6)))
            out = torch.empty(6, n_q * D, device="cuda")
            lse = torch.empty(6, n_q, device="cuda")
            dl.dl_decode_attn_cluster(q.cuda(), kv, sl, plan, out, lse, path=path)
        else:
            plan = dl.dl_attn_plan_build(lens, n_q, n_kv, D, regions=list(range(6)))
            out, lse = dl.decode_attention(q.cuda(), kv, sl, plan, dl.workspace_for(plan), path=path)
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle.attention(q.numpy().astype(np.float64), kp, vp, np.array(lens, np.int32), n_q=n_q,
                                            n_kv=n_kv, head_dim=D, chunk=plan.chunk, n_splits=plan.max_splits,
                                            row_region=np.arange(6, dtype=np.int32))
        assert_attn_close(out.cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse)


@pytest.mark.parametrize("form", ["partials", "cluster", "merged"])
@pytest.mark.parametrize("rows,D,neox,rot,bias", [(1, 128, True, 128, False), (8, 128, True, 128, True),
                                                  (2, 64, False, 32, False)])
def test_q8_fused_rope(dl, form, rows, D, neox, rot, bias):
    """The rope/store inside the attention launch on the q8_0 mirror: stored codes and scales,
    outputs and lse bit-identical to dl_rope_kv_store followed by the attention; outputs within
    the oracle's bars."""
    n_kv = 8
    n_q = 24 if D == 128 else 32
    if form == "merged" and rows * n_q // n_kv > 8:
        pytest.skip("the last piece merges at most 8 queries")
    cap = 5128
    pos = list(range(5120, 5120 + rows))
    seqlen = [p + 1 for p in pos]
    kc, ks, vc, vs = _planes("q8f/%d/%d" % (rows, D), 1, n_kv, cap, D)
    q = synth.normal_f32(4, "q8f/q/%d/%d" % (rows, D), (rows, n_q * D))
    k = synth.normal_f32(4, "q8f/k/%d/%d" % (rows, D), (rows, n_kv * D))
    v = synth.normal_f32(4, "q8f/v/%d/%d" % (rows, D), (rows, n_kv * D))
    b = synth.normal_f32(4, "q8f/b/%d" % D, ((n_q + 2 * n_kv) * D,)).cuda() if bias else None
    rope = dl.make_rope(500000.0, rot, cap, neox=neox)
    dpos = torch.tensor(pos, dtype=torch.int32, device="cuda")
    sl = torch.tensor(seqlen, dtype=torch.int32, device="cuda")
    plan = (dl.dl_attn_plan_build_cluster(seqlen, n_q, n_kv, D) if form == "cluster"
            else dl.dl_attn_plan_build(seqlen, n_q, n_kv, D))
    res = {}
    for mode in ("fused", "separate"):
        kv = _cache(dl, kc, ks, vc, vs)
        qd = q.clone().cuda()
        out = torch.full((rows, n_q * D), float("nan"), device="cuda")
        lse = torch.full((rows, n_q), float("nan"), device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rin = dict(k=k.cuda(), v=v.cuda(), pos=dpos, rope=rope, bias=b) if mode == "fused" else {}
        if mode == "separate":
            dl.dl_rope_kv_store(qd, k.cuda(), v.cuda(), dpos, rope, kv, n_q, bias=b, status=status)
        if form == "cluster":
            dl.dl_decode_attn_cluster(qd, kv, sl, plan, out, lse, status=status, **rin)
        elif form == "merged":
            dl.dl_decode_attn_merged(qd, kv, sl, plan, dl.workspace_for(plan), out, lse, status=status, **rin)
        else:
            ws = dl.workspace_for(plan)
            if mode == "fused":
                dl.dl_decode_attn_rope(qd, k.cuda(), v.cuda(), dpos, rope, kv, sl, plan, ws, bias=b, status=status)
            else:
                dl.dl_decode_attn(qd, kv, sl, plan, ws, status=status)
            dl.dl_attn_merge(ws, plan, sl, out, lse)
        torch.cuda.synchronize()
        assert dl.dl_status_read(status) == 0
        res[mode] = [kv.k.cpu().numpy(), kv.k_scale.cpu().numpy().view(np.uint16), kv.v.cpu().numpy(),
                     kv.v_scale.cpu().numpy().view(np.uint16), out.cpu().numpy(), lse.cpu().numpy()]
    for x, y in zip(res["fused"], res["separate"]):
        assert np.array_equal(x, y)
    kp, vp = _oracle_planes(torch.from_numpy(res["fused"][0]), torch.from_numpy(res["fused"][1].view(np.float16)),
                            torch.from_numpy(res["fused"][2]), torch.from_numpy(res["fused"][3].view(np.float16)))
    qo = q.numpy().astype(np.float64).copy()
    ko = oracle.Q8Plane(kc.numpy().copy(), ks.numpy().view(np.uint16).copy())
    vo = oracle.Q8Plane(vc.numpy().copy(), vs.numpy().view(np.uint16).copy())
    qo = oracle.rope_kv_store(q, k, v, np.array(pos, np.int32), ko, vo, n_q=n_q, n_kv=n_kv, head_dim=D, rot_dim=rot,
                              theta=500000.0, neox=neox, bias=None if b is None else b.cpu().numpy())
    # the attention is checked on the mirror as the GPU stored it (the stored k codes may differ
    # from the oracle's by one: rotation in f32 against double)
    ref_out, ref_lse = oracle.attention(np.asarray(qo, np.float64), kp, vp, np.array(seqlen, np.int32), n_q=n_q,
                                        n_kv=n_kv, head_dim=D, chunk=plan.chunk, n_splits=plan.max_splits)
    assert_attn_close(res["fused"][4], res["fused"][5], ref_out, ref_lse)


def test_q8_refusals(dl):
    """A capacity that is not a multiple of 4 is refused before anything launches."""
    kc, ks, vc, vs = _planes("q8a/refuse", 1, 2, 64, 64)
    q = torch.zeros(1, 256, device="cuda")
    sl = torch.tensor([64], dtype=torch.int32, device="cuda")
    plan = dl.dl_attn_plan_build([64], 4, 2, 64)
    ws = dl.workspace_for(plan)
    kc2, ks2, vc2, vs2 = _planes("q8a/refuse2", 1, 2, 66, 64)
    kv2 = _cache(dl, kc2, ks2, vc2, vs2)
    with pytest.raises(dl.DLError) as e:
        dl.dl_decode_attn(q, kv2, sl, plan, ws)
    assert e.value.code in (dl.DL_E_SHAPE, dl.DL_E_ALIGN)
