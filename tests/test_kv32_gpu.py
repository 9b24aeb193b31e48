"""The f32 KV mirror: dl_rope_kv_store, dl_decode_attn(+merge), dl_decode_attn_rope and
dl_decode_attn_cluster on float32 planes against the oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import assert_attn_close

pytestmark = pytest.mark.gpu

POISON = np.float32(np.nan).view(np.uint32)


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _planes(label, n_reg, n_kv, cap, D):
    k = synth.normal_f32(0, label + "/K32", (n_reg, n_kv, cap, D))
    v = synth.normal_f32(0, label + "/V32", (n_reg, n_kv, cap, D))
    return k, v


def test_kv32_rope_store(dl):
    """Stored k within the f32 rotation bar of the oracle, v bit-exact (one correctly rounded add),
    exactly the computed slots written, nothing clamped to the half range."""
    rows, n_q, n_kv, D, cap = 3, 8, 2, 128, 300
    pos = np.array([5, 299, 100], np.int32)
    regions = np.array([0, 1, 0], np.int32)
    q = synth.normal_f32(1, "kv32/q", (rows, n_q * D))
    k = synth.normal_f32(1, "kv32/k", (rows, n_kv * D)) * 3e4          # pairs past the f16 range
    v = synth.normal_f32(1, "kv32/v", (rows, n_kv * D)) * 3e4
    b = synth.normal_f32(1, "kv32/b", ((n_q + 2 * n_kv) * D,))
    shape = (2, n_kv, cap, D)
    kc_o = np.full(shape, np.nan, np.float32)
    vc_o = np.full(shape, np.nan, np.float32)
    qo = oracle.rope_kv_store(q, k, v, pos, kc_o, vc_o, n_q=n_q, n_kv=n_kv, head_dim=D, rot_dim=D,
                              theta=500000.0, neox=True, bias=b, row_region=regions)
    kv = dl.KVCache(torch.full(shape, float("nan")).cuda(), torch.full(shape, float("nan")).cuda())
    rope = dl.make_rope(500000.0, D, cap)
    qd = q.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dl_rope_kv_store(qd, k.cuda(), v.cuda(), torch.from_numpy(pos).cuda(), rope, kv, n_q, bias=b.cuda(),
                        row_region=torch.from_numpy(regions).cuda(), status=status)
    torch.cuda.synchronize()
    assert dl.dl_status_read(status) == 0
    kg, vg = kv.k.cpu().numpy(), kv.v.cpu().numpy()
    assert np.array_equal(np.isnan(kg), np.isnan(kc_o)) and np.array_equal(np.isnan(vg), np.isnan(vc_o))
    w = ~np.isnan(kc_o)
    np.testing.assert_array_equal(vg[w], vc_o[w])
    np.testing.assert_allclose(kg[w], kc_o[w], rtol=1e-6, atol=2e-6 * 3e4)
    assert np.abs(kg[w]).max() > 65504.0
    np.testing.assert_allclose(qd.cpu().numpy(), qo, rtol=1e-6, atol=2e-6)


@pytest.mark.parametrize("rows,n_q,n_kv,D,cap", [(1, 32, 8, 64, 4097), (1, 24, 8, 128, 5128), (8, 24, 8, 128, 5128),
                                                (4, 32, 8, 64, 3000)])
@pytest.mark.parametrize("path,sm_count", [(0, 0), (1, 0), (2, 0), (0, 76)])
def test_kv32_attention(dl, rows, n_q, n_kv, D, cap, path, sm_count):
    """Both inner products: CUDA cores with 4 (one row), 6 (24 queries per work item) or 8 (32)
    queries per warp; tensor cores on bf16 hi + lo terms (the library's choice above 4 queries).
    sm_count 76 is the one-wave plan for the mirror's one CTA per SM at D = 128."""
    seqlen = list(range(cap - 7, cap - 7 + rows)) if rows > 1 else [cap]
    kc, vc = _planes("kv32/attn/%d/%d" % (rows, D), 1, n_kv, cap, D)
    q = synth.normal_f32(2, "kv32/attn/q/%d/%d" % (rows, D), (rows, n_q * D))
    plan = dl.dl_attn_plan_build(seqlen, n_q, n_kv, D, sm_count=sm_count)
    ws = dl.workspace_for(plan)
    kv = dl.KVCache(kc.cuda(), vc.cuda())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = dl.decode_attention(q.cuda(), kv, torch.tensor(seqlen, dtype=torch.int32, device="cuda"), plan, ws,
                                   status=status, path=path)
    torch.cuda.synchronize()
    assert dl.dl_status_read(status) == 0
    ref_out, ref_lse = oracle.attention(q.numpy().astype(np.float64), kc.numpy(), vc.numpy(),
                                        np.array(seqlen, np.int32), n_q=n_q, n_kv=n_kv, head_dim=D,
                                        chunk=plan.chunk, n_splits=plan.max_splits)
    assert_attn_close(out.cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse)


@pytest.mark.parametrize("cluster", [False, True])
def test_kv32_fused_rope_and_cluster(dl, cluster):
    """Rope and store inside the attention launch on the f32 mirror: the stored values and the
    results equal the separate store followed by the attention, and meet the oracle's bars."""
    rows, n_q, n_kv, D, cap = 8, 24, 8, 128, 5128
    pos = list(range(5120, 5128))
    seqlen = [p + 1 for p in pos]
    kc, vc = _planes("kv32/fused", 1, n_kv, cap, D)
    q = synth.normal_f32(3, "kv32/fused/q", (rows, n_q * D))
    k = synth.normal_f32(3, "kv32/fused/k", (rows, n_kv * D))
    v = synth.normal_f32(3, "kv32/fused/v", (rows, n_kv * D))
    plan = (dl.dl_attn_plan_build_cluster(seqlen, n_q, n_kv, D) if cluster
            else dl.dl_attn_plan_build(seqlen, n_q, n_kv, D))
    rope = dl.make_rope(500000.0, D, cap)
    dpos = torch.tensor(pos, dtype=torch.int32, device="cuda")
    dsl = torch.tensor(seqlen, dtype=torch.int32, device="cuda")
    res = {}
    for mode in ("fused", "separate"):
        kv = dl.KVCache(kc.clone().cuda(), vc.clone().cuda())
        qd = q.clone().cuda()
        out = torch.empty(rows, n_q * D, device="cuda")
        lse = torch.empty(rows, n_q, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if mode == "separate":
            dl.dl_rope_kv_store(qd, k.cuda(), v.cuda(), dpos, rope, kv, n_q, status=status)
        if cluster:
            if mode == "fused":
                dl.dl_decode_attn_cluster(qd, kv, dsl, plan, out, lse, k=k.cuda(), v=v.cuda(), pos=dpos, rope=rope,
                                          status=status)
            else:
                dl.dl_decode_attn_cluster(qd, kv, dsl, plan, out, lse, status=status)
        else:
            ws = dl.workspace_for(plan)
            if mode == "fused":
                dl.dl_decode_attn_rope(qd, k.cuda(), v.cuda(), dpos, rope, kv, dsl, plan, ws, status=status)
            else:
                dl.dl_decode_attn(qd, kv, dsl, plan, ws, status=status)
            dl.dl_attn_merge(ws, plan, dsl, out, lse)
        torch.cuda.synchronize()
        assert dl.dl_status_read(status) == 0
        res[mode] = (kv.k.cpu().numpy(), kv.v.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy())
    for a, b in zip(res["fused"], res["separate"]):
        assert np.array_equal(a, b)
    kc_o, vc_o = kc.numpy().copy(), vc.numpy().copy()
    qo = oracle.rope_kv_store(q, k, v, np.array(pos, np.int32), kc_o, vc_o, n_q=n_q, n_kv=n_kv, head_dim=D, rot_dim=D,
                              theta=500000.0, neox=True)
    ref_out, ref_lse = oracle.attention(qo, kc_o, vc_o, np.array(seqlen, np.int32), n_q=n_q, n_kv=n_kv, head_dim=D,
                                        chunk=plan.chunk, n_splits=plan.max_splits)
    assert_attn_close(res["fused"][2], res["fused"][3], ref_out, ref_lse)


@pytest.mark.parametrize("path", [1, 2])
def test_kv32_keys_past_the_f16_range(dl, path):
    """Keys of magnitude 1e5 (past the f16 range, the reason for the f32 mirror) with small
    queries: both inner products against the oracle (the tensor form's bf16 terms keep f32's
    exponent range)."""
    rows, n_q, n_kv, D, cap = 8, 24, 8, 128, 1024
    seqlen = list(range(cap - 7, cap + 1))
    kc = synth.normal_f32(0, "kv32/wide/K", (1, n_kv, cap, D)) * 1e5
    vc = synth.normal_f32(0, "kv32/wide/V", (1, n_kv, cap, D))
    q = synth.normal_f32(5, "kv32/wide/q", (rows, n_q * D)) * 1e-5
    assert float(kc.abs().max()) > 65504.0
    plan = dl.dl_attn_plan_build(seqlen, n_q, n_kv, D)
    kv = dl.KVCache(kc.cuda(), vc.cuda())
    out, lse = dl.decode_attention(q.cuda(), kv, torch.tensor(seqlen, dtype=torch.int32, device="cuda"), plan,
                                   dl.workspace_for(plan), path=path)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attention(q.numpy().astype(np.float64), kc.numpy(), vc.numpy(),
                                        np.array(seqlen, np.int32), n_q=n_q, n_kv=n_kv, head_dim=D,
                                        chunk=plan.chunk, n_splits=plan.max_splits)
    assert_attn_close(out.cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse)
