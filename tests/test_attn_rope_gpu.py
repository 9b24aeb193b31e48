"""dl_decode_attn_rope (rope and KV store fused into the attention launch) against the two
separate calls and against the oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import as_u16, assert_attn_close, f16_ulp_dist, kv_planes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _inputs(label, rows, n_q, n_kv, D, n_reg, cap, bias):
    q = synth.normal_f32(0, label + "/q", (rows, n_q * D))
    k = synth.normal_f32(0, label + "/k", (rows, n_kv * D))
    v = synth.normal_f32(0, label + "/v", (rows, n_kv * D))
    b = synth.normal_f32(0, label + "/b", ((n_q + 2 * n_kv) * D,)) if bias else None
    kc, vc = kv_planes(label, n_reg, n_kv, cap, D)
    return q, k, v, b, kc, vc


def _both(dl, *, rows, n_q, n_kv, D, cap, pos, regions=None, n_reg=1, seqlen=None, rot=None, neox=True,
          bias=False, force_chunk=0, path=0, label="fused"):
    """Run the fused call and the two separate calls on identical inputs; return both results."""
    rot = D if rot is None else rot
    regions = [0] * rows if regions is None else regions
    seqlen = [p + 1 for p in pos] if seqlen is None else seqlen
    q, k, v, b, kc, vc = _inputs(label, rows, n_q, n_kv, D, n_reg, cap, bias)
    plan = dl.dl_attn_plan_build(seqlen, n_q, n_kv, D, regions=regions, force_chunk=force_chunk)
    rope = dl.make_rope(500000.0, rot, cap, neox=neox)
    dpos = torch.tensor(pos, dtype=torch.int32, device="cuda")
    dsl = torch.tensor(seqlen, dtype=torch.int32, device="cuda")
    dreg = torch.tensor(regions, dtype=torch.int32, device="cuda")
    bd = None if b is None else b.cuda()
    res = {}
    for mode in ("fused", "separate"):
        kv = dl.KVCache(kc.clone().cuda(), vc.clone().cuda())
        ws = dl.workspace_for(plan)
        ws.view(torch.float32)[:ws.numel() // 4].fill_(float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        qd = q.clone().cuda()
        out = torch.empty(rows, n_q * D, device="cuda")
        lse = torch.empty(rows, n_q, device="cuda")
        if mode == "fused":
            dl.dl_decode_attn_rope(qd, k.cuda(), v.cuda(), dpos, rope, kv, dsl, plan, ws, bias=bd, status=status,
                                   path=path)
        else:
            dl.dl_rope_kv_store(qd, k.cuda(), v.cuda(), dpos, rope, kv, n_q, bias=bd, row_region=dreg, status=status)
            dl.dl_decode_attn(qd, kv, dsl, plan, ws, status=status, path=path)
        dl.dl_attn_merge(ws, plan, dsl, out, lse)
        torch.cuda.synchronize()
        res[mode] = dict(q=qd.cpu().numpy(), kc=as_u16(kv.k), vc=as_u16(kv.v), out=out.cpu().numpy(),
                         lse=lse.cpu().numpy(), status=dl.dl_status_read(status))
    return res, (q, k, v, b, kc, vc, plan, seqlen, regions, rot, neox)


def _assert_same(res, q_raw):
    f, s = res["fused"], res["separate"]
    assert np.array_equal(f["kc"], s["kc"]) and np.array_equal(f["vc"], s["vc"])
    assert np.array_equal(f["out"], s["out"]) and np.array_equal(f["lse"], s["lse"])
    assert f["status"] == s["status"]
    # the fused call leaves q as projected
    assert np.array_equal(f["q"], q_raw.numpy())


def _assert_oracle(res, inputs, *, n_q, n_kv, D, pos):
    q, k, v, b, kc, vc, plan, seqlen, regions, rot, neox = inputs
    kc_o = kc.numpy().view(np.uint16).copy()
    vc_o = vc.numpy().view(np.uint16).copy()
    qo = oracle.rope_kv_store(q, k, v, np.array(pos, np.int32), kc_o, vc_o, n_q=n_q, n_kv=n_kv, head_dim=D,
                              rot_dim=rot, theta=500000.0, neox=neox, bias=b,
                              row_region=np.array(regions, np.int32))
    f = res["fused"]
    w = kc_o != kc.numpy().view(np.uint16)
    assert int(f16_ulp_dist(f["kc"][w], kc_o[w]).max()) <= 1
    assert int(f16_ulp_dist(f["vc"][w], vc_o[w]).max()) <= 1
    ref_out, ref_lse = oracle.attention(qo, kc_o, vc_o, np.array(seqlen, np.int32), n_q=n_q, n_kv=n_kv,
                                        head_dim=D, chunk=plan.chunk, n_splits=plan.max_splits,
                                        row_region=np.array(regions, np.int32))
    assert_attn_close(f["out"], f["lse"], ref_out, ref_lse)


@pytest.mark.parametrize("rows,n_q,n_kv,D,cap,pos", [
    (1, 4, 2, 64, 128, [127]),
    (1, 32, 8, 64, 4097, [4096]),
    (1, 24, 8, 128, 5128, [5120]),
    (8, 24, 8, 128, 5128, list(range(5120, 5128))),
    (8, 24, 8, 128, 32768, list(range(32760, 32768))),
])
def test_fused_equals_separate_and_oracle(dl, rows, n_q, n_kv, D, cap, pos):
    """The configs' shapes: stored halves, outputs and LSE bit-identical to rope/store + attention,
    and within the bars of the oracle."""
    res, inputs = _both(dl, rows=rows, n_q=n_q, n_kv=n_kv, D=D, cap=cap, pos=pos, label="fused/%d/%d" % (rows, D))
    _assert_same(res, inputs[0])
    assert res["fused"]["status"] == 0
    _assert_oracle(res, inputs, n_q=n_q, n_kv=n_kv, D=D, pos=pos)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("rows", [1, 8])
def test_fused_both_inner_products(dl, path, rows):
    pos = list(range(5120, 5120 + rows))
    res, inputs = _both(dl, rows=rows, n_q=24, n_kv=8, D=128, cap=5128, pos=pos, path=path,
                        label="fused/path/%d" % rows)
    _assert_same(res, inputs[0])
    _assert_oracle(res, inputs, n_q=24, n_kv=8, D=128, pos=pos)


def test_fused_new_rows_across_a_piece_boundary(dl):
    """Pieces of 32 keys with the 8 new positions straddling a boundary: each piece stores and
    reads its own share."""
    pos = list(range(5116, 5124))
    res, inputs = _both(dl, rows=8, n_q=24, n_kv=8, D=128, cap=5128, pos=pos, force_chunk=32,
                        label="fused/boundary")
    _assert_same(res, inputs[0])
    _assert_oracle(res, inputs, n_q=24, n_kv=8, D=128, pos=pos)


def test_fused_sessions_regions_bias_partial_interleaved(dl):
    """Six one-row sessions in their own regions, a bias, interleaved pairs over half the channels."""
    pos = [700, 1300, 95, 2047, 511, 1800]
    res, inputs = _both(dl, rows=6, n_q=32, n_kv=8, D=64, cap=2048, pos=pos, regions=list(range(6)), n_reg=6,
                        rot=32, neox=False, bias=True, label="fused/sessions")
    _assert_same(res, inputs[0])
    _assert_oracle(res, inputs, n_q=32, n_kv=8, D=64, pos=pos)


def test_fused_position_past_the_keys_is_stored(dl):
    """A row that does not attend its own new key (seqlen = pos) still gets it stored, like the
    separate store does."""
    pos = [300]
    res, inputs = _both(dl, rows=1, n_q=4, n_kv=2, D=64, cap=512, pos=pos, seqlen=[300], label="fused/past")
    _assert_same(res, inputs[0])


def test_fused_out_of_range_position_flagged(dl):
    """A position outside the cache is neither stored nor read out of bounds; the status says so."""
    res, _ = _both(dl, rows=2, n_q=4, n_kv=2, D=64, cap=256, pos=[100, 256], seqlen=[101, 256],
                   label="fused/range")
    f, s = res["fused"], res["separate"]
    assert f["status"] & 1 and s["status"] & 1
    assert np.array_equal(f["kc"], s["kc"]) and np.array_equal(f["vc"], s["vc"])
