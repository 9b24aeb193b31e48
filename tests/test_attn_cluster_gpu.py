"""dl_decode_attn_cluster (the pieces of a KV head merged inside their thread-block cluster) against
the oracle, the partials + merge path and the fused rope (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import as_u16, assert_attn_close, kv_planes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _cluster(dl, q, kc, vc, seqlen, regions, n_q, n_kv, D, max_cluster=0, path=0):
    plan = dl.dl_attn_plan_build_cluster(seqlen, n_q, n_kv, D, regions=regions, max_cluster=max_cluster)
    kv = dl.KVCache(kc.cuda(), vc.cuda())
    rows = len(seqlen)
    out = torch.full((rows, n_q * D), float("nan"), device="cuda")
    lse = torch.full((rows, n_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dl_decode_attn_cluster(q.cuda(), kv, torch.tensor(seqlen, dtype=torch.int32, device="cuda"), plan, out, lse,
                              status=status, path=path)
    torch.cuda.synchronize()
    assert dl.dl_status_read(status) == 0
    return out.cpu().numpy(), lse.cpu().numpy(), plan


def _oracle(q, kc, vc, seqlen, regions, n_q, n_kv, D, plan):
    return oracle.attention(q.numpy().astype(np.float64), kc.numpy().view(np.uint16), vc.numpy().view(np.uint16),
                            np.array(seqlen, np.int32), n_q=n_q, n_kv=n_kv, head_dim=D, chunk=plan.chunk,
                            n_splits=plan.max_splits, row_region=np.array(regions, np.int32))


@pytest.mark.parametrize("rows,n_q,n_kv,D,cap,first", [
    (1, 4, 2, 64, 128, 128),
    (1, 32, 8, 64, 4097, 4097),
    (1, 24, 8, 128, 5128, 5121),
    (8, 24, 8, 128, 5128, 5121),
    (8, 24, 8, 128, 32768, 32761),
])
def test_cluster_configs(dl, rows, n_q, n_kv, D, cap, first):
    seqlen = list(range(first, first + rows))
    q = synth.normal_f32(0, "clu/q/%d/%d" % (rows, cap), (rows, n_q * D))
    kc, vc = kv_planes("clu/%d/%d" % (rows, cap), 1, n_kv, cap, D)
    out, lse, plan = _cluster(dl, q, kc, vc, seqlen, [0] * rows, n_q, n_kv, D)
    assert 1 <= plan.cluster <= 16 and plan.workspace_bytes == 0
    ref_out, ref_lse = _oracle(q, kc, vc, seqlen, [0] * rows, n_q, n_kv, D, plan)
    assert_attn_close(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("max_cluster", [4, 8, 16])
def test_cluster_sessions_with_idle_pieces(dl, max_cluster):
    """Six sessions of very different lengths in one command: the short ones leave pieces of
    their clusters without keys, which take part in the merge and weigh nothing."""
    lens = [513, 8192, 1500, 64, 4097, 2900]
    n_q, n_kv, D = 24, 8, 128
    q = synth.normal_f32(1, "clu/sess/q", (6, n_q * D))
    kc, vc = kv_planes("clu/sess", 6, n_kv, 8192, D)
    out, lse, plan = _cluster(dl, q, kc, vc, lens, list(range(6)), n_q, n_kv, D, max_cluster=max_cluster)
    assert plan.cluster <= max_cluster
    ref_out, ref_lse = _oracle(q, kc, vc, lens, list(range(6)), n_q, n_kv, D, plan)
    assert_attn_close(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("rows", [1, 8])
def test_cluster_both_inner_products_and_partials_path(dl, path, rows):
    """Each inner product meets the bars, and agrees with the partials + merge path."""
    n_q, n_kv, D = 24, 8, 128
    seqlen = list(range(5121, 5121 + rows))
    q = synth.normal_f32(2, "clu/path/%d" % rows, (rows, n_q * D))
    kc, vc = kv_planes("clu/path/%d" % rows, 1, n_kv, 5128, D)
    out, lse, plan = _cluster(dl, q, kc, vc, seqlen, [0] * rows, n_q, n_kv, D, path=path)
    ref_out, ref_lse = _oracle(q, kc, vc, seqlen, [0] * rows, n_q, n_kv, D, plan)
    assert_attn_close(out, lse, ref_out, ref_lse)
    p2 = dl.dl_attn_plan_build(seqlen, n_q, n_kv, D)
    ws = dl.workspace_for(p2)
    kv = dl.KVCache(kc.cuda(), vc.cuda())
    o2, l2 = dl.decode_attention(q.cuda(), kv, torch.tensor(seqlen, dtype=torch.int32, device="cuda"), p2, ws,
                                 path=path)
    torch.cuda.synchronize()
    assert_attn_close(out, lse, o2.cpu().numpy().astype(np.float64), l2.cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("rows", [1, 8])
def test_cluster_with_fused_rope(dl, rows):
    """Rope and store inside the cluster launch: stored halves and results bit-identical to a
    separate store followed by the cluster launch; q stays as projected."""
    n_q, n_kv, D, cap = 24, 8, 128, 5128
    pos = list(range(5120, 5120 + rows))
    seqlen = [p + 1 for p in pos]
    q = synth.normal_f32(3, "clu/rope/q%d" % rows, (rows, n_q * D))
    k = synth.normal_f32(3, "clu/rope/k%d" % rows, (rows, n_kv * D))
    v = synth.normal_f32(3, "clu/rope/v%d" % rows, (rows, n_kv * D))
    kc, vc = kv_planes("clu/rope/%d" % rows, 1, n_kv, cap, D)
    plan = dl.dl_attn_plan_build_cluster(seqlen, n_q, n_kv, D)
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
        if mode == "fused":
            dl.dl_decode_attn_cluster(qd, kv, dsl, plan, out, lse, k=k.cuda(), v=v.cuda(), pos=dpos, rope=rope,
                                      status=status)
        else:
            dl.dl_rope_kv_store(qd, k.cuda(), v.cuda(), dpos, rope, kv, n_q, status=status)
            dl.dl_decode_attn_cluster(qd, kv, dsl, plan, out, lse, status=status)
        torch.cuda.synchronize()
        assert dl.dl_status_read(status) == 0
        res[mode] = (as_u16(kv.k), as_u16(kv.v), out.cpu().numpy(), lse.cpu().numpy(), qd.cpu().numpy())
    f, s = res["fused"], res["separate"]
    for i in range(4):
        assert np.array_equal(f[i], s[i])
    assert np.array_equal(f[4], q.numpy())


def test_cluster_refusals(dl):
    """A cluster plan is refused by the partials calls and the merge, a partials plan by the
    cluster call, before anything launches."""
    n_q, n_kv, D = 4, 2, 64
    kc, vc = kv_planes("clu/refuse", 1, n_kv, 256, D)
    kv = dl.KVCache(kc.cuda(), vc.cuda())
    q = torch.zeros(1, n_q * D, device="cuda")
    sl = torch.tensor([200], dtype=torch.int32, device="cuda")
    pc = dl.dl_attn_plan_build_cluster([200], n_q, n_kv, D)
    pp = dl.dl_attn_plan_build([200], n_q, n_kv, D)
    ws = dl.workspace_for(pp)
    out = torch.zeros(1, n_q * D, device="cuda")
    for call in (lambda: dl.dl_decode_attn(q, kv, sl, pc, ws),
                 lambda: dl.dl_attn_merge(ws, pc, sl, out),
                 lambda: dl.dl_decode_attn_cluster(q, kv, sl, pp, out)):
        with pytest.raises(dl.DLError) as e:
            call()
        assert e.value.code == dl.DL_E_ARG
