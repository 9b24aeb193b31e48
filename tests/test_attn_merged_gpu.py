"""dl_decode_attn_merged (the last piece of each session and KV head merges the partials) against
the two-launch path it replaces (bit-identical) and the oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import assert_attn_close, kv_planes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _both(dl, q, kv, seqlen_dev, plan, rows, n_q, D, path=0, calls=1, fused=None):
    """(out, lse) of the merged launch (called `calls` times on one workspace) and of the
    partials + merge launches; fused = (k, v, pos, rope) runs the rope/store in each launch
    (the caller restores the cache between the two forms)."""
    ws = dl.workspace_for(plan)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(calls):
        out = torch.full((rows, n_q * D), float("nan"), device="cuda")
        lse = torch.full((rows, n_q), float("nan"), device="cuda")
        kw = {} if fused is None else dict(k=fused[0], v=fused[1], pos=fused[2], rope=fused[3])
        dl.dl_decode_attn_merged(q, kv, seqlen_dev, plan, ws, out, lse, status=status, path=path, **kw)
        torch.cuda.synchronize()
        outs.append((out.cpu().numpy(), lse.cpu().numpy()))
    assert dl.dl_status_read(status) == 0
    # every call leaves the counters zero
    pc = (plan.n_sessions * plan.n_kv * 4 + 15) // 16 * 16
    assert int(ws[plan.workspace_bytes - pc:].cpu().count_nonzero()) == 0
    return outs


def _two_launch(dl, q, kv, seqlen_dev, plan, rows, n_q, D, path=0):
    ws = dl.workspace_for(plan)
    out, lse = dl.decode_attention(q, kv, seqlen_dev, plan, ws, path=path)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("rows,n_q,n_kv,D,cap,path", [
    (1, 24, 8, 128, 5128, 0),      # 3B, one row: CUDA cores
    (1, 32, 8, 64, 4097, 0),       # 1B, one row
    (2, 24, 8, 128, 5128, 0),      # two rows of one session: tensor cores (6 queries)
    (2, 24, 8, 128, 5128, 1),
    (1, 4, 2, 64, 128, 2),         # tiny, tensor form on request
])
def test_merged_equals_two_launches(dl, rows, n_q, n_kv, D, cap, path):
    seqlen = list(range(cap - rows + 1, cap + 1))
    kc, vc = kv_planes("merged/%d/%d/%d" % (rows, D, path), 1, n_kv, cap, D)
    kv = dl.KVCache(kc.cuda(), vc.cuda())
    q = synth.normal_f32(1, "merged/q/%d/%d" % (rows, D), (rows, n_q * D)).cuda()
    plan = dl.dl_attn_plan_build(seqlen, n_q, n_kv, D)
    sl = torch.tensor(seqlen, dtype=torch.int32, device="cuda")
    got = _both(dl, q, kv, sl, plan, rows, n_q, D, path=path, calls=3)
    ref = _two_launch(dl, q, kv, sl, plan, rows, n_q, D, path=path)
    for o, l in got:
        assert np.array_equal(o, ref[0]) and np.array_equal(l, ref[1])
    ro, rl = oracle.attention(q.cpu().numpy().astype(np.float64), kc.numpy().view(np.uint16),
                              vc.numpy().view(np.uint16), np.array(seqlen, np.int32), n_q=n_q, n_kv=n_kv,
                              head_dim=D, chunk=plan.chunk, n_splits=plan.max_splits)
    assert_attn_close(got[0][0], got[0][1], ro, rl)


def test_merged_sessions_short_rows_and_empty(dl):
    """Six one-row sessions of different lengths, device lengths below the planned ones (so some
    pieces have no keys and do not count), and a row with no keys at all (out 0, lse -inf)."""
    n_q, n_kv, D = 24, 8, 128
    lens = [513, 4000, 1500, 64, 2049, 2900]
    cap = 4000
    kc, vc = kv_planes("merged/sess", 6, n_kv, cap, D)
    kv = dl.KVCache(kc.cuda(), vc.cuda())
    q = synth.normal_f32(2, "merged/sess/q", (6, n_q * D)).cuda()
    plan = dl.dl_attn_plan_build(lens, n_q, n_kv, D, regions=list(range(6)))
    for dev_lens in (lens, [300, 1200, 1500, 1, 2049, 100]):
        sl = torch.tensor(dev_lens, dtype=torch.int32, device="cuda")
        got = _both(dl, q, kv, sl, plan, 6, n_q, D, calls=2)
        ref = _two_launch(dl, q, kv, sl, plan, 6, n_q, D)
        for o, l in got:
            assert np.array_equal(o, ref[0]) and np.array_equal(l, ref[1])
        ro, rl = oracle.attention(q.cpu().numpy().astype(np.float64), kc.numpy().view(np.uint16),
                                  vc.numpy().view(np.uint16), np.array(dev_lens, np.int32), n_q=n_q, n_kv=n_kv,
                                  head_dim=D, chunk=plan.chunk, n_splits=plan.max_splits,
                                  row_region=np.arange(6, dtype=np.int32))
        assert_attn_close(got[0][0], got[0][1], ro, rl)
    # a session whose row has no keys: every piece is idle, the first writes the empty result
    sl = torch.tensor([0, 4000, 1500, 64, 2049, 2900], dtype=torch.int32, device="cuda")
    ws = dl.workspace_for(plan)
    out = torch.full((6, n_q * D), float("nan"), device="cuda")
    lse = torch.full((6, n_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dl_decode_attn_merged(q, kv, sl, plan, ws, out, lse, status=status)
    torch.cuda.synchronize()
    assert dl.dl_status_read(status) == dl.DL_STATUS_SEQLEN_RANGE
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(l[0]))
    ref = _two_launch(dl, q, kv, sl, plan, 6, n_q, D)
    assert np.array_equal(o, ref[0]) and np.array_equal(l, ref[1])


@pytest.mark.parametrize("mirror", ["f16", "f32", "q8_0"])
def test_merged_mirrors_and_fused_rope(dl, mirror):
    """On each KV mirror; on the f16 and f32 mirrors also with the rope/store in the launch (the
    stored rows and the results equal the separate store followed by the two launches)."""
    n_q, n_kv, D, cap = 24, 8, 128, 5128
    pos = [5120]
    seqlen = [5121]
    q = synth.normal_f32(3, "merged/mir/q", (1, n_q * D))
    if mirror == "q8_0":
        kc, ks = synth.kv_q8_random_planes(0, "merged/mir/K", 1, n_kv, cap, D)
        vc, vs = synth.kv_q8_random_planes(0, "merged/mir/V", 1, n_kv, cap, D)
        mk = lambda: dl.KVCache.q8(kc.cuda(), ks.cuda(), vc.cuda(), vs.cuda())
    else:
        dt = torch.float16 if mirror == "f16" else torch.float32
        kc = synth.normal_f32(0, "merged/mir/K", (1, n_kv, cap, D)).to(dt)
        vc = synth.normal_f32(0, "merged/mir/V", (1, n_kv, cap, D)).to(dt)
        mk = lambda: dl.KVCache(kc.clone().cuda(), vc.clone().cuda())
    plan = dl.dl_attn_plan_build(seqlen, n_q, n_kv, D)
    sl = torch.tensor(seqlen, dtype=torch.int32, device="cuda")
    kv = mk()
    got = _both(dl, q.cuda(), kv, sl, plan, 1, n_q, D, calls=2)
    ref = _two_launch(dl, q.cuda(), kv, sl, plan, 1, n_q, D)
    for o, l in got:
        assert np.array_equal(o, ref[0]) and np.array_equal(l, ref[1])
    if mirror == "q8_0":
        return
    k = synth.normal_f32(3, "merged/mir/k", (1, n_kv * D)).cuda()
    v = synth.normal_f32(3, "merged/mir/v", (1, n_kv * D)).cuda()
    rope = dl.make_rope(500000.0, D, cap)
    dpos = torch.tensor(pos, dtype=torch.int32, device="cuda")
    kv_f = mk()
    got = _both(dl, q.clone().cuda(), kv_f, sl, plan, 1, n_q, D, fused=(k, v, dpos, rope))
    kv_s = mk()
    qs = q.clone().cuda()
    dl.dl_rope_kv_store(qs, k, v, dpos, rope, kv_s, n_q)
    ref = _two_launch(dl, qs, kv_s, sl, plan, 1, n_q, D)
    assert np.array_equal(got[0][0], ref[0]) and np.array_equal(got[0][1], ref[1])
    assert torch.equal(kv_f.k, kv_s.k) and torch.equal(kv_f.v, kv_s.v)


def test_merged_refusals(dl):
    n_q, n_kv, D, cap = 24, 8, 128, 256
    kc, vc = kv_planes("merged/refuse", 1, n_kv, cap, D)
    kv = dl.KVCache(kc.cuda(), vc.cuda())
    q = torch.zeros(8, n_q * D, device="cuda")
    out = torch.zeros(8, n_q * D, device="cuda")
    sl8 = torch.tensor(list(range(249, 257)), dtype=torch.int32, device="cuda")
    plan8 = dl.dl_attn_plan_build(list(range(249, 257)), n_q, n_kv, D)
    with pytest.raises(dl.DLError) as e:                        # 24 queries per work item
        dl.dl_decode_attn_merged(q, kv, sl8, plan8, dl.workspace_for(plan8), out)
    assert e.value.code == dl.DL_E_SHAPE
    plan1 = dl.dl_attn_plan_build([256], n_q, n_kv, D)
    sl1 = sl8[7:]
    with pytest.raises(dl.DLError) as e:                        # workspace too small
        dl.dl_decode_attn_merged(q[:1], kv, sl1, plan1, torch.zeros(16, dtype=torch.uint8, device="cuda"),
                                 out[:1])
    assert e.value.code == dl.DL_E_WORKSPACE
    cplan = dl.dl_attn_plan_build_cluster([256], n_q, n_kv, D)
    with pytest.raises(dl.DLError) as e:                        # a cluster plan
        dl.dl_decode_attn_merged(q[:1], kv, sl1, cplan, dl.workspace_for(plan1), out[:1])
    assert e.value.code == dl.DL_E_ARG
