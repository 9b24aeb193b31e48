"""Cache slots past every row's keys hold NaN (f16 and f32 mirrors: the values; q8_0 mirror: the
scales): no inner product on any mirror may let them into a result (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import assert_attn_close

pytestmark = pytest.mark.gpu

N_Q, N_KV, D, CAP = 24, 8, 128, 1100


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


@pytest.mark.parametrize("mirror", ["f16", "f32", "q8_0"])
@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("rows", [1, 8])
def test_slots_past_the_keys_are_never_read(dl, mirror, path, rows):
    seqlen = list(range(1001 - rows + 1, 1002))           # the last stage of a piece is partial
    lmax = max(seqlen)
    q = synth.normal_f32(7, "poison/q/%d" % rows, (rows, N_Q * D))
    if mirror == "q8_0":
        kc, ks = synth.kv_q8_random_planes(0, "poison/K", 1, N_KV, CAP, D)
        vc, vs = synth.kv_q8_random_planes(0, "poison/V", 1, N_KV, CAP, D)
        ksn, vsn = ks.numpy().view(np.uint16).copy(), vs.numpy().view(np.uint16).copy()
        ksn[:, :, lmax:, :] = 0x7E00                        # NaN scales past the keys
        vsn[:, :, lmax:, :] = 0x7E00
        kv = dl.KVCache.q8(kc.cuda(), torch.from_numpy(ksn.view(np.float16)).cuda(), vc.cuda(),
                           torch.from_numpy(vsn.view(np.float16)).cuda())
        kp = oracle.Q8Plane(kc.numpy().copy(), ksn)
        vp = oracle.Q8Plane(vc.numpy().copy(), vsn)
    else:
        k = synth.normal_f32(0, "poison/K", (1, N_KV, CAP, D))
        v = synth.normal_f32(0, "poison/V", (1, N_KV, CAP, D))
        k[:, :, lmax:, :] = float("nan")
        v[:, :, lmax:, :] = float("nan")
        if mirror == "f16":
            k, v = k.half(), v.half()
            kp, vp = k.numpy().view(np.uint16).copy(), v.numpy().view(np.uint16).copy()
        else:
            kp, vp = k.numpy().copy(), v.numpy().copy()
        kv = dl.KVCache(k.cuda(), v.cuda())
    plan = dl.dl_attn_plan_build(seqlen, N_Q, N_KV, D)
    ws = dl.workspace_for(plan)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = dl.decode_attention(q.cuda(), kv, torch.tensor(seqlen, dtype=torch.int32, device="cuda"), plan, ws,
                                   status=status, path=path)
    torch.cuda.synchronize()
    assert dl.dl_status_read(status) == 0
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    ref_out, ref_lse = oracle.attention(q.numpy().astype(np.float64), kp, vp, np.array(seqlen, np.int32), n_q=N_Q,
                                        n_kv=N_KV, head_dim=D, chunk=plan.chunk, n_splits=plan.max_splits)
    assert_attn_close(o, l, ref_out, ref_lse)
