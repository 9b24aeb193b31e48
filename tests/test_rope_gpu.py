"""dl_rope_kv_store against the oracle (GPU): stored halves within 1 ulp, the
store's indexing bit-exact, q rotated in place."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import as_u16, f16_ulp_dist

pytestmark = pytest.mark.gpu

POISON = 0x7E00   # a NaN pattern no store can produce


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _case(dl, *, rows, n_q, n_kv, D, rot, cap, n_reg, pos, regions, theta=500000.0, neox=True,
          bias=False, label="rope"):
    q = synth.normal_f32(0, label + "/q", (rows, n_q * D))
    k = synth.normal_f32(0, label + "/k", (rows, n_kv * D))
    v = synth.normal_f32(0, label + "/v", (rows, n_kv * D))
    b = synth.normal_f32(0, label + "/b", ((n_q + 2 * n_kv) * D,)) if bias else None
    shape = (n_reg, n_kv, cap, D)
    kc_o = np.full(shape, POISON, np.uint16)
    vc_o = np.full(shape, POISON, np.uint16)
    pos_np = np.array(pos, np.int32)
    reg_np = np.array(regions, np.int32)
    qo = oracle.rope_kv_store(q, k, v, pos_np, kc_o, vc_o, n_q=n_q, n_kv=n_kv, head_dim=D, rot_dim=rot,
                              theta=theta, neox=neox, bias=b, row_region=reg_np)
    kv = dl.KVCache(torch.from_numpy(np.full(shape, POISON, np.uint16).view(np.float16)).cuda(),
                    torch.from_numpy(np.full(shape, POISON, np.uint16).view(np.float16)).cuda())
    rope = dl.make_rope(theta, rot, cap, neox=neox)
    qd = q.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dl_rope_kv_store(qd, k.cuda(), v.cuda(), torch.from_numpy(pos_np).cuda(), rope, kv, n_q,
                        bias=None if b is None else b.cuda(), row_region=torch.from_numpy(reg_np).cuda(),
                        status=status)
    torch.cuda.synchronize()
    return qd.cpu().numpy(), qo, as_u16(kv.k), kc_o, as_u16(kv.v), vc_o, dl.dl_status_read(status)


def _check(qg, qo, kg, ko, vg, vo):
    # indexing: exactly the oracle's slots were written, nothing else
    assert np.array_equal(kg == POISON, ko == POISON)
    assert np.array_equal(vg == POISON, vo == POISON)
    w = ko != POISON
    assert int(f16_ulp_dist(kg[w], ko[w]).max()) <= 1
    assert int(f16_ulp_dist(vg[w], vo[w]).max()) <= 1
    # q: f32 rotation against the double one (table angles rounded to f32)
    np.testing.assert_allclose(qg, qo, rtol=1e-6, atol=2e-6)


@pytest.mark.parametrize("rows,n_q,n_kv,D,cap,pos", [
    (1, 4, 2, 64, 128, [127]),
    (1, 32, 8, 64, 4097, [4096]),
    (8, 24, 8, 128, 5128, list(range(5120, 5128))),
    (8, 24, 8, 128, 32768, list(range(32760, 32768))),
])
def test_rope_store_configs(dl, rows, n_q, n_kv, D, cap, pos):
    _check(*_case(dl, rows=rows, n_q=n_q, n_kv=n_kv, D=D, rot=D, cap=cap, n_reg=1, pos=pos,
                  regions=[0] * rows, label="rope/%d/%d" % (D, cap))[:6])


def test_rope_store_regions_bias_partial_rotation(dl):
    """Rows in several regions, bias rows added first, a rotated width below head_dim."""
    r = _case(dl, rows=5, n_q=6, n_kv=2, D=128, rot=64, cap=300, n_reg=3, pos=[0, 299, 17, 17, 150],
              regions=[2, 0, 1, 2, 0], bias=True, label="rope/mixed")
    _check(*r[:6])
    assert r[6] == 0


def test_rope_store_interleaved_pairs(dl):
    _check(*_case(dl, rows=2, n_q=4, n_kv=2, D=64, rot=64, cap=64, n_reg=1, pos=[5, 63], regions=[0, 0],
                  neox=False, label="rope/norm")[:6])


def test_rope_store_out_of_range_rows_skipped(dl):
    """A position past the cache is never written; the status word says so."""
    n_q, n_kv, D, cap = 4, 2, 64, 16
    q = synth.normal_f32(9, "rope/oob/q", (2, n_q * D)).cuda()
    k = synth.normal_f32(9, "rope/oob/k", (2, n_kv * D)).cuda()
    v = synth.normal_f32(9, "rope/oob/v", (2, n_kv * D)).cuda()
    shape = (1, n_kv, cap, D)
    kv = dl.KVCache(torch.from_numpy(np.full(shape, POISON, np.uint16).view(np.float16)).cuda(),
                    torch.from_numpy(np.full(shape, POISON, np.uint16).view(np.float16)).cuda())
    rope = dl.make_rope(500000.0, D, 64)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dl_rope_kv_store(q, k, v, torch.tensor([3, 16], dtype=torch.int32, device="cuda"), rope, kv, n_q,
                        status=status)
    st = dl.dl_status_read(status)
    assert st & dl.DL_STATUS_POS_RANGE
    kk = as_u16(kv.k)
    assert np.all(kk[:, :, [i for i in range(cap) if i != 3]] == POISON)
    assert np.all(kk[:, :, 3] != POISON)


def test_rope_store_clamps_to_half_range(dl):
    n_q, n_kv, D, cap = 2, 1, 64, 8
    q = torch.zeros(1, n_q * D, device="cuda")
    k = torch.zeros(1, n_kv * D, device="cuda")
    v = torch.zeros(1, n_kv * D, device="cuda")
    k[0, 3] = 1e5
    v[0, 4] = -1e5
    kv = dl.KVCache.empty(1, n_kv, cap, D)
    rope = dl.make_rope(500000.0, D, cap)
    dl.dl_rope_kv_store(q, k, v, torch.tensor([0], dtype=torch.int32, device="cuda"), rope, kv, n_q)
    torch.cuda.synchronize()
    assert as_u16(kv.k)[0, 0, 0, 3] == 0x7BFF and as_u16(kv.v)[0, 0, 0, 4] == 0xFBFF
