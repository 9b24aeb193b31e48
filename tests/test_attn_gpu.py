"""dl_decode_attn + dl_attn_merge against the oracle (GPU)."""
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


def _run(dl, q, k, v, seqlen, regions, n_q, n_kv, D, force_chunk=0, poison=True, path=0):
    plan = dl.dl_attn_plan_build(seqlen, n_q, n_kv, D, regions=regions, force_chunk=force_chunk)
    kv = dl.KVCache(k.cuda(), v.cuda())
    ws = dl.workspace_for(plan)
    if poison:
        ws.view(torch.float32)[:ws.numel() // 4].fill_(float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sl = torch.tensor(seqlen, dtype=torch.int32, device="cuda")
    out, lse = dl.decode_attention(q.cuda(), kv, sl, plan, ws, status=status, path=path)
    torch.cuda.synchronize()
    assert dl.dl_status_read(status) == 0
    return out.cpu().numpy(), lse.cpu().numpy(), plan


def _ref(q, k, v, seqlen, regions, n_q, n_kv, D, plan):
    kc = k.numpy().view(np.uint16)
    vc = v.numpy().view(np.uint16)
    return oracle.attention(q.numpy().astype(np.float64), kc, vc, np.array(seqlen, np.int32), n_q=n_q,
                            n_kv=n_kv, head_dim=D, chunk=plan.chunk, n_splits=plan.max_splits,
                            row_region=None if regions is None else np.array(regions, np.int32))


CONFIGS = {
    # name: (n_q, n_kv, D, n_regions, capacity, seqlens, regions)
    "tiny": (4, 2, 64, 1, 128, [128], None),
    "1b": (32, 8, 64, 1, 4097, [4097], None),
    "3b-1": (24, 8, 128, 1, 5128, [5121], None),
    "3b-2": (24, 8, 128, 1, 5128, [5121, 5122], None),
    "3b-4": (24, 8, 128, 1, 5128, list(range(5121, 5125)), None),
    "3b-8": (24, 8, 128, 1, 5128, list(range(5121, 5129)), None),
    "ragged-tail": (6, 2, 128, 1, 100, [1, 33, 65, 99], None),
}


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("name", list(CONFIGS))
def test_attention_configs(dl, name, path):
    """Both inner products (CUDA cores, tensor cores) and the automatic choice."""
    n_q, n_kv, D, n_reg, cap, seqlen, regions = CONFIGS[name]
    k, v = kv_planes("attn/" + name, n_reg, n_kv, cap, D)
    q = synth.normal_f32(0, "attn/%s/q" % name, (len(seqlen), n_q * D))
    out, lse, plan = _run(dl, q, k, v, seqlen, regions, n_q, n_kv, D, path=path)
    ro, rl = _ref(q, k, v, seqlen, regions, n_q, n_kv, D, plan)
    assert_attn_close(out, lse, ro, rl)


@pytest.mark.parametrize("name,chunk", [("1b", 160), ("1b", 288), ("3b-1", 160), ("3b-2", 32), ("3b-1", 4096)])
def test_attention_cuda_core_stage_counts(dl, name, chunk):
    """CUDA-core form on forced piece lengths: 5 or 9 stages (a ring slot filled twice at head_dim
    64 and 128, one stage group taking two stages), 1 stage per piece (8 queries per warp, 2 rows),
    and 4096 keys (the ring cycling many times); every row ends in a ragged last piece."""
    n_q, n_kv, D, n_reg, cap, seqlen, regions = CONFIGS[name]
    k, v = kv_planes("attn/" + name, n_reg, n_kv, cap, D)
    q = synth.normal_f32(0, "attn/%s/q" % name, (len(seqlen), n_q * D))
    out, lse, plan = _run(dl, q, k, v, seqlen, regions, n_q, n_kv, D, force_chunk=chunk, path=1)
    assert plan.chunk == chunk
    ro, rl = _ref(q, k, v, seqlen, regions, n_q, n_kv, D, plan)
    assert_attn_close(out, lse, ro, rl)


def test_attention_twelve_streams(dl):
    """Twelve one-row streams with their own caches, lengths U{512..8192}, run as 6 + 6."""
    n_q, n_kv, D = 24, 8, 128
    lens = synth.twelve_stream_lengths(0)
    cap = max(lens) + 1
    k, v = kv_planes("attn/streams", 12, n_kv, cap, D)
    q = synth.normal_f32(0, "attn/streams/q", (12, n_q * D))
    assert dl.dl_plan_groups(12) == [6, 6]
    for g in range(2):
        rows = list(range(6 * g, 6 * g + 6))
        seqlen = [lens[r] + 1 for r in rows]
        out, lse, plan = _run(dl, q[rows[0]:rows[-1] + 1], k, v, seqlen, rows, n_q, n_kv, D)
        assert plan.n_sessions == 6
        ro, rl = _ref(q[rows[0]:rows[-1] + 1], k, v, seqlen, rows, n_q, n_kv, D, plan)
        assert_attn_close(out, lse, ro, rl)


def test_attention_long_context_split_invariance(dl):
    """Eight rows at positions 32760..32767: any piece length agrees with one piece."""
    n_q, n_kv, D, cap = 24, 8, 128, 32768
    seqlen = list(range(32761, 32769))
    k, v = kv_planes("attn/long", 1, n_kv, cap, D)
    q = synth.normal_f32(0, "attn/long/q", (8, n_q * D))
    out_auto, lse_auto, plan = _run(dl, q, k, v, seqlen, None, n_q, n_kv, D)
    ro, rl = oracle.attn_full(q.numpy().astype(np.float64), k.numpy().view(np.uint16), v.numpy().view(np.uint16),
                              np.array(seqlen, np.int32), n_q=n_q, n_kv=n_kv, head_dim=D)
    assert_attn_close(out_auto, lse_auto, ro, rl)
    for chunk, path in ((32768, 0), (2 * plan.chunk, 0), (4096, 1), (96, 2), (plan.chunk, 1)):
        out, lse, p2 = _run(dl, q, k, v, seqlen, None, n_q, n_kv, D, force_chunk=chunk, path=path)
        assert_attn_close(out, lse, ro, rl)
        assert np.max(np.abs(out - out_auto)) <= 2e-3


@pytest.mark.parametrize("path", [1, 2])
def test_attention_peaked_query_teeth(dl, path):
    """A query aimed at one key returns that key's value; the control fails on a wrong value row."""
    n_q, n_kv, D, cap = 2, 1, 128, 700
    k, v = kv_planes("attn/peak", 1, n_kv, cap, D)
    K = k.numpy().astype(np.float64)
    j = 613
    q = np.zeros((1, n_q * D), np.float32)
    q[0, :D] = 30.0 * K[0, 0, j] / np.linalg.norm(K[0, 0, j]) * np.sqrt(D)
    q[0, D:] = synth.normal_f32(0, "attn/peak/q2", (D,)).numpy()
    q = torch.from_numpy(q)
    out, lse, plan = _run(dl, q, k, v, [cap], None, n_q, n_kv, D, path=path)
    ro, rl = _ref(q, k, v, [cap], None, n_q, n_kv, D, plan)
    assert_attn_close(out, lse, ro, rl)
    V = v.numpy().astype(np.float64)
    assert np.max(np.abs(out[0, :D] - V[0, 0, j])) < 2e-3
    assert np.max(np.abs(out[0, :D] - V[0, 0, j - 1])) > 2e-3


def test_attention_workspace_too_small(dl):
    n_q, n_kv, D = 4, 2, 64
    plan = dl.dl_attn_plan_build([64], n_q, n_kv, D)
    kv = dl.KVCache.empty(1, n_kv, 64, D)
    q = torch.zeros(1, n_q * D, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(dl.DLError) as e:
        dl.dl_decode_attn(q, kv, torch.tensor([64], dtype=torch.int32, device="cuda"), plan, ws)
    assert e.value.code == dl.DL_E_WORKSPACE


def test_attention_seqlen_past_plan_reported(dl):
    """A device key count past the plan is clipped and flagged, never read past."""
    n_q, n_kv, D, cap = 4, 2, 64, 256
    k, v = kv_planes("attn/clip", 1, n_kv, cap, D)
    q = synth.normal_f32(0, "attn/clip/q", (1, n_q * D))
    plan = dl.dl_attn_plan_build([100], n_q, n_kv, D)
    kv = dl.KVCache(k.cuda(), v.cuda())
    ws = dl.workspace_for(plan)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sl = torch.tensor([200], dtype=torch.int32, device="cuda")
    out, lse = dl.decode_attention(q.cuda(), kv, sl, plan, ws, status=status)
    assert dl.dl_status_read(status) & dl.DL_STATUS_SEQLEN_RANGE
    ro, rl = _ref(q, k, v, [100], None, n_q, n_kv, D, plan)
    assert_attn_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl)
