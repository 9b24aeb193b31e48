"""The attention entry point that allocates nothing, against the ordinary one (GPU).

Callers that may not allocate device memory (a fixed budget after start-up, a
host whose device memory belongs to its own pool, code paths where an
allocation's implicit synchronisation is not allowed) use
dl_decode_attention_noalloc, whose partials live in the library's own fixed
buffer.  Its results must match dl_decode_attn + dl_attn_merge with a caller
workspace bit for bit (the same kernels on the same plan), on two calls in a row
(the buffer keeps the previous call's contents), and the oracle's attention within
the attention bars.  This file is collected last so that a run stopping at the
first failure has run every other test first.
"""
import ctypes

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


def _noalloc(dl, q, kv, seqlen, plan, out, lse, status):
    L = dl.lib()
    rc = L.dl_decode_attention_noalloc(
        ctypes.c_void_p(q.data_ptr()), q.stride(0), ctypes.byref(kv.c), ctypes.c_void_p(seqlen.data_ptr()),
        ctypes.byref(plan), ctypes.c_void_p(out.data_ptr()), out.stride(0), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, L.dl_last_error().decode()


@pytest.mark.parametrize("case", ["3b-8", "streams-6"])
def test_noalloc_matches_workspace_entry(dl, case):
    n_q, n_kv, D = 24, 8, 128
    if case == "3b-8":
        seqlen, regions, n_reg, cap = list(range(5121, 5129)), [0] * 8, 1, 5128
    else:
        lens = synth.twelve_stream_lengths(0)[:6]
        seqlen, regions, n_reg, cap = [l + 1 for l in lens], list(range(6)), 6, max(lens) + 1
    k, v = kv_planes("noalloc/" + case, n_reg, n_kv, cap, D)
    kv = dl.KVCache(k.cuda(), v.cuda())
    rows = len(seqlen)
    plan = dl.dl_attn_plan_build(seqlen, n_q, n_kv, D, regions=regions)
    assert plan.workspace_bytes <= dl.lib().dl_decode_attention_noalloc_max_bytes()
    sl = torch.tensor(seqlen, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        q = synth.normal_f32(call, "noalloc/%s/q" % case, (rows, n_q * D)).cuda()
        ws = dl.workspace_for(plan)
        ref_out, ref_lse = dl.decode_attention(q, kv, sl, plan, ws)
        out = torch.full((rows, n_q * D), float("nan"), device="cuda")
        lse = torch.full((rows, n_q), float("nan"), device="cuda")
        _noalloc(dl, q, kv, sl, plan, out, lse, status)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
        oo, ol = oracle.attention(q.cpu().numpy().astype(np.float64), k.numpy().view(np.uint16), v.numpy().view(np.uint16),
                                  np.array(seqlen, np.int32), n_q=n_q, n_kv=n_kv, head_dim=D, chunk=plan.chunk,
                                  n_splits=plan.max_splits, row_region=np.array(regions, np.int32))
        assert_attn_close(out.cpu().numpy(), lse.cpu().numpy(), oo, ol)
    assert dl.dl_status_read(status) == 0


def test_noalloc_refuses_plans_past_its_buffer(dl):
    n_q, n_kv, D = 32, 4, 128
    plan = dl.dl_attn_plan_build([32768] * 8, n_q, n_kv, D, force_chunk=32)   # thousands of pieces
    assert plan.workspace_bytes > dl.lib().dl_decode_attention_noalloc_max_bytes()
    kv = dl.KVCache.empty(1, n_kv, 32768, D)
    q = torch.zeros(8, n_q * D, device="cuda")
    out = torch.zeros(8, n_q * D, device="cuda")
    lse = torch.zeros(8, n_q, device="cuda")
    sl = torch.full((8,), 32768, dtype=torch.int32, device="cuda")
    L = dl.lib()
    rc = L.dl_decode_attention_noalloc(
        ctypes.c_void_p(q.data_ptr()), q.stride(0), ctypes.byref(kv.c), ctypes.c_void_p(sl.data_ptr()),
        ctypes.byref(plan), ctypes.c_void_p(out.data_ptr()), out.stride(0), ctypes.c_void_p(lse.data_ptr()),
        None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == dl.DL_E_WORKSPACE
    assert "fixed buffer" in L.dl_last_error().decode()


def test_noalloc_refuses_cluster_plans(dl):
    """A cluster plan keeps no partials: the entry sends it to the cluster call before launching."""
    n_q, n_kv, D = 24, 8, 128
    plan = dl.dl_attn_plan_build_cluster([5128] * 8, n_q, n_kv, D, regions=[0] * 8)
    assert plan.cluster > 0 and plan.workspace_bytes == 0
    kv = dl.KVCache.empty(1, n_kv, 5128, D)
    q = torch.zeros(8, n_q * D, device="cuda")
    out = torch.zeros(8, n_q * D, device="cuda")
    lse = torch.zeros(8, n_q, device="cuda")
    sl = torch.full((8,), 5128, dtype=torch.int32, device="cuda")
    L = dl.lib()
    rc = L.dl_decode_attention_noalloc(
        ctypes.c_void_p(q.data_ptr()), q.stride(0), ctypes.byref(kv.c), ctypes.c_void_p(sl.data_ptr()),
        ctypes.byref(plan), ctypes.c_void_p(out.data_ptr()), out.stride(0), ctypes.c_void_p(lse.data_ptr()),
        None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == dl.DL_E_ARG
    assert "dl_decode_attn_cluster" in L.dl_last_error().decode()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
