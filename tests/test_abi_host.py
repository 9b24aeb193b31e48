"""The C-ABI library without a GPU: it loads, exports every symbol include/dl.h
declares, and its host-only logic (packed sizes, grouping, split plans, RoPE
tables, argument refusals) behaves as documented."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import oracle
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "dl.h")


@pytest.fixture(scope="module")
def dl():
    from row_decode_step_gb300 import _build
    _build.build()
    import row_decode_step_gb300 as m
    m.lib()
    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dl_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(dl):
    names = _declared_functions()
    assert len(names) >= 13
    L = ctypes.CDLL(dl.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_version_and_error_text(dl):
    assert dl.lib().dl_version() == 100
    with pytest.raises(dl.DLError) as e:
        dl.dl_q8_packed_size(16, 33)
    assert e.value.code == dl.DL_E_SHAPE and "n_in" in str(e.value)


def test_packed_sizes_match_q8_bytes(dl):
    for n_out, n_in in ((5120, 3072), (3072, 3072), (16384, 3072), (3072, 8192), (2048, 8192)):
        qb, db = dl.dl_q8_packed_size(n_out, n_in)
        assert qb + db == n_out * n_in // 32 * 34
    # ragged shapes pad to whole tiles
    qb, db = dl.dl_q8_packed_size(37, 96)
    assert qb == 3 * 4 * 512 and db == 3 * 4 * 32


def test_f16w_packed_sizes(dl):
    """The f16 device plane is the matrix's f16 bytes on full tiles, padded to whole tiles else;
    widths that are not a multiple of 32 are refused."""
    for n_out, n_in in ((5120, 3072), (16384, 3072), (3072, 8192)):
        assert dl.dl_f16w_packed_size(n_out, n_in) == n_out * n_in * 2
    assert dl.dl_f16w_packed_size(37, 96) == 3 * 4 * 1024
    with pytest.raises(dl.DLError) as e:
        dl.dl_f16w_packed_size(16, 48)
    assert e.value.code == dl.DL_E_SHAPE


def test_grouping_matches_oracle_and_golden(dl):
    for n in range(0, 70):
        assert dl.dl_plan_groups(n) == (oracle.plan_groups(n) if n else [])
    assert dl.dl_plan_groups(12) == [6, 6]


def test_attn_plan_fills_sms(dl):
    for rows, sl, regs in ((1, [5121], None), (8, list(range(5121, 5129)), None),
                           (8, list(range(32761, 32769)), None),
                           (6, [600, 8000, 513, 4000, 2222, 7777], list(range(6)))):
        p = dl.dl_attn_plan_build(sl, 24, 8, 128, regions=regs, sm_count=148)
        assert p.rows == rows and p.chunk % 32 == 0
        # every key of every row is covered by the pieces of its session
        for s in range(p.n_sessions):
            rws = [p.sess_rows[i] for i in range(p.sess_begin[s], p.sess_begin[s + 1])]
            assert p.sess_splits[s] * p.chunk >= max(sl[r] for r in rws)
            assert (p.sess_splits[s] - 1) * p.chunk < max(sl[r] for r in rws)
        assert p.n_work == sum(8 * p.sess_splits[s] for s in range(p.n_sessions))
        # enough work items to cover the SMs whenever the keys allow it
        total_tiles = sum(8 * math.ceil(max(sl) / 32) for _ in range(1))
        assert p.n_work >= min(148, total_tiles)
        assert p.workspace_bytes >= rows * 24 * p.max_splits * 129 * 4
        # partial outputs, partial LSEs, then the last-piece merge's counters, each 16-byte rounded
        r16 = lambda b: (b + 15) // 16 * 16
        assert p.workspace_bytes == (r16(rows * 24 * p.max_splits * 128 * 4) + r16(rows * 24 * p.max_splits * 4) +
                                     r16(p.n_sessions * 8 * 4))


def test_attn_plan_sessions(dl):
    # rows of one region share work items; different regions do not
    p = dl.dl_attn_plan_build([100, 101, 50, 102], 24, 8, 128, regions=[3, 3, 1, 3], sm_count=148)
    assert p.n_sessions == 2
    assert [p.sess_rows[i] for i in range(4)] == [0, 1, 3, 2]
    # a session wider than one work item's 32 queries is split
    p = dl.dl_attn_plan_build([64] * 8, 32, 4, 64, sm_count=148)   # group 8: four rows per item
    assert p.n_sessions == 2


def test_attn_plan_cluster_shapes(dl):
    """Cluster plans: every (session, KV head) has the same C <= max_cluster pieces of a multiple of
    32 keys covering the longest session, laid out as consecutive work items, with no workspace."""
    for lens, regions, mc in (([5121], None, 0), ([5121 + r for r in range(8)], None, 0),
                              ([513, 8192, 1500, 64, 4097, 2900], list(range(6)), 8), ([32761], None, 4)):
        P = dl.dl_attn_plan_build_cluster(lens, 24, 8, 128, regions=regions, sm_count=152, max_cluster=mc)
        C = P.cluster
        assert 1 <= C <= (mc or 16) and P.workspace_bytes == 0
        assert P.chunk % 32 == 0 and C * P.chunk >= max(lens) > (C - 1) * P.chunk
        assert P.n_work == P.n_sessions * 8 * C and P.max_splits == C
        for s in range(P.n_sessions):
            assert P.sess_splits[s] == C and P.sess_item0[s] == s * 8 * C
    with pytest.raises(dl.DLError):
        dl.dl_attn_plan_build_cluster([100], 24, 8, 128, max_cluster=17)


def test_attn_plan_refusals(dl):
    for args, code in ((([5] * 9, 24, 8, 128), dl.DL_E_SHAPE),
                       (([0], 24, 8, 128), dl.DL_E_ARG),
                       (([5], 24, 7, 128), dl.DL_E_SHAPE),
                       (([5], 24, 8, 96), dl.DL_E_SHAPE)):
        with pytest.raises(dl.DLError) as e:
            dl.dl_attn_plan_build(*args, sm_count=148)
        assert e.value.code == code


def test_rope_table_against_double_math(dl):
    t = dl.dl_rope_table_build(500000.0, 128, 40000).numpy()
    for p in (0, 1, 127, 5120, 32767, 39999):
        for j in (0, 1, 31, 63):
            a = p * 500000.0 ** (-2.0 * j / 128)
            assert t[p, j, 0] == np.float32(math.cos(a))
            assert t[p, j, 1] == np.float32(math.sin(a))


def test_null_and_shape_refusals_before_any_launch(dl):
    L = dl.lib()
    assert L.dl_gemv_q8(None, None, 1, 0, None, 0, None) == dl.DL_E_ARG
    assert L.dl_rope_kv_store(None, 0, None, 0, None, 0, None, None, None, 1, 8, None, None, None, None) == dl.DL_E_ARG
    assert L.dl_plan_groups(-1, 8, None) == dl.DL_E_ARG
    assert L.dl_status_read(None, None) == dl.DL_E_ARG
    assert L.dl_decode_attn_merged(None, 0, None, None, None, None, None, 0, None, 0, None, None, 0, None) == dl.DL_E_ARG
    w = dl.dl_q8_weight(16, 16, 64, 100)   # n_in not a multiple of 32
    x = ctypes.c_float(0)
    assert L.dl_gemv_q8(ctypes.byref(w), ctypes.byref(x), 1, 128, ctypes.byref(x), 64, None) == dl.DL_E_SHAPE


def test_l2_prefetch_next_arguments(dl):
    """The prefetch ranges are checked on the host: count, null arrays, 16-byte starts and sizes
    (pointers are host integers here: nothing is dereferenced or launched)."""
    L = dl.lib()
    P, SZ = ctypes.c_void_p, ctypes.c_size_t
    assert L.dl_l2_prefetch_next(0, None, None) == dl.DL_OK
    assert L.dl_l2_prefetch_next(-1, None, None) == dl.DL_E_ARG
    assert L.dl_l2_prefetch_next(17, (P * 17)(*([4096] * 17)), (SZ * 17)(*([16] * 17))) == dl.DL_E_ARG
    assert L.dl_l2_prefetch_next(1, None, None) == dl.DL_E_ARG
    assert L.dl_l2_prefetch_next(2, (P * 2)(4096, 4104), (SZ * 2)(16, 16)) == dl.DL_E_ALIGN   # start
    assert L.dl_l2_prefetch_next(1, (P * 1)(4096), (SZ * 1)(24)) == dl.DL_E_ALIGN            # size
    assert L.dl_l2_prefetch_next(1, (P * 1)(None), (SZ * 1)(16)) == dl.DL_E_ALIGN            # null range
    assert L.dl_l2_prefetch_next(16, (P * 16)(*([4096] * 16)), (SZ * 16)(*([0, 32] * 8))) == dl.DL_OK
    # the next launching call takes them even when it refuses its own arguments
    assert L.dl_gemv_q8(None, None, 1, 0, None, 0, None) == dl.DL_E_ARG
    assert L.dl_l2_prefetch_next(0, None, None) == dl.DL_OK


def test_layer_step_refusals_before_any_launch(dl):
    """dl_layer_step checks its plan and cache on the host first: a cluster plan (no partials in
    the workspace) and a mirror other than f16 are refused before anything is read on the device
    (pointers are host integers here: nothing is dereferenced or launched)."""
    L = dl.lib()
    P = ctypes.c_void_p
    assert L.dl_layer_step(None, None, None, None, None, None, None, None, None, 0, None, 0, None) == dl.DL_E_ARG
    n_q, n_kv, D = 24, 8, 128
    W = dl.dl_layer_weights()
    B = dl.dl_layer_bufs()
    rope = dl.dl_rope()
    kv = dl.dl_kv_cache()
    kv.k, kv.v, kv.head_dim, kv.n_kv, kv.capacity, kv.n_regions = 4096, 8192, D, n_kv, 5128, 1
    kv.region_stride, kv.elem_bytes = n_kv * 5128 * D, 2
    fake = P(4096)
    cplan = dl.dl_attn_plan_build_cluster([5128] * 8, n_q, n_kv, D, regions=[0] * 8, sm_count=152)
    rc = L.dl_layer_step(ctypes.byref(W), ctypes.byref(B), None, fake, ctypes.byref(rope), ctypes.byref(kv),
                         fake, ctypes.byref(cplan), fake, 1 << 20, None, 0, None)
    assert rc == dl.DL_E_ARG and "cluster" in L.dl_last_error().decode()
    plan = dl.dl_attn_plan_build([5128] * 8, n_q, n_kv, D, regions=[0] * 8, sm_count=152)
    kv.elem_bytes = 4
    rc = L.dl_layer_step(ctypes.byref(W), ctypes.byref(B), None, fake, ctypes.byref(rope), ctypes.byref(kv),
                         fake, ctypes.byref(plan), fake, 1 << 20, None, 0, None)
    assert rc == dl.DL_E_SHAPE and "f16" in L.dl_last_error().decode()


@pytest.mark.parametrize("kw", [dict(one_launch=True), dict(gemv_chain=True)])
def test_layer_step_refuses_concurrent_grid_wide_launches(kw):
    """Launches that hold every SM and wait across their CTAs cannot run as concurrent commands:
    the refusal comes before anything is allocated."""
    from row_decode_step_gb300.step import LayerStep
    with pytest.raises(ValueError):
        LayerStep([5120] * 12, list(range(12)), 24, 8, 128, 3072, 8192, "cpu", concurrent=True, **kw)


def test_oracle_results_do_not_depend_on_threads():
    """The oracle's parallel loops give each result to one thread in the stated order: any thread
    count returns the same bits."""
    import synth
    blocks = synth.q8_0_blocks_from_normal(4, "thr/w", 96, 256).numpy()
    x = synth.normal_f32(4, "thr/x", (3, 256)).numpy()
    k = synth.kv_cache_normal(4, "thr/K", 1, 2, 300, 64).numpy().view(np.uint16)
    v = synth.kv_cache_normal(4, "thr/V", 1, 2, 300, 64).numpy().view(np.uint16)
    q = synth.normal_f32(4, "thr/q", (3, 8 * 64)).numpy().astype(np.float64)
    sl = np.array([300, 171, 1], np.int32)
    got = []
    for t in (1, 4):
        oracle.set_threads(t)
        y = oracle.gemv_q8(blocks, x)
        o, l = oracle.attention(q, k, v, sl, n_q=8, n_kv=2, head_dim=64, chunk=64, n_splits=5)
        got.append((y, o, l))
    oracle.set_threads(1)
    for a, b in zip(got[0], got[1]):
        assert np.array_equal(a, b)
