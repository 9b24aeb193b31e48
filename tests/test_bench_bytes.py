"""bench.py's algorithmic byte count of a layer step (the numerator of every GB/s and HBM
fraction it reports), checked on CPU against sums written out from the shapes."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _step(wl):
    from row_decode_step_gb300.step import LayerStep
    S = wl["shape"]
    # host plans only (sm_count given, so no device query); buffers on the CPU
    return LayerStep(wl["positions"], wl["regions"], S.n_q, S.n_kv, S.head_dim, S.hidden, S.ffn, "cpu",
                     sm_count=152)


@pytest.mark.parametrize("kv,kv_read,kv_new", [
    ("f16", 5128 * 8 * 128 * 2 * 2, 8 * 8 * 128 * 2 * 2),
    ("q8_0", 5128 * 8 * 128 * 2 * 34 // 32, 8 * 8 * 128 * 2 * 34 // 32),
    ("f32", 5128 * 8 * 128 * 2 * 4, 8 * 8 * 128 * 2 * 4),
])
def test_step_bytes_3b_8_rows(dl, kv, kv_read, kv_new):
    import bench
    wl = bench.workload("3b-8")
    weights = (5120 * 3072 + 3072 * 3072 + 16384 * 3072 + 3072 * 8192) // 32 * 34
    # f32 activation rows: QKV in/out, rope q in/out and k, v in, attention q in, merge out + lse,
    # O in/out, gate/up in/out, down in/out
    acts = 8 * ((3072 + 5120) + (5120 + 3072) + 2 * 3072 + 24 + (3072 + 3072) + (3072 + 16384) + (8192 + 3072))
    assert bench.step_bytes(wl, _step(wl), kv) == weights + kv_read + kv_new + 4 * acts


def test_step_bytes_twelve_streams(dl):
    """Two commands: the weights twice, each stream's own keys once."""
    import bench
    import synth
    wl = bench.workload("3b-12")
    step = _step(wl)
    assert [c.n for c in step.commands] == [6, 6]
    lens = synth.twelve_stream_lengths(0)
    weights = (5120 * 3072 + 3072 * 3072 + 16384 * 3072 + 3072 * 8192) // 32 * 34
    kv = sum(l + 1 for l in lens) * 8 * 128 * 2 * 2 + 12 * 8 * 128 * 2 * 2
    acts = 12 * ((3072 + 5120) + (5120 + 3072) + 2 * 3072 + 24 + (3072 + 3072) + (3072 + 16384) + (8192 + 3072))
    assert bench.step_bytes(wl, step) == 2 * weights + kv + 4 * acts
