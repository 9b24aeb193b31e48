"""dl_gemv_f16w (the f16-weight reference lane) against the oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import assert_gemv_close, gemv_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _run(dl, w, x, path=0):
    W = dl.dl_f16w_pack(w.cuda())
    y = dl.dl_gemv_f16w(W, x.cuda(), path=path)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("n_out,n_in,rows", [
    (37, 96, 1), (37, 96, 3), (256, 256, 1), (512, 256, 8), (200, 160, 9),
    (64, 1024, 12), (16, 32, 5), (300, 2080, 7), (1000, 4096, 2), (130, 8192, 4),
])
def test_f16w_shapes(dl, n_out, n_in, rows):
    """Several tiles, ragged row tiles, a short last K-slice, 1..12 rows (tiled past eight)."""
    w = synth.f16_weights_from_normal(1, "f16w/%d/%d" % (n_out, n_in), n_out, n_in)
    x = synth.normal_f32(1, "f16w/x/%d" % n_in, (rows, n_in))
    assert_gemv_close(_run(dl, w, x), oracle.gemv_f16w(w, x))


@pytest.mark.parametrize("n_out,n_in", [(5120, 3072), (16384, 3072), (3072, 8192)])
@pytest.mark.parametrize("rows", [1, 8])
def test_f16w_full_size(dl, n_out, n_in, rows):
    """The 3B-shaped QKV, gate/up and down projections as f16 weights, in the launch shapes the
    bench times."""
    w = synth.f16_weights_from_normal(0, "f16w/full/%d/%d" % (n_out, n_in), n_out, n_in, device="cuda")
    x = synth.normal_f32(0, "f16w/full/x/%d/%d" % (n_in, rows), (rows, n_in))
    assert_gemv_close(_run(dl, w, x), oracle.gemv_f16w(w.cpu(), x))


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("rows", [1, 2])
def test_f16w_both_inner_products(dl, path, rows):
    """The CUDA-core and tensor-core inner products each meet the bar."""
    w = synth.f16_weights_from_normal(2, "f16w/paths", 1024, 3072)
    x = synth.normal_f32(2, "f16w/paths/x/%d" % rows, (rows, 3072))
    assert_gemv_close(_run(dl, w, x, path=path), oracle.gemv_f16w(w, x))


def test_f16w_extreme_weights_and_wide_activations(dl):
    """Weights at the ends of the f16 range (65504, subnormals, -0) and activations spanning
    1e-6 .. 1e6 keep the bar on both inner products."""
    n_out, n_in, rows = 64, 512, 3
    w = synth.f16_weights_from_normal(6, "f16w/range", n_out, n_in)
    bits = w.view(torch.int16)
    bits[0, :64] = 0x7BFF                         # 65504
    bits[1, 64:128] = 0x0001                      # 2^-24
    bits[2, 128:192] = -32768                     # -0 (0x8000)
    bits[3, :] = 0x03FF                           # largest subnormal
    x = synth.normal_f32(6, "f16w/range/x", (rows, n_in))
    x = x * torch.logspace(-6, 6, n_in // 32).repeat_interleave(32)
    ref = oracle.gemv_f16w(w, x)
    assert_gemv_close(_run(dl, w, x, path=2), ref)
    assert_gemv_close(_run(dl, w, x[:2], path=1), ref[:2])


@pytest.mark.parametrize("path", [1, 2])
def test_f16w_row_independent_of_other_rows(dl, path):
    """A row's outputs do not depend on the other rows of its command: bit-identical when they change."""
    n_out, n_in = 384, 1024
    rows = 2 if path == 1 else 9
    w = synth.f16_weights_from_normal(2, "f16w/indep", n_out, n_in)
    W = dl.dl_f16w_pack(w.cuda())
    x = synth.normal_f32(2, "f16w/indep/x", (rows, n_in)).cuda()
    y0 = dl.dl_gemv_f16w(W, x, path=path)
    x2 = x.clone()
    x2[1:] = 1e3 * synth.normal_f32(3, "f16w/indep/x2", (rows - 1, n_in)).cuda()
    y1 = dl.dl_gemv_f16w(W, x2, path=path)
    torch.cuda.synchronize()
    assert torch.equal(y0[0], y1[0])
    assert not torch.equal(y0[1], y1[1])


def test_f16w_strides_and_poisoned_padding(dl):
    """Strided rows read only their n_in inputs and write only their n_out outputs."""
    n_out, n_in, rows = 80, 192, 5
    w = synth.f16_weights_from_normal(3, "f16w/stride", n_out, n_in)
    W = dl.dl_f16w_pack(w.cuda())
    xs = torch.full((rows, n_in + 64), float("nan"), device="cuda")
    x = synth.normal_f32(3, "f16w/stride/x", (rows, n_in))
    xs[:, :n_in] = x.cuda()
    ys = torch.full((rows, n_out + 48), -7.0, device="cuda")
    dl.dl_gemv_f16w(W, xs[:, :n_in], ys[:, :n_out])
    torch.cuda.synchronize()
    out = ys.cpu().numpy()
    assert np.all(out[:, n_out:] == -7.0)
    assert_gemv_close(out[:, :n_out], oracle.gemv_f16w(w, x))


def test_f16w_control_detects_planted_error(dl):
    """Teeth: the comparison fails when the oracle is handed one changed weight."""
    n_out, n_in = 64, 256
    w = synth.f16_weights_from_normal(4, "f16w/teeth", n_out, n_in)
    x = synth.normal_f32(4, "f16w/teeth/x", (2, n_in))
    y = _run(dl, w, x)
    bad = w.clone()
    bad[5, 103] = 4.0
    assert gemv_err(y, oracle.gemv_f16w(bad, x)) > 1e-3
    assert_gemv_close(y, oracle.gemv_f16w(w, x))


def test_f16w_refusals(dl):
    """Misaligned activations, a CUDA-core command of 3 rows and a width that is not a multiple of
    32 are refused before anything launches."""
    w = synth.f16_weights_from_normal(5, "f16w/refuse", 32, 64).cuda()
    W = dl.dl_f16w_pack(w)
    buf = torch.zeros(1, 65, device="cuda")
    with pytest.raises(dl.DLError) as e:
        dl.dl_gemv_f16w(W, buf[:, 1:])
    assert e.value.code == dl.DL_E_ALIGN
    with pytest.raises(dl.DLError) as e:
        dl.dl_gemv_f16w(W, torch.zeros(3, 64, device="cuda"), path=1)
    assert e.value.code == dl.DL_E_SHAPE
    with pytest.raises(dl.DLError) as e:
        dl.dl_f16w_pack(torch.zeros(4, 48, dtype=torch.float16, device="cuda"))
    assert e.value.code == dl.DL_E_SHAPE
