"""dl_gemv_q8 against the oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.workloads import assert_gemv_close, gemv_err, layer_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import row_decode_step_gb300 as m
    from row_decode_step_gb300 import _build
    _build.build()
    m.lib()
    return m


def _run(dl, blocks, n_out, n_in, x, path=0):
    W = dl.dl_q8_pack(blocks.cuda(), n_out, n_in)
    y = dl.dl_gemv_q8(W, x.cuda(), path=path)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("n_out,n_in,rows", [
    (37, 96, 1), (37, 96, 3), (256, 256, 1), (512, 256, 8), (200, 160, 9),
    (64, 1024, 12), (48, 128, 16), (16, 32, 5), (300, 2080, 7), (1000, 4096, 2),
])
def test_gemv_shapes(dl, n_out, n_in, rows):
    """Several tiles, ragged row tiles and ragged k groups, 1..16 rows (tiled past eight)."""
    blocks = synth.q8_0_blocks_from_normal(1, "gemv/%d/%d" % (n_out, n_in), n_out, n_in)
    x = synth.normal_f32(1, "gemv/x/%d" % n_in, (rows, n_in))
    y = _run(dl, blocks, n_out, n_in, x)
    assert_gemv_close(y, oracle.gemv_q8(blocks, x))


@pytest.mark.parametrize("shape", ["llama-3.2-1b", "llama-3.2-3b"])
@pytest.mark.parametrize("rows", [1, 2, 4, 8, 12])
def test_gemv_full_layer(dl, shape, rows):
    """Every projection of the full-size layer, the same launch shapes the bench times."""
    for name, blocks in layer_blocks(shape).items():
        n_out, n_in = blocks.shape[0], blocks.shape[1] * 32
        x = synth.normal_f32(0, "%s/x/%s/%d" % (shape, name, rows), (rows, n_in))
        y = _run(dl, blocks, n_out, n_in, x)
        ref = oracle.gemv_q8(blocks, x)
        assert_gemv_close(y, ref)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("rows", [1, 2])
def test_gemv_both_inner_products(dl, path, rows):
    """The CUDA-core and tensor-core inner products each meet the bar on the 3B QKV shape."""
    blocks = layer_blocks("llama-3.2-3b")["wqkv"]
    n_out, n_in = blocks.shape[0], blocks.shape[1] * 32
    x = synth.normal_f32(0, "paths/x/%d" % rows, (rows, n_in))
    assert_gemv_close(_run(dl, blocks, n_out, n_in, x, path=path), oracle.gemv_q8(blocks, x))


def test_gemv_tensor_path_wide_range(dl):
    """Activation blocks spanning 1e-6 .. 1e6 (past the f16 range) keep the bar on the tensor path."""
    n_out, n_in, rows = 64, 512, 3
    blocks = synth.q8_0_blocks_from_normal(6, "gemv/range", n_out, n_in)
    x = synth.normal_f32(6, "gemv/range/x", (rows, n_in))
    scale = torch.logspace(-6, 6, n_in // 32).repeat_interleave(32)
    x = x * scale
    assert_gemv_close(_run(dl, blocks, n_out, n_in, x, path=2), oracle.gemv_q8(blocks, x))


def test_gemv_cuda_core_path_refuses_wide_commands(dl):
    blocks = synth.q8_0_blocks_from_normal(7, "gemv/wide", 32, 64)
    W = dl.dl_q8_pack(blocks.cuda(), 32, 64)
    with pytest.raises(dl.DLError) as e:
        dl.dl_gemv_q8(W, torch.zeros(3, 64, device="cuda"), path=1)
    assert e.value.code == dl.DL_E_SHAPE


def test_gemv_rows_match_single_rows(dl):
    """Rows stepped together agree with the same rows stepped one at a time (tails of 2, 9, 16).

    One or two rows take the CUDA-core inner product (f32 activations and sums); a command
    of more rows takes the tensor-core path, whose activations enter as an f16 hi + lo pair
    after a power-of-two scale per k-tile (about 22 significant bits) and whose products
    are summed in f32.  Both are close to an f32 dot product, so they agree with each other
    at 3e-4 of the output scale (summation order and the lo term's rounding), well inside
    the 1e-3 bar each of them meets against the oracle.  A 9-row command is stepped as
    balanced groups (5 + 4), a 16-row one as 8 + 8.
    """
    n_out, n_in = 384, 1024
    blocks = synth.q8_0_blocks_from_normal(2, "gemv/tail", n_out, n_in)
    W = dl.dl_q8_pack(blocks.cuda(), n_out, n_in)
    x = synth.normal_f32(2, "gemv/tail/x", (16, n_in)).cuda()
    for n in (2, 9, 16):
        y = dl.dl_gemv_q8(W, x[:n])
        ys = torch.cat([dl.dl_gemv_q8(W, x[r:r + 1]) for r in range(n)])
        torch.cuda.synchronize()
        assert gemv_err(y.cpu().numpy(), ys.cpu().numpy().astype(np.float64)) < 3e-4


@pytest.mark.parametrize("path", [1, 2])
def test_gemv_row_independent_of_other_rows(dl, path):
    """A row's outputs do not depend on the other rows of its command: bit-identical when they change."""
    n_out, n_in = 384, 1024
    rows = 2 if path == 1 else 9
    blocks = synth.q8_0_blocks_from_normal(2, "gemv/indep", n_out, n_in)
    W = dl.dl_q8_pack(blocks.cuda(), n_out, n_in)
    x = synth.normal_f32(2, "gemv/indep/x", (rows, n_in)).cuda()
    y0 = dl.dl_gemv_q8(W, x, path=path)
    x2 = x.clone()
    x2[1:] = 1e3 * synth.normal_f32(3, "gemv/indep/x2", (rows - 1, n_in)).cuda()
    y1 = dl.dl_gemv_q8(W, x2, path=path)
    torch.cuda.synchronize()
    assert torch.equal(y0[0], y1[0])
    assert not torch.equal(y0[1], y1[1])


def test_gemv_strides_and_poisoned_padding(dl):
    """Strided rows read only their n_in inputs and write only their n_out outputs."""
    n_out, n_in, rows = 80, 192, 5
    blocks = synth.q8_0_blocks_from_normal(3, "gemv/stride", n_out, n_in)
    W = dl.dl_q8_pack(blocks.cuda(), n_out, n_in)
    xs = torch.full((rows, n_in + 64), float("nan"), device="cuda")
    x = synth.normal_f32(3, "gemv/stride/x", (rows, n_in))
    xs[:, :n_in] = x.cuda()
    ys = torch.full((rows, n_out + 48), -7.0, device="cuda")
    dl.dl_gemv_q8(W, xs[:, :n_in], ys[:, :n_out])
    torch.cuda.synchronize()
    out = ys.cpu().numpy()
    assert np.all(out[:, n_out:] == -7.0)
    assert_gemv_close(out[:, :n_out], oracle.gemv_q8(blocks, x))


def test_gemv_control_detects_planted_error(dl):
    """Teeth: the comparison fails when the oracle is handed one changed weight byte."""
    n_out, n_in = 64, 256
    blocks = synth.q8_0_blocks_from_normal(4, "gemv/teeth", n_out, n_in)
    x = synth.normal_f32(4, "gemv/teeth/x", (2, n_in))
    y = _run(dl, blocks, n_out, n_in, x)
    bad = blocks.clone()
    bad[5, 3, 7] = (int(bad[5, 3, 7]) + 50) % 256
    assert gemv_err(y, oracle.gemv_q8(bad, x)) > 1e-3
    assert_gemv_close(y, oracle.gemv_q8(blocks, x))


def test_gemv_refuses_misaligned_x(dl):
    n_out, n_in = 32, 64
    blocks = synth.q8_0_blocks_from_normal(5, "gemv/align", n_out, n_in)
    W = dl.dl_q8_pack(blocks.cuda(), n_out, n_in)
    buf = torch.zeros(1, n_in + 1, device="cuda")
    with pytest.raises(dl.DLError) as e:
        dl.dl_gemv_q8(W, buf[:, 1:])
    assert e.value.code == dl.DL_E_ALIGN
