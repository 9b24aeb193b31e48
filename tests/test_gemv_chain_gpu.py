"""dl_gemv_q8_chain (GEMV phases in one persistent launch) against the oracle (GPU)."""
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


def _pack(dl, blocks):
    return dl.dl_q8_pack(blocks.cuda(), blocks.shape[0], blocks.shape[1] * 32)


@pytest.mark.parametrize("shape", ["llama-3.2-1b", "llama-3.2-3b"])
@pytest.mark.parametrize("rows", [1, 2, 4, 8])
def test_chain_layer_projections(dl, shape, rows):
    """O, gate/up and down as the three phases of one launch, each within the GEMV bar."""
    blocks = layer_blocks(shape)
    names = ["wo", "wgu", "wdown"]
    Ws = [_pack(dl, blocks[n]) for n in names]
    xs = [synth.normal_f32(0, "chain/%s/%s/%d" % (shape, n, rows), (rows, blocks[n].shape[1] * 32)) for n in names]
    ys = [torch.full((rows, blocks[n].shape[0]), float("nan"), device="cuda") for n in names]
    sync = torch.zeros(4, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dl.dl_gemv_q8_chain(Ws, [x.cuda() for x in xs], ys, sync, status=status)
    torch.cuda.synchronize()
    assert dl.dl_status_read(status) == 0
    for n, x, y in zip(names, xs, ys):
        assert_gemv_close(y.cpu().numpy(), oracle.gemv_q8(blocks[n], x))


def test_chain_dependent_phases_and_reuse(dl):
    """Phase 1 reads phase 0's output; five launches in a row reuse the barrier words."""
    n = 3072
    b0 = synth.q8_0_blocks_from_normal(1, "chain/dep/0", n, n)
    b1 = synth.q8_0_blocks_from_normal(1, "chain/dep/1", n, n)
    W0, W1 = _pack(dl, b0), _pack(dl, b1)
    x = synth.normal_f32(1, "chain/dep/x", (8, n))
    y0_ref = oracle.gemv_q8(b0, x)
    y1_ref = oracle.gemv_q8(b1, y0_ref.astype(np.float32))
    sync = torch.zeros(4, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    xd = x.cuda()
    for _ in range(5):
        y0 = torch.full((8, n), float("nan"), device="cuda")
        y1 = torch.full((8, n), float("nan"), device="cuda")
        dl.dl_gemv_q8_chain([W0, W1], [xd, y0], [y0, y1], sync, status=status)
        torch.cuda.synchronize()
        assert dl.dl_status_read(status) == 0
        assert_gemv_close(y0.cpu().numpy(), y0_ref)
        # the second phase's input carries the first phase's rounding
        assert gemv_err(y1.cpu().numpy(), y1_ref) < 1e-2


@pytest.mark.parametrize("path", [1, 2])
def test_chain_both_inner_products(dl, path):
    rows = 2
    b = synth.q8_0_blocks_from_normal(2, "chain/path", 5120, 3072)
    W = _pack(dl, b)
    x = synth.normal_f32(2, "chain/path/x", (rows, 3072))
    y = torch.empty(rows, 5120, device="cuda")
    dl.dl_gemv_q8_chain([W], [x.cuda()], [y], torch.zeros(4, dtype=torch.int32, device="cuda"), path=path)
    torch.cuda.synchronize()
    assert_gemv_close(y.cpu().numpy(), oracle.gemv_q8(b, x))


def test_chain_refusals(dl):
    sync = torch.zeros(4, dtype=torch.int32, device="cuda")
    b = synth.q8_0_blocks_from_normal(3, "chain/refuse", 64, 512)
    W = _pack(dl, b)
    x = torch.zeros(2, 512, device="cuda")
    with pytest.raises(dl.DLError) as e:                       # n_in not a multiple of 1024
        dl.dl_gemv_q8_chain([W], [x], [torch.zeros(2, 64, device="cuda")], sync)
    assert e.value.code == dl.DL_E_SHAPE
    b2 = synth.q8_0_blocks_from_normal(3, "chain/refuse2", 1024, 1024)
    W2 = _pack(dl, b2)
    buf = torch.zeros(2, 1024, device="cuda")
    with pytest.raises(dl.DLError) as e:                       # output over its own input
        dl.dl_gemv_q8_chain([W2], [buf], [buf], sync)
    assert e.value.code == dl.DL_E_ARG
    with pytest.raises(dl.DLError) as e:                       # nine rows
        dl.dl_gemv_q8_chain([W2], [torch.zeros(9, 1024, device="cuda")], [torch.zeros(9, 1024, device="cuda")], sync)
    assert e.value.code == dl.DL_E_SHAPE
    with pytest.raises(dl.DLError) as e:                       # CUDA cores at three rows
        dl.dl_gemv_q8_chain([W2], [torch.zeros(3, 1024, device="cuda")], [torch.zeros(3, 1024, device="cuda")], sync,
                            path=1)
    assert e.value.code == dl.DL_E_SHAPE
