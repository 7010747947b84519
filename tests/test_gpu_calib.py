"""The data-movement reference kernels (include/spl_calib.h) on the GPU: in either chunk order
they move every value of every chunk (one partial wave, several waves with a partial last one),
and compute what the header says, checked against numpy's fp32 arithmetic on the host."""
import numpy as np
import pytest
import torch

import compressed_pseudo_gradient_gb300 as spl
from compressed_pseudo_gradient_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.mark.parametrize("persistent", [False, True])
@pytest.mark.parametrize("chunks", [1, 5, 1000, 12345])
def test_sender_moves_add_every_value(chunks, persistent):
    n = chunks * spl.CHUNK
    a = synth.laplace(n, 1.0, synth.generator(11 + chunks, DEV), DEV)
    b = synth.laplace(n, 1e-3, synth.generator(12 + chunks, DEV), DEV)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = spl.calib_moves(spl.CALIB_SENDER_MOVES, a, b, flags=flags, persistent=persistent)
    torch.cuda.synchronize()
    want = a.cpu().numpy() + b.cpu().numpy()          # fp32, rounded to nearest
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert int(flags.item()) == 0


@pytest.mark.parametrize("persistent", [False, True])
@pytest.mark.parametrize("chunks", [1, 7, 1000, 12345])
def test_receiver_moves_write_both_outputs(chunks, persistent):
    n = chunks * spl.CHUNK
    a = synth.laplace(n, 1.0, synth.generator(21 + chunks, DEV), DEV)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    neg, same = spl.calib_moves(spl.CALIB_RECEIVER_MOVES, a, flags=flags, persistent=persistent)
    torch.cuda.synchronize()
    ah = a.cpu().numpy()
    assert np.array_equal(neg.cpu().numpy().view(np.uint32), (-ah).view(np.uint32))
    assert np.array_equal(same.cpu().numpy().view(np.uint32), ah.view(np.uint32))
    assert int(flags.item()) == 0


def test_calib_rejects_partial_chunks_and_host_memory():
    a = torch.zeros(spl.CHUNK + 4, device=DEV)
    with pytest.raises(spl.SplError):
        spl.calib_moves(spl.CALIB_SENDER_MOVES, a, torch.zeros_like(a))
    h = torch.zeros(spl.CHUNK).pin_memory()          # the bulk copies read device memory only
    d1 = torch.zeros(spl.CHUNK, device=DEV)
    d2 = torch.zeros(spl.CHUNK, device=DEV)
    st = spl.library().spl_calib_moves(spl.CALIB_SENDER_MOVES, 0, h.data_ptr(), d1.data_ptr(),
                                       d2.data_ptr(), None, spl.CHUNK, None, None)
    assert st == 1                                    # SPL_ERR_INVALID_ARG
