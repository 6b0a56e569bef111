"""The device id-list helpers against the input recipes, bit for bit.

qsa_fill_ids_decode / qsa_fill_ids_even write on the GPU the lists that the
workloads build on the host (decode windows of sink + local + own cell;
evenly spaced unique causal cells), so a run can make its ids without a host
upload.  Both sides are integer closed forms: the comparison is exact.
"""
import numpy as np
import pytest
import torch

from sparse_selected_attention_gb300 import qsa_fill_ids_decode, qsa_fill_ids_even
from sparse_selected_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _ids(T, W):
    return torch.full((T, W), 12345, dtype=torch.int32, device="cuda")  # every slot must be overwritten


@pytest.mark.parametrize("T,pos0,W,sink,local", [
    (1, 320, 384, 64, 256),       # the tiny decode window
    (8, 30000, 384, 64, 256),     # the MTP window
    (70, 0, 384, 64, 256),        # p below the sink, then below sink + local
    (5, 300, 64, 16, 40),
    (3, 10, 128, 0, 0),           # own cell only
])
def test_fill_ids_decode_matches_recipe(cuda_device, T, pos0, W, sink, local):
    ids = _ids(T, W)
    qsa_fill_ids_decode(ids, pos0, sink=sink, local=local)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), wl.decode_ids(T, pos0, W, sink=sink, local=local))


@pytest.mark.parametrize("T,pos0,W,select", [
    (1984, 0, 2048, 2048),        # the short prompt lists (every causal cell up to t = 2047)
    (1984, 30000, 2048, 2048),    # the long prompt lists
    (40, 31900, 2112, 2051),      # the three-cell last chunk
    (33, 4960, 448, 400),
    (3, 0, 64, 2),
])
def test_fill_ids_even_matches_recipe(cuda_device, T, pos0, W, select):
    ids = _ids(T, W)
    qsa_fill_ids_even(ids, pos0, select=select)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), wl.even_ids(T, pos0, W, select=select))
