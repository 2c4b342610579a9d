"""Failure detection without a GPU fault: a bounded device wait is made to
run out and reports through the device status word, and the context stays
usable.  The one-launch scale + quantize kernel's grid barrier counts block
arrivals in its workspace; with the arrival word preset so that the blocks'
arrivals wrap past the grid size, the barrier can never complete (a flag
nothing sets).  Every block's wait gives up after its time limit (~2 s),
records NVFP4_ERR_TIMEOUT * 100 + site and returns without quantizing."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from _gpu import assert_same_quant, dev, oracle_quant

pytestmark = pytest.mark.gpu

ARRIVE_WORD = 32      # the grid barrier's arrival counter in the workspace
SITE_RESIDENT = 7     # wait site of the resident fused kernel
SITE_STREAM = 26      # wait site of the streaming fused kernel's grid barrier


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_device_gb300 as m
    return m


def test_grid_barrier_timeout_reports_status(nv):
    rows, cols = 130, 256                      # 65 blocks of two rows, all resident
    x = synthetic.normal(np.random.default_rng(31), (rows, cols))
    xd = dev(x)
    t = nv.NVFP4Tensor.empty(rows, cols)
    assert nv.device_status() == 0
    ws = nv.workspace(256)
    ws.view(torch.int32)[ARRIVE_WORD] = -(rows // 2)   # 2^32 - 65: 65 arrivals wrap to 0
    nv.nvfp4_scale_quantize(xd, t, ws)
    torch.cuda.synchronize()                   # returns: every wait is bounded
    assert nv.device_status(clear=True) == nv.NVFP4_ERR_TIMEOUT * 100 + SITE_RESIDENT
    assert nv.device_status() == 0
    # the context is still usable: a zeroed workspace gives the exact result
    nv.nvfp4_scale_quantize(xd, t, nv.workspace(256))
    c, s, g = oracle_quant(x)
    assert_same_quant(t, c, s, g, "after timeout")
    assert nv.device_status() == 0


def test_stream_grid_barrier_timeout_reports_status(nv):
    """The streaming variant (more rows than the resident blocks hold; one
    block per SM): its grid barrier runs out the same way, and the block
    returns with no bulk copy in flight (every row of pass 1 was waited
    for), so the next call on a zeroed workspace is exact."""
    rows, cols = 1300, 256
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    x = synthetic.normal(np.random.default_rng(37), (rows, cols))
    xd = dev(x)
    t = nv.NVFP4Tensor.empty(rows, cols)
    assert nv.device_status() == 0
    ws = nv.workspace(256)
    ws.view(torch.int32)[ARRIVE_WORD] = -(nsm // 2)   # half the arrivals wrap to 0
    nv.nvfp4_scale_quantize(xd, t, ws)
    torch.cuda.synchronize()
    assert nv.device_status(clear=True) == nv.NVFP4_ERR_TIMEOUT * 100 + SITE_STREAM
    assert nv.device_status() == 0
    nv.nvfp4_scale_quantize(xd, t, nv.workspace(256))
    c, s, g = oracle_quant(x)
    assert_same_quant(t, c, s, g, "after timeout (streaming)")
    assert nv.device_status() == 0
