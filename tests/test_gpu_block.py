"""GPU tests of the layer-block launch set: the host pipeline (copies of
neighbouring ubatches overlapped with compute, two device buffer pairs,
graphs replayed on alternate buffers) gives bit for bit the outputs of the
plain, stream-ordered forward on the same ubatches."""
import numpy as np
import pytest
import torch

import synthetic
from _gpu import dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_device_gb300 as m
    return m


def make_block(nv, T, H=256, I=512, Nqkv=512):
    from nvfp4_block_scaled_device_gb300.block import PrefillBlock
    ws = nv.workspace(256)
    W = {}
    for j, (k, rows, cols) in enumerate((("qkv", Nqkv, H), ("o", H, H), ("gate", I, H), ("up", I, H),
                                         ("down", H, I))):
        W[k] = nv.quantize_new(dev(synthetic.weight(70 + j, rows, cols)), ws)
    return PrefillBlock(T, W, dev(synthetic.norm_weight(80, H)), dev(synthetic.norm_weight(81, H)))


@pytest.mark.parametrize("T", [130, 1])
def test_host_pipeline_matches_forward(nv, T):
    from nvfp4_block_scaled_device_gb300.block import HostPipeline
    blk = make_block(nv, T)
    xs = [synthetic.activations(T, seed=90 + i, h=256) for i in range(5)]
    stream = torch.cuda.Stream()
    out = torch.empty((T, 256), dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        blk.calibrate(dev(xs[0]), out, stream)
    stream.synchronize()
    # the plain forward, one ubatch at a time
    ref = []
    for xb in xs:
        xd = dev(xb)
        with torch.cuda.stream(stream):
            blk.forward(xd, out, stream)
        stream.synchronize()
        ref.append(host(out).copy())
    # the pipeline, all ubatches in flight
    pipe = HostPipeline(blk, stream)
    x_host = [torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16).pin_memory() for xb in xs]
    o_host = [torch.empty((T, 256), dtype=torch.bfloat16).pin_memory() for _ in xs]
    for xh, oh in zip(x_host, o_host):
        pipe.submit(xh, oh)
    pipe.wait()
    assert nv.device_status() == 0
    for i, oh in enumerate(o_host):
        got = oh.view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, ref[i]), f"ubatch {i}"
    assert not np.array_equal(ref[0], ref[1])


def test_stacked_layers_one_graph(nv):
    """The long-prefill shape in miniature: ubatches through stacked layers,
    each with its own seeded weights and residual adds in bf16, captured as
    ONE CUDA graph (capture fails on any host synchronisation, so the launch
    set has none per layer) and replayed; outputs equal the eager,
    layer-by-layer run bit for bit, and the layers really differ."""
    from nvfp4_block_scaled_device_gb300.block import PrefillBlock
    L, U, T, H, I, Nqkv = 3, 4, 64, 256, 512, 512
    ws = nv.workspace(256)
    blocks = []
    for layer in range(L):
        W = {}
        for j, (k, rows, cols) in enumerate((("qkv", Nqkv, H), ("o", H, H), ("gate", I, H), ("up", I, H),
                                             ("down", H, I))):
            W[k] = nv.quantize_new(dev(synthetic.weight(100 + 10 * layer + j, rows, cols)), ws)
        blocks.append(PrefillBlock(T, W, dev(synthetic.norm_weight(200 + layer, H)),
                                   dev(synthetic.norm_weight(300 + layer, H))))
    stream = torch.cuda.Stream()
    xs = [dev(synthetic.activations(T, seed=400 + u, h=H)) for u in range(U)]
    bufs = [[torch.empty((T, H), dtype=torch.bfloat16, device="cuda") for _ in range(L)] for _ in range(U)]
    with torch.cuda.stream(stream):
        for b in blocks:
            b.calibrate(xs[0], bufs[0][0], stream)

        def run_all():
            for u in range(U):
                inp = xs[u]
                for layer in range(L):
                    blocks[layer].forward(inp, bufs[u][layer], stream)
                    inp = bufs[u][layer]
        run_all()
    stream.synchronize()
    eager = [[host(t).copy() for t in row] for row in bufs]
    for row in bufs:
        for t in row:
            t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run_all()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    assert nv.device_status() == 0
    for u in range(U):
        for layer in range(L):
            assert np.array_equal(host(bufs[u][layer]), eager[u][layer]), (u, layer)
    assert not np.array_equal(eager[0][0], eager[0][1])
