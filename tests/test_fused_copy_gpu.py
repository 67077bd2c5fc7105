"""FP8 activation copies made by the epilogue of the layer before.

Inside dl_decode_stream, an FP8 layer whose x is exactly the whole y of the
layer just before it -- a plain linear (no SwiGLU, no argmax) with the same M --
gets its exact f16 copy from that layer's epilogue instead of a prep kernel:
every output tile of the producer is one 128-column K block of the copy.  The
copy is the same bytes the prep kernel writes, so every output must equal the
same chain run through single calls, bit for bit; with a workspace too small
for the copy regions the layers fall back to their own prep kernels.
"""
import pytest
import torch

import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs

pytestmark = pytest.mark.gpu

BF, F8 = inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128

# (dtype, N, K, bias, act); layer i > 0 reads the y of layer i - 1.  Fed by
# the epilogue before: 1 (bf16 producer), 2 and 3 (FP8 producers), 5 (bf16
# producer, SwiGLU consumer).  Layer 6 follows a SwiGLU layer: own prep.
CHAIN = [(BF, 2048, 512, True, 0), (F8, 1024, 2048, False, 0), (F8, 1536, 1024, True, 0),
         (F8, 512, 1536, False, 0), (BF, 1024, 512, False, 0), (F8, 1024, 1024, True, 1),
         (F8, 256, 512, False, 0)]
FED = 4


def _lib(dt):
    return dl.BF16 if dt == BF else dl.FP8_B128


def chain(dev, specs, M, seed):
    """The layers with their weights; x of layer 0 seeded, later x = earlier y."""
    layers, prev = [], None
    for i, (dt, N, K, bias, act) in enumerate(specs):
        L = inputs.make_layer(dt, M, N, K, bias=bias, config_id=seed, layer_idx=i).to(dev)
        x = L.x if prev is None else prev
        y = torch.empty((M, N // 2 if act == 1 else N), dtype=torch.bfloat16, device=dev)
        layers.append(dl.Layer(_lib(dt), x, L.w, y, L.scales, L.bias, act=act))
        prev = y
    return layers


def single_calls(layers, ws):
    """The same chain, one call per layer (each FP8 layer with its own prep)."""
    out, x = [], layers[0].x
    for L in layers:
        if L.act == 1:
            y = dl.linear_swiglu(x, L.w, L.scales, L.bias, workspace=ws)
        elif L.dtype == dl.BF16:
            y = dl.linear_bf16(x, L.w, L.bias, workspace=ws)
        else:
            y = dl.linear_fp8_block128(x, L.w, L.scales, L.bias, workspace=ws)
        out.append(y)
        x = y
    torch.cuda.synchronize()
    return out


def run(layers, ws, use_graph, st):
    for L in layers:
        L.y.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        dl.decode_stream(layers, ws, use_graph=use_graph, stream=st)
    st.synchronize()
    return [L.y.clone() for L in layers]


@pytest.mark.parametrize("max_ctas", [0, 8])
@pytest.mark.parametrize("M", [1, 6, 16])
def test_epilogue_copies_match_single_calls(cuda_device, M, max_ctas):
    """max_ctas = 8: long segments, so many producer tiles are covered whole by
    one segment (finished through the CTA's own slots); the default grid splits
    most tiles (finished by the fix-up)."""
    layers = chain(cuda_device, CHAIN, M, 120)
    n = len(layers)
    f8 = sum(L.dtype == dl.FP8_B128 for L in layers)
    small = dl.Workspace.for_shapes([L.shape() for L in layers], cuda_device)
    big = dl.Workspace.for_stream(layers)
    assert big.nbytes > small.nbytes
    assert dl.decode_stream_launches(layers, small) == n + f8
    assert dl.decode_stream_launches(layers, big) == n + f8 - FED
    dl.set_override(0, 0, max_ctas)
    try:
        want = single_calls(layers, small)
        st = torch.cuda.Stream()
        for ws in (big, small):
            for use_graph in (False, True, True):
                got = run(layers, ws, use_graph, st)
                for i in range(n):
                    assert torch.equal(got[i], want[i]), (ws.nbytes, use_graph, i)
            assert torch.all(ws.tensor[:dl.WORKSPACE_ZERO_BYTES] == 0)
    finally:
        dl.set_override(0, 0, 0)
        dl.graph_cache_clear()
    assert dl.device_status() == 0


def test_epilogue_copy_follows_new_inputs(cuda_device):
    """One workspace, the same chain with a new x each step: every block of
    every fed copy is rewritten by each call (nothing read from a previous
    step), in both replay modes."""
    M = 4
    layers = chain(cuda_device, CHAIN[:4], M, 121)
    ws = dl.Workspace.for_stream(layers)
    st = torch.cuda.Stream()
    g = torch.Generator(device="cpu").manual_seed(7)
    try:
        for step in range(3):
            layers[0].x.copy_(torch.randn(layers[0].x.shape, generator=g).to(torch.bfloat16))
            want = single_calls(layers, ws)
            for use_graph in (False, True):
                got = run(layers, ws, use_graph, st)
                for i in range(len(layers)):
                    assert torch.equal(got[i], want[i]), (step, use_graph, i)
    finally:
        dl.graph_cache_clear()
    assert dl.device_status() == 0


def test_not_fed_when_x_is_not_the_whole_previous_y(cuda_device):
    """A slice of the previous y, or a y from two layers back, keeps its prep."""
    dev = cuda_device
    M = 2
    a = inputs.make_layer(BF, M, 2048, 512, bias=False, config_id=122, layer_idx=0).to(dev)
    b = inputs.make_layer(F8, M, 1024, 1024, bias=False, config_id=122, layer_idx=1).to(dev)
    c = inputs.make_layer(F8, M, 512, 2048, bias=False, config_id=122, layer_idx=2).to(dev)
    ya = torch.empty((M, 2048), dtype=torch.bfloat16, device=dev)
    yb = torch.empty((M, 1024), dtype=torch.bfloat16, device=dev)
    yc = torch.empty((M, 512), dtype=torch.bfloat16, device=dev)
    yab = torch.randn((M, 1024), generator=torch.Generator().manual_seed(5)).to(dev, torch.bfloat16)
    layers = [dl.Layer(dl.BF16, a.x, a.w, ya),
              dl.Layer(dl.FP8_B128, yab, b.w, yb, b.scales),      # not the previous y
              dl.Layer(dl.FP8_B128, ya, c.w, yc, c.scales)]       # y of two layers back
    ws = dl.Workspace.for_stream(layers)
    assert dl.decode_stream_launches(layers, ws) == 3 + 2
    st = torch.cuda.Stream()
    got = run(layers, ws, True, st)
    y0 = dl.linear_bf16(a.x, a.w, workspace=ws)
    want = [y0, dl.linear_fp8_block128(yab, b.w, b.scales, workspace=ws),
            dl.linear_fp8_block128(y0, c.w, c.scales, workspace=ws)]
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(got[i], want[i]), i
    dl.graph_cache_clear()
    assert dl.device_status() == 0
