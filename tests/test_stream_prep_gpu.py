"""FP8 activation copies made up front inside dl_decode_stream.

An FP8 layer whose x no earlier layer of the list writes has its f16 copy
made ahead (when the workspace has room, dl_decode_stream_workspace_bytes):
layer 0's just before it, the later ones' in batches, one launch right after
every 16th layer (layer 16k) holding the copies of layers 16k+1 .. 16k+16 and
copying while layer 16k runs.  A layer fed by an earlier layer keeps its own
prep kernel.  Either way the outputs must equal the single calls' bit
for bit (the copy is the same bytes, made earlier).
"""
import pytest
import torch

import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs

pytestmark = pytest.mark.gpu

BF, F8 = inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128


def _lib(dt):
    return dl.BF16 if dt == BF else dl.FP8_B128


def independent_layers(dev, specs, M, seed):
    """Layers with their own (seeded) x each."""
    out = []
    for i, (dt, N, K, bias) in enumerate(specs):
        L = inputs.make_layer(dt, M, N, K, bias=bias, config_id=seed, layer_idx=i).to(dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        out.append(dl.Layer(_lib(dt), L.x, L.w, y, L.scales, L.bias))
    return out


def singles(layers, ws):
    want = []
    for L in layers:
        y = torch.empty_like(L.y)
        if L.dtype == dl.BF16:
            dl.linear_bf16(L.x, L.w, L.bias, out=y, workspace=ws)
        else:
            dl.linear_fp8_block128(L.x, L.w, L.scales, L.bias, out=y, workspace=ws)
        want.append(y)
    torch.cuda.synchronize()
    return want


def run(layers, ws, use_graph, st):
    for L in layers:
        L.y.zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        dl.decode_stream(layers, ws, use_graph=use_graph, stream=st)
    st.synchronize()
    return [L.y.clone() for L in layers]


@pytest.mark.parametrize("M", [1, 6, 16])
def test_up_front_copies_match_per_layer_prep_and_single_calls(cuda_device, M):
    specs = [(F8, 1024, 2048, True), (BF, 768, 1024, False), (F8, 512, 4096, False),
             (F8, 2048, 1024, True)]
    layers = independent_layers(cuda_device, specs, M, 95)
    small = dl.Workspace.for_shapes([L.shape() for L in layers], cuda_device)
    big = dl.Workspace.for_stream(layers)
    assert big.nbytes > small.nbytes
    n, f8 = len(layers), sum(L.dtype == dl.FP8_B128 for L in layers)
    assert dl.decode_stream_launches(layers, small) == n + f8        # a prep before each FP8 layer
    # layer 0's copy before it, the other FP8 copies in one launch after it
    assert dl.decode_stream_launches(layers, big) == 2 + n
    want = singles(layers, small)
    st = torch.cuda.Stream()
    for ws in (small, big):
        for use_graph in (False, True, True):
            got = run(layers, ws, use_graph, st)
            for i in range(n):
                assert torch.equal(got[i], want[i]), (ws.nbytes, use_graph, i)
        assert torch.all(ws.tensor[:dl.WORKSPACE_ZERO_BYTES] == 0)
    assert dl.device_status() == 0
    dl.graph_cache_clear()


def test_layers_fed_by_earlier_layers_keep_their_prep(cuda_device):
    """x = an earlier y is not copied up front: the whole y of the layer just
    before gets its copy from that layer's epilogue, a slice its own prep."""
    dev = cuda_device
    M = 1
    a = inputs.make_layer(F8, M, 2048, 1024, bias=False, config_id=96, layer_idx=0).to(dev)
    b = inputs.make_layer(F8, M, 1024, 2048, bias=True, config_id=96, layer_idx=1).to(dev)
    c = inputs.make_layer(F8, M, 640, 1024, bias=False, config_id=96, layer_idx=2).to(dev)
    d = inputs.make_layer(F8, M, 512, 1024, bias=False, config_id=96, layer_idx=3).to(dev)
    ya = torch.empty((M, 2048), dtype=torch.bfloat16, device=dev)
    yb = torch.empty((M, 1024), dtype=torch.bfloat16, device=dev)
    yc = torch.empty((M, 640), dtype=torch.bfloat16, device=dev)
    yd = torch.empty((M, 512), dtype=torch.bfloat16, device=dev)
    layers = [dl.Layer(dl.FP8_B128, a.x, a.w, ya, a.scales),
              dl.Layer(dl.FP8_B128, ya, b.w, yb, b.scales, b.bias),          # all of an earlier y
              dl.Layer(dl.FP8_B128, ya[:, 512:1536], c.w, yc, c.scales),     # part of an earlier y
              dl.Layer(dl.FP8_B128, d.x, d.w, yd, d.scales)]                 # ready at the start
    ws = dl.Workspace.for_stream(layers)
    # layer 0's copy, layer 3's copy (after layer 0), 1 from layer 0's epilogue,
    # 2 with its own prep
    assert dl.decode_stream_launches(layers, ws) == 2 + 4 + 1
    st = torch.cuda.Stream()
    got = run(layers, ws, True, st)
    # the same chain through single calls
    want = []
    y0 = dl.linear_fp8_block128(a.x, a.w, a.scales, workspace=ws)
    want.append(y0)
    want.append(dl.linear_fp8_block128(y0, b.w, b.scales, b.bias, workspace=ws))
    want.append(dl.linear_fp8_block128(y0[:, 512:1536].contiguous(), c.w, c.scales, workspace=ws))
    want.append(dl.linear_fp8_block128(d.x, d.w, d.scales, workspace=ws))
    torch.cuda.synchronize()
    for i in range(4):
        assert torch.equal(got[i], want[i]), i
    assert dl.device_status() == 0
    dl.graph_cache_clear()


def test_copies_made_ahead_in_windows_of_16(cuda_device):
    """70 small FP8 layers with their own x: layer 0's copy alone before it, then
    the copies of layers 16k+1 .. 16k+16 in one launch right after layer 16k
    (five launches), no per-layer prep; with a workspace that holds no copy
    region every layer has its own prep."""
    specs = [(F8, 128 * (1 + i % 3), 128 * (1 + i % 4), i % 2 == 0) for i in range(70)]
    layers = independent_layers(cuda_device, specs, 2, 97)
    ws = dl.Workspace.for_stream(layers)
    assert dl.decode_stream_launches(layers, ws) == 1 + 5 + 70
    small = dl.Workspace.for_shapes([L.shape() for L in layers], cuda_device)
    assert dl.decode_stream_launches(layers, small) == 70 + 70
    want = singles(layers, ws)
    st = torch.cuda.Stream()
    got = run(layers, ws, True, st)
    for i in range(70):
        assert torch.equal(got[i], want[i]), i
    assert dl.device_status() == 0
    dl.graph_cache_clear()


def test_bf16_first_layer_puts_the_copies_before_it(cuda_device):
    """Layer 0 is bf16: the FP8 copies go in one launch before it (waiting for the
    kernels before the stream first)."""
    specs = [(BF, 1024, 2048, False), (F8, 512, 4096, True), (F8, 2048, 1024, False)]
    layers = independent_layers(cuda_device, specs, 6, 98)
    ws = dl.Workspace.for_stream(layers)
    assert dl.decode_stream_launches(layers, ws) == 1 + 3
    want = singles(layers, ws)
    st = torch.cuda.Stream()
    for use_graph in (False, True, True):
        got = run(layers, ws, use_graph, st)
        for i in range(3):
            assert torch.equal(got[i], want[i]), (use_graph, i)
    assert dl.device_status() == 0
    dl.graph_cache_clear()


def test_one_later_copy_covers_every_block(cuda_device):
    """Exactly one FP8 layer after layer 0 copied ahead, with more (K block,
    token slot) pairs (96 x 16) than the copy launch has warps (at most 8 per
    SM): every block of its copy must be made by this call.  The workspace
    first serves a list whose layer 1 has the same region but another x, so
    a block left out would be read stale and give wrong outputs."""
    M = 4
    shapes = [(F8, 256, 1024, False), (F8, 256, 12288, True), (F8, 256, 1024, False)]
    first = independent_layers(cuda_device, shapes, M, 99)
    second = [first[0], independent_layers(cuda_device, shapes[:2], M, 100)[1]]
    ws = dl.Workspace.for_stream(first)
    # layer 0's copy, then layer 1's alone in the launch after layer 0
    assert dl.decode_stream_launches(second, ws) == 2 + 2
    st = torch.cuda.Stream()
    want_first = singles(first, ws)
    want = singles(second, ws)
    for use_graph in (False, True):
        got = run(first, ws, use_graph, st)
        for i in range(3):
            assert torch.equal(got[i], want_first[i]), (use_graph, i)
        got = run(second, ws, use_graph, st)
        for i in range(2):
            assert torch.equal(got[i], want[i]), (use_graph, i)
    assert dl.device_status() == 0
    dl.graph_cache_clear()


@pytest.mark.parametrize("M", [1, 16])
def test_tensor_memory_family_stream_matches_single_calls(cuda_device, M):
    """The tensor-memory family (forced): copies made ahead, and the prep
    launches of layers fed by an earlier layer, write its e4m3 activation
    parts; the stream equals single calls bit for bit."""
    specs = [(F8, 1024, 2048, True), (BF, 768, 1024, False), (F8, 512, 4096, False),
             (F8, 2048, 1024, True)]
    layers = independent_layers(cuda_device, specs, M, 101)
    L4 = inputs.make_layer(F8, M, 256, 512, bias=False, config_id=101, layer_idx=4).to(cuda_device)
    y4 = torch.empty((M, 256), dtype=torch.bfloat16, device=cuda_device)
    layers.append(dl.Layer(dl.FP8_B128, layers[2].y, L4.w, y4, L4.scales))    # x = y of layer 2
    dl.set_override(dl.KERNEL_TC, 0, 0)
    try:
        ws = dl.Workspace.for_stream(layers)
        # layer 0's copy, layers 2 and 3 after it, layer 4 (x = y of layer 2) with its own prep
        assert dl.decode_stream_launches(layers, ws) == 2 + 5 + 1
        want = []
        for i, L in enumerate(layers):
            x = want[2] if i == 4 else L.x
            y = torch.empty_like(L.y)
            if L.dtype == dl.BF16:
                dl.linear_bf16(x, L.w, L.bias, out=y, workspace=ws)
            else:
                dl.linear_fp8_block128(x, L.w, L.scales, L.bias, out=y, workspace=ws)
            want.append(y)
        torch.cuda.synchronize()
        st = torch.cuda.Stream()
        for use_graph in (False, True):
            got = run(layers, ws, use_graph, st)
            for i in range(len(layers)):
                assert torch.equal(got[i], want[i]), (use_graph, i)
    finally:
        dl.set_override(0, 0, 0)
        dl.graph_cache_clear()
    assert dl.device_status() == 0
