"""The CUDA-graph cache of dl_decode_stream: keyed on the layers' fields (not on
the struct's padding bytes) and bounded, least recently used first out."""
import ctypes

import pytest
import torch

import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs

pytestmark = pytest.mark.gpu


def _layers(dev, n_out=1, seed=60):
    A = inputs.make_layer(inputs.DTYPE_BF16, 1, 256, 512, bias=True, config_id=seed).to(dev)
    B = inputs.make_layer(inputs.DTYPE_BF16, 1, 128, 256, bias=False, config_id=seed,
                          layer_idx=1).to(dev)
    ya = torch.empty((1, 256), dtype=torch.bfloat16, device=dev)
    outs = [torch.empty((1, 128), dtype=torch.bfloat16, device=dev) for _ in range(n_out)]
    lists = [[dl.Layer(dl.BF16, A.x, A.w, ya, None, A.bias), dl.Layer(dl.BF16, ya, B.w, yb)]
             for yb in outs]
    return lists, outs


def test_key_ignores_struct_padding(cuda_device):
    """Two calls with the same fields but different tail-padding bytes reuse one graph."""
    dl.graph_cache_clear()
    (layers,), (yb,) = _layers(cuda_device)
    ws = dl.Workspace.for_stream(layers)
    st = torch.cuda.Stream()
    size = ctypes.sizeof(dl._Layer)
    results = []
    for fill in (0x00, 0xA5, 0x5A):
        raw = (ctypes.c_ubyte * (size * len(layers)))(*([fill] * (size * len(layers))))
        arr = ctypes.cast(raw, ctypes.POINTER(dl._Layer))
        for i, L in enumerate(layers):
            s = dl._layer_struct(L)
            ctypes.memmove(ctypes.addressof(raw) + i * size, ctypes.addressof(s),
                           dl._Layer.act.offset + 4)      # the fields only, not the padding
        assert bytes(raw)[size - 1] == fill
        st_ptr = ctypes.c_void_p(st.cuda_stream)
        assert dl.load().dl_decode_stream(arr, len(layers), ws.ptr, ws.nbytes, st_ptr, 1) == 0
        st.synchronize()
        results.append(yb.clone())
    assert dl.graph_cache_size() == 1
    assert all(torch.equal(r, results[0]) for r in results)
    dl.graph_cache_clear()
    assert dl.graph_cache_size() == 0


def test_cache_is_bounded_and_evicted_lists_recapture(cuda_device):
    dl.graph_cache_clear()
    lists, outs = _layers(cuda_device, n_out=20)
    ws = dl.Workspace.for_stream(lists[0])
    st = torch.cuda.Stream()
    # reference: every list without graphs (same kernels, same bits)
    for layers in lists:
        dl.decode_stream(layers, ws, use_graph=False, stream=st)
    st.synchronize()
    ref = outs[0].clone()
    assert all(torch.equal(o, ref) for o in outs)
    for o in outs:
        o.zero_()
    for layers in lists:
        dl.decode_stream(layers, ws, use_graph=True, stream=st)
    st.synchronize()
    assert dl.graph_cache_size() == 16
    assert all(torch.equal(o, ref) for o in outs)
    # the first lists were evicted: replaying them captures them again, correctly
    outs[0].zero_()
    dl.decode_stream(lists[0], ws, use_graph=True, stream=st)
    st.synchronize()
    assert torch.equal(outs[0], ref)
    assert dl.graph_cache_size() == 16
    dl.graph_cache_clear()
