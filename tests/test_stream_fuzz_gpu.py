"""Randomised decode streams against the same chains run as single calls.

dl_decode_stream decides per layer how an FP8 layer's activation copy is made:
ahead of the stream (x ready at the start), by the epilogue of the layer just
before (x is that plain linear's whole y), or by its own prep launch; it also
places workspace regions and caches graphs.  Seeded random chains mix bf16
and FP8 layers, SwiGLU and argmax layers, chained and fresh inputs, several
token counts and kernel families, and two workspace sizes.  Every output must
equal the single-call chain bit for bit.
"""
import random

import pytest
import torch

import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs

pytestmark = pytest.mark.gpu

BF, F8 = inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128


def random_chain(rng, dev, seed):
    """(layers, spec): 5-9 layers of one token count; each layer reads the
    previous layer's y when the shapes allow it and a coin says so."""
    M = rng.choice([1, 2, 6, 9, 16])
    n = rng.randint(5, 9)
    layers, spec = [], []
    prev_y, prev_cols = None, None
    for i in range(n):
        dt = rng.choice([BF, F8, F8])
        last = i == n - 1
        act = 2 if (last and rng.random() < 0.4) else (1 if rng.random() < 0.2 else 0)
        N = 128 * rng.randint(1, 6)
        if act == 1:
            N = 256 * rng.randint(1, 3)                 # y has N/2 columns, a multiple of 128
        chain = (prev_y is not None and prev_cols is not None and rng.random() < 0.7
                 and (prev_cols % 128 == 0 if dt == F8 else prev_cols % 8 == 0))
        K = prev_cols if chain else 128 * rng.randint(1, 8)
        L = inputs.make_layer(dt, M, N, K, bias=rng.random() < 0.3, config_id=seed, layer_idx=i).to(dev)
        x = prev_y if chain else L.x
        if act == 2:
            y = torch.empty((M,), dtype=torch.int32, device=dev)
            prev_y, prev_cols = None, None
        else:
            cols = N // 2 if act == 1 else N
            y = torch.empty((M, cols), dtype=torch.bfloat16, device=dev)
            prev_y, prev_cols = y, cols
        layers.append(dl.Layer(dl.BF16 if dt == BF else dl.FP8_B128, x, L.w, y, L.scales, L.bias, act=act))
        spec.append((dt, M, N, K, act, chain))
    return layers, spec


def single_calls(layers, spec, ws):
    out, prev = [], None
    for L, (dt, M, N, K, act, chain) in zip(layers, spec):
        x = prev if chain else L.x
        if act == 2:
            y = dl.linear_argmax(x, L.w, L.scales, L.bias, workspace=ws)
        elif act == 1:
            y = dl.linear_swiglu(x, L.w, L.scales, L.bias, workspace=ws)
        elif L.dtype == dl.BF16:
            y = dl.linear_bf16(x, L.w, L.bias, workspace=ws)
        else:
            y = dl.linear_fp8_block128(x, L.w, L.scales, L.bias, workspace=ws)
        out.append(y)
        prev = y
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("family", [0, dl.KERNEL_MMA, dl.KERNEL_TC])
@pytest.mark.parametrize("seed", range(6))
def test_random_streams_match_single_calls(cuda_device, seed, family):
    rng = random.Random(1000 * family + seed)
    layers, spec = random_chain(rng, cuda_device, 300 + seed)
    dl.set_override(family, 0, 0)
    try:
        big = dl.Workspace.for_stream(layers)
        small = dl.Workspace.for_shapes([L.shape() for L in layers], cuda_device)
        want = single_calls(layers, spec, small)
        st = torch.cuda.Stream()
        for ws in (big, small):
            for use_graph in (False, True, True):
                for L in layers:
                    L.y.zero_()
                torch.cuda.synchronize()
                with torch.cuda.stream(st):
                    dl.decode_stream(layers, ws, use_graph=use_graph, stream=st)
                st.synchronize()
                for i, L in enumerate(layers):
                    assert torch.equal(L.y, want[i]), (seed, family, ws.nbytes, use_graph, i, spec[i])
            assert torch.all(ws.tensor[:dl.WORKSPACE_ZERO_BYTES] == 0)
    finally:
        dl.set_override(0, 0, 0)
        dl.graph_cache_clear()
    assert dl.device_status() == 0
