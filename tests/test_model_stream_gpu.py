"""The whole-model decode weight stream at full size, checked against the oracle.

80 Qwen2.5-72B-shaped decoder layers with weight-only FP8 block-128 weights
(QKV with bias, O, gate_up with the fused SwiGLU epilogue, down) and the bf16
lm_head with the fused argmax, M = 1, built exactly as the benchmark builds
them (same seeds, the same chaining: down -> next QKV, O -> gate_up, gate_up ->
down, last down -> lm_head) and run through dl_decode_stream as one cached
CUDA graph with the benchmark's workspace, so that every activation-copy path
of the stream is exercised: copies made ahead, copies written by the layer
before (down -> QKV, O -> gate_up), prep launches (SwiGLU -> down), and the
argmax after 320 layers.  Every decoded token streams every weight once
("Developing a custom Qwen2.5 72B inference engine from scratch", §2) and the
next token is picked on the GPU (same page, §5).

For decoder layers 0, 41 and 79 each linear is checked on the device input
bytes it actually read: the stream's output equals a single call's output bit
for bit, and that call's fp32 values match the oracle on sampled rows (every
tile edge, the ragged end, random rows) within the acceptance tolerance.  The
token id equals the argmax of the lm_head's own fp32 logits, which match the
oracle on sampled rows, and the oracle's logit at that id is within tolerance
of the oracle's maximum over all 152064 rows.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs
from parity_util import assert_parity, oracle_for, sample_rows
from test_argmax_gpu import check_decision, check_near_true_max
from test_swiglu_gpu import check as check_swiglu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLED_LAYERS = (0, 41, 79)


@pytest.fixture(scope="module")
def model(cuda_device):
    dl.set_override(0, 0, 0)
    layers = bench.build_layers("qwen72b_model_fp8_m1", cuda_device)
    ys = [bench.out_buffer(L, cuda_device) for _, L in layers]
    for j in range(1, len(layers)):
        if layers[j][1].x is None:
            layers[j][1].x = ys[j - 1]
    dl_layers = [dl.Layer(dl.BF16 if L.dtype == "bf16" else dl.FP8_B128, L.x, L.w, ys[j],
                          L.scales, L.bias, act=L.act) for j, (_, L) in enumerate(layers)]
    ws = dl.Workspace.for_stream(dl_layers)
    st = torch.cuda.Stream(cuda_device)
    dl.decode_stream(dl_layers, ws, use_graph=True, stream=st)
    st.synchronize()
    first = [y.clone() for y in ys]
    dl.decode_stream(dl_layers, ws, use_graph=True, stream=st)     # the cached graph, replayed
    st.synchronize()
    assert dl.device_status() == 0
    yield layers, ys, first
    dl.graph_cache_clear()
    del dl_layers, ws


def test_stream_is_the_benchmark_stream(model):
    layers, ys, _ = model
    assert len(layers) == 4 * inputs.QWEN72B_LAYERS + 1
    chained = [j for j in range(1, len(layers)) if layers[j][1].x is ys[j - 1]]
    # every decoder layer's QKV (from the previous down, or x for layer 0),
    # gate_up (from O), down (from gate_up) and the lm_head are chained
    assert len(chained) == 3 * inputs.QWEN72B_LAYERS
    assert layers[-1][0] == "lm_head" and layers[-1][1].act == 2


def test_replay_is_bitwise_identical(model):
    _, ys, first = model
    for j, (a, b) in enumerate(zip(ys, first)):
        assert torch.equal(a, b), j


@pytest.mark.parametrize("layer", SAMPLED_LAYERS)
def test_sampled_decoder_layer_against_oracle(model, cuda_device, layer):
    layers, ys, _ = model
    for j in range(4 * layer, 4 * layer + 4):
        name, L = layers[j]
        Lx = inputs.LayerInputs(L.dtype, L.M, L.N, L.K, L.x.clone(), L.w, L.scales, L.bias)
        ws = dl.Workspace(dl.workspace_bytes(L.M, L.N, L.K, dl.FP8_B128), cuda_device)
        if L.act == 1:
            I = L.N // 2
            y32 = torch.empty((L.M, I), dtype=torch.float32, device=cuda_device)
            y = dl.linear_swiglu(Lx.x, Lx.w, Lx.scales, Lx.bias, out_f32=y32, workspace=ws)
            torch.cuda.synchronize(cuda_device)
            assert torch.equal(y, ys[j]), f"{name}: stream output differs from a single call"
            check_swiglu(Lx, y, y32, outputs=sample_rows(I, seed=40 + layer), what=name)
        else:
            y32 = torch.empty((L.M, L.N), dtype=torch.float32, device=cuda_device)
            y = dl.linear_fp8_block128(Lx.x, Lx.w, Lx.scales, Lx.bias, out_f32=y32, workspace=ws)
            torch.cuda.synchronize(cuda_device)
            assert torch.equal(y, ys[j]), f"{name}: stream output differs from a single call"
            rows = sample_rows(L.N, seed=40 + layer)
            ref, a = oracle_for(Lx, rows=rows)
            assert_parity(y, y32, ref, a, rows=rows, what=name)
    assert dl.device_status() == 0


def test_lm_head_token_against_oracle(model, cuda_device):
    layers, ys, _ = model
    name, L = layers[-1]
    Lx = inputs.LayerInputs(L.dtype, L.M, L.N, L.K, L.x.clone(), L.w, L.scales, L.bias)
    ws = dl.Workspace(dl.workspace_bytes(L.M, L.N, L.K, dl.BF16), cuda_device)
    y32 = torch.empty((L.M, L.N), dtype=torch.float32, device=cuda_device)
    y = torch.empty((L.M, L.N), dtype=torch.bfloat16, device=cuda_device)
    mx = torch.empty(L.M, dtype=torch.float32, device=cuda_device)
    idx = dl.linear_argmax(Lx.x, Lx.w, None, Lx.bias, out_max=mx, out=y, out_f32=y32, workspace=ws)
    torch.cuda.synchronize(cuda_device)
    assert torch.equal(idx, ys[-1]), "the stream's token differs from a single call's"
    check_decision(idx, mx, y32, name)
    rows = sample_rows(L.N, seed=49)
    ref, a = oracle_for(Lx, rows=rows)
    assert_parity(y, y32, ref, a, rows=rows, what=name)
    check_near_true_max(Lx, idx)                      # over all 152064 logits
    assert dl.device_status() == 0
