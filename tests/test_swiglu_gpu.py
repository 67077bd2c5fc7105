"""gate_up with the fused SwiGLU epilogue (dl_linear_swiglu) against the oracle.

Tolerance, per output (written out in swiglu_bound): the kernel's fp32 sums
g~, u~ of the gate and up rows obey the linear layer's bound
|g~ - g| <= dg = 2e-3 A_g + 1e-6 (the same for u), A = sum_k |x_k w_k|.  silu
is Lipschitz with constant sup |silu'| = 1.0998... < 1.1, so
|silu(g~) u~ - silu(g) u| <= 1.1 dg (|u| + du) + |silu(g)| du; the fp32
evaluation of g / (1 + e^-g) * u adds a few roundings (expf within 2 ulp), at
most 1e-6 |y| for safety, plus 1e-6 absolute.  y is RNE(y_f32) bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs
from parity_util import ABS_TOL, REL_TOL, sample_rows

pytestmark = pytest.mark.gpu

FAMILIES = [dl.KERNEL_SIMT, dl.KERNEL_MMA, dl.KERNEL_TC]   # TC: FP8 only (bf16 runs its auto family)


def swiglu_bound(g, u, ag, au):
    dg = REL_TOL * ag + ABS_TOL
    du = REL_TOL * au + ABS_TOL
    y = oracle.silu(g) * u
    return 1.1 * dg * (np.abs(u) + du) + np.abs(oracle.silu(g)) * du + 1e-6 * np.abs(y) + 1e-6


def run_swiglu(L, dev, workspace=None):
    I = L.N // 2
    y32 = torch.empty((L.M, I), dtype=torch.float32, device=dev)
    y = dl.linear_swiglu(L.x, L.w, L.scales, L.bias, out_f32=y32, workspace=workspace)
    torch.cuda.synchronize(dev)
    return y, y32


def oracle_swiglu(L, outputs=None):
    xb = inputs.bf16_bits(L.x)
    bb = inputs.bf16_bits(L.bias) if L.bias is not None else None
    if L.dtype == inputs.DTYPE_BF16:
        return oracle.swiglu(oracle.BF16, xb, inputs.bf16_bits(L.w), bias_bits=bb, outputs=outputs)
    return oracle.swiglu(oracle.FP8_B128, xb, inputs.u8_codes(L.w), L.scales.cpu().numpy(),
                         bias_bits=bb, outputs=outputs)


def check(L, y, y32, outputs=None, what=""):
    ref, g, u, ag, au = oracle_swiglu(L, outputs)
    got = y32.detach().cpu().double().numpy()
    yb = inputs.bf16_bits(y)
    if outputs is not None:
        got = got[:, outputs]
        yb = yb[:, outputs]
    bound = swiglu_bound(g, u, ag, au)
    bad = ~(np.abs(got - ref) <= bound)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first "
                           f"{np.argwhere(bad)[:3].tolist()}")
    rne = oracle.round_to_bf16(y32.detach().cpu().numpy())
    if outputs is not None:
        rne = rne[:, outputs]
    assert np.array_equal(rne, yb), f"{what}: y differs from RNE(y_f32)"


SHAPES = [(8, 128), (72, 1024), (200, 256), (1000, 2048)]      # (I outputs, K)


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("M", [1, 2, 6, 9, 16])
@pytest.mark.parametrize("dtype", [inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128])
def test_swiglu_small_shapes(cuda_device, dtype, M, family):
    dl.set_override(family, 0, 0)
    for i, (I, K) in enumerate(SHAPES):
        L = inputs.make_layer(dtype, M, 2 * I, K, bias=(i % 2 == 1), config_id=60 + i)
        y, y32 = run_swiglu(L.to(cuda_device), cuda_device)
        check(L, y, y32, what=f"{dtype} M={M} I={I} K={K} fam={family}")


@pytest.mark.parametrize("ctas", [1, 2, 3, 17])
@pytest.mark.parametrize("dtype", [inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128])
def test_swiglu_split_k_fixup(cuda_device, dtype, ctas):
    """Few CTAs: most tiles are finished by the fix-up, which pairs the slots."""
    dl.set_override(0, 0, ctas)
    L = inputs.make_layer(dtype, 6, 2 * 504, 4096, bias=True, config_id=64)
    y, y32 = run_swiglu(L.to(cuda_device), cuda_device)
    check(L, y, y32, what=f"{dtype} ctas={ctas}")


def test_swiglu_in_decode_stream_matches_single_calls(cuda_device):
    """act = 1 layers inside dl_decode_stream, the SwiGLU output chained into a
    down projection, against single calls."""
    dl.set_override(0, 0, 0)
    M, H, I = 2, 1024, 1536
    gu = inputs.make_layer(inputs.DTYPE_FP8_B128, M, 2 * I, H, bias=False, config_id=65).to(cuda_device)
    dn = inputs.make_layer(inputs.DTYPE_BF16, M, H, I, bias=False, config_id=66).to(cuda_device)
    act = torch.empty((M, I), dtype=torch.bfloat16, device=cuda_device)
    out = torch.empty((M, H), dtype=torch.bfloat16, device=cuda_device)
    layers = [dl.Layer(dl.FP8_B128, gu.x, gu.w, act, scales=gu.scales, act=1),
              dl.Layer(dl.BF16, act, dn.w, out)]
    ws = dl.Workspace(max(dl.workspace_bytes(M, 2 * I, H, dl.FP8_B128),
                          dl.workspace_bytes(M, H, I, dl.BF16)), cuda_device)
    side = torch.cuda.Stream(cuda_device)
    for use_graph in (False, True, True):
        with torch.cuda.stream(side):
            dl.decode_stream(layers, ws, use_graph=use_graph, stream=side)
        side.synchronize()
        ref_act = dl.linear_swiglu(gu.x, gu.w, gu.scales, workspace=ws)
        ref_out = dl.linear_bf16(ref_act, dn.w, workspace=ws)
        torch.cuda.synchronize(cuda_device)
        assert torch.equal(act, ref_act) and torch.equal(out, ref_out)
    assert dl.device_status() == 0


@pytest.mark.slow
@pytest.mark.parametrize("dtype,M", [(inputs.DTYPE_BF16, 1), (inputs.DTYPE_FP8_B128, 6)])
def test_swiglu_full_size_gate_up(cuda_device, dtype, M):
    """Qwen2.5-72B gate_up (2 x 29568 rows, K = 8192) in the launch configuration
    the bench uses, on sampled outputs (every tile edge, the tail, random)."""
    dl.set_override(0, 0, 0)
    I, K = 29568, 8192
    L = inputs.make_layer(dtype, M, 2 * I, K, bias=False, config_id=67, device=cuda_device)
    y, y32 = run_swiglu(L, cuda_device)
    outs = sample_rows(I, count=160, seed=3)
    check(L, y, y32, outputs=outs, what=f"full gate_up {dtype} M={M}")


def test_swiglu_rejects_n_not_multiple_of_16(cuda_device):
    L = inputs.make_layer(inputs.DTYPE_BF16, 1, 40, 128, bias=False, config_id=68).to(cuda_device)
    y = torch.empty((1, 20), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(ValueError):
        dl.linear_swiglu(L.x, L.w, out=y)
