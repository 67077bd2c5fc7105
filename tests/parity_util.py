"""Shared helpers for the GPU parity tests: run the library through its binding
and compare with the CPU oracle on the same bytes."""
import numpy as np
import torch

import oracle
import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs

# The acceptance bound, per element, before bf16 rounding:
#   |y_gpu - y_ref| <= 2e-3 * sum_k |x_k w_nk| + 1e-6
REL_TOL = 2e-3
ABS_TOL = 1e-6


def run_gpu(L: inputs.LayerInputs, dev, *, workspace=None):
    """y (bf16) and y_f32 from the library for a layer already on `dev`."""
    y32 = torch.empty((L.M, L.N), dtype=torch.float32, device=dev)
    if L.dtype == inputs.DTYPE_BF16:
        y = dl.linear_bf16(L.x, L.w, L.bias, out_f32=y32, workspace=workspace)
    else:
        y = dl.linear_fp8_block128(L.x, L.w, L.scales, L.bias, out_f32=y32, workspace=workspace)
    torch.cuda.synchronize(dev)
    return y, y32


def oracle_for(L: inputs.LayerInputs, rows=None, k_range=None, with_bias=True):
    """Oracle y and sum|x w| for a layer (tensors on any device; copied to host)."""
    xb = inputs.bf16_bits(L.x)
    bb = inputs.bf16_bits(L.bias) if (L.bias is not None and with_bias) else None
    if L.dtype == inputs.DTYPE_BF16:
        return oracle.linear(oracle.BF16, xb, inputs.bf16_bits(L.w), bias_bits=bb, rows=rows,
                             k_range=k_range)
    return oracle.linear(oracle.FP8_B128, xb, inputs.u8_codes(L.w), L.scales.cpu().numpy(),
                         bias_bits=bb, rows=rows, k_range=k_range)


def assert_parity(y, y32, ref, a, rows=None, what=""):
    """Tolerance on y_f32, and y == RNE(y_f32) bit for bit."""
    got32 = y32.detach().cpu()
    ybits = inputs.bf16_bits(y)
    if rows is not None:
        got32 = got32[:, rows]
        ybits = ybits[:, rows]
    g = got32.double().numpy()
    bound = REL_TOL * a + ABS_TOL
    err = np.abs(g - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                             f"first {idx}; max err/bound {float(np.nanmax(err / bound)):.3g}")
    rne = oracle.round_to_bf16(got32.numpy())
    if not np.array_equal(rne, ybits):
        n = int((rne != ybits).sum())
        raise AssertionError(f"{what}: {n} bf16 outputs differ from RNE(y_f32)")
    return float(np.max(err / bound)) if err.size else 0.0


def sample_rows(N, count=192, seed=0):
    """Rows across the whole range: both ends of every 128-row tile edge sampled,
    plus random rows; always includes row 0 and row N-1 (the ragged tail)."""
    rng = np.random.default_rng(seed)
    picks = {0, N - 1, min(127, N - 1), min(128, N - 1), max(0, N - 128), max(0, N - 129)}
    picks.update(rng.integers(0, N, size=count).tolist())
    return np.array(sorted(picks), dtype=np.int64)
