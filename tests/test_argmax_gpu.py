"""lm_head with the fused on-device argmax (dl_linear_argmax) against the oracle.

The decision is an integer taken from floating point, so both sides take it in
the kernel's precision: idx must equal the lowest-index argmax of the kernel's
own fp32 logits (exactly), and those logits must match the oracle within the
linear layer's tolerance, so the chosen logit is within tolerance of the true
maximum.  Ties and NaN are placed on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs
from parity_util import ABS_TOL, REL_TOL, assert_parity, oracle_for, sample_rows

pytestmark = pytest.mark.gpu

FAMILIES = [dl.KERNEL_SIMT, dl.KERNEL_MMA, dl.KERNEL_TC]   # TC: FP8 only (bf16 runs its auto family)


def run_argmax(L, dev, logits=True, workspace=None):
    M = L.M
    y32 = torch.empty((M, L.N), dtype=torch.float32, device=dev) if logits else None
    y = torch.empty((M, L.N), dtype=torch.bfloat16, device=dev) if logits else None
    mx = torch.empty(M, dtype=torch.float32, device=dev)
    idx = dl.linear_argmax(L.x, L.w, L.scales, L.bias, out_max=mx, out=y, out_f32=y32,
                           workspace=workspace)
    torch.cuda.synchronize(dev)
    return idx, mx, y, y32


def check_decision(idx, mx, y32, what):
    got = y32.cpu().numpy()
    want = oracle.argmax_lowest(got)
    assert np.array_equal(idx.cpu().numpy(), want), f"{what}: idx {idx.tolist()} != {want.tolist()}"
    chosen = got[np.arange(got.shape[0]), want]
    m = mx.cpu().numpy()
    assert np.array_equal(np.isnan(m), np.isnan(chosen)) and np.array_equal(
        m[~np.isnan(m)], chosen[~np.isnan(chosen)]), f"{what}: maxval"


def check_near_true_max(L, idx, rows=None):
    """The oracle's value at the chosen index is within tolerance of its maximum."""
    ref, a = oracle_for(L, rows=rows)
    bound = REL_TOL * a + ABS_TOL
    cols = np.arange(ref.shape[1]) if rows is None else np.asarray(rows)
    pos = {int(c): i for i, c in enumerate(cols)}
    for m, n in enumerate(idx.cpu().numpy().tolist()):
        if n not in pos:
            continue
        best = int(np.argmax(ref[m]))
        assert ref[m, pos[n]] >= ref[m, best] - bound[m, pos[n]] - bound[m, best]


SHAPES = [(1, 128), (300, 1024), (129, 256), (5000, 2048)]


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("M", [1, 2, 6, 9, 16])
@pytest.mark.parametrize("dtype", [inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128])
def test_argmax_small_shapes(cuda_device, dtype, M, family):
    dl.set_override(family, 0, 0)
    for i, (N, K) in enumerate(SHAPES):
        L = inputs.make_layer(dtype, M, N, K, bias=(i % 2 == 1), config_id=70 + i)
        Ld = L.to(cuda_device)
        idx, mx, y, y32 = run_argmax(Ld, cuda_device)
        ref, a = oracle_for(L)
        assert_parity(y, y32, ref, a, what=f"argmax logits {dtype} M={M} N={N}")
        check_decision(idx, mx, y32, f"{dtype} M={M} N={N} fam={family}")
        check_near_true_max(L, idx)
        # the same decision without writing the logits
        idx2, mx2, _, _ = run_argmax(Ld, cuda_device, logits=False)
        assert torch.equal(idx, idx2) and torch.equal(mx, mx2)


@pytest.mark.parametrize("ctas", [1, 2, 3, 17])
@pytest.mark.parametrize("dtype", [inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128])
def test_argmax_through_split_k_fixups(cuda_device, dtype, ctas):
    dl.set_override(0, 0, ctas)
    L = inputs.make_layer(dtype, 6, 1000, 4096, bias=True, config_id=75)
    idx, mx, y, y32 = run_argmax(L.to(cuda_device), cuda_device)
    check_decision(idx, mx, y32, f"{dtype} ctas={ctas}")
    check_near_true_max(L, idx)


def _one_hot_layer(dtype, N, K, col0, M=1):
    """x = e_0 (every token), so logit n = W[n][0] exactly (FP8 scales 1)."""
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    x[:, 0] = 1.0
    if dtype == inputs.DTYPE_BF16:
        w = torch.zeros((N, K), dtype=torch.bfloat16)
        w[:, 0] = torch.tensor(col0, dtype=torch.float32).to(torch.bfloat16)
        return inputs.LayerInputs(dtype, M, N, K, x, w, None, None)
    w = torch.zeros((N, K), dtype=torch.uint8)
    w[:, 0] = torch.tensor(col0, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)
    s = torch.ones(((N + 127) // 128, K // 128), dtype=torch.float32)
    return inputs.LayerInputs(dtype, M, N, K, x, w, s, None)


@pytest.mark.parametrize("ctas", [0, 3])
@pytest.mark.parametrize("dtype", [inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128])
def test_argmax_ties_go_to_the_lowest_index(cuda_device, dtype, ctas):
    dl.set_override(0, 0, ctas)
    N, K = 5000, 1024
    col = np.full(N, -2.0)
    col[[4000, 37, 300, 2999]] = 8.0               # equal maxima; lowest is 37
    col[5] = -0.0
    L = _one_hot_layer(dtype, N, K, col, M=3).to(cuda_device)
    idx, mx, _, y32 = run_argmax(L, cuda_device)
    assert idx.tolist() == [37, 37, 37] and mx.tolist() == [8.0, 8.0, 8.0]
    check_decision(idx, mx, y32, "ties")
    # all equal (including -0 and +0): index 0
    L0 = _one_hot_layer(dtype, N, K, np.where(np.arange(N) % 2 == 0, 0.0, -0.0)).to(cuda_device)
    assert run_argmax(L0, cuda_device)[0].tolist() == [0]


@pytest.mark.parametrize("dtype", [inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128])
def test_argmax_nan_counts_as_largest(cuda_device, dtype):
    dl.set_override(0, 0, 0)
    N, K = 3000, 256
    col = np.linspace(-3.0, 3.0, N).astype(np.float32)
    col[[2500, 250, 1000]] = np.nan
    L = _one_hot_layer(dtype, N, K, col, M=2).to(cuda_device)
    idx, mx, _, y32 = run_argmax(L, cuda_device)
    assert idx.tolist() == [250, 250] and torch.isnan(mx).all()
    check_decision(idx, mx, y32, "nan")


def test_argmax_in_decode_stream(cuda_device):
    """act = 2 as the last layer of a stream: y receives the indices."""
    dl.set_override(0, 0, 0)
    M, H, V = 2, 2048, 12000
    a = inputs.make_layer(inputs.DTYPE_FP8_B128, M, H, H, bias=False, config_id=76).to(cuda_device)
    lm = inputs.make_layer(inputs.DTYPE_BF16, M, V, H, bias=False, config_id=77).to(cuda_device)
    h = torch.empty((M, H), dtype=torch.bfloat16, device=cuda_device)
    ids = torch.empty(M, dtype=torch.int32, device=cuda_device)
    layers = [dl.Layer(dl.FP8_B128, a.x, a.w, h, scales=a.scales),
              dl.Layer(dl.BF16, h, lm.w, ids, act=2)]
    ws = dl.Workspace(max(dl.workspace_bytes(M, H, H, dl.FP8_B128),
                          dl.workspace_bytes(M, V, H, dl.BF16)), cuda_device)
    side = torch.cuda.Stream(cuda_device)
    for use_graph in (False, True, True):
        with torch.cuda.stream(side):
            dl.decode_stream(layers, ws, use_graph=use_graph, stream=side)
        side.synchronize()
        ref_h = dl.linear_fp8_block128(a.x, a.w, a.scales, workspace=ws)
        ref_ids = dl.linear_argmax(ref_h, lm.w, workspace=ws)
        torch.cuda.synchronize(cuda_device)
        assert torch.equal(h, ref_h) and torch.equal(ids, ref_ids)
    assert torch.all(ws.tensor[:dl.WORKSPACE_ZERO_BYTES] == 0)
    assert dl.device_status() == 0


def test_argmax_repeatable_and_zero_prefix_restored(cuda_device):
    dl.set_override(0, 0, 0)
    L = inputs.make_layer(inputs.DTYPE_BF16, 4, 20000, 1024, bias=True, config_id=78).to(cuda_device)
    ws = dl.Workspace(dl.workspace_bytes(4, 20000, 1024, dl.BF16), cuda_device)
    first = run_argmax(L, cuda_device, logits=False, workspace=ws)[:2]
    for _ in range(5):
        again = run_argmax(L, cuda_device, logits=False, workspace=ws)[:2]
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
        assert torch.all(ws.tensor[:dl.WORKSPACE_ZERO_BYTES] == 0)


@pytest.mark.slow
def test_argmax_full_size_lm_head(cuda_device):
    """Qwen2.5-72B lm_head (152064 x 8192, bf16) at M = 1 in the bench's launch
    configuration: exact decision on the kernel's logits, sampled logits against
    the oracle, and the chosen logit against the oracle's maximum over all rows."""
    dl.set_override(0, 0, 0)
    N, K, _ = inputs.QWEN72B_LM_HEAD
    L = inputs.make_layer(inputs.DTYPE_BF16, 1, N, K, bias=False, config_id=79, device=cuda_device)
    idx, mx, y, y32 = run_argmax(L, cuda_device)
    check_decision(idx, mx, y32, "lm_head")
    rows = np.union1d(sample_rows(N, count=128, seed=7), idx.cpu().numpy())
    ref, a = oracle_for(L, rows=rows)
    assert_parity(y, y32, ref, a, rows=rows, what="lm_head logits")
    check_near_true_max(L, idx)
