"""GPU parity: the CUDA path against the CPU oracle on identical seeded bytes.

Bar: |y_f32 - y_ref| <= 2e-3 * sum_k |x w| + 1e-6 per element before rounding,
y == RNE(y_f32) bit for bit, e4m3 decode bit-exact, repeated runs bitwise
identical.  Shapes span several 128-row tiles, ragged N and K tails, every
M in 1..16 and both kernel families.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs
from parity_util import assert_parity, oracle_for, run_gpu, sample_rows

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FAMILIES = [dl.KERNEL_SIMT, dl.KERNEL_MMA, dl.KERNEL_TC]   # TC: FP8 only (bf16 runs its auto family)


@pytest.fixture(autouse=True)
def _reset_overrides():
    dl.set_override(0, 0, 0)
    yield
    dl.set_override(0, 0, 0)


def _bits_tensor(values, dev):
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(np.asarray(values, dtype=np.float32)))
    return t.to(dev)


def _codes_tensor(values, dev):
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.float8_e4m3fn)
    assert torch.equal(t.float(), torch.tensor(np.asarray(values, dtype=np.float32)))
    return t.view(torch.uint8).to(dev)


# ------------------------------------------------------------------ configs / shapes

@pytest.mark.parametrize("family", [0] + FAMILIES)
def test_bf16_gemv_1024_with_bias(cuda_device, family):
    """BF16 GEMV M=1, K=N=1024, bias: every output against the oracle."""
    dl.set_override(family, 0, 0)
    L = inputs.make_layer(inputs.DTYPE_BF16, 1, 1024, 1024, bias=True, config_id=0)
    y, y32 = run_gpu(L.to(cuda_device), cuda_device)
    ref, a = oracle_for(L)
    assert_parity(y, y32, ref, a, what=f"cfg0 family {family}")


SMALL_BF16 = [(1, 128), (127, 136), (129, 256), (300, 1000), (257, 8), (5, 4104)]
SMALL_FP8 = [(1, 128), (127, 256), (129, 384), (300, 1024), (257, 128)]


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("M", [1, 2, 3, 5, 6, 8, 9, 16])
def test_small_shapes_bf16(cuda_device, family, M):
    dl.set_override(family, 0, 0)
    for i, (N, K) in enumerate(SMALL_BF16):
        L = inputs.make_layer(inputs.DTYPE_BF16, M, N, K, bias=(i % 2 == 0), config_id=10 + i)
        y, y32 = run_gpu(L.to(cuda_device), cuda_device)
        ref, a = oracle_for(L)
        assert_parity(y, y32, ref, a, what=f"bf16 M={M} N={N} K={K} fam={family}")


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("M", [1, 2, 3, 5, 6, 8, 9, 16])
def test_small_shapes_fp8(cuda_device, family, M):
    dl.set_override(family, 0, 0)
    for i, (N, K) in enumerate(SMALL_FP8):
        L = inputs.make_layer(inputs.DTYPE_FP8_B128, M, N, K, bias=(i % 2 == 1), config_id=20 + i)
        y, y32 = run_gpu(L.to(cuda_device), cuda_device)
        ref, a = oracle_for(L)
        assert_parity(y, y32, ref, a, what=f"fp8 M={M} N={N} K={K} fam={family}")


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("ctas", [1, 2, 3, 17, 0])
def test_split_count_does_not_break_parity(cuda_device, family, ctas):
    """Any number of K splits (grid sizes) is correct within tolerance."""
    dl.set_override(family, 0, ctas)
    for dtype in (inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128):
        L = inputs.make_layer(dtype, 6, 1000, 2048, bias=True, config_id=30)
        y, y32 = run_gpu(L.to(cuda_device), cuda_device)
        ref, a = oracle_for(L)
        assert_parity(y, y32, ref, a, what=f"{dtype} ctas={ctas} fam={family}")


@pytest.mark.parametrize("family", FAMILIES)
def test_two_ctas_per_sm(cuda_device, family):
    dl.set_override(family, 2, 0)
    for dtype in (inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128):
        L = inputs.make_layer(dtype, 4, 2000, 4096, bias=False, config_id=31)
        y, y32 = run_gpu(L.to(cuda_device), cuda_device)
        ref, a = oracle_for(L)
        assert_parity(y, y32, ref, a, what=f"{dtype} 2 CTAs/SM fam={family}")


# ------------------------------------------------------------------ exactness pins

@pytest.mark.parametrize("family", FAMILIES)
def test_e4m3_dequant_bit_exact_all_codes(cuda_device, family):
    """Row n holds code n at column k0; x = e_k0: y_f32[n] = e4m3(n) * scale exactly."""
    dl.set_override(family, 0, 0)
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    K = 256
    for k0 in (0, 5, 127, 128, 250):
        for sc in ([[1.0, 1.0], [1.0, 1.0]], [[2.0, 0.25], [8.0, 0.5]]):
            codes = torch.zeros(256, K, dtype=torch.uint8)
            codes[:, k0] = torch.arange(256, dtype=torch.uint8)
            x = torch.zeros(1, K)
            x[0, k0] = 1.0
            scales = torch.tensor(sc, dtype=torch.float32)
            y32 = torch.empty(1, 256, dtype=torch.float32, device=cuda_device)
            dl.linear_fp8_block128(x.to(torch.bfloat16).to(cuda_device), codes.to(cuda_device),
                                   scales.to(cuda_device), out_f32=y32)
            got = y32.cpu().double().numpy()[0]
            expect = table * np.array([sc[n // 128][k0 // 128] for n in range(256)])
            nan = np.isnan(expect)
            assert np.array_equal(np.isnan(got), nan), (k0, family)
            assert np.array_equal(got[~nan], expect[~nan]), (k0, family)


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("M", [1, 2, 6, 16])
def test_fp8_activations_not_exact_in_f16(cuda_device, family, M):
    """FP8 units whose activation block spans more than f16 can hold after one
    power-of-two scaling (here ~60 binades, and values below f16's reach) take
    the exact bf16 route; the rest of the layer keeps the f16 route."""
    dl.set_override(family, 0, 0)
    N, K = 300, 1024
    L = inputs.make_layer(inputs.DTYPE_FP8_B128, M, N, K, bias=True, config_id=47)
    x = L.x.float()
    x[0, 128 + 5] = 2.0 ** 40                    # token 0, block 1: huge and tiny values
    x[0, 128 + 6] = -1.5 * 2.0 ** -20
    x[M - 1, 3] = 2.0 ** -100                    # last token, block 0: far below the rest
    x[M - 1, 700] = 3.0 * 2.0 ** 30              # and block 5: one large value
    L.x = x.to(torch.bfloat16)
    y, y32 = run_gpu(L.to(cuda_device), cuda_device)
    ref, a = oracle_for(L)
    assert_parity(y, y32, ref, a, what=f"fp8 wide-range x M={M} fam={family}")


@pytest.mark.parametrize("family", FAMILIES)
def test_one_hot_bf16_selects_column_exactly(cuda_device, family):
    dl.set_override(family, 0, 0)
    N, K = 300, 1024
    L = inputs.make_layer(inputs.DTYPE_BF16, 1, N, K, bias=True, config_id=40)
    for k0 in (0, 63, 64, 1000):
        x = torch.zeros(1, K, dtype=torch.bfloat16)
        x[0, k0] = 1.0
        y32 = torch.empty(1, N, dtype=torch.float32, device=cuda_device)
        dl.linear_bf16(x.to(cuda_device), L.w.to(cuda_device), L.bias.to(cuda_device), out_f32=y32)
        expect = L.w[:, k0].float() + L.bias.float()       # one IEEE fp32 addition
        assert torch.equal(y32.cpu()[0], expect), k0


@pytest.mark.parametrize("family", FAMILIES)
def test_power_of_two_scales_scale_outputs_exactly(cuda_device, family):
    dl.set_override(family, 0, 0)
    L = inputs.make_layer(inputs.DTYPE_FP8_B128, 6, 640, 2048, bias=False, config_id=41).to(cuda_device)
    _, y1 = run_gpu(L, cuda_device)
    L4 = inputs.LayerInputs(L.dtype, L.M, L.N, L.K, L.x, L.w, L.scales * 4.0, None)
    _, y4 = run_gpu(L4, cuda_device)
    assert torch.equal(y4, y1 * 4.0)


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("off", [1, 2, 3])
def test_fp8_scales_not_16_byte_aligned(cuda_device, family, off):
    """Block scales 4, 8 or 12 bytes past a 16-byte boundary, with an odd
    number of K blocks (K = 640: a stage's two scales may straddle a 16-byte
    block, the last unit of a tile has one) and a ragged last tile.  The
    floats around the scales are NaN, so reading a neighbour as a scale would
    show.  Same outputs, bit for bit, as with the scales at an aligned
    address, and within the oracle's bound."""
    dl.set_override(family, 0, 0)
    L = inputs.make_layer(inputs.DTYPE_FP8_B128, 6, 300, 640, bias=True, config_id=42).to(cuda_device)
    y_al, y32_al = run_gpu(L, cuda_device)
    n = L.scales.numel()
    buf = torch.full((n + 8,), float("nan"), dtype=torch.float32, device=cuda_device)
    view = buf[off:off + n].view(L.scales.shape)
    view.copy_(L.scales)
    assert view.data_ptr() % 16 == 4 * off
    Lo = inputs.LayerInputs(L.dtype, L.M, L.N, L.K, L.x, L.w, view, L.bias)
    y, y32 = run_gpu(Lo, cuda_device)
    assert torch.equal(y32, y32_al) and torch.equal(y, y_al)
    ref, a = oracle_for(L)
    assert_parity(y, y32, ref, a, what=f"fp8 scales at +{4 * off} B fam={family}")


@pytest.mark.parametrize("family", FAMILIES)
def test_row_permutation_within_tiles_permutes_outputs_bitwise(cuda_device, family):
    dl.set_override(family, 0, 0)
    for dtype in (inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128):
        L = inputs.make_layer(dtype, 3, 512, 1024, bias=False, config_id=42).to(cuda_device)
        perm = torch.cat([t * 128 + torch.randperm(128, generator=torch.Generator().manual_seed(t))
                          for t in range(4)]).to(cuda_device)
        _, y1 = run_gpu(L, cuda_device)
        Lp = inputs.LayerInputs(L.dtype, L.M, L.N, L.K, L.x, L.w[perm].contiguous(), L.scales, None)
        _, yp = run_gpu(Lp, cuda_device)
        assert torch.equal(yp, y1[:, perm])


@pytest.mark.parametrize("family", FAMILIES)
def test_repeated_runs_bitwise_identical(cuda_device, family):
    dl.set_override(family, 0, 0)
    for dtype in (inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128):
        L = inputs.make_layer(dtype, 6, 1000, 8192, bias=True, config_id=43).to(cuda_device)
        ya, a32 = run_gpu(L, cuda_device)
        for _ in range(3):
            yb, b32 = run_gpu(L, cuda_device)
            assert torch.equal(a32, b32) and torch.equal(ya, yb)


# ------------------------------------------------------------------ worked examples

@pytest.mark.parametrize("family", FAMILIES)
def test_column_split_example_on_gpu(cuda_device, family):
    dl.set_override(family, 0, 0)
    g = json.load(open(os.path.join(GOLDEN, "column_split_example.json")))
    x = np.zeros((2, 128)); x[:, :4] = g["x"]
    w = np.zeros((6, 128)); w[:, :4] = np.array(g["w_inputs_by_outputs"]).T
    want = torch.tensor(g["printed_one_device"], dtype=torch.float32)
    y32 = torch.empty(2, 6, dtype=torch.float32, device=cuda_device)
    dl.linear_bf16(_bits_tensor(x, cuda_device), _bits_tensor(w, cuda_device), out_f32=y32)
    assert torch.equal(y32.cpu(), want)
    dl.linear_fp8_block128(_bits_tensor(x, cuda_device), _codes_tensor(w, cuda_device),
                           torch.ones(1, 1, device=cuda_device), out_f32=y32)
    assert torch.equal(y32.cpu(), want)


@pytest.mark.parametrize("family", FAMILIES)
def test_mlp_split_example_two_way_split_k_on_gpu(cuda_device, family):
    """Second linear of the MLP example with K split over two CTAs at hidden unit 4.
    A work unit is 128 columns of bf16 and 256 columns of FP8, so the second half
    of the hidden units starts at column 128 (bf16) or 256 (FP8): two units,
    exactly two CTAs, one per unit."""
    dl.set_override(family, 0, 2)
    g = json.load(open(os.path.join(GOLDEN, "mlp_split_example.json")))
    x, a, b = (np.array(g[k], dtype=np.float64) for k in ("x", "a", "b"))
    h = np.maximum(x @ a, 0.0)             # small integers: exact; the example's ReLU
    y32 = torch.empty(2, 4, dtype=torch.float32, device=cuda_device)
    for fmt in ("bf16", "fp8"):
        half = 128 if fmt == "bf16" else 256
        hp = np.zeros((2, 2 * half)); hp[:, 0:4] = h[:, 0:4]; hp[:, half:half + 4] = h[:, 4:8]
        wp = np.zeros((4, 2 * half)); wp[:, 0:4] = b.T[:, 0:4]; wp[:, half:half + 4] = b.T[:, 4:8]
        def run(xx):
            if fmt == "bf16":
                dl.linear_bf16(_bits_tensor(xx, cuda_device), _bits_tensor(wp, cuda_device), out_f32=y32)
            else:
                dl.linear_fp8_block128(_bits_tensor(xx, cuda_device), _codes_tensor(wp, cuda_device),
                                       torch.ones(1, 4, device=cuda_device), out_f32=y32)
            return y32.cpu()
        assert torch.equal(run(hp), torch.tensor(g["printed_all_reduce_sum"], dtype=torch.float32))
        h0 = hp.copy(); h0[:, half:] = 0
        h1 = hp.copy(); h1[:, :half] = 0
        assert torch.equal(run(h0), torch.tensor(g["printed_device0_partial"], dtype=torch.float32))
        assert torch.equal(run(h1), torch.tensor(g["printed_device1_partial"], dtype=torch.float32))


# ------------------------------------------------------------------ bounds and errors

@pytest.mark.parametrize("family", FAMILIES)
def test_guard_bands_untouched(cuda_device, family):
    """Writes stay inside y, y_f32 and the workspace (sentinel bands around each)."""
    dl.set_override(family, 0, 0)
    G = 4096
    for dtype, (M, N, K) in ((inputs.DTYPE_BF16, (3, 129, 1000)), (inputs.DTYPE_FP8_B128, (9, 1, 256)),
                             (inputs.DTYPE_FP8_B128, (16, 10240 + 128, 1024))):
        L = inputs.make_layer(dtype, M, N, K, bias=True, config_id=44).to(cuda_device)
        ybuf = torch.full((2 * G + M * N,), -7.0, dtype=torch.bfloat16, device=cuda_device)
        fbuf = torch.full((2 * G + M * N,), -7.0, dtype=torch.float32, device=cuda_device)
        need = dl.workspace_bytes(M, N, K, dl.BF16 if dtype == inputs.DTYPE_BF16 else dl.FP8_B128)
        Z = dl.WORKSPACE_ZERO_BYTES
        wsbuf = torch.full((need + G,), 0xAB, dtype=torch.uint8, device=cuda_device)
        # zero prefix (counters, tickets); the scratch after it starts as NaN
        # bytes, so a partial sum read before it was written would show
        wsbuf[:Z] = 0
        wsbuf[Z:need] = 0xFF
        ws = dl.Workspace.__new__(dl.Workspace)
        ws.nbytes, ws.tensor = need, wsbuf
        y = ybuf[G:G + M * N]
        y32 = fbuf[G:G + M * N]
        if dtype == inputs.DTYPE_BF16:
            dl.linear_bf16(L.x, L.w, L.bias, out=y, out_f32=y32, workspace=ws)
        else:
            dl.linear_fp8_block128(L.x, L.w, L.scales, L.bias, out=y, out_f32=y32, workspace=ws)
        torch.cuda.synchronize()
        assert torch.all(ybuf[:G] == -7.0) and torch.all(ybuf[G + M * N:] == -7.0)
        assert torch.all(fbuf[:G] == -7.0) and torch.all(fbuf[G + M * N:] == -7.0)
        assert torch.all(wsbuf[need:] == 0xAB)
        # the counters and tickets are back to zero after the call
        assert torch.all(wsbuf[:Z] == 0)
        ref, a = oracle_for(L)
        assert_parity(y.view(M, N), y32.view(M, N), ref, a, what=f"guard bands {dtype} M={M} N={N}")


@pytest.mark.parametrize("family", FAMILIES)
def test_one_workspace_serves_calls_of_any_shape(cuda_device, family):
    """Calls with few tiles then many tiles share one workspace: every call leaves
    its zero prefix (counters, tickets) zero, so no call ever reads a stale
    arrival ticket, and the scratch after it is written before it is read."""
    dl.set_override(family, 0, 0)
    shapes = [(inputs.DTYPE_BF16, 1, 300, 8192), (inputs.DTYPE_FP8_B128, 6, 640, 8192),
              (inputs.DTYPE_BF16, 2, 20000, 1024), (inputs.DTYPE_FP8_B128, 9, 30000, 1024),
              (inputs.DTYPE_BF16, 16, 300, 8192), (inputs.DTYPE_BF16, 1, 40000, 512)]
    need = max(dl.workspace_bytes(M, N, K, dl.BF16 if dt == inputs.DTYPE_BF16 else dl.FP8_B128)
               for dt, M, N, K in shapes)
    ws = dl.Workspace(need, cuda_device)
    for i, (dt, M, N, K) in enumerate(shapes):
        L = inputs.make_layer(dt, M, N, K, bias=(i % 2 == 0), config_id=46, layer_idx=i)
        y, y32 = run_gpu(L.to(cuda_device), cuda_device, workspace=ws)
        rows = sample_rows(N, count=64, seed=i)
        ref, a = oracle_for(L, rows=rows)
        assert_parity(y, y32, ref, a, rows=rows, what=f"shared workspace call {i}")
        assert torch.all(ws.tensor[:dl.WORKSPACE_ZERO_BYTES] == 0), f"zero prefix dirty after call {i}"


def test_workspace_too_small_is_rejected_before_launch(cuda_device):
    L = inputs.make_layer(inputs.DTYPE_BF16, 1, 1024, 1024, bias=False, config_id=45).to(cuda_device)
    need = dl.workspace_bytes(1, 1024, 1024, dl.BF16)
    ws = dl.Workspace(need // 2, cuda_device)
    with pytest.raises(dl.DLError) as e:
        dl.linear_bf16(L.x, L.w, workspace=ws)
    assert e.value.status == 4


# ------------------------------------------------------------------ decode stream

def _chain(dev, dtypes, M=2, seed=50):
    """A chain of layers where each layer's x is the previous layer's y."""
    dims = [384, 1000, 256, 640, 128][: len(dtypes) + 1]
    layers, host = [], []
    x = inputs.normal_bf16((M, dims[0]), 1.0, inputs.seed_for(seed, 0, "x"), dev)
    for i, dt in enumerate(dtypes):
        K, N = dims[i], dims[i + 1]
        Li = inputs.make_layer(dt, M, N, K, bias=(i == 0), config_id=seed, layer_idx=i + 1).to(dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        layers.append(dl.Layer(dl.BF16 if dt == inputs.DTYPE_BF16 else dl.FP8_B128, x, Li.w, y,
                               Li.scales, Li.bias))
        host.append(Li)
        x = y
    return layers, host


def test_decode_stream_matches_single_calls_and_oracle(cuda_device):
    dts = [inputs.DTYPE_FP8_B128, inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128, inputs.DTYPE_BF16]
    layers, host = _chain(cuda_device, dts)
    ws = dl.Workspace.for_shapes([L.shape() for L in layers], cuda_device)
    # layer by layer through the single-call entry points
    singles = []
    for L in layers:
        if L.dtype == dl.BF16:
            dl.linear_bf16(L.x, L.w, L.bias, out=L.y, workspace=ws)
        else:
            dl.linear_fp8_block128(L.x, L.w, L.scales, L.bias, out=L.y, workspace=ws)
        singles.append(L.y.clone())
    torch.cuda.synchronize()
    st = torch.cuda.Stream()          # graph capture needs a non-default stream
    for use_graph in (False, True, True):
        for L in layers:
            L.y.fill_(0)
        torch.cuda.synchronize()
        dl.decode_stream(layers, ws, use_graph=use_graph, stream=st)
        st.synchronize()
        for i, L in enumerate(layers):
            assert torch.equal(L.y, singles[i]), (use_graph, i)
    # oracle, one layer at a time on the GPU's own input bytes
    for i, (L, Lh) in enumerate(zip(layers, host)):
        Lc = inputs.LayerInputs(Lh.dtype, Lh.M, Lh.N, Lh.K, L.x, Lh.w, Lh.scales, Lh.bias)
        ref, a = oracle_for(Lc)
        y32 = torch.empty(Lh.M, Lh.N, dtype=torch.float32, device=cuda_device)
        if L.dtype == dl.BF16:
            dl.linear_bf16(L.x, L.w, L.bias, out_f32=y32, workspace=ws)
        else:
            dl.linear_fp8_block128(L.x, L.w, L.scales, L.bias, out_f32=y32, workspace=ws)
        torch.cuda.synchronize()
        assert_parity(L.y, y32, ref, a, what=f"stream layer {i}")
    dl.graph_cache_clear()


def test_graph_replay_soak_stays_bitwise_constant(cuda_device):
    """Many back-to-back replays: the arrival tickets never drift (long-run check)."""
    dts = [inputs.DTYPE_FP8_B128, inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128]
    layers, _ = _chain(cuda_device, dts, M=1, seed=51)
    ws = dl.Workspace.for_shapes([L.shape() for L in layers], cuda_device)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        dl.decode_stream(layers, ws, use_graph=True, stream=st)
        st.synchronize()
        first = [L.y.clone() for L in layers]
        for _ in range(2000):
            dl.decode_stream(layers, ws, use_graph=True, stream=st)
        st.synchronize()
    for i, L in enumerate(layers):
        assert torch.equal(L.y, first[i]), i
    ticket_bytes = 4 * max((L.w.shape[0] + 127) // 128 for L in layers)
    assert torch.all(ws.tensor[:ticket_bytes] == 0)       # every arrival ticket reset
    dl.graph_cache_clear()


# ------------------------------------------------------------------ full-size workloads

QWEN = inputs.QWEN72B_SHAPES


def _full_layer(dtype, name, M, config_id, dev, layer_idx=0):
    N, K, bias = QWEN[name]
    return inputs.make_layer(dtype, M, N, K, bias=bias, config_id=config_id,
                             layer_idx=layer_idx, device=dev)


@pytest.mark.slow
@pytest.mark.parametrize("name", list(QWEN))
def test_qwen_layer_bf16_m1_sampled(cuda_device, name):
    """Qwen2.5-72B-shaped layer linears, BF16, M=1 (the launch the benchmark times)."""
    L = _full_layer(inputs.DTYPE_BF16, name, 1, 1, cuda_device)
    y, y32 = run_gpu(L, cuda_device)
    rows = sample_rows(L.N, seed=1)
    ref, a = oracle_for(L, rows=rows)
    assert_parity(y, y32, ref, a, rows=rows, what=f"bf16 {name}")


@pytest.mark.slow
@pytest.mark.parametrize("name", list(QWEN))
def test_qwen_layer_fp8_m6_sampled(cuda_device, name):
    """Same four shapes, weight-only FP8 block-128, M=6 (speculative verify step)."""
    L = _full_layer(inputs.DTYPE_FP8_B128, name, 6, 2, cuda_device)
    y, y32 = run_gpu(L, cuda_device)
    rows = sample_rows(L.N, seed=2)
    ref, a = oracle_for(L, rows=rows)
    assert_parity(y, y32, ref, a, rows=rows, what=f"fp8 {name}")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["qkv", "o"])
def test_qwen_layer_fp8_m1_sampled(cuda_device, name):
    """FP8 QKV (with bias) and O at M=1, the shapes of the whole-model stream
    (gate_up and down at M=1 are in the token sweep)."""
    L = _full_layer(inputs.DTYPE_FP8_B128, name, 1, 4, cuda_device)
    y, y32 = run_gpu(L, cuda_device)
    rows = sample_rows(L.N, seed=4)
    ref, a = oracle_for(L, rows=rows)
    assert_parity(y, y32, ref, a, rows=rows, what=f"fp8 M=1 {name}")


@pytest.mark.slow
@pytest.mark.parametrize("dtype", [inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128])
@pytest.mark.parametrize("name", ["gate_up", "down"])
def test_token_sweep_sampled(cuda_device, dtype, name):
    """M in {1,2,4,6,8,16} on gate_up and down."""
    base = _full_layer(dtype, name, 16, 3, cuda_device)
    rows = sample_rows(base.N, count=96, seed=3)
    for M in (1, 2, 4, 6, 8, 16):
        L = inputs.LayerInputs(dtype, M, base.N, base.K, base.x[:M].contiguous(), base.w,
                               base.scales, base.bias)
        y, y32 = run_gpu(L, cuda_device)
        ref, a = oracle_for(L, rows=rows)
        assert_parity(y, y32, ref, a, rows=rows, what=f"{dtype} {name} M={M}")


def test_device_error_word_clear(cuda_device):
    assert dl.device_status() == 0
