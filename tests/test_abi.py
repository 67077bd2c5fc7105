"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments before any CUDA call (host-side failure tests; no GPU needed)."""
import ctypes

import pytest
import torch

import weight_streaming_skinny_gb300 as dl

EXPECTED = {"dl_workspace_bytes", "dl_linear_bf16", "dl_linear_fp8_block128", "dl_decode_stream",
            "dl_graph_cache_clear", "dl_set_override", "dl_device_status", "dl_last_error",
            "dl_version", "dl_linear_swiglu", "dl_linear_bf16_static_scratch", "dl_linear_argmax",
            "dl_decode_stream_workspace_bytes", "dl_decode_stream_launches", "dl_set_wait_test",
            "dl_graph_cache_size"}


def test_library_exports_every_header_symbol():
    declared = set(dl.header_symbols())
    assert EXPECTED <= declared
    assert set(dl.exported_symbols()) == declared


def test_version():
    import re
    m = re.search(r"#define\s+DL_VERSION\s+(\d+)", open(dl._HEADER).read())
    assert m and dl.version() == int(m.group(1)) == dl.ABI_VERSION


# fake, well-aligned device addresses: never dereferenced, validation fails first
X, W, Y, S, B, WS = (0x10000 * (i + 1) for i in range(6))


def _bf16(x=X, w=W, bias=None, y=Y, yf=None, M=1, N=128, K=128, ws=WS, nbytes=1 << 20):
    lib = dl.load()
    return lib.dl_linear_bf16(x, w, bias, y, yf, M, N, K, ws, nbytes, None)


def _fp8(x=X, w=W, s=S, bias=None, y=Y, M=1, N=128, K=128, ws=WS, nbytes=1 << 20):
    lib = dl.load()
    return lib.dl_linear_fp8_block128(x, w, s, bias, y, None, M, N, K, ws, nbytes, None)


@pytest.mark.parametrize("M", [0, -1, 17, 1000])
def test_rejects_M_outside_decode_range(M):
    assert _bf16(M=M) == 2
    assert _fp8(M=M) == 2
    assert b"M=" in dl.load().dl_last_error()


def test_rejects_bad_K_and_N():
    assert _bf16(K=12) == 2        # bf16 needs K % 8 == 0
    assert _fp8(K=136) == 2        # FP8 needs K % 128 == 0
    assert _bf16(N=0) == 2
    assert _bf16(K=0) == 2


def test_rejects_null_pointers():
    assert _bf16(x=None) == 1
    assert _bf16(w=None) == 1
    assert _bf16(y=None) == 1
    assert _fp8(s=None) == 1
    assert _bf16(ws=None) == 4


def test_rejects_misaligned_pointers():
    assert _bf16(x=X + 8) == 3
    assert _bf16(w=W + 2) == 3
    assert _bf16(y=Y + 1) == 3
    assert _bf16(bias=B + 1) == 3
    assert _bf16(yf=Y + 2) == 3
    assert _fp8(s=S + 2) == 3


def test_workspace_bytes_zero_for_invalid_shapes():
    lib = dl.load()
    assert lib.dl_workspace_bytes(0, 128, 128, 0) == 0
    assert lib.dl_workspace_bytes(17, 128, 128, 0) == 0
    assert lib.dl_workspace_bytes(1, 128, 100, 1) == 0
    assert lib.dl_workspace_bytes(1, 128, 128, 7) == 0


def test_override_validation():
    lib = dl.load()
    assert lib.dl_set_override(4, 0, 0) == 1
    assert lib.dl_set_override(0, 3, 0) == 1
    assert lib.dl_set_override(0, 0, -1) == 1
    assert lib.dl_set_override(0, 0, 0) == 0


def test_decode_stream_validates_every_layer_before_launching():
    lib = dl.load()
    good = dl._Layer(0, 1, 128, 128, X, W, None, None, Y)
    bad = dl._Layer(1, 1, 128, 100, X, W, S, None, Y)      # FP8 with K % 128 != 0
    arr = (dl._Layer * 2)(good, bad)
    assert lib.dl_decode_stream(arr, 2, WS, 1 << 20, None, 0) == 2
    assert b"layer 1" in lib.dl_last_error()
    assert lib.dl_decode_stream(None, 1, WS, 1 << 20, None, 0) == 1
    assert lib.dl_decode_stream(arr, 1, WS, 1 << 20, None, 5) == 1
    assert lib.dl_decode_stream(arr, 0, None, 0, None, 0) == 0     # empty list: nothing to do


def test_python_binding_refuses_cpu_tensors():
    x = torch.zeros(1, 128, dtype=torch.bfloat16)
    w = torch.zeros(128, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        dl.linear_bf16(x, w)
    with pytest.raises(ValueError, match="CUDA"):
        dl.linear_fp8_block128(x, torch.zeros(128, 128, dtype=torch.uint8),
                               torch.ones(1, 1))


def test_error_message_is_thread_local_and_cleared():
    lib = dl.load()
    assert _bf16(M=99) == 2
    assert lib.dl_last_error() != b""
    assert lib.dl_set_override(0, 0, 0) == 0
    assert lib.dl_last_error() == b""
    # dl_layer: 4 ints, 5 pointers, int act (+ 4 bytes of tail padding)
    assert ctypes.sizeof(dl._Layer) == 4 * 4 + 5 * 8 + 8
    assert dl._Layer.act.offset == 4 * 4 + 5 * 8


def test_workspace_zero_prefix_matches_header():
    import re
    text = open(dl._HEADER).read()
    m = re.search(r"#define\s+DL_WORKSPACE_ZERO_BYTES\s+\((\d+)u\s*\+\s*(\d+)u\s*\*\s*(\d+)u\)", text)
    assert m and int(m.group(1)) + int(m.group(2)) * int(m.group(3)) == dl.WORKSPACE_ZERO_BYTES


def test_swiglu_validation_before_any_cuda_call():
    """Bad SwiGLU arguments fail on the host: unknown dtype, N not a multiple of 16."""
    lib = dl.load()
    p = ctypes.c_void_p(1 << 20)
    ws = ctypes.c_void_p(1 << 24)
    assert lib.dl_linear_swiglu(7, p, p, None, None, p, None, 1, 32, 128, ws, 1 << 20, None) == 1
    assert lib.dl_linear_swiglu(0, p, p, None, None, p, None, 1, 40, 128, ws, 1 << 20, None) == 2
    assert b"16" in lib.dl_last_error()


def test_interleave_gate_up_layout():
    g = torch.arange(24 * 2, dtype=torch.float32).reshape(24, 2)
    u = -g - 1
    w = dl.interleave_gate_up(g, u)
    for j in range(24):
        b, i = divmod(j, 8)
        assert torch.equal(w[16 * b + i], g[j]) and torch.equal(w[16 * b + 8 + i], u[j])


def test_argmax_validation_before_any_cuda_call():
    """idx is required and aligned; y may be omitted (host-side checks only)."""
    lib = dl.load()
    p = ctypes.c_void_p(1 << 20)
    ws = ctypes.c_void_p(1 << 24)
    assert lib.dl_linear_argmax(0, p, p, None, None, None, None, None, None, 1, 256, 128, ws,
                                1 << 20, None) == 1
    assert lib.dl_linear_argmax(0, p, p, None, None, ctypes.c_void_p((1 << 20) + 2), None, None,
                                None, 1, 256, 128, ws, 1 << 20, None) == 3
    assert lib.dl_linear_argmax(0, p, p, None, None, p, None, None, None, 17, 256, 128, ws,
                                1 << 20, None) == 2


def test_wait_test_hook_validation():
    """The bounded-wait test hooks: a withheld stage needs a short wait limit."""
    lib = dl.load()
    assert lib.dl_set_wait_test(-1, 0) == 1
    assert lib.dl_set_wait_test(0, -1) == 1
    assert lib.dl_set_wait_test(0, 2) == 1               # withholding needs a limit ...
    assert lib.dl_set_wait_test(10**9, 2) == 1           # ... of at most 100 ms
    assert b"100 ms" in lib.dl_last_error()
    assert lib.dl_set_wait_test(20_000_000, 2) == 0
    assert lib.dl_set_wait_test(0, 0) == 0


def test_graph_cache_empty_without_a_gpu_call():
    dl.graph_cache_clear()
    assert dl.graph_cache_size() == 0
