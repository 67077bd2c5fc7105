"""dl_linear_bf16_static_scratch: the entry point that allocates nothing and
keeps its split-K state in the library's static device scratch.  Checked
against the oracle at the acceptance tolerance and bit for bit against
dl_linear_bf16 (caller workspace: same plan, same kernel) on calls issued back
to back, so that each call starts from what the previous one left in the
shared scratch; and checked to allocate no device memory while it runs.

This file is collected last on purpose: it must pass in a fresh process (the
first call on the device does the scratch set-up) and after every other test
(the scratch and the overrides then carry earlier state)."""
import re

import numpy as np
import pytest
import torch

import oracle
import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs
from parity_util import ABS_TOL, REL_TOL, oracle_for

# (M, N, K, bias): split-K tiles with partial sums and a ragged tail; a second
# shape with more tiles (its tickets lie over the first call's partials); the
# first shape again.
CALLS = [(1, 4096, 8192, True), (6, 1000, 2048, False), (1, 4096, 8192, True)]


def _within_tolerance(y32, ref, a, what):
    """|y_f32 - y_ref| <= 2e-3 * sum|x w| + 1e-6 against the oracle's values."""
    g = y32.detach().cpu().double().numpy()
    bound = REL_TOL * a + ABS_TOL
    bad = ~(np.abs(g - ref) <= bound)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance"


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point(cuda_device):
    dl.set_override(0, 0, 0)
    host = [inputs.make_layer(inputs.DTYPE_BF16, M, N, K, bias=b, config_id=90 + (i % 2))
            for i, (M, N, K, b) in enumerate(CALLS)]
    dev = [L.to(cuda_device) for L in host]
    for L in dev:
        assert dl.workspace_bytes(L.M, L.N, L.K, dl.BF16) <= dl.STATIC_SCRATCH_BYTES
    outs = [(torch.empty((L.M, L.N), dtype=torch.bfloat16, device=cuda_device),
             torch.empty((L.M, L.N), dtype=torch.float32, device=cuda_device)) for L in dev]
    # Back to back on one stream, no host synchronisation in between.
    for L, (y, y32) in zip(dev, outs):
        dl.linear_bf16_static_scratch(L.x, L.w, L.bias, out=y, out_f32=y32)
    torch.cuda.synchronize(cuda_device)
    assert dl.device_status() == 0

    for i, (Lh, L, (y, y32)) in enumerate(zip(host, dev, outs)):
        ws = dl.Workspace(dl.workspace_bytes(L.M, L.N, L.K, dl.BF16), cuda_device)
        y32_ref = torch.empty_like(y32)
        y_ref = dl.linear_bf16(L.x, L.w, L.bias, out_f32=y32_ref, workspace=ws)
        torch.cuda.synchronize(cuda_device)
        ref, a = oracle_for(Lh)
        _within_tolerance(y32, ref, a, f"call {i} M={L.M} N={L.N} K={L.K}")
        # y is y_f32 rounded once to nearest even
        assert np.array_equal(oracle.round_to_bf16(y32.cpu().numpy()), inputs.bf16_bits(y))
        # the workspace entry point runs the same plan and kernel: the same bits
        assert torch.equal(y32, y32_ref) and torch.equal(y, y_ref), f"call {i}"
    # The third call repeats the first one's inputs after another shape used the
    # scratch: same plan, same kernel, so the same bits.
    assert torch.equal(outs[0][1], outs[2][1]) and torch.equal(outs[0][0], outs[2][0])


@pytest.mark.gpu
def test_static_scratch_allocates_nothing(cuda_device):
    """After a warm-up call, many calls leave the device's free memory and the
    caching allocator's counters exactly as they were."""
    dl.set_override(0, 0, 0)
    L = inputs.make_layer(inputs.DTYPE_BF16, 1, 4096, 8192, bias=True, config_id=92).to(cuda_device)
    y = torch.empty((1, 4096), dtype=torch.bfloat16, device=cuda_device)
    y32 = torch.empty((1, 4096), dtype=torch.float32, device=cuda_device)
    for _ in range(2):                                   # set-up happens here
        dl.linear_bf16_static_scratch(L.x, L.w, L.bias, out=y, out_f32=y32)
    torch.cuda.synchronize(cuda_device)
    first = y32.clone()
    free0, _ = torch.cuda.mem_get_info(cuda_device)
    stats0 = torch.cuda.memory_stats(cuda_device)
    for _ in range(50):
        dl.linear_bf16_static_scratch(L.x, L.w, L.bias, out=y, out_f32=y32)
    torch.cuda.synchronize(cuda_device)
    free1, _ = torch.cuda.mem_get_info(cuda_device)
    stats1 = torch.cuda.memory_stats(cuda_device)
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    for k in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
        assert stats1.get(k, 0) == stats0.get(k, 0), k
    assert torch.equal(y32, first)
    assert dl.device_status() == 0


@pytest.mark.gpu
def test_static_scratch_rejects_oversize_plans(cuda_device):
    dl.set_override(0, 0, 0)
    K = 8192
    # the largest N the library takes (16,384 tiles) splits into enough segments
    for M, N in [(9, 59136), (16, 152064), (16, 2097152)]:
        if dl.workspace_bytes(M, N, K, dl.BF16) > dl.STATIC_SCRATCH_BYTES:
            break
    else:
        pytest.skip("no candidate shape needs more scratch than the limit on this device")
    # contents are never read: the plan is rejected before anything is enqueued
    x = torch.empty((M, K), dtype=torch.bfloat16, device=cuda_device)
    w = torch.empty((N, K), dtype=torch.bfloat16, device=cuda_device)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(dl.DLError) as e:
        dl.linear_bf16_static_scratch(x, w, out=y)
    assert e.value.status == 4
    assert "static scratch" in str(e.value)


def test_static_scratch_limit_matches_header():
    text = open(dl._HEADER).read()
    m = re.search(r"#define\s+DL_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m and (int(m.group(1)) << int(m.group(2))) == dl.STATIC_SCRATCH_BYTES
