"""Parity at the size limits the library accepts.

N up to 2,097,152 rows (16,384 tiles of 128), one row less for a ragged last
tile, a K of 262,144 columns (2,048 K blocks: many K units per tile and the
largest minimum segment), and rejection just past the N limit.  Outputs are
compared with the oracle (sampled rows for the tall layers, every row for the
long-K one), within the acceptance tolerance, y == RNE(y_f32).
"""
import numpy as np
import pytest
import torch

import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs
from parity_util import assert_parity, oracle_for, run_gpu, sample_rows

pytestmark = pytest.mark.gpu

BF, F8 = inputs.DTYPE_BF16, inputs.DTYPE_FP8_B128
N_MAX = 16384 * 128


@pytest.mark.parametrize("N", [N_MAX, N_MAX - 1])
@pytest.mark.parametrize("dtype", [BF, F8])
def test_tallest_layer_sampled(cuda_device, dtype, N):
    dl.set_override(0, 0, 0)
    L = inputs.make_layer(dtype, 2, N, 128, bias=True, config_id=110, device=cuda_device)
    y, y32 = run_gpu(L, cuda_device)
    rows = np.union1d(sample_rows(N, count=256, seed=11), np.array([N - 1, N - 2, 128 * 16383]))
    ref, a = oracle_for(L, rows=rows)
    assert_parity(y, y32, ref, a, rows=rows, what=f"{dtype} N={N}")
    assert dl.device_status() == 0


@pytest.mark.parametrize("dtype", [BF, F8])
def test_longest_k(cuda_device, dtype):
    dl.set_override(0, 0, 0)
    L = inputs.make_layer(dtype, 3, 256, 262144, bias=False, config_id=111, device=cuda_device)
    y, y32 = run_gpu(L, cuda_device)
    ref, a = oracle_for(L)
    assert_parity(y, y32, ref, a, what=f"{dtype} K=262144")
    assert dl.device_status() == 0


@pytest.mark.parametrize("dtype", [BF, F8])
def test_one_row_past_the_limit_is_rejected(cuda_device, dtype):
    dev = cuda_device
    N, K = N_MAX + 1, 128
    x = torch.zeros((1, K), dtype=torch.bfloat16, device=dev)
    y = torch.empty((1, N), dtype=torch.bfloat16, device=dev)
    assert dl.workspace_bytes(1, N, K, dl.BF16 if dtype == BF else dl.FP8_B128) == 0
    ws = dl.Workspace(1 << 20, dev)
    with pytest.raises(dl.DLError) as e:
        if dtype == BF:
            w = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
            dl.linear_bf16(x, w, out=y, workspace=ws)
        else:
            w = torch.empty((N, K), dtype=torch.uint8, device=dev)
            s = torch.ones(((N + 127) // 128, 1), dtype=torch.float32, device=dev)
            dl.linear_fp8_block128(x, w, s, out=y, workspace=ws)
    assert e.value.status == 2
