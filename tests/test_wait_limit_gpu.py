"""The bounded device waits: a wait that runs out returns an error status
instead of hanging, and the context stays usable.

Every device-side wait of the kernel gives up after a limit, ORs a bit into
the device error word and lets its CTA leave (the bounded barrier waits that
guard against a barrier that drifts over a long run, "Developing a custom
Qwen2.5 72B inference engine from scratch", §7).  Here the limit is shortened
to 20 ms and CTA 0 withholds the copies of one pipeline stage -- the stage's
barrier expects bytes that nobody sends, a flag that nothing sets -- so its
consumers' wait runs out.  Nothing is in flight for the withheld stage, so the
CTA can leave safely.  The test checks that the call returns, that
dl_device_status reports the consumer-wait bit, and that the next normal call
on the same workspace, once its zero prefix is reset, matches the oracle.
"""
import time

import pytest
import torch

import weight_streaming_skinny_gb300 as dl
from weight_streaming_skinny_gb300 import inputs
from parity_util import assert_parity, oracle_for, run_gpu

pytestmark = pytest.mark.gpu

WAIT_NS = 20_000_000          # 20 ms
CONSUMER_WAIT_BIT = 1


@pytest.fixture(autouse=True)
def _reset_hooks():
    dl.set_override(0, 0, 0)
    dl.set_wait_test(0, 0)
    yield
    dl.set_wait_test(0, 0)
    dl.set_override(0, 0, 0)


@pytest.mark.parametrize("dtype,M,withhold", [(inputs.DTYPE_BF16, 1, 2),
                                              (inputs.DTYPE_FP8_B128, 6, 2),
                                              (inputs.DTYPE_FP8_B128, 1, 5)])
def test_withheld_stage_runs_out_and_reports(cuda_device, dtype, M, withhold):
    assert dl.device_status() == 0
    # 32 tiles x 8192 columns: CTA 0 streams at least 6 stages (a single FP8
    # call prefetches its first 3 before the dependency wait, so withholding
    # stage 2 covers that path and stage 5 the main loop).
    N, K = 4096, 8192
    L = inputs.make_layer(dtype, M, N, K, bias=True, config_id=95).to(cuda_device)
    ws = dl.Workspace(dl.workspace_bytes(M, N, K,
                                         dl.BF16 if dtype == inputs.DTYPE_BF16 else dl.FP8_B128),
                      cuda_device)
    dl.set_wait_test(WAIT_NS, withhold)
    t0 = time.perf_counter()
    run_gpu(L, cuda_device, workspace=ws)          # returns: launch OK, device synchronised
    elapsed = time.perf_counter() - t0
    dl.set_wait_test(0, 0)
    flags = dl.device_status()
    assert flags & CONSUMER_WAIT_BIT, f"error word 0x{flags:x}: the consumers' wait did not run out"
    assert elapsed < 5.0, f"the call took {elapsed:.2f} s with a 20 ms wait limit"
    assert dl.device_status() == 0                 # read and cleared
    # The same workspace after its arrival counters are zeroed again: correct.
    ws.reset()
    y, y32 = run_gpu(L, cuda_device, workspace=ws)
    ref, a = oracle_for(L)
    assert_parity(y, y32, ref, a, what=f"{dtype} M={M} after a withheld stage")
    assert dl.device_status() == 0


def test_wait_limit_alone_changes_nothing(cuda_device):
    """A short limit with nothing withheld: no wait runs out, results exact."""
    L = inputs.make_layer(inputs.DTYPE_FP8_B128, 6, 1000, 2048, bias=True, config_id=96)
    Ld = L.to(cuda_device)
    y0, y320 = run_gpu(Ld, cuda_device)
    dl.set_wait_test(WAIT_NS, 0)
    y1, y321 = run_gpu(Ld, cuda_device)
    dl.set_wait_test(0, 0)
    assert dl.device_status() == 0
    assert torch.equal(y320, y321) and torch.equal(y0, y1)

