"""Failure detection on the GPU without a fault: the pipeline wait that every
decode and prefill kernel uses gives up after its limit on a barrier that
nothing completes, the CTA's other warps drain through its abort flag, the
device status word reports PKV_DEV_TIMEOUT, and the context keeps running
ticks that match the oracle."""
import time

import pytest
import torch

from paged_kv_attention_mapping_gb300 import binding
from paged_kv_attention_mapping_gb300 import workloads as W

from test_gpu_parity import run_and_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def test_bounded_wait_gives_up_and_reports(dev):
    assert binding.device_status() == 0
    result = torch.full((2,), -1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    binding.selftest_bounded_wait(20000, result)  # 20 ms for the producer warp; 2 s for the others
    st = binding.device_status()                  # waits for the stream
    dt = time.perf_counter() - t0
    assert st == binding.DEV_TIMEOUT
    assert dt >= 0.015, dt
    assert dt < 1.0, dt                           # the other warps left through the abort flag, not their own limit
    err_word, drained = (int(x) for x in result.cpu())
    assert err_word == binding.DEV_TIMEOUT
    assert drained == 10                          # every warp of the CTA returned without its barrier
    # the status was read and cleared; the context still runs a tick exactly
    assert binding.device_status() == 0
    w = W.random_workload(41, 4, 8, 2, 64, 16, "bf16", (1, 70), 200)
    run_and_compare(w, dev)
    assert binding.device_status() == 0


def test_bounded_wait_rejects_limits_outside_its_range(dev):
    for bad in (0, -5, 1000001):
        with pytest.raises(RuntimeError):
            binding.selftest_bounded_wait(bad)
    assert binding.device_status() == 0
