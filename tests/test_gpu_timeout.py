"""Failure detection without a fault: a bounded pipeline wait that runs out.

Every wait inside the pipelined kernels gives up after a limit, records
PA_DEV_ERR_TIMEOUT, lets the copies and tensor-core work in flight complete,
frees its tensor memory and returns ("vLLM V1 engine architecture", the
failure-handling section: a dead engine must be detected and reported, not
left hanging).  The test makes one wait run out on purpose: with the limit at
1 ms, CTA 0 of each pipelined kernel leaves out the copy of one pipeline
stage (pa_test_skip_copy), so the waits on that stage can only time out.
Nothing faults, traps or hangs.  The call must come back quickly with the
flag set, and the next ordinary step in the same process must be exact (its
kernels allocate tensor memory again, so a leak would show).
"""
import time

import pytest

import paged_kv_cache_82_gb300 as pa
from tests._gpu_step import gpu_step
from tests.test_gpu_parity import _check_step, _custom

pytestmark = pytest.mark.gpu

STEPS = {
    # head-group decode kernel: CTA 0 streams several stages
    "decode": lambda: _custom([(3000, 1)] * 8, 32, 8),
    # tensor-core prefill tiles (16 chunks of 128 keys per tile)
    "prefill": lambda: _custom([(2000, 1000)], 32, 8),
}


@pytest.mark.parametrize("kind", sorted(STEPS))
def test_a_wait_that_runs_out_is_reported_and_the_next_step_is_exact(kind):
    wl = STEPS[kind]()
    pa.pa_set_wait_limit_ns(1_000_000)   # 1 ms
    pa.pa_test_skip_copy(2)
    try:
        t0 = time.perf_counter()
        _, _, _, _, flags = gpu_step(wl)  # synchronises (device error read)
        elapsed = time.perf_counter() - t0
    finally:
        pa.pa_test_skip_copy(-1)
        pa.pa_set_wait_limit_ns(0)
    assert flags & pa.PA_DEV_ERR_TIMEOUT, hex(flags)
    assert elapsed < 5.0, elapsed
    # the context is usable and the same step is exact again
    _check_step(STEPS[kind]())


def test_wait_limit_and_hook_arguments():
    with pytest.raises(pa.PaError):
        pa.pa_set_wait_limit_ns(10)            # below 0.1 ms
    with pytest.raises(pa.PaError):
        pa.pa_test_skip_copy(-2)
    pa.pa_set_wait_limit_ns(0)
    pa.pa_test_skip_copy(-1)
    assert pa.pa_get_device_error() == 0
