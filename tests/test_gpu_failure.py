"""Device-side failure detection: the bounded wait that every kernel of the
library uses gives up after its limit, records PLX_ERR_TIMEOUT in the device
status word and returns, and the device stays usable.  The wait runs out on a
barrier that nothing arrives on, in a one-thread kernel with nothing
asynchronous in flight (plx_selftest_wait); no test faults, traps or hangs the
GPU."""
import time

import numpy as np
import pytest

import plx_inputs
from parity import assert_f32

PLX_ERR_TIMEOUT = 5


@pytest.mark.gpu
def test_a_wait_that_completes_leaves_the_status_word_clear():
    import parameterized_local_linear_02_b300 as plx
    plx.plx_last_device_error()            # start from a clear word
    plx.plx_selftest_wait(1000, arrive=True)
    assert plx.plx_last_device_error() == 0


@pytest.mark.gpu
def test_a_wait_that_runs_out_reports_a_timeout_and_the_device_stays_usable():
    import torch
    import oracle
    import parameterized_local_linear_02_b300 as plx
    plx.plx_last_device_error()
    t0 = time.perf_counter()
    plx.plx_selftest_wait(20000, arrive=False)       # 20 ms, nothing arrives
    assert plx.plx_last_device_error() == PLX_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.015 <= elapsed < 2.0, f"the wait gave up after {elapsed:.3f} s"
    # the status word was cleared by the read, and the next calls compute normally
    assert plx.plx_last_device_error() == 0
    x = plx_inputs.decode(2, 2, 128, 300, seed=81, seqlens=np.array([300, 77]))
    t = x.device_tensors("cuda")
    out, _ = plx.plx_decode(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"], num_splits=2,
                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    res = oracle.decode("stream", x.q, x.rho, x.k_cache, x.v_cache, x.seqlens, x.scale)
    ref = np.stack([res[(b, h)][0] for b in range(2) for h in range(2)]).reshape(2, 2, 128)
    assert_f32(out.cpu().numpy(), ref, "decode after a device-side timeout")
