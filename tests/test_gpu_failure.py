"""Failure detection on the GPU without a fault: every kernel's waits are bounded, and a wait
that runs out records TQ_ERR_TIMEOUT in the context's device error word and returns. The
self-test entry point runs exactly that path on a barrier nothing completes; the context must
then report the timeout once, and go on decoding correctly."""

import time

import numpy as np
import pytest
import torch

from quantised_kv_cache_gb300 import tq
from quantised_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_kv_cache_gb300 import build
    build.build()


def _decode(ctx, seed):
    w = wl.Workload(99, "fail", 2, 4, 4, 200, torch.float32, "KQV", 4, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, DEV, seed=seed)
    cache = tq.Cache(ctx, 2, 4, 256, device=DEV)
    tq.tq_append_quantize(ctx.handle, cache, k, v, torch.zeros(2, dtype=torch.int32, device=DEV))
    lens = torch.full((2,), 200, dtype=torch.int32, device=DEV)
    return tq.tq_decode_attention(ctx.handle, cache, q, lens, 256).cpu().numpy()


def test_a_wait_that_runs_out_reports_a_timeout_and_the_context_stays_usable():
    ctx = tq.Context(128, 4, "KQV", 5)
    before = _decode(ctx, 1)
    assert tq.tq_get_device_error(ctx.handle) == 0
    t0 = time.perf_counter()
    tq.tq_selftest_bounded_wait(ctx.handle, 5_000_000)  # 5 ms
    assert tq.tq_get_device_error(ctx.handle) == tq.TQ_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.004 < elapsed < 2.0, elapsed  # the wait lasted its budget, not more
    assert tq.tq_get_device_error(ctx.handle) == 0  # read and cleared
    after = _decode(ctx, 1)
    np.testing.assert_array_equal(before, after)
    assert tq.tq_get_device_error(ctx.handle) == 0
    ctx.close()


def test_the_self_test_refuses_a_budget_above_the_kernels_own():
    ctx = tq.Context(128, 4, "KQV", 5)
    with pytest.raises(tq.TQError) as e:
        tq.tq_selftest_bounded_wait(ctx.handle, 3_000_000_000)
    assert e.value.status == tq.TQ_ERR_ARG
    ctx.close()
