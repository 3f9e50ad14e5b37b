"""Device-side failure detection, exercised without faulting or hanging the GPU.

The tensor-core kernels bound every mbarrier wait by a cycle budget; a wait that
runs out records a timeout in the context's sticky status and its kernel
returns.  ae_selftest_wait_timeout runs that same bounded wait on an mbarrier
that nothing completes (no copy or MMA in flight), with a short budget, so the
give-up path runs for real: the status becomes sticky, the host reports
AE_ERR_DEVICE, and a fresh context on the same GPU still samples correctly.
"""
import dataclasses

import numpy as np
import pytest

from flow_matching_action_gb300 import synth

from .helpers import GpuRunner, oracle_actions

pytestmark = pytest.mark.gpu

AE_ERR_DEVICE = -5


def test_wait_timeout_is_sticky_and_a_fresh_context_works():
    import torch
    from flow_matching_action_gb300 import ae
    dims = dataclasses.replace(synth.TINY, dtype="bf16")
    w = synth.make_weights(dims, 0)
    wl = synth.tiny_variant("masked")
    r = GpuRunner(dims, w, max_batch=1, max_rows=64)
    try:
        before = r.run(wl)  # the context works before the self-test
        ae.ae_selftest_wait_timeout(r.expert.ctx, 200_000)  # ~0.1 ms budget
        with pytest.raises(ae.AEError) as e:
            r.expert.synchronize()
        assert e.value.status == AE_ERR_DEVICE
        k, v, mask, noise = r.upload(wl)
        with pytest.raises(ae.AEError) as e:
            r.expert.sample(noise, wl.n_steps, torch.empty_like(noise))
        assert e.value.status == AE_ERR_DEVICE
        with pytest.raises(ae.AEError) as e:  # sticky: still reported
            r.expert.synchronize()
        assert e.value.status == AE_ERR_DEVICE
    finally:
        r.close()
    r2 = GpuRunner(dims, w, max_batch=1, max_rows=64)
    try:
        after = r2.run(wl)
    finally:
        r2.close()
    np.testing.assert_array_equal(after, before)
    assert np.abs(after - oracle_actions(wl, w)).max() <= 1e-2


def test_selftest_rejects_negative_budget():
    from flow_matching_action_gb300 import ae
    dims = dataclasses.replace(synth.TINY, dtype="bf16")
    r = GpuRunner(dims, synth.make_weights(dims, 0), max_batch=1, max_rows=8)
    try:
        with pytest.raises(ae.AEError) as e:
            ae.ae_selftest_wait_timeout(r.expert.ctx, -1)
        assert e.value.status == -1
        r.expert.synchronize()  # nothing was launched: the context is clean
    finally:
        r.close()
