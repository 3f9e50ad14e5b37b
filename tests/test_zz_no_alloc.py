"""ae_sample_noalloc: sampling for callers that cannot allocate device memory.

Callers that sample while a CUDA stream capture is open, under a device-memory
budget owned by someone else, or inside a control loop that forbids allocator
calls after start-up need a sampling call that never allocates.  This file
checks, through the C ABI, that ae_sample_noalloc gives the same actions as
ae_sample (within the bf16 tolerance of the parity tests) on two calls in a
row, and that its second and third calls leave the device's free memory
unchanged.  It sits last in collection order on purpose.
"""
import dataclasses

import numpy as np
import pytest

from flow_matching_action_gb300 import synth

from .helpers import GpuRunner, weights

pytestmark = pytest.mark.gpu

BF16_ACT_TOL = 1e-2


def _run_pair(dims, w, wl, max_rows):
    import torch
    from flow_matching_action_gb300 import ae
    r = GpuRunner(dims, w, max_batch=wl.batch, max_rows=max_rows)
    try:
        k, v, mask, noise = r.upload(wl)
        r.expert.bind_prefix(k, v, [int(c) for c in wl.cu_lens], mask)
        ref = torch.empty_like(noise)
        ae.ae_sample(r.expert.ctx, noise, wl.n_steps, ref)  # also builds the time table
        outs = []
        free = []
        for _ in range(3):
            out = torch.full_like(noise, float("nan"))
            ae.ae_sample_noalloc(r.expert.ctx, noise, wl.n_steps, out)
            torch.cuda.synchronize()
            ae.ae_synchronize(r.expert.ctx)
            free.append(torch.cuda.mem_get_info()[0])
            outs.append(out.cpu().numpy().astype(np.float64))
        return ref.cpu().numpy().astype(np.float64), outs, free
    finally:
        r.close()


def test_noalloc_matches_sample_tiny_bf16():
    dims = dataclasses.replace(synth.TINY, dtype="bf16")
    w = synth.make_weights(dims, 0)
    wl = synth.build_workload("na", dims, 2, [[("v", 40), ("m", 8), ("v", 16)], [("v", 30)]], seed=3)
    ref, outs, free = _run_pair(dims, w, wl, max_rows=64)
    for out in outs[:2]:
        assert np.isfinite(out).all()
        assert np.abs(out - ref).max() <= BF16_ACT_TOL
    assert free[1] == free[2]


def test_noalloc_matches_sample_pi05_two_camera():
    wl = synth.pi05_two_camera()
    ref, outs, free = _run_pair(synth.PI05, weights("pi05"), wl, max_rows=712)
    for out in outs[:2]:
        assert np.isfinite(out).all()
        assert np.abs(out - ref).max() <= BF16_ACT_TOL
    assert free[1] == free[2]


def test_noalloc_rejects_unprepared_steps_and_fp32():
    import torch
    from flow_matching_action_gb300 import ae
    dims = dataclasses.replace(synth.TINY, dtype="bf16")
    wl = synth.tiny_variant("plain")
    r = GpuRunner(dims, synth.make_weights(dims, 0), max_batch=1, max_rows=64)
    try:
        k, v, mask, noise = r.upload(wl)
        r.expert.bind_prefix(k, v, [int(c) for c in wl.cu_lens], mask)
        out = torch.empty_like(noise)
        with pytest.raises(ae.AEError) as e:
            ae.ae_sample_noalloc(r.expert.ctx, noise, 3, out)  # no table for 3 steps yet
        assert e.value.status == -3
    finally:
        r.close()
    r = GpuRunner(synth.TINY, weights("tiny"), max_batch=1, max_rows=64)
    try:
        k, v, mask, noise = r.upload(wl)
        r.expert.bind_prefix(k, v, [int(c) for c in wl.cu_lens], mask)
        with pytest.raises(ae.AEError) as e:
            ae.ae_sample_noalloc(r.expert.ctx, noise, 2, torch.empty_like(noise))
        assert e.value.status == -7
    finally:
        r.close()
