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

from .helpers import GpuRunner, golden_b16, oracle_actions, weights

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
    oracle = oracle_actions(wl, weights("pi05"))
    for out in outs[:2]:
        assert np.isfinite(out).all()
        assert np.abs(out - ref).max() <= BF16_ACT_TOL
        assert np.abs(out - oracle).max() <= BF16_ACT_TOL
    assert free[1] == free[2]


def test_noalloc_pi05_batch_of_16():
    """At batch 16 the fixed scratch holds fewer attention work units than
    ae_sample would use, so the planner gives each CTA a longer range of key
    chunks; the result must still match ae_sample and the oracle."""
    wl = synth.pi05_batched(0)
    ref, outs, free = _run_pair(synth.PI05, weights("pi05"), wl, max_rows=2048)
    oracle = golden_b16(0)
    for out in outs[:2]:
        assert np.isfinite(out).all()
        assert np.abs(out - ref).max() <= BF16_ACT_TOL
        assert np.abs(out - oracle).max() <= BF16_ACT_TOL
    assert free[1] == free[2]


def test_noalloc_rejects_a_batch_beyond_the_fixed_scratch():
    """32 requests of 4 query tiles each need 128 attention work units; the
    16 MiB array holds 127 at head_dim 256."""
    import torch
    from flow_matching_action_gb300 import ae
    wl = synth.build_workload("b32", synth.PI05, 1, [[("v", 8)]] * 32, seed=2)
    r = GpuRunner(synth.PI05, weights("pi05"), max_batch=32, max_rows=8)
    try:
        k, v, mask, noise = r.upload(wl)
        r.expert.bind_prefix(k, v, [int(c) for c in wl.cu_lens], mask)
        out = torch.empty_like(noise)
        ae.ae_sample(r.expert.ctx, noise, 1, out)  # builds the table; allowed to allocate
        with pytest.raises(ae.AEError) as e:
            ae.ae_sample_noalloc(r.expert.ctx, noise, 1, out)
        assert e.value.status == -2
        r.expert.synchronize()
    finally:
        r.close()


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
