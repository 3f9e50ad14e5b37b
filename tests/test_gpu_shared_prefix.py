"""Many action samples of one observation over one shared prefix (OxyGen,
"Cross-task KV Sharing": the prefill's KV is read in place by every consumer).

ae_bind_prefix_shared binds one request's prefix K/V for n samples, each with
its own noise.  Its result must equal ae_bind_prefix of n copies of the prefix
bitwise (the same kernels see the same values), and every sample must match
the oracle run on that prefix with the sample's noise: 1e-4 on the fp32 path,
final-action max |delta| <= 1e-2 on the bf16 path.
"""
import dataclasses

import numpy as np
import pytest

from flow_matching_action_gb300 import synth

from .helpers import GpuRunner, oracle_actions, weights

pytestmark = pytest.mark.gpu


def copies_of(wl, n_samples, noise_seed):
    """The request of `wl` repeated n_samples times (prefix rows copied), with
    a fresh noise per sample: what the shared binding must reproduce."""
    assert wl.batch == 1
    rows = wl.n_rows[0]
    d = wl.dims
    noise = np.stack([synth.request_noise(d, noise_seed, s) for s in range(n_samples)])
    return dataclasses.replace(
        wl, name=wl.name + f"_x{n_samples}", layouts=[list(wl.layouts[0]) for _ in range(n_samples)],
        prefix_k=np.concatenate([wl.prefix_k] * n_samples, axis=1),
        prefix_v=np.concatenate([wl.prefix_v] * n_samples, axis=1),
        mask=np.concatenate([wl.mask] * n_samples),
        cu_lens=np.arange(n_samples + 1, dtype=np.int32) * rows, noise=noise)


def run_shared(runner, wl, noise):
    import torch
    k, v, mask, _ = runner.upload(wl)
    x = torch.from_numpy(np.ascontiguousarray(noise)).cuda()
    runner.expert.bind_prefix_shared(noise.shape[0], k, v, wl.n_rows[0], mask)
    out = torch.empty_like(x)
    runner.expert.sample(x, wl.n_steps, out)
    runner.expert.synchronize()
    runner._keep = (k, v, mask, x)
    return out.cpu().numpy().astype(np.float64)


def test_tiny_f32_shared_prefix_matches_oracle_and_copies():
    wl = synth.tiny_variant("masked")
    many = copies_of(wl, 3, noise_seed=11)
    r = GpuRunner(synth.TINY, weights("tiny"), max_batch=4, max_rows=256)
    try:
        shared = run_shared(r, wl, many.noise)
        copied = r.run(many)
    finally:
        r.close()
    np.testing.assert_array_equal(shared, copied)
    assert np.abs(shared - oracle_actions(many, weights("tiny"))).max() <= 1e-4
    # different noise, same prefix: the samples differ
    assert np.abs(shared[0] - shared[1]).max() > 1e-3


@pytest.mark.parametrize("layout", ["two_camera", "masked_slot"])
def test_pi05_bf16_shared_prefix(layout):
    wl = synth.pi05_two_camera() if layout == "two_camera" else synth.pi05_masked_slot()
    many = copies_of(wl, 4, noise_seed=21)
    r = GpuRunner(synth.PI05, weights("pi05"), max_batch=4, max_rows=4096)
    try:
        shared = run_shared(r, wl, many.noise)
        copied = r.run(many)
    finally:
        r.close()
    assert np.isfinite(shared).all()
    np.testing.assert_array_equal(shared, copied)
    if layout == "two_camera":
        # first and last sample against the oracle on their own
        for s in (0, 3):
            one = dataclasses.replace(wl, noise=many.noise[s:s + 1])
            ref = oracle_actions(one, weights("pi05"))
            assert np.abs(shared[s] - ref[0]).max() <= 1e-2, s


def test_shared_prefix_host_checks():
    from flow_matching_action_gb300 import ae
    r = GpuRunner(synth.TINY, weights("tiny"), max_batch=2, max_rows=64)
    try:
        ctx = r.expert.ctx
        with pytest.raises(ae.AEError) as e:
            ae.ae_bind_prefix_shared(ctx, 3, None, None, 10)
        assert e.value.status == -2  # more samples than max_batch
        with pytest.raises(ae.AEError) as e:
            ae.ae_bind_prefix_shared(ctx, 1, None, None, 65)
        assert e.value.status == -2  # longer than max_prefix_rows
        with pytest.raises(ae.AEError) as e:
            ae.ae_bind_prefix_shared(ctx, 1, None, None, 10)
        assert e.value.status == -1  # rows but no K / V
        ae.ae_bind_prefix_shared(ctx, 0, None, None, 0)  # nothing bound: legal
    finally:
        r.close()
