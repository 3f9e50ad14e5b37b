"""Parity of the persistent bf16 path (the whole sample as one cooperative
kernel, phases separated by a grid barrier) with the float64 oracle.

Same bars as the per-kernel bf16 path: final action max |delta| <= 1e-2 and
per-layer hidden relative L2 <= 1e-2 against the oracle; pad and mask variants
equal their unpadded run bitwise; and, because every unit of work is dealt in a
fixed order and every sum runs in a fixed order, two runs are bitwise equal.
Every test also checks that the sample really was one kernel launch.
"""
import os

import numpy as np
import pytest

from flow_matching_action_gb300 import synth

from .helpers import GpuRunner, oracle_actions, rel_l2, weights

pytestmark = pytest.mark.gpu

BF16_ACT_TOL, BF16_HID_TOL = 1e-2, 1e-2


def persistent_runner(dims, w, **kw):
    old = os.environ.get("AE_PERSIST")
    os.environ["AE_PERSIST"] = "1"
    try:
        return GpuRunner(dims, w, dtype="bf16", **kw)
    finally:
        if old is None:
            del os.environ["AE_PERSIST"]
        else:
            os.environ["AE_PERSIST"] = old


def run_one_launch(runner, wl, **kw):
    out = runner.run(wl, **kw)
    assert runner.expert.info()["launches_last_sample"] == 1
    return out


@pytest.fixture(scope="module")
def pi05_persist():
    r = persistent_runner(synth.PI05, weights("pi05"), max_batch=16, max_rows=2048)
    yield r
    r.close()


@pytest.fixture(scope="module")
def tiny_persist():
    r = persistent_runner(synth.TINY, weights("tiny"), max_batch=4, max_rows=256)
    yield r
    r.close()


def test_pi05_two_camera_matches_oracle(pi05_persist):
    wl = synth.pi05_two_camera()
    ref, ref_dump = oracle_actions(wl, weights("pi05"), dump=True)
    (got, dump) = run_one_launch(pi05_persist, wl, dump=True)
    assert np.abs(got - ref).max() <= BF16_ACT_TOL
    assert rel_l2(dump, ref_dump, axis=(2, 3, 4)).max() <= BF16_HID_TOL


def test_pi05_repeatable_and_masked_slot_bitwise(pi05_persist):
    a = run_one_launch(pi05_persist, synth.pi05_two_camera())
    b = run_one_launch(pi05_persist, synth.pi05_two_camera(), in_place=True)
    np.testing.assert_array_equal(a, b)
    masked = run_one_launch(pi05_persist, synth.pi05_masked_slot())
    assert np.isfinite(masked).all()
    np.testing.assert_array_equal(masked, a)


def test_pi05_padded_equals_unpadded_bitwise(pi05_persist):
    padded = run_one_launch(pi05_persist, synth.pi05_padded(0, padded=True))
    unpadded = run_one_launch(pi05_persist, synth.pi05_padded(0, padded=False))
    assert np.isfinite(padded).all()
    np.testing.assert_array_equal(padded, unpadded)
    ref = oracle_actions(synth.pi05_padded(0, padded=False), weights("pi05"))
    assert np.abs(padded - ref).max() <= BF16_ACT_TOL


def test_pi05_batched_ragged_sampled_requests(pi05_persist):
    wl = synth.pi05_batched(0)
    got = run_one_launch(pi05_persist, wl)
    assert np.isfinite(got).all()
    lens = wl.n_valid
    for b in (int(np.argmin(lens)), int(np.argmax(lens))):
        single = synth.pi05_request(0, b, lens[b])
        ref = oracle_actions(single, weights("pi05"))
        assert np.abs(got[b] - ref[0]).max() <= BF16_ACT_TOL


def test_tiny_head_dim_64_ragged_batch(tiny_persist):
    """head_dim 64 (the RoPE epilogue's direct-store form), a ragged batch with
    a masked slot and a request far longer than the others."""
    wl = synth.build_workload("b3", synth.TINY, 3, [[("v", 30)], [("v", 5), ("m", 3)], [("v", 200)]],
                              seed=4)
    got = run_one_launch(tiny_persist, wl)
    assert np.abs(got - oracle_actions(wl, weights("tiny"))).max() <= BF16_ACT_TOL


def test_tiny_empty_prefixes_and_single_step(tiny_persist):
    wl = synth.build_workload("e", synth.TINY, 1, [[("m", 7)], []], seed=5)
    got = run_one_launch(tiny_persist, wl)
    assert np.isfinite(got).all()
    assert np.abs(got - oracle_actions(wl, weights("tiny"))).max() <= BF16_ACT_TOL
