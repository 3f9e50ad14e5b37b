"""Parity of the pipelined attention kernel (eight warps, S double buffered in
TMEM, separate K and V buffers) with the float64 oracle, through the C ABI.

Same bars as the rest of the bf16 path: final action max |delta| <= 1e-2 and
per-layer hidden relative L2 <= 1e-2 against the oracle; pad and mask
variants equal their unpadded run bitwise.  The batch of 16 ragged requests
gives every work unit several chunks, so the K/V and S pipelines turn over;
the tiny expert covers head_dim 64 and gathered chunks with action rows.
"""
import os

import numpy as np
import pytest

from flow_matching_action_gb300 import synth

from .helpers import GpuRunner, oracle_actions, rel_l2, weights

pytestmark = pytest.mark.gpu

BF16_ACT_TOL, BF16_HID_TOL = 1e-2, 1e-2


def pipe_runner(dims, w, **kw):
    old = os.environ.get("AE_ATTN_PIPE")
    os.environ["AE_ATTN_PIPE"] = "1"
    try:
        return GpuRunner(dims, w, dtype="bf16", **kw)
    finally:
        if old is None:
            del os.environ["AE_ATTN_PIPE"]
        else:
            os.environ["AE_ATTN_PIPE"] = old


@pytest.fixture(scope="module")
def pi05_pipe():
    r = pipe_runner(synth.PI05, weights("pi05"), max_batch=16, max_rows=2048)
    yield r
    r.close()


@pytest.fixture(scope="module")
def tiny_pipe():
    r = pipe_runner(synth.TINY, weights("tiny"), max_batch=4, max_rows=256)
    yield r
    r.close()


def test_pi05_two_camera_matches_oracle(pi05_pipe):
    wl = synth.pi05_two_camera()
    ref, ref_dump = oracle_actions(wl, weights("pi05"), dump=True)
    got, dump = pi05_pipe.run(wl, dump=True)
    assert np.abs(got - ref).max() <= BF16_ACT_TOL
    assert rel_l2(dump, ref_dump, axis=(2, 3, 4)).max() <= BF16_HID_TOL


def test_pi05_masked_slot_and_padding_bitwise(pi05_pipe):
    base = pi05_pipe.run(synth.pi05_two_camera())
    masked = pi05_pipe.run(synth.pi05_masked_slot())
    assert np.isfinite(masked).all()
    np.testing.assert_array_equal(masked, base)
    padded = pi05_pipe.run(synth.pi05_padded(1, padded=True))
    unpadded = pi05_pipe.run(synth.pi05_padded(1, padded=False))
    np.testing.assert_array_equal(padded, unpadded)


def test_pi05_batched_multi_chunk_units(pi05_pipe):
    wl = synth.pi05_batched(0)
    got = pi05_pipe.run(wl)
    assert np.isfinite(got).all()
    lens = wl.n_valid
    for b in (int(np.argmin(lens)), int(np.argmax(lens))):
        single = synth.pi05_request(0, b, lens[b])
        ref = oracle_actions(single, weights("pi05"))
        assert np.abs(got[b] - ref[0]).max() <= BF16_ACT_TOL


def test_tiny_head_dim_64_ragged_batch(tiny_pipe):
    wl = synth.build_workload("b3", synth.TINY, 3, [[("v", 30)], [("v", 5), ("m", 3)], [("v", 200)]], seed=4)
    got = tiny_pipe.run(wl)
    assert np.abs(got - oracle_actions(wl, weights("tiny"))).max() <= BF16_ACT_TOL


def test_tiny_empty_prefixes(tiny_pipe):
    wl = synth.build_workload("e", synth.TINY, 1, [[("m", 7)], []], seed=5)
    got = tiny_pipe.run(wl)
    assert np.isfinite(got).all()
    assert np.abs(got - oracle_actions(wl, weights("tiny"))).max() <= BF16_ACT_TOL
