"""Parity of the CUDA library (through the C ABI) with the float64 oracle.

Tolerances (stated by the spec of this path): the bf16 path must match the
oracle to final-action max |delta| <= 1e-2 and per-layer hidden relative L2
<= 1e-2 at every step and layer; the fp32 path to <= 1e-4 on both.  Pad and
mask variants must equal their unpadded GPU run bitwise: masked rows are
skipped (they hold NaN here), and every reduction runs in a fixed order over
the valid rows only.
"""
import numpy as np
import pytest

from flow_matching_action_gb300 import synth

from .helpers import GOLDEN_SEEDS, GpuRunner, golden_b16, golden_pad2048, oracle_actions, rel_l2, weights

pytestmark = pytest.mark.gpu

BF16_ACT_TOL, BF16_HID_TOL = 1e-2, 1e-2
F32_TOL = 1e-4


@pytest.fixture(scope="module")
def tiny_runner():
    r = GpuRunner(synth.TINY, weights("tiny"), max_batch=4, max_rows=256)
    yield r
    r.close()


@pytest.fixture(scope="module")
def pi05_runner():
    r = GpuRunner(synth.PI05, weights("pi05"), max_batch=16, max_rows=2048)
    yield r
    r.close()


@pytest.fixture(scope="module")
def pi05_two_camera_oracle():
    wl = synth.pi05_two_camera()
    out, dump = oracle_actions(wl, weights("pi05"), dump=True)
    return wl, out, dump


# ------------------------------------------------------------------ tiny, fp32
def test_tiny_f32_matches_oracle(tiny_runner):
    wl = synth.tiny()
    ref, ref_dump = oracle_actions(wl, weights("tiny"), dump=True)
    got, dump = tiny_runner.run(wl, dump=True)
    assert np.abs(got - ref).max() <= F32_TOL
    assert rel_l2(dump, ref_dump, axis=(2, 3, 4)).max() <= F32_TOL


@pytest.mark.parametrize("kind", ["masked", "padded"])
def test_tiny_pad_and_mask_bitwise(tiny_runner, kind):
    plain = tiny_runner.run(synth.tiny_variant("plain"))
    other = tiny_runner.run(synth.tiny_variant(kind))
    assert np.isfinite(other).all()
    np.testing.assert_array_equal(other, plain)
    ref = oracle_actions(synth.tiny_variant("plain"), weights("tiny"))
    assert np.abs(plain - ref).max() <= F32_TOL


def test_tiny_batch_of_three_matches_oracle(tiny_runner):
    wl = synth.build_workload("b3", synth.TINY, 3, [[("v", 30)], [("v", 5), ("m", 3)], [("v", 200)]],
                              seed=4)
    w = weights("tiny")
    got = tiny_runner.run(wl)
    assert np.abs(got - oracle_actions(wl, w)).max() <= F32_TOL


def test_tiny_empty_prefix_and_single_step(tiny_runner):
    w = weights("tiny")
    wl = synth.build_workload("e", synth.TINY, 1, [[("m", 7)], []], seed=5)
    got = tiny_runner.run(wl)
    assert np.isfinite(got).all()
    assert np.abs(got - oracle_actions(wl, w)).max() <= F32_TOL


def test_tiny_in_place_and_rebind_free_resample(tiny_runner):
    wl = synth.tiny_variant("masked")
    a = tiny_runner.run(wl)
    b = tiny_runner.run(wl, in_place=True)
    np.testing.assert_array_equal(a, b)
    # bind once, sample again without rebinding: hoisted binding == recomputed
    c = tiny_runner.run(wl, rebind=False)
    np.testing.assert_array_equal(a, c)


# ------------------------------------------------------------------ Pi0.5-shaped, bf16
def test_pi05_two_camera_bf16(pi05_runner, pi05_two_camera_oracle):
    wl, ref, ref_dump = pi05_two_camera_oracle
    got, dump = pi05_runner.run(wl, dump=True)
    err = np.abs(got - ref).max()
    hid = rel_l2(dump, ref_dump, axis=(2, 3, 4))
    assert err <= BF16_ACT_TOL, err
    assert hid.max() <= BF16_HID_TOL, hid.max()


def test_pi05_masked_slot_equals_two_camera_bitwise(pi05_runner, pi05_two_camera_oracle):
    base = pi05_runner.run(synth.pi05_two_camera())
    masked = pi05_runner.run(synth.pi05_masked_slot())
    assert np.isfinite(masked).all()
    np.testing.assert_array_equal(masked, base)


@pytest.mark.parametrize("seed", GOLDEN_SEEDS)
def test_pi05_padded_equals_unpadded_bitwise(pi05_runner, seed):
    """The 2048-padded workload (1621..1634 valid rows, NaN pads) equals its
    unpadded run bitwise and the oracle's stored actions within 1e-2."""
    padded = pi05_runner.run(synth.pi05_padded(seed, padded=True))
    unpadded = pi05_runner.run(synth.pi05_padded(seed, padded=False))
    assert np.isfinite(padded).all()
    np.testing.assert_array_equal(padded, unpadded)
    err = np.abs(padded - golden_pad2048(seed)).max()
    assert err <= BF16_ACT_TOL, err


def test_pi05_padded_per_layer_hidden(pi05_runner):
    """Per-layer residual stream of the 2048-padded workload against the oracle's."""
    wl = synth.pi05_padded(0, padded=True)
    got, dump = pi05_runner.run(wl, dump=True)
    ref, ref_dump = oracle_actions(synth.pi05_padded(0, padded=False), weights("pi05"), dump=True)
    assert np.abs(got - ref).max() <= BF16_ACT_TOL
    hid = rel_l2(dump, ref_dump, axis=(2, 3, 4))
    assert hid.max() <= BF16_HID_TOL, hid.max()


@pytest.mark.parametrize("seed", GOLDEN_SEEDS)
def test_pi05_batched_ragged_every_request(pi05_runner, seed):
    """Batch of 16 ragged prefixes (600..2048 valid rows): every request against
    the oracle's stored actions."""
    wl = synth.pi05_batched(seed)
    got = pi05_runner.run(wl)
    assert np.isfinite(got).all()
    err = np.abs(got - golden_b16(seed)).max(axis=(1, 2))
    assert err.max() <= BF16_ACT_TOL, err


def test_pi05_batched_per_layer_hidden_and_alone(pi05_runner):
    """Per-layer residual stream of the shortest and the longest request of the
    batch of 16 against the oracle run on that request alone, and each equal
    (within tolerance) to the library's own batch-1 run of the request."""
    wl = synth.pi05_batched(0)
    got, dump = pi05_runner.run(wl, dump=True)
    lens = wl.n_valid
    for b in (int(np.argmin(lens)), int(np.argmax(lens))):
        single = synth.pi05_request(0, b, lens[b])
        ref, ref_dump = oracle_actions(single, weights("pi05"), dump=True)
        assert np.abs(got[b] - ref[0]).max() <= BF16_ACT_TOL
        hid = rel_l2(dump[:, :, b:b + 1], ref_dump, axis=(2, 3, 4))
        assert hid.max() <= BF16_HID_TOL, (b, hid.max())
        alone = pi05_runner.run(single)
        assert np.abs(got[b] - alone[0]).max() <= BF16_ACT_TOL


def test_pi05_batch_of_three_masked_and_ragged(pi05_runner):
    """A batch between 1 and 16: 150 action tokens make one 160-token GEMM tile
    (eight epilogue warps), one request has a masked camera slot, and the
    lengths leave split-K token runs that end in partial 4-token groups."""
    wl = synth.build_workload("pi05_b3", synth.PI05, 3,
                              [[("v", 300)], [("v", 128), ("m", 256), ("v", 77)], [("v", 1100)]], seed=7)
    got = pi05_runner.run(wl)
    assert np.isfinite(got).all()
    assert np.abs(got - oracle_actions(wl, weights("pi05"))).max() <= BF16_ACT_TOL


def test_pi05_batched_long_request_then_short_ones(pi05_runner):
    """One 2048-row request, then fifteen of 600 rows.  The attention work
    split that minimizes the wave makespan here would index more partial
    units than the partial buffers hold; the planner must lengthen the chunk
    ranges instead.  The long and the last short request against the oracle
    (two Euler steps)."""
    lay = [[("v", 2048)]] + [[("v", 600)] for _ in range(15)]
    wl = synth.build_workload("pi05_long_then_short", synth.PI05, 2, lay, seed=3)
    got = pi05_runner.run(wl)
    assert np.isfinite(got).all()
    for b in (0, 15):
        ref = oracle_actions(synth.pi05_request(3, b, wl.n_valid[b], n_steps=2), weights("pi05"))
        assert np.abs(got[b] - ref[0]).max() <= BF16_ACT_TOL, b


def test_pi05_f32_debug_path_matches_oracle():
    """The same Pi0.5 weights, upcast exactly to fp32, through the fp32 path."""
    wl = synth.pi05_two_camera(n_steps=2)
    w = weights("pi05")
    r = GpuRunner(synth.PI05, w, dtype="f32", max_batch=1, max_rows=1024)
    try:
        got, dump = r.run(wl, dump=True)
    finally:
        r.close()
    ref, ref_dump = oracle_actions(wl, w, dump=True)
    assert np.abs(got - ref).max() <= F32_TOL
    assert rel_l2(dump, ref_dump, axis=(2, 3, 4)).max() <= F32_TOL


def test_debug_launch_switches_change_nothing(monkeypatch):
    """AE_GRAPH=0 (kernels launched one by one instead of one graph replay) and
    AE_PDL=0 (no programmatic dependent launch) are debugging aids read at
    ae_create: the same kernels run and the actions are bitwise the same."""
    wl = synth.pi05_masked_slot(n_steps=2)
    w = weights("pi05")
    outs = []
    for env in ({}, {"AE_GRAPH": "0"}, {"AE_GRAPH": "0", "AE_PDL": "0"}):
        for k in ("AE_GRAPH", "AE_PDL"):
            monkeypatch.delenv(k, raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        r = GpuRunner(synth.PI05, w, max_batch=1, max_rows=1024)
        try:
            outs.append(r.run(wl))
        finally:
            r.close()
    assert np.isfinite(outs[0]).all()
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


# ------------------------------------------------------------------ bf16 path, small shapes and edges
@pytest.fixture(scope="module")
def tiny_bf16_runner():
    r = GpuRunner(synth.TINY, weights("tiny"), dtype="bf16", max_batch=4, max_rows=256)
    yield r
    r.close()


def test_tiny_bf16_ragged_batch_and_empty_prefixes(tiny_bf16_runner):
    """head_dim 64 on the tensor-core path: a ragged batch with a masked slot
    and a long request, then a single Euler step with no valid prefix at all."""
    w = weights("tiny")
    wl = synth.build_workload("b3", synth.TINY, 3, [[("v", 30)], [("v", 5), ("m", 3)], [("v", 200)]], seed=4)
    assert np.abs(tiny_bf16_runner.run(wl) - oracle_actions(wl, w)).max() <= BF16_ACT_TOL
    wl = synth.build_workload("e", synth.TINY, 1, [[("m", 7)], []], seed=5)
    got = tiny_bf16_runner.run(wl)
    assert np.isfinite(got).all()
    assert np.abs(got - oracle_actions(wl, w)).max() <= BF16_ACT_TOL


def test_tiny_bf16_in_place_and_rebind_free(tiny_bf16_runner):
    wl = synth.tiny_variant("masked")
    a = tiny_bf16_runner.run(wl)
    np.testing.assert_array_equal(a, tiny_bf16_runner.run(wl, in_place=True))
    np.testing.assert_array_equal(a, tiny_bf16_runner.run(wl, rebind=False))
    np.testing.assert_array_equal(a, tiny_bf16_runner.run(synth.tiny_variant("plain")))


def test_pi05_bf16_single_euler_step(pi05_runner):
    wl = synth.pi05_two_camera(n_steps=1)
    got = pi05_runner.run(wl)
    assert np.abs(got - oracle_actions(wl, weights("pi05"))).max() <= BF16_ACT_TOL


# ------------------------------------------------------------------ errors through the ABI
def test_abi_errors_on_gpu(tiny_runner):
    from flow_matching_action_gb300 import ae
    import torch
    ctx = tiny_runner.expert.ctx
    x = torch.zeros(1, 16, 8, device="cuda")
    with pytest.raises(ae.AEError) as e:
        ae.ae_sample(ctx, x, 0, x)
    assert e.value.status == -2
    with pytest.raises(ae.AEError) as e:
        ae.ae_bind_prefix(ctx, 5, x, x, [0, 1, 2, 3, 4, 5])
    assert e.value.status == -2
    with pytest.raises(ae.AEError) as e:
        ae.ae_bind_prefix(ctx, 1, x, x, [0, 257])
    assert e.value.status == -2
    # a fresh context is unbound
    r = GpuRunner(synth.TINY, weights("tiny"), max_batch=1, max_rows=8)
    try:
        with pytest.raises(ae.AEError) as e:
            ae.ae_sample(r.expert.ctx, x, 2, x)
        assert e.value.status == -3
    finally:
        r.close()
