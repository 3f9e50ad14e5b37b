"""The cross-attention form of the prefix (MolmoBot PR, Part 2): per-layer VLM
hidden states bound with ae_bind_context are projected into K/V once, inside
the library, and reused by every flow step.

Against the oracle run on the same hidden states (sample(context=...)): 1e-4
on the fp32 path, final-action max |delta| <= 1e-2 on the bf16 path (the
Pi0.5 shape projects on the tensor cores, the tiny shape with SIMT kernels).
Masked and padded context rows hold NaN and must change nothing (bitwise).
"""
import dataclasses

import numpy as np
import pytest

from flow_matching_action_gb300 import synth

from .helpers import GpuRunner, device_weights, oracle_actions, weights

pytestmark = pytest.mark.gpu


def ctx_weights(dims, seed=0):
    base = weights("pi05" if dims.width == synth.PI05.width else "tiny", seed)
    return {**base, **synth.make_context_weights(dims, seed)}


def oracle_ctx(wl, w, dump=False):
    return oracle_actions(wl, w, dump=dump, context=(wl.context, w["w_ck"], w["w_cv"]))


def run_ctx(runner, wl, dump=False):
    import torch
    hid = torch.from_numpy(np.ascontiguousarray(wl.context)).cuda()
    if runner.dtype == "bf16":
        hid = hid.to(torch.bfloat16)
    mask = torch.from_numpy(wl.mask).cuda()
    noise = torch.from_numpy(wl.noise).cuda()
    d = runner.dims
    buf = None
    if dump:
        buf = torch.full((wl.n_steps, d.layers + 1, wl.batch, d.horizon, d.width), float("nan"), device="cuda")
    runner.expert.set_debug_dump(buf)
    runner.expert.bind_context(hid, [int(c) for c in wl.cu_lens], mask)
    out = torch.empty_like(noise)
    runner.expert.sample(noise, wl.n_steps, out)
    runner.expert.synchronize()
    runner.expert.set_debug_dump(None)
    res = out.cpu().numpy().astype(np.float64)
    return (res, buf.cpu().numpy().astype(np.float64)) if dump else res


@pytest.mark.parametrize("dtype,tol", [("f32", 1e-4), ("bf16", 1e-2)])
def test_tiny_context_matches_oracle_and_skips_masked_rows(dtype, tol):
    dims = dataclasses.replace(synth.TINY_CTX, dtype=dtype)
    w = ctx_weights(synth.TINY_CTX)
    r = GpuRunner(dims, w, max_batch=2, max_rows=128)
    try:
        outs = {k: run_ctx(r, synth.tiny_context(0, k)) for k in ("plain", "masked", "padded")}
    finally:
        r.close()
    ref = oracle_ctx(synth.tiny_context(0, "plain"), w)
    assert np.abs(outs["plain"] - ref).max() <= tol
    assert np.isfinite(outs["masked"]).all()
    np.testing.assert_array_equal(outs["masked"], outs["plain"])
    np.testing.assert_array_equal(outs["padded"], outs["plain"])


@pytest.fixture(scope="module")
def pi05_ctx_runner():
    r = GpuRunner(synth.PI05_CTX, ctx_weights(synth.PI05_CTX), max_batch=2, max_rows=1024)
    yield r
    r.close()


def test_pi05_context_matches_oracle_per_layer(pi05_ctx_runner):
    """Tensor-core projection of 2048-wide hidden states (712 valid rows):
    final actions within 1e-2 and the per-layer residual stream within 1e-2
    relative L2 of the oracle's."""
    wl = synth.pi05_context(0, n_steps=3)
    w = ctx_weights(synth.PI05_CTX)
    got, dump = run_ctx(pi05_ctx_runner, wl, dump=True)
    ref, ref_dump = oracle_ctx(wl, w, dump=True)
    assert np.abs(got - ref).max() <= 1e-2
    rel = np.sqrt(((dump - ref_dump) ** 2).sum(axis=(2, 3, 4))) / np.sqrt((ref_dump ** 2).sum(axis=(2, 3, 4)))
    assert rel.max() <= 1e-2, rel.max()


def test_pi05_context_masked_slot_bitwise_and_rebind(pi05_ctx_runner):
    """The 968-row layout with an empty 256-row slot (NaN) equals the plain
    712-row one bitwise; binding another context of the same shape afterwards
    (K/V buffers rewritten, sample graph reused) gives that context's result."""
    plain = run_ctx(pi05_ctx_runner, synth.pi05_context(0))
    masked = run_ctx(pi05_ctx_runner, synth.pi05_context(0, padded=True))
    assert np.isfinite(masked).all()
    np.testing.assert_array_equal(masked, plain)
    other = synth.pi05_context(5, n_steps=10)
    got = run_ctx(pi05_ctx_runner, other)
    again = run_ctx(pi05_ctx_runner, synth.pi05_context(0))
    np.testing.assert_array_equal(again, plain)
    ref = oracle_ctx(other, ctx_weights(synth.PI05_CTX))
    assert np.abs(got - ref).max() <= 1e-2


def test_context_requires_ctx_dim():
    from flow_matching_action_gb300 import ae
    r = GpuRunner(synth.TINY, weights("tiny"), max_batch=1, max_rows=64)
    try:
        with pytest.raises(ae.AEError) as e:
            ae.ae_bind_context(r.expert.ctx, 0, None, [0])
        assert e.value.status == -7
    finally:
        r.close()
