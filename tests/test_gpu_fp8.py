"""fp8 e4m3 block-Linear weights (AE_WEIGHTS_FP8_E4M3) against the oracle.

MolmoBot PR, Part 3 and the LoongForge Pi0.5 blog, section 7 quantize the
block Linears per tensor (amax -> scale -> e4m3 cast, the GEMM result restored
by the scale).  The library quantizes the weights it is given in ae_create;
the oracle's quantize_e4m3_per_tensor takes the same fp32 decisions, so:

* every code and every tensor's factor r must equal the oracle's bitwise;
* sampling must match the oracle run on the fp8 weights (value(code) * r) to
  the bf16 path's tolerances (final actions max |delta| <= 1e-2, per-layer
  hidden relative L2 <= 1e-2): the kernels apply exactly those weights, and
  the remaining differences are the bf16 activations and fp32 sums the bf16
  path has too;
* weights already on the e4m3 grid times a power of two are quantized
  losslessly, so the fp8 context applies the bf16 context's weights exactly.
  Its pipeline stages span 128 K columns instead of 64, so a split-K GEMM may
  cut K at other columns and add the same products in another order: where
  every split falls on a 128-column boundary in both (the batch-16 Pi0.5
  plans) the two contexts must agree bitwise (every scaling by a power of
  two is exact), elsewhere to 2e-3 (fp32 sums in another order, then bf16
  activations).
"""
import dataclasses
import functools

import numpy as np
import pytest

from flow_matching_action_gb300 import ae, synth
from oracle import ae_oracle as O

from .helpers import GpuRunner, oracle_actions, rel_l2, weights

pytestmark = pytest.mark.gpu

ACT_TOL, HID_TOL = 1e-2, 1e-2
TINY16 = dataclasses.replace(synth.TINY, dtype="bf16")


@functools.lru_cache(maxsize=2)
def bf16_weights(name):
    """The weights as the bf16 context stores them (the oracle must quantize the same values)."""
    return synth.make_weights(TINY16, 0) if name == "tiny" else weights("pi05")


@functools.lru_cache(maxsize=2)
def fp8_oracle_weights(name):
    return O.fp8_expert_weights(bf16_weights(name))[0]


def tiny16_workload():
    """The masked tiny workload with its prefix K/V in bf16 (as a bf16 context reads it)."""
    wl = synth.tiny_variant("masked")
    return dataclasses.replace(wl, dims=TINY16, prefix_k=synth.round_to_bf16(wl.prefix_k),
                               prefix_v=synth.round_to_bf16(wl.prefix_v))


def on_grid(w, p=2.0 ** -13):
    """Block Linears moved onto the e4m3 grid times p (largest magnitude 448 p)."""
    out = dict(w)
    for name in O.FP8_LINEARS:
        out[name] = [O.e4m3_round(W / np.abs(W).max() * 448.0) * p for W in w[name]]
    return out


@pytest.mark.parametrize("name,layers", [("tiny", None), ("pi05", (0, 17))])
def test_codes_and_factors_equal_the_oracle_quantizer(name, layers):
    dims = TINY16 if name == "tiny" else synth.PI05
    w = bf16_weights(name)
    r = GpuRunner(dims, w, max_batch=1, max_rows=64, fp8_weights=True)
    try:
        for l in (layers or range(dims.layers)):
            for which, wn in enumerate(ae.FP8_LINEARS):
                W = np.asarray(w[wn][l])
                codes = np.empty(W.shape, dtype=np.uint8)
                got_r = ae.ae_get_fp8_weight(r.expert.ctx, l, which, codes)
                ref_codes, ref_r = O.quantize_e4m3_per_tensor(W)
                np.testing.assert_array_equal(codes, ref_codes, err_msg=f"{wn}[{l}]")
                assert np.float32(got_r) == ref_r, (wn, l, got_r, ref_r)
    finally:
        r.close()


def test_tiny_fp8_matches_oracle():
    wl = tiny16_workload()
    r = GpuRunner(TINY16, bf16_weights("tiny"), max_batch=4, max_rows=256, fp8_weights=True)
    try:
        got, dump = r.run(wl, dump=True)
    finally:
        r.close()
    ref, ref_dump = oracle_actions(wl, fp8_oracle_weights("tiny"), dump=True)
    assert np.abs(got - ref).max() <= ACT_TOL
    assert rel_l2(dump, ref_dump, axis=(2, 3, 4)).max() <= HID_TOL


@pytest.fixture(scope="module")
def pi05_fp8_runner():
    r = GpuRunner(synth.PI05, weights("pi05"), max_batch=16, max_rows=2048, fp8_weights=True)
    yield r
    r.close()


def test_pi05_fp8_two_camera_matches_oracle(pi05_fp8_runner):
    wl = synth.pi05_two_camera()
    got, dump = pi05_fp8_runner.run(wl, dump=True)
    ref, ref_dump = oracle_actions(wl, fp8_oracle_weights("pi05"), dump=True)
    err = np.abs(got - ref).max()
    hid = rel_l2(dump, ref_dump, axis=(2, 3, 4)).max()
    assert err <= ACT_TOL, err
    assert hid <= HID_TOL, hid
    # the fp8 weights move the actions away from the bf16 weights' by
    # quantization noise, far less than the actions themselves
    bf16_ref = oracle_actions(wl, weights("pi05"))
    assert 0 < np.abs(ref - bf16_ref).max() < 0.1 * np.abs(bf16_ref).max()


def test_pi05_fp8_batched_shortest_and_longest_match_oracle(pi05_fp8_runner):
    wl = synth.pi05_batched(0)
    got = pi05_fp8_runner.run(wl)
    assert np.isfinite(got).all()
    lens = [int(n) for n in wl.n_rows]
    for b in (int(np.argmin(lens)), int(np.argmax(lens))):
        one = synth.pi05_request(0, b, lens[b])
        ref = oracle_actions(one, fp8_oracle_weights("pi05"))
        assert np.abs(got[b] - ref[0]).max() <= ACT_TOL, b


@pytest.mark.parametrize("case", ["tiny_b2", "pi05_b1", "pi05_b16"])
def test_on_grid_weights_fp8_context_equals_bf16_context(case):
    if case == "tiny_b2":
        dims, w, wl, mb, rows = TINY16, bf16_weights("tiny"), tiny16_workload(), 4, 256
    else:
        dims, w, mb, rows = synth.PI05, weights("pi05"), 16, 2048
        wl = synth.pi05_two_camera() if case == "pi05_b1" else synth.pi05_batched(0)
    wg = on_grid(w)
    outs = []
    for fp8 in (False, True):
        r = GpuRunner(dims, wg, max_batch=mb, max_rows=rows, fp8_weights=fp8)
        try:
            outs.append(r.run(wl))
        finally:
            r.close()
    assert np.isfinite(outs[0]).all()
    if case == "pi05_b16":
        np.testing.assert_array_equal(outs[1], outs[0])
    else:
        assert np.abs(outs[1] - outs[0]).max() <= 2e-3


def test_fp8_noalloc_matches_sample(pi05_fp8_runner):
    """ae_sample_noalloc on an fp8 context (its attention keeps fp32 split-KV
    partials where ae_sample keeps bf16 ones: equal within the bf16 tolerance)."""
    import torch
    wl = synth.pi05_two_camera()
    base = pi05_fp8_runner.run(wl)
    x = torch.from_numpy(wl.noise).cuda()
    out = torch.empty_like(x)
    ae.ae_sample_noalloc(pi05_fp8_runner.expert.ctx, x, wl.n_steps, out)
    pi05_fp8_runner.expert.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    assert np.abs(got - base).max() <= ACT_TOL


def test_fp8_export_rejected_on_bf16_context():
    r = GpuRunner(TINY16, bf16_weights("tiny"), max_batch=1, max_rows=64)
    try:
        with pytest.raises(ae.AEError) as e:
            ae.ae_get_fp8_weight(r.expert.ctx, 0, 0)
        assert e.value.status == -7
        rf = GpuRunner(TINY16, bf16_weights("tiny"), max_batch=1, max_rows=64, fp8_weights=True)
        try:
            for layer, which in ((-1, 0), (TINY16.layers, 0), (0, 7)):
                with pytest.raises(ae.AEError) as e:
                    ae.ae_get_fp8_weight(rf.expert.ctx, layer, which)
                assert e.value.status == -1
            info = rf.expert.info()
            assert info["device_bytes"] < r.expert.info()["device_bytes"]  # codes replace the bf16 copies
        finally:
            rf.close()
    finally:
        r.close()


def test_pi05_fp8_shared_prefix_equals_bound_copies(pi05_fp8_runner):
    """One prefix shared by 4 samples (OxyGen cross-task KV sharing) on an fp8
    context: bitwise the result of binding 4 copies (the same kernels)."""
    from .test_gpu_shared_prefix import copies_of, run_shared
    wl = synth.pi05_two_camera()
    many = copies_of(wl, 4, noise_seed=31)
    shared = run_shared(pi05_fp8_runner, wl, many.noise)
    copied = pi05_fp8_runner.run(many)
    assert np.isfinite(shared).all()
    np.testing.assert_array_equal(shared, copied)


def test_pi05_fp8_context_projection_matches_oracle():
    """The projected-context prefix (MolmoBot PR, Part 2) with fp8 block
    Linears: the context projections stay bf16, the expert's Linears are e4m3."""
    from .test_gpu_context import run_ctx
    dims = synth.PI05_CTX
    wc = synth.make_context_weights(dims, 0)
    wl = synth.pi05_context(0)
    r = GpuRunner(dims, {**weights("pi05"), **wc}, max_batch=1, max_rows=max(wl.n_rows), fp8_weights=True)
    try:
        got = run_ctx(r, wl)
    finally:
        r.close()
    ref = oracle_actions(wl, {**fp8_oracle_weights("pi05"), **wc}, context=(wl.context, wc["w_ck"], wc["w_cv"]))
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= ACT_TOL


@pytest.mark.parametrize("which", ["tiny", "pi05_2l"])
def test_vlm_prefill_with_fp8_weights_matches_oracle(which):
    """ae_prefill (OxyGen: the prefill produces KV[t]) through the e4m3 GEMMs,
    including the long-K down projection of a 16384-wide MLP, against the
    oracle's prefill on the same fp8 weights: every layer's K and V within
    relative L2 1e-2."""
    from .test_gpu_prefill import gpu_prefill, oracle_prefill, rel_l2 as rl2
    if which == "tiny":
        d = dataclasses.replace(synth.TINY_VLM, dtype="bf16")
        w, emb, batch = synth.make_vlm_weights(d, 3), synth.prefix_embeddings(d, 3, 2), 2
    else:
        d = synth.PI05_VLM_2L
        w, emb, batch = synth.make_vlm_weights(d, 0), synth.prefix_embeddings(d, 0, 1), 1
    k, v = gpu_prefill(d, w, emb, batch, fp8_weights=True)
    rk, rv = oracle_prefill(d, O.fp8_expert_weights(w)[0], emb, batch)
    for l in range(d.layers):
        assert rl2(k[l], rk[l]) <= 1e-2, (l, rl2(k[l], rk[l]))
        assert rl2(v[l], rv[l]) <= 1e-2, (l, rl2(v[l], rv[l]))
