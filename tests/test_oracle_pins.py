"""Pins of the float64 oracle to facts other than itself (no GPU needed).

Each test checks one oracle function against a library routine that defines
the same operation, a closed form, an invariant, or a brute-force formulation
of the same mathematics, so that a dropped term, a wrong sign, a wrong pairing
or a transposed operand in the oracle fails here.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from flow_matching_action_gb300 import synth
from oracle import ae_oracle as O

T = lambda a: torch.as_tensor(np.asarray(a, dtype=np.float64))  # noqa: E731


# --------------------------------------------------------------------------- time
def test_time_embedding_t0_is_sin0_cos1():
    e = O.time_embedding(0.0, 256, 4e-3, 4.0)
    assert np.array_equal(e[:128], np.zeros(128)) and np.array_equal(e[128:], np.ones(128))


def test_time_embedding_pairs_on_unit_circle():
    for t in (1.0, 0.7, 0.1, 0.0375):
        e = O.time_embedding(t, 1024, 4e-3, 4.0)
        np.testing.assert_allclose(e[:512] ** 2 + e[512:] ** 2, 1.0, atol=1e-14)


def test_time_embedding_periods_recovered_from_output():
    """Invert the embedding at a small t to recover each index's period: the
    periods must run geometrically from min_period to max_period."""
    t = 1e-4  # small enough that every angle is below pi
    e = O.time_embedding(t, 64, 4e-3, 4.0)
    ang = np.arctan2(e[:32], e[32:])
    period = 2 * math.pi * t / ang
    assert period[0] == pytest.approx(4e-3, rel=1e-9)
    assert period[-1] == pytest.approx(4.0, rel=1e-9)
    ratios = period[1:] / period[:-1]
    np.testing.assert_allclose(ratios, ratios[0], rtol=1e-9)


def test_time_mlp_matches_torch_linear_silu_chain():
    rng = np.random.default_rng(5)
    D = 48
    w1, w2 = rng.standard_normal((D, D)), rng.standard_normal((D, D))
    b1, b2 = rng.standard_normal(D), rng.standard_normal(D)
    e = rng.standard_normal(D)
    ref = F.silu(F.linear(F.silu(F.linear(T(e), T(w1), T(b1))), T(w2), T(b2))).numpy()
    np.testing.assert_allclose(O.time_mlp(e, w1, b1, w2, b2), ref, rtol=1e-12, atol=1e-12)


def test_modulation_chunks_in_order():
    rng = np.random.default_rng(6)
    c = rng.standard_normal(8)
    w = rng.standard_normal((24, 8))
    b = rng.standard_normal(24)
    full = F.linear(T(c), T(w), T(b)).numpy()
    s, sh, g = O.modulation(c, w, b, 3)
    np.testing.assert_allclose(np.concatenate([s, sh, g]), full, rtol=1e-12, atol=1e-12)
    assert s.shape == sh.shape == g.shape == (8,)


# --------------------------------------------------------------------------- norm / act
def test_ada_rms_identity_modulation_is_torch_rms_norm():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 96)) * 3
    ref = F.rms_norm(T(x), (96,), eps=1e-6).numpy()
    np.testing.assert_allclose(O.ada_rms(x, np.zeros(96), np.zeros(96), 1e-6), ref, rtol=1e-12, atol=1e-12)


def test_ada_rms_scale_minus_one_gives_shift():
    rng = np.random.default_rng(2)
    x, sh = rng.standard_normal((3, 16)), rng.standard_normal(16)
    np.testing.assert_array_equal(O.ada_rms(x, -np.ones(16), sh, 1e-6), np.broadcast_to(sh, (3, 16)))


def test_gelu_tanh_matches_torch():
    x = np.linspace(-8, 8, 1001)
    ref = F.gelu(T(x), approximate="tanh").numpy()
    np.testing.assert_allclose(O.gelu_tanh(x), ref, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------- rope
def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(3)
    dh, theta = 64, 10000.0
    x = rng.standard_normal((5, dh))
    pos = np.array([0, 1, 17, 712, 2100], dtype=np.float64)
    z = x[:, : dh // 2] + 1j * x[:, dh // 2:]
    freq = 1.0 / theta ** (np.arange(0, dh, 2) / dh)
    zr = z * np.exp(1j * pos[:, None] * freq[None, :])
    ref = np.concatenate([zr.real, zr.imag], axis=-1)
    np.testing.assert_allclose(O.rope(x, pos, theta), ref, rtol=1e-11, atol=1e-11)


def test_rope_identity_at_zero_and_norm_preserving():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 256))
    np.testing.assert_array_equal(O.rope(x, np.zeros(3), 1e4), x)
    r = O.rope(x, np.array([5.0, 900.0, 2047.0]), 1e4)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_relative_position_invariance():
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal((1, 128)), rng.standard_normal((1, 128))
    a = (O.rope(q, np.array([30.0]), 1e4) * O.rope(k, np.array([11.0]), 1e4)).sum()
    b = (O.rope(q, np.array([830.0]), 1e4) * O.rope(k, np.array([811.0]), 1e4)).sum()
    assert a == pytest.approx(b, rel=1e-10, abs=1e-10)


# --------------------------------------------------------------------------- attention
def _joint_mask(phys_valid: np.ndarray, n_act: int) -> np.ndarray:
    """Full [(P+H) x (P+H)] prefix-LM visibility as the LoongForge blog's section 3
    states it: prefix rows see valid prefix columns only (bidirectional, never
    the actions); action rows see valid prefix columns and all action columns;
    rows and columns of masked/pad prefix tokens are masked out."""
    P = phys_valid.size
    n = P + n_act
    vis = np.zeros((n, n), dtype=bool)
    pv = phys_valid.astype(bool)
    vis[:P, :P] = pv[:, None] & pv[None, :]
    vis[P:, :P] = pv[None, :]
    vis[P:, P:] = True
    # a fully masked pad row attends to nothing; give it itself so SDPA stays finite
    for i in range(P):
        if not pv[i]:
            vis[i, i] = True
    return vis


def _brute_force_action_rows(q_act, k_act, v_act, kp_phys, vp_phys, phys_valid, hq, hkv):
    """Joint attention over [physical prefix || actions] with an explicit mask, via torch SDPA."""
    P, H = kp_phys.shape[0], q_act.shape[1]
    dh = q_act.shape[-1]
    kp = np.where(phys_valid[:, None, None].astype(bool), kp_phys.reshape(P, hkv, dh), 0.0)
    vp = np.where(phys_valid[:, None, None].astype(bool), vp_phys.reshape(P, hkv, dh), 0.0)
    kj = np.concatenate([kp.transpose(1, 0, 2), k_act], axis=1)          # [hkv, P+H, dh]
    vj = np.concatenate([vp.transpose(1, 0, 2), v_act], axis=1)
    # prefix queries are irrelevant to action rows; use zeros
    qj = np.concatenate([np.zeros((hq, P, dh)), q_act], axis=1)         # [hq, P+H, dh]
    rep = hq // hkv
    kj, vj = np.repeat(kj, rep, axis=0), np.repeat(vj, rep, axis=0)
    mask = torch.as_tensor(_joint_mask(phys_valid, H))
    o = F.scaled_dot_product_attention(T(qj)[None], T(kj)[None], T(vj)[None], attn_mask=mask)[0]
    return o[:, P:].numpy()


@pytest.mark.parametrize("hq,hkv", [(4, 1), (4, 2)])
@pytest.mark.parametrize("layout", [[("v", 64)], [("v", 16), ("m", 16), ("v", 32)],
                                    [("v", 48), ("m", 16)], [("m", 8)]])
def test_attention_matches_brute_force_prefix_lm(layout, hq, hkv):
    rng = np.random.default_rng(11)
    dh, H = 64, 16
    phys_valid = np.concatenate([np.full(n, k == "v", dtype=np.uint8) for k, n in layout])
    P = phys_valid.size
    kp = rng.standard_normal((P, hkv * dh))
    vp = rng.standard_normal((P, hkv * dh))
    kp[phys_valid == 0] = np.nan
    vp[phys_valid == 0] = np.nan
    q = rng.standard_normal((hq, H, dh)) * 2
    k = rng.standard_normal((hkv, H, dh))
    v = rng.standard_normal((hkv, H, dh))
    idx = np.nonzero(phys_valid)[0]
    n = idx.size
    k_all = np.concatenate([kp[idx].reshape(n, hkv, dh).transpose(1, 0, 2), k], axis=1)
    v_all = np.concatenate([vp[idx].reshape(n, hkv, dh).transpose(1, 0, 2), v], axis=1)
    got = O.attention(q, k_all, v_all)
    ref = _brute_force_action_rows(q, k, v, kp, vp, phys_valid, hq, hkv)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_attention_rows_sum_to_one():
    """With every value row equal to ones, each output row is the sum of its
    attention weights, which must be 1."""
    rng = np.random.default_rng(12)
    q = rng.standard_normal((8, 50, 256)) * 4
    k = rng.standard_normal((1, 762, 256))
    o = O.attention(q, k, np.ones((1, 762, 256)))
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- layer
def _standard_block(h, w, l, kp, vp, positions, d):
    """A plain pre-RMSNorm transformer block built from torch library routines
    (rms_norm, linear, scaled_dot_product_attention, gelu): what an expert
    layer must reduce to when scale = shift = 0 and gate = 1."""
    H = h.shape[0]
    hq, hkv, dh = d.n_q_heads, d.n_kv_heads, d.head_dim
    th = T(h)
    y = F.rms_norm(th, (d.width,), eps=d.rms_eps)
    q = F.linear(y, T(w["wq"][l])).reshape(H, hq, dh).transpose(0, 1).numpy()
    k = F.linear(y, T(w["wk"][l])).reshape(H, hkv, dh).transpose(0, 1).numpy()
    v = F.linear(y, T(w["wv"][l])).reshape(H, hkv, dh).transpose(0, 1).numpy()
    # RoPE in its complex form
    def rot(x):
        z = x[..., : dh // 2] + 1j * x[..., dh // 2:]
        f = 1.0 / d.rope_theta ** (np.arange(0, dh, 2) / dh)
        z = z * np.exp(1j * positions[:, None] * f[None, :])
        return np.concatenate([z.real, z.imag], axis=-1)
    q, k = rot(q), rot(k)
    n = kp.shape[0]
    o = _brute_force_action_rows(q, k, v, kp, vp, np.ones(n, np.uint8), hq, hkv)
    o = T(o.transpose(1, 0, 2).reshape(H, hq * dh))
    th = th + F.linear(o, T(w["wo"][l]))
    y2 = F.rms_norm(th, (d.width,), eps=d.rms_eps)
    m = F.gelu(F.linear(y2, T(w["wg"][l])), approximate="tanh") * F.linear(y2, T(w["wu"][l]))
    return (th + F.linear(m, T(w["wd"][l]))).numpy()


def test_expert_layer_identity_modulation_is_standard_block():
    d = synth.TINY
    w = synth.make_weights(d, seed=3)
    rng = np.random.default_rng(13)
    h = rng.standard_normal((d.horizon, d.width))
    kp = rng.standard_normal((40, d.kv_dim))
    vp = rng.standard_normal((40, d.kv_dim))
    pos = 40 + np.arange(d.horizon, dtype=np.float64)
    z, one = np.zeros(d.width), np.ones(d.width)
    got = O.expert_layer(h, (z, z, one), (z, z, one), w, 1, kp, vp, pos, d)
    ref = _standard_block(h, w, 1, kp, vp, pos, d)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10)


def test_expert_layer_zero_gates_leave_residual_unchanged():
    d = synth.TINY
    w = synth.make_weights(d, seed=3)
    rng = np.random.default_rng(14)
    h = rng.standard_normal((d.horizon, d.width))
    kp = rng.standard_normal((10, d.kv_dim))
    z = np.zeros(d.width)
    s = rng.standard_normal(d.width)
    out = O.expert_layer(h, (s, s, z), (s, s, z), w, 0, kp, kp, 10 + np.arange(d.horizon), d)
    np.testing.assert_array_equal(out, h)


# --------------------------------------------------------------------------- the loop
def _run(wl, w=None, **kw):
    w = synth.make_weights(wl.dims, wl.seed) if w is None else w
    return O.sample(wl.dims, w, wl.prefix_k, wl.prefix_v, wl.cu_lens, wl.mask, wl.noise,
                    wl.n_steps, **kw)


def test_zero_velocity_leaves_noise_unchanged():
    wl = synth.tiny()
    w = synth.make_weights(wl.dims, 0)
    w["w_out"] = np.zeros_like(w["w_out"])
    w["b_out"] = np.zeros_like(w["b_out"])
    out = _run(wl, w)
    np.testing.assert_array_equal(out, wl.noise.astype(np.float64))


def _velocity_only_final_shift(d, w, rng):
    """Zero every gate and set (1 + scale_f) = 0: then v = W_out shift_f(t) + b_out."""
    D = d.width
    for l in range(d.layers):
        for j in ("1", "2"):
            wm, bm = w["w_mod" + j][l].copy(), w["b_mod" + j][l].copy()
            wm[2 * D:] = 0.0
            bm[2 * D:] = 0.0
            w["w_mod" + j][l], w["b_mod" + j][l] = wm, bm
    wf, bf = w["w_mod_f"].copy(), w["b_mod_f"].copy()
    wf[:D] = 0.0
    bf[:D] = -1.0
    w["w_mod_f"], w["b_mod_f"] = wf, bf
    return w


@pytest.mark.parametrize("n_steps", [1, 2, 5])
def test_euler_schedule_closed_form(n_steps):
    """With zero gates and (1+scale_f)=0 the velocity depends on t only:
    x_S = x_0 + delta * sum_k v(t_k), delta = -1/S, t_k = 1 - k/S."""
    d = synth.TINY
    wl = synth.build_workload("t", d, n_steps, [[("v", 20), ("m", 4)]], seed=1)
    w = _velocity_only_final_shift(d, synth.make_weights(d, 1), None)
    out = _run(wl, w)
    x = T(wl.noise[0])
    for k in range(n_steps):
        t = 1.0 - k / n_steps
        e = T(O.time_embedding(t, d.width, d.time_min_period, d.time_max_period))
        c = F.silu(F.linear(F.silu(F.linear(e, T(w["w_t1"]), T(w["b_t1"]))), T(w["w_t2"]), T(w["b_t2"])))
        shift_f = F.linear(c, T(w["w_mod_f"][d.width:]), T(w["b_mod_f"][d.width:]))
        v = F.linear(shift_f, T(w["w_out"]), T(w["b_out"]))
        x = x + (-1.0 / n_steps) * v[None, :]
    np.testing.assert_allclose(out[0], x.numpy(), rtol=1e-12, atol=1e-12)


def test_constant_velocity_moves_by_minus_v():
    """Constant v over S steps of -1/S moves x by exactly -v (up to rounding)."""
    d = synth.TINY
    wl = synth.tiny()
    w = _velocity_only_final_shift(d, synth.make_weights(d, 0), None)
    w["w_mod_f"][d.width:] = 0.0         # shift_f = b_shift: independent of t
    out = _run(wl, w)
    v = F.linear(T(w["b_mod_f"][d.width:]), T(w["w_out"]), T(w["b_out"])).numpy()
    np.testing.assert_allclose(out[0], wl.noise[0] - v[None, :], rtol=1e-12, atol=1e-12)


def test_pad_and_mask_invariance_bitwise():
    outs = {k: _run(synth.tiny_variant(k)) for k in ("plain", "masked", "padded")}
    assert np.isfinite(outs["masked"]).all()      # NaN rows never read
    np.testing.assert_array_equal(outs["masked"], outs["plain"])
    np.testing.assert_array_equal(outs["padded"], outs["plain"])


def test_hoisted_equals_recomputed_bitwise():
    wl = synth.tiny_variant("masked")
    np.testing.assert_array_equal(_run(wl, hoist=True), _run(wl, hoist=False))


def test_batch_independence_bitwise():
    d = synth.TINY
    wl = synth.build_workload("b3", d, 2, [[("v", 30)], [("v", 5), ("m", 3)], [("v", 64)]], seed=2)
    w = synth.make_weights(d, 2)
    both = _run(wl, w)
    for b, lay in enumerate(wl.layouts):
        single = synth.build_workload("b1", d, 2, [lay], seed=2)
        kb, vb = synth.valid_prefix(d, wl.n_valid[b], 2, b)
        idx = np.nonzero(single.mask)[0]
        single.prefix_k[:, idx], single.prefix_v[:, idx] = kb, vb
        single.noise = synth.request_noise(d, 2, b)[None]
        np.testing.assert_array_equal(_run(single, w)[0], both[b])


def test_empty_prefix_is_legal():
    wl = synth.build_workload("e", synth.TINY, 2, [[("m", 4)]], seed=0)
    out = _run(wl)
    assert np.isfinite(out).all()
    wl0 = synth.build_workload("e0", synth.TINY, 2, [[]], seed=0)
    np.testing.assert_array_equal(_run(wl0), out)


def test_dump_entry_is_input_projection():
    wl = synth.tiny()
    w = synth.make_weights(wl.dims, 0)
    d = wl.dims
    dump = np.zeros((wl.n_steps, d.layers + 1, 1, d.horizon, d.width))
    _run(wl, w, dump=dump)
    ref = F.linear(T(wl.noise[0]), T(w["w_in"]), T(w["b_in"])).numpy()
    np.testing.assert_allclose(dump[0, 0, 0], ref, rtol=1e-13, atol=1e-13)
    assert np.abs(dump[1, 0, 0] - dump[0, 0, 0]).max() > 0   # x moved between steps


def test_golden_tiny_regression():
    """The oracle still produces the committed tiny-case actions (written by
    tests/golden/make_golden.py from the oracle alone)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_actions.txt")
    ref = np.loadtxt(path).reshape(1, synth.TINY.horizon, synth.TINY.action_dim)
    np.testing.assert_allclose(_run(synth.tiny()), ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- context projection
def _ctx_run(wl, w, wc, hoist=True):
    return O.sample(wl.dims, w, None, None, wl.cu_lens, wl.mask, wl.noise, wl.n_steps, hoist=hoist,
                    context=(wl.context, wc["w_ck"], wc["w_cv"]))


def test_project_request_matches_torch_linear_and_complex_rotation():
    d = synth.TINY_CTX
    wl = synth.tiny_context(1, "masked")
    wc = synth.make_context_weights(d, 1)
    ks, vs, n = O.project_request(d, wl.context, wc["w_ck"], wc["w_cv"], wl.mask, 0, wl.n_rows[0])
    idx = np.nonzero(wl.mask)[0]
    assert n == idx.size == 48
    half = d.head_dim // 2
    freq = 1.0 / d.rope_theta ** (np.arange(0, d.head_dim, 2) / d.head_dim)
    for l in range(d.layers):
        x = T(wl.context[l, idx])
        k = F.linear(x, T(wc["w_ck"][l])).numpy()
        v = F.linear(x, T(wc["w_cv"][l])).numpy()
        z = k[:, :half] + 1j * k[:, half:]
        zr = z * np.exp(1j * np.arange(n)[:, None] * freq[None, :])
        np.testing.assert_allclose(ks[l], np.concatenate([zr.real, zr.imag], -1), rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(vs[l], v, rtol=1e-12, atol=1e-12)


def test_project_request_identity_weights_reduce_to_rope():
    import dataclasses
    d = dataclasses.replace(synth.TINY_CTX, ctx_dim=synth.TINY.kv_dim)
    rng = np.random.default_rng(5)
    hidden = rng.standard_normal((d.layers, 10, d.ctx_dim))
    eye = [np.eye(d.kv_dim)] * d.layers
    ks, vs, n = O.project_request(d, hidden, eye, eye, None, 0, 10)
    np.testing.assert_array_equal(vs, hidden)
    for l in range(d.layers):
        np.testing.assert_allclose(ks[l], O.rope(hidden[l], np.arange(10.0), d.rope_theta), rtol=1e-13)


def test_context_projected_once_equals_recomputed_bitwise():
    d = synth.TINY_CTX
    wl = synth.tiny_context(2, "masked")
    w, wc = synth.make_weights(d, 2), synth.make_context_weights(d, 2)
    np.testing.assert_array_equal(_ctx_run(wl, w, wc, hoist=True), _ctx_run(wl, w, wc, hoist=False))


def test_context_masked_and_padded_rows_are_skipped_bitwise():
    d = synth.TINY_CTX
    w, wc = synth.make_weights(d, 0), synth.make_context_weights(d, 0)
    outs = {k: _ctx_run(synth.tiny_context(0, k), w, wc) for k in ("plain", "masked", "padded")}
    assert np.isfinite(outs["masked"]).all()      # NaN hidden rows never projected
    np.testing.assert_array_equal(outs["masked"], outs["plain"])
    np.testing.assert_array_equal(outs["padded"], outs["plain"])


def test_context_equals_its_projection_bound_as_prefix_bitwise():
    d = synth.TINY_CTX
    wl = synth.tiny_context(3, "padded")
    w, wc = synth.make_weights(d, 3), synth.make_context_weights(d, 3)
    ks, vs, n = O.project_request(d, wl.context, wc["w_ck"], wc["w_cv"], wl.mask, 0, wl.n_rows[0])
    pk = np.full((d.layers, wl.n_rows[0], d.kv_dim), np.nan)
    pv = pk.copy()
    idx = np.nonzero(wl.mask)[0]
    pk[:, idx], pv[:, idx] = ks, vs
    ref = O.sample(d, w, pk, pv, wl.cu_lens, wl.mask, wl.noise, wl.n_steps)
    np.testing.assert_array_equal(_ctx_run(wl, w, wc), ref)


# --------------------------------------------------------------------------- VLM prefill
def test_prefill_one_layer_matches_torch_norm_linear_and_rotation():
    import dataclasses
    d = dataclasses.replace(synth.TINY_VLM, layers=1)
    w = synth.make_vlm_weights(d, 1)
    emb = synth.prefix_embeddings(d, 1, 1)
    ks, vs = O.prefill_request(d, w, emb)
    norm1 = w["b_mod1"][0][: d.width]
    y = F.rms_norm(T(emb), (d.width,), eps=d.rms_eps) * (1.0 + T(norm1))
    k = F.linear(y, T(w["wk"][0])).numpy()
    v = F.linear(y, T(w["wv"][0])).numpy()
    half = d.head_dim // 2
    z = k[:, :half] + 1j * k[:, half:]
    freq = 1.0 / d.rope_theta ** (np.arange(0, d.head_dim, 2) / d.head_dim)
    zr = z * np.exp(1j * np.arange(d.horizon)[:, None] * freq[None, :])
    np.testing.assert_allclose(ks[0], np.concatenate([zr.real, zr.imag], -1), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(vs[0], v, rtol=1e-10, atol=1e-10)


def test_prefill_layer0_is_per_token_and_deeper_layers_see_every_token():
    d = synth.TINY_VLM
    w = synth.make_vlm_weights(d, 2)
    emb = synth.prefix_embeddings(d, 2, 1)
    ks, vs = O.prefill_request(d, w, emb)
    emb2 = emb.copy()
    emb2[-1] += 1.0                                   # change the last token only
    ks2, vs2 = O.prefill_request(d, w, emb2)
    np.testing.assert_array_equal(ks2[0][:-1], ks[0][:-1])   # layer 0: K/V of a token is its own
    np.testing.assert_array_equal(vs2[0][:-1], vs[0][:-1])
    assert np.abs(ks2[1][0] - ks[1][0]).max() > 1e-6          # layer 1: token 0 saw the last token


# --------------------------------------------------------------------------- fp8 e4m3 weights
def test_e4m3_value_matches_torch_float8_e4m3fn_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_value(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])
    np.testing.assert_array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))  # -0 is code 0x80
    assert np.nanmax(got) == 448.0 and got[1] == 2.0 ** -9


def _e4m3_grid():
    v = O.e4m3_value(np.arange(0x7F))          # the 127 non-negative finite values, ascending
    assert np.all(np.diff(v) > 0)
    return v


def test_e4m3_round_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    grid = _e4m3_grid()
    mids = (grid[1:] + grid[:-1]) / 2                                # every tie
    near = np.concatenate([mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20)])
    rand = np.concatenate([rng.normal(0, s, 4000) for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = np.concatenate([grid, mids, near, rand, [0.0, -0.0, 1e-6, -1e-6]]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    x = np.concatenate([x, -x])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_round(x)
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(np.signbit(got), np.signbit(ref))


def test_e4m3_round_ties_go_to_even_mantissa_and_saturate():
    grid = _e4m3_grid()
    codes = np.arange(0x7F)
    mids = (grid[1:] + grid[:-1]) / 2
    got = O.e4m3_encode(mids)
    even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])   # the even code of each pair
    np.testing.assert_array_equal(got, even.astype(np.uint8))
    # 464 is the tie between 448 and 480 (= the NaN pattern): above 448 saturates
    for v in (448.0, 449.0, 463.9, 464.0, 470.0, 1e6):
        assert O.e4m3_round(v) == 448.0 and O.e4m3_round(-v) == -448.0


def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.arange(256)
    v = O.e4m3_value(codes)
    fin = ~np.isnan(v)
    np.testing.assert_array_equal(O.e4m3_encode(v[fin]), codes[fin].astype(np.uint8))


def test_quantize_per_tensor_amax_lands_on_448_and_error_bound():
    rng = np.random.default_rng(1)
    for scale in (0.02, 3.0, 1e-4):
        w = synth.round_to_bf16(rng.normal(0, scale, (96, 64)))
        codes, r = O.quantize_e4m3_per_tensor(w)
        assert codes.dtype == np.uint8 and codes.shape == w.shape and r.dtype == np.float32
        i = np.unravel_index(np.argmax(np.abs(w)), w.shape)
        assert abs(O.e4m3_value(codes[i])) == 448.0
        s = 1.0 / np.float64(r)
        deq = O.e4m3_value(codes) * np.float64(r)
        # half a mantissa step of w * s (2^-4 relative; 2^-10 absolute among
        # subnormals), back in w's units, plus the fp32 roundings of s, w * s and r
        bound = np.maximum(np.abs(w) * s * 2.0 ** -4, 2.0 ** -10) / s * (1 + 1e-6) + np.abs(w) * 4e-7
        assert np.all(np.abs(deq - w) <= bound)


def test_quantize_per_tensor_power_of_two_invariance_and_zero():
    rng = np.random.default_rng(2)
    w = synth.round_to_bf16(rng.normal(0, 0.02, (64, 32)))
    c0, r0 = O.quantize_e4m3_per_tensor(w)
    for k in (-3, 5):
        c1, r1 = O.quantize_e4m3_per_tensor(w * 2.0 ** k)
        np.testing.assert_array_equal(c1, c0)
        assert r1 == np.float32(r0 * np.float32(2.0 ** k))
    cz, rz = O.quantize_e4m3_per_tensor(np.zeros((4, 8)))
    assert not cz.any() and rz == 1.0


def _on_e4m3_grid(w, p):
    """w moved onto the e4m3 grid times the power of two p, largest magnitude 448 p."""
    out = dict(w)
    for name in O.FP8_LINEARS:
        out[name] = [O.e4m3_round(W / np.abs(W).max() * 448.0) * p for W in w[name]]
    return out


def test_fp8_weights_on_the_grid_reproduce_the_bf16_oracle_bitwise():
    wl = synth.tiny_variant("masked")
    w = _on_e4m3_grid(synth.make_weights(synth.TINY, 4), 2.0 ** -14)
    w8, q = O.fp8_expert_weights(w)
    assert len(q) == len(O.FP8_LINEARS) * synth.TINY.layers
    for name in O.FP8_LINEARS:
        for l in range(synth.TINY.layers):
            np.testing.assert_array_equal(w8[name][l], w[name][l])
            assert q[(name, l)][1] == np.float32(2.0 ** -14)
    ref = O.sample(synth.TINY, w, wl.prefix_k, wl.prefix_v, wl.cu_lens, wl.mask, wl.noise, 3)
    got = O.sample(synth.TINY, w8, wl.prefix_k, wl.prefix_v, wl.cu_lens, wl.mask, wl.noise, 3)
    np.testing.assert_array_equal(got, ref)
    # off the grid the fp8 weights do move the actions, by quantization noise only
    w0 = synth.make_weights(synth.TINY, 4)
    a = O.sample(synth.TINY, w0, wl.prefix_k, wl.prefix_v, wl.cu_lens, wl.mask, wl.noise, 3)
    b = O.sample(synth.TINY, O.fp8_expert_weights(w0)[0], wl.prefix_k, wl.prefix_v, wl.cu_lens, wl.mask,
                 wl.noise, 3)
    assert 0 < np.abs(a - b).max() < 0.05 * np.abs(a).max()
