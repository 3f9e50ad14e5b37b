"""VLM prefill producing the prefix KV (OxyGen: the prefill of a frame produces
KV[t]; MolmoBot PR, Part 2: the VLM backbone runs once per query), through
ae_prefill, against the oracle's prefill_request on the same synthetic VLM and
embeddings: every layer's K and V within relative L2 1e-2 (the bf16 tolerance
of this path for hidden values), and, fed to an action expert as its bound
prefix, final actions within 1e-2 of the oracle's chain.
"""
import dataclasses

import numpy as np
import pytest

from flow_matching_action_gb300 import synth

from .helpers import GpuRunner, device_weights, oracle_actions

pytestmark = pytest.mark.gpu


def rel_l2(a, b):
    return float(np.sqrt(((a - b) ** 2).sum()) / np.sqrt((b ** 2).sum()))


def gpu_prefill(dims, w, emb, batch, fp8_weights=False):
    import torch
    from flow_matching_action_gb300 import ae
    dev_w = device_weights(w, "bf16")
    ex = ae.ActionExpert(dims, dev_w, batch, 0, dtype="bf16", fp8_weights=fp8_weights)
    try:
        e = torch.from_numpy(np.ascontiguousarray(emb)).cuda().to(torch.bfloat16)
        k = torch.empty((dims.layers, batch * dims.horizon, dims.kv_dim), dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        ae.ae_prefill(ex.ctx, batch, e, k, v)
        ex.synchronize()
        return k.float().cpu().numpy().astype(np.float64), v.float().cpu().numpy().astype(np.float64)
    finally:
        ex.close()


def oracle_prefill(dims, w, emb, batch):
    from oracle import ae_oracle
    n = dims.horizon
    ks, vs = zip(*[ae_oracle.prefill_request(dims, w, emb[b * n:(b + 1) * n]) for b in range(batch)])
    return np.concatenate(ks, axis=1), np.concatenate(vs, axis=1)


def test_tiny_vlm_prefill_matches_oracle():
    d = dataclasses.replace(synth.TINY_VLM, dtype="bf16")
    w = synth.make_vlm_weights(d, 3)
    emb = synth.prefix_embeddings(d, 3, 2)
    k, v = gpu_prefill(d, w, emb, 2)
    rk, rv = oracle_prefill(d, w, emb, 2)
    for l in range(d.layers):
        assert rel_l2(k[l], rk[l]) <= 1e-2, l
        assert rel_l2(v[l], rv[l]) <= 1e-2, l


def test_pi05_vlm_prefill_two_layers_matches_oracle():
    """The widths of Pi0.5's VLM (D 2048, MLP 16384, 8 q heads, one KV head,
    head_dim 256) over the 712-token two-camera prefix, two layers."""
    d = synth.PI05_VLM_2L
    w = synth.make_vlm_weights(d, 0)
    emb = synth.prefix_embeddings(d, 0, 1)
    k, v = gpu_prefill(d, w, emb, 1)
    rk, rv = oracle_prefill(d, w, emb, 1)
    for l in range(d.layers):
        assert rel_l2(k[l], rk[l]) <= 1e-2, (l, rel_l2(k[l], rk[l]))
        assert rel_l2(v[l], rv[l]) <= 1e-2, (l, rel_l2(v[l], rv[l]))


def test_prefilled_kv_drives_the_action_expert():
    """Prefill (GPU) -> bind as the expert's prefix -> sample, against the same
    chain in the oracle (prefill_request, then sample)."""
    import torch
    dv = dataclasses.replace(synth.TINY_VLM, dtype="bf16")
    de = dataclasses.replace(synth.TINY, dtype="bf16")
    wv, we = synth.make_vlm_weights(dv, 4), synth.make_weights(de, 4)
    emb = synth.prefix_embeddings(dv, 4, 1)
    k, v = gpu_prefill(dv, wv, emb, 1)
    rk, rv = oracle_prefill(dv, wv, emb, 1)
    wl = synth.build_workload("prefilled", de, 2, [[("v", dv.horizon)]], seed=4)
    r = GpuRunner(de, we, dtype="bf16", max_batch=1, max_rows=dv.horizon)
    try:
        wl_gpu = dataclasses.replace(wl, prefix_k=k.astype(np.float32), prefix_v=v.astype(np.float32))
        got = r.run(wl_gpu)
    finally:
        r.close()
    wl_ref = dataclasses.replace(wl, prefix_k=rk, prefix_v=rv)
    ref = oracle_actions(wl_ref, we)
    assert np.abs(got - ref).max() <= 1e-2


def test_prefill_host_checks():
    from flow_matching_action_gb300 import ae
    r = GpuRunner(synth.TINY, synth.make_weights(synth.TINY, 0), max_batch=1, max_rows=8)
    try:
        with pytest.raises(ae.AEError) as e:
            ae.ae_prefill(r.expert.ctx, 1, None, None, None)
        assert e.value.status == -7  # fp32 context
    finally:
        r.close()
