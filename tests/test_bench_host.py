"""Host-side pieces of bench.py that need no GPU: the digest that ties the
committed DRAM-traffic counters to the CUDA sources they were taken on, and
the algorithmic bytes and FLOPs the roofline fractions divide."""
import json
import os

import numpy as np

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_tokens_drop_comments_and_keep_strings():
    text = 'int a = 1; // note\n/* block\n comment */ const char* s = "//x /*y*/";\n  int   b;'
    assert bench._code_tokens(text) == 'int a = 1; const char* s = "//x /*y*/"; int b;'


def test_code_tokens_see_code_changes_but_not_comment_edits():
    base = "__global__ void k(int* p) { p[0] = 1; } // writes one\n"
    assert bench._code_tokens(base) == bench._code_tokens(base.replace("writes one", "stores 1"))
    assert bench._code_tokens(base) != bench._code_tokens(base.replace("= 1", "= 2"))


def test_traffic_record_is_used_only_for_its_own_sources():
    """The committed counters count only while the CUDA code they were taken
    on is unchanged; otherwise bench.py reports no traffic."""
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)
    assert rec["bytes_per_flow_step"]["pi05_b1"] > 622e6  # the weights stream once per flow step
    got = bench.measured_traffic("pi05_b1")
    if rec["source_sha256"] == bench.source_digest():
        assert got == rec["bytes_per_flow_step"]["pi05_b1"]
    else:
        assert got is None


def test_fp8_traffic_and_algorithmic_bytes():
    """e4m3 block Linears: one byte a weight plus a 4-byte factor per weight
    row; the measured traffic of that path streams the codes once, at about
    half the bf16 path's bytes."""
    from flow_matching_action_gb300 import synth
    d = synth.PI05
    b16, f16 = bench.algorithmic(d, [712])
    b8, f8 = bench.algorithmic(d, [712], fp8_weights=True)
    per_layer = (d.q_dim + 2 * d.kv_dim) * d.width + d.width * d.q_dim + 3 * d.mlp * d.width
    rows = (d.q_dim + 2 * d.kv_dim) + d.width + 2 * d.mlp + d.width
    kv = d.layers * 2 * 712 * d.kv_dim * 2
    assert b16 == d.layers * per_layer * 2 + kv == 635977728
    assert b8 == d.layers * (per_layer + 4 * rows) + kv == 325472256
    assert f8 == f16  # the arithmetic is the same bf16 MMA work
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)["bytes_per_flow_step"]
    assert 311e6 < rec["pi05_b1_fp8"] < 0.55 * rec["pi05_b1"]


def test_flop_model_equals_torch_flop_counter():
    """The FLOPs the tensor roofline divides by (the block Linears of every
    token plus Q K^T and P V over each request's valid prefix rows and its own
    action rows) equal what torch's FLOP counter counts when the same
    contractions of one flow step run as plain torch ops, for a ragged batch
    with an empty prefix in it."""
    import torch
    import torch.nn.functional as F
    from torch.utils.flop_counter import FlopCounterMode

    from flow_matching_action_gb300 import synth
    d = synth.TINY
    w = synth.make_weights(d, 0)
    T = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    H, hq, hkv, dh = d.horizon, d.n_q_heads, d.n_kv_heads, d.head_dim
    n_valid = [40, 7, 0]
    with FlopCounterMode(display=False) as fc:
        for n in n_valid:
            h = torch.ones(H, d.width, dtype=torch.float64)
            prefix = torch.ones(n, d.kv_dim, dtype=torch.float64)
            for l in range(d.layers):
                q = F.linear(h, T(w["wq"][l])).reshape(H, hq, dh).transpose(0, 1)
                k = torch.cat([prefix, F.linear(h, T(w["wk"][l]))]).reshape(n + H, hkv, dh).transpose(0, 1)
                v = torch.cat([prefix, F.linear(h, T(w["wv"][l]))]).reshape(n + H, hkv, dh).transpose(0, 1)
                p = torch.softmax(torch.matmul(q, k.transpose(-1, -2)), dim=-1)
                o = torch.matmul(p, v).transpose(0, 1).reshape(H, hq * dh)
                h = h + F.linear(o, T(w["wo"][l]))
                m = F.gelu(F.linear(h, T(w["wg"][l])), approximate="tanh") * F.linear(h, T(w["wu"][l]))
                h = h + F.linear(m, T(w["wd"][l]))
    assert bench.algorithmic(d, n_valid)[1] == fc.get_total_flops()


def test_byte_model_counts_the_block_linears_and_valid_prefix_rows():
    """The HBM roofline's bytes are the block Linears the weight generator
    makes (7 per layer, 2 bytes an element; 1 byte plus a 4-byte factor per
    output row with e4m3 codes) and the K and V rows each request reads at
    every layer: its valid prefix rows, not the masked or padded ones."""
    from flow_matching_action_gb300 import synth
    d = synth.TINY
    w = synth.make_weights(d, 0)
    block = [np.asarray(a) for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd") for a in w[name]]
    assert len(block) == 7 * d.layers
    wl = synth.tiny_variant("masked")  # a masked slot inside the prefix
    n_valid = [int(m.sum()) for m in np.split(wl.mask, np.asarray(wl.cu_lens[1:-1]))]
    assert sum(n_valid) < int(wl.cu_lens[-1])
    kv = sum(d.layers * 2 * n * d.kv_dim * 2 for n in n_valid)
    assert bench.algorithmic(d, n_valid)[0] == sum(a.size for a in block) * 2 + kv
    assert bench.algorithmic(d, n_valid, fp8_weights=True)[0] == sum(a.size + 4 * a.shape[0] for a in block) + kv
