"""Shared test plumbing: upload synthetic workloads, run the CUDA library and
the oracle on the same inputs, and cache what is expensive to rebuild."""
from __future__ import annotations

import functools
import os

import numpy as np

from flow_matching_action_gb300 import synth

MAX_ROWS = 2048
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
GOLDEN_SEEDS = (0, 1, 2, 3, 4)


@functools.lru_cache(maxsize=4)
def golden(name: str) -> np.ndarray:
    """A stored oracle output (written by tests/golden/make_golden.py from the oracle alone)."""
    return np.loadtxt(os.path.join(GOLDEN, name))


def golden_pad2048(seed: int) -> np.ndarray:
    """Oracle actions [1, 50, 32] of the 2048-padded Pi0.5 workload of `seed`."""
    g = golden("pi05_pad2048_actions.txt.gz").reshape(len(GOLDEN_SEEDS), 1, 50, 32)
    return g[GOLDEN_SEEDS.index(seed)]


def golden_b16(seed: int) -> np.ndarray:
    """Oracle actions [16, 50, 32] of the batch-16 ragged Pi0.5 workload of `seed`."""
    g = golden("pi05_b16_ragged_actions.txt.gz").reshape(len(GOLDEN_SEEDS), 16, 50, 32)
    return g[GOLDEN_SEEDS.index(seed)]


@functools.lru_cache(maxsize=4)
def weights(dims_name: str, seed: int = 0):
    dims = {"tiny": synth.TINY, "pi05": synth.PI05}[dims_name]
    return synth.make_weights(dims, seed)


def oracle_actions(wl, w, dump: bool = False, **kw):
    from oracle import ae_oracle
    d = wl.dims
    buf = np.zeros((wl.n_steps, d.layers + 1, wl.batch, d.horizon, d.width)) if dump else None
    out = ae_oracle.sample(d, w, wl.prefix_k, wl.prefix_v, wl.cu_lens, wl.mask, wl.noise,
                           wl.n_steps, dump=buf, **kw)
    return (out, buf) if dump else out


def _dev(x, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def device_weights(w, dtype):
    out = {}
    for k, v in w.items():
        out[k] = [_dev(a, dtype) for a in v] if isinstance(v, list) else _dev(v, dtype)
    return out


class GpuRunner:
    """One library context for a dims/weights pair; runs workloads through the C ABI."""

    def __init__(self, dims, w, dtype=None, max_batch=16, max_rows=MAX_ROWS, fp8_weights=False):
        from flow_matching_action_gb300 import ae
        self.dtype = dtype or dims.dtype
        self.dims = dims
        self.dev_w = device_weights(w, self.dtype)
        self.expert = ae.ActionExpert(dims, self.dev_w, max_batch, max_rows, dtype=self.dtype,
                                      fp8_weights=fp8_weights)

    def upload(self, wl):
        import torch
        k = _dev(wl.prefix_k, self.dtype)
        v = _dev(wl.prefix_v, self.dtype)
        mask = torch.from_numpy(wl.mask).cuda()
        noise = torch.from_numpy(wl.noise).cuda()
        return k, v, mask, noise

    def run(self, wl, dump=False, use_mask=True, n_steps=None, in_place=False, rebind=True):
        import torch
        k, v, mask, noise = self.upload(wl)
        n_steps = n_steps or wl.n_steps
        d = self.dims
        hid = None
        if dump:
            hid = torch.full((n_steps, d.layers + 1, wl.batch, d.horizon, d.width), float("nan"),
                             device="cuda")
        self.expert.set_debug_dump(hid)
        if rebind:
            self.expert.bind_prefix(k, v, [int(c) for c in wl.cu_lens], mask if use_mask else None)
        out = noise if in_place else torch.empty_like(noise)
        self.expert.sample(noise, n_steps, out)
        self.expert.synchronize()
        self.expert.set_debug_dump(None)
        res = out.cpu().numpy().astype(np.float64)
        self._keep = (k, v, mask, noise)
        return (res, hid.cpu().numpy().astype(np.float64)) if dump else res

    def close(self):
        self.expert.close()


def rel_l2(a, b, axis):
    return np.sqrt(((a - b) ** 2).sum(axis=axis)) / np.sqrt((b ** 2).sum(axis=axis))
