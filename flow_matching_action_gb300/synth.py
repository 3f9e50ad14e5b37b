"""Seeded synthetic inputs for the action-expert denoise loop.

This module only draws random numbers and lays them out in memory.  It holds
none of the method's arithmetic, so both the CPU oracle (driven by the tests)
and the CUDA library consume exactly the same inputs from here.

Shapes follow the Pi0.5-style action expert described by the LoongForge blog
("How to Speed Up VLA Training Step by Step", sections 1-3: two or three
256-token camera slots plus an instruction, 50 action tokens, 18 expert
layers) and the MolmoBot PR ("Inference optimization for MolmoBot VLA",
Part 1: about 1600 image tokens plus a few instruction tokens, padded to 2048).
No dataset is read; every tensor is N(0, sigma) from a counter-seeded
``numpy.random.default_rng`` stream:

* stream ``[seed, 0]``       weights, in the fixed order of ``WEIGHT_ORDER``
* stream ``[seed, 1]``       prefix lengths (only where a workload draws them)
* stream ``[seed, 2, b]``    valid prefix K then V rows of request ``b``
* stream ``[seed, 3, b]``    initial noise of request ``b``
* stream ``[seed, 4]``       context K/V projection weights (cross-attention form)
* stream ``[seed, 5, b]``    valid context hidden-state rows of request ``b``
* stream ``[seed, 6]``       synthetic VLM weights (prefill)
* stream ``[seed, 7, b]``    prefix token embeddings of request ``b`` (prefill)

Because request ``b`` owns its own streams, request ``b`` of a batch is the
same as a batch-1 workload built from the same ``(seed, b)``.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Sequence, Tuple

import numpy as np

WEIGHT_STD = 0.02


@dataclasses.dataclass(frozen=True)
class ExpertDims:
    """Dimensions of the action expert (names follow the pages' notation)."""

    layers: int
    width: int          # D, residual width (also the time-embedding width)
    mlp: int            # F, GeGLU hidden width
    n_q_heads: int      # Hq
    n_kv_heads: int     # Hkv (GQA: Hq % Hkv == 0)
    head_dim: int       # dh
    horizon: int        # H, action tokens per chunk
    action_dim: int     # A
    dtype: str          # "bf16" or "f32": storage type of weights and prefix K/V
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0
    time_min_period: float = 4e-3
    time_max_period: float = 4.0
    ctx_dim: int = 0    # C, width of the VLM hidden states projected into K/V (0: none)

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim


# 2-layer fp32 case the oracle finishes in well under a second.
TINY = ExpertDims(layers=2, width=256, mlp=1024, n_q_heads=4, n_kv_heads=1,
                  head_dim=64, horizon=16, action_dim=8, dtype="f32")
# Pi0.5-shaped action expert (Gemma-300M-like width, 18 layers, MQA).
PI05 = ExpertDims(layers=18, width=1024, mlp=4096, n_q_heads=8, n_kv_heads=1,
                  head_dim=256, horizon=50, action_dim=32, dtype="bf16")


def layer_weight_shapes(d: ExpertDims) -> List[Tuple[str, Tuple[int, ...]]]:
    D, F = d.width, d.mlp
    return [
        ("wq", (d.q_dim, D)), ("wk", (d.kv_dim, D)), ("wv", (d.kv_dim, D)),
        ("wo", (D, d.q_dim)), ("wg", (F, D)), ("wu", (F, D)), ("wd", (D, F)),
        ("w_mod1", (3 * D, D)), ("b_mod1", (3 * D,)),
        ("w_mod2", (3 * D, D)), ("b_mod2", (3 * D,)),
    ]


def global_weight_shapes(d: ExpertDims) -> List[Tuple[str, Tuple[int, ...]]]:
    D, A = d.width, d.action_dim
    return [
        ("w_in", (D, A)), ("b_in", (D,)),
        ("w_t1", (D, D)), ("b_t1", (D,)), ("w_t2", (D, D)), ("b_t2", (D,)),
        ("w_mod_f", (2 * D, D)), ("b_mod_f", (2 * D,)),
        ("w_out", (A, D)), ("b_out", (A,)),
    ]


LAYER_WEIGHTS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd",
                 "w_mod1", "b_mod1", "w_mod2", "b_mod2")
GLOBAL_WEIGHTS = ("w_in", "b_in", "w_t1", "b_t1", "w_t2", "b_t2",
                  "w_mod_f", "b_mod_f", "w_out", "b_out")


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.

    Input preparation only: weights and prefix K/V are stored in bf16, and both
    sides must see the same bf16 values.  Quiet NaNs stay NaN.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    src, dst = x.reshape(-1).view(np.uint32), out.reshape(-1).view(np.uint32)
    chunk = 1 << 20
    lsb = np.empty(min(chunk, src.size), dtype=np.uint32)
    for i in range(0, src.size, chunk):
        s, d = src[i:i + chunk], dst[i:i + chunk]
        t = lsb[: s.size]
        np.right_shift(s, 16, out=t)
        np.bitwise_and(t, 1, out=t)
        # finite inputs cannot overflow 32 bits here (|x| < 2^128)
        np.add(s, 0x7FFF, out=d)
        np.add(d, t, out=d)
        np.bitwise_and(d, 0xFFFF0000, out=d)
    return out.reshape(x.shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _normal(rng, shape, std=1.0) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def _store(d: ExpertDims, x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float32, copy=False)
    return round_to_bf16(x) if d.dtype == "bf16" else x


def make_weights(d: ExpertDims, seed: int = 0) -> Dict[str, object]:
    """All expert weights, N(0, 0.02), rounded to the storage dtype.

    Returns a dict: global names -> float32 arrays, and each per-layer name ->
    list of ``layers`` float32 arrays.  Matrices are row-major ``[out, in]``.
    """
    rng = np.random.default_rng([seed, 0])
    w: Dict[str, object] = {}
    for name, shape in global_weight_shapes(d)[:6]:
        w[name] = _store(d, _normal(rng, shape, WEIGHT_STD))
    for name in LAYER_WEIGHTS:
        w[name] = []
    for _ in range(d.layers):
        for name, shape in layer_weight_shapes(d):
            w[name].append(_store(d, _normal(rng, shape, WEIGHT_STD)))
    for name, shape in global_weight_shapes(d)[6:]:
        w[name] = _store(d, _normal(rng, shape, WEIGHT_STD))
    return w


def make_context_weights(d: ExpertDims, seed: int = 0) -> Dict[str, List[np.ndarray]]:
    """Per-layer context projections w_ck, w_cv [Hkv*dh, C], N(0, 0.02), from
    their own stream (the expert's other weights are unchanged by them)."""
    rng = np.random.default_rng([seed, 4])
    w: Dict[str, List[np.ndarray]] = {"w_ck": [], "w_cv": []}
    for _ in range(d.layers):
        w["w_ck"].append(_store(d, _normal(rng, (d.kv_dim, d.ctx_dim), WEIGHT_STD)))
        w["w_cv"].append(_store(d, _normal(rng, (d.kv_dim, d.ctx_dim), WEIGHT_STD)))
    return w


def build_context_workload(name: str, d: ExpertDims, n_steps: int, layouts, seed: int = 0,
                           fill=np.nan) -> "Workload":
    """As build_workload, but every request's prefix arrives as per-layer VLM
    hidden states ``context`` [L, total_rows, C] (N(0, 1) valid rows from
    stream [seed, 5, b], ``fill`` elsewhere) instead of pre-projected K/V."""
    wl = build_workload(name, d, n_steps, layouts, seed, fill)
    total = int(sum(wl.n_rows))
    ctx = np.full((d.layers, total, d.ctx_dim), fill, dtype=np.float32)
    for b, lay in enumerate(wl.layouts):
        rng = np.random.default_rng([seed, 5, b])
        rows = _store(d, _normal(rng, (d.layers, wl.n_valid[b], d.ctx_dim)))
        phys, used = int(wl.cu_lens[b]), 0
        for kind, n in lay:
            if kind == "v":
                ctx[:, phys:phys + n] = rows[:, used:used + n]
                used += n
            phys += n
    wl.context = ctx
    wl.prefix_k = wl.prefix_v = None
    return wl


# A request's prefix layout is a list of segments ("v", n) for n valid rows or
# ("m", n) for n masked / padded rows.  Valid rows are consumed in order, so two
# layouts with the same total of valid rows hold the same valid K/V.
Segment = Tuple[str, int]


@dataclasses.dataclass
class Workload:
    name: str
    dims: ExpertDims
    n_steps: int
    layouts: List[List[Segment]]
    seed: int = 0
    # filled by build_workload
    prefix_k: np.ndarray = None       # [layers, total_rows, kv_dim] float32 (NaN in masked rows)
    prefix_v: np.ndarray = None
    mask: np.ndarray = None           # [total_rows] uint8, 1 = valid
    cu_lens: np.ndarray = None        # [batch + 1] int32 physical row offsets
    noise: np.ndarray = None          # [batch, horizon, action_dim] float32
    context: np.ndarray = None        # [layers, total_rows, ctx_dim] hidden states (context workloads)

    @property
    def batch(self) -> int:
        return len(self.layouts)

    @property
    def n_valid(self) -> List[int]:
        return [sum(n for kind, n in lay if kind == "v") for lay in self.layouts]

    @property
    def n_rows(self) -> List[int]:
        return [sum(n for _, n in lay) for lay in self.layouts]


def valid_prefix(d: ExpertDims, n_valid: int, seed: int, b: int) -> Tuple[np.ndarray, np.ndarray]:
    """Valid K and V rows of request b: two [layers, n_valid, kv_dim] arrays, N(0, 1)."""
    rng = np.random.default_rng([seed, 2, b])
    k = _store(d, _normal(rng, (d.layers, n_valid, d.kv_dim)))
    v = _store(d, _normal(rng, (d.layers, n_valid, d.kv_dim)))
    return k, v


def request_noise(d: ExpertDims, seed: int, b: int) -> np.ndarray:
    rng = np.random.default_rng([seed, 3, b])
    return _normal(rng, (d.horizon, d.action_dim))


def build_workload(name: str, d: ExpertDims, n_steps: int, layouts: Sequence[Sequence[Segment]],
                   seed: int = 0, fill=np.nan) -> Workload:
    """Lay out every request's valid rows into its physical layout (masked rows = ``fill``)."""
    layouts = [list(l) for l in layouts]
    wl = Workload(name=name, dims=d, n_steps=n_steps, layouts=layouts, seed=seed)
    rows = wl.n_rows
    total = int(sum(rows))
    K = np.full((d.layers, total, d.kv_dim), fill, dtype=np.float32)
    V = np.full((d.layers, total, d.kv_dim), fill, dtype=np.float32)
    mask = np.zeros(total, dtype=np.uint8)
    cu = np.zeros(len(layouts) + 1, dtype=np.int32)
    for b, lay in enumerate(layouts):
        cu[b + 1] = cu[b] + rows[b]
        kb, vb = valid_prefix(d, wl.n_valid[b], seed, b)
        phys = int(cu[b])
        used = 0
        for kind, n in lay:
            if kind == "v":
                K[:, phys:phys + n] = kb[:, used:used + n]
                V[:, phys:phys + n] = vb[:, used:used + n]
                mask[phys:phys + n] = 1
                used += n
            elif kind != "m":
                raise ValueError(f"unknown segment kind {kind!r}")
            phys += n
    wl.prefix_k, wl.prefix_v, wl.mask, wl.cu_lens = K, V, mask, cu
    wl.noise = np.stack([request_noise(d, seed, b) for b in range(len(layouts))]) \
        if layouts else np.zeros((0, d.horizon, d.action_dim), np.float32)
    return wl


def draw_lengths(seed: int, lo: int, hi: int, count: int) -> List[int]:
    """``count`` lengths uniform on the integers [lo, hi] from stream [seed, 1]."""
    rng = np.random.default_rng([seed, 1])
    return [int(x) for x in rng.integers(lo, hi + 1, size=count)]


# ---------------------------------------------------------------------------
# The named workloads.  Sizes follow the pages: a LIBERO-style two-camera
# prefix of 2 x 256 image tokens plus instruction text (712 valid rows); the
# same with a third, empty camera slot that is masked out; a MolmoBot-style
# ~1600-image-token prefix of 1621..1634 valid rows padded to 2048; and a batch
# of 16 requests with ragged prefixes of 600..2048 rows.
# ---------------------------------------------------------------------------

def tiny(seed: int = 0) -> Workload:
    return build_workload("tiny", TINY, 2, [[("v", 64)]], seed)


def tiny_variant(kind: str, seed: int = 0) -> Workload:
    """48 valid rows: plain, with a 16-row masked slot inside, or padded to 64."""
    lay = {"plain": [("v", 48)],
           "masked": [("v", 16), ("m", 16), ("v", 32)],
           "padded": [("v", 48), ("m", 16)]}[kind]
    return build_workload(f"tiny48_{kind}", TINY, 2, [lay], seed)


def pi05_two_camera(seed: int = 0, n_steps: int = 10) -> Workload:
    return build_workload("pi05_b1_712", PI05, n_steps, [[("v", 712)]], seed)


def pi05_masked_slot(seed: int = 0, n_steps: int = 10) -> Workload:
    # img0 [0,256), img1 [256,512), empty camera slot [512,768) masked, text [768,968)
    return build_workload("pi05_b1_968_masked", PI05, n_steps,
                          [[("v", 512), ("m", 256), ("v", 200)]], seed)


def pi05_padded(seed: int = 0, n_steps: int = 10, padded: bool = True) -> Workload:
    n = draw_lengths(seed, 1621, 1634, 1)[0]
    lay = [("v", n), ("m", 2048 - n)] if padded else [("v", n)]
    return build_workload(f"pi05_b1_pad2048_{'padded' if padded else 'unpadded'}", PI05,
                          n_steps, [lay], seed)


def pi05_batched(seed: int = 0, n_steps: int = 10, batch: int = 16) -> Workload:
    lens = draw_lengths(seed, 600, 2048, batch)
    return build_workload(f"pi05_b{batch}_ragged", PI05, n_steps, [[("v", n)] for n in lens], seed)


def pi05_request(seed: int, b: int, n_valid: int, n_steps: int = 10) -> Workload:
    """Request b of a batched workload, rebuilt on its own (batch 1)."""
    wl = build_workload(f"pi05_req{b}", PI05, n_steps, [[("v", n_valid)]], seed)
    # request b's own streams, not request 0's
    k, v = valid_prefix(PI05, n_valid, seed, b)
    wl.prefix_k[:], wl.prefix_v[:] = k, v
    wl.noise = request_noise(PI05, seed, b)[None]
    return wl


# Context (cross-attention) workloads: the same expert with C = 2048-wide VLM
# hidden states (a Gemma-2B-sized VLM, as in Pi0.5) projected into the prefix
# K/V at bind time; the tiny case uses C = 128.
TINY_CTX = dataclasses.replace(TINY, ctx_dim=128)
PI05_CTX = dataclasses.replace(PI05, ctx_dim=2048)


def tiny_context(seed: int = 0, kind: str = "plain") -> Workload:
    lay = {"plain": [("v", 48)], "masked": [("v", 16), ("m", 16), ("v", 32)],
           "padded": [("v", 48), ("m", 16)]}[kind]
    return build_context_workload(f"tiny_ctx_{kind}", TINY_CTX, 2, [lay], seed)


def pi05_context(seed: int = 0, n_steps: int = 10, padded: bool = False) -> Workload:
    """The two-camera 712-row prefix as 2048-wide hidden states (optionally padded to 968 rows)."""
    lay = [("v", 512), ("m", 256), ("v", 200)] if padded else [("v", 712)]
    return build_context_workload("pi05_ctx_712" + ("_masked" if padded else ""), PI05_CTX, n_steps, [lay], seed)


# Synthetic VLM for the prefill that produces the prefix KV: a Gemma-style
# decoder with the expert's layer; ``horizon`` is the number of prefix tokens a
# request carries.  TINY_VLM is the oracle-sized case; PI05_VLM_2L has the
# widths of Pi0.5's 2B VLM (D 2048, F 16384, 8 query heads, one KV head) over
# the two-camera 712-token prefix, with 2 layers so that the oracle stays fast.
TINY_VLM = ExpertDims(layers=2, width=256, mlp=1024, n_q_heads=4, n_kv_heads=1,
                      head_dim=64, horizon=48, action_dim=8, dtype="f32")
PI05_VLM_2L = ExpertDims(layers=2, width=2048, mlp=16384, n_q_heads=8, n_kv_heads=1,
                         head_dim=256, horizon=712, action_dim=32, dtype="bf16")


def make_vlm_weights(d: ExpertDims, seed: int = 0, norm_std: float = 0.1) -> Dict[str, object]:
    """Weights of a synthetic VLM in the expert's weight layout: its layers'
    projections N(0, 0.02); its RMSNorm weights w N(0, norm_std) stored as the
    biases (w, 0, 1) of modulation Linears whose weights are zero; the time
    MLP and action projections (unused by a prefill) N(0, 0.02)."""
    rng = np.random.default_rng([seed, 6])
    D = d.width
    w: Dict[str, object] = {}
    for name, shape in global_weight_shapes(d):
        w[name] = _store(d, _normal(rng, shape, WEIGHT_STD))
    for name in LAYER_WEIGHTS:
        w[name] = []
    for _ in range(d.layers):
        for name, shape in layer_weight_shapes(d):
            if name in ("w_mod1", "w_mod2"):
                w[name].append(np.zeros(shape, dtype=np.float32))
            elif name in ("b_mod1", "b_mod2"):
                norm = _store(d, _normal(rng, (D,), norm_std))
                w[name].append(np.concatenate([norm, np.zeros(D, np.float32), np.ones(D, np.float32)]))
            else:
                w[name].append(_store(d, _normal(rng, shape, WEIGHT_STD)))
    return w


def prefix_embeddings(d: ExpertDims, seed: int, batch: int) -> np.ndarray:
    """[batch * n, D] token embeddings, N(0, 1), request b from stream [seed, 7, b]."""
    return np.concatenate([_store(d, _normal(np.random.default_rng([seed, 7, b]), (d.horizon, d.width)))
                           for b in range(batch)]) if batch else np.zeros((0, d.width), np.float32)
