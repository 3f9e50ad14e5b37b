"""Plain float64 CPU oracle of the flow-matching action-expert denoise loop.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library
never calls it, and it shares no code with the CUDA library: it reads plain
NumPy arrays and writes plain NumPy arrays.

Everything is computed in float64 with NumPy; inputs that are stored in bf16 on
the GPU arrive here as the exact float values of those bf16 numbers.  The steps
follow the pages in order; where the pages are silent the plainest reading is
taken and named in the docstring of the function that takes it.

Sources (page title, section):

* [MolmoBot] "Inference optimization for MolmoBot VLA: torch.compile + CUDA
  graphs + action-expert KV cache", Part 2 (the VLM runs once, the action expert
  is integrated for ``num_steps`` Euler steps from noise; the context K/V is
  computed once and reused by every step) and Part 1 (padded positions are
  masked out and leave the actions unchanged).
* [LoongForge] "How to Speed Up VLA Training Step by Step: A 3x Acceleration
  Case Study on Pi0.5", section 1 (empty camera slots are masked; pad tokens do
  not advance position_ids), section 2 (adaRMS: fp32, square, mean, rsqrt,
  scale/shift/gate chunks; RoPE with rotate_half; gelu*up; gated residuals),
  section 3 (MQA, the prefix-LM mask: prefix bidirectional, actions see every
  valid prefix token and each other, pad rows/cols masked), section 5.3 (action
  input projection, time MLP, action output projection).
* [sglang] sglang PR #34599 summary, implementation items 1-2 (merged Q/K/V and
  gate/up projections; mask, positions and sinusoidal time scaling computed once
  per request instead of once per step).
* [MolmoBot] Part 2 also describes the cross-attention form of the prefix: the
  VLM hands over per-layer hidden states of its context, and the action expert
  projects them into K/V; the fix computes that projection once per query and
  reuses it for every flow step (``project_request``, ``sample(context=...)``).
* [OxyGen] "Unified KV Cache Management for VLA Inference under Multi-Task
  Parallelism": the VLM prefill of a frame's observation and instruction
  produces the KV cache KV[t] that the action expert reads (``prefill_request``).

Parity status of each function is listed in ``PINS``: every function has a
test that pins it to something other than itself, except the end-to-end action
values, for which no page prints a worked example ("parity unpinned" for the
end-to-end values; each of their ingredients is pinned).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

PINS = {
    "time_embedding": "tests/test_oracle_pins.py: unit-circle pairs, t=0 value, per-index period",
    "time_mlp": "tests/test_oracle_pins.py: torch.nn.functional silu/linear chain",
    "ada_rms": "tests/test_oracle_pins.py: scale=shift=0 equals torch rms_norm",
    "rope": "tests/test_oracle_pins.py: complex-rotation form, p=0 identity, relative invariance",
    "gelu_tanh": "tests/test_oracle_pins.py: torch gelu(approximate='tanh')",
    "attention": "tests/test_oracle_pins.py: brute-force joint prefix-LM attention via torch SDPA",
    "expert_layer": "tests/test_oracle_pins.py: identity modulation equals a standard pre-norm block",
    "project_request": "tests/test_oracle_pins.py: torch F.linear + complex-rotation RoPE, identity "
                       "weights reduce to rope(), masked rows skipped, projected once == recomputed",
    "prefill_request": "tests/test_oracle_pins.py: one layer against torch rms_norm/linear and the "
                       "complex-rotation RoPE; layer-0 K/V per token, deeper K/V see every token",
    "e4m3_value": "tests/test_oracle_pins.py: all 256 codes against torch float8_e4m3fn",
    "e4m3_round / e4m3_encode": "tests/test_oracle_pins.py: torch float8_e4m3fn casts of in-range values, "
                                "ties to even at every midpoint, saturation closed form, code round trip",
    "quantize_e4m3_per_tensor": "tests/test_oracle_pins.py: amax lands on 448, error bound of half a "
                                "mantissa step, power-of-two scale invariance, amax 0",
    "fp8_expert_weights": "tests/test_oracle_pins.py: weights already on the e4m3 grid (times a power "
                          "of two) give the bf16 oracle's actions bitwise",
    "sample": "tests/test_oracle_pins.py: zero velocity, constant velocity closed form, pad/mask "
              "invariance (bitwise), hoisted == recomputed (bitwise), batch independence; "
              "end-to-end values: parity unpinned (no page prints an expected action)",
}


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# Time conditioning
# ---------------------------------------------------------------------------

def time_embedding(t: float, width: int, min_period: float, max_period: float) -> np.ndarray:
    """Sinusoidal embedding of the flow time t, length ``width``.

    [sglang] item 2 and [LoongForge] section 5.3 name a sinusoidal time scaling
    followed by a time MLP but print neither.  Reading: ``width/2`` periods
    spaced geometrically from ``min_period`` to ``max_period`` (inclusive);
    the embedding is [sin(2 pi t / p_j) for all j] followed by
    [cos(2 pi t / p_j) for all j].
    """
    half = width // 2
    if half == 1:
        frac = np.zeros(1)
    else:
        frac = np.arange(half, dtype=np.float64) / (half - 1)
    period = min_period * (max_period / min_period) ** frac
    angle = 2.0 * math.pi * float(t) / period
    return np.concatenate([np.sin(angle), np.cos(angle)])


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def time_mlp(e: np.ndarray, w_t1, b_t1, w_t2, b_t2) -> np.ndarray:
    """Time MLP ([LoongForge] section 5.3): c = silu(W2 silu(W1 e + b1) + b2).

    Reading: two D->D Linears, each followed by SiLU; c conditions every adaRMS.
    """
    a = silu(_f64(w_t1) @ e + _f64(b_t1))
    return silu(_f64(w_t2) @ a + _f64(b_t2))


def modulation(c: np.ndarray, w_mod, b_mod, n_chunks: int) -> List[np.ndarray]:
    """Chunk ``W_mod c + b_mod`` into ``n_chunks`` vectors of width D.

    [LoongForge] section 2 chunks adaRMS's conditioning into scale, shift and
    gate, in that order.  The final norm before the action output projection
    has scale and shift only (no residual follows it).
    """
    m = _f64(w_mod) @ c + _f64(b_mod)
    return list(np.split(m, n_chunks))


# ---------------------------------------------------------------------------
# Layer pieces
# ---------------------------------------------------------------------------

def ada_rms(x: np.ndarray, scale: np.ndarray, shift: np.ndarray, eps: float) -> np.ndarray:
    """Adaptive RMSNorm ([LoongForge] section 2): x * rsqrt(mean(x^2) + eps) * (1 + scale) + shift.

    Reading: no separate learned norm weight; the mean runs over the last axis.
    """
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * (1.0 + scale) + shift


def rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotary embedding with the rotate_half pairing ([LoongForge] section 2).

    x: [..., T, dh]; positions: [T].  Pair i rotates (x[i], x[i + dh/2]) by the
    angle positions * theta^(-2i/dh):  x*cos + rotate_half(x)*sin with
    rotate_half(x) = [-x2, x1].
    """
    dh = x.shape[-1]
    half = dh // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / dh)
    ang = _f64(positions)[:, None] * inv_freq[None, :]          # [T, half]
    cos, sin = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """GELU, tanh approximation (the "gelu" of gelu*up, [LoongForge] section 2)."""
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


def attention(q: np.ndarray, k_all: np.ndarray, v_all: np.ndarray) -> np.ndarray:
    """Action-row attention of one request under the prefix-LM mask.

    q: [Hq, H, dh] action queries.  k_all, v_all: [Hkv, n + H, dh] = the request's
    VALID prefix rows (in order) followed by its H action rows.  Per
    [LoongForge] section 3, action rows see every valid prefix token and every
    action token (including themselves), so the key set is exactly the rows
    passed in: masked and padded prefix rows are excluded from the set, not
    added with -inf.  Query head h reads KV head h // (Hq / Hkv) (MQA/GQA).
    Scale 1/sqrt(dh) (the pages are silent; the standard choice).
    """
    hq, _, dh = q.shape
    group = hq // k_all.shape[0]
    out = np.empty_like(q)
    for h in range(hq):
        kh, vh = k_all[h // group], v_all[h // group]
        s = (q[h] @ kh.T) / math.sqrt(dh)                       # [H, n + H]
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=-1, keepdims=True)
        out[h] = p @ vh
    return out


def expert_layer(h: np.ndarray, mods1, mods2, w: Dict, l: int, kp: np.ndarray, vp: np.ndarray,
                 positions: np.ndarray, dims, trace: Optional[Dict] = None) -> np.ndarray:
    """One Gemma-style action-expert layer on the H action rows of one request.

    h: [H, D] residual stream.  kp, vp: [n, Hkv*dh] valid prefix rows of layer l
    (prefix K is already rotated at the VLM's own positions and is not re-roped).
    Steps ([LoongForge] section 2; merged projections per [sglang] item 1 are
    a layout choice and compute the same q, k, v and gate/up):
      y = adaRMS1(h); q,k,v = y Wq^T, y Wk^T, y Wv^T; RoPE(q, k) at positions;
      o = attention; h += gate1 * (o Wo^T);
      y2 = adaRMS2(h); h += gate2 * ((gelu_tanh(y2 Wg^T) * (y2 Wu^T)) Wd^T).
    """
    H, D = h.shape
    hq, hkv, dh = dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    s1, sh1, g1 = mods1
    s2, sh2, g2 = mods2
    y = ada_rms(h, s1, sh1, dims.rms_eps)
    q = (y @ _f64(w["wq"][l]).T).reshape(H, hq, dh).transpose(1, 0, 2)
    k = (y @ _f64(w["wk"][l]).T).reshape(H, hkv, dh).transpose(1, 0, 2)
    v = (y @ _f64(w["wv"][l]).T).reshape(H, hkv, dh).transpose(1, 0, 2)
    q = rope(q, positions, dims.rope_theta)
    k = rope(k, positions, dims.rope_theta)
    n = kp.shape[0]
    k_all = np.concatenate([_f64(kp).reshape(n, hkv, dh).transpose(1, 0, 2), k], axis=1)
    v_all = np.concatenate([_f64(vp).reshape(n, hkv, dh).transpose(1, 0, 2), v], axis=1)
    o = attention(q, k_all, v_all).transpose(1, 0, 2).reshape(H, hq * dh)
    if trace is not None:
        trace.update(y=y, q=q, k=k, v=v, o=o)
    h = h + g1 * (o @ _f64(w["wo"][l]).T)
    y2 = ada_rms(h, s2, sh2, dims.rms_eps)
    m = gelu_tanh(y2 @ _f64(w["wg"][l]).T) * (y2 @ _f64(w["wu"][l]).T)
    if trace is not None:
        trace.update(y2=y2, m=m)
    return h + g2 * (m @ _f64(w["wd"][l]).T)


# ---------------------------------------------------------------------------
# fp8 e4m3 weights of the block Linears
# ---------------------------------------------------------------------------

# The Linears of the attention and MLP blocks: [MolmoBot] Part 3 converts the
# blocks' fused QKV, attention output, gate/up and down Linears and keeps the
# norms, embeddings and input/output projections in bf16; [LoongForge]
# section 7 likewise keeps the action/time projections at their precision.
FP8_LINEARS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")
E4M3_MAX = 448.0


def e4m3_value(codes) -> np.ndarray:
    """Value of fp8 E4M3 codes (the e4m3 of [MolmoBot] Part 3 and [LoongForge] section 7).

    The pages name the format without its bit layout.  Reading: the OCP 8-bit
    floating-point E4M3 format ("e4m3fn"): bit 7 sign, bits 6..3 exponent with
    bias 7, bits 2..0 mantissa; exponent field 0 holds subnormals m/8 * 2^-6;
    S.1111.111 is NaN; there are no infinities, so the largest value is
    1.75 * 2^8 = 448.
    """
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 0xF) & (c & 0x7 == 0x7), np.nan, mag)
    return sign * mag


def e4m3_round(v) -> np.ndarray:
    """Nearest E4M3 value of each (finite) v, ties to the even mantissa; a
    magnitude above 448 after rounding saturates to 448 (the saturating cast of
    a per-tensor scaled weight, whose largest magnitude lands on 448).  The sign
    of a value that rounds to zero is kept."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                      # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)               # binade of a; subnormals share 2^-6's
    q = np.exp2(e - 3.0)                     # spacing of the 3-bit mantissa there
    r = np.minimum(np.rint(a / q) * q, E4M3_MAX)  # rint: half to even
    return np.copysign(r, v)


def e4m3_encode(v) -> np.ndarray:
    """Codes of e4m3_round(v) (uint8), the sign bit set for negative values and -0."""
    r = e4m3_round(v)
    a = np.abs(r)
    _, ex = np.frexp(a)
    e = ex - 1
    normal = a >= 2.0 ** -6
    mant_n = np.where(normal, a / np.exp2(np.where(normal, e, 0)) * 8.0 - 8.0, 0.0)
    code_n = ((np.where(normal, e, 0) + 7) << 3) + mant_n.astype(np.int64)
    code_s = (a / 2.0 ** -9).astype(np.int64)
    code = np.where(normal, code_n, code_s)
    return (code | np.where(np.signbit(r), 0x80, 0)).astype(np.uint8)


def quantize_e4m3_per_tensor(w):
    """Per-tensor fp8 of one weight matrix ([MolmoBot] Part 3: per-tensor dynamic
    e4m3, amax -> scale -> cast, with the GEMM result restored by the scale;
    [LoongForge] section 7: TorchAO's tensorwise recipe, inputs and weights
    cast to fp8 and the result restored using the scales).

    The pages print no formula.  Reading (the tensorwise convention): amax =
    max |w|; s = fp32(448 / amax) (s = 1 when amax = 0); codes =
    E4M3(fp32(w * s)); the Linear applies value(code) * r with r = fp32(1 / s).
    Every step is one fp32 operation, rounded to nearest.  Only the weights
    are quantized here: the activations of the path stay bf16 (the expert's
    Linears see at most a few hundred action rows, and the pages' own fp8
    passes drop GEMMs that small).  Returns (codes uint8 like w, r float32).
    """
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.float32(np.max(np.abs(w32))) if w32.size else np.float32(0.0)
    s = np.float32(E4M3_MAX) / amax if amax > 0 else np.float32(1.0)
    codes = e4m3_encode(w32 * np.float32(s))
    return codes, np.float32(np.float32(1.0) / np.float32(s))


def fp8_expert_weights(w: Dict):
    """The weights with every block Linear (FP8_LINEARS, every layer) replaced
    by its fp8 form value(code) * r, in float64 (exact: 4 significant bits
    times the 24 of r); every other weight unchanged.  Returns (weights,
    {(name, layer): (codes, r)})."""
    out = dict(w)
    q = {}
    for name in FP8_LINEARS:
        deq = []
        for l, W in enumerate(w[name]):
            codes, r = quantize_e4m3_per_tensor(W)
            q[(name, l)] = (codes, r)
            deq.append(e4m3_value(codes) * np.float64(r))
        out[name] = deq
    return out, q


# ---------------------------------------------------------------------------
# Binding and the denoise loop
# ---------------------------------------------------------------------------

def bind_request(prefix_k, prefix_v, mask, row0: int, row1: int):
    """Valid prefix rows of one request, in physical order, for every layer.

    [LoongForge] section 1: masked camera slots and pads are invisible and do
    not advance positions, so a request's prefix is its valid rows in order and
    its action token i sits at position n_valid + i ([LoongForge] section 3:
    actions follow the prefix).  Returns (K [L, n, kv], V [L, n, kv], n).
    """
    if mask is None:
        idx = np.arange(row0, row1)
    else:
        idx = row0 + np.nonzero(np.asarray(mask[row0:row1]))[0]
    return prefix_k[:, idx, :], prefix_v[:, idx, :], int(idx.size)


def project_request(dims, hidden, w_ck, w_cv, mask, row0: int, row1: int):
    """Cross-attention K/V of one request's VLM context ([MolmoBot] Part 2).

    hidden: [L, total_rows, C] per-layer hidden states of the packed context
    (rows outside the request's valid set may hold anything, NaN included);
    w_ck, w_cv: per layer [Hkv*dh, C].  For layer l and the request's valid
    rows in order (the same valid set and order as ``bind_request``):
        K = RoPE(hidden W_ck^T) at positions 0..n-1,   V = hidden W_cv^T.
    Readings: no bias (Gemma style); the projected K is rotated at the row's
    position among the request's valid rows, which is the convention the
    joint attention of this path already assumes for a pre-projected prefix
    (prefix keys rotated at their positions, action token i at n + i), so a
    projected context is used exactly like a bound prefix.  Returns
    (K [L, n, Hkv*dh], V [L, n, Hkv*dh], n).
    """
    if mask is None:
        idx = np.arange(row0, row1)
    else:
        idx = row0 + np.nonzero(np.asarray(mask[row0:row1]))[0]
    n = int(idx.size)
    hkv, dh = dims.n_kv_heads, dims.head_dim
    L = len(w_ck)
    ks = np.empty((L, n, hkv * dh))
    vs = np.empty((L, n, hkv * dh))
    pos = np.arange(n, dtype=np.float64)
    for l in range(L):
        x = _f64(hidden[l, idx, :])                                   # [n, C]
        k = (x @ _f64(w_ck[l]).T).reshape(n, hkv, dh).transpose(1, 0, 2)
        ks[l] = rope(k, pos, dims.rope_theta).transpose(1, 0, 2).reshape(n, hkv * dh)
        vs[l] = x @ _f64(w_cv[l]).T
    return ks, vs, n


def prefill_request(dims, w: Dict, emb: np.ndarray):
    """Per-layer K and V of a VLM prefill over one request's prefix tokens.

    [OxyGen] (the VLM prefill of the observation produces KV[t]) and
    [MolmoBot] Part 2 (the VLM backbone runs once per query) put this step
    before the path.  Readings: the VLM is a Gemma-style decoder with the same
    layer as the action expert ([LoongForge] section 2) under constant
    conditioning: its RMSNorm is x * rsqrt(mean(x^2) + eps) * (1 + w_norm)
    and its residuals are plain, i.e. adaRMS with (scale, shift, gate) =
    (w_norm, 0, 1), stored as the biases of modulation Linears whose weights
    are zero; the prefix tokens attend to each other bidirectionally (the
    prefix half of [LoongForge] section 3's prefix-LM mask) at positions
    0..n-1, and K is stored after RoPE (the prefix convention of this path).
    emb: [n, D] token embeddings.  Returns (K [L, n, Hkv*dh], V [L, n, Hkv*dh]).
    """
    n, D = emb.shape
    L, hkv, dh = dims.layers, dims.n_kv_heads, dims.head_dim
    zero_c = np.zeros(D)
    pos = np.arange(n, dtype=np.float64)
    empty = np.zeros((0, hkv * dh))
    ks = np.empty((L, n, hkv * dh))
    vs = np.empty((L, n, hkv * dh))
    h = _f64(emb)
    for l in range(L):
        m1 = modulation(zero_c, w["w_mod1"][l], w["b_mod1"][l], 3)
        m2 = modulation(zero_c, w["w_mod2"][l], w["b_mod2"][l], 3)
        trace: Dict = {}
        h = expert_layer(h, m1, m2, w, l, empty, empty, pos, dims, trace=trace)
        ks[l] = trace["k"].transpose(1, 0, 2).reshape(n, hkv * dh)
        vs[l] = trace["v"].transpose(1, 0, 2).reshape(n, hkv * dh)
    return ks, vs


def step_times(n_steps: int) -> List[float]:
    """Euler schedule: n_steps steps of delta = -1/n_steps from t = 1.

    [MolmoBot] Part 2 integrates ``num_steps`` Euler steps from noise at t=1.
    Reading: the velocity of step k is evaluated at t_k = 1 - k/n_steps
    (k = 0..n_steps-1), in float64.
    """
    return [1.0 - k / n_steps for k in range(n_steps)]


def sample(dims, w: Dict, prefix_k, prefix_v, cu_lens, mask, noise, n_steps: int,
           hoist: bool = True, dump: Optional[np.ndarray] = None, context=None) -> np.ndarray:
    """Integrate the action chunk of every request from ``noise`` for ``n_steps`` Euler steps.

    prefix_k, prefix_v: [L, total_rows, Hkv*dh]; cu_lens: [B+1] physical row
    offsets; mask: [total_rows] (1 = valid) or None; noise: [B, H, A].
    Each step: h = x W_in^T + b_in; L expert layers; v = adaRMS_f(h) W_out^T
    + b_out; x <- x + delta * v with delta = -1/n_steps ([MolmoBot] Part 2).

    ``hoist=True`` computes the request binding (valid rows, positions) and
    each step's time conditioning once, as [MolmoBot] Part 2 and [sglang]
    item 2 do; ``hoist=False`` recomputes them inside every step and layer.
    The two must agree bitwise.  ``dump`` (optional, [S, L+1, B, H, D]) receives
    the residual stream entering each layer and leaving the last one.
    Requests are processed one at a time: request b's result does not depend
    on the others.

    ``context=(hidden, w_ck, w_cv)`` replaces prefix_k / prefix_v by the
    cross-attention K/V projected from the per-layer hidden states
    (``project_request``): once per request when hoisted, as [MolmoBot] Part 2
    does, or again in every step and layer when not.
    """
    B = len(cu_lens) - 1
    x_all = _f64(noise).copy()
    delta = -1.0 / n_steps
    times = step_times(n_steps)
    L = dims.layers
    D, H = dims.width, dims.horizon

    def cond(t):
        e = time_embedding(t, D, dims.time_min_period, dims.time_max_period)
        return time_mlp(e, w["w_t1"], w["b_t1"], w["w_t2"], w["b_t2"])

    hoisted_c = [cond(t) for t in times] if hoist else None

    def bind(r0, r1):
        if context is not None:
            hidden, w_ck, w_cv = context
            return project_request(dims, hidden, w_ck, w_cv, mask, r0, r1)
        return bind_request(prefix_k, prefix_v, mask, r0, r1)

    for b in range(B):
        r0, r1 = int(cu_lens[b]), int(cu_lens[b + 1])
        if hoist:
            kp, vp, n = bind(r0, r1)
            positions = n + np.arange(H, dtype=np.float64)
        x = x_all[b]
        for s, t in enumerate(times):
            c = hoisted_c[s] if hoist else cond(t)
            h = x @ _f64(w["w_in"]).T + _f64(w["b_in"])
            for l in range(L):
                if dump is not None:
                    dump[s, l, b] = h
                if not hoist:
                    kp, vp, n = bind(r0, r1)
                    positions = n + np.arange(H, dtype=np.float64)
                    c = cond(t)
                m1 = modulation(c, w["w_mod1"][l], w["b_mod1"][l], 3)
                m2 = modulation(c, w["w_mod2"][l], w["b_mod2"][l], 3)
                h = expert_layer(h, m1, m2, w, l, kp[l], vp[l], positions, dims)
            if dump is not None:
                dump[s, L, b] = h
            sf, shf = modulation(c, w["w_mod_f"], w["b_mod_f"], 2)
            v = ada_rms(h, sf, shf, dims.rms_eps) @ _f64(w["w_out"]).T + _f64(w["b_out"])
            x = x + delta * v
        x_all[b] = x
    return x_all
