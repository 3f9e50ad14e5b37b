"""ctypes binding of ``include/ae.h``: same names, argument marshalling only.

Every step of the denoise loop runs in the CUDA library; this module only turns
torch tensors into raw pointers and status codes into exceptions.  There is no
CPU or PyTorch fallback: if ``libae.so`` has not been built, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libae.so")

AE_OK = 0
AE_DTYPE_BF16 = 0
AE_DTYPE_F32 = 1
AE_WEIGHTS_AS_DTYPE = 0
AE_WEIGHTS_FP8_E4M3 = 1
AE_MAX_BATCH = 64
AE_MAX_STEPS = 128

STATUS_NAMES = {0: "AE_OK", -1: "AE_ERR_INVALID_ARG", -2: "AE_ERR_SHAPE", -3: "AE_ERR_NOT_BOUND",
                -4: "AE_ERR_CUDA", -5: "AE_ERR_DEVICE", -6: "AE_ERR_OOM", -7: "AE_ERR_UNSUPPORTED"}


class AEError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class ae_config(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int), ("width", ctypes.c_int), ("mlp", ctypes.c_int),
                ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("action_dim", ctypes.c_int), ("horizon", ctypes.c_int),
                ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
                ("time_min_period", ctypes.c_double), ("time_max_period", ctypes.c_double),
                ("dtype", ctypes.c_int), ("ctx_dim", ctypes.c_int), ("weight_format", ctypes.c_int)]


_GLOBAL = ("w_in", "b_in", "w_t1", "b_t1", "w_t2", "b_t2", "w_mod_f", "b_mod_f", "w_out", "b_out")
_LAYER = ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "w_mod1", "b_mod1", "w_mod2", "b_mod2")
_CONTEXT = ("w_ck", "w_cv")  # per layer, only with ctx_dim > 0


class ae_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _GLOBAL] + \
               [(n, ctypes.POINTER(ctypes.c_void_p)) for n in _LAYER + _CONTEXT]


class ae_info(ctypes.Structure):
    _fields_ = [("launches_last_sample", ctypes.c_int64), ("launches_last_bind", ctypes.c_int64),
                ("device_bytes", ctypes.c_int64), ("sm_count", ctypes.c_int), ("path", ctypes.c_int)]


# Every symbol include/ae.h declares, with its ctypes signature.
_SIGNATURES = {
    "ae_create": (ctypes.c_int, [ctypes.POINTER(ae_config), ctypes.POINTER(ae_weights), ctypes.c_int,
                                 ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    "ae_destroy": (None, [ctypes.c_void_p]),
    "ae_set_stream": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "ae_bind_prefix": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]),
    "ae_bind_prefix_shared": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int32, ctypes.c_void_p]),
    "ae_bind_context": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                       ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]),
    "ae_prefill": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "ae_sample": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]),
    "ae_sample_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]),
    "ae_set_debug_dump": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]),
    "ae_synchronize": (ctypes.c_int, [ctypes.c_void_p]),
    "ae_last_error": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_size_t]),
    "ae_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ae_get_info": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ae_info)]),
    "ae_get_fp8_weight": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.POINTER(ctypes.c_float)]),
    "ae_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m flow_matching_action_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _msg(ctx) -> str:
    buf = ctypes.create_string_buffer(512)
    lib().ae_last_error(ctx, buf, 512)
    return buf.value.decode(errors="replace")


def _check(status: int, ctx=None):
    if status != AE_OK:
        raise AEError(status, _msg(ctx))


def ae_status_string(status: int) -> str:
    return lib().ae_status_string(status).decode()


def make_config(dims, dtype: Optional[str] = None, fp8_weights: bool = False) -> ae_config:
    """An ae_config from any object with the expert-dimension attributes."""
    dt = dtype or dims.dtype
    return ae_config(dims.layers, dims.width, dims.mlp, dims.n_q_heads, dims.n_kv_heads, dims.head_dim,
                     dims.action_dim, dims.horizon, dims.rms_eps, dims.rope_theta,
                     dims.time_min_period, dims.time_max_period,
                     AE_DTYPE_BF16 if dt == "bf16" else AE_DTYPE_F32, getattr(dims, "ctx_dim", 0),
                     AE_WEIGHTS_FP8_E4M3 if fp8_weights else AE_WEIGHTS_AS_DTYPE)


def make_weights(w: Dict) -> ae_weights:
    """An ae_weights from a dict of tensors (global names -> tensor, layer names -> list).

    The returned struct keeps the per-layer pointer arrays alive as attributes.
    """
    s = ae_weights()
    keep = []
    for n in _GLOBAL:
        setattr(s, n, _ptr(w[n]))
    for n in _LAYER + _CONTEXT:
        if n not in w:  # context projections are optional
            continue
        arr = (ctypes.c_void_p * len(w[n]))(*[_ptr(t) for t in w[n]])
        keep.append(arr)
        setattr(s, n, ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)))
    s._keep = keep
    return s


def ae_create(config: ae_config, weights: ae_weights, max_batch: int, max_prefix_rows: int,
              stream=None) -> ctypes.c_void_p:
    out = ctypes.c_void_p()
    st = lib().ae_create(ctypes.byref(config), ctypes.byref(weights), max_batch, max_prefix_rows,
                         stream, ctypes.byref(out))
    _check(st, None)
    return out


def ae_destroy(ctx) -> None:
    lib().ae_destroy(ctx)


def ae_set_stream(ctx, stream) -> None:
    _check(lib().ae_set_stream(ctx, stream), ctx)


def ae_bind_prefix(ctx, batch: int, prefix_k, prefix_v, cu_lens: Sequence[int], prefix_mask=None) -> None:
    cu = (ctypes.c_int32 * (len(cu_lens)))(*[int(v) for v in cu_lens]) if cu_lens is not None else None
    _check(lib().ae_bind_prefix(ctx, batch, _ptr(prefix_k), _ptr(prefix_v), cu, _ptr(prefix_mask)), ctx)


def ae_bind_prefix_shared(ctx, n_samples: int, prefix_k, prefix_v, n_rows: int, prefix_mask=None) -> None:
    _check(lib().ae_bind_prefix_shared(ctx, n_samples, _ptr(prefix_k), _ptr(prefix_v), int(n_rows),
                                       _ptr(prefix_mask)), ctx)


def ae_bind_context(ctx, batch: int, hidden, cu_lens: Sequence[int], prefix_mask=None) -> None:
    cu = (ctypes.c_int32 * (len(cu_lens)))(*[int(v) for v in cu_lens]) if cu_lens is not None else None
    _check(lib().ae_bind_context(ctx, batch, _ptr(hidden), cu, _ptr(prefix_mask)), ctx)


def ae_prefill(ctx, batch: int, embeddings, out_k, out_v) -> None:
    _check(lib().ae_prefill(ctx, batch, _ptr(embeddings), _ptr(out_k), _ptr(out_v)), ctx)


def ae_sample(ctx, noise, n_steps: int, out_actions) -> None:
    _check(lib().ae_sample(ctx, _ptr(noise), n_steps, _ptr(out_actions)), ctx)


def ae_sample_noalloc(ctx, noise, n_steps: int, out_actions) -> None:
    """ae_sample without device-memory allocation (see include/ae.h): for callers
    that sample inside a stream capture or under a fixed HBM budget."""
    _check(lib().ae_sample_noalloc(ctx, _ptr(noise), n_steps, _ptr(out_actions)), ctx)


def ae_selftest_wait_timeout(ctx, budget_cycles: int) -> None:
    """Run one bounded device wait that nothing completes (see include/ae.h):
    the context's sticky status becomes AE_ERR_DEVICE."""
    _check(lib().ae_selftest_wait_timeout(ctx, int(budget_cycles)), ctx)


def ae_set_debug_dump(ctx, hidden, capacity: int) -> None:
    _check(lib().ae_set_debug_dump(ctx, _ptr(hidden), capacity), ctx)


def ae_synchronize(ctx) -> None:
    _check(lib().ae_synchronize(ctx), ctx)


def ae_last_error(ctx) -> str:
    return _msg(ctx)


FP8_LINEARS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")  # the `which` of ae_get_fp8_weight


def ae_get_fp8_weight(ctx, layer: int, which: int, codes=None) -> float:
    """Copy one quantized block Linear's e4m3 codes into `codes` (a writable
    uint8 numpy array of the tensor's shape, or None) and return its factor r."""
    r = ctypes.c_float(0.0)
    ptr = None if codes is None else codes.ctypes.data_as(ctypes.c_void_p)
    _check(lib().ae_get_fp8_weight(ctx, layer, which, ptr, ctypes.byref(r)), ctx)
    return r.value


def ae_get_info(ctx) -> dict:
    info = ae_info()
    _check(lib().ae_get_info(ctx, ctypes.byref(info)), ctx)
    return {f: getattr(info, f) for f, _ in ae_info._fields_}


class ActionExpert:
    """Convenience owner of one context: create / bind / sample / destroy.

    Holds references to the borrowed prefix tensors so they outlive the binding.
    """

    def __init__(self, dims, weights: Dict, max_batch: int, max_prefix_rows: int, stream=None,
                 dtype: Optional[str] = None, fp8_weights: bool = False):
        self.dims = dims
        self.config = make_config(dims, dtype, fp8_weights)
        self._wstruct = make_weights(weights)
        self.ctx = ae_create(self.config, self._wstruct, max_batch, max_prefix_rows, stream)
        self._bound = None

    def bind_prefix(self, prefix_k, prefix_v, cu_lens, prefix_mask=None):
        batch = len(cu_lens) - 1
        ae_bind_prefix(self.ctx, batch, prefix_k, prefix_v, cu_lens, prefix_mask)
        self._bound = (prefix_k, prefix_v, prefix_mask)

    def bind_context(self, hidden, cu_lens, prefix_mask=None):
        """Per-layer VLM hidden states projected into K/V once, then bound."""
        ae_bind_context(self.ctx, len(cu_lens) - 1, hidden, cu_lens, prefix_mask)
        self._bound = (None, None, prefix_mask)

    def bind_prefix_shared(self, n_samples: int, prefix_k, prefix_v, n_rows: int, prefix_mask=None):
        """One request's prefix bound for n_samples samples of the same observation."""
        ae_bind_prefix_shared(self.ctx, n_samples, prefix_k, prefix_v, n_rows, prefix_mask)
        self._bound = (prefix_k, prefix_v, prefix_mask)

    def sample(self, noise, n_steps: int, out=None):
        if out is None:
            out = noise.new_empty(noise.shape)
        ae_sample(self.ctx, noise, n_steps, out)
        return out

    def set_debug_dump(self, hidden):
        ae_set_debug_dump(self.ctx, hidden, 0 if hidden is None else hidden.numel())
        self._dump = hidden

    def synchronize(self):
        ae_synchronize(self.ctx)

    def info(self) -> dict:
        return ae_get_info(self.ctx)

    def close(self):
        if self.ctx is not None and self.ctx.value:
            ae_destroy(self.ctx)
        self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
