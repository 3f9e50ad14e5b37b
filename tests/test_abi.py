"""The C-ABI library loads and exports every symbol include/ae.h declares, and
its host-side checks reject bad arguments (no GPU needed)."""
import ctypes
import os
import re

import pytest

from flow_matching_action_gb300 import ae, synth
from flow_matching_action_gb300 import build as ae_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ae_build.build()
    return ae.lib()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "ae.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"AE_API\s+[\w\s\*]+?\b(ae_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("ae_create", "ae_bind_prefix", "ae_sample", "ae_destroy"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert syms
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) == set(ae._SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    for code, name in ae.STATUS_NAMES.items():
        assert ae.ae_status_string(code) == name


def _weights_struct(dims, n_layers=None):
    # fake non-NULL pointers: host checks run before any CUDA call
    fake = 0x1000
    w = {n: fake for n in ae._GLOBAL}
    for n in ae._LAYER:
        w[n] = [fake] * (n_layers if n_layers is not None else dims.layers)
    return ae.make_weights(w)


@pytest.mark.parametrize("field,value,status", [
    ("layers", 0, -1), ("width", 30, -2), ("head_dim", 48, -2), ("head_dim", 512, -2),
    ("n_kv_heads", 3, -2), ("dtype", 7, -1), ("rms_eps", 0.0, -1), ("mlp", -4, -1),
    ("ctx_dim", -8, -2), ("ctx_dim", 100, -2), ("weight_format", 2, -1),
    ("weight_format", 1, -1)])  # TINY is fp32: fp8 weights need a bf16 context
def test_create_rejects_bad_config(lib, field, value, status):
    cfg = ae.make_config(synth.TINY)
    setattr(cfg, field, value)
    with pytest.raises(ae.AEError) as e:
        ae.ae_create(cfg, _weights_struct(synth.TINY), 1, 64)
    assert e.value.status == status


def test_create_rejects_null_weights_and_bad_batch(lib):
    cfg = ae.make_config(synth.TINY)
    with pytest.raises(ae.AEError) as e:
        ae.ae_create(cfg, ae.ae_weights(), 1, 64)
    assert e.value.status == -1
    for mb in (0, ae.AE_MAX_BATCH + 1):
        with pytest.raises(ae.AEError) as e:
            ae.ae_create(cfg, _weights_struct(synth.TINY), mb, 64)
        assert e.value.status == -2


def test_calls_on_null_context_are_rejected(lib):
    assert lib.ae_get_fp8_weight(None, 0, 0, None, None) == -1
    assert lib.ae_sample(None, None, 1, None) == -1
    assert lib.ae_bind_prefix(None, 0, None, None, None, None) == -1
    assert lib.ae_bind_prefix_shared(None, 1, None, None, 10, None) == -1
    assert lib.ae_bind_context(None, 0, None, None, None) == -1
    assert lib.ae_synchronize(None) == -1
    lib.ae_destroy(None)  # ignored


def test_create_without_sm103_device_is_unsupported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cfg = ae.make_config(synth.TINY)
    with pytest.raises(ae.AEError) as e:
        ae.ae_create(cfg, _weights_struct(synth.TINY), 1, 64)
    assert e.value.status == -7
