"""The C ABI library loads, exports every symbol include/mg.h declares, and
rejects bad descriptors before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from static_graph_nn_gb300 import binding
from static_graph_nn_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "mg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mg_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("mg_step_plan_create", "mg_forward", "mg_train_step", "mg_step_plan_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_symbols():
        assert hasattr(lib, n), n
    assert set(declared_symbols()) == set(binding.exported_symbols())


def _create(lib, layers, batch=8, loss="ce_dense", precision="strict", optimizer="adam"):
    arr = (binding.mg_layer * max(1, len(layers)))(*[binding.layer_struct(l) for l in layers])
    d = binding.mg_graph_desc()
    d.batch, d.n_layers, d.layers = batch, len(layers), arr
    d.loss = binding.LOSSES[loss]
    d.precision = binding.PRECISIONS[precision]
    d.optimizer = binding.OPTIMIZERS[optimizer]
    d.beta1, d.beta2, d.adam_eps = 0.9, 0.999, 1e-8
    h = ctypes.c_void_p()
    st = lib.mg_step_plan_create(ctypes.byref(d), ctypes.byref(h))
    if st == 0:
        lib.mg_step_plan_destroy(h)
    return st, lib.mg_last_error(None).decode()


BAD = {
    "widths_do_not_chain": ([W.linear(4, 8, True), W.relu(), W.linear(7, 2, False)], binding.MG_ERR_SHAPE),
    "zero_batch": ([W.linear(4, 8, True)], binding.MG_ERR_SHAPE, 0),
    "activation_first": ([W.relu(), W.linear(4, 2, False)], binding.MG_ERR_UNSUPPORTED),
    "activation_before_loss": ([W.linear(4, 2, False), W.relu()], binding.MG_ERR_UNSUPPORTED),
    "residual_unbalanced": ([W.residual_begin(), W.linear(4, 4, False)], binding.MG_ERR_INVALID_ARG),
    "residual_width": ([W.residual_begin(), W.linear(4, 6, False), W.residual_end()], binding.MG_ERR_SHAPE),
    "attention_strict": ([W.linear(64, 192, False), W.causal_attention(1, 64, 64)], binding.MG_ERR_UNSUPPORTED),
    "attention_head_dim": ([W.linear(32, 96, False), W.causal_attention(1, 32, 64)], binding.MG_ERR_UNSUPPORTED, 64, "bf16"),
    "attention_batch": ([W.linear(64, 192, False), W.causal_attention(1, 64, 64), W.linear(64, 4, False)], binding.MG_ERR_SHAPE, 100, "bf16"),
    "bf16_input_row_alignment": ([W.linear(10, 8, False)], binding.MG_ERR_ALIGN, 8, "bf16"),
    "no_layers": ([], binding.MG_ERR_INVALID_ARG),
}


@pytest.mark.parametrize("case", sorted(BAD))
def test_descriptor_validation(lib, case):
    spec = BAD[case]
    layers, want = spec[0], spec[1]
    batch = spec[2] if len(spec) > 2 else 8
    prec = spec[3] if len(spec) > 3 else "strict"
    st, msg = _create(lib, layers, batch=batch, precision=prec)
    assert st == want, (st, msg)
    assert msg


def test_null_arguments(lib):
    assert lib.mg_step_plan_create(None, None) == binding.MG_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert lib.mg_step_plan_create(None, ctypes.byref(h)) == binding.MG_ERR_INVALID_ARG
    assert h.value is None
    lib.mg_step_plan_destroy(None)  # no-op
    assert lib.mg_param_count(None) == 0
    assert lib.mg_train_step(None, None, None, None, None, None, None, 0.1, 1, None) == binding.MG_ERR_INVALID_ARG
    assert lib.mg_forward(None, None, None, None, None) == binding.MG_ERR_INVALID_ARG
    assert lib.mg_last_error(None)


def _create_raw(lib, layers, loss=0, precision=0, optimizer=1, beta1=0.9, beta2=0.999, eps=1e-8):
    arr = (binding.mg_layer * max(1, len(layers)))(*[binding.layer_struct(l) for l in layers])
    d = binding.mg_graph_desc()
    d.batch, d.n_layers, d.layers = 8, len(layers), arr
    d.loss, d.precision, d.optimizer = loss, precision, optimizer
    d.beta1, d.beta2, d.adam_eps = beta1, beta2, eps
    h = ctypes.c_void_p()
    st = lib.mg_step_plan_create(ctypes.byref(d), ctypes.byref(h))
    if st == 0:
        lib.mg_step_plan_destroy(h)
    return st, h.value


BAD_SETTINGS = {
    "loss_kind": dict(loss=3),
    "negative_loss_kind": dict(loss=-1),
    "precision": dict(precision=2),
    "optimizer": dict(optimizer=4),
    "negative_optimizer": dict(optimizer=-1),
    "adam_beta1_one": dict(optimizer=binding.OPTIMIZERS["adam"], beta1=1.0),
    "adam_beta2_negative": dict(optimizer=binding.OPTIMIZERS["adam"], beta2=-0.5),
    "adam_eps_zero": dict(optimizer=binding.OPTIMIZERS["adam"], eps=0.0),
    "adam_beta_nan": dict(optimizer=binding.OPTIMIZERS["adam"], beta1=float("nan")),
    "laprop_eps_negative": dict(optimizer=binding.OPTIMIZERS["laprop"], eps=-1e-8),
    "laprop_beta2_one": dict(optimizer=binding.OPTIMIZERS["laprop"], beta2=1.0),
    "momentum_one": dict(optimizer=binding.OPTIMIZERS["sgd_momentum"], beta1=1.0),
}


@pytest.mark.parametrize("case", sorted(BAD_SETTINGS))
def test_settings_validation(lib, case):
    """Out-of-range loss, precision and optimizer settings are rejected at
    creation, before any device work, and no plan is returned."""
    st, h = _create_raw(lib, [W.linear(4, 2, False)], **BAD_SETTINGS[case])
    assert st == binding.MG_ERR_INVALID_ARG
    assert h is None
    assert lib.mg_last_error(None)


def test_null_plan_in_every_entry_point(lib):
    """Every call that takes a plan answers a NULL plan with an error status
    (or zero / NULL), without touching a device."""
    E = binding.MG_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(64)
    n = ctypes.c_size_t()
    assert lib.mg_param_tensor_count(None) == 0
    assert lib.mg_workspace_bytes(None) == 0
    assert lib.mg_param_info(None, 0, None, None, None) == E
    assert lib.mg_loss(None, None, None) == E
    assert lib.mg_loss_async(None, buf, None) == E
    assert lib.mg_loss_device_ptr(None) is None
    assert lib.mg_refresh_params(None, None, None) == E
    assert lib.mg_plan_dump(None, buf, 64) == 0
    assert lib.mg_debug_check_finite(None, None, 0, None, None) == E
    assert lib.mg_last_launch_count(None) == 0
    assert lib.mg_graph_replays(None) == 0
    assert lib.mg_profile_begin(None, 1) == E
    assert lib.mg_profile_end(None) == E
    assert lib.mg_profile_entries(None) == 0
    assert lib.mg_profile_entry(None, 0, None, 0, None, None, None, None) == E
    assert lib.mg_checkpoint_bytes(None, 1, 1) == 0
    assert lib.mg_checkpoint_save(None, None, None, None, buf, 64, ctypes.byref(n), None) == E
    assert lib.mg_checkpoint_load(None, buf, 64, None, None, None, None) == E
