"""The oracle against facts that do not come from it (CPU only)."""
import numpy as np
import pytest

import pins


@pytest.mark.parametrize("name", sorted(pins.tiny_graphs()))
def test_finite_differences(name):
    layers, rows, d_in, loss = pins.tiny_graphs()[name]
    assert pins.fd_error(layers, rows, d_in, loss) < 1e-6


def test_ce_closed_form():
    assert pins.ce_closed_form_error() < 1e-13


def test_mse_closed_form():
    assert pins.mse_closed_form_error() < 1e-15


def test_adam_first_step_closed_form():
    assert pins.adam_t1_error() < 1e-6


def test_adam_second_step_by_hand():
    assert pins.adam_t2_error() < 1e-6


def test_sgd_exact():
    assert pins.sgd_error() < 1e-7


def test_gelu_special_values():
    assert pins.gelu_special_error() < 1e-12


def test_attention_special_cases():
    assert pins.attention_special_error() < 1e-12


def test_attention_brute_force():
    assert pins.attention_brute_force_error() < 1e-12


def test_rmsnorm_invariants():
    assert pins.rmsnorm_invariant_error() < 1e-10


def test_bf16_rounding():
    assert pins.bf16_round_error() == 0.0


def test_brute_force_2x3x2():
    assert pins.brute_force_error() < 1e-12


def test_loss_decreases_on_repeated_batch():
    assert pins.loss_decrease_ok()
