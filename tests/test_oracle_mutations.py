"""Plant plausible mistakes in the oracle (on the CPU) and check that at least
one pin catches each: the pins are strong enough to trust the oracle."""
import importlib.util
import os
import types

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "step.py")

MUTATIONS = {
    "gelu_grad_drops_term": ("return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * du",
                             "return 0.5 * (1.0 + t)"),
    "gelu_wrong_constant": ("GELU_C = 0.044715", "GELU_C = 0.0447"),
    "ce_dense_sign": ("grad = (p * y.sum(axis=1, keepdims=True) - y) / rows",
                      "grad = (y - p * y.sum(axis=1, keepdims=True)) / rows"),
    "ce_no_mean": ("loss = -(y * lp).sum() / rows", "loss = -(y * lp).sum()"),
    "ce_index_off_by_one": ("grad[np.arange(rows), t] -= 1.0",
                            "grad[np.arange(rows), (t + 1) % grad.shape[1]] -= 1.0"),
    "mse_factor": ("2.0 * diff / n", "diff / n"),
    "rmsnorm_drops_mean_term": ("dh = r * (gy - x * r * r * (gy * x).mean(axis=1, keepdims=True))",
                                "dh = r * gy"),
    "rmsnorm_eps_outside": ("r = 1.0 / np.sqrt((h * h).mean(axis=1, keepdims=True) + l[\"eps\"])",
                            "r = 1.0 / (np.sqrt((h * h).mean(axis=1, keepdims=True)) + l[\"eps\"])"),
    "linear_dx_transposed": ("dh = dh @ t[\"w\"].T", "dh = dh @ t[\"w\"].T[::-1]"),
    "linear_dw_transposed": ("grads[sl[0]] = t[\"x\"].T @ dh", "grads[sl[0]] = (dh.T @ t[\"x\"]).T[::-1]"),
    "bias_grad_mean": ("grads[sl[1]] = dh.sum(axis=0)", "grads[sl[1]] = dh.mean(axis=0)"),
    "relu_grad_ge": ("dh = dh * (t[\"z\"] > 0.0)", "dh = dh * (t[\"z\"] >= -0.5)"),
    "residual_skip_grad_dropped": ("dh = dh + skip_grads.pop()", "skip_grads.pop()"),
    "attn_mask_wrong_side": ("mask = np.triu(np.ones((s_len, s_len), dtype=bool), k=1)",
                             "mask = np.tril(np.ones((s_len, s_len), dtype=bool), k=-1)"),
    "attn_no_scale": ("scale = 1.0 / math.sqrt(dh)\n    s = (q @ k.T) * scale",
                      "scale = 1.0 / math.sqrt(dh)\n    s = (q @ k.T)"),
    "attn_dk_no_scale": ("dk = (ds.T @ q) * scale", "dk = (ds.T @ q)"),
    "attn_ds_sign": ("ds = p * (dp - (dp * p).sum(axis=1, keepdims=True))",
                     "ds = p * (dp + (dp * p).sum(axis=1, keepdims=True))"),
    "attn_heads_swapped_v": ("v = qkv[r, 2 * d + hh * dh: 2 * d + (hh + 1) * dh]",
                             "v = qkv[r, 2 * d + ((hh + 1) % h) * dh: 2 * d + ((hh + 1) % h + 1) * dh]"),
    "adam_no_bias_correction": ("mhat = m2 / (1.0 - beta1 ** step)", "mhat = m2"),
    "adam_eps_inside": ("lr * mhat / (np.sqrt(vhat) + eps)", "lr * mhat / np.sqrt(vhat + eps)"),
    "laprop_raw_gradient_in_momentum": ("(1.0 - beta1) * g / (np.sqrt(vhat) + eps)", "(1.0 - beta1) * g"),
    "laprop_no_second_moment_correction": ("vhat = v2 / (1.0 - beta2 ** step)\n    m2", "vhat = v2\n    m2"),
    "laprop_no_momentum_correction": ("lr * m2 / (1.0 - beta1 ** step)", "lr * m2"),
    "laprop_root_after_eps": ("g / (np.sqrt(vhat) + eps)", "g / np.sqrt(vhat + eps)"),
    "momentum_dampened": ("b2 = mu * np.asarray(b, np.float64) + g", "b2 = mu * np.asarray(b, np.float64) + (1.0 - mu) * g"),
    "momentum_old_buffer": ("p2 = np.asarray(p, np.float64) - lr * b2", "p2 = np.asarray(p, np.float64) - lr * (b2 - g)"),
    "sgd_sign": ("return (np.asarray(p, np.float64) - lr * g)", "return (np.asarray(p, np.float64) + lr * g)"),
    "bf16_truncate": ("u + np.uint64(0x7FFF) + lsb", "u"),
}

NAMES = ["forward", "backward", "loss_and_grad", "train_step", "run_steps", "adam_update",
         "sgd_update", "gelu_tanh", "gelu_tanh_grad", "attention_fwd", "attention_bwd",
         "bf16_round", "laprop_update", "sgd_momentum_update"]


def _load_mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def test_unmutated_oracle_passes_every_pin():
    assert all(ok for _, ok in pins.all_checks())


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(mutation, monkeypatch):
    mod = _load_mutant(*MUTATIONS[mutation])
    for n in NAMES:
        monkeypatch.setattr(oracle, n, getattr(mod, n))
    failed = [name for name, ok in pins.all_checks() if not ok]
    assert failed, f"no pin caught {mutation}"
