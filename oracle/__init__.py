"""CPU oracle for the training step (test infrastructure only; see ``step``)."""
from .step import (MOMENTS, adam_update, attention_bwd, attention_fwd, backward,  # noqa: F401
                   bf16_round, forward, gelu_tanh, gelu_tanh_grad, laprop_update,
                   loss_and_grad, run_steps, sgd_momentum_update, sgd_update, train_step)
