"""CPU oracle for the training step (test infrastructure only; see ``step``)."""
from .step import (adam_update, attention_bwd, attention_fwd, backward, bf16_round,  # noqa: F401
                   forward, gelu_tanh, gelu_tanh_grad, loss_and_grad, run_steps,
                   sgd_update, train_step)
