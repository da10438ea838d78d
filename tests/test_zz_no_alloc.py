"""The allocation-free softmax cross-entropy entry point, for callers that may
not allocate device memory (a plugin or enqueue hook of another framework, or
a process whose device memory is reserved by its own caching allocator).

It is compared, through the C ABI, with the training step's own loss kernel as
reached through the existing entry points: the loss that mg_train_step reports
and the last layer's bias gradient (the column sums of dlogits), on two calls
in a row.  This file sorts last so that a run stopping at the first failure has
already run every other test; it passes alone and after the others."""
import ctypes

import numpy as np
import pytest

from static_graph_nn_gb300 import Plan, binding
from static_graph_nn_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-4     # the strict-f32 gate of the parity tests


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _noalloc_ce(lib, logits, labels):
    rows, cols = logits.shape
    dlogits = torch.empty_like(logits)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    st = lib.mg_softmax_ce_noalloc(0, logits.data_ptr(), rows, cols, 0, labels.data_ptr(),
                                   dlogits.data_ptr(), loss.data_ptr(), None)
    assert st == binding.MG_OK, lib.mg_last_error(None)
    torch.cuda.synchronize()
    return float(loss.item()), dlogits.double().cpu().numpy()


def test_noalloc_ce_matches_the_training_step():
    lib = binding.load()
    w = W.workload("c2")                       # 4096 x 10 logits, last Linear has a bias
    plan = Plan.for_workload(w, "strict")
    info = plan.param_info()
    flat = torch.zeros(plan.param_count, dtype=torch.float32)
    for (off, r, c), t in zip(info, W.init_params(w)):
        flat[off:off + r * c] = torch.from_numpy(t.reshape(-1))
    params = flat.cuda()
    grads = torch.zeros_like(params)
    m, v = torch.zeros_like(params), torch.zeros_like(params)
    x = torch.from_numpy(W.make_x(w)).cuda()
    y = torch.from_numpy(W.make_labels(w)).cuda()
    b_off, _, b_cols = info[-1]
    for step in (1, 2):                        # two calls in a row
        logits = torch.empty((w.batch, w.d_out), dtype=torch.float32, device="cuda")
        plan.forward(params, x, logits)
        loss_na, dlogits = _noalloc_ce(lib, logits, y)
        plan.train_step(params, grads, m, v, x, y, w.lr, step)   # same params, then updates them
        loss_step = plan.loss()
        db = grads[b_off:b_off + b_cols].double().cpu().numpy()
        assert abs(loss_na - loss_step) <= TOL * abs(loss_step), (step, loss_na, loss_step)
        db_na = dlogits.sum(axis=0)
        assert np.abs(db_na - db).max() <= TOL * np.abs(db).max(), step
    plan.close()


def test_noalloc_ce_rejects_too_many_rows():
    lib = binding.load()
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    p = dummy.data_ptr()
    st = lib.mg_softmax_ce_noalloc(0, p, 65537, 1, 0, p, p, p, None)
    assert st == binding.MG_ERR_INVALID_ARG
    assert b"65536" in lib.mg_last_error(None)
