"""The allocation-free softmax cross-entropy entry point, for callers that may
not allocate device memory (a plugin or enqueue hook of another framework, or
a process whose device memory is reserved by its own caching allocator).

Checked through the C ABI in two ways:

* against the float64 CPU oracle (``oracle.loss_and_grad``), element by element
  on the full dlogits and on the loss, for both logit types (fp32, bf16), both
  label kinds (dense fp32 rows, int32 class ids) and widths whose rows are and
  are not multiples of 16 bytes (the vector and the scalar kernel), on two
  calls in a row with different row counts, so that nothing the first call
  left in the shared scratch array reaches the second;
* against the training step's own loss kernel reached through the existing
  entry points: the loss that mg_train_step reports and the last layer's bias
  gradient (the column sums of dlogits), on two calls in a row.

This file sorts last so that a run stopping at the first failure has already
run every other test; it passes alone and after the others."""
import numpy as np
import pytest

import oracle
from static_graph_nn_gb300 import Plan, binding
from static_graph_nn_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-4          # the strict-f32 gate of the parity tests (max|a-b| / max|b|)
BF16_REL = 2.0 ** -7  # one bf16 rounding step of the stored dlogits, relative


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _noalloc_ce(lib, logits, labels, label_kind):
    rows, cols = logits.shape
    dtype = 1 if logits.dtype == torch.bfloat16 else 0
    dlogits = torch.full_like(logits, float("nan"))
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    st = lib.mg_softmax_ce_noalloc(dtype, logits.data_ptr(), rows, cols, label_kind,
                                   labels.data_ptr(), dlogits.data_ptr(), loss.data_ptr(), None)
    assert st == binding.MG_OK, lib.mg_last_error(None)
    torch.cuda.synchronize()
    return float(loss.item()), dlogits.double().cpu().numpy()


def _inputs(rows, cols, label_kind, dtype, seed):
    """Seeded logits N(0, 3^2) and labels: int32 class ids, or dense rows that
    are one-hot except every fifth row, which holds soft weights summing to 1.3
    (the general (softmax * sum(y) - y) / rows form)."""
    rng = np.random.default_rng(seed)
    z = (3.0 * rng.standard_normal((rows, cols))).astype(np.float32)
    ids = rng.integers(0, cols, size=rows)
    if label_kind == 1:
        y = ids.astype(np.int32)
    else:
        y = np.zeros((rows, cols), np.float32)
        y[np.arange(rows), ids] = 1.0
        soft = rng.random((rows, cols)).astype(np.float32)
        soft *= 1.3 / soft.sum(axis=1, keepdims=True)
        y[::5] = soft[::5]
    zt = torch.from_numpy(z).cuda()
    if dtype == "bf16":
        zt = zt.to(torch.bfloat16)
    # what the kernel reads: the logits as stored
    z_stored = zt.double().cpu().numpy()
    return zt.contiguous(), torch.from_numpy(y).cuda().contiguous(), z_stored, y


def _check(dtype, label_kind, got_loss, got_d, z_stored, y):
    want_loss, want_d = oracle.loss_and_grad("ce_index" if label_kind else "ce_dense",
                                             z_stored, y)
    assert np.isfinite(got_d).all()
    assert abs(got_loss - want_loss) <= TOL * abs(want_loss), (got_loss, want_loss)
    scale = np.abs(want_d).max()
    err = np.abs(got_d - want_d)
    if dtype == "f32":
        assert err.max() <= TOL * scale, err.max() / scale
    else:
        # each stored value is the bf16 rounding of an fp32 value within the
        # strict gate of the exact one
        assert (err <= BF16_REL * np.abs(want_d) + TOL * scale).all(), \
            float((err - BF16_REL * np.abs(want_d)).max() / scale)
    return err.max() / scale


@pytest.mark.parametrize("cols", [10, 1000, 1003])
@pytest.mark.parametrize("label_kind", [0, 1])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_ce_matches_the_oracle(dtype, label_kind, cols):
    """Two calls in a row, the second with fewer rows and other data."""
    lib = binding.load()
    worst = 0.0
    for call, rows in enumerate((777, 301)):
        zt, yt, z_stored, y = _inputs(rows, cols, label_kind, dtype, seed=100 * cols + call)
        loss, d = _noalloc_ce(lib, zt, yt, label_kind)
        worst = max(worst, _check(dtype, label_kind, loss, d, z_stored, y))
    print(dtype, label_kind, cols, "max|a-b|/max|b| =", worst)


def test_noalloc_ce_many_classes_index_labels():
    """A 32000-class head (the residual network's) with index labels, bf16."""
    lib = binding.load()
    zt, yt, z_stored, y = _inputs(64, 32000, 1, "bf16", seed=7)
    loss, d = _noalloc_ce(lib, zt, yt, 1)
    _check("bf16", 1, loss, d, z_stored, y)


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
        loss_na, dlogits = _noalloc_ce(lib, logits, y, 0)
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
