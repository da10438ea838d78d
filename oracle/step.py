"""CPU oracle: one training step of a typed static graph, written out plainly.

TEST INFRASTRUCTURE ONLY.  This package is the independent checker of the CUDA
library.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
import it; the library never calls it and shares no code with it.

What it computes follows "Meganeura: Portable GPU Training and Inference through
Vulkan and Metal" (abstract: a typed static graph, automatic differentiation,
optimizer) and the "Meganeura" README (Example section: matmul(x, w) with
w[in, out], relu, cross_entropy_loss against a dense label tensor; Contents
section: SGD and Adam optimizers).  The pages print no formulas, so each step
below is the textbook definition, in float64 (numpy), with the reading taken
where the pages are silent:

* Linear: Z = X W (+ b), W stored [in, out] row-major as in the Example.
* ReLU, derivative 1 if z > 0 else 0 (0 at z = 0).
* GELU, tanh form: 0.5 z (1 + tanh(u)), u = sqrt(2/pi) (z + 0.044715 z^3).
* RMSNorm: r = 1/sqrt(mean(x^2) + eps), y = x r gamma.
* Residual: out = skip + branch.
* Causal attention per (batch, head): S = Q K^T / sqrt(d_h), keys j > i masked,
  P = softmax(S), O = P V; heads are column blocks of the fused QKV tensor.
* Cross-entropy, mean over rows: L = -(1/B) sum_b sum_c y_bc log softmax(z_b)_c
  (dense labels) or -(1/B) sum_b log softmax(z_b)[t_b] (integer labels).
* Mean squared error over all elements.
* Backward: the chain rule applied layer by layer in reverse.
* SGD: p -= lr g.  Adam (t = step, from 1): bias-corrected moments, eps added
  after the square root, no weight decay.
* LaProp (named beside Adam in the paper's checkpoint notes; its update is the
  published algorithm of Ziyin, Wang & Ueda, "LaProp: Separating Momentum and
  Adaptivity in Adam", 2020): the gradient is divided by the bias-corrected
  root of its second moment before it enters the momentum.
* SGD with momentum (heavy ball, no dampening): b = mu b + g, p -= lr b, with
  mu in the descriptor's beta1.

Precision: float64 arithmetic throughout, with the storage types of the typed
static graph.  Three modes:

* "exact": every value kept in float64 (used by the finite-difference pins);
* "strict": every graph value -- each layer's output and the gradient with
  respect to each value -- is stored as float32 (strict f32);
* "bf16": x, the weight matrices, the MSE target and every graph value and
  value gradient are stored as bf16 (round to nearest even), as the bf16
  workloads specify, with the master weights and Adam moments in fp32.

Arithmetic inside an op is float64 on the stored operands, rounded once to the
value type.  Parameter gradients are float64; parameters and Adam moments are
stored back as float32 after each update (fp32 master weights).

Parity status: every function here is pinned by the CPU tests (finite
differences, closed forms, brute force on tiny graphs, invariants, and PyTorch
CPU float64 autograd as an outside opinion).
"""
from __future__ import annotations

import math

import numpy as np

SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
GELU_C = 0.044715


# --------------------------------------------------------------------------
# bf16 rounding (round to nearest, ties to even) of float32 values
# --------------------------------------------------------------------------

def bf16_round(a) -> np.ndarray:
    """float32 -> bf16 -> float64, round to nearest even on the 16 dropped bits."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def store(a, precision):
    """Round a value to the storage type of the graph's values."""
    if precision == "bf16":
        return bf16_round(a)
    if precision == "strict":
        return np.asarray(a, np.float64).astype(np.float32).astype(np.float64)
    return np.asarray(a, np.float64)


# --------------------------------------------------------------------------
# Pointwise functions
# --------------------------------------------------------------------------

def gelu_tanh(z):
    u = SQRT_2_OVER_PI * (z + GELU_C * z ** 3)
    return 0.5 * z * (1.0 + np.tanh(u))


def gelu_tanh_grad(z):
    u = SQRT_2_OVER_PI * (z + GELU_C * z ** 3)
    t = np.tanh(u)
    du = SQRT_2_OVER_PI * (1.0 + 3.0 * GELU_C * z ** 2)
    return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * du


def log_softmax_rows(z):
    m = z.max(axis=1, keepdims=True)
    s = z - m
    return s - np.log(np.exp(s).sum(axis=1, keepdims=True))


# --------------------------------------------------------------------------
# Attention (one batch element, one head, full S x S matrix)
# --------------------------------------------------------------------------

def _attn_head_fwd(q, k, v):
    s_len, dh = q.shape
    scale = 1.0 / math.sqrt(dh)
    s = (q @ k.T) * scale
    mask = np.triu(np.ones((s_len, s_len), dtype=bool), k=1)   # j > i
    s = np.where(mask, -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    p = e / e.sum(axis=1, keepdims=True)
    return p @ v, p


def _attn_head_bwd(q, k, v, p, do):
    dh = q.shape[1]
    scale = 1.0 / math.sqrt(dh)
    dv = p.T @ do
    dp = do @ v.T
    ds = p * (dp - (dp * p).sum(axis=1, keepdims=True))
    dq = (ds @ k) * scale
    dk = (ds.T @ q) * scale
    return dq, dk, dv


def _attn_split(layer, rows):
    h, dh, s_len = layer["n_heads"], layer["head_dim"], layer["seq_len"]
    if rows % s_len:
        raise ValueError("rows must be a multiple of seq_len")
    return h, dh, s_len, rows // s_len


def attention_fwd(layer, qkv):
    """qkv [rows, 3*d] = [Q | K | V]; head h is columns h*dh..h*dh+dh-1 of each third."""
    rows = qkv.shape[0]
    h, dh, s_len, nb = _attn_split(layer, rows)
    d = h * dh
    out = np.zeros((rows, d))
    probs = {}
    for b in range(nb):
        r = slice(b * s_len, (b + 1) * s_len)
        for hh in range(h):
            c = slice(hh * dh, (hh + 1) * dh)
            q = qkv[r, c]
            k = qkv[r, d + hh * dh: d + (hh + 1) * dh]
            v = qkv[r, 2 * d + hh * dh: 2 * d + (hh + 1) * dh]
            o, p = _attn_head_fwd(q, k, v)
            out[r, c] = o
            probs[(b, hh)] = p
    return out, probs


def attention_bwd(layer, qkv, probs, dout):
    rows = qkv.shape[0]
    h, dh, s_len, nb = _attn_split(layer, rows)
    d = h * dh
    dqkv = np.zeros_like(qkv)
    for b in range(nb):
        r = slice(b * s_len, (b + 1) * s_len)
        for hh in range(h):
            cq = slice(hh * dh, (hh + 1) * dh)
            ck = slice(d + hh * dh, d + (hh + 1) * dh)
            cv = slice(2 * d + hh * dh, 2 * d + (hh + 1) * dh)
            dq, dk, dv = _attn_head_bwd(qkv[r, cq], qkv[r, ck], qkv[r, cv],
                                        probs[(b, hh)], dout[r, cq])
            dqkv[r, cq] = dq
            dqkv[r, ck] = dk
            dqkv[r, cv] = dv
    return dqkv


# --------------------------------------------------------------------------
# Graph forward / loss / backward
# --------------------------------------------------------------------------

def _param_slots(layers):
    """For each layer, the indices of its tensors in the flat parameter list."""
    slots, i = [], 0
    for l in layers:
        if l["op"] == "linear":
            if l["bias"]:
                slots.append((i, i + 1))
                i += 2
            else:
                slots.append((i, None))
                i += 1
        elif l["op"] == "rmsnorm":
            slots.append((i,))
            i += 1
        else:
            slots.append(())
    return slots, i


def forward(layers, params, x, precision="exact"):
    """Returns (output [rows, d_out] float64, tape for backward).  Each layer's
    output is a graph value, stored in the precision's value type."""
    slots, _ = _param_slots(layers)
    bf16 = precision == "bf16"
    h = store(x, precision)
    tape, skips = [], []
    for l, sl in zip(layers, slots):
        op = l["op"]
        if op == "linear":
            w = params[sl[0]]
            w = bf16_round(w) if bf16 else np.asarray(w, dtype=np.float64)
            z = h @ w
            if sl[1] is not None:
                z = z + np.asarray(params[sl[1]], dtype=np.float64)
            tape.append({"x": h, "w": w})
            h = z
        elif op == "relu":
            tape.append({"z": h})
            h = np.maximum(h, 0.0)
        elif op == "gelu_tanh":
            tape.append({"z": h})
            h = gelu_tanh(h)
        elif op == "rmsnorm":
            g = np.asarray(params[sl[0]], dtype=np.float64)
            r = 1.0 / np.sqrt((h * h).mean(axis=1, keepdims=True) + l["eps"])
            tape.append({"x": h, "r": r, "g": g})
            h = h * r * g
        elif op == "residual_begin":
            skips.append(h)
            tape.append({})
            continue                       # no new value
        elif op == "residual_end":
            h = skips.pop() + h
            tape.append({})
        elif op == "causal_attention":
            o, probs = attention_fwd(l, h)
            tape.append({"qkv": h, "p": probs})
            h = o
        else:
            raise ValueError(op)
        h = store(h, precision)
    if skips:
        raise ValueError("unbalanced residual_begin")
    return h, tape


def loss_and_grad(kind, out, labels, precision="exact"):
    """Loss (float) and dLoss/dout (in float64; backward stores it) for the
    output of the last layer."""
    rows = out.shape[0]
    if kind == "ce_dense":
        y = np.asarray(labels, dtype=np.float64)
        lp = log_softmax_rows(out)
        loss = -(y * lp).sum() / rows
        p = np.exp(lp)
        grad = (p * y.sum(axis=1, keepdims=True) - y) / rows
        return float(loss), grad
    if kind == "ce_index":
        t = np.asarray(labels, dtype=np.int64)
        lp = log_softmax_rows(out)
        loss = -lp[np.arange(rows), t].sum() / rows
        grad = np.exp(lp)
        grad[np.arange(rows), t] -= 1.0
        return float(loss), grad / rows
    if kind == "mse":
        tgt = bf16_round(labels) if precision == "bf16" else np.asarray(labels, dtype=np.float64)
        diff = out - tgt
        n = diff.size
        return float((diff * diff).sum() / n), 2.0 * diff / n
    raise ValueError(kind)


def backward(layers, params, tape, dout, precision="exact"):
    """Gradients of every parameter (float64), in declaration order, and the
    gradient with respect to x.  The gradient with respect to each graph value
    is stored in the value type once all its contributions are summed (a
    residual's skip source receives two)."""
    slots, n = _param_slots(layers)
    grads = [None] * n
    dh = store(dout, precision)
    skip_grads = []
    rev = list(zip(layers, slots, tape))[::-1]
    for k, (l, sl, t) in enumerate(rev):
        op = l["op"]
        if op == "linear":
            grads[sl[0]] = t["x"].T @ dh
            if sl[1] is not None:
                grads[sl[1]] = dh.sum(axis=0)
            dh = dh @ t["w"].T
        elif op == "relu":
            dh = dh * (t["z"] > 0.0)
        elif op == "gelu_tanh":
            dh = dh * gelu_tanh_grad(t["z"])
        elif op == "rmsnorm":
            x, r, g = t["x"], t["r"], t["g"]
            grads[sl[0]] = (dh * x * r).sum(axis=0)
            gy = dh * g
            dh = r * (gy - x * r * r * (gy * x).mean(axis=1, keepdims=True))
        elif op == "residual_end":
            skip_grads.append(dh)
            continue                       # the same value gradient flows to both
        elif op == "residual_begin":
            dh = dh + skip_grads.pop()
        elif op == "causal_attention":
            dh = attention_bwd(l, t["qkv"], t["p"], dh)
        else:
            raise ValueError(op)
        # the value whose gradient dh now is: complete unless a residual_begin
        # (which adds the skip's share) comes next in the reverse walk
        if k + 1 < len(rev) and rev[k + 1][0]["op"] == "residual_begin":
            continue
        dh = store(dh, precision)
    return grads, dh


# --------------------------------------------------------------------------
# Optimizers
# --------------------------------------------------------------------------

def sgd_update(p, g, lr):
    return (np.asarray(p, np.float64) - lr * g).astype(np.float32)


def adam_update(p, g, m, v, lr, step, beta1, beta2, eps):
    """One Adam step, t = step (1-based).  Returns float32 (p, m, v)."""
    m2 = beta1 * np.asarray(m, np.float64) + (1.0 - beta1) * g
    v2 = beta2 * np.asarray(v, np.float64) + (1.0 - beta2) * g * g
    mhat = m2 / (1.0 - beta1 ** step)
    vhat = v2 / (1.0 - beta2 ** step)
    p2 = np.asarray(p, np.float64) - lr * mhat / (np.sqrt(vhat) + eps)
    return p2.astype(np.float32), m2.astype(np.float32), v2.astype(np.float32)


def laprop_update(p, g, m, v, lr, step, beta1, beta2, eps):
    """One LaProp step, t = step (1-based), in the published algorithm's order:
    v = b2 v + (1-b2) g^2; the gradient divided by sqrt(v / (1 - b2^t)) + eps
    enters the momentum m = b1 m + (1-b1) (that quotient); p -= lr m /
    (1 - b1^t).  Returns float32 (p, m, v)."""
    v2 = beta2 * np.asarray(v, np.float64) + (1.0 - beta2) * g * g
    vhat = v2 / (1.0 - beta2 ** step)
    m2 = beta1 * np.asarray(m, np.float64) + (1.0 - beta1) * g / (np.sqrt(vhat) + eps)
    p2 = np.asarray(p, np.float64) - lr * m2 / (1.0 - beta1 ** step)
    return p2.astype(np.float32), m2.astype(np.float32), v2.astype(np.float32)


def sgd_momentum_update(p, g, b, lr, mu):
    """Heavy-ball SGD: b = mu b + g, p -= lr b.  Returns float32 (p, b)."""
    b2 = mu * np.asarray(b, np.float64) + g
    p2 = np.asarray(p, np.float64) - lr * b2
    return p2.astype(np.float32), b2.astype(np.float32)


# optimizer name -> moments it keeps: (first, second)
MOMENTS = {"sgd": (False, False), "adam": (True, True), "laprop": (True, True),
           "sgd_momentum": (True, False)}


# --------------------------------------------------------------------------
# One full training step
# --------------------------------------------------------------------------

def train_step(layers, params, x, labels, loss_kind, precision, optimizer, lr, step,
               adam_m=None, adam_v=None, beta1=0.9, beta2=0.999, eps=1e-8):
    """Forward, loss, backward, update.  Returns a dict with the loss, the
    output, the float64 gradients (before the update) and the updated float32
    params / moments."""
    out, tape = forward(layers, params, x, precision)
    loss, dout = loss_and_grad(loss_kind, out, labels, precision)
    grads, _ = backward(layers, params, tape, dout, precision)
    new_p, new_m, new_v = [], [], []
    for i, (p, g) in enumerate(zip(params, grads)):
        if optimizer == "sgd":
            new_p.append(sgd_update(p, g, lr))
        elif optimizer in ("adam", "laprop"):
            upd = adam_update if optimizer == "adam" else laprop_update
            a, b, c = upd(p, g, adam_m[i], adam_v[i], lr, step, beta1, beta2, eps)
            new_p.append(a)
            new_m.append(b)
            new_v.append(c)
        elif optimizer == "sgd_momentum":
            a, b = sgd_momentum_update(p, g, adam_m[i], lr, beta1)
            new_p.append(a)
            new_m.append(b)
        else:
            raise ValueError(optimizer)
    return {"loss": loss, "out": out, "grads": grads, "params": new_p,
            "adam_m": new_m, "adam_v": new_v}


def run_steps(layers, params, x, labels, loss_kind, precision, optimizer, lr, n_steps,
              beta1=0.9, beta2=0.999, eps=1e-8):
    """n_steps steps on one fixed batch; returns the per-step results."""
    p = [np.asarray(a, np.float32).copy() for a in params]
    has_m, has_v = MOMENTS[optimizer]
    m = [np.zeros_like(a) for a in p] if has_m else None
    v = [np.zeros_like(a) for a in p] if has_v else None
    hist = []
    for t in range(1, n_steps + 1):
        r = train_step(layers, p, x, labels, loss_kind, precision, optimizer, lr, t,
                       m, v, beta1, beta2, eps)
        p = r["params"]
        if has_m:
            m = r["adam_m"]
        if has_v:
            v = r["adam_v"]
        hist.append(r)
    return hist
