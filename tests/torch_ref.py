"""PyTorch CPU float64 autograd version of a layer list: an outside opinion on
the oracle (library routines: F.gelu(tanh), F.rms_norm, scaled_dot_product_attention,
F.cross_entropy, F.mse_loss, torch.optim).  Test-only; never used by the library."""
import math

import numpy as np
import torch
import torch.nn.functional as F


def bf16(t):
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)


def f32(t):
    return t.to(torch.float32).to(torch.float64)


class Store(torch.autograd.Function):
    """A graph value in its storage type: rounds the value going forward and the
    (summed) gradient with respect to it going backward."""

    @staticmethod
    def forward(ctx, t, precision):
        ctx.precision = precision
        return _round(t, precision)

    @staticmethod
    def backward(ctx, g):
        return _round(g, ctx.precision), None


def _round(t, precision):
    if precision == "bf16":
        return bf16(t)
    if precision == "strict":
        return f32(t)
    return t


def forward(layers, params, x, precision):
    h = _round(x, precision)
    skips, i = [], 0
    for l in layers:
        op = l["op"]
        if op == "residual_begin":
            skips.append(h)
            continue
        if op == "linear":
            w = params[i]
            i += 1
            if precision == "bf16":
                w = w + (bf16(w) - w).detach()      # forward in bf16, gradient to w
            h = h @ w
            if l["bias"]:
                h = h + params[i]
                i += 1
        elif op == "relu":
            h = F.relu(h)
        elif op == "gelu_tanh":
            h = F.gelu(h, approximate="tanh")
        elif op == "rmsnorm":
            h = F.rms_norm(h, (l["d"],), weight=params[i], eps=l["eps"])
            i += 1
        elif op == "residual_end":
            h = skips.pop() + h
        elif op == "causal_attention":
            nh, dh, s = l["n_heads"], l["head_dim"], l["seq_len"]
            d = nh * dh
            nb = h.shape[0] // s
            q, k, v = h[:, :d], h[:, d:2 * d], h[:, 2 * d:]
            sh = lambda t: t.reshape(nb, s, nh, dh).transpose(1, 2)  # noqa: E731
            o = F.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True)
            h = o.transpose(1, 2).reshape(nb * s, d)
        h = Store.apply(h, precision)
    return h


def loss(kind, out, labels, precision):
    if kind == "ce_dense":
        return F.cross_entropy(out, labels)
    if kind == "ce_index":
        return F.cross_entropy(out, labels.long())
    t = bf16(labels) if precision == "bf16" else labels
    return F.mse_loss(out, t)


def run(w_layers, params, x, labels, kind, precision, optimizer, lr, steps,
        betas=(0.9, 0.999), eps=1e-8):
    ps = [torch.tensor(np.asarray(p, np.float64), requires_grad=True) for p in params]
    xt = torch.tensor(np.asarray(x, np.float64))
    lt = torch.tensor(np.asarray(labels))
    if kind != "ce_index":
        lt = lt.to(torch.float64)
    if optimizer == "sgd":
        opt = torch.optim.SGD(ps, lr=lr)
    else:
        opt = torch.optim.Adam(ps, lr=lr, betas=betas, eps=eps)
    hist = []
    for _ in range(steps):
        opt.zero_grad()
        out = forward(w_layers, ps, xt, precision)
        L = loss(kind, out, lt, precision)
        L.backward()
        grads = [p.grad.detach().numpy().copy() for p in ps]
        opt.step()
        hist.append({"loss": float(L.detach()), "grads": grads,
                     "params": [p.detach().numpy().copy() for p in ps]})
    return hist
