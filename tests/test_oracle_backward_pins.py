"""Pins of the oracle's backward pass (CPU only).

The page ("Folding Tensor and Sequence Parallelism for Memory-Efficient Transformer
Training & Inference") names training but prints no backward formulas, so the
backward is the chain rule of the forward layer. It is pinned to torch autograd in
float64 (a library the oracle does not use), to central finite differences on tiny
inputs, to closed forms, and its rank-by-rank restatement (the forward schedules
run in reverse) to the plain one for several D. Planted mistakes must be caught.
"""
import math
import types

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _weights(H, F, seed, scale=0.3):
    rng = np.random.default_rng(seed)
    W = {k: rng.standard_normal((H, H)) * scale for k in ("Wq", "Wk", "Wv", "Wo")}
    W["W1"] = rng.standard_normal((F, H)) * scale
    W["W3"] = rng.standard_normal((F, H)) * scale
    W["W2"] = rng.standard_normal((H, F)) * scale
    return W


def _torch_layer(x, W, heads):
    S, H = x.shape
    d = H // heads
    sp = lambda a: a.view(S, heads, d).transpose(0, 1)
    att = torch.nn.functional.scaled_dot_product_attention(
        sp(x @ W["Wq"].T), sp(x @ W["Wk"].T), sp(x @ W["Wv"].T), is_causal=True)
    h = x + att.transpose(0, 1).reshape(S, H) @ W["Wo"].T
    return h + (torch.nn.functional.silu(h @ W["W1"].T) * (h @ W["W3"].T)) @ W["W2"].T


def check_layer_backward_vs_autograd(o):
    S, H, heads, F = 12, 8, 2, 6
    x, dout = _rand((S, H), 1), _rand((S, H), 2)
    W = _weights(H, F, 3)
    got = o.layer_backward(x, W, heads, dout)
    tx = torch.from_numpy(x).requires_grad_()
    tW = {k: torch.from_numpy(v).requires_grad_() for k, v in W.items()}
    _torch_layer(tx, tW, heads).backward(torch.from_numpy(dout))
    assert np.abs(got["dx"] - tx.grad.numpy()).max() < 1e-10
    for k in W:
        assert np.abs(got["d" + k] - tW[k].grad.numpy()).max() < 1e-10, k


def _torch_layer_batched(x, W, heads):
    """The layer on a micro-batch [B, S, H]: torch's batched causal attention keeps
    every sequence to itself."""
    Bn, S, H = x.shape
    d = H // heads
    sp = lambda a: a.view(Bn, S, heads, d).transpose(1, 2)
    att = torch.nn.functional.scaled_dot_product_attention(
        sp(x @ W["Wq"].T), sp(x @ W["Wk"].T), sp(x @ W["Wv"].T), is_causal=True)
    h = x + att.transpose(1, 2).reshape(Bn, S, H) @ W["Wo"].T
    return h + (torch.nn.functional.silu(h @ W["W1"].T) * (h @ W["W3"].T)) @ W["W2"].T


def check_batched_backward_vs_autograd(o):
    # the gradient of the summed micro-batch loss, against torch autograd in float64
    Bn, S, H, heads, F = 3, 10, 8, 2, 6
    x, dout = _rand((Bn, S, H), 4), _rand((Bn, S, H), 5)
    W = _weights(H, F, 6)
    got = o.layer_backward_batched(x, W, heads, dout)
    tx = torch.from_numpy(x).requires_grad_()
    tW = {k: torch.from_numpy(v).requires_grad_() for k, v in W.items()}
    _torch_layer_batched(tx, tW, heads).backward(torch.from_numpy(dout))
    assert got["dx"].shape == x.shape
    assert np.abs(got["dx"] - tx.grad.numpy()).max() < 1e-10
    for k in W:
        assert np.abs(got["d" + k] - tW[k].grad.numpy()).max() < 1e-10, k


def check_attention_backward_finite_differences(o):
    n, d = 5, 3
    q, k, v, do = (_rand((n, d), s) for s in (4, 5, 6, 7))
    pos = np.arange(n)
    dq, dk, dv = o.causal_attention_head_backward(q, k, v, pos, pos, do)
    loss = lambda q_, k_, v_: float((o.causal_attention_head(q_, k_, v_, pos, pos) * do).sum())
    eps = 1e-6
    for arr, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        for idx in np.ndindex(arr.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += eps
            up = loss(*args)
            args[which][idx] -= 2 * eps
            num = (up - loss(*args)) / (2 * eps)
            assert abs(num - g[idx]) < 1e-7, (which, idx, num, g[idx])


def check_closed_forms(o):
    assert o.silu_grad(np.array(0.0)) == 0.5
    z = np.linspace(-6, 6, 25)
    num = (o.silu(z + 1e-6) - o.silu(z - 1e-6)) / 2e-6
    assert np.abs(o.silu_grad(z) - num).max() < 1e-8
    # query 0 attends only to key 0: its gradient reaches v_0 alone (dv_0 += do_0)
    # and none reaches q_0 or k_0 (a one-key softmax is constant)
    q, k, v, do = (_rand((1, 4), s) for s in (8, 9, 10, 11))
    dq, dk, dv = o.causal_attention_head_backward(q, k, v, np.array([0]), np.array([0]), do)
    assert np.abs(dv - do).max() < 1e-15 and np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
    # a zero output gradient gives zero gradients everywhere
    S, H = 6, 4
    W = _weights(H, 4, 12)
    g = o.layer_backward(_rand((S, H), 13), W, 2, np.zeros((S, H)))
    assert all(np.abs(v).max() == 0 for v in g.values())


def check_tsp_backward_equals_plain(o):
    S, H, heads, F = 16, 16, 4, 8
    x, dout = _rand((S, H), 14), _rand((S, H), 15)
    W = _weights(H, F, 16)
    plain = o.layer_backward(x, W, heads, dout)
    for D in (1, 2, 4):
        tsp = o.tsp_layer_backward(x, W, heads, D, dout)
        for key in plain:
            err = np.abs(tsp[key] - plain[key]).max() / max(np.abs(plain[key]).max(), 1e-30)
            assert err < 1e-11, (D, key, err)


def check_block_backwards_vs_autograd(o):
    S, H, heads, F = 10, 8, 2, 6
    x, dy = _rand((S, H), 17), _rand((S, H), 18)
    W = _weights(H, F, 19)
    tW = {k: torch.from_numpy(v).requires_grad_() for k, v in W.items()}
    # MLP block alone
    th = torch.from_numpy(x).requires_grad_()
    ((torch.nn.functional.silu(th @ tW["W1"].T) * (th @ tW["W3"].T)) @ tW["W2"].T).backward(
        torch.from_numpy(dy))
    m = o.swiglu_mlp_backward(x, W["W1"], W["W3"], W["W2"], dy)
    assert np.abs(m["dh"] - th.grad.numpy()).max() < 1e-10
    for k in ("W1", "W3", "W2"):
        assert np.abs(m["d" + k] - tW[k].grad.numpy()).max() < 1e-10, k
    # attention block alone
    tx = torch.from_numpy(x).requires_grad_()
    sp = lambda a: a.view(S, heads, H // heads).transpose(0, 1)
    att = torch.nn.functional.scaled_dot_product_attention(
        sp(tx @ tW["Wq"].T), sp(tx @ tW["Wk"].T), sp(tx @ tW["Wv"].T), is_causal=True)
    (att.transpose(0, 1).reshape(S, H) @ tW["Wo"].T).backward(torch.from_numpy(dy))
    a = o.attention_block_backward(x, W["Wq"], W["Wk"], W["Wv"], W["Wo"], heads, dy)
    assert np.abs(a["dx"] - tx.grad.numpy()).max() < 1e-10
    for k in ("Wq", "Wk", "Wv", "Wo"):
        assert np.abs(a["d" + k] - tW[k].grad.numpy()).max() < 1e-10, k


def check_sampled_backwards(o):
    """The row / column sampled forms give the full forms' entries."""
    S, H, F = 12, 8, 10
    h, dy = _rand((S, H), 20), _rand((S, H), 21)
    W = _weights(H, F, 22)
    full = o.swiglu_mlp_backward(h, W["W1"], W["W3"], W["W2"], dy)
    rows, cols = np.array([0, 5, 11]), np.array([1, 4, 9])
    part = o.swiglu_mlp_backward(h, W["W1"], W["W3"], W["W2"], dy, rows=rows, ffn_cols=cols)
    assert np.abs(part["dh"] - full["dh"][rows]).max() < 1e-12
    assert np.abs(part["dW1"] - full["dW1"][cols]).max() < 1e-12
    assert np.abs(part["dW3"] - full["dW3"][cols]).max() < 1e-12
    assert np.abs(part["dW2"] - full["dW2"][:, cols]).max() < 1e-12
    n, d = 11, 4
    q, k, v, do = (_rand((n, d), s) for s in (23, 24, 25, 26))
    pos = np.array([0, 1, 2, 8, 9, 10, 3, 4, 5, 6, 7])  # zigzag-like query order
    kpos = np.arange(n)
    dq, dk, dv = o.causal_attention_head_backward(q, k, v, pos, kpos, do)
    qr, kr = np.array([0, 3, 10]), np.array([0, 2, 7, 10])
    sq, sk, sv = o.causal_attention_head_backward_rows(q, k, v, pos, kpos, do, qr, kr, q_block=3)
    assert np.abs(sq - dq[qr]).max() < 1e-12
    assert np.abs(sk - dk[kr]).max() < 1e-12
    assert np.abs(sv - dv[kr]).max() < 1e-12


def check_rounded_output_delta(o):
    """Delta from the output itself (identity rounding) is the same gradient; a
    rounded output changes dq/dk but not dv; the sampled form takes the same option."""
    n, d = 10, 4
    q, k, v, do = (_rand((n, d), s) for s in (31, 32, 33, 34))
    pos = np.arange(n)
    exact = o.causal_attention_head_backward(q, k, v, pos, pos, do)
    ident = o.causal_attention_head_backward(q, k, v, pos, pos, do, o_round=lambda x: x)
    for a, b in zip(exact, ident):
        assert np.abs(a - b).max() < 1e-12
    coarse = lambda x: np.round(x * 8) / 8
    rq, rk, rv = o.causal_attention_head_backward(q, k, v, pos, pos, do, o_round=coarse)
    assert np.abs(rv - exact[2]).max() < 1e-12
    assert np.abs(rq - exact[0]).max() > 1e-3 and np.abs(rk - exact[1]).max() > 1e-3
    qr, kr = np.array([1, 7]), np.array([0, 5])
    sq, sk, sv = o.causal_attention_head_backward_rows(q, k, v, pos, pos, do, qr, kr, q_block=4,
                                                       o_round=coarse)
    assert np.abs(sq - rq[qr]).max() < 1e-12 and np.abs(sk - rk[kr]).max() < 1e-12


def check_attention_gradient_sums(o):
    """Per head, the key gradients sum to zero (each softmax row's dS sums to zero)
    and the value gradients sum to the output gradients (each P row sums to one)."""
    n, d = 9, 5
    q, k, v, do = (_rand((n, d), s) for s in (27, 28, 29, 30))
    pos = np.arange(n)
    dq, dk, dv = o.causal_attention_head_backward(q, k, v, pos, pos, do)
    assert np.abs(dk.sum(axis=0)).max() < 1e-12
    assert np.abs(dv.sum(axis=0) - do.sum(axis=0)).max() < 1e-12


def check_stored_backward(o):
    """The stored-precision backward (store=...): with the identity it is the exact
    backward; with a coarse grid (multiples of 1/16, so that each rounding point
    matters) the head's and the MLP's gradients equal library computations that
    round at the stated points: torch's softmax and autograd (scores -> dS,
    silu(a1) * a3 -> dA1, dA3), rounded where the docstrings say."""
    ident = lambda a: a
    S, H, heads, F = 10, 8, 2, 6
    x, dout = _rand((S, H), 40), _rand((S, H), 41)
    W = _weights(H, F, 42)
    ex, st = o.layer_backward(x, W, heads, dout), o.layer_backward(x, W, heads, dout, store=ident)
    for k in ex:
        assert np.abs(ex[k] - st[k]).max() < 1e-12, k
    coarse = lambda a: np.round(np.asarray(a) * 16) / 16
    # one head: P rounded before dv, dS before dq and dk (Delta from the exact O)
    n, d = 9, 4
    q, k, v, do = (_rand((n, d), s) for s in (43, 44, 45, 46))
    pos = np.arange(n)
    dq, dk, dv = o.causal_attention_head_backward(q, k, v, pos, pos, do, store=coarse)
    ts = (torch.from_numpy(q) @ torch.from_numpy(k).T / math.sqrt(d)).requires_grad_()
    mask = torch.ones(n, n, dtype=torch.bool).tril()
    P = torch.softmax(ts.masked_fill(~mask, float("-inf")), dim=1)
    (P @ torch.from_numpy(v)).backward(torch.from_numpy(do))
    dS = coarse(ts.grad.numpy())
    assert np.abs(dv - coarse(P.detach().numpy()).T @ do).max() < 1e-12
    assert np.abs(dq - dS @ k / math.sqrt(d)).max() < 1e-12
    assert np.abs(dk - dS.T @ q / math.sqrt(d)).max() < 1e-12
    # MLP: A1, A3 kept rounded; dA1, dA3 from them, rounded; G rounded before dW2
    h, dy = coarse(_rand((S, H), 47)), _rand((S, H), 48)
    g = o.swiglu_mlp_backward(h, W["W1"], W["W3"], W["W2"], dy, store=coarse)
    a1 = torch.from_numpy(coarse(h @ W["W1"].T)).requires_grad_()
    a3 = torch.from_numpy(coarse(h @ W["W3"].T)).requires_grad_()
    (torch.nn.functional.silu(a1) * a3).backward(torch.from_numpy(dy @ W["W2"]))
    dA1, dA3 = coarse(a1.grad.numpy()), coarse(a3.grad.numpy())
    G = coarse((torch.nn.functional.silu(torch.from_numpy(h @ W["W1"].T))
                * torch.from_numpy(h @ W["W3"].T)).numpy())
    assert np.abs(g["dh"] - (dA1 @ W["W1"] + dA3 @ W["W3"])).max() < 1e-12
    assert np.abs(g["dW1"] - dA1.T @ h).max() < 1e-12
    assert np.abs(g["dW3"] - dA3.T @ h).max() < 1e-12
    assert np.abs(g["dW2"] - dy.T @ G).max() < 1e-12
    # the sampled forms take the same rounding
    qr, kr = np.array([0, 4, 8]), np.array([0, 3, 8])
    sq, sk, sv = o.causal_attention_head_backward_rows(q, k, v, pos, pos, do, qr, kr, q_block=4,
                                                       store=coarse)
    assert np.abs(sq - dq[qr]).max() < 1e-12 and np.abs(sk - dk[kr]).max() < 1e-12
    assert np.abs(sv - dv[kr]).max() < 1e-12


PINS = [check_layer_backward_vs_autograd, check_attention_backward_finite_differences,
        check_closed_forms, check_tsp_backward_equals_plain, check_block_backwards_vs_autograd,
        check_sampled_backwards, check_attention_gradient_sums, check_rounded_output_delta,
        check_batched_backward_vs_autograd, check_stored_backward]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_backward_pin(pin):
    pin(oracle)


def _mutant(**overrides):
    ns = types.SimpleNamespace(**{k: getattr(oracle, k) for k in oracle.__all__})
    for k, v in overrides.items():
        setattr(ns, k, v)
    return ns


def _attn_bwd_no_rowsum(q, k, v, q_pos, k_pos, do, o_round=None, store=None):
    d = q.shape[1]
    s = (q @ k.T) / math.sqrt(d)
    s = np.where(np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None], s, -np.inf)
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ds = p * (do @ v.T)  # the rowsum term dropped
    return ds @ k / math.sqrt(d), ds.T @ q / math.sqrt(d), p.T @ do


def _layer_bwd_wrong_dw2(x, W, heads, dout, store=None):
    g = oracle.layer_backward(x, W, heads, dout, store=store)
    g["dW2"] = g["dW2"] * 2.0
    return g


def _mlp_bwd_no_w3_path(h, W1, W3, W2, dmlp, rows=None, ffn_cols=None, store=None):
    g = oracle.swiglu_mlp_backward(h, W1, W3, W2, dmlp, rows, ffn_cols, store=store)
    r = slice(None) if rows is None else rows
    g["dh"] = g["dh"] - ((dmlp[r] @ W2) * oracle.silu(h[r] @ W1.T)) @ W3
    return g


def _attn_rows_unnormalised(q, k, v, q_pos, k_pos, do, q_rows, k_rows, q_block=1024,
                            o_round=None, store=None):
    dq, dk, dv = oracle.causal_attention_head_backward_rows(q, k, v, q_pos, k_pos, do,
                                                            q_rows, k_rows, q_block, o_round, store)
    return dq, dk, dv * 1.5


def _batched_bwd_mean(x, W, heads, dout, store=None):
    """Mistake: weight gradients averaged over the micro-batch instead of summed."""
    g = oracle.layer_backward_batched(x, W, heads, dout, store=store)
    return {k: (v if k == "dx" else v / x.shape[0]) for k, v in g.items()}


def _attn_bwd_store_skips_p(q, k, v, q_pos, k_pos, do, o_round=None, store=None):
    """Mistake: dv from the unrounded P (the stored form rounds P before dv)."""
    dq, dk, _ = oracle.causal_attention_head_backward(q, k, v, q_pos, k_pos, do, o_round, store)
    _, _, dv = oracle.causal_attention_head_backward(q, k, v, q_pos, k_pos, do, o_round)
    return dq, dk, dv


def _mlp_bwd_store_late(h, W1, W3, W2, dmlp, rows=None, ffn_cols=None, store=None):
    """Mistake: dA1, dA3 formed from the unrounded pre-activations."""
    if store is None:
        return oracle.swiglu_mlp_backward(h, W1, W3, W2, dmlp, rows, ffn_cols)
    g = oracle.swiglu_mlp_backward(h, W1, W3, W2, dmlp, rows, ffn_cols)
    r = slice(None) if rows is None else rows
    A1, A3 = h[r] @ W1.T, h[r] @ W3.T
    dG = dmlp[r] @ W2
    g["dh"] = store(dG * A3 * oracle.silu_grad(A1)) @ W1 + store(dG * oracle.silu(A1)) @ W3
    return g


MUTANTS = {
    "stored backward: dv from the unrounded P": dict(causal_attention_head_backward=_attn_bwd_store_skips_p),
    "stored backward: MLP pre-activations unrounded": dict(swiglu_mlp_backward=_mlp_bwd_store_late),
    "micro-batch weight gradients averaged": dict(layer_backward_batched=_batched_bwd_mean),
    "MLP dh without the W3 path": dict(swiglu_mlp_backward=_mlp_bwd_no_w3_path),
    "sampled attention dv scaled": dict(causal_attention_head_backward_rows=_attn_rows_unnormalised),
    "attention dS without the row-sum term": dict(causal_attention_head_backward=_attn_bwd_no_rowsum),
    "silu gradient without the z term": dict(silu_grad=lambda z: 1.0 / (1.0 + np.exp(-z))),
    "dW2 scaled": dict(layer_backward=_layer_bwd_wrong_dw2),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_backward_planted_mistake_is_caught(name):
    caught = 0
    for pin in PINS:
        try:
            pin(_mutant(**MUTANTS[name]))
        except AssertionError:
            caught += 1
    assert caught >= 1, name
