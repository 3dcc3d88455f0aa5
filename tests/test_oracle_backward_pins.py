"""Pins of the oracle's attention backward and log-sum-exp (CPU only).

attention_backward is checked against torch float64 autograd through
scaled_dot_product_attention (a library routine), against central finite
differences of the oracle's own forward attention, and against identities the
definition fixes: the key gradients of a head sum to zero (softmax rows sum to
one, so the score gradients of a row sum to zero), and the value gradients sum
to the output gradients of the rows that see every key.  Planted mistakes must
be caught.  attention_lse is checked against torch.logsumexp.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import stack as ofw


def _torch_grads(q, k, v, do, H, length, causal):
    S, D = q.shape
    hd = D // H
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    qt, kt, vt = t(q), t(k), t(v)
    j = torch.arange(S)
    allowed = (j[None, :] < length).expand(S, -1)
    if causal:
        allowed = allowed & (j[None, :] <= j[:, None])
    heads = lambda a: a.view(S, H, hd).transpose(0, 1)
    o = F.scaled_dot_product_attention(heads(qt), heads(kt), heads(vt), attn_mask=allowed)
    o = o.transpose(0, 1).reshape(S, D)
    dom = torch.tensor(do, dtype=torch.float64)
    dom[length:] = 0.0
    (o * dom).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("length", [1, 6, 11])
def test_backward_matches_torch_autograd(causal, length):
    r = np.random.default_rng(50 + length)
    S, D, H = 11, 24, 3
    q, k, v, do = (r.normal(size=(S, D)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, H, length, causal)
    tq, tk, tv = _torch_grads(q, k, v, do, H, length, causal)
    np.testing.assert_allclose(dq[:length], tq[:length], atol=1e-12)
    np.testing.assert_allclose(dk, tk, atol=1e-12)
    np.testing.assert_allclose(dv, tv, atol=1e-12)
    assert np.all(dq[length:] == 0.0)
    assert np.all(dk[length:] == 0.0) and np.all(dv[length:] == 0.0)


def test_backward_matches_finite_differences_of_the_forward():
    r = np.random.default_rng(60)
    S, D, H, length = 6, 8, 2, 5
    q, k, v, do = (r.normal(size=(S, D)) for _ in range(4))
    do[length:] = 0.0
    dq, dk, dv = oracle.attention_backward(q, k, v, do, H, length, True)
    loss = lambda q_, k_, v_: float((oracle.attention(q_, k_, v_, H, length, True) * do).sum())
    eps = 1e-6
    for name, a, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0), (2, 3), (4, 7), (1, 5)]:
            ap, am = a.copy(), a.copy()
            ap[idx] += eps
            am[idx] -= eps
            args_p = {"q": (ap, k, v), "k": (q, ap, v), "v": (q, k, ap)}[name]
            args_m = {"q": (am, k, v), "k": (q, am, v), "v": (q, k, am)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[idx]) < 1e-8, (name, idx, fd, g[idx])


def test_backward_identities():
    r = np.random.default_rng(70)
    S, D, H, length = 9, 16, 2, 9
    q, k, v, do = (r.normal(size=(S, D)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, H, length, False)
    # every row's score gradients sum to zero, so the key gradients of each head sum to zero
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    # without a mask every row's probabilities sum to one over all keys: sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)


def test_lse_matches_torch_logsumexp():
    r = np.random.default_rng(80)
    S, D, H, length = 10, 12, 3, 7
    q, k = r.normal(size=(S, D)), r.normal(size=(S, D))
    lse = oracle.attention_lse(q, k, H, length, True)
    hd = D // H
    for h in range(H):
        c = slice(h * hd, (h + 1) * hd)
        s = torch.tensor(q[:, c] @ k[:, c].T / np.sqrt(hd))
        j = torch.arange(S)
        s = s.masked_fill(~((j[None, :] < length) & (j[None, :] <= j[:, None])), float("-inf"))
        np.testing.assert_allclose(lse[h], torch.logsumexp(s, dim=1).numpy(), atol=1e-12)


def _plant_no_scale(q, k, v, dout, n_heads, length, causal):
    dq, dk, dv = ORIG(q, k, v, dout, n_heads, length, causal)
    hd = q.shape[1] // n_heads
    return dq * np.sqrt(hd), dk, dv


def _plant_sign(q, k, v, dout, n_heads, length, causal):
    dq, dk, dv = ORIG(q, k, v, dout, n_heads, length, causal)
    return dq, -dk, dv


def _plant_causal_strict(q, k, v, dout, n_heads, length, causal):
    # keys j < i instead of j <= i: emulate by shifting the keys one row down
    return ORIG(q, np.vstack([k[:1] * 0, k[:-1]]), np.vstack([v[:1] * 0, v[:-1]]), dout, n_heads, length, causal)


ORIG = ofw.attention_backward


@pytest.mark.parametrize("mut", [_plant_no_scale, _plant_sign, _plant_causal_strict])
def test_planted_backward_mistakes_are_caught(mut):
    r = np.random.default_rng(90)
    S, D, H, length = 8, 16, 2, 7
    q, k, v, do = (r.normal(size=(S, D)) for _ in range(4))
    dq, dk, dv = mut(q, k, v, do, H, length, True)
    tq, tk, tv = _torch_grads(q, k, v, do, H, length, True)
    diff = max(np.abs(dq[:length] - tq[:length]).max(), np.abs(dk - tk).max(), np.abs(dv - tv).max())
    assert diff > 1e-6, mut.__name__
