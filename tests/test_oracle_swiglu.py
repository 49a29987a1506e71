"""Pins for the fp64 fused gate-up SwiGLU oracle (CPU): PyTorch autograd of
silu(gate) * up in fp64 (library special case), central finite differences of
the backward, and closed forms (silu(0) = 0, silu'(0) = 1/2, silu(a) - silu(-a)
= a, the derivative's zero near a = -1.2785)."""
import numpy as np
import torch

from oracle import swiglu as osw


def test_forward_and_backward_match_torch_autograd():
    g = np.random.default_rng(3)
    T, n = 7, 13
    x = g.normal(0, 3, (T, 2 * n))
    dy = g.normal(0, 1, (T, n))
    xt = torch.tensor(x, requires_grad=True)
    yt = torch.nn.functional.silu(xt[:, :n]) * xt[:, n:]
    yt.backward(gradient=torch.tensor(dy))
    np.testing.assert_allclose(osw.forward(x, n), yt.detach().numpy(), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(osw.backward(x, dy, n), xt.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_backward_matches_central_differences():
    g = np.random.default_rng(4)
    T, n = 3, 5
    x = g.normal(0, 2, (T, 2 * n))
    dy = g.normal(0, 1, (T, n))
    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = ((osw.forward(xp, n) - osw.forward(xm, n)) * dy).sum() / (2 * h)
    got = osw.backward(x, dy, n)
    assert np.abs(fd - got).max() <= 1e-7 * max(1.0, np.abs(got).max())


def test_closed_forms():
    a = np.array([[0.0, 3.0, -3.0, 40.0, -40.0, -800.0]])
    n = a.shape[1]
    x = np.concatenate([a, np.ones_like(a)], axis=1)
    y = osw.forward(x, n)[0]
    assert y[0] == 0.0 and y[5] == 0.0
    np.testing.assert_allclose(y[1] - y[2], 3.0, rtol=1e-15)   # silu(a) - silu(-a) = a
    np.testing.assert_allclose(y[3], 40.0, rtol=1e-15)
    dx = osw.backward(x, np.ones_like(a), n)[0]
    assert dx[0] == 0.5                                         # silu'(0) = 1/2
    # silu' has one zero, near a = -1.27846454
    r = -1.2784645427610738
    xr = np.array([[r, 1.0]])
    assert abs(osw.backward(xr, np.ones((1, 1)), 1)[0, 0]) < 1e-12


def test_backward_terms_bound_the_gradient_and_equal_it_without_cancellation():
    # |d_gate| <= t_gate with equality when both products share a sign (gate
    # a >= 0), and d_up is a single product, so t_up = |d_up|
    g = np.random.default_rng(6)
    T, n = 9, 17
    x = g.normal(0, 3, (T, 2 * n))
    dy = g.normal(0, 1, (T, n))
    d = osw.backward(x, dy, n)
    t = osw.backward_terms(x, dy, n)
    assert np.all(np.abs(d) <= t * (1 + 1e-14))
    a = x[:, :n]
    np.testing.assert_allclose(t[:, :n][a >= 0], np.abs(d[:, :n][a >= 0]), rtol=1e-14)
    np.testing.assert_allclose(t[:, n:], np.abs(d[:, n:]), rtol=1e-14)


def test_backward_terms_against_torch_pieces():
    # the two products of d_gate from torch: dy b sigmoid(a), and dy b a sigmoid'(a)
    # with sigmoid' from autograd; the product of d_up as dy silu(a)
    g = np.random.default_rng(7)
    T, n = 5, 11
    x = g.normal(0, 4, (T, 2 * n))
    dy = g.normal(0, 1, (T, n))
    a = torch.tensor(x[:, :n], requires_grad=True)
    b = torch.tensor(x[:, n:])
    dyt = torch.tensor(dy)
    s = torch.sigmoid(a)
    s.backward(torch.ones_like(s))
    ds = a.grad
    t_gate = (dyt * b * s).abs() + (dyt * b * a.detach() * ds).abs()
    t_up = (dyt * torch.nn.functional.silu(a.detach())).abs()
    want = torch.cat([t_gate, t_up], dim=1).detach().numpy()
    np.testing.assert_allclose(osw.backward_terms(x, dy, n), want, rtol=1e-13, atol=1e-300)


def test_backward_terms_hand_worked():
    # a = 0: sigmoid = 1/2 -> t_gate = |dy b| / 2, t_up = 0
    # a = 2, b = 3, dy = -1: sigmoid(2) = 0.8807970779778823;
    #   t_gate = 3 s + 3 * 2 * s (1 - s), t_up = 2 s
    # at the zero r of silu' (1 + r (1 - s) = 0), t_gate = 2 |dy b s(r)| while d_gate = 0
    s2 = 0.8807970779778823
    r = -1.2784645427610738
    sr = 1.0 / (1.0 + np.exp(-r))
    x = np.array([[0.0, 2.0, r, 5.0, 3.0, 1.5]])
    dy = np.array([[2.0, -1.0, 1.0]])
    t = osw.backward_terms(x, dy, 3)[0]
    np.testing.assert_allclose(t[0], 5.0, rtol=1e-15)
    np.testing.assert_allclose(t[1], 3 * s2 + 6 * s2 * (1 - s2), rtol=1e-14)
    np.testing.assert_allclose(t[2], 2 * 1.5 * sr, rtol=1e-12)
    assert t[3] == 0.0
    np.testing.assert_allclose(t[4], 2 * s2, rtol=1e-14)
    np.testing.assert_allclose(t[5], abs(r) * sr, rtol=1e-14)
