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
