"""Pins for the fp64 fused-linear-cross-entropy oracle (CPU): PyTorch autograd
on the same loss (library special case), central finite differences of the
hidden and weight gradients, the zero row-sum of grad_weight without softcap,
and the streamed / sampled evaluation against the direct one."""
import numpy as np
import pytest
import torch

from oracle import ce as oc
from oracle import flce as of

IGN = -100


def rng(seed):
    return np.random.default_rng(seed)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


@pytest.mark.parametrize("T,eps,red", [(0.0, 0.0, "mean"), (30.0, 0.0, "mean"), (5.0, 0.2, "sum")])
def test_matches_torch_autograd(T, eps, red):
    g = rng(1)
    N, H, V = 24, 40, 97
    h = g.normal(0, 1, (N, H))
    W = g.normal(0, 0.3, (V, H))
    lab = g.integers(0, V, N)
    lab[[3, 10]] = IGN
    gs = 0.7
    r = of.flce_fwd_bwd(h, W, lab, label_smoothing=eps, softcap=T, reduction=red, grad_scale=gs)
    ht = torch.tensor(h, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    S = ht @ Wt.T
    z = T * torch.tanh(S / T) if T > 0 else S
    loss = torch.nn.functional.cross_entropy(z, torch.tensor(lab), ignore_index=IGN,
                                             label_smoothing=eps, reduction=red)
    (gs * loss).backward()
    assert abs(r["reduced_loss"] - loss.item()) < 1e-10 * max(1, abs(loss.item()))
    np.testing.assert_allclose(r["grad_hidden"], ht.grad.numpy(), rtol=1e-9, atol=1e-14)
    np.testing.assert_allclose(r["grad_weight"], Wt.grad.numpy(), rtol=1e-9, atol=1e-14)


def test_gradients_match_central_differences():
    g = rng(2)
    N, H, V = 4, 5, 7
    h = g.normal(0, 1, (N, H))
    W = g.normal(0, 0.5, (V, H))
    lab = np.array([1, IGN, 6, 0])
    kw = dict(label_smoothing=0.15, softcap=2.5, reduction="mean", grad_scale=1.3)
    r = of.flce_fwd_bwd(h, W, lab, **kw)

    def f(hh, WW):
        return 1.3 * of.flce_fwd_bwd(hh, WW, lab, want_grad=False, **kw)["reduced_loss"]

    eps = 1e-6
    for M, G, which in ((h, r["grad_hidden"], 0), (W, r["grad_weight"], 1)):
        fd = np.zeros_like(M)
        for idx in np.ndindex(M.shape):
            Mp, Mm = M.copy(), M.copy()
            Mp[idx] += eps
            Mm[idx] -= eps
            args_p = (Mp, W) if which == 0 else (h, Mp)
            args_m = (Mm, W) if which == 0 else (h, Mm)
            fd[idx] = (f(*args_p) - f(*args_m)) / (2 * eps)
        assert np.abs(fd - G).max() <= 1e-6 * np.abs(G).max()


def test_weight_gradient_rows_sum_to_zero_without_softcap():
    g = rng(3)
    N, H, V = 30, 16, 50
    h = g.normal(0, 1, (N, H))
    W = g.normal(0, 0.4, (V, H))
    lab = g.integers(0, V, N)
    r = of.flce_fwd_bwd(h, W, lab, label_smoothing=0.1)
    # sum_j G[r, j] = 0 for every row, so sum_j grad_W[j, :] = (G 1)^T h = 0
    np.testing.assert_allclose(r["grad_weight"].sum(axis=0), 0, atol=1e-13)


@pytest.mark.parametrize("T,eps", [(0.0, 0.0), (30.0, 0.1)])
def test_streamed_and_sampled_match_the_direct_evaluation(T, eps):
    g = rng(4)
    N, H, V = 33, 24, 101
    hb = bf16_bits(g.normal(0, 1, (N, H)))
    Wb = bf16_bits(g.normal(0, 0.5, (V, H)))
    lab = g.integers(0, V, N)
    lab[[0, 7]] = IGN
    h, W = of.widen_bf16(hb), of.widen_bf16(Wb)
    full = of.flce_fwd_bwd(h, W, lab, label_smoothing=eps, softcap=T, reduction="mean")
    rows = np.array([0, 1, 5, 32])
    cols = np.array([0, 3, 50, 100])
    s = of.sampled(hb, Wb, lab, rows, cols, label_smoothing=eps, softcap=T, reduction="mean",
                   block=7)
    np.testing.assert_allclose(s["loss"], full["loss"], rtol=1e-12, atol=1e-12)
    assert np.array_equal(s["argmax"], full["argmax"])
    assert abs(s["reduced_loss"] - full["reduced_loss"]) < 1e-12
    assert s["n_correct"] == full["n_correct"] and s["n_valid"] == full["n_valid"]
    np.testing.assert_allclose(s["grad_hidden_rows"], full["grad_hidden"][rows], rtol=1e-10,
                               atol=1e-15)
    np.testing.assert_allclose(s["grad_weight_cols"], full["grad_weight"][cols], rtol=1e-10,
                               atol=1e-15)


def test_grad_columns_equals_the_row_gradient_given_the_row_lse():
    g = rng(5)
    n, V = 9, 40
    x = g.normal(0, 3, (n, V))
    lab = g.integers(0, V, n)
    lab[2] = IGN
    r = oc.ce_fwd_bwd(x, "f64", V, lab, label_smoothing=0.3, softcap=6.0, reduction="sum",
                      grad_scale=0.5)
    from scipy.special import logsumexp
    lse = logsumexp(6.0 * np.tanh(x / 6.0), axis=1)
    cols = np.array([0, 5, 39, 17])
    gc = oc.grad_columns(x[:, cols], cols, V, lab, lse, np.full(n, 0.5), label_smoothing=0.3,
                         softcap=6.0)
    np.testing.assert_allclose(gc, r["grad"][:, cols], rtol=1e-11, atol=1e-16)


@pytest.mark.parametrize("block", [1, 3, 7, 64])
def test_row_stats_two_largest_logits_against_a_full_sort(block):
    # brute force: the two largest entries of each fully formed row of S
    # (with multiplicity), including maxima duplicated in one block, across
    # blocks, and rows whose runner-up sits in an earlier block
    g = rng(8)
    N, H, V = 12, 16, 37
    h = g.normal(0, 1, (N, H))
    Wf = g.normal(0, 0.5, (V, H))
    Wf[20] = Wf[5]          # exact duplicate column (any h): duplicated maximum possible
    Wf[6] = Wf[5]           # in the same block as column 5 for blocks >= 7
    h[0] = 0.0              # a row of all-equal logits
    Wb = bf16_bits(Wf)
    lab = g.integers(0, V, N)
    st = of.row_stats(h, Wb, lab, block=block)
    # one product per row and column, in Python loops (fp64 dot products; the
    # blocked matmuls may round the last bit differently)
    W64 = of.widen_bf16(Wb)
    S = np.array([[float(np.dot(h[i], W64[j])) for j in range(V)] for i in range(N)])
    srt = np.sort(S, axis=1)
    np.testing.assert_allclose(st["top"], srt[:, -1], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(st["second"], srt[:, -2], rtol=1e-13, atol=1e-15)
    # the argmax is a column holding the maximum (up to the last-bit rounding
    # of duplicated columns)
    at = S[np.arange(N), st["argmax"]]
    np.testing.assert_allclose(at, srt[:, -1], rtol=1e-13, atol=1e-15)
    # the duplicated columns make near-exact ties: second = top on those rows
    dup = np.isclose(S[:, 5], srt[:, -1], rtol=1e-13, atol=1e-15)
    assert dup.any()
    np.testing.assert_allclose(st["second"][dup], st["top"][dup], rtol=1e-13, atol=1e-15)
