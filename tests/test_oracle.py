"""Pins for the fp64 cross-entropy oracle, against facts that do not come from
the oracle itself: closed forms, invariants, finite differences, brute force
and the library special case (PyTorch's cross_entropy, which the pages name
as the same operation).  CPU only."""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

from oracle import ce as oc

IGN = -100


def rng(seed):
    return np.random.default_rng(seed)


def f64_rows(x):
    return np.ascontiguousarray(x, dtype=np.float64)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("V", [1, 2, 7, 100])
@pytest.mark.parametrize("eps", [0.0, 0.1, 1.0])
@pytest.mark.parametrize("T", [0.0, 30.0])
def test_uniform_logits_give_ln_V(V, eps, T):
    c = 1.75
    n = 3
    x = np.full((n, V), c)
    lab = np.array([0, V - 1, IGN])
    r = oc.ce_fwd_bwd(x, "f64", V, lab, label_smoothing=eps, softcap=T, reduction="sum",
                      grad_scale=0.5)
    assert abs(r["loss"][0] - math.log(V)) < 1e-12
    assert abs(r["loss"][1] - math.log(V)) < 1e-12
    assert r["loss"][2] == 0.0
    assert list(r["argmax"]) == [0, 0, 0]
    dz = 1.0 - math.tanh(c / T) ** 2 if T > 0 else 1.0
    for row, y in ((0, 0), (1, V - 1)):
        q = np.full(V, eps / V)
        q[y] += 1 - eps
        np.testing.assert_allclose(r["grad"][row], 0.5 * (1.0 / V - q) * dz, rtol=0, atol=1e-15)
    assert np.all(r["grad"][2] == 0)


def test_two_class_softplus():
    g = rng(1)
    x = g.normal(0, 3, size=(50, 2))
    lab = g.integers(0, 2, 50)
    r = oc.ce_fwd_bwd(x, "f64", 2, lab, reduction="sum")
    d = x[np.arange(50), 1 - lab] - x[np.arange(50), lab]
    np.testing.assert_allclose(r["loss"], np.logaddexp(0.0, d), rtol=1e-13, atol=1e-14)


def test_full_smoothing_is_lse_minus_mean():
    g = rng(2)
    x = g.normal(0, 2, size=(20, 33))
    lab = g.integers(0, 33, 20)
    r = oc.ce_fwd_bwd(x, "f64", 33, lab, label_smoothing=1.0, reduction="sum")
    np.testing.assert_allclose(r["loss"], logsumexp(x, axis=1) - x.mean(axis=1), rtol=1e-13)


@pytest.mark.parametrize("T", [0.0, 5.0])
def test_smoothed_loss_is_cross_entropy_to_q(T):
    g = rng(3)
    V = 57
    x = g.normal(0, 4, size=(30, V))
    lab = g.integers(0, V, 30)
    eps = 0.37
    r = oc.ce_fwd_bwd(x, "f64", V, lab, label_smoothing=eps, softcap=T, reduction="sum")
    z = T * np.tanh(x / T) if T > 0 else x
    logp = z - logsumexp(z, axis=1, keepdims=True)
    q = np.full((30, V), eps / V)
    q[np.arange(30), lab] += 1 - eps
    np.testing.assert_allclose(r["loss"], -(q * logp).sum(axis=1), rtol=1e-12)


# ------------------------------------------------------------------ invariants

def test_shift_invariance_without_softcap():
    g = rng(4)
    x = g.normal(0, 3, size=(16, 40))
    lab = g.integers(0, 40, 16)
    a = oc.ce_fwd_bwd(x, "f64", 40, lab, label_smoothing=0.2)
    b = oc.ce_fwd_bwd(x + 11.0, "f64", 40, lab, label_smoothing=0.2)
    np.testing.assert_allclose(a["loss"], b["loss"], rtol=1e-12)
    np.testing.assert_allclose(a["grad"], b["grad"], rtol=1e-10, atol=1e-17)


def test_column_permutation_equivariance():
    g = rng(5)
    V = 64
    x = g.normal(0, 3, size=(12, V))
    lab = g.integers(0, V, 12)
    perm = g.permutation(V)
    inv = np.argsort(perm)
    a = oc.ce_fwd_bwd(x, "f64", V, lab, label_smoothing=0.1, softcap=7.0)
    b = oc.ce_fwd_bwd(x[:, perm], "f64", V, inv[lab], label_smoothing=0.1, softcap=7.0)
    np.testing.assert_allclose(a["loss"], b["loss"], rtol=1e-12)
    np.testing.assert_allclose(a["grad"], b["grad"][:, inv], rtol=1e-10, atol=1e-17)


def test_huge_softcap_reduces_to_no_softcap():
    g = rng(6)
    x = g.normal(0, 3, size=(10, 90))
    lab = g.integers(0, 90, 10)
    a = oc.ce_fwd_bwd(x, "f64", 90, lab, label_smoothing=0.1, softcap=1e6)
    b = oc.ce_fwd_bwd(x, "f64", 90, lab, label_smoothing=0.1, softcap=0.0)
    np.testing.assert_allclose(a["loss"], b["loss"], atol=1e-9, rtol=0)
    np.testing.assert_allclose(a["grad"], b["grad"], atol=1e-9, rtol=0)


@pytest.mark.parametrize("T", [0.0, 3.0])
def test_gradient_rows_sum_to_zero(T):
    g = rng(7)
    V = 301
    x = g.normal(0, 2, size=(25, V))
    lab = g.integers(0, V, 25)
    r = oc.ce_fwd_bwd(x, "f64", V, lab, label_smoothing=0.3, softcap=T, reduction="sum")
    dz = 1 - np.tanh(x / T) ** 2 if T > 0 else np.ones_like(x)
    # sum_j (p_j - q_j) = 0 for a valid row
    np.testing.assert_allclose((r["grad"] / dz).sum(axis=1), 0, atol=1e-13)


@pytest.mark.parametrize("T,eps", [(0.0, 0.0), (0.0, 0.25), (2.5, 0.0), (2.5, 0.4)])
def test_gradient_matches_central_differences(T, eps):
    g = rng(8)
    n, V = 6, 13
    x = g.normal(0, 2, size=(n, V))
    lab = g.integers(0, V, n)
    lab[2] = IGN
    gs = 0.75
    r = oc.ce_fwd_bwd(x, "f64", V, lab, label_smoothing=eps, softcap=T, reduction="mean",
                      grad_scale=gs)

    def total(xx):
        rr = oc.ce_fwd_bwd(xx, "f64", V, lab, label_smoothing=eps, softcap=T, reduction="mean",
                           grad_scale=gs, want_grad=False)
        return gs * rr["reduced_loss"]

    h = 1e-6
    fd = np.zeros_like(x)
    for i in range(n):
        for j in range(V):
            xp = x.copy()
            xm = x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fd[i, j] = (total(xp) - total(xm)) / (2 * h)
    err = np.abs(fd - r["grad"]).max() / np.abs(r["grad"]).max()
    assert err < 1e-6, err
    assert np.all(r["grad"][2] == 0)


# ------------------------------------------------------- ignored rows, reductions

def test_ignored_rows_and_mean_over_valid_only():
    g = rng(9)
    V = 50
    x = g.normal(0, 2, size=(40, V))
    lab = g.integers(0, V, 40)
    lab[::4] = IGN
    s = oc.ce_fwd_bwd(x, "f64", V, lab, reduction="sum")
    m = oc.ce_fwd_bwd(x, "f64", V, lab, reduction="mean")
    assert s["n_valid"] == 30 and m["n_valid"] == 30
    assert np.all(s["loss"][::4] == 0) and np.all(s["grad"][::4] == 0)
    assert abs(s["reduced_loss"] / m["reduced_loss"] - 30) < 1e-12
    assert abs(s["loss"].sum() - s["reduced_loss"]) < 1e-10
    # the mean's gradient is the sum's divided by n_valid
    np.testing.assert_allclose(m["grad"] * 30, s["grad"], rtol=1e-12, atol=1e-18)


def test_all_rows_ignored():
    x = rng(10).normal(size=(5, 9))
    lab = np.full(5, IGN)
    r = oc.ce_fwd_bwd(x, "f64", 9, lab, reduction="mean")
    assert r["n_valid"] == 0 and r["reduced_loss"] == 0.0 and r["accuracy"] == 0.0
    assert np.all(r["grad"] == 0)


def test_bad_labels_are_flagged():
    x = rng(11).normal(size=(4, 9))
    lab = np.array([3, 9, -1, IGN])
    r = oc.ce_fwd_bwd(x, "f64", 9, lab, reduction="mean")
    assert r["n_valid"] == 1 and r["n_bad"] == 2
    assert np.isfinite(r["loss"][0]) and np.isnan(r["loss"][1]) and np.isnan(r["loss"][2])
    assert r["loss"][3] == 0.0
    assert np.all(r["grad"][1:] == 0)
    assert math.isnan(r["reduced_loss"])


# ----------------------------------------------------------- argmax / accuracy

def test_argmax_brute_force_with_ties():
    g = rng(12)
    V = 1000
    x = np.round(g.normal(0, 2, size=(200, V)) * 4) / 4  # many exact ties
    for i in range(0, 200, 3):
        j = int(np.argmax(x[i]))
        k = g.integers(0, V)
        x[i, k] = x[i, j]
    lab = g.integers(0, V, 200)
    lab[5] = IGN
    r = oc.ce_fwd_bwd(x, "f64", V, lab)
    first = np.array([min(np.flatnonzero(row == row.max())) for row in x])
    assert np.array_equal(r["argmax"], first)
    valid = lab != IGN
    assert r["n_correct"] == int(np.sum((first == lab) & valid))
    assert r["accuracy"] == r["n_correct"] / int(valid.sum())


# ---------------------------------------------------- library special case

@pytest.mark.parametrize("reduction", ["mean", "sum"])
@pytest.mark.parametrize("eps", [0.0, 0.1])
@pytest.mark.parametrize("T", [0.0, 30.0])
def test_matches_torch_cross_entropy(reduction, eps, T):
    g = rng(13)
    n, V = 64, 1024
    x = g.normal(0, 4, size=(n, V))
    lab = g.integers(0, V, n)
    lab[g.permutation(n)[:5]] = IGN
    gs = 0.3
    r = oc.ce_fwd_bwd(x, "f64", V, lab, label_smoothing=eps, softcap=T, reduction=reduction,
                      grad_scale=gs)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    z = T * torch.tanh(xt / T) if T > 0 else xt
    yt = torch.tensor(lab)
    per = torch.nn.functional.cross_entropy(z, yt, ignore_index=IGN, label_smoothing=eps,
                                            reduction="none")
    red = torch.nn.functional.cross_entropy(z, yt, ignore_index=IGN, label_smoothing=eps,
                                            reduction=reduction)
    (red * gs).backward()
    np.testing.assert_allclose(r["loss"], per.detach().numpy(), rtol=1e-12, atol=1e-12)
    assert abs(r["reduced_loss"] - red.item()) < 1e-10 * max(1.0, abs(red.item()))
    np.testing.assert_allclose(r["grad"], xt.grad.numpy(), rtol=1e-9, atol=1e-16)


def test_stored_dtypes_widen_exactly():
    g = rng(14)
    x32 = g.normal(0, 3, size=(8, 77)).astype(np.float32)
    xb = torch.tensor(x32).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    lab = g.integers(0, 77, 8)
    a = oc.ce_fwd_bwd(x32, "f32", 77, lab, label_smoothing=0.1)
    b = oc.ce_fwd_bwd(x32.astype(np.float64), "f64", 77, lab, label_smoothing=0.1)
    c = oc.ce_fwd_bwd(bits, "bf16", 77, lab, label_smoothing=0.1)
    d = oc.ce_fwd_bwd(xb.to(torch.float64).numpy(), "f64", 77, lab, label_smoothing=0.1)
    assert np.array_equal(a["loss"], b["loss"]) and np.array_equal(a["grad"], b["grad"])
    assert np.array_equal(c["loss"], d["loss"]) and np.array_equal(c["grad"], d["grad"])


def test_row_stride_reads_only_first_V_columns():
    g = rng(15)
    x = g.normal(size=(6, 40))
    padded = np.full((6, 47), np.nan)
    padded[:, :40] = x
    lab = g.integers(0, 40, 6)
    a = oc.ce_fwd_bwd(x, "f64", 40, lab)
    b = oc.ce_fwd_bwd(padded, "f64", 40, lab)
    assert np.array_equal(a["loss"], b["loss"]) and np.array_equal(a["grad"], b["grad"])


def test_result_does_not_depend_on_thread_count():
    g = rng(16)
    x = g.normal(0, 3, size=(37, 500))
    lab = g.integers(0, 500, 37)
    a = oc.ce_fwd_bwd(x, "f64", 500, lab, label_smoothing=0.1, softcap=9.0, threads=1)
    b = oc.ce_fwd_bwd(x, "f64", 500, lab, label_smoothing=0.1, softcap=9.0, threads=7)
    assert np.array_equal(a["loss"], b["loss"]) and np.array_equal(a["grad"], b["grad"])


# --------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_on_fp32_values():
    g = rng(17)
    v = np.concatenate([g.normal(0, 1, 20000), g.normal(0, 1e-30, 2000),
                        g.normal(0, 1e30, 2000)]).astype(np.float32)
    ref = torch.tensor(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oc.round_bf16(v.astype(np.float64)), ref)


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_round_bf16_is_nearest_even_in_fp64():
    g = rng(18)
    v = g.normal(0, 1, 20000) * np.exp2(g.integers(-140, 120, 20000))
    out = oc.round_bf16(v)
    got = _bf16_to_f64(out)
    # brute force: the two bf16 neighbours bracketing v, by stepping the bit pattern
    b32 = v.astype(np.float32).view(np.uint32) >> 16
    cands = []
    for d in (-1, 0, 1, 2):
        bits = (b32.astype(np.int64) + d).astype(np.uint16)
        cands.append(_bf16_to_f64(bits))
    cands = np.stack(cands)
    dist = np.abs(cands - v)
    best = np.nanmin(dist, axis=0)
    assert np.all(np.abs(got - v) == best)
    # exact ties go to the even pattern: 1 + 2^-8 lies between 1 and 1 + 2^-7
    assert oc.round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert oc.round_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82
    # a value a hair above the tie must not be double-rounded down
    assert oc.round_bf16(np.array([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81


# ---- reduction "none" with per-token upstream gradients (library special case:
# torch's cross_entropy(reduction="none") and autograd with a gradient vector)
@pytest.mark.parametrize("T,eps", [(0.0, 0.0), (0.0, 0.25), (7.0, 0.1)])
def test_none_reduction_with_per_token_upstream_gradient_matches_torch(T, eps):
    g = np.random.default_rng(41)
    n, V = 9, 23
    x = g.normal(0, 2, (n, V))
    lab = g.integers(0, V, n)
    lab[[2, 6]] = -100
    up = g.normal(0, 1, n)
    r = oc.ce_fwd_bwd(x, "f64", V, lab, label_smoothing=eps, softcap=T, reduction="none",
                      grad_scale=0.5, grad_per_token=up)
    xt = torch.tensor(x, requires_grad=True)
    z = T * torch.tanh(xt / T) if T > 0 else xt
    lt = torch.nn.functional.cross_entropy(z, torch.tensor(lab), ignore_index=-100,
                                           label_smoothing=eps, reduction="none")
    lt.backward(gradient=0.5 * torch.tensor(up))
    np.testing.assert_allclose(r["loss"], lt.detach().numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["grad"], xt.grad.numpy(), rtol=1e-10, atol=1e-15)
    valid = lab != -100
    assert abs(r["reduced_loss"] - r["loss"][valid].sum()) < 1e-12


def test_uniform_per_token_gradient_equals_sum_reduction():
    g = np.random.default_rng(42)
    x = g.normal(0, 2, (7, 31))
    lab = g.integers(0, 31, 7)
    a = oc.ce_fwd_bwd(x, "f64", 31, lab, reduction="sum", grad_scale=0.3)
    b = oc.ce_fwd_bwd(x, "f64", 31, lab, reduction="none", grad_scale=1.0,
                      grad_per_token=np.full(7, 0.3))
    np.testing.assert_allclose(b["grad"], a["grad"], rtol=1e-15, atol=0)
    assert a["reduced_loss"] == b["reduced_loss"]
