"""Pins for the vocabulary-sharded CE oracle (CPU): one shard and any cut of
the vocabulary reproduce the (separately pinned) unsharded CE oracle; the
merge does not depend on the order of the shards; uniform logits give ln V;
ties of the maximum across shards go to the smallest global column."""
import itertools

import numpy as np
import pytest

from oracle import ce as oc
from oracle import ce_shard as osh

IGN = -100


def data(seed, n=12, V=37, sigma=2.0):
    g = np.random.default_rng(seed)
    x = g.normal(0, sigma, (n, V))
    lab = g.integers(0, V, n)
    lab[1] = IGN
    return x, lab


@pytest.mark.parametrize("T,eps,red", [(0.0, 0.0, "mean"), (4.0, 0.2, "sum"), (30.0, 0.1, "mean")])
@pytest.mark.parametrize("bounds", [[], [1], [36], [5, 6, 20], list(range(1, 37))])
def test_any_cut_reproduces_the_unsharded_oracle(T, eps, red, bounds):
    x, lab = data(1)
    lab[2] = 0        # label in the first column
    lab[3] = 36       # label in the last column
    if bounds:
        lab[4] = bounds[0]        # label on a shard's first column
        lab[5] = bounds[-1] - 1   # label on a shard's last column
    full = oc.ce_fwd_bwd(x, "f64", x.shape[1], lab, label_smoothing=eps, softcap=T, reduction=red,
                         grad_scale=0.7)
    sh = osh.sharded_fwd_bwd(x, bounds, lab, label_smoothing=eps, softcap=T, reduction=red,
                             grad_scale=0.7)
    np.testing.assert_allclose(sh["loss"], full["loss"], rtol=1e-12, atol=1e-12)
    assert np.array_equal(sh["argmax"], full["argmax"])
    np.testing.assert_allclose(sh["grad"], full["grad"], rtol=1e-11, atol=1e-15)
    assert abs(sh["reduced_loss"] - full["reduced_loss"]) <= 1e-12 * max(1, abs(full["reduced_loss"]))
    assert sh["n_correct"] == full["n_correct"]


def test_merge_is_independent_of_shard_order():
    x, lab = data(2, V=40)
    cuts = [(0, 7), (7, 8), (8, 25), (25, 40)]
    parts = [osh.shard_stats(x[:, a:b], a, lab, 5.0) for a, b in cuts]
    ref = osh.merge_stats(parts)
    for perm in itertools.permutations(range(4)):
        m = osh.merge_stats([parts[i] for i in perm])
        assert np.array_equal(m["argmax"], ref["argmax"])
        np.testing.assert_allclose(m["lse"], ref["lse"], rtol=1e-14)
        np.testing.assert_allclose(m["sum_z"], ref["sum_z"], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(m["z_y"], ref["z_y"], rtol=0, atol=0)


def test_uniform_logits_give_log_v():
    V = 50
    x = np.full((3, V), 1.25)
    lab = np.array([0, 49, 17])
    sh = osh.sharded_fwd_bwd(x, [10, 11, 30], lab, label_smoothing=0.3)
    np.testing.assert_allclose(sh["loss"], np.log(V), rtol=1e-14)
    assert np.all(sh["argmax"] == 0)


def test_tied_maximum_across_shards_goes_to_the_smallest_column():
    x = np.zeros((2, 10))
    x[0, [3, 8]] = 5.0     # tie split over shards [0, 6) and [6, 10)
    x[1, [7, 9]] = 4.0     # tie inside the second shard
    lab = np.array([3, 9])
    p0 = osh.shard_stats(x[:, :6], 0, lab)
    p1 = osh.shard_stats(x[:, 6:], 6, lab)
    for order in ([p0, p1], [p1, p0]):
        m = osh.merge_stats(order)
        assert list(m["argmax"]) == [3, 7]
