"""The seeded workload generator draws what its recipe says (CPU, small sizes)."""
import torch

from vocabulary_lm_cross_gb300.workloads import (CE_WORKLOADS, FLCE_WORKLOADS, HEADLINE_CE,
                                                 IGNORE_INDEX, make_ce_inputs, make_flce_inputs)


def test_headline_workload_recipe_at_small_size():
    w = CE_WORKLOADS[HEADLINE_CE].resized(N=400, V=3000)
    x, lab = make_ce_inputs(w)
    assert x.shape == (400, 3000) and x.dtype == torch.bfloat16 and lab.dtype == torch.int64
    assert int((lab == IGNORE_INDEX).sum()) == round(0.03 * 400)
    valid = lab != IGNORE_INDEX
    assert bool(((lab[valid] >= 0) & (lab[valid] < 3000)).all())
    xf = x.float()
    n_ties = int(((xf == xf.max(dim=1, keepdim=True).values).sum(dim=1) >= 2).sum())
    assert n_ties >= 4  # round(0.01 * 400) rows carry an exact duplicate maximum
    # the label boost makes the label logit larger on average than the row mean
    y = lab.clamp(min=0)
    assert float((xf[torch.arange(400), y] - xf.mean(dim=1))[valid].mean()) > 1.0


def test_generator_is_deterministic_and_pads_with_nan():
    w = CE_WORKLOADS["ce-bf16-8192x151936-stride152064-softcap30-sum"].resized(
        N=64, V=1000, row_stride=1016)
    a, la = make_ce_inputs(w)
    b, lb = make_ce_inputs(w)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)) and torch.equal(la, lb)
    assert a.shape == (64, 1016)
    assert bool(torch.isnan(a[:, 1000:].float()).all())
    assert bool(torch.isfinite(a[:, :1000].float()).all())


def test_flce_inputs_shapes():
    w = FLCE_WORKLOADS["flce-bf16-4096x6656x202048-softcap30"].resized(N=50, H=64, V=300)
    h, W, lab = make_flce_inputs(w)
    assert h.shape == (50, 64) and W.shape == (300, 64) and lab.shape == (50,)
    assert h.dtype == torch.bfloat16 and W.dtype == torch.bfloat16
    assert int((lab == IGNORE_INDEX).sum()) == 1
