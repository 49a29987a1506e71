"""The oracle against closed-form cross-entropy calls (tests/golden/
ce_closed_forms.jsonl and flce_closed_forms.jsonl, written by
tests/golden/make_ce_closed_forms.py from the method's definition with
Python's math module only): per-token losses, gradients, argmax with ties,
reduced loss, accuracy and counts; for the fused linear form also the hidden
and weight gradients."""
import importlib.util
import json
import os

import numpy as np
import pytest

from oracle import ce as oc
from oracle import flce as of

HERE = os.path.dirname(os.path.abspath(__file__))


def load_cases(name):
    with open(os.path.join(HERE, "golden", name)) as f:
        return [json.loads(line) for line in f if line.strip()]


CASES = load_cases("ce_closed_forms.jsonl")
FLCE_CASES = load_cases("flce_closed_forms.jsonl")


def test_fixture_is_what_its_generator_writes():
    spec = importlib.util.spec_from_file_location(
        "make_ce_closed_forms", os.path.join(HERE, "golden", "make_ce_closed_forms.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    assert [json.loads(json.dumps(c)) for c in gen.CASES] == CASES
    assert [json.loads(json.dumps(c)) for c in gen.FLCE_CASES] == FLCE_CASES


@pytest.mark.parametrize("c", CASES, ids=[c["case"] for c in CASES])
def test_oracle_matches_closed_forms(c):
    x = np.asarray(c["x"], dtype=np.float64)
    lab = np.asarray(c["labels"], dtype=np.int64)
    r = oc.ce_fwd_bwd(x, "f64", c["V"], lab, label_smoothing=c["label_smoothing"],
                      softcap=c["softcap"], reduction=c["reduction"], grad_scale=c["grad_scale"])
    np.testing.assert_allclose(r["loss"], c["loss"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(r["grad"], np.asarray(c["grad"]), rtol=1e-12, atol=1e-15)
    assert r["argmax"].tolist() == c["argmax"]
    assert r["n_valid"] == c["n_valid"] and r["n_correct"] == c["n_correct"]
    assert abs(r["reduced_loss"] - c["reduced_loss"]) <= 1e-13 * max(1.0, abs(c["reduced_loss"]))
    assert r["accuracy"] == pytest.approx(c["accuracy"], abs=0.0)


@pytest.mark.parametrize("c", FLCE_CASES, ids=[c["case"] for c in FLCE_CASES])
def test_flce_oracle_matches_closed_forms(c):
    h = np.asarray(c["h"], dtype=np.float64)
    W = np.asarray(c["W"], dtype=np.float64)
    lab = np.asarray(c["labels"], dtype=np.int64)
    r = of.flce_fwd_bwd(h, W, lab, label_smoothing=c["label_smoothing"], softcap=c["softcap"],
                        reduction=c["reduction"], grad_scale=c["grad_scale"])
    np.testing.assert_allclose(r["loss"], c["loss"], rtol=1e-13, atol=1e-15)
    assert r["argmax"].tolist() == c["argmax"]
    np.testing.assert_allclose(r["grad_hidden"], np.asarray(c["grad_hidden"]), rtol=1e-12,
                               atol=1e-15)
    np.testing.assert_allclose(r["grad_weight"], np.asarray(c["grad_weight"]), rtol=1e-12,
                               atol=1e-15)
    assert abs(r["reduced_loss"] - c["reduced_loss"]) <= 1e-13 * max(1.0, abs(c["reduced_loss"]))
