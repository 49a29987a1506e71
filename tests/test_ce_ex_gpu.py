"""GPU parity of ce_fwd_bwd_ex (through the C ABI): reduction "none" and
per-token upstream gradients on both kernels against the fp64 oracle, and the
forward-only mode (logits untouched; losses, argmax and reduced values equal
to those of the call that also writes the gradient)."""
import numpy as np
import pytest
import torch

from oracle import ce as oc
from tests.parity import bf16_bits_np, bits_to_f64, check_grad, check_loss, check_reduced
from vocabulary_lm_cross_gb300 import ce_fwd_bwd
from vocabulary_lm_cross_gb300.workloads import CEWorkload, make_ce_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def wl(N, V, dtype, T, eps, red, seed, stride=0):
    return CEWorkload(f"ex-{N}x{V}", N=N, V=V, dtype=dtype, sigma=3.0, ignore_frac=0.05,
                      label_smoothing=eps, softcap=T, reduction=red, grad_scale=0.5, seed=seed,
                      row_stride=stride, dup_max_frac=0.02, label_boost=2.0)


def host(x, dtype):
    return bf16_bits_np(x) if dtype == "bf16" else x.cpu().numpy()


@pytest.mark.parametrize("path", ["rows", "split"])
@pytest.mark.parametrize("N,V,dtype,T,eps,red", [
    (64, 40000, "bf16", 0.0, 0.1, "none"),
    (48, 33333, "f32", 30.0, 0.0, "none"),
    (80, 50001, "bf16", 5.0, 0.2, "mean"),
])
def test_per_token_upstream_gradients(monkeypatch, path, N, V, dtype, T, eps, red):
    monkeypatch.setenv("VLMCE_CE_PATH", path)
    w = wl(N, V, dtype, T, eps, red, seed=N + V)
    x, lab = make_ce_inputs(w, device=DEV)
    g = torch.Generator(device="cpu")
    g.manual_seed(N)
    up = torch.randn(N, generator=g, dtype=torch.float32)
    up[3] = 0.0
    up[5] = -2.0
    xh, labh = host(x, dtype), lab.cpu().numpy()
    r = ce_fwd_bwd(x[:, :V], lab, label_smoothing=eps, softcap=T, reduction=red, grad_scale=0.5,
                   grad_per_token=up.to(DEV))
    torch.cuda.synchronize()
    ref = oc.ce_fwd_bwd(xh, dtype, V, labh, label_smoothing=eps, softcap=T, reduction=red,
                        grad_scale=0.5, grad_per_token=up.double().numpy())
    check_loss(r.loss.cpu().numpy(), ref["loss"])
    assert np.array_equal(r.argmax.cpu().numpy(), ref["argmax"])
    check_reduced(float(r.reduced[0]), ref["reduced_loss"], "sum" if red == "none" else red)
    scale = ref["row_scale"] * up.double().numpy()[:, None]
    x64 = bits_to_f64(xh[:, :V]) if dtype == "bf16" else xh[:, :V].astype(np.float64)
    check_grad(host(x, dtype)[:, :V], ref["grad"], labh, V, eps, scale, dtype, softcap=T,
               x64=x64)


@pytest.mark.parametrize("path", ["rows", "split"])
@pytest.mark.parametrize("dtype,T,eps,red,V,stride", [
    ("bf16", 0.0, 0.1, "mean", 20011, 20016), ("f32", 30.0, 0.0, "sum", 20011, 20016),
    ("bf16", 5.0, 0.2, "none", 20011, 20016),
    ("bf16", 30.0, 0.1, "sum", 70001, 70008),  # wide softcap rows (row kernel)
])
def test_forward_only_leaves_the_logits_and_matches_the_full_call(monkeypatch, path, dtype, T, eps,
                                                                  red, V, stride):
    monkeypatch.setenv("VLMCE_CE_PATH", path)
    w = wl(100, V, dtype, T, eps, red, seed=7, stride=stride)
    x0, lab = make_ce_inputs(w, device=DEV)
    iv = torch.int16 if dtype == "bf16" else torch.int32
    xf = x0.clone()
    rf = ce_fwd_bwd(xf[:, :w.V], lab, label_smoothing=eps, softcap=T, reduction=red,
                    compute_grad=False)
    xg = x0.clone()
    rg = ce_fwd_bwd(xg[:, :w.V], lab, label_smoothing=eps, softcap=T, reduction=red)
    torch.cuda.synchronize()
    assert torch.equal(xf.view(iv), x0.view(iv))            # untouched, padding included
    assert not torch.equal(xg[:, :w.V].view(iv), x0[:, :w.V].view(iv))
    assert torch.equal(rf.loss.view(torch.int32), rg.loss.view(torch.int32))
    assert torch.equal(rf.argmax, rg.argmax)
    assert torch.equal(rf.reduced.view(torch.int32), rg.reduced.view(torch.int32))
    assert torch.equal(rf.counts, rg.counts)
