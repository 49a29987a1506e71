"""ce_fwd_bwd_noalloc, the entry point for callers that cannot allocate device
memory (its scratch is a fixed array in the library's device image), gives the
same results as ce_fwd_bwd with a caller workspace, call after call.

Collected last on purpose: a failure here leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import vocabulary_lm_cross_gb300 as v
from tests.parity import bf16_bits_np, check_grad, check_loss
from vocabulary_lm_cross_gb300 import capi
from vocabulary_lm_cross_gb300.workloads import (CE_WORKLOADS, HEADLINE_CE, CEWorkload,
                                                 make_ce_inputs)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from vocabulary_lm_cross_gb300 import build
    build.build()


def _noalloc(x: torch.Tensor, lab: torch.Tensor, w: CEWorkload, row_outputs: bool = True):
    """One ce_fwd_bwd_noalloc call; without row outputs the per-row losses and
    argmaxes live only in the library's fixed scratch."""
    N, V = w.N, w.V
    out = dict(loss=torch.empty(N, dtype=torch.float32, device=DEV),
               argmax=torch.empty(N, dtype=torch.int64, device=DEV),
               reduced=torch.empty(2, dtype=torch.float32, device=DEV),
               counts=torch.empty(4, dtype=torch.int64, device=DEV))
    st = capi.lib().ce_fwd_bwd_noalloc(
        x.data_ptr(), capi.BF16 if w.dtype == "bf16" else capi.F32, lab.data_ptr(), N, V,
        x.stride(0), -100, w.label_smoothing, w.softcap,
        capi.MEAN if w.reduction == "mean" else capi.SUM, w.grad_scale,
        out["loss"].data_ptr() if row_outputs else None,
        out["argmax"].data_ptr() if row_outputs else None, out["reduced"].data_ptr(),
        out["counts"].data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    capi.check(st, "ce_fwd_bwd_noalloc")
    return out


def _rows(x: torch.Tensor, dtype: str) -> np.ndarray:
    return bf16_bits_np(x) if dtype == "bf16" else x.cpu().numpy()


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    cases = [
        CE_WORKLOADS[HEADLINE_CE].resized(N=300),
        CEWorkload("f32-strided-softcap", N=97, V=20011, dtype="f32", sigma=6.0, ignore_frac=0.1,
                   label_smoothing=0.1, softcap=30.0, reduction="sum", grad_scale=0.25, seed=77,
                   row_stride=20016),
    ]
    for w in cases:
        x, lab = make_ce_inputs(w, device=DEV)
        xa, xb = x.clone(), x.clone()
        ref = v.ce_fwd_bwd(xa[:, :w.V], lab, label_smoothing=w.label_smoothing, softcap=w.softcap,
                           reduction=w.reduction, grad_scale=w.grad_scale)
        got = _noalloc(xb, lab, w)
        torch.cuda.synchronize()
        # within the parity tolerances (the kernels are the same, so in fact identical)
        check_loss(got["loss"].cpu().numpy(), ref.loss.cpu().numpy().astype(np.float64))
        assert np.array_equal(got["argmax"].cpu().numpy(), ref.argmax.cpu().numpy())
        assert got["counts"].cpu().tolist() == ref.counts.cpu().tolist()
        assert np.array_equal(got["reduced"].cpu().numpy(), ref.reduced.cpu().numpy())
        ga, gb = _rows(xa, w.dtype)[:, :w.V], _rows(xb, w.dtype)[:, :w.V]
        ref_grad = ga.astype(np.float64) if w.dtype == "f32" else \
            (ga.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        scale = w.grad_scale / int(ref.counts[0]) if w.reduction == "mean" else w.grad_scale
        check_grad(gb, ref_grad, lab.cpu().numpy(), w.V, w.label_smoothing, scale, w.dtype,
                   softcap=w.softcap)
        assert np.array_equal(ga.view(np.uint8), gb.view(np.uint8))


def test_noalloc_at_its_row_limit_without_row_outputs_twice_in_a_row():
    # N = 65536 rows with no per-row outputs: the losses and argmaxes the
    # finalize step reduces live in the fixed scratch, all of it in use.  Two
    # calls back to back on one stream with different inputs: the second
    # call's results must not depend on what the first left in the scratch.
    base = CEWorkload("noalloc-limit", N=65536, V=64, dtype="bf16", sigma=2.0, ignore_frac=0.05,
                      label_smoothing=0.1, softcap=0.0, reduction="mean", grad_scale=1.0,
                      seed=91, label_boost=2.0)
    ws = [base, base.resized(seed=92)]
    ins = [make_ce_inputs(w, device=DEV) for w in ws]
    refs = []
    for w, (x, lab) in zip(ws, ins):
        xa = x.clone()
        refs.append((v.ce_fwd_bwd(xa, lab, label_smoothing=w.label_smoothing,
                                  reduction=w.reduction, grad_scale=w.grad_scale), xa))
    xbs = [x.clone() for x, _ in ins]
    gots = [_noalloc(xb, lab, w, row_outputs=False) for xb, (_, lab), w in zip(xbs, ins, ws)]
    torch.cuda.synchronize()
    for (ref, xa), got, xb in zip(refs, gots, xbs):
        assert got["counts"].cpu().tolist() == ref.counts.cpu().tolist()
        assert np.array_equal(got["reduced"].cpu().numpy(), ref.reduced.cpu().numpy())
        assert np.array_equal(bf16_bits_np(xa), bf16_bits_np(xb))
    # the two inputs differ, and so do their results
    assert not np.array_equal(gots[0]["reduced"].cpu().numpy(), gots[1]["reduced"].cpu().numpy())


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    n_max = int(capi.lib().vlmce_ce_noalloc_max_rows())
    assert n_max == 65536
    st = capi.lib().ce_fwd_bwd_noalloc(1 << 20, capi.BF16, 1 << 20, n_max + 1, 100, 100, -100,
                                       0.0, 0.0, capi.MEAN, 1.0, None, None, None, None, None)
    assert st == capi.ERR_TOO_LARGE
