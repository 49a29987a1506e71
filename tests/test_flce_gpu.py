"""GPU parity of the tcgen05 GEMM engine and of flce_fwd_bwd (through the C
ABI) against matmuls of the same bf16 values and the fp64 FLCE oracle.

Tolerances: GEMM fp32 results within 1e-5 of the largest reference magnitude
(fp32 accumulation of exact bf16 products); FLCE per-token loss 1e-4
absolute; argmax exact except on rows whose two largest fp64 logits are
closer than 1e-3 max(1, |top|) (fp32 accumulation may order such near-ties
differently; such rows are counted and reported); gradients within 1e-2
relative L2 (the gradient tile is rounded to bf16 before the two gradient
products, as the pages' fused path does); reduced loss 1e-4 (mean) /
1e-6 relative (sum).
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import flce as of
from tests.parity import bf16_bits_np, check_loss, check_reduced
from vocabulary_lm_cross_gb300 import capi
from vocabulary_lm_cross_gb300.flce import flce_fwd_bwd
from vocabulary_lm_cross_gb300.workloads import (FLCE_WORKLOADS, IGNORE_INDEX, FLCEWorkload,
                                                 make_flce_inputs)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from vocabulary_lm_cross_gb300 import build
    build.build()


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def gemm(A, a_mn, B, b_mn, C, M, N, K, accumulate=False):
    st = capi.lib().vlmce_gemm_bf16(A.data_ptr(), int(a_mn), B.data_ptr(), int(b_mn), C.data_ptr(),
                                    M, N, K, A.stride(0), B.stride(0), C.stride(0), int(accumulate),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    capi.check(st, "vlmce_gemm_bf16")


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (296, 520, 200), (1000, 264, 1032),
                                   (520, 136, 72)])
def test_gemm_engine_against_matmul(a_mn, b_mn, M, N, K):
    g = torch.Generator(device=DEV)
    g.manual_seed(M * 7 + N * 3 + K + 10 * a_mn + b_mn)
    Al = torch.randn(M, K, generator=g, device=DEV).to(torch.bfloat16)  # logical A [M, K]
    Bl = torch.randn(N, K, generator=g, device=DEV).to(torch.bfloat16)  # logical B [N, K]
    A = Al.t().contiguous() if a_mn else Al
    B = Bl.t().contiguous() if b_mn else Bl
    ref = Al.double() @ Bl.double().t()
    C = torch.full((M, N), 3.0, dtype=torch.float32, device=DEV)
    gemm(A, a_mn, B, b_mn, C, M, N, K)
    torch.cuda.synchronize()
    err = (C.double() - ref).abs().max().item()
    assert err <= 1e-5 * ref.abs().max().item(), err
    gemm(A, a_mn, B, b_mn, C, M, N, K, accumulate=True)
    torch.cuda.synchronize()
    err = (C.double() - 2 * ref).abs().max().item()
    assert err <= 2e-5 * ref.abs().max().item(), err


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 1)])
def test_gemm_engine_fp16_against_matmul(a_mn, b_mn):
    M, N, K = 520, 264, 1032
    g = torch.Generator(device=DEV)
    g.manual_seed(17 + a_mn)
    Al = torch.randn(M, K, generator=g, device=DEV).to(torch.float16)
    Bl = torch.randn(N, K, generator=g, device=DEV).to(torch.float16)
    A = Al.t().contiguous() if a_mn else Al
    B = Bl.t().contiguous() if b_mn else Bl
    ref = Al.double() @ Bl.double().t()
    C = torch.empty((M, N), dtype=torch.float32, device=DEV)
    st = capi.lib().vlmce_gemm(A.data_ptr(), a_mn, B.data_ptr(), b_mn, C.data_ptr(), M, N, K,
                               A.stride(0), B.stride(0), C.stride(0), 0, capi.F16,
                               torch.cuda.current_stream().cuda_stream)
    capi.check(st, "vlmce_gemm")
    torch.cuda.synchronize()
    assert (C.double() - ref).abs().max().item() <= 1e-5 * ref.abs().max().item()


def near_tie_rows(h64, W64, labels=None):
    S = h64 @ W64.T
    top2 = np.sort(S, axis=1)[:, -2:]
    return np.abs(top2[:, 1] - top2[:, 0]) < 1e-3 * np.maximum(1.0, np.abs(top2[:, 1]))


def widen(t):
    return t.double().cpu().numpy() if t.dtype == torch.float16 else of.widen_bf16(bf16_bits_np(t))


def run_small(w: FLCEWorkload, accumulate=False, chunk_rows=None):
    h, W, lab = make_flce_inputs(w, device=DEV)
    gw0 = None
    if accumulate:
        gw0 = torch.randn(w.V, w.H, device=DEV, dtype=torch.float32)
    res = flce_fwd_bwd(h, W, lab, label_smoothing=w.label_smoothing, softcap=w.softcap,
                       reduction=w.reduction, grad_scale=w.grad_scale,
                       grad_weight=gw0.clone() if accumulate else None,
                       accumulate_grad_weight=accumulate, chunk_rows=chunk_rows)
    torch.cuda.synchronize()
    h64 = widen(h)
    W64 = widen(W)
    labh = lab.cpu().numpy()
    ref = of.flce_fwd_bwd(h64, W64, labh, label_smoothing=w.label_smoothing, softcap=w.softcap,
                          reduction=w.reduction, grad_scale=w.grad_scale)
    check_loss(res.loss.cpu().numpy(), ref["loss"])
    ties = near_tie_rows(h64, W64)
    amax = res.argmax.cpu().numpy()
    mism = (amax != ref["argmax"])
    assert not np.any(mism & ~ties), np.flatnonzero(mism & ~ties)
    counts = res.counts.cpu().numpy()
    assert counts[0] == ref["n_valid"] and counts[2] == ref["n_bad"] and counts[3] == 0
    # counts and accuracy exactly, the GPU's choice deciding on exempt near-tie rows
    valid = (labh != IGNORE_INDEX) & (labh >= 0) & (labh < w.V)
    n_correct = int(np.sum(valid & (np.where(mism, amax, ref["argmax"]) == labh)))
    assert counts[1] == n_correct
    assert float(res.reduced[1]) == np.float32(n_correct / max(ref["n_valid"], 1))
    check_reduced(float(res.reduced[0]), ref["reduced_loss"], w.reduction)
    gh = res.grad_hidden.float().cpu().numpy()
    assert rel_l2(gh, ref["grad_hidden"]) < 1e-2
    gw = res.grad_weight.cpu().numpy().astype(np.float64)
    if accumulate:
        gw = gw - gw0.cpu().numpy()
    assert rel_l2(gw, ref["grad_weight"]) < 1e-2
    return res, ref


def small(N, H, V, T=0.0, eps=0.0, red="mean", gs=1.0, seed=11, wsig=0.05, dtype="bf16"):
    return FLCEWorkload(f"f{N}x{H}x{V}", N=N, H=H, V=V, hidden_sigma=1.0, weight_sigma=wsig,
                        multiplier=0.5, ignore_frac=0.05, label_smoothing=eps, softcap=T,
                        reduction=red, grad_scale=gs, seed=seed, dtype=dtype)


@pytest.mark.parametrize("N,H,V,T,eps,red", [(256, 512, 8192, 30.0, 0.1, "mean"),
                                             (600, 264, 17000, 0.0, 0.0, "sum"),
                                             (130, 128, 300, 5.0, 0.2, "mean")])
def test_flce_fp16(N, H, V, T, eps, red):
    run_small(small(N, H, V, T=T, eps=eps, red=red, gs=0.5, seed=N + 1, dtype="f16"))


@pytest.mark.parametrize("N,H,V", [(256, 512, 8192), (200, 264, 5000), (130, 128, 300),
                                   (1, 64, 1000), (3, 200, 513)])
@pytest.mark.parametrize("T,eps,red", [(0.0, 0.0, "mean"), (30.0, 0.1, "sum")])
def test_flce_small_single_chunk(N, H, V, T, eps, red):
    run_small(small(N, H, V, T=T, eps=eps, red=red, gs=0.5))


def test_flce_several_chunks_and_accumulated_weight_gradient():
    run_small(small(200, 264, 20000, T=30.0, eps=0.1), accumulate=False)
    run_small(small(150, 136, 17000, T=0.0, eps=0.0, red="sum"), accumulate=True)


@pytest.mark.parametrize("N,H,V,T,eps", [(600, 264, 17000, 30.0, 0.1), (520, 128, 9000, 0.0, 0.0),
                                         (1030, 200, 700, 5.0, 0.2)])
def test_flce_two_pairs_per_cluster(N, H, V, T, eps):
    # more than one 256-row pair tile: clusters of two CTA pairs share each
    # weight tile; ragged rows in the second pair, several vocabulary chunks
    run_small(small(N, H, V, T=T, eps=eps, red="sum", gs=0.25, seed=N), accumulate=(N == 520))


# The row-chunked schedule (flce_fwd_bwd_rows): one block, ragged blocks with
# an accumulated weight gradient, vocabularies that are not multiples of 8
# (padded logits / gradient rows), many small blocks (few rows per CE call),
# fp16.
@pytest.mark.parametrize("N,H,V,T,eps,red,chunk,dtype,acc", [
    (256, 512, 8192, 30.0, 0.1, "mean", 256, "bf16", False),
    (600, 264, 17000, 0.0, 0.0, "sum", 256, "bf16", True),
    (200, 264, 5001, 5.0, 0.2, "mean", 64, "bf16", False),
    (130, 128, 303, 30.0, 0.1, "sum", 7, "f16", False),
    (1030, 200, 700, 0.0, 0.0, "mean", 1000, "f16", True),
])
def test_flce_row_chunked(N, H, V, T, eps, red, chunk, dtype, acc):
    run_small(small(N, H, V, T=T, eps=eps, red=red, gs=0.5, seed=N + V, dtype=dtype),
              accumulate=acc, chunk_rows=chunk)


def test_flce_row_chunked_one_row_blocks():
    run_small(small(5, 64, 1000, T=30.0, eps=0.1, red="sum", seed=9), chunk_rows=1)


@pytest.mark.parametrize("chunk_rows", [None, 16])
@pytest.mark.parametrize("accumulate", [False, True])
def test_flce_no_rows(chunk_rows, accumulate):
    # no rows: zero losses and counts; d loss / dW = 0, so an overwritten
    # grad_weight is cleared and an accumulated one kept
    h = torch.zeros(0, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.randn(100, 64, device=DEV).to(torch.bfloat16)
    lab = torch.zeros(0, dtype=torch.int64, device=DEV)
    gw = torch.full((100, 64), 7.0, device=DEV)
    r = flce_fwd_bwd(h, W, lab, chunk_rows=chunk_rows, grad_weight=gw,
                     accumulate_grad_weight=accumulate)
    torch.cuda.synchronize()
    assert r.loss.numel() == 0 and int(r.counts[0]) == 0 and int(r.counts[3]) == 0
    assert float(r.reduced[0]) == 0.0
    assert torch.equal(gw, torch.full_like(gw, 7.0) if accumulate else torch.zeros_like(gw))


def test_flce_row_chunked_agrees_with_vocab_chunked():
    # both schedules form fp32 logits and a 16-bit gradient between the products:
    # losses agree to rounding, argmax exactly (the same fp32 products), the
    # gradients to the 16-bit rounding of the gradient tile
    w = small(520, 256, 12000, T=30.0, eps=0.1, red="mean", gs=0.5, seed=3)
    h, W, lab = make_flce_inputs(w, device=DEV)
    kw = dict(label_smoothing=w.label_smoothing, softcap=w.softcap, reduction=w.reduction,
              grad_scale=w.grad_scale)
    a = flce_fwd_bwd(h, W, lab, **kw)
    b = flce_fwd_bwd(h, W, lab, chunk_rows=200, **kw)
    torch.cuda.synchronize()
    assert torch.allclose(a.loss, b.loss, rtol=0, atol=2e-5)
    assert torch.equal(a.argmax, b.argmax)
    assert torch.equal(a.counts, b.counts)
    assert rel_l2(a.grad_hidden.float().cpu().numpy(), b.grad_hidden.float().cpu().numpy()) < 2e-3
    assert rel_l2(a.grad_weight.cpu().numpy(), b.grad_weight.cpu().numpy()) < 2e-3


def test_flce_agrees_with_torch_matmuls_around_the_ce_kernel():
    # an independent composition: fp32 torch matmul logits -> ce_fwd_bwd (the
    # row kernel on fp32 logits) -> torch matmuls for the two gradients
    from vocabulary_lm_cross_gb300 import ce_fwd_bwd
    w = small(300, 192, 7000, T=30.0, eps=0.1, red="mean", gs=0.5, seed=5)
    h, W, lab = make_flce_inputs(w, device=DEV)
    res = flce_fwd_bwd(h, W, lab, label_smoothing=w.label_smoothing, softcap=w.softcap,
                       reduction=w.reduction, grad_scale=w.grad_scale)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        hf, Wf = h.float(), W.float()
        S = hf @ Wf.T
        ce = ce_fwd_bwd(S, lab, label_smoothing=w.label_smoothing, softcap=w.softcap,
                        reduction=w.reduction, grad_scale=w.grad_scale)
        gh = S @ Wf     # S now holds d loss / d S
        gw = S.T @ hf
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    torch.cuda.synchronize()
    assert torch.allclose(res.loss, ce.loss, rtol=0, atol=2e-5)
    assert abs(float(res.reduced[0]) - float(ce.reduced[0])) < 1e-5
    assert int(res.counts[0]) == int(ce.counts[0]) and int(res.counts[2]) == int(ce.counts[2])
    assert rel_l2(res.grad_hidden.float().cpu().numpy(), gh.cpu().numpy()) < 1e-2
    assert rel_l2(res.grad_weight.cpu().numpy(), gw.cpu().numpy()) < 1e-2


def test_flce_deterministic():
    w = small(256, 512, 9000, T=30.0)
    outs = []
    for _ in range(2):
        h, W, lab = make_flce_inputs(w, device=DEV)
        r = flce_fwd_bwd(h, W, lab, softcap=30.0)
        torch.cuda.synchronize()
        outs.append((r.grad_hidden.view(torch.int16).cpu(), r.grad_weight.cpu(), r.loss.cpu()))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1].view(torch.int32), outs[1][1].view(torch.int32))
    assert torch.equal(outs[0][2].view(torch.int32), outs[1][2].view(torch.int32))


def _golden_flce():
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "flce_closed_forms.jsonl")
    with open(path) as f:
        return [json.loads(line) for line in f if line.strip()]


GOLDEN = _golden_flce()


# The closed-form fused linear CE calls of tests/golden (exact small inputs,
# so the logits are exact in fp32): losses within 1e-4, argmax and counts
# exact, both gradients within 1e-2 relative L2 (the gradient tile is rounded
# to bf16 before the two products).
@pytest.mark.parametrize("chunk_rows", [None, 2])
@pytest.mark.parametrize("c", GOLDEN, ids=[c["case"] for c in GOLDEN])
def test_flce_closed_form_golden_calls(c, chunk_rows):
    h = torch.tensor(c["h"], dtype=torch.float64).to(torch.bfloat16).to(DEV)
    W = torch.tensor(c["W"], dtype=torch.float64).to(torch.bfloat16).to(DEV)
    lab = torch.tensor(c["labels"], dtype=torch.int64, device=DEV)
    r = flce_fwd_bwd(h, W, lab, label_smoothing=c["label_smoothing"], softcap=c["softcap"],
                     reduction=c["reduction"], grad_scale=c["grad_scale"], chunk_rows=chunk_rows)
    torch.cuda.synchronize()
    np.testing.assert_allclose(r.loss.cpu().numpy(), c["loss"], rtol=0, atol=1e-4)
    assert r.argmax.cpu().tolist() == c["argmax"]
    counts = r.counts.cpu().tolist()
    assert counts[0] == c["n_valid"] and counts[1] == c["n_correct"] and counts[2:] == [0, 0]
    assert abs(float(r.reduced[0]) - c["reduced_loss"]) <= 1e-4 * max(1.0, abs(c["reduced_loss"]))
    assert rel_l2(r.grad_hidden.float().cpu().numpy(), np.asarray(c["grad_hidden"])) < 1e-2
    assert rel_l2(r.grad_weight.cpu().numpy(), np.asarray(c["grad_weight"])) < 1e-2


# The GEMM launches of a call take their tiles from counters in that call's
# workspace: two calls in flight on two streams at once give the same bits as
# one after the other.
def test_flce_concurrent_calls_on_two_streams():
    ws = [small(256, 512, 9000, T=30.0, seed=21), small(192, 512, 7000, eps=0.1, seed=22)]
    inputs = [make_flce_inputs(w, device=DEV) for w in ws]

    def call(w, h, W, lab):
        return flce_fwd_bwd(h, W, lab, label_smoothing=w.label_smoothing, softcap=w.softcap)

    ref = []
    for w, (h, W, lab) in zip(ws, inputs):
        ref.append(call(w, h, W, lab))
        torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for st, w, (h, W, lab) in zip(streams, ws, inputs):
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            outs.append(call(w, h, W, lab))
    torch.cuda.synchronize()
    for a, b in zip(ref, outs):
        assert torch.equal(a.grad_hidden.view(torch.int16), b.grad_hidden.view(torch.int16))
        assert torch.equal(a.grad_weight.view(torch.int32), b.grad_weight.view(torch.int32))
        assert torch.equal(a.loss.view(torch.int32), b.loss.view(torch.int32))
        assert torch.equal(a.argmax, b.argmax)
        assert torch.equal(a.counts, b.counts)


@pytest.mark.parametrize("chunk_rows", [None, 1024])
def test_flce_full_size_workload_sampled(chunk_rows):
    w = FLCE_WORKLOADS["flce-bf16-4096x6656x202048-softcap30"]
    h, W, lab = make_flce_inputs(w, device=DEV)
    hb = bf16_bits_np(h)
    Wb = bf16_bits_np(W)
    labh = lab.cpu().numpy()
    res = flce_fwd_bwd(h, W, lab, label_smoothing=w.label_smoothing, softcap=w.softcap,
                       reduction=w.reduction, grad_scale=w.grad_scale, chunk_rows=chunk_rows)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, w.N - 1], np.flatnonzero(labh == IGNORE_INDEX)[:2],
                                     rng.choice(w.N, 28, replace=False)]))
    cols = np.unique(np.concatenate([[0, w.V - 1, 8191, 8192], labh[labh >= 0][:6],
                                     rng.choice(w.V, 22, replace=False)]))
    ref = of.sampled(hb, Wb, labh, rows, cols, label_smoothing=w.label_smoothing,
                     softcap=w.softcap, reduction=w.reduction, grad_scale=w.grad_scale)
    check_loss(res.loss.cpu().numpy(), ref["loss"])
    # argmax: exact except on oracle near-ties (top two fp64 logits closer than
    # 1e-3 max(1, |top|)); there the GPU's column must itself be a near-maximum
    amax = res.argmax.cpu().numpy()
    top, second = ref["top"], ref["second"]
    tie_tol = 1e-3 * np.maximum(1.0, np.abs(top))
    near = (top - second) < tie_tol
    mism = np.flatnonzero(amax != ref["argmax"])
    assert not np.any(~near[mism]), mism[~near[mism]]
    h64 = of.widen_bf16(hb)
    for r in mism:
        s_gpu = float(h64[r] @ of.widen_bf16(Wb[amax[r]]))
        assert top[r] - s_gpu < tie_tol[r], (r, amax[r], s_gpu, top[r])
    # counts and accuracy, exactly: on the exempt rows the GPU's (validated)
    # choice decides correctness
    valid = (labh != IGNORE_INDEX) & (labh >= 0) & (labh < w.V)
    decided = np.where(amax != ref["argmax"], amax, ref["argmax"])
    n_correct = int(np.sum(valid & (decided == labh)))
    counts = res.counts.cpu().numpy()
    assert counts[0] == ref["n_valid"] and counts[2] == ref["n_bad"] and counts[3] == 0, counts
    assert counts[1] == n_correct, (counts[1], n_correct)
    if mism.size == 0:
        assert n_correct == ref["n_correct"]
    assert float(res.reduced[1]) == np.float32(n_correct / max(ref["n_valid"], 1))
    check_reduced(float(res.reduced[0]), ref["reduced_loss"], w.reduction)
    gh = res.grad_hidden.float().cpu().numpy()[rows]
    gw = res.grad_weight.cpu().numpy()[cols]
    e_h = rel_l2(gh, ref["grad_hidden_rows"])
    e_w = rel_l2(gw, ref["grad_weight_cols"])
    print("full-size FLCE (chunk_rows", chunk_rows, "): oracle near-tie rows", int(near.sum()),
          "argmax mismatches", mism.size, "rel-L2 grad_hidden", e_h, "grad_weight", e_w)
    assert e_h < 1e-2 and e_w < 1e-2
