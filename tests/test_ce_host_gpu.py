"""GPU checks of ce_fwd_bwd_host (through the C ABI): logits in page-locked
host memory streamed through the device in chunks of rows (one chunk, several
ragged chunks, more chunks than staging slots, rows off the 16-byte grid),
labels and outputs in host memory.  The results must be bit-identical to
ce_fwd_bwd on a device copy of the same inputs run on the same (row) kernel,
padding columns untouched; pageable host memory is refused before anything is
launched."""
import ctypes

import numpy as np
import pytest
import torch

from vocabulary_lm_cross_gb300 import capi, ce_fwd_bwd, ce_fwd_bwd_host
from vocabulary_lm_cross_gb300.workloads import CEWorkload, make_ce_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def wl(N, V, stride, dtype, T, eps, red, seed):
    return CEWorkload(f"host-{N}x{V}", N=N, V=V, dtype=dtype, sigma=3.0, ignore_frac=0.05,
                      label_smoothing=eps, softcap=T, reduction=red, grad_scale=0.5, seed=seed,
                      row_stride=stride, dup_max_frac=0.02, label_boost=2.0)


def bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("N,V,stride,dtype,T,eps,red", [
    (300, 5003, 5011, "bf16", 0.0, 0.1, "mean"),
    (40, 20000, 20000, "bf16", 30.0, 0.0, "sum"),
    (200, 4096, 4100, "f32", 5.0, 0.2, "mean"),
    (1, 131072, 131072, "bf16", 0.0, 0.0, "mean"),
    (700, 65536, 65544, "bf16", 0.0, 0.1, "mean"),     # 3 chunks of 256 rows, last ragged
    (2100, 32768, 32768, "bf16", 30.0, 0.0, "sum"),    # 5 chunks through 3 slots
    (600, 20000, 20004, "f32", 0.0, 0.0, "mean"),      # 2 chunks, fp32
    (60, 70001, 70007, "bf16", 30.0, 0.1, "sum"),      # wide softcap rows on 256-thread CTAs
    (600, 40000, 40000, "f32", 30.0, 0.0, "mean"),     # the same, 3 chunks, fp32
    (2048, 131072, 131072, "bf16", 0.0, 0.1, "mean"),  # the headline shape, as bench.py's e2e
])
def test_host_results_equal_device_results(monkeypatch, N, V, stride, dtype, T, eps, red):
    monkeypatch.setenv("VLMCE_CE_PATH", "rows")  # the kernel the host path uses
    w = wl(N, V, stride, dtype, T, eps, red, seed=N + V)
    x, lab = make_ce_inputs(w, device="cpu")
    xh, labh = x.pin_memory(), lab.pin_memory()
    xd, labd = x.to(DEV), lab.to(DEV)
    kw = dict(label_smoothing=eps, softcap=T, reduction=red, grad_scale=0.5)
    rd = ce_fwd_bwd(xd[:, :V], labd, **kw)
    rh = ce_fwd_bwd_host(xh[:, :V], labh, device=DEV, **kw)
    torch.cuda.synchronize()
    assert torch.equal(bits(xh), bits(xd.cpu()))  # gradient, and the NaN padding untouched
    assert torch.equal(bits(rh.loss), bits(rd.loss.cpu()))
    assert torch.equal(rh.argmax, rd.argmax.cpu())
    assert torch.equal(bits(rh.reduced), bits(rd.reduced.cpu()))
    assert torch.equal(rh.counts, rd.counts.cpu())
    assert int(rh.counts[3]) == 0


def test_host_rows_off_the_16_byte_grid(monkeypatch):
    monkeypatch.setenv("VLMCE_CE_PATH", "rows")
    N, V, S = 530, 70001, 70011
    w = wl(N, V, S, "bf16", 0.0, 0.05, "mean", seed=9)
    x, lab = make_ce_inputs(w, device="cpu")
    buf = torch.full((N, S + 8), float("nan"), dtype=torch.bfloat16)
    buf[:, 3:3 + V] = x[:, :V]
    bh = buf.pin_memory()
    bd = buf.to(DEV)
    rd = ce_fwd_bwd(bd[:, 3:3 + V], lab.to(DEV), label_smoothing=0.05)
    rh = ce_fwd_bwd_host(bh[:, 3:3 + V], lab.pin_memory(), device=DEV, label_smoothing=0.05)
    torch.cuda.synchronize()
    assert torch.equal(bits(bh), bits(bd.cpu()))
    assert torch.equal(bits(rh.loss), bits(rd.loss.cpu()))
    assert torch.equal(rh.argmax, rd.argmax.cpu())


def test_host_outputs_with_device_logits():
    w = wl(160, 3000, 3000, "bf16", 0.0, 0.0, "mean", seed=3)
    x, lab = make_ce_inputs(w, device="cpu")
    xd, xd2, labd = x.to(DEV), x.to(DEV), lab.to(DEV)
    rd = ce_fwd_bwd(xd, labd)
    loss_h = torch.empty(w.N, dtype=torch.float32).pin_memory()
    ws = torch.empty(capi.lib().vlmce_ce_workspace_bytes(w.N, w.V, capi.BF16), dtype=torch.uint8,
                     device=DEV)
    st = capi.lib().ce_fwd_bwd_host(xd2.data_ptr(), capi.BF16, labd.data_ptr(), w.N, w.V, w.V,
                                    -100, 0.0, 0.0, capi.MEAN, 1.0, loss_h.data_ptr(), None, None,
                                    None, ws.data_ptr(), ws.numel(),
                                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == capi.OK
    assert torch.equal(bits(xd2), bits(xd))
    assert torch.equal(bits(loss_h), bits(rd.loss.cpu()))


def test_pageable_host_memory_is_refused():
    N, V = 8, 64
    x = np.zeros((N, V), np.float32)       # pageable: the device cannot address it
    lab = np.zeros(N, np.int64)
    ws = torch.empty(4096, dtype=torch.uint8, device=DEV)
    lib = capi.lib()
    st = lib.ce_fwd_bwd_host(x.ctypes.data, capi.F32, lab.ctypes.data, N, V, V, -100, 0.0, 0.0,
                             capi.MEAN, 1.0, None, None, None, None, ws.data_ptr(), ws.numel(),
                             torch.cuda.current_stream().cuda_stream)
    assert st == capi.ERR_INVALID_ARG
    xp = torch.zeros((N, V), dtype=torch.float32).pin_memory()
    st = lib.ce_fwd_bwd_host(xp.data_ptr(), capi.F32, lab.ctypes.data, N, V, V, -100, 0.0, 0.0,
                             capi.MEAN, 1.0, None, None, None, None, ws.data_ptr(), ws.numel(),
                             torch.cuda.current_stream().cuda_stream)
    assert st == capi.ERR_INVALID_ARG  # pinned logits, pageable labels
    torch.cuda.synchronize()
    assert np.all(x == 0)
