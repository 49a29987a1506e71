"""The C ABI calls are stream-ordered and allocate nothing, so a caller can
capture them in a CUDA graph: a replayed ce_fwd_bwd and a replayed shard rank
step (statistics, merge, loss and gradient) give the same bits as eager calls."""
import pytest
import torch

from vocabulary_lm_cross_gb300 import ce_fwd_bwd
from vocabulary_lm_cross_gb300 import shard as sh
from vocabulary_lm_cross_gb300.ce import CEResult, workspace_bytes
from vocabulary_lm_cross_gb300.workloads import CEWorkload, make_ce_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def result(N):
    return CEResult(loss=torch.empty(N, dtype=torch.float32, device=DEV),
                    argmax=torch.empty(N, dtype=torch.int64, device=DEV),
                    reduced=torch.empty(2, dtype=torch.float32, device=DEV),
                    counts=torch.empty(4, dtype=torch.int64, device=DEV))


def test_replayed_ce_fwd_bwd_equals_eager():
    w = CEWorkload("graph", N=400, V=30011, dtype="bf16", sigma=3.0, ignore_frac=0.05,
                   label_smoothing=0.1, softcap=0.0, reduction="mean", grad_scale=1.0, seed=21)
    x0, lab = make_ce_inputs(w, device=DEV)
    xe = x0.clone()
    re = ce_fwd_bwd(xe, lab, label_smoothing=0.1)
    xg = x0.clone()
    out = result(w.N)
    ws = torch.empty(workspace_bytes(w.N, w.V, xg.dtype), dtype=torch.uint8, device=DEV)
    ce_fwd_bwd(xg, lab, label_smoothing=0.1, out=out, workspace=ws)  # warm-up (attributes, plans)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ce_fwd_bwd(xg, lab, label_smoothing=0.1, out=out, workspace=ws)
    for _ in range(2):
        xg.copy_(x0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(xg.view(torch.int16), xe.view(torch.int16))
        assert torch.equal(out.loss.view(torch.int32), re.loss.view(torch.int32))
        assert torch.equal(out.argmax, re.argmax)
        assert torch.equal(out.reduced.view(torch.int32), re.reduced.view(torch.int32))


def test_replayed_shard_step_equals_eager():
    N, V, tp = 300, 8 * 2048, 8
    w = CEWorkload("graph-shard", N=N, V=V, dtype="bf16", sigma=3.0, ignore_frac=0.05,
                   label_smoothing=0.0, softcap=30.0, reduction="sum", grad_scale=0.25, seed=22)
    x0, lab = make_ce_inputs(w, device=DEV)
    vl = V // tp
    gathered = torch.stack([sh.shard_stats(x0[:, i * vl:(i + 1) * vl].contiguous(), lab, i * vl, V,
                                           softcap=30.0) for i in range(tp)]).contiguous()
    mine0 = x0[:, vl:2 * vl].contiguous()  # rank 1's shard
    kw = dict(softcap=30.0, reduction="sum", grad_scale=0.25)

    def step(b, out, merged, ws):
        sh.shard_stats(b, lab, vl, V, softcap=30.0, out=gathered[1])
        sh.merge_stats(gathered, out=merged)
        sh.shard_fwd_bwd(b, lab, vl, V, merged, out=out, workspace=ws, **kw)

    ws = torch.empty(workspace_bytes(N, V, mine0.dtype), dtype=torch.uint8, device=DEV)
    be, oute, me = mine0.clone(), result(N), torch.empty((N, 8), device=DEV)
    step(be, oute, me, ws)
    torch.cuda.synchronize()
    bg, outg, mg = mine0.clone(), result(N), torch.empty((N, 8), device=DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(bg, outg, mg, ws)
    bg.copy_(mine0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(bg.view(torch.int16), be.view(torch.int16))
    assert torch.equal(mg.view(torch.int32), me.view(torch.int32))
    assert torch.equal(outg.loss.view(torch.int32), oute.loss.view(torch.int32))
    assert torch.equal(outg.reduced.view(torch.int32), oute.reduced.view(torch.int32))
