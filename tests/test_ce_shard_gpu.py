"""GPU parity of the vocabulary-sharded cross-entropy (through the C ABI):
shard statistics and their merge against the fp64 shard oracle; the protocol
(statistics per shard -> merge -> loss and gradient per shard) against the
unsharded fp64 oracle with the gradient tolerance of the unsharded kernels;
one shard equal, bit for bit, to ce_fwd_bwd on its row kernel; every shard
reporting identical losses; argument errors before any launch."""
import numpy as np
import pytest
import torch

from oracle import ce as oc
from oracle import ce_shard as osh
from tests.parity import bf16_bits_np, check_grad, check_loss, check_reduced
from vocabulary_lm_cross_gb300 import capi, ce_fwd_bwd
from vocabulary_lm_cross_gb300 import shard as sh
from vocabulary_lm_cross_gb300.workloads import CEWorkload, make_ce_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def wl(N, V, dtype, T, eps, red, seed, stride=0):
    return CEWorkload(f"shard-{N}x{V}", N=N, V=V, dtype=dtype, sigma=3.0, ignore_frac=0.05,
                      label_smoothing=eps, softcap=T, reduction=red, grad_scale=0.5, seed=seed,
                      row_stride=stride, dup_max_frac=0.05, label_boost=3.0)


def stats_lse(stats):
    """log-sum-exp of z per row from the [N, 8] row-statistics records (m + log s)."""
    return stats[:, 2] + torch.log(stats[:, 3])


def stats_argmax(stats):
    """The argmax column stored as int32 bits in word 1 of each record."""
    return stats.view(torch.int32)[:, 1]


def host_x(x, dtype):
    return bf16_bits_np(x) if dtype == "bf16" else x.cpu().numpy()


def widen(xh, dtype):
    if dtype == "bf16":
        return (xh.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return xh.astype(np.float64)


def run_protocol(x_dev, lab_dev, V, cuts, *, eps, T, red, gs):
    """Statistics per shard (copies of the column ranges), merge, fwd_bwd per shard."""
    edges = [0] + list(cuts) + [V]
    shards = [x_dev[:, a:b].contiguous() for a, b in zip(edges[:-1], edges[1:])]
    stats = torch.stack([sh.shard_stats(s, lab_dev, a, V, softcap=T)
                         for s, a in zip(shards, edges[:-1])])
    g = sh.merge_stats(stats)
    outs = [sh.shard_fwd_bwd(s, lab_dev, a, V, g, label_smoothing=eps, softcap=T, reduction=red,
                             grad_scale=gs) for s, a in zip(shards, edges[:-1])]
    torch.cuda.synchronize()
    return edges, shards, stats, g, outs


CASES = [
    # N, V, dtype, T, eps, red, cuts
    (300, 20011, "bf16", 0.0, 0.1, "mean", [1, 9000, 9001, 15000]),
    (160, 4099, "f32", 30.0, 0.0, "sum", [2048]),
    (97, 32768, "bf16", 5.0, 0.2, "mean", [8192, 16384, 24576]),
    (64, 1000, "bf16", 0.0, 0.0, "mean", list(range(100, 1000, 100))),
    # the benchmarked layouts: the headline row length in TP = 8 shards, and the
    # softcap workload's row length in TP = 8 shards
    (256, 131072, "bf16", 0.0, 0.1, "mean", [16384 * i for i in range(1, 8)]),
    (64, 151936, "bf16", 30.0, 0.1, "sum", [18992 * i for i in range(1, 8)]),
]


@pytest.mark.parametrize("N,V,dtype,T,eps,red,cuts", CASES)
def test_shard_protocol_against_the_oracle(N, V, dtype, T, eps, red, cuts):
    w = wl(N, V, dtype, T, eps, red, seed=N * 7 + V)
    x, lab = make_ce_inputs(w, device=DEV)
    xh = host_x(x, dtype)
    labh = lab.cpu().numpy()
    # put some labels on shard edges
    edges = [0] + cuts + [V]
    for i, e in enumerate(edges[1:-1]):
        if 3 * i + 5 < N and labh[3 * i + 5] != -100:
            labh[3 * i + 5] = e
            labh[3 * i + 6] = e - 1 if labh[3 * i + 6] != -100 else -100
    lab = torch.from_numpy(labh).to(DEV)
    edges, shards, stats, g, outs = run_protocol(x, lab, V, cuts, eps=eps, T=T, red=red, gs=0.5)
    x64 = widen(xh, dtype)
    # shard statistics against the shard oracle
    for i, (a, b) in enumerate(zip(edges[:-1], edges[1:])):
        o = osh.shard_stats(x64[:, a:b], a, labh, T)
        s = stats[i].cpu()
        assert np.array_equal(stats_argmax(s).numpy(), o["argmax"]), i
        assert np.array_equal(s[:, 0].numpy().astype(np.float64), o["x_max"]), i
        np.testing.assert_allclose(stats_lse(s).double().numpy(), o["lse"], rtol=2e-6, atol=2e-5)
        np.testing.assert_allclose(s[:, 5].double().numpy(), o["z_y"], rtol=1e-6, atol=1e-5)
        zabs = np.abs(osh._z(x64[:, a:b], T)).sum(axis=1)
        assert np.all(np.abs(s[:, 4].double().numpy() - o["sum_z"]) <= 1e-5 * (zabs + 1))
    # merged statistics against the oracle merge
    om = osh.merge_stats([osh.shard_stats(x64[:, a:b], a, labh, T)
                          for a, b in zip(edges[:-1], edges[1:])])
    gc = g.cpu()
    assert np.array_equal(stats_argmax(gc).numpy(), om["argmax"])
    np.testing.assert_allclose(stats_lse(gc).double().numpy(), om["lse"], rtol=2e-6, atol=2e-5)
    # the protocol's results against the unsharded oracle
    ref = oc.ce_fwd_bwd(xh, dtype, V, labh, label_smoothing=eps, softcap=T, reduction=red,
                        grad_scale=0.5)
    for o in outs:  # identical on every shard
        assert torch.equal(o.loss.view(torch.int32), outs[0].loss.view(torch.int32))
        assert torch.equal(o.argmax, outs[0].argmax)
        assert torch.equal(o.reduced.view(torch.int32), outs[0].reduced.view(torch.int32))
        assert torch.equal(o.counts, outs[0].counts)
    check_loss(outs[0].loss.cpu().numpy(), ref["loss"])
    assert np.array_equal(outs[0].argmax.cpu().numpy(), ref["argmax"])
    counts = outs[0].counts.cpu().numpy()
    assert counts[0] == ref["n_valid"] and counts[1] == ref["n_correct"] and counts[3] == 0
    check_reduced(float(outs[0].reduced[0]), ref["reduced_loss"], red)
    got = np.concatenate([host_x(s, dtype) for s in shards], axis=1)
    check_grad(got, ref["grad"], labh, V, eps, ref["row_scale"], dtype, softcap=T,
               x64=x64[:, :V])


@pytest.mark.parametrize("dtype,T,eps", [("bf16", 0.0, 0.1), ("f32", 30.0, 0.0), ("bf16", 30.0, 0.2)])
def test_one_shard_is_ce_fwd_bwd_bit_for_bit(monkeypatch, dtype, T, eps):
    monkeypatch.setenv("VLMCE_CE_PATH", "rows")
    w = wl(257, 12345, dtype, T, eps, "mean", seed=5, stride=12352)
    x, lab = make_ce_inputs(w, device=DEV)
    V = w.V
    xa = x.clone()
    ra = ce_fwd_bwd(xa[:, :V], lab, label_smoothing=eps, softcap=T, grad_scale=0.5)
    xb = x.clone()
    s = sh.shard_stats(xb[:, :V], lab, 0, V, softcap=T)
    g = sh.merge_stats(s[None])
    rb = sh.shard_fwd_bwd(xb[:, :V], lab, 0, V, g, label_smoothing=eps, softcap=T, grad_scale=0.5)
    torch.cuda.synchronize()
    iv = torch.int16 if dtype == "bf16" else torch.int32
    assert torch.equal(xa.view(iv), xb.view(iv))
    assert torch.equal(ra.loss.view(torch.int32), rb.loss.view(torch.int32))
    assert torch.equal(ra.argmax, rb.argmax)
    assert torch.equal(ra.reduced.view(torch.int32), rb.reduced.view(torch.int32))


# The shard statistics resolve the argmax column of each shard's maximum
# after the merge of the warps; the record merge keeps the smallest column.
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [0.0, 30.0])
def test_argmax_at_planted_maxima_across_shards(dtype, T):
    from tests.test_ce_gpu import planted_maxima
    V = 20001
    x, lab = planted_maxima(64, V, V + 3, dtype)
    cuts = [17, 1000, 1005, V // 2 + 1, V - 19]
    edges, shards, stats, g, outs = run_protocol(x[:, :V], lab, V, cuts, eps=0.1, T=T,
                                                 red="mean", gs=1.0)
    xh = host_x(x[:, :V].contiguous(), dtype)
    labh = lab.cpu().numpy()
    ref = oc.ce_fwd_bwd(xh, dtype, V, labh, label_smoothing=0.1, softcap=T, reduction="mean",
                        want_grad=False)
    for i, (a, b) in enumerate(zip(edges[:-1], edges[1:])):
        o = osh.shard_stats(widen(xh[:, a:b], dtype), a, labh, T)
        assert np.array_equal(stats_argmax(stats[i]).cpu().numpy(), o["argmax"]), i
    assert np.array_equal(stats_argmax(g).cpu().numpy(), ref["argmax"])
    assert np.array_equal(outs[0].argmax.cpu().numpy(), ref["argmax"])


def test_merge_in_place_and_of_identical_shards():
    N = 33
    x = torch.randn(N, 500, device=DEV).to(torch.bfloat16)
    lab = torch.randint(0, 1000, (N,), device=DEV)
    s = sh.shard_stats(x, lab, 500, 1000)
    two = torch.stack([s, s]).contiguous()
    st = capi.lib().ce_merge_stats(two.data_ptr(), 2, N, two.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == capi.OK
    m = two[0]
    assert torch.equal(stats_argmax(m), stats_argmax(s))
    torch.testing.assert_close(stats_lse(m), stats_lse(s) + np.log(2.0), rtol=1e-6, atol=1e-6)


def test_shard_argument_errors():
    lib = capi.lib()
    x = torch.zeros((4, 16), device=DEV)
    lab = torch.zeros(4, dtype=torch.int64, device=DEV)
    out = torch.empty((4, 8), device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    # shard past the vocabulary, negative start, V_local > row_stride
    assert lib.ce_shard_stats(x.data_ptr(), capi.F32, lab.data_ptr(), 4, 16, 16, 10, 20, 0.0,
                              out.data_ptr(), s) == capi.ERR_INVALID_ARG
    assert lib.ce_shard_stats(x.data_ptr(), capi.F32, lab.data_ptr(), 4, 16, 16, -1, 20, 0.0,
                              out.data_ptr(), s) == capi.ERR_INVALID_ARG
    assert lib.ce_shard_stats(x.data_ptr(), capi.F32, lab.data_ptr(), 4, 16, 8, 0, 20, 0.0,
                              out.data_ptr(), s) == capi.ERR_INVALID_ARG
    assert lib.ce_merge_stats(out.data_ptr(), 0, 4, out.data_ptr(), s) == capi.ERR_INVALID_ARG
    ws = torch.empty(64, dtype=torch.uint8, device=DEV)
    assert lib.ce_shard_fwd_bwd(x.data_ptr(), capi.F32, lab.data_ptr(), 4, 16, 16, 0, 16, -100, 0.0,
                                0.0, capi.MEAN, 1.0, out.data_ptr(), None, None, None, None,
                                ws.data_ptr(), ws.numel(), s) == capi.ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("N,V,dtype,T,eps,red,cuts", [CASES[0], CASES[1], CASES[4], CASES[5]])
def test_gathered_call_is_merge_then_fwd_bwd_bit_for_bit(N, V, dtype, T, eps, red, cuts):
    # ce_shard_fwd_bwd_gathered merges the [k, N] records inside the gradient
    # kernel: every output equals ce_merge_stats + ce_shard_fwd_bwd, bit for bit
    w = wl(N, V, dtype, T, eps, red, seed=N * 3 + V)
    x, lab = make_ce_inputs(w, device=DEV)
    edges, shards, stats, g, outs = run_protocol(x, lab, V, cuts, eps=eps, T=T, red=red, gs=0.5)
    fresh = [x[:, a:b].contiguous() for a, b in zip(edges[:-1], edges[1:])]
    for s_ref, s_new, a, o in zip(shards, fresh, edges[:-1], outs):
        r = sh.shard_fwd_bwd(s_new, lab, a, V, stats, label_smoothing=eps, softcap=T,
                             reduction=red, grad_scale=0.5)
        torch.cuda.synchronize()
        assert torch.equal(host_bits(s_new, dtype), host_bits(s_ref, dtype)), a
        assert torch.equal(r.loss.view(torch.int32), o.loss.view(torch.int32))
        assert torch.equal(r.argmax, o.argmax)
        assert torch.equal(r.reduced.view(torch.int32), o.reduced.view(torch.int32))
        assert torch.equal(r.counts, o.counts)


def host_bits(t, dtype):
    return t.view(torch.int16 if dtype == "bf16" else torch.int32).cpu()


def test_gathered_argument_errors():
    lib = capi.lib()
    x = torch.zeros((4, 16), device=DEV)
    lab = torch.zeros(4, dtype=torch.int64, device=DEV)
    recs = torch.zeros((2, 4, 8), device=DEV)
    ws = torch.empty(v_ws(4, 16), dtype=torch.uint8, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    args = (x.data_ptr(), capi.F32, lab.data_ptr(), 4, 16, 16, 0, 16, -100, 0.0, 0.0, capi.MEAN,
            1.0)
    tail = (None, None, None, None, ws.data_ptr(), ws.numel(), s)
    assert lib.ce_shard_fwd_bwd_gathered(*args, recs.data_ptr(), 0, *tail) == capi.ERR_INVALID_ARG
    assert lib.ce_shard_fwd_bwd_gathered(*args, None, 2, *tail) == capi.ERR_INVALID_ARG
    assert lib.ce_shard_fwd_bwd_gathered(*args, recs.data_ptr() + 4, 2, *tail) == \
        capi.ERR_MISALIGNED
    torch.cuda.synchronize()


def v_ws(N, V):
    from vocabulary_lm_cross_gb300.ce import workspace_bytes
    return workspace_bytes(N, V, torch.float32)
