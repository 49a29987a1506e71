"""GPU parity of the fused gate-up SwiGLU (through the C ABI) against the fp64
oracle: vector and scalar paths, bf16 and fp32, strided rows, an in-place
backward; bf16 results within 1 ulp of the rounded oracle wherever an fp32
evaluation can resolve them.  Tolerance: |r - r_o| <= ulp(r_o) + kappa T with
kappa = 4e-6 (MUFU exp2 and reciprocal ~2^-22 plus a few fp32 roundings) and
T the sum of the magnitudes of the products forming the element."""
import numpy as np
import pytest
import torch

from oracle import ce as oc
from oracle import swiglu as osw
from tests.parity import bf16_bits_np, bits_to_f64, ordered, ulp
from vocabulary_lm_cross_gb300 import capi
from vocabulary_lm_cross_gb300.swiglu import swiglu_bwd, swiglu_fwd

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KAPPA = 4e-6


def inputs(T, n, dtype, seed, x_pad=0, sigma=2.0):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = torch.full((T, 2 * n + x_pad), float("nan"), dtype=dt)
    x[:, :2 * n] = (torch.randn((T, 2 * n), generator=g) * sigma).to(dt)
    dy = torch.randn((T, n), generator=g).to(dt)
    return x, dy


def to64(t, dtype):
    return bits_to_f64(bf16_bits_np(t)) if dtype == "bf16" else t.cpu().double().numpy()


def check(got, ref, terms, dtype, what):
    g = to64(got, dtype)
    u = ulp(ref, dtype)
    cond = KAPPA * terms
    err = np.abs(g - ref)
    bad = ~(err <= u + cond)
    assert not bad.any(), (what, int(bad.sum()), np.argwhere(bad)[0])
    if dtype == "bf16":
        d = np.abs(ordered(bf16_bits_np(got)) - ordered(oc.round_bf16(ref)))
        well = cond <= 0.5 * u
        assert not (well & (d > 1)).any(), (what, "more than 1 ulp from RN(oracle)")


@pytest.mark.parametrize("T,n,dtype,pad", [(300, 4096, "bf16", 0), (97, 1001, "bf16", 0),
                                           (64, 512, "f32", 0), (130, 2048, "bf16", 16),
                                           (33, 257, "f32", 3), (1, 8, "bf16", 0)])
def test_forward_and_backward_against_the_oracle(T, n, dtype, pad):
    x, dy = inputs(T, n, dtype, seed=T + n, x_pad=pad)
    xd, dyd = x.to(DEV), dy.to(DEV)
    y = swiglu_fwd(xd[:, :2 * n])
    dx = swiglu_bwd(xd[:, :2 * n], dyd)
    torch.cuda.synchronize()
    x64, dy64 = to64(x[:, :2 * n], dtype), to64(dy, dtype)
    yo = osw.forward(x64, n)
    check(y.cpu(), yo, np.abs(yo), dtype, "y")
    check(dx.cpu(), osw.backward(x64, dy64, n), osw.backward_terms(x64, dy64, n), dtype, "dx")
    assert torch.isnan(xd[:, 2 * n:]).all()  # padding untouched


def test_in_place_backward_equals_out_of_place():
    T, n = 200, 3000
    x, dy = inputs(T, n, "bf16", seed=5)
    a, b, dyd = x.to(DEV), x.to(DEV), dy.to(DEV)
    ref = swiglu_bwd(a, dyd)
    swiglu_bwd(b, dyd, out=b)
    torch.cuda.synchronize()
    assert torch.equal(ref.view(torch.int16), b.view(torch.int16))


def test_extreme_gates():
    a = torch.tensor([[0.0, 100.0, -100.0, 88.0, -88.0, 1e-30, -1.2785, 3.0]])
    x = torch.cat([a, torch.ones_like(a)], dim=1).to(DEV)
    y = swiglu_fwd(x)
    dx = swiglu_bwd(x, torch.ones((1, 8), device=DEV))
    torch.cuda.synchronize()
    yh, dxh = y.cpu().double().numpy()[0], dx.cpu().double().numpy()[0]
    assert yh[0] == 0.0 and yh[1] == 100.0 and abs(yh[2]) < 1e-30
    assert dxh[0] == 0.5 and abs(dxh[1] - 1.0) < 1e-6 and abs(dxh[2]) < 1e-30
    np.testing.assert_allclose(yh, osw.forward(x.cpu().double().numpy(), 8)[0], rtol=1e-6,
                               atol=1e-30)


def test_argument_errors():
    lib = capi.lib()
    x = torch.zeros((4, 16), device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    assert lib.swiglu_fwd(x.data_ptr(), capi.F32, 4, 8, 15, x.data_ptr(), 8, s) == \
        capi.ERR_INVALID_ARG                                  # x_stride < 2n
    assert lib.swiglu_fwd(x.data_ptr(), capi.F32, 4, 8, 16, x.data_ptr(), 8, s) == \
        capi.ERR_INVALID_ARG                                  # y overlaps x
    assert lib.swiglu_fwd(x.data_ptr(), 7, 4, 8, 16, None, 8, s) == capi.ERR_UNSUPPORTED_DTYPE
    assert lib.swiglu_bwd(x.data_ptr(), 16, None, 8, x.data_ptr(), 16, capi.F32, 4, 8, s) == \
        capi.ERR_INVALID_ARG                                  # no dy
