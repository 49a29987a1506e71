"""The C-ABI library loads, exports every symbol include/vlmce.h declares, and
rejects bad arguments on the host before touching the GPU.  CPU only: no
compute call is made."""
import ctypes
import math
import os
import re

import pytest
import torch

from vocabulary_lm_cross_gb300 import build, capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", text):
            name = m.group(1)
            if name in ("if", "sizeof", "defined"):
                continue
            names.add(name)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"ce_fwd_bwd", "vlmce_ce_workspace_bytes", "vlmce_status_string",
            "vlmce_ce_max_vocab"} <= names
    for n in names:
        assert hasattr(lib, n), n
        assert n in capi.SIGNATURES, n


def test_status_strings(lib):
    for code in range(8):
        s = capi.status_string(code)
        assert s.startswith("VLMCE_")
    assert "unknown" in capi.status_string(99)


def test_sizes(lib):
    assert lib.vlmce_ce_max_vocab(capi.BF16) >= 262144
    assert lib.vlmce_ce_max_vocab(capi.F32) >= 131072
    assert lib.vlmce_ce_max_vocab(7) == 0
    assert lib.vlmce_ce_workspace_bytes(2048, 131072, capi.BF16) >= 2048 * 12
    assert lib.vlmce_ce_workspace_bytes(0, 10, capi.BF16) > 0


# Fake, suitably aligned device addresses: the checks below fail before any use.
P = 1 << 20


def call(lib, **kw):
    a = dict(logits=P, dtype=capi.BF16, labels=P, N=4, V=100, row_stride=100, ignore_index=-100,
             eps=0.0, softcap=0.0, reduction=capi.MEAN, grad_scale=1.0, out_loss=P,
             out_argmax=P, out_reduced=P, out_counts=P, ws=P, ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return lib.ce_fwd_bwd(a["logits"], a["dtype"], a["labels"], a["N"], a["V"], a["row_stride"],
                          a["ignore_index"], a["eps"], a["softcap"], a["reduction"],
                          a["grad_scale"], a["out_loss"], a["out_argmax"], a["out_reduced"],
                          a["out_counts"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=5), capi.ERR_UNSUPPORTED_DTYPE),
    (dict(N=-1), capi.ERR_INVALID_ARG),
    (dict(V=0), capi.ERR_INVALID_ARG),
    (dict(row_stride=99), capi.ERR_INVALID_ARG),
    (dict(logits=None), capi.ERR_INVALID_ARG),
    (dict(labels=None), capi.ERR_INVALID_ARG),
    (dict(eps=-0.1), capi.ERR_INVALID_ARG),
    (dict(eps=1.5), capi.ERR_INVALID_ARG),
    (dict(eps=math.nan), capi.ERR_INVALID_ARG),
    (dict(softcap=-1.0), capi.ERR_INVALID_ARG),
    (dict(softcap=math.inf), capi.ERR_INVALID_ARG),
    (dict(softcap=math.nan), capi.ERR_INVALID_ARG),
    (dict(grad_scale=math.nan), capi.ERR_INVALID_ARG),
    (dict(grad_scale=math.inf), capi.ERR_INVALID_ARG),
    (dict(reduction=-1), capi.ERR_INVALID_ARG),
    (dict(reduction=3), capi.ERR_INVALID_ARG),
    (dict(V=(1 << 28) + 1, row_stride=(1 << 28) + 1), capi.ERR_TOO_LARGE),
    (dict(N=(1 << 31), row_stride=100), capi.ERR_TOO_LARGE),
    (dict(ws=None), capi.ERR_WORKSPACE_TOO_SMALL),
    (dict(ws_bytes=16), capi.ERR_WORKSPACE_TOO_SMALL),
    (dict(ws=P + 8), capi.ERR_MISALIGNED),
    (dict(logits=P + 1), capi.ERR_MISALIGNED),
    (dict(logits=P + 2, dtype=capi.F32), capi.ERR_MISALIGNED),
    (dict(labels=P + 4), capi.ERR_MISALIGNED),
    (dict(out_argmax=P + 4), capi.ERR_MISALIGNED),
    (dict(out_counts=P + 4), capi.ERR_MISALIGNED),
    (dict(out_loss=P + 2), capi.ERR_MISALIGNED),
])
def test_argument_errors_are_reported_before_any_launch(lib, kw, code):
    assert call(lib, **kw) == code


def call_ex(lib, gpt, **kw):
    a = dict(logits=P, dtype=capi.BF16, labels=P, N=4, V=100, row_stride=100, ignore_index=-100,
             eps=0.0, softcap=0.0, reduction=capi.NONE, grad_scale=1.0, out_loss=P,
             out_argmax=P, out_reduced=P, out_counts=P, ws=P, ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return lib.ce_fwd_bwd_ex(a["logits"], a["dtype"], a["labels"], a["N"], a["V"],
                             a["row_stride"], a["ignore_index"], a["eps"], a["softcap"],
                             a["reduction"], a["grad_scale"], gpt, 1, a["out_loss"],
                             a["out_argmax"], a["out_reduced"], a["out_counts"], a["ws"],
                             a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("gpt,kw,code", [
    (P + 2, {}, capi.ERR_MISALIGNED),              # per-token gradients not 4-byte aligned
    (P, dict(reduction=3), capi.ERR_INVALID_ARG),
    (P, dict(eps=2.0), capi.ERR_INVALID_ARG),
])
def test_ex_argument_errors_are_reported_before_any_launch(lib, gpt, kw, code):
    assert call_ex(lib, gpt, **kw) == code


def call_flce_rows(lib, **kw):
    a = dict(hidden=P, dtype=capi.BF16, hs=64, weight=P, ws_=64, labels=P, N=4, H=64, V=100,
             ignore_index=-100, eps=0.0, softcap=0.0, reduction=capi.MEAN, grad_scale=1.0,
             out_loss=P, out_argmax=P, out_reduced=P, out_counts=P, gh=P, gw=P, acc=0, chunk=2,
             ws=P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.flce_fwd_bwd_rows(a["hidden"], a["dtype"], a["hs"], a["weight"], a["ws_"],
                                 a["labels"], a["N"], a["H"], a["V"], a["ignore_index"], a["eps"],
                                 a["softcap"], a["reduction"], a["grad_scale"], a["out_loss"],
                                 a["out_argmax"], a["out_reduced"], a["out_counts"], a["gh"],
                                 a["gw"], a["acc"], a["chunk"], a["ws"], a["ws_bytes"],
                                 a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(chunk=0), capi.ERR_INVALID_ARG),
    (dict(chunk=-3), capi.ERR_INVALID_ARG),
    (dict(dtype=capi.F32), capi.ERR_UNSUPPORTED_DTYPE),
    (dict(reduction=capi.NONE), capi.ERR_INVALID_ARG),
    (dict(ws_bytes=1000), capi.ERR_WORKSPACE_TOO_SMALL),
    (dict(ws=P + 16), capi.ERR_MISALIGNED),
    (dict(H=60, hs=64, ws_=64), capi.ERR_MISALIGNED),
    (dict(N=-1), capi.ERR_INVALID_ARG),
])
def test_flce_rows_argument_errors_are_reported_before_any_launch(lib, kw, code):
    assert call_flce_rows(lib, **kw) == code


def test_flce_rows_workspace_bytes(lib):
    f = lib.vlmce_flce_rows_workspace_bytes
    assert f(4096, 6656, 202048, 0) == 0
    assert f(-1, 64, 100, 8) == 0
    small, big = f(4096, 6656, 202048, 512), f(4096, 6656, 202048, 1024)
    # the fp32 logits (4 B) and 16-bit gradient (2 B) of one block dominate
    assert big - small >= 512 * 202048 * 6
    assert f(4096, 6656, 202048, 1 << 20) == f(4096, 6656, 202048, 4096)


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_valid_call_without_a_gpu_fails_cleanly(lib):
    st = call(lib)
    assert st in (capi.ERR_CUDA, capi.ERR_UNSUPPORTED_DEVICE)


def test_binding_raises_loudly_on_bad_input():
    import vocabulary_lm_cross_gb300 as v
    with pytest.raises((ValueError, TypeError)):
        v.ce_fwd_bwd(torch.zeros(3, 4), torch.zeros(3, dtype=torch.int64))


def test_missing_library_raises_instead_of_falling_back(monkeypatch, tmp_path):
    # with no compiled library there is no CPU path: every call raises
    import vocabulary_lm_cross_gb300 as v
    monkeypatch.setattr(capi, "_lib", None)
    monkeypatch.setattr(capi, "LIB", str(tmp_path / "libvlmce.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        capi.lib()
    with pytest.raises(RuntimeError):
        v.ce.workspace_bytes(4, 100, torch.bfloat16)
