"""Host-side checks of adam_step (no GPU): every call here fails argument
checking before any CUDA call, so the fake device addresses are never
dereferenced (safe on a GPU machine too); n_tensors = 0 is a no-op."""

import ctypes
import os

import pytest

from newton_schulz_08_gb300 import muon

BASE = 0x7F0000000000  # fake, 16-byte aligned device addresses


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(muon.LIB_PATH):
        from newton_schulz_08_gb300 import build
        build.build()
    return muon.lib()


def desc(p=BASE, g=BASE + 0x10000000, m=BASE + 0x20000000, v=BASE + 0x30000000, numel=1000,
         dtype=muon.MUON_BF16):
    return muon.adam_tensor_desc(p, g, m, v, numel, dtype, 0)


def call(L, descs, lr=1e-3, b1=0.9, b2=0.999, eps=1e-8, wd=0.0, step=1, cautious=1):
    arr = (muon.adam_tensor_desc * max(len(descs), 1))(*descs)
    return L.adam_step(arr, len(descs), lr, b1, b2, eps, wd, step, cautious, None)


def test_empty_list_is_a_no_op(L):
    assert L.adam_step(None, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1, None) == muon.MUON_OK


@pytest.mark.parametrize("kw", [dict(step=0), dict(step=-3), dict(b1=1.0), dict(b2=1.5), dict(b1=-0.1),
                                dict(eps=-1e-8), dict(lr=float("inf")), dict(wd=float("nan")),
                                dict(eps=float("nan"))])
def test_bad_hyper_parameters(L, kw):
    bad_first = desc()
    assert call(L, [bad_first], **kw) == muon.MUON_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value", [("param", 0), ("grad", 0), ("exp_avg", 0), ("exp_avg_sq", 0),
                                         ("numel", 0), ("numel", -5), ("grad_dtype", 7)])
def test_bad_descriptor(L, field, value):
    d = desc()
    setattr(d, field, value)
    assert call(L, [d]) == muon.MUON_ERR_INVALID_ARG
    assert L.adam_step(None, 2, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1, None) == muon.MUON_ERR_INVALID_ARG


@pytest.mark.parametrize("field", ["param", "grad", "exp_avg", "exp_avg_sq"])
def test_misaligned(L, field):
    d = desc()
    setattr(d, field, getattr(d, field) + 4)
    assert call(L, [d]) == muon.MUON_ERR_MISALIGNED


def test_aliasing(L):
    # a moment on top of the parameter
    assert call(L, [desc(m=BASE + 16)]) == muon.MUON_ERR_ALIASING
    # the gradient inside a written array
    assert call(L, [desc(g=BASE + 0x30000000 + 64)]) == muon.MUON_ERR_ALIASING
    # two tensors whose parameters overlap
    d2 = desc(p=BASE + 2000, g=BASE + 0x40000000, m=BASE + 0x50000000, v=BASE + 0x60000000)
    assert call(L, [desc(), d2]) == muon.MUON_ERR_ALIASING
    # adjacent, not overlapping: argument checks pass, so it is not called here
    # (it would launch); the check is exercised by the GPU tests


def test_too_large(L):
    assert call(L, [desc(numel=(1 << 40) + 1)]) == muon.MUON_ERR_TOO_LARGE


def test_binding_rejects_mismatched_lists():
    with pytest.raises(ValueError):
        muon.adam_step([1], [], [], [], 1)
