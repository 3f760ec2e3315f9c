"""moda_pack_depth reading its source straight from page-locked host memory
(the host-to-device transfer fused with the relayout) gives the same bytes as
the device-to-device relayout; pageable host memory is refused before any
kernel runs."""
import ctypes

import pytest
import torch

import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300.inputs import Workload, make_inputs

import gpu_common as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


@pytest.mark.parametrize("w", [Workload("hp-d128", T=300, Hq=8, Hk=2, d=128, L=13, seed=2),
                               Workload("hp-d64", T=1000, Hq=4, Hk=4, d=64, L=64, seed=3)],
                         ids=lambda w: w.name)
def test_pack_from_pinned_host_equals_device(w):
    x = make_inputs(w)
    host = x["kd"].pin_memory()
    ref = moda.moda_pack_depth(x["kd"].cuda())
    got = moda.moda_pack_depth(host)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    assert torch.equal(got, ref)
    # and again into the same destination, as a step loop does
    got.zero_()
    moda.moda_pack_depth(host, got)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


def test_pack_refuses_pageable_host_memory():
    src = torch.zeros((2, 4, 1, 64), dtype=torch.bfloat16)  # pageable
    dst = torch.empty((1, 4, 2, 64), dtype=torch.bfloat16, device="cuda")
    lib = moda.load()
    lib.moda_pack_depth.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    st = lib.moda_pack_depth(ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(dst.data_ptr()), 2, 4, 1, 64, None)
    assert st == 1  # MODA_ERR_INVALID_ARG
    # and a host destination is refused too
    hdst = torch.empty((1, 4, 2, 64), dtype=torch.bfloat16).pin_memory()
    hsrc = torch.zeros((2, 4, 1, 64), dtype=torch.bfloat16, device="cuda")
    st = lib.moda_pack_depth(ctypes.c_void_p(hsrc.data_ptr()), ctypes.c_void_p(hdst.data_ptr()), 2, 4, 1, 64, None)
    assert st == 1
    assert moda.moda_get_device_error() == 0
