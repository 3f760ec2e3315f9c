"""Failure detection on the GPU without a fault: a bounded wait on a barrier
nothing arrives on gives up, latches MODA_ERR_TIMEOUT, and the context stays
usable for the next forward call."""
import numpy as np
import pytest
import torch

import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300.inputs import Workload, make_inputs

import gpu_common as gc

pytestmark = pytest.mark.gpu

TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


def test_bounded_wait_reports_timeout_and_context_survives():
    assert moda.moda_get_device_error() == 0
    moda.moda_selftest_wait_timeout(50)
    assert moda.moda_get_device_error() == TIMEOUT
    assert moda.moda_get_device_error() == 0          # read clears the word
    w = Workload("after-timeout", T=300, Hq=8, Hk=2, d=128, L=6, seed=12)
    gc.check_workload(w)                              # a normal call still runs and matches
    assert moda.moda_get_device_error() == 0
