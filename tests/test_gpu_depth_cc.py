"""moda_fwd_depth_cc (the depth slots on CUDA cores, merged into the L = 0
forward) against the fp64 oracle, with the forward's tolerances, and against
moda_fwd on the same inputs."""
import pytest
import torch

import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300 import inputs as wl
from sequence_depth_attention_gb300.inputs import Workload, make_inputs

import gpu_common as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gc.ensure_built()


CASES = [
    wl.TINY,
    Workload("cc-T1", T=1, Hq=4, Hk=2, d=128, L=3),
    Workload("cc-T3-G16", T=3, Hq=16, Hk=1, d=64, L=2),
    Workload("cc-T200-G1-L33", T=200, Hq=3, Hk=3, d=64, L=33),
    Workload("cc-T300-G8-L70", T=300, Hq=16, Hk=2, d=128, L=70, seed=5),
    wl.LAYER_700M,
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_depth_cc_vs_oracle(w):
    gc.check_workload(w, depth_on_cuda_cores=True)


def test_depth_cc_long_sampled():
    gc.check_workload(wl.DEPTH_SWEEP[3], sampled=True, device_inputs=True, depth_on_cuda_cores=True)


def test_depth_cc_equals_fused_depth():
    w = Workload("cc-vs-fused", T=1000, Hq=16, Hk=4, d=128, L=24, seed=9)
    x = make_inputs(w, device="cuda")
    kd, vd = moda.moda_pack_depth(x["kd"]), moda.moda_pack_depth(x["vd"])
    o1, l1 = moda.moda_fwd(x["q"], x["k"], x["v"], kd, vd, w.scale)
    o2, l2 = moda.moda_fwd(x["q"], x["k"], x["v"], kd, vd, w.scale, depth_on_cuda_cores=True)
    torch.cuda.synchronize()
    assert moda.moda_get_device_error() == 0
    assert (o1.float() - o2.float()).abs().max().item() <= gc.TOL_O
    assert (l1 - l2).abs().max().item() <= gc.TOL_LSE
