"""The two device measurements of include/mg_diag.h on the GPU: the launch floor of the fused
kernel's launch shapes and the exponential rate of its two exp paths."""

import pytest
import torch

import attention_mugraph_gb300 as mg
from attention_mugraph_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    mg.load_library()


@pytest.mark.parametrize("ctas,cluster,pdl", [(64, 16, True), (64, 16, False), (16, 8, True), (152, 1, True)])
def test_launch_floor_is_a_few_microseconds(ctas, cluster, pdl):
    us = mg.diag_launch_floor(ctas, cluster, 215296, pdl, 200)
    assert 0.1 < us < 50.0, us


def test_launch_floor_refuses_small_shared_memory():
    # Below 120 KB two CTAs could share an SM and wait on each other's tensor memory.
    with pytest.raises(mg.MgAttnError) as e:
        mg.diag_launch_floor(64, 16, 64 * 1024, True, 10)
    assert e.value.status == mg.MG_ERR_INVALID_ARG


@pytest.mark.parametrize("poly", [False, True])
def test_exp_rate_is_plausible(poly):
    clk, ns = mg.diag_exp_rate(500, poly=poly)
    # Per SM: at least 1 and at most 128 fp32 exponentials per clock (4 sub-partitions x 32 lanes).
    assert 1.0 < clk <= 128.0, clk
    assert 0.5 < ns < 300.0, ns
