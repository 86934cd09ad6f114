"""GPU parity of QK-norm attention (MG_FLAG_QK_NORM) against the fp64 oracle.

The graph (Mirage documentation, tutorials/attention-with-kv-norm): Q = rms_norm(Q),
K = rms_norm(K), then A = matmul(Q, K); E = exp(A); S = reduction(E, 2); D = div(E, S);
O = matmul(D, V), rms_norm over the head dimension with eps = 1e-6 and no weight. The oracle
normalises in double; the kernels apply the two normalisations as a row and a column scale of A
in fp32 (with each row's maximum subtracted, since normalised scores reach +-d). Bound:
|O_gpu - O_ref| <= 2e-3 * (1 + |O_ref|) elementwise.
"""

import numpy as np
import pytest
import torch

import oracle
import attention_mugraph_gb300 as mg
from attention_mugraph_gb300 import _lib, build, inputs

pytestmark = pytest.mark.gpu

RTOL = 2e-3
QK = mg.MG_FLAG_QK_NORM


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _lib.load_library()
    yield
    torch.cuda.synchronize()


def run_gpu(q, k, v, **opts):
    B, M, d = q.shape
    N = k.shape[2]
    plan = mg.Plan(B, M, N, d, **opts)
    O = torch.full((B, M, d), float("nan"), dtype=torch.float16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), O)
    torch.cuda.synchronize()
    assert plan.status() == mg.MG_OK
    return O, plan


def assert_parity(O, ref, what):
    o = O.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - ref)
    bound = RTOL * (1.0 + np.abs(ref))
    assert (err <= bound).all(), f"{what}: max err {err.max():.3e}"


def qk_ref(q, k, v):
    return oracle.attention_qknorm(q, k, v, eps=mg.MG_QKNORM_EPS)


@pytest.mark.parametrize("name", inputs.CONFIG_ORDER)
def test_workloads(name):
    q, k, v, _ = inputs.make_config(name)
    O, plan = run_gpu(q, k, v, flags=QK)
    assert_parity(O, qk_ref(q, k, v), f"{name} n_split={plan.info['n_split']}")


@pytest.mark.parametrize("B,M,N,d,n_split,flags", [
    (3, 129, 136, 64, 0, 0), (2, 300, 1000, 64, 3, 0), (2, 300, 1000, 64, 3, mg.MG_FLAG_NO_CLUSTER),
    (1, 127, 4104, 128, 0, 0), (4, 64, 6216, 64, 7, 0), (1, 513, 256, 128, 2, 0), (2, 17, 65544, 64, 0, 0),
    (7, 3, 1024, 128, 8, mg.MG_FLAG_NO_CLUSTER), (1, 128, 128, 64, 1, 0), (2, 200, 2056, 64, 1, 0),
    (1, 1, 8, 128, 0, 0), (2, 64, 1024, 128, 1, 0), (16, 8, 4096, 128, 9, mg.MG_FLAG_NO_CLUSTER)])
def test_shapes_and_combines(B, M, N, d, n_split, flags):
    q, k, v = inputs.make_inputs(B, M, N, d, 0.5 if d == 64 else 0.25, seed=11 * B + M + N)
    O, plan = run_gpu(q, k, v, n_split=n_split, flags=QK | flags)
    assert_parity(O, qk_ref(q, k, v), f"{B, M, N, d} n_split={plan.info['n_split']} "
                                      f"cluster={plan.info['cluster_ctas']} stages={plan.info['stages']}")


def test_normal_draws_and_scale_of_inputs():
    # N(0,1) draws (the tutorial's launch example shapes) and the same inputs with K scaled by 4
    # (exact in fp16): QK-norm removes the scale, so both match the oracle of the unscaled graph
    # up to eps.
    q, k, v = inputs.make_inputs_normal(64, 1, 4096, 128, seed=1)
    ref = qk_ref(q, k, v)
    O, _ = run_gpu(q, k, v, flags=QK)
    assert_parity(O, ref, "N(0,1) draws")
    k4 = (k.float() * 4).half()
    O4, _ = run_gpu(q, k4, v, flags=QK)
    assert_parity(O4, ref, "K scaled by 4")


def test_deterministic_and_combines_agree():
    q, k, v, _ = inputs.make_config("gqa")
    ref = qk_ref(q, k, v)
    O1, p1 = run_gpu(q, k, v, flags=QK)
    O2, _ = run_gpu(q, k, v, flags=QK)
    O3, p3 = run_gpu(q, k, v, flags=QK | mg.MG_FLAG_NO_CLUSTER)
    assert p1.info["cluster_ctas"] > 0 and p3.info["cluster_ctas"] == 0
    assert torch.equal(O1, O2)
    assert_parity(O3, ref, "second-kernel combine")
