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


# ---------------------------------------------------------------------------------------------
# The few-row kernel's QK-norm form (head dim 128, at most 16 rows per batch): one pass, the
# query scales once per CTA and each tile's key scales from the K tile in shared memory.

QK_SWAP_SHAPES = [  # (B, M, N, n_split, flags)
    (16, 8, 32768, 0, 0),                        # decode
    (16, 8, 32768, 0, mg.MG_FLAG_NO_CLUSTER),
    (64, 1, 4096, 0, 0),                         # the launch example's shapes: 2-CTA clusters
    (3, 16, 1032, 1, 0),                         # one split; ragged N
    (2, 1, 8, 0, 0),                             # one ragged tile
    (5, 3, 5000, 7, 0),
    (5, 3, 5000, 7, mg.MG_FLAG_NO_CLUSTER),
    (4, 8, 8192, 16, 0),
]


@pytest.mark.parametrize("B,M,N,n_split,flags", QK_SWAP_SHAPES)
def test_few_row_kernel(B, M, N, n_split, flags):
    q, k, v = inputs.make_inputs_normal(B, M, N, 128, seed=3 * B + M + N)
    O, plan = run_gpu(q, k, v, n_split=n_split, flags=QK | flags)
    assert plan.info["swap_ab"] == 1
    assert_parity(O, qk_ref(q, k, v), f"{B, M, N} n_split={plan.info['n_split']} "
                                      f"cluster={plan.info['cluster_ctas']}")
    O2, _ = run_gpu(q, k, v, n_split=n_split, flags=QK | flags)
    assert torch.equal(O, O2)


@pytest.mark.parametrize("n_split", [1, 0])
def test_few_row_kernel_scales_per_key_and_row(n_split):
    # Every key vector and query row multiplied by its own power of two (exact in fp16), from
    # 2^-3 to 2^3: the normalisation removes each factor, so the result is the unscaled inputs'
    # up to eps. A key scale applied to the wrong key (or a query scale to the wrong row) is off
    # by up to 2^6 and fails the bound.
    B, M, N = 4, 13, 2056
    q, k, v = inputs.make_inputs_normal(B, M, N, 128, seed=17)
    ref = qk_ref(q, k, v)
    kf = 2.0 ** (torch.arange(N) % 7 - 3).float()
    qf = 2.0 ** (torch.arange(M) % 5 - 2).float()
    ks = (k.float() * kf).half().contiguous()
    qs = (q.float() * qf[:, None]).half().contiguous()
    O, plan = run_gpu(qs, ks, v, n_split=n_split, flags=QK)
    assert plan.info["swap_ab"] == 1
    assert_parity(O, ref, f"per-key and per-row factors n_split={plan.info['n_split']}")


def test_few_row_kernel_matches_one_tile_kernel():
    q, k, v, _ = inputs.make_config("decode_m1")
    ref = qk_ref(q, k, v)
    a, pa = run_gpu(q, k, v, flags=QK)
    b, pb = run_gpu(q, k, v, flags=QK | mg.MG_FLAG_NO_SWAP_AB)
    assert pa.info["swap_ab"] == 1 and pb.info["swap_ab"] == 0
    assert_parity(a, ref, "few-row kernel")
    assert_parity(b, ref, "one-tile kernel")


@pytest.mark.parametrize("flags", [0, mg.MG_FLAG_NO_CLUSTER])
def test_few_row_kernel_bounded_wait(flags):
    # The load warp waits on a barrier nothing arrives on: the wait for Q behind the query scales'
    # barrier, the key-scale waits and the group barriers unwind within the bound.
    q, k, v, (B, M, N, d) = inputs.make_config("decode")
    plan = mg.Plan(B, M, N, d, flags=QK | flags | mg.MG_FLAG_INJECT_TIMEOUT, timeout_ns=2_000_000)
    assert plan.info["swap_ab"] == 1
    O = torch.zeros((B, M, d), dtype=torch.float16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), O)
    assert plan.status() == mg.MG_ERR_TIMEOUT
    O2, _ = run_gpu(q, k, v, flags=QK | flags)
    assert_parity(O2, qk_ref(q, k, v), "after timeout")
