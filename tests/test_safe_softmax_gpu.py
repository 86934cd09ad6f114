"""GPU parity of the max-subtracted variant (MG_FLAG_SAFE_SOFTMAX) against the fp64 oracle.

The oracle is the graph as written, O = (exp(A) / rowsum(exp(A))) . V, evaluated in fp64, where
exp(A) cannot overflow for these inputs. Subtracting each row's maximum before exp is cancelled
by the normalisation, so the variant must match the same oracle within the same bound,
|O_gpu - O_ref| <= 2e-3 * (1 + |O_ref|), on every workload and on scores far past the fp16 range
of exp(A) (the tutorial's launch example draws Q, K ~ N(0, 1) with d = 128: |A| reaches ~45).
"""

import numpy as np
import pytest
import torch

import oracle
import attention_mugraph_gb300 as mg
from attention_mugraph_gb300 import _lib, build, inputs

pytestmark = pytest.mark.gpu

RTOL = 2e-3
SAFE = mg.MG_FLAG_SAFE_SOFTMAX


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


@pytest.mark.parametrize("name", inputs.CONFIG_ORDER)
def test_workloads(name):
    q, k, v, _ = inputs.make_config(name)
    O, plan = run_gpu(q, k, v, flags=SAFE)
    assert_parity(O, oracle.attention(q, k, v), f"{name} n_split={plan.info['n_split']}")


@pytest.mark.parametrize("B,M,N,d,n_split,flags", [
    (3, 129, 136, 64, 0, 0), (2, 300, 1000, 64, 3, 0), (2, 300, 1000, 64, 3, mg.MG_FLAG_NO_CLUSTER),
    (1, 127, 4104, 128, 0, 0), (4, 64, 6216, 64, 7, 0), (1, 513, 256, 128, 2, 0), (2, 17, 65544, 64, 0, 0),
    (7, 3, 1024, 128, 8, mg.MG_FLAG_NO_CLUSTER), (1, 128, 128, 64, 1, 0), (2, 200, 2056, 64, 1, 0),
    (1, 256, 2048, 64, 5, 0), (1, 1, 8, 128, 0, 0), (16, 8, 32768, 128, 9, mg.MG_FLAG_NO_CLUSTER)])
def test_shapes_and_combines(B, M, N, d, n_split, flags):
    q, k, v = inputs.make_inputs(B, M, N, d, 0.5 if d == 64 else 0.25, seed=7 * B + M + N)
    O, plan = run_gpu(q, k, v, n_split=n_split, flags=SAFE | flags)
    assert_parity(O, oracle.attention(q, k, v), f"{B, M, N, d} n_split={plan.info['n_split']} "
                                                f"cluster={plan.info['cluster_ctas']}")


def test_tutorial_launch_example_normal_draws():
    # Q (64,1,128), K (64,128,4096), V (64,4096,128), all ~ N(0,1).
    q, k, v = inputs.make_inputs_normal(64, 1, 4096, 128, seed=0)
    a = (q.double() @ k.double()).abs().max().item()
    assert a > 20.0  # far past ln(65504) ~ 11.09
    O, _ = run_gpu(q, k, v, flags=SAFE)
    assert_parity(O, oracle.attention(q, k, v), "launch example, N(0,1) draws")


@pytest.mark.parametrize("n_split,flags", [(0, 0), (1, 0), (4, 0), (4, mg.MG_FLAG_NO_CLUSTER), (32, 0)])
def test_large_scores(n_split, flags):
    # Q, K ~ U(-2, 2) at d = 64: scores with a standard deviation near 10.7. The graph as written
    # overflows fp16 (documented precondition); the variant matches the oracle.
    B, M, N, d = 2, 256, 4096, 64
    q, k, v = inputs.make_inputs(B, M, N, d, 2.0, seed=3)
    ref = oracle.attention(q, k, v)
    O, _ = run_gpu(q, k, v, n_split=n_split, flags=SAFE | flags)
    assert_parity(O, ref, f"large scores n_split={n_split} flags={flags}")
    if n_split == 0 and flags == 0:
        plain, _ = run_gpu(q, k, v)
        assert not torch.isfinite(plain).all()


def test_deterministic():
    q, k, v, _ = inputs.make_config("long_kv")
    O1, _ = run_gpu(q, k, v, flags=SAFE)
    O2, _ = run_gpu(q, k, v, flags=SAFE)
    assert torch.equal(O1, O2)


def test_matches_plain_path_on_small_scores():
    # Where the graph as written is in range, both evaluations agree to within the bound too.
    q, k, v, _ = inputs.make_config("gqa")
    ref = oracle.attention(q, k, v)
    a, _ = run_gpu(q, k, v)
    b, _ = run_gpu(q, k, v, flags=SAFE)
    assert_parity(a, ref, "plain")
    assert_parity(b, ref, "safe")


@pytest.mark.parametrize("flags,n_split", [(SAFE, 0), (mg.MG_FLAG_QK_NORM, 0), (SAFE | mg.MG_FLAG_NO_CLUSTER, 0),
                                           (mg.MG_FLAG_QK_NORM | mg.MG_FLAG_NO_CLUSTER, 4)])
def test_bounded_wait_in_variants(flags, n_split):
    # The load warp waits on a barrier nothing arrives on; every role of the variant (row-maximum
    # pass, maximum exchange, cluster or second-kernel combine) unwinds within the bound and the
    # context stays usable.
    q, k, v, _ = inputs.make_config("gqa")
    plan = mg.Plan(2, 256, 4096, 64, n_split=n_split, flags=flags | mg.MG_FLAG_INJECT_TIMEOUT, timeout_ns=2_000_000)
    O = torch.zeros((2, 256, 64), dtype=torch.float16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), O)
    assert plan.status() == mg.MG_ERR_TIMEOUT
    O2, _ = run_gpu(q, k, v, flags=SAFE)
    assert_parity(O2, oracle.attention(q, k, v), "after timeout")


# ---------------------------------------------------------------------------------------------
# The few-row kernel's one-pass form (head dim 128, at most 16 rows per batch): the running
# maximum per softmax group, the rescale of the partial sums and of the O^T accumulator when it
# grows, the merge of the two groups, and split partials that carry their maximum.

ONLINE_SHAPES = [  # (B, M, N, n_split, flags, normal draws)
    (16, 8, 32768, 0, 0, False),                        # decode: 8-CTA clusters
    (16, 8, 32768, 0, mg.MG_FLAG_NO_CLUSTER, False),    # the second kernel, with the maxima
    (64, 1, 4096, 0, 0, True),                          # the launch example's draws: |A| ~ 45
    (64, 1, 4096, 0, mg.MG_FLAG_NO_CLUSTER, True),
    (3, 16, 1032, 1, 0, True),                          # one split: O written directly; ragged N
    (3, 16, 384, 1, 0, False),                          # 3 tiles: group 0 takes two, group 1 one
    (2, 1, 8, 0, 0, True),                              # one ragged tile: group 1 has none
    (5, 3, 5000, 7, 0, True),                           # 7 ranks; ragged N
    (5, 3, 5000, 7, mg.MG_FLAG_NO_CLUSTER, True),
    (4, 8, 8192, 16, 0, True),                          # 16 ranks
    (2, 5, 1032, 9, 0, False),                          # one tile per rank: no group 1 anywhere
]


@pytest.mark.parametrize("B,M,N,n_split,flags,normal", ONLINE_SHAPES)
def test_online_few_row_kernel(B, M, N, n_split, flags, normal):
    d = 128
    if normal:
        q, k, v = inputs.make_inputs_normal(B, M, N, d, seed=B * 11 + M + N)
    else:
        q, k, v = inputs.make_inputs(B, M, N, d, 0.25, seed=B * 11 + M + N)
    O, plan = run_gpu(q, k, v, n_split=n_split, flags=SAFE | flags)
    assert plan.info["swap_ab"] == 1
    assert_parity(O, oracle.attention(q, k, v), f"{B, M, N, d} n_split={plan.info['n_split']} "
                                                f"cluster={plan.info['cluster_ctas']}")
    O2, _ = run_gpu(q, k, v, n_split=n_split, flags=SAFE | flags)
    assert torch.equal(O, O2)


def ramped_keys(B, M, N, rising, seed):
    # N(0, 1) draws with key n scaled by 0.25 + 6 n / N (rising) or its reverse: the rows' maxima
    # climb from ~13 to ~320 across the tiles, so a group's maximum jumps past the kernel's
    # rescale slack (8) on most of its tiles (O^T rescaled in tensor memory), or on none after the
    # first. exp(A) stays finite in the fp64 oracle (A < 709).
    q, k, v = inputs.make_inputs_normal(B, M, N, 128, seed=seed)
    ramp = 0.25 + 6.0 * torch.arange(N, dtype=torch.float32) / N
    if not rising:
        ramp = ramp.flip(0)
    return q, (k.float() * ramp).half().contiguous(), v


@pytest.mark.parametrize("rising", [True, False])
@pytest.mark.parametrize("n_split,flags", [(1, 0), (0, 0), (4, mg.MG_FLAG_NO_CLUSTER)])
def test_online_running_maximum(rising, n_split, flags):
    B, M, N = 4, 16, 4104
    q, k, v = ramped_keys(B, M, N, rising, seed=5)
    ref = oracle.attention(q, k, v)
    O, plan = run_gpu(q, k, v, n_split=n_split, flags=SAFE | flags)
    assert plan.info["swap_ab"] == 1
    assert_parity(O, ref, f"ramp rising={rising} n_split={plan.info['n_split']}")


def test_online_matches_two_pass_kernel():
    # The one-tile kernel's two-pass form (MG_FLAG_NO_SWAP_AB) on the same inputs: both within the
    # bound of the oracle.
    q, k, v, _ = inputs.make_config("decode_m1")
    ref = oracle.attention(q, k, v)
    a, pa = run_gpu(q, k, v, flags=SAFE)
    b, pb = run_gpu(q, k, v, flags=SAFE | mg.MG_FLAG_NO_SWAP_AB)
    assert pa.info["swap_ab"] == 1 and pb.info["swap_ab"] == 0
    assert_parity(a, ref, "one pass")
    assert_parity(b, ref, "two passes")


@pytest.mark.parametrize("flags", [0, mg.MG_FLAG_NO_CLUSTER])
def test_online_bounded_wait(flags):
    # The load warp waits on a barrier nothing arrives on: the group barriers, the rescale's wait
    # and the combine unwind within the bound, and the context stays usable.
    q, k, v, (B, M, N, d) = inputs.make_config("decode")
    plan = mg.Plan(B, M, N, d, flags=SAFE | flags | mg.MG_FLAG_INJECT_TIMEOUT, timeout_ns=2_000_000)
    assert plan.info["swap_ab"] == 1
    O = torch.zeros((B, M, d), dtype=torch.float16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), O)
    assert plan.status() == mg.MG_ERR_TIMEOUT
    O2, _ = run_gpu(q, k, v, flags=SAFE | flags)
    assert_parity(O2, oracle.attention(q, k, v), "after timeout")
