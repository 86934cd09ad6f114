"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on the same seeded
fp16 inputs, elementwise within max|O_gpu - O_ref| <= 2e-3 * (1 + |O_ref|).

Covers the six workloads at full size, a shape sweep with ragged M and N tails over both head
dims, every N split and pipeline depth, both combines, the two-Q-tile kernel, degenerate inputs
with closed forms, the largest N, determinism, the host-buffer entry point, CUDA-graph capture and
the bounded-wait status path.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import attention_mugraph_gb300 as mg
from attention_mugraph_gb300 import _lib, build, inputs

pytestmark = pytest.mark.gpu

RTOL = 2e-3  # the acceptance bound: |err| <= RTOL * (1 + |ref|)


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _lib.load_library()
    yield
    torch.cuda.synchronize()


def assert_parity(o_gpu, ref, what=""):
    o = o_gpu.float().cpu().numpy().astype(np.float64) if isinstance(o_gpu, torch.Tensor) else o_gpu
    assert o.shape == ref.shape, what
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - ref)
    bound = RTOL * (1.0 + np.abs(ref))
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (f"{what}: max err {err.max():.3e}; worst at {worst}: gpu {o[worst]} "
                                  f"ref {ref[worst]}")
    return float(err.max())


def run_gpu(q, k, v, **opts):
    B, M, d = q.shape
    N = k.shape[2]
    plan = mg.Plan(B, M, N, d, **opts)
    Q, K, V = q.cuda(), k.cuda(), v.cuda()
    O = torch.full((B, M, d), float("nan"), dtype=torch.float16, device="cuda")
    plan.run(Q, K, V, O)
    torch.cuda.synchronize()
    assert plan.status() == mg.MG_OK
    return O, plan


@pytest.mark.parametrize("name", inputs.CONFIG_ORDER)
def test_workload_parity_full_size(name):
    q, k, v, _ = inputs.make_config(name)
    ref = oracle.attention(q, k, v)
    O, plan = run_gpu(q, k, v)
    assert_parity(O, ref, f"{name} n_split={plan.info['n_split']}")


@pytest.mark.parametrize("name", inputs.CONFIG_ORDER)
def test_workload_parity_in_the_bench_launch_configuration(name):
    # The benchmark's timed launch: back-to-back calls captured in one CUDA graph over rotating
    # input sets (so every call but the graph's first loads its inputs early, while the previous
    # call runs), the default plan (cluster placement included), replayed twice. Every output is
    # checked: in full against the oracle for the smaller workloads, on 64 sampled rows per
    # batch set for the two largest.
    sets = [inputs.make_config(name, seed=s)[:3] for s in range(3)]
    B, M, N, d = inputs.CONFIGS[name][:4]
    plan = mg.Plan(B, M, N, d)
    dev = [tuple(t.cuda() for t in x) for x in sets]
    outs = [torch.full((B, M, d), float("nan"), dtype=torch.float16, device="cuda") for _ in range(6)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.run(*dev[0], outs[0])  # an eager call first, as the bench's warm-up
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        for i, o in enumerate(outs):
            plan.run(*dev[i % 3], o)
        g.capture_end()
    for _ in range(2):
        with torch.cuda.stream(s):
            g.replay()
    s.synchronize()
    assert plan.status() == mg.MG_OK
    big = B * N * d * 2 * 2 > 100_000_000
    rng = np.random.default_rng(5)
    for j, (q, k, v) in enumerate(sets):
        if big:
            rows = np.sort(rng.choice(B * M, size=min(64, B * M), replace=False))
            ref = oracle.attention_rows(q, k, v, rows)
        else:
            ref = oracle.attention(q, k, v)
        for i in range(j, 6, 3):
            o = outs[i].float().cpu().numpy().astype(np.float64)
            got = o.reshape(B * M, d)[rows] if big else o
            err = np.abs(got - ref)
            assert np.isfinite(got).all() and (err <= 2e-3 * (1.0 + np.abs(ref))).all(), \
                f"{name} call {i} (set {j}) n_split={plan.info['n_split']}: max err {err.max():.3e}"


SWEEP = [  # (B, M, N, d, n_split) with ragged M (not a multiple of 128) and N (not of 128)
    (1, 1, 8, 64, 0), (1, 1, 8, 128, 0), (3, 129, 136, 64, 0), (2, 300, 1000, 64, 3),
    (1, 127, 4104, 128, 0), (2, 200, 2056, 64, 1), (1, 128, 128, 64, 1), (4, 64, 6216, 64, 7),
    (1, 513, 256, 128, 2), (2, 17, 65544, 64, 0), (5, 33, 520, 128, 5), (1, 256, 384, 64, 3),
    (7, 3, 1024, 128, 8), (1, 1000, 8192, 64, 0),
]


@pytest.mark.parametrize("B,M,N,d,n_split", SWEEP)
def test_shape_sweep(B, M, N, d, n_split):
    q, k, v = inputs.make_inputs(B, M, N, d, 0.5 if d == 64 else 0.25, seed=B * 1000 + M + N)
    ref = oracle.attention(q, k, v)
    O, _ = run_gpu(q, k, v, n_split=n_split)
    assert_parity(O, ref, f"{B, M, N, d, n_split}")


@pytest.mark.parametrize("n_split,stages", [(1, 4), (2, 2), (3, 3), (5, 4), (32, 2), (31, 3), (7, 5), (4, 6)])
def test_split_and_pipeline_depth(n_split, stages):
    q, k, v, _ = inputs.make_config("gqa")
    ref = oracle.attention(q, k, v)
    O, _ = run_gpu(q, k, v, n_split=n_split, stages=stages)
    assert_parity(O, ref, f"n_split={n_split} stages={stages}")


@pytest.mark.parametrize("n_split,stages", [(1, 2), (3, 3), (9, 2)])
def test_split_and_pipeline_depth_d128(n_split, stages):
    q, k, v = inputs.make_inputs(4, 100, 4104, 128, 0.25, seed=12)
    ref = oracle.attention(q, k, v)
    O, _ = run_gpu(q, k, v, n_split=n_split, stages=stages)
    assert_parity(O, ref, f"d=128 n_split={n_split} stages={stages}")


@pytest.mark.parametrize("B,M,N,d,n_split", [(2, 256, 4096, 64, 16), (1, 200, 2056, 64, 3), (4, 100, 4104, 128, 9),
                                             (3, 129, 1032, 64, 8), (2, 17, 1024, 128, 2), (1, 384, 8192, 64, 13)])
def test_cluster_combine_matches_second_kernel(B, M, N, d, n_split):
    # The cluster combine (the split CTAs of a row tile in one thread-block cluster, partials
    # through L2 after one cluster barrier) and the second-kernel combine of the same split, each
    # against the oracle.
    q, k, v = inputs.make_inputs(B, M, N, d, 0.5 if d == 64 else 0.25, seed=n_split * 7 + d)
    ref = oracle.attention(q, k, v)
    O_cl, plan = run_gpu(q, k, v, n_split=n_split)
    O_k2, plan2 = run_gpu(q, k, v, n_split=n_split, flags=mg.MG_FLAG_NO_CLUSTER)
    assert plan2.info["cluster_ctas"] == 0 and plan2.info["kernels_per_run"] == 2
    assert_parity(O_cl, ref, f"cluster {plan.info['cluster_ctas']}")
    assert_parity(O_k2, ref, "second kernel")


@pytest.mark.parametrize("n_split,flags", [(2, 0), (16, 0), (16, mg.MG_FLAG_SAFE_SOFTMAX)])
def test_cluster_combine_of_cancelling_splits(n_split, flags):
    # Two splits each dominated by one V row, of opposite signs: O is the small difference of two
    # large partials, where any rounding of the exchanged partials shows most.
    B, M, N, d = 1, 3, 2048, 64
    q = torch.zeros((B, M, d))
    q[0, :, 0] = torch.tensor([1.0, 1.25, 1.5])
    k = torch.zeros((B, d, N))
    k[0, 0, :] = -5.0
    k[0, 0, 0] = 5.0      # split 0
    k[0, 0, N // 2] = 5.0  # split n_split / 2
    v = torch.randn((B, N, d), generator=torch.Generator().manual_seed(9)) * 0.01
    v[0, 0, :] = 3.9
    v[0, N // 2, :] = -3.7
    q, k, v = q.half(), k.half(), v.half()
    ref = oracle.attention(q, k, v)
    assert np.abs(ref).max() < 0.2  # the partials (~3.8) nearly cancel
    O, plan = run_gpu(q, k, v, n_split=n_split, flags=flags)
    assert plan.info["cluster_ctas"] == n_split
    assert_parity(O, ref, f"cancelling splits, cluster {n_split}, flags {flags}")


@pytest.mark.parametrize("n_split", [2, 16])
@pytest.mark.parametrize("flags", [0, mg.MG_FLAG_SAFE_SOFTMAX])
def test_cluster_combine_of_cancelling_splits_large_v(n_split, flags):
    # Two splits each dominated by one V row of magnitude ~30, of opposite signs: O (~0.8) is the
    # small difference of two large partials, and the bound 2e-3 * (1 + |O|) does not grow with
    # them. Split j takes column tiles j, j + n_split, ..., so the dominant columns sit in tiles 0
    # and 1: splits 0 and 1 for every n_split >= 2. V is the earlier test's values times 8, which
    # fp16 holds exactly.
    B, M, N, d = 1, 3, 2048, 64
    q = torch.zeros((B, M, d))
    q[0, :, 0] = torch.tensor([1.0, 1.25, 1.5])
    k = torch.zeros((B, d, N))
    k[0, 0, :] = -5.0
    k[0, 0, 0] = 5.0    # column tile 0: split 0
    k[0, 0, 128] = 5.0  # column tile 1: split 1
    v = torch.randn((B, N, d), generator=torch.Generator().manual_seed(9)) * 0.01
    v[0, 0, :] = 3.9
    v[0, 128, :] = -3.7
    q, k, v = q.half(), k.half(), (v.half() * 8)
    ref = oracle.attention(q, k, v)
    assert np.abs(ref).max() < 1.2  # the partials (~30) nearly cancel
    O, plan = run_gpu(q, k, v, n_split=n_split, flags=flags)
    assert plan.info["cluster_ctas"] == n_split
    assert_parity(O, ref, f"cancelling splits |V| ~ 30, cluster {n_split}, flags {flags}")


@pytest.mark.parametrize("d", [64, 128])
def test_cluster_combine_mixed_slices(d):
    # As above, but only some 32-column slices of the dominant V rows are large: in one row, the
    # on-chip exchange adds the fp16 remainders of those slices and not of the others.
    B, M, N = 2, 40, 1024
    g = torch.Generator().manual_seed(17)
    q = torch.zeros((B, M, d))
    q[:, :, 0] = torch.rand((B, M), generator=g) * 0.5 + 1.0
    k = torch.full((B, d, N), -5.0)
    k[:, 1:, :] = 0.0
    k[:, 0, 0] = 5.0
    k[:, 0, 128] = 5.0
    v = torch.randn((B, N, d), generator=g) * 0.5
    wide = [c for c in range(d) if (c // 32) % 2 == 0]  # slices 0, 2: large; 1, 3: small
    v[:, 0, wide] = 29.5
    v[:, 128, wide] = -31.25
    q, k, v = q.half(), k.half(), v.half()
    ref = oracle.attention(q, k, v)
    O, plan = run_gpu(q, k, v, n_split=4)
    assert plan.info["cluster_ctas"] == 4
    assert_parity(O, ref, f"mixed slices d={d}")


PUSH_SHAPES = [  # (B, M, N, n_split, large V slices): head dim 64, cluster combine
    (2, 256, 4096, 16, False),   # the GQA graph's own split
    (1, 200, 2056, 3, True),     # ragged M and N; 3 owners of 42, 43, 43 rows
    (3, 129, 1032, 8, False),    # the second row tile holds one row
    (1, 384, 8192, 13, True),    # 13 owners of 9 or 10 rows
    (2, 17, 1024, 2, True),      # one partial row tile
    (1, 128, 3072, 7, False),    # 7 owners, 24 column tiles
    (2, 64, 1024, 5, True),
    (1, 256, 2048, 11, False),
]


@pytest.mark.parametrize("B,M,N,n_split,large", PUSH_SHAPES)
def test_pushed_combine_matches_pulled_bit_for_bit(B, M, N, n_split, large):
    # The pushed exchange (opt-in: each CTA copies every owner's rows into that owner's receive
    # area) and the pulled one (owners read every CTA's staging) combine the same staged values in the same
    # rank order, so their outputs agree bit for bit; both match the oracle. With large V slices,
    # some rows carry fp16 remainders (pushed only to the owners of those rows).
    d = 64
    q, k, v = inputs.make_inputs(B, M, N, d, 0.5, seed=n_split * 11 + M)
    if large:
        # Batch 0: slice 0 of V around 6, so every partial x there has |x| >= 4 (remainders);
        # other slices and batches stay small (none).
        v = v.float()
        v[0, :, :32] = v[0, :, :32] * 0.5 + 6.0
        v = v.half()
    ref = oracle.attention(q, k, v)
    O_push, plan = run_gpu(q, k, v, n_split=n_split, flags=mg.MG_FLAG_PUSH_COMBINE)
    O_pull, plan2 = run_gpu(q, k, v, n_split=n_split)
    assert plan.info["cluster_ctas"] == n_split and plan.info["xchg_push"] == 1
    assert plan2.info["cluster_ctas"] == n_split and plan2.info["xchg_push"] == 0
    assert_parity(O_push, ref, f"pushed, {n_split} ranks")
    assert torch.equal(O_push, O_pull)
    O_again, _ = run_gpu(q, k, v, n_split=n_split, flags=mg.MG_FLAG_PUSH_COMBINE)
    assert torch.equal(O_push, O_again)


PAIR_SHAPES = [  # (B, M, N, d, n_split, stages): the two-Q-tile kernel forced (MG_FLAG_Q_PAIRS)
    (1, 256, 1024, 64, 1, 0),      # one split: TMA store of both tiles
    (2, 200, 2056, 64, 0, 0),      # ragged M (tile 1 holds rows 128..199) and ragged N
    (1, 129, 8, 64, 0, 0),         # tile 1 holds one row; one ragged column tile
    (3, 512, 1032, 64, 3, 0),      # two pairs per batch, cluster of 3
    (1, 256, 8192, 64, 16, 0),     # cluster of 16
    (2, 256, 4096, 64, 2, 0),      # cluster of 2
    (2, 256, 4096, 64, 20, 0),     # 20 splits: second kernel
    (4, 256, 520, 64, 5, 2),       # two-stage ring
    (1, 256, 3072, 64, 1, 3),      # one split, 24 tiles through a three-stage ring
    (2, 384, 2048, 64, 4, 0),      # three row tiles: odd, so the one-tile kernel serves it
]


@pytest.mark.parametrize("B,M,N,d,n_split,stages", PAIR_SHAPES)
def test_two_q_tile_kernel(B, M, N, d, n_split, stages):
    q, k, v = inputs.make_inputs(B, M, N, d, 0.5, seed=B * 31 + M + N + n_split)
    ref = oracle.attention(q, k, v)
    O, plan = run_gpu(q, k, v, n_split=n_split, stages=stages, flags=mg.MG_FLAG_Q_PAIRS)
    want_pairs = (-(-M // 128)) % 2 == 0
    assert plan.info["q_tiles_per_cta"] == (2 if want_pairs else 1)
    assert_parity(O, ref, f"pairs {B, M, N, d} n_split={plan.info['n_split']} cluster={plan.info['cluster_ctas']}")


@pytest.mark.parametrize("flags", [0, mg.MG_FLAG_NO_CLUSTER])
def test_two_q_tile_kernel_matches_one_tile_kernel(flags):
    # The batch-8 GQA shape through both kernels, each against the oracle; the two-tile kernel is
    # reproducible bit for bit, run to run.
    q, k, v, _ = inputs.make_config("gqa_b8")
    ref = oracle.attention(q, k, v)
    O2, p2 = run_gpu(q, k, v, flags=flags | mg.MG_FLAG_Q_PAIRS)
    O2b, _ = run_gpu(q, k, v, flags=flags | mg.MG_FLAG_Q_PAIRS)
    O1, p1 = run_gpu(q, k, v, flags=flags | mg.MG_FLAG_NO_Q_PAIRS)
    assert p2.info["q_tiles_per_cta"] == 2 and p1.info["q_tiles_per_cta"] == 1
    assert_parity(O2, ref, "two-tile")
    assert_parity(O1, ref, "one-tile")
    assert torch.equal(O2, O2b)


SK_SHAPES = [  # (B, M, N, d): the stream-K schedule forced (MG_FLAG_STREAM_K)
    (20, 5, 3000, 64),     # runs of 3-4 units crossing batches; ragged N
    (37, 16, 1032, 64),    # 16 rows; runs of 2-3 units; ragged N
    (7, 3, 1000, 128),     # fewer units than SMs: one unit per CTA
    (64, 1, 4096, 128),    # the launch example's shapes
    (16, 8, 32768, 128),   # decode-like
    (3, 9, 262144, 64),    # long runs: 1536 units over 152 CTAs, 2 batches touched by many
]


@pytest.mark.parametrize("B,M,N,d", SK_SHAPES)
def test_stream_k_schedule(B, M, N, d):
    q, k, v = inputs.make_inputs(B, M, N, d, 0.5 if d == 64 else 0.25, seed=B + M + N)
    ref = oracle.attention(q, k, v)
    O, plan = run_gpu(q, k, v, flags=mg.MG_FLAG_STREAM_K)
    assert plan.info["schedule"] == 1
    assert_parity(O, ref, f"stream-K {B, M, N, d} slots={plan.info['n_split']} ctas={plan.info['grid_ctas']}")
    # Reproducible bit for bit, and on a second call (every partial slot rewritten or re-zeroed).
    O2 = torch.full_like(O, float("nan"))
    plan.run(q.cuda(), k.cuda(), v.cuda(), O2)
    torch.cuda.synchronize()
    assert torch.equal(O, O2)


def test_stream_k_matches_split_schedule():
    q, k, v, _ = inputs.make_config("decode_m1")
    ref = oracle.attention(q, k, v)
    O_sk, p_sk = run_gpu(q, k, v, flags=mg.MG_FLAG_STREAM_K)
    O_sp, p_sp = run_gpu(q, k, v, flags=mg.MG_FLAG_NO_STREAM_K)
    assert p_sk.info["schedule"] == 1 and p_sp.info["schedule"] == 0
    assert_parity(O_sk, ref, "stream-K")
    assert_parity(O_sp, ref, "split")


SWAP_SHAPES = [  # (B, M, N, d, n_split): the few-row specialisation forced (MG_FLAG_SWAP_AB)
    (16, 8, 32768, 128, 0),    # decode-like, the second kernel
    (64, 1, 4096, 128, 0),     # the launch example's shapes
    (3, 16, 1032, 128, 1),     # 16 rows, one split: O written directly; ragged N
    (5, 3, 5000, 128, 7),      # 3 rows; ragged N; 7 splits
    (2, 1, 8, 128, 0),         # one query row, one ragged column tile
]


@pytest.mark.parametrize("B,M,N,d,n_split", SWAP_SHAPES)
def test_swap_ab_specialisation(B, M, N, d, n_split):
    q, k, v = inputs.make_inputs(B, M, N, d, 0.25, seed=B * 7 + M + N)
    ref = oracle.attention(q, k, v)
    O, plan = run_gpu(q, k, v, n_split=n_split, flags=mg.MG_FLAG_SWAP_AB)
    assert plan.info["swap_ab"] == 1
    assert_parity(O, ref, f"swap-AB {B, M, N, d} n_split={plan.info['n_split']}")


# The few-row kernel releases each stage's K half after its S^T product (in the QK-norm form also
# after the softmax warps' reads of the key scales) and issues K tiles two ahead of V: rings of 2
# and 3 stages, several tiles per CTA and a ragged last tile (N a multiple of 8, the layout rule),
# for the graph as written and both one-pass variants.
SWAP_RING_CASES = [  # (B, M, N, n_split, stages)
    (2, 8, 128 * 11 + 40, 2, 2),
    (2, 8, 128 * 11 + 40, 2, 3),
    (3, 1, 128 * 7 + 8, 1, 2),
    (1, 16, 128 * 13, 3, 3),
]


@pytest.mark.parametrize("flags", [0, mg.MG_FLAG_SAFE_SOFTMAX, mg.MG_FLAG_QK_NORM])
@pytest.mark.parametrize("B,M,N,n_split,stages", SWAP_RING_CASES)
def test_swap_ab_split_ring_release(B, M, N, n_split, stages, flags):
    d = 128
    q, k, v = inputs.make_inputs(B, M, N, d, 0.25, seed=B * 31 + M + N + stages)
    ref = (oracle.attention_qknorm(q, k, v, eps=mg.MG_QKNORM_EPS) if flags == mg.MG_FLAG_QK_NORM
           else oracle.attention(q, k, v))
    O, plan = run_gpu(q, k, v, n_split=n_split, stages=stages, flags=flags | mg.MG_FLAG_SWAP_AB)
    assert plan.info["swap_ab"] == 1 and plan.info["stages"] == stages
    assert_parity(O, ref, f"swap-AB ring {B, M, N} n_split={n_split} stages={stages} flags={flags:#x}")


SWAP_CLUSTER_SHAPES = [  # (B, M, N, n_split): head dim 128, few rows, split partials
    (64, 1, 4096, 2),     # the launch example's shapes, as planned
    (4, 8, 8192, 16),     # 16 ranks of 8 columns each
    (5, 3, 5000, 7),      # 7 ranks of 18 or 19 columns; 3 rows; ragged N
    (3, 16, 2048, 3),     # 16 rows
    (2, 5, 1032, 9),      # ragged N (9 column tiles, one per rank)
]


@pytest.mark.parametrize("B,M,N,n_split", SWAP_CLUSTER_SHAPES)
def test_swap_ab_cluster_combine(B, M, N, n_split):
    # The few-row kernel's split partials combined on chip (fp32 O^T columns and row sums across
    # the cluster) and by the second kernel: each against the oracle, and each reproducible.
    d = 128
    q, k, v = inputs.make_inputs(B, M, N, d, 0.25, seed=B * 13 + M + n_split)
    ref = oracle.attention(q, k, v)
    O_cl, plan = run_gpu(q, k, v, n_split=n_split)
    O_k2, plan2 = run_gpu(q, k, v, n_split=n_split, flags=mg.MG_FLAG_NO_CLUSTER)
    assert plan.info["swap_ab"] == 1 and plan2.info["swap_ab"] == 1
    assert plan2.info["cluster_ctas"] == 0 and plan2.info["kernels_per_run"] == 2
    assert_parity(O_cl, ref, f"swap-AB cluster {plan.info['cluster_ctas']} of {n_split}")
    assert_parity(O_k2, ref, "swap-AB second kernel")
    O_again, _ = run_gpu(q, k, v, n_split=n_split)
    assert torch.equal(O_cl, O_again)


def test_swap_ab_matches_one_tile_kernel_and_is_reproducible():
    q, k, v, _ = inputs.make_config("decode")
    ref = oracle.attention(q, k, v)
    O1, _ = run_gpu(q, k, v, flags=mg.MG_FLAG_SWAP_AB)
    O2, _ = run_gpu(q, k, v, flags=mg.MG_FLAG_SWAP_AB)
    O3, p3 = run_gpu(q, k, v, flags=mg.MG_FLAG_NO_SWAP_AB)
    assert p3.info["swap_ab"] == 0
    assert torch.equal(O1, O2)
    assert_parity(O1, ref, "swap-AB")
    assert_parity(O3, ref, "one-tile")


def test_cluster_placement_for_back_to_back_calls():
    # Without an explicit n_split, the plan asks the device how many clusters it holds at once
    # (GB300: 23 of 6 CTAs, 15 of 7-9, 8 of 11-12, 7 of 13-16). It first keeps the clusters of one
    # call placeable (a smaller cluster, else the second kernel), then, for calls that start early,
    # takes the split count that lets the most calls be in flight (up to 4) within max(8, placed)
    # column tiles per CTA. An explicit n_split is kept.
    gqa = mg.Plan(2, 256, 4096, 64).info
    assert gqa["cluster_ctas"] == gqa["n_split"] == 6
    assert mg.Plan(2, 256, 4096, 64, n_split=16).info["cluster_ctas"] == 16
    # Planned for calls that do not overlap: the count placed for one call's latency.
    assert mg.Plan(2, 256, 4096, 64, flags=mg.MG_FLAG_ISOLATED).info["n_split"] == 12
    # MG_FLAG_NO_EARLY_LOADS changes when a call's kernels run, not the plan.
    assert mg.Plan(2, 256, 4096, 64, flags=mg.MG_FLAG_NO_EARLY_LOADS).info["n_split"] == 6
    assert mg.Plan(1, 256, 4096, 64).info["n_split"] == 12
    assert mg.Plan(2, 64, 1024, 64).info["n_split"] == 8  # 4 tiny calls in flight already
    b4 = mg.Plan(4, 256, 4096, 64).info
    assert b4["cluster_ctas"] == b4["n_split"] == 4 and b4["kernels_per_run"] == 1
    b8 = mg.Plan(8, 256, 4096, 64).info  # 9-CTA clusters do not fit once: a smaller cluster
    assert b8["cluster_ctas"] == b8["n_split"] == 4 and b8["kernels_per_run"] == 1
    # One call of 4 splits fills the device: up to twice its tiles per CTA for a second call,
    # except in the two-pass variants.
    assert mg.Plan(16, 256, 4096, 64).info["n_split"] == 2
    assert mg.Plan(16, 256, 4096, 64, flags=mg.MG_FLAG_SAFE_SOFTMAX).info["n_split"] == 4
    # QK-norm's one-tile form starts early only with its key scales in shared memory: there it
    # takes the same count; at head dim 128 (no room beside the ring) it keeps the placed one.
    assert mg.Plan(2, 256, 4096, 64, flags=mg.MG_FLAG_QK_NORM).info["n_split"] == 6
    assert mg.Plan(2, 256, 4096, 128, flags=mg.MG_FLAG_QK_NORM).info["n_split"] == 16
    for shape in [(2, 256, 4096, 64), (4, 256, 4096, 64), (8, 256, 4096, 64), (1, 256, 4096, 64)]:
        q, k, v = inputs.make_inputs(*shape, 0.5, seed=sum(shape))
        O, plan = run_gpu(q, k, v)
        assert_parity(O, oracle.attention(q, k, v), f"{shape} n_split={plan.info['n_split']}")


def test_k_zero_gives_mean_of_v_with_ragged_tail():
    # Scores 0 everywhere -> every weight is exp(0)=1: any column past N that leaked into the row
    # sum (zero-filled K gives exp(0)=1 too) would pull the mean toward 0.
    B, M, N, d = 2, 130, 1032, 64
    _, _, v = inputs.make_inputs(B, M, N, d, seed=3)
    q = torch.randn((B, M, d)).half()
    k = torch.zeros((B, d, N), dtype=torch.float16)
    O, _ = run_gpu(q, k, v, n_split=3)
    want = v.double().numpy().mean(axis=1, keepdims=True).repeat(M, axis=1)
    assert_parity(O, want, "K=0")


def test_constant_v():
    B, M, N, d = 1, 64, 2048, 128
    q, k, _ = inputs.make_inputs(B, M, N, d, 0.25, seed=4)
    v = torch.full((B, N, d), -1.5, dtype=torch.float16)
    O, _ = run_gpu(q, k, v)
    assert torch.all(O.float() == -1.5) or assert_parity(O, np.full((B, M, d), -1.5), "V=const") is not None


def test_single_query_eight_keys():
    # The smallest problem the layout allows: one query row, N = 8 (one ragged column tile).
    q, k, v = inputs.make_inputs(3, 1, 8, 64, 0.5, seed=5)
    ref = oracle.attention(q, k, v)
    O, _ = run_gpu(q, k, v)
    assert_parity(O, ref, "M=1,N=8")


def test_largest_n_sampled_rows():
    # N = 2^20 keys: row sums of a million fp32 terms; checked on sampled rows.
    B, M, N, d = 1, 256, 1 << 20, 64
    q, k, v = inputs.make_inputs(B, M, N, d, 0.5, seed=6)
    O, plan = run_gpu(q, k, v)
    rows = list(range(0, B * M, 17)) + [B * M - 1]
    ref = oracle.attention_rows(q, k, v, rows)
    got = O.float().cpu().numpy().astype(np.float64).reshape(-1, d)[rows]
    assert_parity(got, ref, f"N=2^20 n_split={plan.info['n_split']}")


def test_deterministic_and_pdl_invariant():
    q, k, v, _ = inputs.make_config("gqa")
    O1, _ = run_gpu(q, k, v)
    O2, _ = run_gpu(q, k, v)
    O3, _ = run_gpu(q, k, v, flags=mg.MG_FLAG_NO_PDL)
    assert torch.equal(O1, O2) and torch.equal(O1, O3)


def test_back_to_back_runs_on_side_stream():
    # Many calls queued on one non-default stream, alternating two input sets, each checked.
    sets = [inputs.make_inputs(2, 256, 4096, 64, 0.5, seed=s) for s in (10, 11)]
    refs = [oracle.attention(*s) for s in sets]
    plan = mg.Plan(2, 256, 4096, 64)
    dev = [[t.cuda() for t in s] for s in sets]
    outs = [torch.empty((2, 256, 64), dtype=torch.float16, device="cuda") for _ in range(6)]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i, o in enumerate(outs):
            plan.run(*dev[i % 2], o, stream=stream)
    stream.synchronize()
    for i, o in enumerate(outs):
        assert_parity(o, refs[i % 2], f"call {i}")


def test_cuda_graph_capture_replay():
    q, k, v, _ = inputs.make_config("gqa")
    ref = oracle.attention(q, k, v)
    plan = mg.Plan(2, 256, 4096, 64)
    Q, K, V = q.cuda(), k.cuda(), v.cuda()
    O = torch.zeros((2, 256, 64), dtype=torch.float16, device="cuda")
    plan.run(Q, K, V, O)  # warm-up outside capture
    torch.cuda.synchronize()
    O.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.capture_begin()
        plan.run(Q, K, V, O, stream=s)
        g.capture_end()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert_parity(O, ref, "graph replay")


@pytest.mark.parametrize("kw", [{}, {"n_split": 1}, {"flags": mg.MG_FLAG_NO_CLUSTER}])
def test_host_buffer_entry_point(kw):
    # Pinned buffers: O is written straight to the host buffer when N is split (the cluster
    # combine, the second kernel), and staged and copied back with one split.
    q, k, v, _ = inputs.make_config("tiny")
    ref = oracle.attention(q, k, v)
    plan = mg.Plan(2, 64, 1024, 64, **kw)
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    ho = torch.empty((2, 64, 64), dtype=torch.float16).pin_memory()
    for _ in range(2):
        plan.run_host(hq, hk, hv, ho)
        torch.cuda.synchronize()
        assert_parity(ho, ref, "run_host")


@pytest.mark.parametrize("kw", [{}, {"n_split": 1}])
def test_host_buffer_back_to_back_calls(kw):
    # Calls enqueued back to back without synchronising: each call's copy kernel loads its pinned
    # inputs while the previous call's kernels may still run (and stores them only after those
    # end). Distinct inputs per call, each result checked; then calls chained in place (O of one
    # call is Q of the next, one host buffer), where the loads must wait for the previous call.
    B, M, N, d = 2, 64, 1024, 64
    plan = mg.Plan(B, M, N, d, **kw)
    sets = [inputs.make_inputs(B, M, N, d, 0.5, seed=40 + i) for i in range(4)]
    pinned = [tuple(t.pin_memory() for t in s) for s in sets]
    outs = [torch.full((B, M, d), float("nan"), dtype=torch.float16).pin_memory() for _ in sets]
    for (hq, hk, hv), ho in zip(pinned, outs):
        plan.run_host(hq, hk, hv, ho)
    torch.cuda.synchronize()
    for (q, k, v), ho in zip(sets, outs):
        assert_parity(ho, oracle.attention(q, k, v), "back to back")
    q, k, v = sets[0]
    h = q.clone().pin_memory()
    hk, hv = k.pin_memory(), v.pin_memory()
    for _ in range(3):
        plan.run_host(h, hk, hv, h)
    torch.cuda.synchronize()
    cur = q.clone()
    for i in range(3):  # the same chain, one synchronised call at a time, separate buffers
        o = torch.full((B, M, d), float("nan"), dtype=torch.float16).pin_memory()
        hc = cur.pin_memory()
        plan.run_host(hc, hk, hv, o)
        torch.cuda.synchronize()
        if i == 0:
            assert_parity(o, oracle.attention(cur, k, v), "chain, first call")
        cur = o.clone()
    assert torch.equal(h, cur)


@pytest.mark.parametrize("kw", [{}, {"n_split": 1}])
def test_host_buffer_chained_calls(kw):
    # Back to back without synchronising, each call's Q is the previous call's O in another
    # pinned buffer: the copy kernel must not load that input before the previous call has
    # written it (the entry point compares its inputs with the previous call's output on the
    # stream). Compared bit for bit with the same chain run one synchronised call at a time.
    B, M, N, d = 2, 64, 1024, 64
    plan = mg.Plan(B, M, N, d, **kw)
    q, k, v = inputs.make_inputs(B, M, N, d, 0.5, seed=71)
    hk, hv = k.pin_memory(), v.pin_memory()
    bufs = [q.clone().pin_memory()] + [torch.full((B, M, d), float("nan"), dtype=torch.float16).pin_memory()
                                       for _ in range(4)]
    for i in range(4):
        plan.run_host(bufs[i], hk, hv, bufs[i + 1])
    torch.cuda.synchronize()
    cur = q.clone()
    for i in range(4):
        hc = cur.pin_memory()
        o = torch.full((B, M, d), float("nan"), dtype=torch.float16).pin_memory()
        plan.run_host(hc, hk, hv, o)
        torch.cuda.synchronize()
        assert torch.equal(o, bufs[i + 1]), f"call {i} of the chain"
        cur = o.clone()


EARLY_OFF = mg.MG_FLAG_NO_EARLY_LOADS | mg.MG_FLAG_NO_PDL


def chain_inputs(q, k, v, which, prev):
    # The call's (Q, K, V), with the one named by `which` replaced by the previous call's O (the
    # same bytes, viewed in that input's shape).
    x = {"q": q, "k": k, "v": v}
    if prev is not None:
        x[which] = prev.view(x[which].shape)
    return x["q"], x["k"], x["v"]


@pytest.mark.parametrize("which", ["q", "k", "v"])
@pytest.mark.parametrize("kw", [{}, {"n_split": 1}, {"flags": mg.MG_FLAG_NO_CLUSTER}])
def test_device_chained_calls(which, kw):
    # Back to back on one stream without synchronising, each call's Q (or K, or V) is the previous
    # call's O: the fused kernel may load its inputs before the previous kernel on the stream has
    # completed, and must not do so here (its inputs share bytes with the previous call's output).
    # Compared bit for bit with the same chain run one synchronised call at a time with the early
    # loads and dependent launch off. M = N so that O has the shape of Q, V and (viewed) K.
    B, M, N, d = 2, 256, 256, 64
    plan = mg.Plan(B, M, N, d, **kw)
    q, k, v = (t.cuda() for t in inputs.make_inputs(B, M, N, d, 0.5, seed=83))
    outs = [torch.full((B, M, d), float("nan"), dtype=torch.float16, device="cuda") for _ in range(6)]
    prev = None
    for o in outs:
        plan.run(*chain_inputs(q, k, v, which, prev), o)
        prev = o
    torch.cuda.synchronize()
    ref_plan = mg.Plan(B, M, N, d, n_split=kw.get("n_split", 0), flags=kw.get("flags", 0) | EARLY_OFF)
    prev = None
    for i, o in enumerate(outs):
        r = torch.full((B, M, d), float("nan"), dtype=torch.float16, device="cuda")
        ref_plan.run(*chain_inputs(q, k, v, which, prev), r)
        torch.cuda.synchronize()
        assert torch.equal(r, o), f"call {i} of the {which} chain"
        prev = r


@pytest.mark.parametrize("shape,back", [((2, 256, 4096, 64), 2), ((2, 64, 1024, 64), 5), ((16, 8, 32768, 128), 2)])
def test_device_calls_reading_an_output_further_back(shape, back):
    # Back to back on one stream, call i's Q is call (i - back)'s O. These plans start at level 2
    # (dependents released at the start: a call may run while calls before the previous one still
    # do); the library compares the inputs with the outputs of its recent calls, not only the
    # previous one. Bit for bit against the same calls run one at a time, synchronised.
    B, M, N, d = shape
    plan = mg.Plan(B, M, N, d)
    n = back + 6
    qs = [t.cuda() for t in (inputs.make_inputs(B, M, N, d, 0.5 if d == 64 else 0.25, seed=200 + i)[0] for i in range(n))]
    _, k, v = inputs.make_inputs(B, M, N, d, 0.5 if d == 64 else 0.25, seed=199)
    k, v = k.cuda(), v.cuda()
    outs = [torch.full((B, M, d), float("nan"), dtype=torch.float16, device="cuda") for _ in range(n)]
    for i in range(n):
        plan.run(outs[i - back] if i >= back else qs[i], k, v, outs[i])
    torch.cuda.synchronize()
    ref_plan = mg.Plan(B, M, N, d, flags=EARLY_OFF)
    refs = []
    for i in range(n):
        r = torch.full((B, M, d), float("nan"), dtype=torch.float16, device="cuda")
        ref_plan.run(refs[i - back] if i >= back else qs[i], k, v, r)
        torch.cuda.synchronize()
        refs.append(r)
        assert torch.equal(r, outs[i]), f"call {i} (reads call {i - back})"


def test_device_chain_in_captured_graph():
    # Two calls captured into one graph, the second reading the first's O as Q, replayed three
    # times: within the capture the first call has no known predecessor (no early loads) and the
    # second sees the first's output.
    B, M, N, d = 2, 256, 256, 64
    plan = mg.Plan(B, M, N, d)
    q, k, v = (t.cuda() for t in inputs.make_inputs(B, M, N, d, 0.5, seed=89))
    o1 = torch.full((B, M, d), float("nan"), dtype=torch.float16, device="cuda")
    o2 = torch.full_like(o1, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.run(q, k, v, torch.empty_like(o1))  # an eager call on the stream first
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        plan.run(q, k, v, o1)
        plan.run(o1, k, v, o2)
        g.capture_end()
    for _ in range(3):
        with torch.cuda.stream(s):
            o1.fill_(float("nan"))
            o2.fill_(float("nan"))
            g.replay()
    s.synchronize()
    ref_plan = mg.Plan(B, M, N, d, flags=EARLY_OFF)
    r1 = torch.empty_like(o1)
    r2 = torch.empty_like(o1)
    ref_plan.run(q, k, v, r1)
    torch.cuda.synchronize()
    ref_plan.run(r1, k, v, r2)
    torch.cuda.synchronize()
    assert torch.equal(o1, r1) and torch.equal(o2, r2)


def test_eager_call_after_a_capture():
    # An eager call X, a capture of an unrelated call on the same stream, then an eager call Z
    # whose Q is X's O: Z's predecessor on the stream is X (the captured call has not run), so Z
    # must compare its inputs with X's output, not with the captured call's. X is long (~30 us)
    # so that Z, if it loaded early, would read Q before X wrote it.
    d = 64
    px = mg.Plan(16, 256, 16384, d)
    pz = mg.Plan(16, 256, 4096, d)
    qx, kx, vx = (t.cuda() for t in inputs.make_inputs(16, 256, 16384, d, 0.5, seed=97))
    qz, kz, vz = (t.cuda() for t in inputs.make_inputs(16, 256, 4096, d, 0.5, seed=98))
    ox = torch.full((16, 256, d), float("nan"), dtype=torch.float16, device="cuda")
    oy = torch.empty_like(ox)
    oz = torch.full_like(ox, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        px.run(qx, kx, vx, ox)
        g.capture_begin()
        pz.run(qz, kz, vz, oy)
        g.capture_end()
        pz.run(ox, kz, vz, oz)
    s.synchronize()
    rx = torch.empty_like(ox)
    rz = torch.empty_like(ox)
    mg.Plan(16, 256, 16384, d, flags=EARLY_OFF).run(qx, kx, vx, rx)
    torch.cuda.synchronize()
    mg.Plan(16, 256, 4096, d, flags=EARLY_OFF).run(rx, kz, vz, rz)
    torch.cuda.synchronize()
    assert torch.equal(ox, rx) and torch.equal(oz, rz)


def test_early_loads_leave_results_unchanged():
    # Distinct buffers back to back (the early loads taken) against the same calls with them off.
    q, k, v, (B, M, N, d) = inputs.make_config("gqa")
    sets = [tuple(t.cuda() for t in inputs.make_inputs(B, M, N, d, 0.5, seed=100 + i)) for i in range(4)]
    for flags in (0, mg.MG_FLAG_NO_CLUSTER):
        a = mg.Plan(B, M, N, d, flags=flags)
        b = mg.Plan(B, M, N, d, flags=flags | EARLY_OFF)
        oa = [torch.empty((B, M, d), dtype=torch.float16, device="cuda") for _ in sets]
        ob = [torch.empty_like(x) for x in oa]
        for x, o in zip(sets, oa):
            a.run(*x, o)
        torch.cuda.synchronize()
        for x, o in zip(sets, ob):
            b.run(*x, o)
        torch.cuda.synchronize()
        assert all(torch.equal(x, y) for x, y in zip(oa, ob))


def test_host_buffer_entry_point_pageable_and_large():
    # Pageable host tensors take the copy-engine path; pinned ones the mapped-copy kernels. Both
    # on a shape with a split combine and several copy rounds per thread.
    q, k, v, _ = inputs.make_config("long_kv")
    ref = oracle.attention(q, k, v)
    B, M, N, d = 2, 256, 65536, 64
    plan = mg.Plan(B, M, N, d)
    for pinned in (False, True):
        hq, hk, hv = ((t.pin_memory() if pinned else t.clone()) for t in (q, k, v))
        ho = torch.full((B, M, d), float("nan"), dtype=torch.float16)
        ho = ho.pin_memory() if pinned else ho
        plan.run_host(hq, hk, hv, ho)
        torch.cuda.synchronize()
        assert_parity(ho, ref, f"run_host pinned={pinned}")


def test_misaligned_pointer_rejected():
    plan = mg.Plan(1, 128, 1024, 64)
    buf = torch.zeros(1 * 128 * 64 + 8, dtype=torch.float16, device="cuda")
    k = torch.zeros((1, 64, 1024), dtype=torch.float16, device="cuda")
    v = torch.zeros((1, 1024, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(mg.MgAttnError) as e:
        plan.run_ptr(buf.data_ptr() + 2, k.data_ptr(), v.data_ptr(), buf.data_ptr())
    assert e.value.status == mg.MG_ERR_LAYOUT


@pytest.mark.parametrize("flags", [0, mg.MG_FLAG_NO_CLUSTER])
def test_bounded_wait_with_early_start(flags):
    # Two calls back to back on distinct buffers, each with a wait that runs out after 2 ms: the
    # second starts early (its dependents released at its start, everything but its global writes
    # before its wait), so both unwind while overlapping; the status is written only after the
    # wait for the previous grid, and the context stays usable.
    q, k, v, _ = inputs.make_config("tiny")
    plan = mg.Plan(2, 64, 1024, 64, flags=mg.MG_FLAG_INJECT_TIMEOUT | flags, timeout_ns=2_000_000)
    assert plan.info["grid_ctas"] >= 10
    sets = [tuple(t.cuda() for t in (q, k, v)) for _ in range(2)]
    outs = [torch.zeros((2, 64, 64), dtype=torch.float16, device="cuda") for _ in range(2)]
    for x, o in zip(sets, outs):
        plan.run(*x, o)
    assert plan.status() == mg.MG_ERR_TIMEOUT
    O2, _ = run_gpu(q, k, v, flags=flags)
    assert_parity(O2, oracle.attention(q, k, v), "after timeouts")


@pytest.mark.parametrize("flags", [0, mg.MG_FLAG_PUSH_COMBINE, mg.MG_FLAG_NO_CLUSTER])
def test_bounded_wait_reports_timeout_and_context_survives(flags):
    # The load warp waits on a barrier nothing arrives on (before issuing any copy); the wait
    # runs out after 2 ms, every role unwinds (with each on-chip exchange form, and without one),
    # and the plan's sticky status says so.
    q, k, v, _ = inputs.make_config("tiny")
    plan = mg.Plan(2, 64, 1024, 64, flags=mg.MG_FLAG_INJECT_TIMEOUT | flags, timeout_ns=2_000_000)
    assert plan.info["xchg_push"] == (1 if flags == mg.MG_FLAG_PUSH_COMBINE else 0)
    Q, K, V = q.cuda(), k.cuda(), v.cuda()
    O = torch.zeros((2, 64, 64), dtype=torch.float16, device="cuda")
    plan.run(Q, K, V, O)
    assert plan.status() == mg.MG_ERR_TIMEOUT
    assert b"barrier" in _lib.load_library().mg_attn_last_error()
    # The context is still usable: a normal plan runs and matches the oracle.
    O2, _ = run_gpu(q, k, v)
    assert_parity(O2, oracle.attention(q, k, v), "after timeout")
