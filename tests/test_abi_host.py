"""Host-side checks of the C ABI that need no GPU: the library builds and loads, exports every
symbol include/mg_attn.h declares, its structs match the header's layout, the planner's
decisions and validation, and the product package's independence from the oracle."""

import ctypes
import os
import re
import subprocess

import pytest
import torch

import attention_mugraph_gb300 as mg
from attention_mugraph_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mg_attn.h")
DIAG_HEADER = os.path.join(ROOT, "include", "mg_diag.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load_library()


def declared_functions(header=HEADER, prefix="mg_attn_"):
    text = open(header).read()
    return sorted(set(re.findall(rf"^\s*(?:mg_status|const char \*|int32_t)\s*\*?\s*({prefix}\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    diag = declared_functions(DIAG_HEADER, "mg_diag_")
    assert len(names) >= 10 and len(diag) == 3
    assert sorted(_lib.EXPORTS) == names
    assert sorted(_lib.DIAG_EXPORTS) == diag
    names = names + diag
    for name in names:
        assert hasattr(lib, name), f"{name} not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    for name in names:
        assert re.search(rf"\bT {name}$", out, re.M), f"{name} is not a defined text symbol"


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "mg_attn.h"
int main(void) {
  printf("%zu %zu %zu\\n", sizeof(mg_attn_options), offsetof(mg_attn_options, timeout_ns), offsetof(mg_attn_options, flags));
  printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(mg_attn_plan_info), offsetof(mg_attn_plan_info, block_m),
         offsetof(mg_attn_plan_info, num_sms), offsetof(mg_attn_plan_info, workspace_bytes),
         offsetof(mg_attn_plan_info, cluster_ctas), offsetof(mg_attn_plan_info, schedule));
  printf("%zu\\n", offsetof(mg_attn_plan_info, xchg_push));
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    l1, l2, l3 = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")[:3]
    O, I = _lib.MgAttnOptions, _lib.MgAttnPlanInfo
    assert [int(x) for x in l1.split()] == [ctypes.sizeof(O), O.timeout_ns.offset, O.flags.offset]
    assert [int(x) for x in l2.split()] == [ctypes.sizeof(I), I.block_m.offset, I.num_sms.offset,
                                            I.workspace_bytes.offset, I.cluster_ctas.offset, I.schedule.offset]
    assert int(l3) == I.xchg_push.offset


def test_status_strings_and_version(lib):
    for s in range(0, 8):
        assert lib.mg_attn_status_string(s)
    assert b"unknown" in lib.mg_attn_status_string(99)
    assert lib.mg_attn_version() == 10000


def split_tiles(n_tiles, n_split):
    # The fused kernel's split j owns the column tiles j, j + n_split, j + 2 n_split, ...
    return [list(range(j, n_tiles, n_split)) for j in range(n_split)]


@pytest.mark.parametrize("B,M,N,d", [(2, 64, 1024, 64), (2, 256, 4096, 64), (16, 256, 4096, 64),
                                     (16, 8, 32768, 128), (2, 256, 65536, 64), (1, 1, 8, 64), (300, 256, 256, 64)])
def test_query_decisions(B, M, N, d):
    info = mg.mg_attn_query(B, M, N, d, num_sms=152)
    m_tiles = B * -(-M // 128)
    n_tiles = -(-N // 128)
    assert info["m_tiles"] == m_tiles and info["n_tiles"] == n_tiles
    assert 1 <= info["n_split"] <= n_tiles
    q = info["q_tiles_per_cta"]
    # Two Q tiles per CTA only where the two-tile kernel applies (d = 64, the graph as written, an
    # even number of row tiles per batch), and then only for throughput-bound shapes.
    assert q in (1, 2) and (q == 1 or (d == 64 and -(-M // 128) % 2 == 0))
    units = m_tiles // q
    if info["schedule"] == 1:  # stream-K: one CTA per SM (or per unit), n_split partial slots per row
        assert info["grid_ctas"] == min(152, m_tiles * n_tiles) and M <= 16
        return
    assert info["grid_ctas"] == units * info["n_split"]
    if units >= 152:
        assert info["n_split"] == 1
    else:
        assert info["grid_ctas"] <= 152  # one wave
    cluster = info["cluster_ctas"]
    assert cluster in (0, info["n_split"]) and cluster <= 16
    if 2 <= info["n_split"] <= 16:
        assert cluster == info["n_split"]  # small splits combine on chip (where the device fits the cluster)
    assert info["kernels_per_run"] == (2 if info["n_split"] > 1 and cluster == 0 else 1)
    assert info["smem_bytes"] <= 232448
    # Every column tile belongs to exactly one split, every split has one (n_split <= n_tiles),
    # and the splits' counts differ by at most one.
    own = split_tiles(n_tiles, info["n_split"])
    assert sorted(t for ts in own for t in ts) == list(range(n_tiles))
    counts = [len(ts) for ts in own]
    assert min(counts) >= 1 and max(counts) - min(counts) <= 1
    # Every split plan keeps its fp32 partials in the workspace (read by the cluster's CTAs through
    # L2, or by the second kernel); one split needs only the status words.
    # Split partials live in the workspace for the second kernel; the one-tile kernel's cluster
    # combine exchanges them on chip; one split needs only the status words.
    ws = 256 + (info["n_split"] * B * M * (d + 1) * 4 if info["n_split"] > 1 and cluster == 0 else 0)
    assert info["workspace_bytes"] == ws


def test_query_pair_choices():
    # The two-Q-tile kernel is opt-in: by default every workload takes the one-tile kernel.
    for shape in [(16, 256, 4096, 64), (2, 256, 65536, 64), (2, 256, 4096, 64), (16, 256, 4096, 128)]:
        assert mg.mg_attn_query(*shape, 152)["q_tiles_per_cta"] == 1
    lkv = mg.mg_attn_query(2, 256, 65536, 64, 152, flags=mg.MG_FLAG_Q_PAIRS)
    assert lkv["q_tiles_per_cta"] == 2 and lkv["n_split"] == 76 and lkv["grid_ctas"] == 152
    assert mg.mg_attn_query(16, 256, 4096, 128, 152, flags=mg.MG_FLAG_Q_PAIRS)["q_tiles_per_cta"] == 1
    # Flags force either kernel; variants and odd row-tile counts keep the one-tile kernel.
    assert mg.mg_attn_query(2, 256, 4096, 64, 152, flags=mg.MG_FLAG_Q_PAIRS)["q_tiles_per_cta"] == 2
    assert mg.mg_attn_query(16, 256, 4096, 64, 152, flags=mg.MG_FLAG_NO_Q_PAIRS)["q_tiles_per_cta"] == 1
    assert mg.mg_attn_query(16, 256, 4096, 64, 152, flags=mg.MG_FLAG_SAFE_SOFTMAX)["q_tiles_per_cta"] == 1
    assert mg.mg_attn_query(16, 384, 4096, 64, 152, flags=mg.MG_FLAG_Q_PAIRS)["q_tiles_per_cta"] == 1
    with pytest.raises(mg.MgAttnError):
        mg.mg_attn_query(2, 256, 4096, 64, 152, flags=mg.MG_FLAG_Q_PAIRS | mg.MG_FLAG_NO_Q_PAIRS)


def test_query_split_fills_its_tiles_when_hbm_bound():
    # Few query rows (HBM-bound): among split counts down to 4/5 of one wave, the plan takes the one
    # that leaves the fewest idle tile slots. Decode-like (16, 8, 32768, 128): 16 row tiles, one wave
    # is 9 splits (28 or 29 of 256 tiles each); 8 splits give every CTA 32.
    info = mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_NO_STREAM_K)
    assert info["n_split"] == 8 and info["grid_ctas"] == 128
    # A shape whose one-wave split already divides its tiles evenly keeps it.
    assert mg.mg_attn_query(64, 1, 4096, 128, 152, flags=mg.MG_FLAG_NO_STREAM_K)["n_split"] == 2
    # Many query rows per batch: every SM is used (one wave, 38 splits of 13 or 14 tiles).
    assert mg.mg_attn_query(2, 256, 65536, 64, 152)["n_split"] == 38


def _sk_slots(rows, n_tiles, G):
    # Restated from the schedule's definition: CTA c takes units [c U / G, (c+1) U / G).
    U = rows * n_tiles
    owner = [0] * U
    for c in range(G):
        for u in range(c * U // G, (c + 1) * U // G):
            owner[u] = c
    return max(owner[(r + 1) * n_tiles - 1] - owner[r * n_tiles] + 1 for r in range(rows))


@pytest.mark.parametrize("B,M,N,d", [(16, 8, 32768, 128), (64, 1, 4096, 128), (20, 5, 3000, 64), (37, 16, 1032, 64)])
def test_query_stream_k(B, M, N, d):
    info = mg.mg_attn_query(B, M, N, d, 152, flags=mg.MG_FLAG_STREAM_K)
    n_tiles = -(-N // 128)
    U = B * n_tiles
    G = min(U, 152)
    assert info["schedule"] == 1 and info["grid_ctas"] == G and info["cluster_ctas"] == 0
    assert info["kernels_per_run"] == 2 and info["n_split"] == _sk_slots(B, n_tiles, G)
    assert info["workspace_bytes"] == 256 + info["n_split"] * B * M * (d + 1) * 4
    assert -(-U // G) <= n_tiles  # a run touches at most two batches


def test_query_stream_k_choices():
    # Opt-in: the default plans keep the split schedule.
    assert mg.mg_attn_query(16, 8, 32768, 128, 152)["schedule"] == 0
    assert mg.mg_attn_query(64, 1, 4096, 128, 152)["schedule"] == 0
    assert mg.mg_attn_query(64, 1, 4096, 128, 152, flags=mg.MG_FLAG_STREAM_K)["schedule"] == 1
    # Not where it does not apply: more than 16 rows per batch, the variants, an explicit split.
    assert mg.mg_attn_query(2, 256, 4096, 64, 152, flags=mg.MG_FLAG_STREAM_K)["schedule"] == 0
    assert mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_SAFE_SOFTMAX)["schedule"] == 0
    assert mg.mg_attn_query(16, 8, 32768, 128, 152, n_split=8)["schedule"] == 0
    assert mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_NO_STREAM_K)["schedule"] == 0
    # Where the runs would exceed one batch's tiles (more batches than SMs), it does not apply.
    assert mg.mg_attn_query(5, 16, 40000, 64, 152, flags=mg.MG_FLAG_STREAM_K)["schedule"] == 1
    assert mg.mg_attn_query(400, 4, 1024, 64, 152, flags=mg.MG_FLAG_STREAM_K)["schedule"] == 0
    with pytest.raises(mg.MgAttnError):
        mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_STREAM_K | mg.MG_FLAG_NO_STREAM_K)


def test_query_swap_ab():
    info = mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_SWAP_AB)
    assert info["swap_ab"] == 1 and info["schedule"] == 0
    # Its split partials combine on chip like the one-tile kernel's (the query cannot see whether
    # the device fits the cluster; a plan falls back to the second kernel when it does not).
    assert info["cluster_ctas"] == info["n_split"] == 8 and info["kernels_per_run"] == 1
    k2 = mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_NO_CLUSTER)
    assert k2["swap_ab"] == 1 and k2["cluster_ctas"] == 0 and k2["kernels_per_run"] == 2
    assert k2["workspace_bytes"] == 256 + 8 * 16 * 8 * (128 + 1) * 4 and info["workspace_bytes"] == 256
    assert info["smem_bytes"] < mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_NO_SWAP_AB)["smem_bytes"]
    # The default where it applies: head dim 128, at most 16 rows, the graph as written.
    assert mg.mg_attn_query(16, 8, 32768, 128, 152)["swap_ab"] == 1
    assert mg.mg_attn_query(64, 1, 4096, 128, 152)["swap_ab"] == 1
    assert mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_NO_SWAP_AB)["swap_ab"] == 0
    assert mg.mg_attn_query(16, 8, 32768, 64, 152, flags=mg.MG_FLAG_SWAP_AB)["swap_ab"] == 0
    assert mg.mg_attn_query(16, 17, 32768, 128, 152, flags=mg.MG_FLAG_SWAP_AB)["swap_ab"] == 0
    # The max-subtracted evaluation and QK-norm run there in one pass (running maxima exchanged
    # between warps, the query scales: 1152 more bytes of shared memory).
    safe = mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_SAFE_SOFTMAX)
    assert safe["swap_ab"] == 1 and safe["smem_bytes"] == info["smem_bytes"] + 1152
    assert safe["cluster_ctas"] == 8 and safe["workspace_bytes"] == 256
    k2s = mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_SAFE_SOFTMAX | mg.MG_FLAG_NO_CLUSTER)
    assert k2s["swap_ab"] == 1 and k2s["workspace_bytes"] == 256 + 8 * 16 * 8 * (128 + 2) * 4
    qk = mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_QK_NORM)
    assert qk["swap_ab"] == 1 and qk["smem_bytes"] == safe["smem_bytes"]
    with pytest.raises(mg.MgAttnError):
        mg.mg_attn_query(16, 8, 32768, 128, 152, flags=mg.MG_FLAG_SWAP_AB | mg.MG_FLAG_NO_SWAP_AB)


def test_query_cluster_choices():
    # The GQA tutorial shape takes a 16-CTA cluster (2 column tiles per CTA) instead of 32 splits.
    assert mg.mg_attn_query(2, 256, 4096, 64, 152)["cluster_ctas"] == 16
    # A long KV axis keeps one wave of splits and the second kernel.
    lkv = mg.mg_attn_query(2, 256, 65536, 64, 152)
    assert lkv["n_split"] == 38 and lkv["cluster_ctas"] == 0 and lkv["kernels_per_run"] == 2
    # The flag forces the second kernel.
    nc = mg.mg_attn_query(2, 256, 4096, 64, 152, flags=mg.MG_FLAG_NO_CLUSTER)
    assert nc["cluster_ctas"] == 0 and nc["n_split"] == 32 and nc["kernels_per_run"] == 2


def test_query_safe_softmax_workspace():
    # The max-subtracted variant adds one fp32 row maximum per split and row to the partials of
    # the second kernel; the on-chip combine and single-split plans need no extra memory.
    B, M, N, d = 2, 256, 65536, 64
    plain = mg.mg_attn_query(B, M, N, d, 152)
    safe = mg.mg_attn_query(B, M, N, d, 152, flags=mg.MG_FLAG_SAFE_SOFTMAX)
    n = safe["n_split"]
    assert n == plain["n_split"] and safe["kernels_per_run"] == 2
    assert safe["workspace_bytes"] == 256 + n * B * M * (d + 2) * 4
    assert safe["workspace_bytes"] - plain["workspace_bytes"] == n * B * M * 4
    for shape in [(2, 256, 4096, 64), (16, 8, 32768, 128)]:
        for kw in [{}, {"n_split": 1}]:
            a = mg.mg_attn_query(*shape, 152, **kw)
            b = mg.mg_attn_query(*shape, 152, flags=mg.MG_FLAG_SAFE_SOFTMAX, **kw)
            if a["kernels_per_run"] == 1:
                assert b["workspace_bytes"] == a["workspace_bytes"] == 256


def test_query_qk_norm_plan():
    # QK-norm computes its scales inside the fused kernel (no extra launch). The workspace has
    # room for the key scales (B*N of them and 128 spare floats); as QK-norm implies the
    # max-subtracted evaluation, also one row maximum per split and row. Where they fit beside the
    # ring, the CTA's key scales stay in shared memory instead (128 floats per column tile of the
    # CTA), so that nothing global is written before the epilogue. Stages are unchanged.
    plain = mg.mg_attn_query(2, 256, 4096, 64, 152)
    qk = mg.mg_attn_query(2, 256, 4096, 64, 152, flags=mg.MG_FLAG_QK_NORM)
    tiles = -(-qk["n_tiles"] // qk["n_split"])
    assert qk["smem_bytes"] == plain["smem_bytes"] + tiles * 128 * 4 and qk["stages"] == 6
    assert qk["kernels_per_run"] == plain["kernels_per_run"]
    assert qk["workspace_bytes"] == plain["workspace_bytes"] + 256 + (2 * 4096 + 128) * 4
    # Head dim 128, three stages: no room beside the ring; the scales go through global memory.
    qk128 = mg.mg_attn_query(2, 256, 4096, 128, 152, flags=mg.MG_FLAG_QK_NORM)
    assert qk128["stages"] == 3
    assert qk128["smem_bytes"] == mg.mg_attn_query(2, 256, 4096, 128, 152)["smem_bytes"]
    # 64 column tiles per CTA do not fit either (32 KB of scales).
    one = mg.mg_attn_query(1, 128, 8192, 64, 152, n_split=1, flags=mg.MG_FLAG_QK_NORM)
    assert one["smem_bytes"] == mg.mg_attn_query(1, 128, 8192, 64, 152, n_split=1)["smem_bytes"]
    B, M, N, d = 2, 256, 65536, 64
    a = mg.mg_attn_query(B, M, N, d, 152, flags=mg.MG_FLAG_QK_NORM)
    b = mg.mg_attn_query(B, M, N, d, 152, flags=mg.MG_FLAG_SAFE_SOFTMAX)
    assert a["workspace_bytes"] == b["workspace_bytes"] + 256 + (B * N + 128) * 4
    assert b["workspace_bytes"] == 256 + b["n_split"] * B * M * (d + 2) * 4


def test_query_options():
    info = mg.mg_attn_query(2, 256, 4096, 64, 152, n_split=5, stages=2)
    assert info["n_split"] == 5 and info["stages"] == 2
    assert mg.mg_attn_query(2, 256, 4096, 128, 152)["stages"] == 3
    assert mg.mg_attn_query(2, 256, 4096, 64, 152)["stages"] == 6


def fwd_smem(d, stages, push):
    # Restated from the kernel's layout: alignment slack, Q, the ring, the pushed combine's receive
    # area (144 rows of x, remainders and kLmw floats), the row-sum exchange, the barrier area.
    lmw = 4 if d == 64 else 8
    recv = 144 * (2 * (d + 8) * 2 + lmw * 4) if push else 0
    return 1024 + 128 * d * 2 + stages * 2 * d * 128 * 2 + recv + 2 * 128 * 4 + 512


def test_query_push_combine():
    # On request, the graph as written at head dim 64 with an on-chip combine pushes each owner's
    # rows into its receive area, which takes the place of one K/V stage; everything else pulls.
    P = mg.MG_FLAG_PUSH_COMBINE
    for shape in [(2, 256, 4096, 64), (2, 64, 1024, 64), (16, 256, 4096, 64), (1, 128, 2048, 64)]:
        info = mg.mg_attn_query(*shape, 152, flags=P)
        assert info["cluster_ctas"] > 0 and info["xchg_push"] == 1 and info["stages"] == 5
        assert info["smem_bytes"] == fwd_smem(64, 5, True) <= 232448
        pull = mg.mg_attn_query(*shape, 152)
        assert pull["xchg_push"] == 0 and pull["stages"] == 6 and pull["smem_bytes"] == fwd_smem(64, 6, False)
        assert pull["n_split"] == info["n_split"] and pull["cluster_ctas"] == info["cluster_ctas"]
    q = dict(num_sms=152)
    assert mg.mg_attn_query(2, 256, 4096, 64, stages=6, flags=P, **q)["xchg_push"] == 0  # no room at this depth
    assert mg.mg_attn_query(2, 256, 4096, 64, stages=3, flags=P, **q)["xchg_push"] == 1
    assert mg.mg_attn_query(2, 256, 4096, 64, stages=3, flags=P, **q)["stages"] == 3
    for flags in (mg.MG_FLAG_SAFE_SOFTMAX, mg.MG_FLAG_QK_NORM, mg.MG_FLAG_NO_CLUSTER, mg.MG_FLAG_Q_PAIRS):
        assert mg.mg_attn_query(2, 256, 4096, 64, flags=flags | P, **q)["xchg_push"] == 0
    assert mg.mg_attn_query(2, 256, 4096, 128, flags=P, **q)["xchg_push"] == 0            # d = 128: no room
    assert mg.mg_attn_query(2, 256, 65536, 64, flags=P, **q)["xchg_push"] == 0            # second kernel
    assert mg.mg_attn_query(2, 256, 4096, 64, n_split=1, flags=P, **q)["xchg_push"] == 0  # nothing to combine


@pytest.mark.parametrize("args,kw,code", [
    ((0, 256, 4096, 64), {}, mg.MG_ERR_INVALID_ARG),
    ((2, -1, 4096, 64), {}, mg.MG_ERR_INVALID_ARG),
    ((2, 256, 4096, 32), {}, mg.MG_ERR_UNSUPPORTED),
    ((2, 256, 4100, 64), {}, mg.MG_ERR_LAYOUT),
    ((2, 256, 4096, 64), {"n_split": 33}, mg.MG_ERR_CONFIG),
    ((2, 256, 4096, 64), {"stages": 7}, mg.MG_ERR_CONFIG),
    ((2, 256, 4096, 64), {"flags": 0x4000}, mg.MG_ERR_CONFIG),
    ((2, 256, 4096, 64), {"flags": 0x8000}, mg.MG_ERR_CONFIG),
    ((2, 256, 4096, 64), {"flags": 0x10000}, mg.MG_ERR_CONFIG),
    ((2, 256, 4096, 64), {"timeout_ns": 5}, mg.MG_ERR_CONFIG),
    ((2, 256, 4096, 128), {"stages": 4}, mg.MG_ERR_INSUFFICIENT_SMEM),
    ((2, 256, 4096, 64), {"max_smem_optin": 100000}, mg.MG_ERR_INSUFFICIENT_SMEM),
    ((2, 1 << 31, 4096, 64), {}, mg.MG_ERR_INVALID_ARG),
])
def test_query_rejects(args, kw, code):
    with pytest.raises(mg.MgAttnError) as e:
        mg.mg_attn_query(*args, num_sms=152, **kw)
    assert e.value.status == code


def test_null_arguments_rejected_without_gpu(lib):
    assert lib.mg_attn_run(None, None, None, None, None, None) == mg.MG_ERR_INVALID_ARG
    assert lib.mg_attn_run_host(None, None, None, None, None, None) == mg.MG_ERR_INVALID_ARG
    assert lib.mg_attn_destroy(None) == mg.MG_ERR_INVALID_ARG
    assert lib.mg_attn_get_status(None) == mg.MG_ERR_INVALID_ARG
    assert lib.mg_attn_plan(2, 256, 4096, 64, None) == mg.MG_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_plan_without_device_fails_cleanly(lib):
    h = ctypes.c_void_p()
    st = lib.mg_attn_plan(2, 256, 4096, 64, ctypes.byref(h))
    assert st == mg.MG_ERR_CUDA and not h.value
    assert lib.mg_attn_last_error()


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "attention_mugraph_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "mg_oracle" not in text and "libmgoracle" not in text, f


@pytest.mark.parametrize("args", [(0, 1, 215296, 1, 10), (64, 3, 215296, 1, 10), (64, 17, 215296, 1, 10),
                                  (64, 16, 215296, 1, 0), (64, 16, 215296, 1, 100001)])
def test_diag_launch_floor_rejects_bad_arguments_before_any_cuda_call(lib, args):
    out = ctypes.c_float(-1.0)
    assert lib.mg_diag_launch_floor(*args, ctypes.byref(out)) == mg.MG_ERR_INVALID_ARG
    assert out.value == -1.0 and lib.mg_diag_last_error()
    assert lib.mg_diag_launch_floor(64, 16, 215296, 1, 10, None) == mg.MG_ERR_INVALID_ARG


def test_diag_exp_rate_rejects_bad_arguments_before_any_cuda_call(lib):
    a, b = ctypes.c_double(), ctypes.c_double()
    assert lib.mg_diag_exp_rate(0, 0, ctypes.byref(a), ctypes.byref(b)) == mg.MG_ERR_INVALID_ARG
    assert lib.mg_diag_exp_rate(1000001, 1, ctypes.byref(a), ctypes.byref(b)) == mg.MG_ERR_INVALID_ARG
    assert lib.mg_diag_exp_rate(10, 0, None, ctypes.byref(b)) == mg.MG_ERR_INVALID_ARG
