"""The allocation-free entry point, mg_attn_run_noalloc, through the C ABI.

It serves callers that cannot call cudaMalloc (device memory handed to another allocator, a
latency path that cannot take cudaMalloc's implicit synchronisation, rules against allocating
after start-up): its split partials live in a fixed 8 MiB device array inside the library. These
checks compare it with the planned entry point (mg_attn_run) on the same inputs, on two calls in a
row (the array keeps the previous call's contents): bit for bit, since both run the same kernels
with the same split, and within the parity bound of the other GPU tests. One check runs in a fresh
child process whose first library call is mg_attn_run_noalloc, before any plan exists, so that the
first call's own set-up decides its path. A shape needing more scratch than the array holds is
refused. This file is collected last so that a failure here never hides the other tests; it also
passes alone in a fresh process.
"""

import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import attention_mugraph_gb300 as mg
from attention_mugraph_gb300 import _lib, build, inputs

pytestmark = pytest.mark.gpu

RTOL = 2e-3  # the parity bound the other GPU tests use: |err| <= RTOL * (1 + |ref|)
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return _lib.load_library()


def _call(lib, shape, Q, K, V, O, stream):
    B, M, N, d = shape
    return lib.mg_attn_run_noalloc(B, M, N, d, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                                   ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("name", ["gqa", "decode", "tiny", "decode_m1"])
def test_noalloc_matches_planned_entry_point_on_two_calls(lib, name):
    q, k, v, shape = inputs.make_config(name)
    B, M, N, d = shape
    Q, K, V = q.cuda(), k.cuda(), v.cuda()
    stream = torch.cuda.current_stream()

    plan = mg.Plan(B, M, N, d)
    ref = torch.empty((B, M, d), dtype=torch.float16, device="cuda")
    plan.run(Q, K, V, ref)
    torch.cuda.synchronize()
    want = ref.double().cpu().numpy()

    for call in range(2):
        O = torch.full((B, M, d), float("nan"), dtype=torch.float16, device="cuda")
        if call == 0:
            st = _call(lib, shape, Q, K, V, O, stream)
            assert st == mg.MG_OK, lib.mg_attn_last_error()
        else:
            mg.run_noalloc(Q, K, V, O)  # the Python binding of the same entry point
        torch.cuda.synchronize()
        got = O.double().cpu().numpy()
        assert np.isfinite(got).all(), f"{name} call {call}: non-finite output"
        err = np.abs(got - want)
        assert (err <= RTOL * (1 + np.abs(want))).all(), f"{name} call {call}: max err {err.max():.3e}"
        assert torch.equal(O, ref), f"{name} call {call}: not bit-identical to mg_attn_run"
    plan.destroy()


# Run in a child interpreter: the library's first call there is mg_attn_run_noalloc. The second
# shape's cluster plan needs no partials, while its second-kernel plan (64 splits) would need
# 8.45 MB, more than the array: a first call that misjudged the cluster would be refused.
_CHILD = r"""
import ctypes, json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from attention_mugraph_gb300 import _lib, build, inputs
import attention_mugraph_gb300 as mg
import oracle

build.build()
lib = _lib.load_library()
out = {}
for name, shape in (("gqa", (2, 256, 4096, 64)), ("d128_long", (2, 128, 8192, 128))):
    B, M, N, d = shape
    q, k, v = inputs.make_inputs(B, M, N, d, 0.5 if d == 64 else 0.25, seed=21)
    Q, K, V = q.cuda(), k.cuda(), v.cuda()
    s = torch.cuda.current_stream()
    got = []
    for call in range(2):
        O = torch.full((B, M, d), float("nan"), dtype=torch.float16, device="cuda")
        st = lib.mg_attn_run_noalloc(B, M, N, d, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                                     ctypes.c_void_p(s.cuda_stream))
        if st != 0:
            out[name] = {"status": st, "error": lib.mg_attn_last_error().decode()}
            break
        torch.cuda.synchronize()
        got.append(O.clone())
    else:
        plan = mg.Plan(B, M, N, d)
        ref = torch.empty((B, M, d), dtype=torch.float16, device="cuda")
        plan.run(Q, K, V, ref)
        torch.cuda.synchronize()
        want = oracle.attention(q, k, v)
        errs = [float(np.max(np.abs(g.double().cpu().numpy() - want) / (1 + np.abs(want)))) for g in got]
        out[name] = {"status": 0, "bit_equal": [bool(torch.equal(g, ref)) for g in got], "rel_err": errs,
                     "cluster_ctas": plan.info["cluster_ctas"], "n_split": plan.info["n_split"]}
        plan.destroy()
print(json.dumps(out))
"""


def test_noalloc_first_call_in_a_fresh_process(lib):
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    for name, got in res.items():
        assert got["status"] == mg.MG_OK, f"{name}: first noalloc call refused: {got.get('error')}"
        assert got["bit_equal"] == [True, True], f"{name}: noalloc calls differ from mg_attn_run: {got}"
        assert max(got["rel_err"]) <= RTOL, f"{name}: {got}"
    assert res["d128_long"]["cluster_ctas"] > 0


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    # d = 128 with 4 row tiles and a long N splits 38 ways and combines them with the second kernel:
    # 38 * 512 * 129 * 4 bytes of partials > 8 MiB.
    B, M, N, d = 4, 128, 16384, 128
    info = mg.mg_attn_query(B, M, N, d, num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    assert info["workspace_bytes"] > 8 << 20
    buf = torch.zeros(16, dtype=torch.float16, device="cuda")
    st = lib.mg_attn_run_noalloc(B, M, N, d, buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mg.MG_ERR_INVALID_ARG
    assert b"static scratch" in lib.mg_attn_last_error()
