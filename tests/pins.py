"""Checks that pin the CPU oracle to facts other than itself.

Each pin takes an implementation ``fn(Q, K, V) -> O`` (fp16 CPU tensors in,
float64 numpy array (B, M, d) out) and raises ``AssertionError`` when the
implementation disagrees with a closed form, a brute-force evaluation written
independently, a library special case, or an invariant of the graph
``O = (exp(Q.K) / rowsum(exp(Q.K))) . V`` (Mirage documentation,
tutorials/group-query-attention, "Define GQA Computation Graph").

They are chosen so that a plausible slip anywhere in the oracle (a wrong sign
on the exponent, a dropped normalisation or term, a transposed operand, a
wrong row/batch index, a stray 1/sqrt(d) scale) fails at least one of them;
``test_oracle_mutants.py`` plants such slips in a copy of the oracle and
checks exactly that.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand_inputs(B, M, N, d, a=0.5, seed=0):
    # Local draw (not the shared recipe) so pins do not depend on its details.
    g = torch.Generator("cpu").manual_seed(seed)
    q = (torch.rand((B, M, d), generator=g) * 2 * a - a).half()
    k = (torch.rand((B, d, N), generator=g) * 2 * a - a).half()
    v = torch.randn((B, N, d), generator=g).half()
    return q, k, v


def _close(got, want, rtol, atol, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = err > bound
    assert not bad.any(), (f"{what}: max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
                           f" (bound {bound.flat[err.argmax()]:.3e})")


# ---------------------------------------------------------------- closed forms

def pin_k_zero(fn):
    """K = 0 makes every score 0, every weight 1/N: O[b,m,:] is the mean of V[b] over N."""
    for (B, M, N, d) in [(2, 5, 37, 8), (1, 3, 130, 4)]:
        q, _, v = _rand_inputs(B, M, N, d, seed=1)
        k = torch.zeros((B, d, N), dtype=torch.float16)
        want = v.double().numpy().mean(axis=1, keepdims=True).repeat(M, axis=1)
        _close(fn(q, k, v), want, 1e-12, 1e-14, f"K=0 {B,M,N,d}")


def pin_q_zero(fn):
    """Q = 0 likewise gives the mean of V over N for every row."""
    B, M, N, d = 2, 4, 19, 6
    _, k, v = _rand_inputs(B, M, N, d, seed=2)
    q = torch.zeros((B, M, d), dtype=torch.float16)
    want = v.double().numpy().mean(axis=1, keepdims=True).repeat(M, axis=1)
    _close(fn(q, k, v), want, 1e-12, 1e-14, "Q=0")


def pin_v_constant(fn):
    """V = c everywhere: the weights sum to one, so O = c."""
    B, M, N, d = 2, 6, 23, 5
    q, k, _ = _rand_inputs(B, M, N, d, a=1.0, seed=3)
    v = torch.full((B, N, d), 0.75, dtype=torch.float16)
    _close(fn(q, k, v), np.full((B, M, d), 0.75), 1e-13, 0.0, "V=const")


def pin_single_key(fn):
    """M = N = 1: one weight, equal to one, so O = V[b, 0, :] exactly."""
    q, k, v = _rand_inputs(3, 1, 1, 7, a=2.0, seed=4)
    got = np.asarray(fn(q, k, v))
    want = v.double().numpy()
    assert np.array_equal(got, want), f"M=N=1: {got} != {want}"


def pin_one_hot(fn):
    """d = 1, Q[m] = t_m, K[n] = 1 at n* else 0: the score row is t_m at n* and 0 elsewhere, so
    O[m] = (e^t_m V[n*] + sum_{n != n*} V[n]) / (e^t_m + N - 1). Fails for exp(-s), shifted exps
    or any missing exponential."""
    ts = [0.5, -1.25, 2.0, 3.0, 0.0]
    N, nstar = 11, 4
    q = torch.tensor(ts, dtype=torch.float16).reshape(1, len(ts), 1)
    k = torch.zeros((1, 1, N), dtype=torch.float16)
    k[0, 0, nstar] = 1.0
    g = torch.Generator("cpu").manual_seed(5)
    v = torch.randn((1, N, 1), generator=g).half()
    vv = [float(x) for x in v.double().flatten()]
    rest = math.fsum(vv[n] for n in range(N) if n != nstar)
    want = np.array([(math.exp(t) * vv[nstar] + rest) / (math.exp(t) + N - 1) for t in ts])
    _close(fn(q, k, v), want.reshape(1, len(ts), 1), 1e-13, 1e-15, "one-hot")


def pin_golden_worked_examples(fn):
    """Hand-derived examples (tests/golden/worked_examples.json): exact fp16 inputs whose
    outputs have short closed forms, evaluated here with the math module."""
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    env = {"e": math.e, "exp": math.exp}
    for case in cases:
        q = torch.tensor(case["Q"], dtype=torch.float16)
        k = torch.tensor(case["K"], dtype=torch.float16)
        v = torch.tensor(case["V"], dtype=torch.float16)
        want = np.array([[[eval(expr, {"__builtins__": {}}, env) for expr in row]
                          for row in batch] for batch in case["O"]], dtype=np.float64)
        _close(fn(q, k, v), want, 1e-13, 1e-15, case["name"])


# ----------------------------------------------------------------- brute force

def brute_force(q, k, v):
    """Pure-Python evaluation of the definition, one output element at a time:
    O[b,m,c] = sum_n w_n V[b,n,c] / sum_n w_n, w_n = exp(sum_k Q[b,m,k] K[b,k,n]).
    Uses exactly rounded sums (math.fsum) so it is independent of summation order."""
    Q = q.double().tolist()
    K = k.double().tolist()
    V = v.double().tolist()
    B, M, d = len(Q), len(Q[0]), len(Q[0][0])
    N = len(K[0][0])
    out = np.zeros((B, M, d))
    for b in range(B):
        for m in range(M):
            w = [math.exp(math.fsum(Q[b][m][kk] * K[b][kk][n] for kk in range(d))) for n in range(N)]
            tot = math.fsum(w)
            for c in range(d):
                out[b, m, c] = math.fsum(w[n] * V[b][n][c] for n in range(N)) / tot
    return out


def pin_brute_force(fn):
    """Odd tiny shapes (B <= 2, M, N <= 17, d in {1, 2, 4}) against the pure-Python loop."""
    for i, (B, M, N, d) in enumerate([(1, 1, 3, 1), (2, 3, 5, 2), (2, 7, 17, 4), (1, 17, 9, 4),
                                      (2, 2, 16, 1)]):
        q, k, v = _rand_inputs(B, M, N, d, a=1.5, seed=10 + i)
        _close(fn(q, k, v), brute_force(q, k, v), 1e-12, 1e-14, f"brute {B,M,N,d}")


# -------------------------------------------------------- library special case

def pin_torch_softmax(fn):
    """Softmax is shift-invariant, so the graph equals torch.softmax(Q@K, -1) @ V (float64)."""
    for i, (B, M, N, d) in enumerate([(2, 64, 96, 64), (1, 9, 200, 128), (3, 5, 40, 16)]):
        q, k, v = _rand_inputs(B, M, N, d, seed=20 + i)
        want = (torch.softmax(q.double() @ k.double(), dim=-1) @ v.double()).numpy()
        _close(fn(q, k, v), want, 1e-11, 1e-13, f"softmax {B,M,N,d}")


# ------------------------------------------------------------------ invariants

def pin_joint_permutation(fn):
    """Reordering the N axis of K (columns) and V (rows) together leaves O unchanged."""
    B, M, N, d = 2, 6, 29, 8
    q, k, v = _rand_inputs(B, M, N, d, seed=30)
    perm = torch.randperm(N, generator=torch.Generator("cpu").manual_seed(31))
    _close(fn(q, k[:, :, perm].contiguous(), v[:, perm, :].contiguous()), fn(q, k, v),
           1e-12, 1e-14, "permutation")


def pin_convex_hull(fn):
    """Each O[b,m,:] is a convex combination of V[b] rows: within V's per-column min/max."""
    B, M, N, d = 3, 7, 33, 5
    q, k, v = _rand_inputs(B, M, N, d, a=2.0, seed=40)
    o = np.asarray(fn(q, k, v))
    vv = v.double().numpy()
    lo = vv.min(axis=1, keepdims=True) - 1e-14
    hi = vv.max(axis=1, keepdims=True) + 1e-14
    assert (o >= lo).all() and (o <= hi).all(), "O leaves the convex hull of V"


def pin_batch_independence(fn):
    """Batch b of a B=3 run equals a B=1 run on that slice, bit for bit."""
    B, M, N, d = 3, 5, 21, 6
    q, k, v = _rand_inputs(B, M, N, d, seed=50)
    full = np.asarray(fn(q, k, v))
    for b in range(B):
        one = np.asarray(fn(q[b:b + 1].contiguous(), k[b:b + 1].contiguous(), v[b:b + 1].contiguous()))
        assert np.array_equal(full[b:b + 1], one), f"batch {b} depends on other batches"


def pin_score_shift(fn):
    """With Q's last column set to one, adding c to K's last row adds c to every score of a row;
    the normalisation cancels it, so O is unchanged. K's last row is drawn on a 1/64 grid so that
    the shifted values stay exact in fp16."""
    B, M, N, d = 2, 4, 27, 6
    q, k, v = _rand_inputs(B, M, N, d, seed=60)
    q[:, :, -1] = 1.0
    g = torch.Generator("cpu").manual_seed(61)
    k[:, -1, :] = (torch.randint(-64, 65, (B, N), generator=g).float() / 64).half()
    k2 = k.clone()
    k2[:, -1, :] = (k[:, -1, :].float() + 1.5).half()
    assert torch.equal(k2[:, -1, :].float() - 1.5, k[:, -1, :].float())
    _close(fn(q, k2, v), fn(q, k, v), 1e-12, 1e-14, "score shift")


def pin_v_linearity(fn):
    """O is linear in V: doubling V (exact in fp16) doubles O exactly."""
    B, M, N, d = 1, 4, 15, 3
    q, k, v = _rand_inputs(B, M, N, d, seed=70)
    assert np.array_equal(np.asarray(fn(q, k, (v.float() * 2).half())), 2 * np.asarray(fn(q, k, v)))



# ---------------------------------------------------------------- the fp16 decode, every bit pattern

def _all_half_patterns():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)


def pin_half_decode_exhaustive(fn):
    # Every IEEE binary16 bit pattern (subnormals, both zeros, infinities, NaNs included) as V with
    # M = N = d = 1 and Q = K = 0: the weight is exp(0) / exp(0) = 1, so O = V exactly. numpy's
    # float16 -> float64 widening is the independent reference.
    v16 = _all_half_patterns()
    B = v16.size
    q = torch.zeros((B, 1, 1), dtype=torch.float16)
    k = torch.zeros((B, 1, 1), dtype=torch.float16)
    v = torch.from_numpy(v16.copy()).reshape(B, 1, 1)
    got = np.asarray(fn(q, k, v), dtype=np.float64).reshape(-1)
    want = v16.astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan), "NaN patterns must decode to NaN and nothing else"
    assert np.array_equal(got[~nan], want[~nan]), (
        f"{int((got[~nan] != want[~nan]).sum())} finite or infinite patterns decode wrongly")


def pin_half_decode_scores(fn):
    # The same decode on the score side: Q = x (or K = x) with d = 1, N = 2, K = [1, 0] (or Q = 1,
    # K = [x, 0]) and V = [1, 0] gives O = e^x / (e^x + 1), the logistic function of the decoded x.
    # Every finite pattern with |x| <= 30 (where the logistic still resolves x), subnormals included.
    x16 = _all_half_patterns()
    x64 = x16.astype(np.float64)
    keep = np.isfinite(x64) & (np.abs(x64) <= 30.0)
    x16, x64 = x16[keep], x64[keep]
    B = x16.size
    want = np.exp(x64) / (np.exp(x64) + 1.0)
    xs = torch.from_numpy(x16.copy())
    v = torch.zeros((B, 2, 1), dtype=torch.float16)
    v[:, 0, 0] = 1.0
    one = torch.ones((B, 1, 1), dtype=torch.float16)
    k_side = torch.zeros((B, 1, 2), dtype=torch.float16)
    k_side[:, 0, 0] = 1.0
    got_q = np.asarray(fn(xs.reshape(B, 1, 1), k_side, v), dtype=np.float64).reshape(-1)
    k_x = torch.zeros((B, 1, 2), dtype=torch.float16)
    k_x[:, 0, 0] = xs
    got_k = np.asarray(fn(one, k_x, v), dtype=np.float64).reshape(-1)
    _close(got_q, want, 1e-13, 0.0, "Q decode through the logistic")
    _close(got_k, want, 1e-13, 0.0, "K decode through the logistic")

PINS = [pin_k_zero, pin_q_zero, pin_v_constant, pin_single_key, pin_one_hot,
        pin_golden_worked_examples, pin_brute_force, pin_torch_softmax, pin_joint_permutation,
        pin_convex_hull, pin_batch_independence, pin_score_shift, pin_v_linearity,
        pin_half_decode_exhaustive, pin_half_decode_scores]


# ================================================================ QK-norm attention
# Pins for ``fn(Q, K, V, eps) -> O`` of the QK-norm graph (Mirage documentation,
# tutorials/attention-with-kv-norm): Q = rms_norm(Q), K = rms_norm(K), then the graph above,
# rms_norm over the head dimension d: x / sqrt(mean(x^2) + eps).

def qk_brute_force(q, k, v, eps):
    """Pure-Python evaluation, one element at a time, exactly rounded sums."""
    Q = q.double().tolist()
    K = k.double().tolist()
    V = v.double().tolist()
    B, M, d = len(Q), len(Q[0]), len(Q[0][0])
    N = len(K[0][0])
    out = np.zeros((B, M, d))
    for b in range(B):
        kn = [[0.0] * N for _ in range(d)]
        for n in range(N):
            r = 1.0 / math.sqrt(math.fsum(K[b][kk][n] ** 2 for kk in range(d)) / d + eps)
            for kk in range(d):
                kn[kk][n] = K[b][kk][n] * r
        for m in range(M):
            rq = 1.0 / math.sqrt(math.fsum(x * x for x in Q[b][m]) / d + eps)
            qn = [x * rq for x in Q[b][m]]
            w = [math.exp(math.fsum(qn[kk] * kn[kk][n] for kk in range(d))) for n in range(N)]
            tot = math.fsum(w)
            for c in range(d):
                out[b, m, c] = math.fsum(w[n] * V[b][n][c] for n in range(N)) / tot
    return out


def qk_pin_brute_force(fn):
    for i, (B, M, N, d) in enumerate([(1, 2, 5, 3), (2, 3, 7, 4), (1, 5, 16, 8)]):
        q, k, v = _rand_inputs(B, M, N, d, a=1.0, seed=80 + i)
        _close(fn(q, k, v, 1e-6), qk_brute_force(q, k, v, 1e-6), 1e-12, 1e-14, f"qk brute {B,M,N,d}")


def qk_pin_torch_rms_norm(fn):
    """torch.nn.functional.rms_norm over d (K transposed to put d last), then softmax in float64."""
    F = torch.nn.functional
    for i, (B, M, N, d) in enumerate([(2, 16, 64, 64), (1, 9, 130, 128)]):
        q, k, v = _rand_inputs(B, M, N, d, seed=90 + i)
        qn = F.rms_norm(q.double(), (d,), eps=1e-6)
        kn = F.rms_norm(k.double().transpose(1, 2), (d,), eps=1e-6).transpose(1, 2)
        want = (torch.softmax(qn @ kn, dim=-1) @ v.double()).numpy()
        _close(fn(q, k, v, 1e-6), want, 1e-11, 1e-13, f"qk torch {B,M,N,d}")


def qk_pin_key_scale(fn):
    """With eps = 0 a key vector's scale cancels in its normalisation: multiplying K[b,:,n*] by 4
    (exact in fp16) leaves O unchanged. Normalising K over N instead of d would not."""
    B, M, N, d = 2, 5, 13, 6
    q, k, v = _rand_inputs(B, M, N, d, seed=95)
    k2 = k.clone()
    k2[:, :, 7] = (k[:, :, 7].float() * 4).half()
    _close(fn(q, k2, v, 0.0), fn(q, k, v, 0.0), 1e-12, 1e-14, "key scale")


def qk_pin_query_scale(fn):
    """With eps = 0 scaling one query row by 8 leaves every output unchanged."""
    B, M, N, d = 2, 6, 11, 5
    q, k, v = _rand_inputs(B, M, N, d, seed=96)
    q2 = q.clone()
    q2[1, 3, :] = (q[1, 3, :].float() * 8).half()
    _close(fn(q2, k, v, 0.0), fn(q, k, v, 0.0), 1e-12, 1e-14, "query scale")


def qk_pin_d1_sign(fn):
    """d = 1 and eps = 0: rms_norm(x) = sign(x), so A = sign(q) sign(k_n) = +-1 and
    O = (e^{+-1} weighted mean of V) in closed form."""
    q = torch.tensor([[[0.75], [-2.0]]], dtype=torch.float16)
    k = torch.tensor([[[0.5, -0.25, 3.0, -1.0]]], dtype=torch.float16)
    g = torch.Generator("cpu").manual_seed(97)
    v = torch.randn((1, 4, 1), generator=g).half()
    vv = [float(x) for x in v.double().flatten()]
    sk = [1.0, -1.0, 1.0, -1.0]
    want = []
    for sq in (1.0, -1.0):
        w = [math.exp(sq * s) for s in sk]
        want.append(math.fsum(wi * x for wi, x in zip(w, vv)) / math.fsum(w))
    _close(fn(q, k, v, 0.0), np.array(want).reshape(1, 2, 1), 1e-13, 1e-15, "d=1 sign")


def qk_pin_zero_query_row(fn):
    """A zero query row with eps > 0 normalises to zero: every score 0, O = mean of V."""
    B, M, N, d = 1, 3, 9, 4
    q, k, v = _rand_inputs(B, M, N, d, seed=98)
    q[0, 1, :] = 0.0
    o = np.asarray(fn(q, k, v, 1e-6))
    _close(o[0, 1], v.double().numpy()[0].mean(axis=0), 1e-13, 1e-15, "zero query row")


QK_PINS = [qk_pin_brute_force, qk_pin_torch_rms_norm, qk_pin_key_scale, qk_pin_query_scale,
           qk_pin_d1_sign, qk_pin_zero_query_row]
