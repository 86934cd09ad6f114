"""The CPU oracle against its pins (closed forms, brute force, a library special case,
invariants), plus its own API behaviour. No GPU needed."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from attention_mugraph_gb300 import inputs
from tests import pins


def _fn(q, k, v):
    return oracle.attention(q, k, v, threads=2)


@pytest.mark.parametrize("pin", pins.PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(_fn)


def test_brute_force_itself_on_closed_form():
    # The brute force is a pin too: check it once against the K = 0 closed form.
    q, _, v = pins._rand_inputs(1, 2, 5, 3, seed=99)
    k = torch.zeros((1, 3, 5), dtype=torch.float16)
    want = v.double().numpy().mean(axis=1, keepdims=True).repeat(2, axis=1)
    np.testing.assert_allclose(pins.brute_force(q, k, v), want, rtol=1e-14, atol=1e-15)


def test_rows_match_full_bit_for_bit():
    q, k, v = pins._rand_inputs(2, 9, 70, 16, seed=7)
    full = oracle.attention(q, k, v)
    rows = [0, 5, 8, 9, 17, 3]
    sub = oracle.attention_rows(q, k, v, rows)
    assert np.array_equal(sub, full.reshape(-1, 16)[rows])


def test_thread_count_does_not_change_result():
    q, k, v = pins._rand_inputs(2, 33, 257, 64, seed=8)
    assert np.array_equal(oracle.attention(q, k, v, threads=1), oracle.attention(q, k, v, threads=4))


def test_bad_arguments_rejected():
    q, k, v = pins._rand_inputs(1, 2, 8, 4)
    with pytest.raises(ValueError):
        oracle.attention(q, k[:, :3], v)
    with pytest.raises(TypeError):
        oracle.attention(q.float(), k, v)
    with pytest.raises(RuntimeError):
        oracle.attention_rows(q, k, v, [2])  # row index out of range (B*M = 2)


def test_config_shapes_follow_the_printed_graph():
    # tests/golden/gqa_graph.json records the shapes the tutorial and the benchmark print.
    with open(os.path.join(pins.GOLDEN, "gqa_graph.json")) as f:
        g = json.load(f)
    B, M, N, d, _ = inputs.CONFIGS["gqa"]
    assert [B, M, d] == g["tutorial_shapes"]["Q"]
    assert [B, d, N] == g["tutorial_shapes"]["K"]
    assert [B, N, d] == g["tutorial_shapes"]["V"]
    B8, M8, N8, d8, _ = inputs.CONFIGS["gqa_b8"]
    assert (B8, M8, N8, d8) == (2 * 8, 256, 4096, 64)  # benchmark shapes at batch_size = 8
    q, k, v, shape = inputs.make_config("tiny")
    o = oracle.attention(q, k, v)
    assert o.shape == (shape[0], shape[1], shape[3])


def test_input_recipe_is_seeded_and_shaped():
    a = inputs.make_inputs(2, 3, 16, 8, 0.5, seed=0)
    b = inputs.make_inputs(2, 3, 16, 8, 0.5, seed=0)
    c = inputs.make_inputs(2, 3, 16, 8, 0.5, seed=1)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert not torch.equal(a[0], c[0])
    q, k, v = a
    assert q.shape == (2, 3, 8) and k.shape == (2, 8, 16) and v.shape == (2, 16, 8)
    assert q.dtype == k.dtype == v.dtype == torch.float16
    assert float(q.abs().max()) <= 0.5 and float(k.abs().max()) <= 0.5


@pytest.mark.parametrize("pin", pins.QK_PINS, ids=lambda p: p.__name__)
def test_qknorm_oracle_pin(pin):
    pin(lambda q, k, v, eps: oracle.attention_qknorm(q, k, v, eps=eps, threads=2))


def test_qknorm_rows_match_full():
    q, k, v = pins._rand_inputs(2, 7, 40, 16, seed=8)
    full = oracle.attention_qknorm(q, k, v)
    rows = [0, 6, 9, 13]
    assert np.array_equal(oracle.attention_qknorm(q, k, v, rows=rows), full.reshape(-1, 16)[rows])
