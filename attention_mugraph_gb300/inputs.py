"""Seeded synthetic inputs for the exp-normalised GQA attention graph.

This module is shared by the tests, the bench and the smoke check. It draws
random numbers and nothing else: none of the method's arithmetic lives here,
so the CPU oracle and the CUDA path can both consume its output without
sharing any code with each other.

Recipe (one ``torch.Generator('cpu')`` seeded with ``seed``; every draw in
fp32, in this order, then rounded to fp16 with round-to-nearest-even):

* ``Q`` of shape (B, M, d) ~ U(-a, a)
* ``K`` of shape (B, d, N) ~ U(-a, a)   (already transposed: d rows, N columns)
* ``V`` of shape (B, N, d) ~ N(0, 1)

The shapes follow the Mirage GQA tutorial graph (Q (2,256,64), K (2,64,4096),
V (2,4096,64), fp16) and the benchmark that scales its leading dimension by the
batch size (blog "Reading Mirage's muGraph search and backend generation
through the GQA example", section 1). The pages use no public dataset; these
synthetic draws are the whole workload.
"""

from __future__ import annotations

import torch

# name -> (B, M, N, d, a). "a" is the half-width of the uniform draw for Q and K.
CONFIGS = {
    # small case: M below one 128-row tile, 8 column tiles
    "tiny": (2, 64, 1024, 64, 0.5),
    # the tutorial graph exactly: batch 1, 2 kv heads, q_per_kv*head_dim = 256
    "gqa": (2, 256, 4096, 64, 0.5),
    # the benchmark's batch_size = 8
    "gqa_b8": (16, 256, 4096, 64, 0.5),
    # decode-like: 8 query rows against a 32768-long KV axis, head dim 128
    "decode": (16, 8, 32768, 128, 0.25),
    # long KV axis: row sums of 65536 terms
    "long_kv": (2, 256, 65536, 64, 0.5),
    # one query row per head, the shapes of the tutorial's launch example (Q (64,1,128),
    # K (64,128,4096), V (64,4096,128)); its values follow the decode-like recipe
    "decode_m1": (64, 1, 4096, 128, 0.25),
}

# Order matters: it mirrors the configuration list the bench and tests quote.
CONFIG_ORDER = ["tiny", "gqa", "gqa_b8", "decode", "long_kv", "decode_m1"]


def make_inputs(B: int, M: int, N: int, d: int, a: float = 0.5, seed: int = 0):
    """Draw (Q, K, V) as contiguous fp16 CPU tensors following the recipe above."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    q = torch.rand((B, M, d), generator=g, dtype=torch.float32) * (2.0 * a) - a
    k = torch.rand((B, d, N), generator=g, dtype=torch.float32) * (2.0 * a) - a
    v = torch.randn((B, N, d), generator=g, dtype=torch.float32)
    return q.half().contiguous(), k.half().contiguous(), v.half().contiguous()


def make_inputs_normal(B: int, M: int, N: int, d: int, seed: int = 0):
    """Q, K, V all ~ N(0, 1) in that order (fp32, then fp16): the draws of the tutorial's launch
    example (Mirage documentation, tutorials/group-query-attention, "Launch Mirage-Generated GQA
    Kernel"). With d = 128 its scores reach |A| ~ 45, past the fp16 range of exp(A)."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    q = torch.randn((B, M, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, d, N), generator=g, dtype=torch.float32)
    v = torch.randn((B, N, d), generator=g, dtype=torch.float32)
    return q.half().contiguous(), k.half().contiguous(), v.half().contiguous()


def make_config(name: str, seed: int = 0):
    """Inputs for one named workload: returns (Q, K, V, (B, M, N, d))."""
    B, M, N, d, a = CONFIGS[name]
    q, k, v = make_inputs(B, M, N, d, a, seed)
    return q, k, v, (B, M, N, d)
