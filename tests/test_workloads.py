"""The seeded input recipe (no GPU needed): the workloads' sizes and length mixes are
the ones the design notes and the bench lines state, and the generators are
deterministic, so every test, the bench and the oracle see the same inputs."""
import numpy as np
import torch

from paged_kv_cache_166_gb300 import workloads as W


def test_length_mixes_as_stated():
    want = {  # sequences, total tokens, shortest, longest, bounds of the recipe
        "tiny": (4, 158, 1, 100, (1, 100)),
        "mha13b": (64, 24_860, 20, 2048, (1, 2048)),
        "gqa70b": (256, 451_896, 55, 8192, (1, 8192)),
        "longctx": (8, 854_921, 40_714, 128_737, (32_768, 131_072)),
    }
    for name, (n, total, lo, hi, (blo, bhi)) in want.items():
        lens = W.context_lengths(W.WORKLOADS[name])
        got = (len(lens), int(lens.sum()), int(lens.min()), int(lens.max()))
        assert got == (n, total, lo, hi), name
        assert blo <= lens.min() and lens.max() <= bhi, name
    assert list(W.context_lengths(W.WORKLOADS["tiny"])) == [1, 17, 40, 100]
    suf = W.suffix_lengths(W.WORKLOADS["prefix"])
    assert (len(suf), int(suf.sum()), int(suf.min()), int(suf.max())) == (256, 66_972, 2, 512)


def test_shapes_as_stated():
    shapes = {name: (w.num_q_heads, w.num_kv_heads, w.head_dim, w.dtype, w.block_size)
              for name, w in W.WORKLOADS.items()}
    assert shapes["mha13b"] == (40, 40, 128, "f16", 16)
    assert shapes["gqa70b"] == (64, 8, 128, "bf16", 16)
    assert shapes["longctx"] == (64, 8, 128, "bf16", 16)
    assert shapes["prefix"] == (32, 8, 128, "bf16", 16)
    assert shapes["tiny"] == (4, 4, 64, "f32", 16)


def test_generators_are_deterministic_and_streams_independent():
    a = W.normal_tensor((3, 4, 64), "bf16", 7, W.STREAM_Q)
    b = W.normal_tensor((3, 4, 64), "bf16", 7, W.STREAM_Q)
    c = W.normal_tensor((3, 4, 64), "bf16", 7, W.STREAM_K_NEW)
    d = W.normal_tensor((3, 4, 64), "bf16", 8, W.STREAM_Q)
    assert torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, d)
    assert a.dtype == torch.bfloat16
    x = W.normal_tensor((4096,), "f32", 1, W.STREAM_K_POOL).double()
    assert abs(float(x.mean())) < 0.1 and abs(float(x.std()) - 1) < 0.1   # N(0, 1) draws
    n = 97
    order = W.pool_order(n, 3)
    assert sorted(order.tolist()) == list(range(n))              # a permutation of the pool
    assert np.array_equal(order, W.pool_order(n, 3))
    assert not np.array_equal(order, np.arange(n))               # ids handed out scattered
