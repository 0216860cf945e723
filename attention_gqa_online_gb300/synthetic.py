"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers; it holds none of the attention
arithmetic.  Every tensor is fp32 on the CPU, drawn from one
``torch.Generator`` seeded per workload, in the order Q, K, V.

Distributions follow the workloads the library is measured on:
  * ``normal``  -- i.i.d. N(0, sigma^2) (sigma = 1 unless stated)
  * ``uniform`` -- i.i.d. U(-1, 1)
"""
import torch


def _draw(gen, shape, dist, sigma=1.0):
    if dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        return x * sigma if sigma != 1.0 else x
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    raise ValueError("unknown distribution " + dist)


def forward_inputs(q_seq, kv_seq, H, G, D, seed=0, qk_sigma=1.0, v_dist="normal"):
    """Q [q_seq, H*D], K and V [kv_seq, G*D]."""
    gen = torch.Generator().manual_seed(seed)
    q = _draw(gen, (q_seq, H * D), "normal", qk_sigma)
    k = _draw(gen, (kv_seq, G * D), "normal", qk_sigma)
    v = _draw(gen, (kv_seq, G * D), v_dist)
    return q, k, v


def decode_inputs(max_seq, H, G, D, seed=0):
    """Q [1, H*D], K and V caches [max_seq, G*D]."""
    gen = torch.Generator().manual_seed(seed)
    q = _draw(gen, (1, H * D), "normal")
    k = _draw(gen, (max_seq, G * D), "normal")
    v = _draw(gen, (max_seq, G * D), "normal")
    return q, k, v


def prefill_inputs(q_rows, q_stride, max_seq, kv_dim, seed=0):
    """Q batch [q_rows, q_stride], K and V caches [max_seq, kv_dim]."""
    gen = torch.Generator().manual_seed(seed)
    q = _draw(gen, (q_rows, q_stride), "normal")
    k = _draw(gen, (max_seq, kv_dim), "normal")
    v = _draw(gen, (max_seq, kv_dim), "normal")
    return q, k, v
