"""Allocating helpers over the C entry points (output tensors come from torch)."""
import math

import torch

from . import _binding as B


def rope_table(max_pos, head_dim, base=10000.0, device="cuda", stream=None):
    """[max_pos, head_dim] RoPE table (cos of the head_dim/2 pair angles, then their sin)."""
    t = torch.empty((max_pos, head_dim), device=device, dtype=torch.float32)
    B.attn_rope_table(t, max_pos, head_dim, base, stream)
    return t


def forward(q, k, v, num_heads, num_kv_heads, mask=B.ATTN_CAUSAL, prec=B.ATTN_FP32, want_lse=True,
            stream=None, window=0, rope=None):
    """q [q_seq, H*D], k/v [kv_seq, G*D] (CUDA fp32) -> (out [q_seq, H*D], lse [q_seq, H, 2] or None).
    window > 0 keeps each row's last `window` keys; rope (a table from rope_table) turns q and k
    by their row positions first."""
    q_seq, kv_seq = q.shape[0], k.shape[0]
    D = q.shape[1] // num_heads
    out = torch.empty_like(q)
    lse = torch.empty((q_seq, num_heads, 2), device=q.device, dtype=torch.float32) if want_lse else None
    if rope is not None:
        B.attn_forward_rope(q, k, v, out, lse, q_seq, kv_seq, num_heads, num_kv_heads, D, mask, prec, window, rope,
                            None, stream)
    elif window:
        B.attn_forward_window(q, k, v, out, lse, q_seq, kv_seq, num_heads, num_kv_heads, D, mask, prec, window,
                              stream)
    else:
        B.attn_forward(q, k, v, out, lse, q_seq, kv_seq, num_heads, num_kv_heads, D, mask, prec, stream)
    return out, lse


def backward(q, k, v, out, lse, dout, num_heads, num_kv_heads, mask=B.ATTN_CAUSAL, window=0, stream=None):
    """Gradients (dq, dk, dv) of forward(q, k, v, ...)'s out for upstream dout, given its out and lse."""
    q_seq, kv_seq = q.shape[0], k.shape[0]
    D = q.shape[1] // num_heads
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    B.attn_backward(q, k, v, out, dout, lse, dq, dk, dv, q_seq, kv_seq, num_heads, num_kv_heads, D, mask,
                    B.ATTN_FP32, window, stream)
    return dq, dk, dv


def prefill(q_batch, k_cache, v_cache, n_queries, n_heads, n_kv_heads, head_dim, start_pos, q_base=0,
            scale=None, out=None, prec=B.ATTN_FP32, stream=None, window=0):
    """Causal prefill of rows q_base .. q_base+n_queries-1 of q_batch (row stride = its width)."""
    max_seq, kv_dim = k_cache.shape
    if out is None:
        out = torch.zeros((q_batch.shape[0], n_heads * head_dim), device=q_batch.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    if window:
        B.attn_prefill_window(q_batch, k_cache, v_cache, out, n_queries, n_heads, n_kv_heads, head_dim, kv_dim,
                              max_seq, scale, start_pos, q_batch.shape[1], out.shape[1], q_base, prec, window, stream)
    else:
        B.attn_prefill(q_batch, k_cache, v_cache, out, n_queries, n_heads, n_kv_heads, head_dim, kv_dim, max_seq,
                       scale, start_pos, q_batch.shape[1], out.shape[1], q_base, prec, stream)
    return out


class DecodeState:
    """A decode workspace (zeroed once) and the device-resident kv_pos word."""

    def __init__(self, num_heads, num_kv_heads, head_dim, max_seq, device="cuda"):
        self.num_heads, self.num_kv_heads, self.head_dim, self.max_seq = num_heads, num_kv_heads, head_dim, max_seq
        nbytes = B.attn_decode_workspace_bytes(num_heads, num_kv_heads, head_dim, max_seq)
        if nbytes == 0:
            raise ValueError("unsupported decode sizes")
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.kv_pos = torch.zeros(1, dtype=torch.int32, device=device)

    def set_pos(self, kv_pos):
        self.kv_pos.fill_(int(kv_pos))


def decode(state, q, k_cache, v_cache, out=None, stream=None, window=0):
    """One decode step at the position held in state.kv_pos (over its last
    `window` positions when window > 0)."""
    if out is None:
        out = torch.empty_like(q)
    if window:
        B.attn_decode_cached_window(q, k_cache, v_cache, state.kv_pos, out, state.num_heads, state.num_kv_heads,
                                    state.head_dim, state.max_seq, state.workspace, None, window, stream)
    else:
        B.attn_decode_cached(q, k_cache, v_cache, state.kv_pos, out, state.num_heads, state.num_kv_heads,
                             state.head_dim, state.max_seq, state.workspace, None, stream)
    return out
