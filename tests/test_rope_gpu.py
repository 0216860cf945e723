"""RoPE-fused forward (attn_forward_rope) and its table (attn_rope_table) on the
GPU against the fp64 oracle, which turns q and k in fp64 itself (no table)."""
import math

import numpy as np
import pytest
import torch

from attention_gqa_online_gb300 import synthetic
from helpers import BF16, FP32, TF32, assert_lse_close, assert_out_close, dev, tc_supported

pytestmark = pytest.mark.gpu
CAUSAL, FULL, CROSS = 0, 1, 2
PRECS = [FP32, TF32, BF16]


def table(A, rows, D, base):
    t = torch.empty((rows, D), device="cuda")
    A.attn_rope_table(t, rows, D, base)
    return t


def test_table_values(cuda_lib):
    """Each entry within fp32 rounding (6e-8) of cos / sin of p * base^(-2d/D) in fp64."""
    rows, D, base = 16384, 128, 10000.0
    t = table(cuda_lib, rows, D, base).cpu().numpy().astype(np.float64)
    p = np.arange(rows, dtype=np.float64)[:, None]
    ang = p * base ** (-2.0 * np.arange(D // 2, dtype=np.float64) / D)
    assert np.abs(t[:, :D // 2] - np.cos(ang)).max() < 1.2e-7
    assert np.abs(t[:, D // 2:] - np.sin(ang)).max() < 1.2e-7


def check(A, orc, q_seq, kv_seq, H, G, D, mask, prec, seed, window=0, base=10000.0, rows=None, **kw):
    q, k, v = synthetic.forward_inputs(q_seq, kv_seq, H, G, D, seed=seed, **kw)
    tab = table(A, max(q_seq, kv_seq), D, base)
    out = torch.full((q_seq, H * D), float("nan"), device="cuda")
    lse = torch.full((q_seq, H, 2), float("nan"), device="cuda")
    A.attn_forward_rope(dev(q), dev(k), dev(v), out, lse, q_seq, kv_seq, H, G, D, mask, prec, window, tab)
    torch.cuda.synchronize()
    assert A.attn_get_status() == 0
    ro, rl = orc.forward_rope(q.numpy(), k.numpy(), v.numpy(), q_seq, kv_seq, H, G, D, mask, base, rows=rows,
                              window=window)
    sel = slice(None) if rows is None else np.asarray(rows)
    got, gl = out.cpu().numpy()[sel], lse.cpu().numpy()[sel]
    where = "rope q%d kv%d H%d G%d D%d mask%d prec%d window%d" % (q_seq, kv_seq, H, G, D, mask, prec, window)
    assert_out_close(got, ro[sel], prec, float(v.abs().max()), where)
    assert_lse_close(gl, rl[sel], prec, float(np.abs(rl[sel][..., 0]).max()), where)


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("mask,kv", [(CAUSAL, 300), (FULL, 300), (CROSS, 421)])
def test_rope_forward(cuda_lib, orc, prec, mask, kv):
    """300 queries, 8 heads over 2 kv heads, D=64."""
    check(cuda_lib, orc, 300, kv, 8, 2, 64, mask, prec, seed=40 + mask)


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("q_seq,kv_seq,H,G,D,mask,window,base", [
    (67, 67, 6, 2, 80, CAUSAL, 0, 10000.0),    # gs = 3 (fp32 only)
    (130, 130, 16, 2, 128, CAUSAL, 0, 10000.0),  # gs = 8
    (45, 131, 8, 8, 64, CROSS, 0, 500.0),       # MHA, other base
    (200, 200, 4, 2, 128, CAUSAL, 77, 10000.0),  # sliding window
    (1, 1, 4, 2, 64, CAUSAL, 0, 10000.0),
    (100, 100, 6, 2, 128, CAUSAL, 0, 10000.0),  # gs = 3 on the tensor cores
])
def test_rope_shapes(cuda_lib, orc, prec, q_seq, kv_seq, H, G, D, mask, window, base):
    if prec != FP32 and not tc_supported(H, G, D):
        pytest.skip("tensor-core precisions need D in {64, 128}")
    check(cuda_lib, orc, q_seq, kv_seq, H, G, D, mask, prec, seed=q_seq + D, window=window, base=base)


@pytest.mark.parametrize("prec,qk_sigma", [(FP32, 3.0), (TF32, 3.0), (BF16, 3.0)])
def test_rope_long_causal(cuda_lib, orc, prec, qk_sigma):
    """q_seq 8193, 32 heads over 8 kv heads, D=128: sampled rows up to position 8192."""
    rng = np.random.default_rng(3)
    rows = sorted(set(range(4)) | set(range(8189, 8193)) | set(rng.integers(0, 8193, 12).tolist()))
    check(cuda_lib, orc, 8193, 8193, 32, 8, 128, CAUSAL, prec, seed=6, rows=rows, qk_sigma=qk_sigma)


def test_rope_rejects(cuda_lib):
    q, k, v = synthetic.forward_inputs(8, 8, 2, 1, 12, seed=1)
    tab = table(cuda_lib, 8, 12, 10000.0)
    out = torch.empty((8, 24), device="cuda")
    with pytest.raises(cuda_lib.AttnError) as e:  # head_dim 12: pairs not in float4 groups
        cuda_lib.attn_forward_rope(dev(q), dev(k), dev(v), out, None, 8, 8, 2, 1, 12, CAUSAL, FP32, 0, tab)
    assert e.value.code == cuda_lib.ATTN_ERR_UNSUPPORTED
    q, k, v = synthetic.forward_inputs(8, 8, 2, 1, 64, seed=1)
    tab = table(cuda_lib, 7, 64, 10000.0)
    out = torch.empty((8, 128), device="cuda")
    with pytest.raises(cuda_lib.AttnError) as e:  # table one row short
        cuda_lib.attn_forward_rope(dev(q), dev(k), dev(v), out, None, 8, 8, 2, 1, 64, CAUSAL, FP32, 0, tab)
    assert e.value.code == cuda_lib.ATTN_ERR_INVALID_ARG


def test_python_helpers_match_the_entry_point(cuda_lib, orc):
    """forward(..., rope=rope_table(...)) is attn_forward_rope (same bits)."""
    q, k, v = synthetic.forward_inputs(100, 100, 4, 2, 64, seed=12)
    tab = cuda_lib.rope_table(100, 64)
    out, lse = cuda_lib.forward(dev(q), dev(k), dev(v), 4, 2, mask=CAUSAL, prec=FP32, rope=tab)
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    cuda_lib.attn_forward_rope(dev(q), dev(k), dev(v), out2, lse2, 100, 100, 4, 2, 64, CAUSAL, FP32, 0, tab)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    ro, _ = orc.forward_rope(q.numpy(), k.numpy(), v.numpy(), 100, 100, 4, 2, 64, CAUSAL, 10000.0)
    assert_out_close(out.cpu().numpy(), ro, FP32, float(v.abs().max()), "rope helper")


@pytest.mark.parametrize("prec,tol", [(FP32, None), (BF16, 2e-2)])
@pytest.mark.parametrize("q_seq,kv_seq,H,G,D,mask,window", [
    (130, 130, 8, 2, 64, CAUSAL, 0),
    (300, 300, 4, 2, 128, CAUSAL, 77),
    (45, 131, 8, 8, 64, CROSS, 0),
])
def test_rope_backward(cuda_lib, orc, prec, tol, q_seq, kv_seq, H, G, D, mask, window):
    """attn_backward_rope after attn_forward_rope against the oracle's RoPE backward
    (fp32: 1e-5 + 1e-4 max|ref| per gradient; bf16 operands: 2e-2 max|ref|)."""
    q, k, v = synthetic.forward_inputs(q_seq, kv_seq, H, G, D, seed=q_seq + D)
    do = np.random.default_rng(q_seq).standard_normal((q_seq, H * D)).astype(np.float32)
    tab = table(cuda_lib, max(q_seq, kv_seq), D, 10000.0)
    out = torch.empty((q_seq, H * D), device="cuda")
    lse = torch.empty((q_seq, H, 2), device="cuda")
    cuda_lib.attn_forward_rope(dev(q), dev(k), dev(v), out, lse, q_seq, kv_seq, H, G, D, mask, FP32, window, tab)
    grads = [torch.full(x.shape, float("nan"), device="cuda") for x in (q, k, v)]
    cuda_lib.attn_backward_rope(dev(q), dev(k), dev(v), out, dev(torch.from_numpy(do)), lse, *grads, q_seq, kv_seq,
                                H, G, D, mask, prec, window, tab)
    torch.cuda.synchronize()
    assert cuda_lib.attn_get_status() == 0
    refs = orc.backward_rope(q.numpy(), k.numpy(), v.numpy(), do, q_seq, kv_seq, H, G, D, mask, 10000.0,
                             window=window)
    for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
        g = g.cpu().numpy()
        bound = (1e-5 + 1e-4 * np.abs(r).max()) if tol is None else tol * np.abs(r).max()
        assert np.abs(g - r).max() <= bound, (name, float(np.abs(g - r).max()), bound)
