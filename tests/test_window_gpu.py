"""Sliding-window entry points (attn_*_window) on the GPU against the fp64 oracle.

Each row whose window is keys [0, n) attends keys [max(0, n - window), n).
The cases span several 64/128-key tiles with ragged tails, windows that end
inside a tile, on a tile boundary and one past it, window 1, and windows as
long as the sequence (which must reproduce the unwindowed call bit for bit).
"""
import math

import numpy as np
import pytest
import torch

from attention_gqa_online_gb300 import synthetic
from helpers import BF16, FP32, TF32, assert_lse_close, assert_out_close, dev, tc_supported

pytestmark = pytest.mark.gpu
CAUSAL, FULL, CROSS = 0, 1, 2
PRECS = [FP32, TF32, BF16]


def run_forward_window(A, q, k, v, q_seq, kv_seq, H, G, D, mask, prec, window):
    out = torch.full((q_seq, H * D), float("nan"), device="cuda")
    lse = torch.full((q_seq, H, 2), float("nan"), device="cuda")
    A.attn_forward_window(dev(q), dev(k) if kv_seq else None, dev(v) if kv_seq else None, out, lse, q_seq, kv_seq,
                          H, G, D, mask, prec, window)
    torch.cuda.synchronize()
    assert A.attn_get_status() == 0
    return out.cpu().numpy(), lse.cpu().numpy()


def check_forward(A, orc, q_seq, kv_seq, H, G, D, mask, prec, window, seed, rows=None, **kw):
    q, k, v = synthetic.forward_inputs(q_seq, kv_seq, H, G, D, seed=seed, **kw)
    out, lse = run_forward_window(A, q, k, v, q_seq, kv_seq, H, G, D, mask, prec, window)
    ro, rl = orc.forward(q.numpy(), k.numpy(), v.numpy(), q_seq, kv_seq, H, G, D, mask, rows=rows, window=window)
    sel = slice(None) if rows is None else np.asarray(rows)
    where = "q%d kv%d H%d G%d D%d mask%d prec%d window%d" % (q_seq, kv_seq, H, G, D, mask, prec, window)
    assert_out_close(out[sel], ro[sel], prec, float(v.abs().max()), where)
    assert_lse_close(lse[sel], rl[sel], prec, float(np.abs(rl[sel][..., 0]).max()), where)
    return out, lse


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("window", [1, 5, 63, 64, 65, 127, 128, 129, 200])
@pytest.mark.parametrize("mask,kv", [(CAUSAL, 300), (FULL, 300), (CROSS, 421)])
def test_forward_window(cuda_lib, orc, prec, window, mask, kv):
    """300 queries, 8 heads over 2 kv heads, D=64: windows inside, on and past tile edges."""
    check_forward(cuda_lib, orc, 300, kv, 8, 2, 64, mask, prec, window, seed=window + 31 * mask)


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("q_seq,kv_seq,H,G,D,mask,window", [
    (67, 67, 6, 2, 80, CAUSAL, 10),      # gs = 3 (fp32 only), ragged tail
    (130, 130, 16, 2, 128, CAUSAL, 40),  # gs = 8: 16 queries per 128-row block
    (45, 131, 8, 8, 64, CROSS, 100),     # MHA, ragged key tail
    (200, 200, 1, 1, 128, CAUSAL, 77),
    (20, 20, 2, 1, 12, FULL, 3),         # small odd head_dim (fp32 only)
    (300, 300, 6, 2, 128, CAUSAL, 129),  # gs = 3 on the tensor cores
])
def test_forward_window_shapes(cuda_lib, orc, prec, q_seq, kv_seq, H, G, D, mask, window):
    if prec != FP32 and not tc_supported(H, G, D):
        pytest.skip("tensor-core precisions need D in {64, 128}")
    check_forward(cuda_lib, orc, q_seq, kv_seq, H, G, D, mask, prec, window, seed=q_seq + window)


def long_rows(q_seq, w):
    """The first rows, rows around the window length, the ragged tail, and a few at random."""
    rng = np.random.default_rng(7)
    return sorted(set(range(8)) | set(range(w - 4, w + 4)) | set(range(q_seq - 8, q_seq)) |
                  set(rng.integers(0, q_seq, 12).tolist()))


@pytest.mark.parametrize("prec", PRECS)
def test_forward_window_long_causal(cuda_lib, orc, prec):
    """q_seq 8193, 32 heads over 8 kv heads, D=128, window 4096, Q,K N(0,3^2): sampled rows."""
    q_seq, w = 8193, 4096
    check_forward(cuda_lib, orc, q_seq, q_seq, 32, 8, 128, CAUSAL, prec, w, seed=8, rows=long_rows(q_seq, w),
                  qk_sigma=3.0)


def f16_scaled(x, axis_max):
    """x * 2^(14 - E) rounded to fp16 and scaled back, with E the binary exponent of
    axis_max (the largest magnitude of x's set), as the 16-bit path stores its
    Q K^T operands."""
    e = np.clip(np.floor(np.log2(np.maximum(axis_max, 1e-38))), -100, 127)
    up = np.exp2(14.0 - e)
    return (x * up).astype(np.float16).astype(np.float64) / up


def test_forward_window_long_causal_bf16_operand_model(cuda_lib, orc):
    """The 16-bit path computes what it states: Q and each 128-key K tile rounded to
    fp16 under their own power of two, P and V rounded to bf16, fp32 accumulation.
    An fp64 evaluation of that rounding model on the windowed 8193-row case with
    Q,K N(0,3^2) (scores of standard deviation 9) must sit close to the kernel,
    and both within the 2e-2 bound of the exact result."""
    q_seq, w, H, G, D = 8193, 4096, 32, 8, 128
    rows = long_rows(q_seq, w)
    q, k, v = synthetic.forward_inputs(q_seq, q_seq, H, G, D, seed=8, qk_sigma=3.0)
    out, _ = run_forward_window(cuda_lib, q, k, v, q_seq, q_seq, H, G, D, CAUSAL, BF16, w)
    ro, _ = orc.forward(q.numpy(), k.numpy(), v.numpy(), q_seq, q_seq, H, G, D, CAUSAL, rows=rows, window=w)
    vmax = float(v.abs().max())
    sl2 = np.float32(1.0 / math.sqrt(D)) * np.float32(math.log2(math.e))
    kn, vn = k.numpy(), v.numpy()
    vb = v.to(torch.bfloat16).to(torch.float64).numpy()
    # K tiles of 128 keys per kv head, each under its own power of two.
    kq = np.empty(kn.shape, np.float64)
    for t0 in range(0, q_seq, 128):
        blk = kn[t0:t0 + 128].reshape(-1, G, D)
        m = np.abs(blk).max(axis=(0, 2))                    # per kv head
        kq[t0:t0 + 128] = f16_scaled(blk.astype(np.float64), m[None, :, None]).reshape(-1, G * D)
    model_err = kernel_err = 0.0
    for r in rows:
        lo = max(0, r + 1 - w)
        for h in range(H):
            g = h // (H // G)
            qs = (q[r, h * D:(h + 1) * D].numpy() * sl2).astype(np.float32).astype(np.float64)
            qr = f16_scaled(qs, np.abs(qs).max())
            s = kq[lo:r + 1, g * D:(g + 1) * D] @ qr
            p = np.exp2(s - s.max())
            pb = torch.from_numpy(p).to(torch.bfloat16).to(torch.float64).numpy()
            o = (pb @ vb[lo:r + 1, g * D:(g + 1) * D]) / p.sum()
            model_err = max(model_err, np.abs(o - ro[r, h * D:(h + 1) * D]).max())
            kernel_err = max(kernel_err, np.abs(out[r, h * D:(h + 1) * D] - o).max())
    assert model_err / vmax < 2e-2
    assert kernel_err / vmax < 3e-3, kernel_err / vmax
    assert np.abs(out[rows] - ro[rows]).max() / vmax < 2e-2


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("mask", [CAUSAL, FULL])
def test_forward_wide_window_is_unwindowed(cuda_lib, prec, mask):
    """window 0 and window >= n give the unwindowed call's bits."""
    q, k, v = synthetic.forward_inputs(150, 150, 4, 2, 64, seed=3)
    out = torch.empty((150, 256), device="cuda")
    lse = torch.empty((150, 4, 2), device="cuda")
    cuda_lib.attn_forward(dev(q), dev(k), dev(v), out, lse, 150, 150, 4, 2, 64, mask, prec)
    for w in (0, 150, 151, 2 ** 32 - 1):
        o2, l2 = run_forward_window(cuda_lib, q, k, v, 150, 150, 4, 2, 64, mask, prec, w)
        assert np.array_equal(out.cpu().numpy(), o2) and np.array_equal(lse.cpu().numpy(), l2), w


@pytest.mark.parametrize("prec", PRECS)
def test_forward_window_one_is_last_v(cuda_lib, prec):
    """window 1: causal row p returns V[p] of its kv head, log-sum 0."""
    q, k, v = synthetic.forward_inputs(140, 140, 4, 2, 64, seed=9)
    out, lse = run_forward_window(cuda_lib, q, k, v, 140, 140, 4, 2, 64, CAUSAL, prec, 1)
    vv = v.to(torch.bfloat16).float() if prec == BF16 else v  # bf16 operands: V itself is rounded
    ref = np.repeat(vv.numpy().reshape(140, 2, 64), 2, axis=1).reshape(140, 256)
    # TF32 operands keep 10 mantissa bits of V (relative error below 2^-10).
    np.testing.assert_allclose(out, ref, rtol=2.0 ** -10 if prec == TF32 else 0, atol=1e-6)
    assert np.max(np.abs(lse[..., 1])) < 1e-6


# ---------------------------------------------------------------- prefill
def check_prefill(A, orc, n_queries, H, G, D, kv_dim, max_seq, start_pos, q_stride, out_stride, q_base, prec,
                  window, seed):
    q_rows = q_base + n_queries
    qb, kc, vc = synthetic.prefill_inputs(q_rows, q_stride, max_seq, kv_dim, seed=seed)
    scale = np.float32(1.0 / math.sqrt(D))
    sentinel = 12345.0
    out = torch.full((q_rows, out_stride), sentinel, device="cuda")
    A.attn_prefill_window(dev(qb), dev(kc), dev(vc), out, n_queries, H, G, D, kv_dim, max_seq, float(scale),
                          start_pos, q_stride, out_stride, q_base, prec, window)
    torch.cuda.synchronize()
    assert A.attn_get_status() == 0
    got = out.cpu().numpy()
    ref = orc.prefill(qb.numpy(), kc.numpy(), vc.numpy(), q_rows, n_queries, H, G, D, kv_dim, max_seq, scale,
                      start_pos, q_stride, out_stride, q_base, window=window)
    written = np.zeros_like(got, dtype=bool)
    written[q_base:q_base + n_queries, :H * D] = True
    assert np.all(got[~written] == sentinel), "prefill wrote outside its rows / head columns"
    where = "nq%d H%d G%d D%d start%d qbase%d window%d" % (n_queries, H, G, D, start_pos, q_base, window)
    assert_out_close(got[written].reshape(n_queries, H * D), ref[written].reshape(n_queries, H * D), prec,
                     float(vc.abs().max()), where)


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("window", [1, 100, 128, 1000, 1537])
def test_prefill_window_config(cuda_lib, orc, prec, window):
    """512 queries from start_pos 1536 into a 2048-row cache, 32 heads over 8, D=128."""
    check_prefill(cuda_lib, orc, 512, 32, 8, 128, 1024, 2048, 1536, 4096, 4096, 0, prec, window, seed=window)


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("n_queries,H,G,D,kv_dim,max_seq,start_pos,q_stride,out_stride,q_base,window", [
    (37, 6, 2, 80, 200, 300, 100, 500, 520, 5, 33),      # gs = 3 (fp32 only)
    (129, 8, 1, 64, 96, 1000, 700, 520, 512, 3, 300),    # gs = 8, kv_dim > G*D
    (64, 32, 8, 128, 1024, 128, 0, 4096, 4096, 64, 50),  # start 0, q_base 64
])
def test_prefill_window_shapes(cuda_lib, orc, prec, n_queries, H, G, D, kv_dim, max_seq, start_pos, q_stride,
                               out_stride, q_base, window):
    if prec != FP32 and not tc_supported(H, G, D):
        pytest.skip("tensor-core precisions need D in {64, 128}")
    check_prefill(cuda_lib, orc, n_queries, H, G, D, kv_dim, max_seq, start_pos, q_stride, out_stride, q_base, prec,
                  window, seed=n_queries + window)


# ---------------------------------------------------------------- decode
def run_decode_window(A, dq, dk, dv, pos_t, ws, kv_pos, H, G, D, max_seq, window):
    pos_t.fill_(int(kv_pos))
    out = torch.full((1, H * D), float("nan"), device="cuda")
    A.attn_decode_cached_window(dq, dk, dv, pos_t, out, H, G, D, max_seq, ws, None, window)
    torch.cuda.synchronize()
    assert A.attn_get_status() == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("H,G,D,max_seq,cases", [
    (32, 8, 128, 16384, [(16383, 4096), (16383, 1), (4095, 4096), (4096, 4096), (9000, 31), (511, 64)]),
    (16, 2, 64, 3000, [(2999, 65), (2999, 3000), (100, 7)]),   # split kernel, gs = 8
    (6, 2, 80, 513, [(512, 100), (5, 3), (300, 1)]),           # generic kernel (D = 80)
    (64, 8, 128, 2048, [(2047, 300), (1000, 1)]),              # split kernel, two head groups per kv head
])
def test_decode_window(cuda_lib, orc, H, G, D, max_seq, cases):
    q, kc, vc = synthetic.decode_inputs(max_seq, H, G, D, seed=max_seq + 1)
    dq, dk, dv = dev(q), dev(kc), dev(vc)
    nbytes = cuda_lib.attn_decode_workspace_bytes(H, G, D, max_seq)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    for kp, w in cases:
        ref = orc.decode(q.numpy(), kc.numpy(), vc.numpy(), kp, H, G, D, max_seq, window=w)
        for _ in range(2):  # the workspace is reusable across windowed calls too
            out = run_decode_window(cuda_lib, dq, dk, dv, pos, ws, kp, H, G, D, max_seq, w)
            assert_out_close(out, ref, FP32, float(vc.abs().max()), "H%d G%d D%d kv_pos=%d window=%d" % (
                H, G, D, kp, w))
