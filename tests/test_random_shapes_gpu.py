"""Seeded random shapes through forward, prefill, decode and backward, every precision, against the fp64 oracle.

Each case draws its own sizes from a generator seeded by the case number:
head_dim (64 and 128, and sizes only the fp32 path takes), kv heads, query
heads per kv head (including groups that do not divide 128), mask, ragged
sequence lengths, sliding windows (none, short, past the sequence), strides
with padding, q_base, and score spreads of N(0,1) and N(0,3^2).  The oracle
runs once per case; every precision the shape supports is compared with it at
that precision's tolerance.
"""
import math

import numpy as np
import pytest
import torch

from attention_gqa_online_gb300 import synthetic
from helpers import BF16, FP32, TF32, assert_lse_close, assert_out_close, dev, tc_supported

pytestmark = pytest.mark.gpu
CAUSAL, FULL, CROSS = 0, 1, 2


def precisions(H, G, D):
    return [FP32, TF32, BF16] if tc_supported(H, G, D) else [FP32]


def forward_case(i):
    rng = np.random.default_rng(7000 + i)
    D = int(rng.choice([64, 128, 64, 128, 32, 96, 8]))
    G = int(rng.integers(1, 5))
    gs = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 16]))
    mask = int(rng.integers(0, 3))
    q_seq = int(rng.integers(1, 320))
    kv_seq = q_seq if mask != CROSS else int(rng.integers(1, 420))
    window = 0 if rng.random() < 0.4 else int(rng.integers(1, kv_seq + 40))
    sigma = float(rng.choice([1.0, 3.0]))
    rows = None
    if q_seq > 96:
        rows = sorted(set(range(8)) | set(range(q_seq - 8, q_seq)) | set(rng.integers(0, q_seq, 40).tolist()))
    return G * gs, G, D, mask, q_seq, kv_seq, window, sigma, rows


@pytest.mark.parametrize("case", range(30))
def test_random_forward(cuda_lib, orc, case):
    H, G, D, mask, q_seq, kv_seq, window, sigma, rows = forward_case(case)
    q, k, v = synthetic.forward_inputs(q_seq, kv_seq, H, G, D, seed=case, qk_sigma=sigma)
    ro, rl = orc.forward(q.numpy(), k.numpy(), v.numpy(), q_seq, kv_seq, H, G, D, mask, rows=rows, window=window)
    sel = slice(None) if rows is None else np.asarray(rows)
    dq, dk, dvv = dev(q), dev(k), dev(v)
    for prec in precisions(H, G, D):
        out = torch.full((q_seq, H * D), float("nan"), device="cuda")
        lse = torch.full((q_seq, H, 2), float("nan"), device="cuda")
        cuda_lib.attn_forward_window(dq, dk, dvv, out, lse, q_seq, kv_seq, H, G, D, mask, prec, window)
        torch.cuda.synchronize()
        assert cuda_lib.attn_get_status() == 0
        where = "case %d: q%d kv%d H%d G%d D%d mask%d window%d sigma%g prec%d" % (
            case, q_seq, kv_seq, H, G, D, mask, window, sigma, prec)
        got, gl = out.cpu().numpy()[sel], lse.cpu().numpy()[sel]
        assert_out_close(got, ro[sel], prec, float(v.abs().max()), where)
        assert_lse_close(gl, rl[sel], prec, float(np.abs(rl[sel][..., 0]).max()), where)


def prefill_case(i):
    rng = np.random.default_rng(8000 + i)
    D = int(rng.choice([64, 128, 64, 128, 80, 32]))
    G = int(rng.integers(1, 4))
    gs = int(rng.choice([1, 2, 3, 4, 8]))
    H = G * gs
    n_queries = int(rng.integers(1, 121))
    max_seq = n_queries + int(rng.integers(0, 380))
    start_pos = int(rng.integers(0, max_seq - n_queries + 1))
    kv_dim = G * D + 4 * int(rng.integers(0, 3))
    q_stride = H * D + 4 * int(rng.integers(0, 3))
    out_stride = H * D + 4 * int(rng.integers(0, 3))
    q_base = int(rng.integers(0, 6))
    window = 0 if rng.random() < 0.4 else int(rng.integers(1, max_seq + 20))
    return n_queries, H, G, D, kv_dim, max_seq, start_pos, q_stride, out_stride, q_base, window


@pytest.mark.parametrize("case", range(20))
def test_random_prefill(cuda_lib, orc, case):
    n_queries, H, G, D, kv_dim, max_seq, start_pos, q_stride, out_stride, q_base, window = prefill_case(case)
    q_rows = q_base + n_queries
    qb, kc, vc = synthetic.prefill_inputs(q_rows, q_stride, max_seq, kv_dim, seed=100 + case)
    scale = np.float32(1.0 / math.sqrt(D))
    ref = orc.prefill(qb.numpy(), kc.numpy(), vc.numpy(), q_rows, n_queries, H, G, D, kv_dim, max_seq, scale,
                      start_pos, q_stride, out_stride, q_base, window=window)
    written = np.zeros((q_rows, out_stride), dtype=bool)
    written[q_base:q_base + n_queries, :H * D] = True
    dqb, dkc, dvc = dev(qb), dev(kc), dev(vc)
    sentinel = 12345.0
    for prec in precisions(H, G, D):
        out = torch.full((q_rows, out_stride), sentinel, device="cuda")
        # K/V row strides that are not multiples of 8 floats run the
        # tensor-core precisions on the fp32 kernel.
        cuda_lib.attn_prefill_window(dqb, dkc, dvc, out, n_queries, H, G, D, kv_dim, max_seq, float(scale),
                                     start_pos, q_stride, out_stride, q_base, prec, window)
        torch.cuda.synchronize()
        assert cuda_lib.attn_get_status() == 0
        got = out.cpu().numpy()
        where = "case %d: nq%d H%d G%d D%d max_seq%d start%d strides %d/%d/%d qbase%d window%d prec%d" % (
            case, n_queries, H, G, D, max_seq, start_pos, kv_dim, q_stride, out_stride, q_base, window, prec)
        assert np.all(got[~written] == sentinel), where + ": wrote outside its rows / head columns"
        assert_out_close(got[written].reshape(n_queries, H * D), ref[written].reshape(n_queries, H * D), prec,
                         float(vc.abs().max()), where)


def decode_case(i):
    rng = np.random.default_rng(9000 + i)
    D = int(rng.choice([64, 128, 64, 128, 80]))
    G = int(rng.integers(1, 9))
    gs = int(rng.choice([1, 2, 3, 4, 8, 16]))
    max_seq = int(rng.integers(1, 4000))
    positions = sorted({0, max_seq - 1, int(rng.integers(0, max_seq)), int(rng.integers(0, max_seq))})
    windows = [0, int(rng.integers(1, max_seq + 50))]
    return G * gs, G, D, max_seq, positions, windows


@pytest.mark.parametrize("case", range(16))
def test_random_decode(cuda_lib, orc, case):
    H, G, D, max_seq, positions, windows = decode_case(case)
    q, kc, vc = synthetic.decode_inputs(max_seq, H, G, D, seed=200 + case)
    dq, dk, dvv = dev(q), dev(kc), dev(vc)
    ws = torch.zeros(cuda_lib.attn_decode_workspace_bytes(H, G, D, max_seq), dtype=torch.uint8, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    vmax = float(vc.abs().max())
    for kp in positions:
        for w in windows:
            ref = orc.decode(q.numpy(), kc.numpy(), vc.numpy(), kp, H, G, D, max_seq, window=w)
            pos.fill_(kp)
            out = torch.full((1, H * D), float("nan"), device="cuda")
            cuda_lib.attn_decode_cached_window(dq, dk, dvv, pos, out, H, G, D, max_seq, ws, None, w)
            torch.cuda.synchronize()
            assert cuda_lib.attn_get_status() == 0
            assert_out_close(out.cpu().numpy(), ref, FP32, vmax, "case %d: H%d G%d D%d max_seq%d kv_pos%d window%d" % (
                case, H, G, D, max_seq, kp, w))


def backward_case(i):
    rng = np.random.default_rng(10000 + i)
    D = int(rng.choice([64, 128, 64, 48]))
    G = int(rng.integers(1, 4))
    gs = int(rng.choice([1, 2, 3, 4, 8]))
    mask = int(rng.integers(0, 3))
    q_seq = int(rng.integers(1, 200))
    kv_seq = q_seq if mask != CROSS else int(rng.integers(1, 260))
    window = 0 if rng.random() < 0.5 else int(rng.integers(1, kv_seq + 20))
    return G * gs, G, D, mask, q_seq, kv_seq, window


@pytest.mark.parametrize("case", range(12))
def test_random_backward(cuda_lib, orc, case):
    """dq, dk, dv per gradient tensor: fp32 within 1e-5 + 1e-4 max|ref|; bf16 operands
    (D in {64, 128}, power-of-two groups) within 2e-2 max|ref|."""
    H, G, D, mask, q_seq, kv_seq, window = backward_case(case)
    q, k, v = synthetic.forward_inputs(q_seq, kv_seq, H, G, D, seed=300 + case)
    dout = torch.from_numpy(np.random.default_rng(400 + case).standard_normal((q_seq, H * D)).astype(np.float32))
    ref = orc.backward(q.numpy(), k.numpy(), v.numpy(), dout.numpy(), q_seq, kv_seq, H, G, D, mask, window=window)
    gs = H // G
    precs = [FP32, BF16] if D in (64, 128) and gs & (gs - 1) == 0 else [FP32]
    dq_, dk_, dv_, do_ = dev(q), dev(k), dev(v), dev(dout)
    out = torch.empty((q_seq, H * D), device="cuda")
    lse = torch.empty((q_seq, H, 2), device="cuda")
    cuda_lib.attn_forward_window(dq_, dk_, dv_, out, lse, q_seq, kv_seq, H, G, D, mask, FP32, window)
    for prec in precs:
        grads = [torch.full(shape, float("nan"), device="cuda") for shape in
                 ((q_seq, H * D), (kv_seq, G * D), (kv_seq, G * D))]
        cuda_lib.attn_backward(dq_, dk_, dv_, out, do_, lse, *grads, q_seq, kv_seq, H, G, D, mask, prec, window)
        torch.cuda.synchronize()
        assert cuda_lib.attn_get_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
            got = g.cpu().numpy()
            where = "case %d: q%d kv%d H%d G%d D%d mask%d window%d prec%d %s" % (
                case, q_seq, kv_seq, H, G, D, mask, window, prec, name)
            assert np.all(np.isfinite(got)), where + ": non-finite gradient"
            err = float(np.abs(got - r).max())
            tol = (1e-5 + 1e-4 * float(np.abs(r).max())) if prec == FP32 else 2e-2 * float(np.abs(r).max())
            assert err <= tol, "%s: max|err| = %.3g > %.3g" % (where, err, tol)


def offset_view(x, shape):
    """x's values in a device buffer that starts one float past a 16-byte boundary."""
    buf = torch.zeros(x.numel() + 4, device="cuda")
    v = buf[1:1 + x.numel()].view(shape)
    v.copy_(x.reshape(shape).to("cuda"))
    assert v.data_ptr() % 16 == 4
    return v


@pytest.mark.parametrize("prec", [TF32, BF16])
def test_tensor_core_precision_layouts_off_the_kernels(cuda_lib, orc, prec):
    """Layouts the tensor-core kernels do not take run on the fp32 kernel and meet the
    precision's bound: pointers 4 bytes past a 16-byte boundary, and 160 query heads
    over one kv head (more than a thread block's 128 rows)."""
    q_seq, H, G, D = 70, 6, 2, 64
    q, k, v = synthetic.forward_inputs(q_seq, q_seq, H, G, D, seed=41, qk_sigma=3.0)
    ro, rl = orc.forward(q.numpy(), k.numpy(), v.numpy(), q_seq, q_seq, H, G, D, CAUSAL)
    out = offset_view(torch.full((q_seq, H * D), float("nan")), (q_seq, H * D))
    lse = torch.full((q_seq, H, 2), float("nan"), device="cuda")
    cuda_lib.attn_forward(offset_view(q, (q_seq, H * D)), offset_view(k, (q_seq, G * D)),
                          offset_view(v, (q_seq, G * D)), out, lse, q_seq, q_seq, H, G, D, CAUSAL, prec)
    torch.cuda.synchronize()
    assert cuda_lib.attn_get_status() == 0
    assert_out_close(out.cpu().numpy(), ro, prec, float(v.abs().max()), "offset pointers")
    assert_lse_close(lse.cpu().numpy(), rl, prec, float(np.abs(rl[..., 0]).max()), "offset pointers")

    q_seq, H, G, D = 9, 160, 1, 64
    q, k, v = synthetic.forward_inputs(q_seq, q_seq, H, G, D, seed=42)
    ro, rl = orc.forward(q.numpy(), k.numpy(), v.numpy(), q_seq, q_seq, H, G, D, FULL)
    out = torch.full((q_seq, H * D), float("nan"), device="cuda")
    lse = torch.full((q_seq, H, 2), float("nan"), device="cuda")
    cuda_lib.attn_forward(dev(q), dev(k), dev(v), out, lse, q_seq, q_seq, H, G, D, FULL, prec)
    torch.cuda.synchronize()
    assert cuda_lib.attn_get_status() == 0
    assert_out_close(out.cpu().numpy(), ro, prec, float(v.abs().max()), "160 query heads per kv head")
    assert_lse_close(lse.cpu().numpy(), rl, prec, float(np.abs(rl[..., 0]).max()), "160 query heads per kv head")


def test_bf16_backward_group_of_three(cuda_lib, orc):
    """bf16 operands with 3 query heads per kv head (not a power of two) run the fp32
    backward: within the bf16 bound (2e-2 max|ref|), indeed within fp32's."""
    q_seq, H, G, D = 90, 6, 2, 64
    q, k, v = synthetic.forward_inputs(q_seq, q_seq, H, G, D, seed=43)
    dout = torch.from_numpy(np.random.default_rng(44).standard_normal((q_seq, H * D)).astype(np.float32))
    ref = orc.backward(q.numpy(), k.numpy(), v.numpy(), dout.numpy(), q_seq, q_seq, H, G, D, CAUSAL)
    dq_, dk_, dv_, do_ = dev(q), dev(k), dev(v), dev(dout)
    out = torch.empty((q_seq, H * D), device="cuda")
    lse = torch.empty((q_seq, H, 2), device="cuda")
    cuda_lib.attn_forward(dq_, dk_, dv_, out, lse, q_seq, q_seq, H, G, D, CAUSAL, FP32)
    grads = [torch.full(shape, float("nan"), device="cuda") for shape in ((q_seq, H * D), (q_seq, G * D), (q_seq, G * D))]
    cuda_lib.attn_backward(dq_, dk_, dv_, out, do_, lse, *grads, q_seq, q_seq, H, G, D, CAUSAL, BF16)
    torch.cuda.synchronize()
    assert cuda_lib.attn_get_status() == 0
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        err = float(np.abs(g.cpu().numpy() - r).max())
        assert err <= 1e-5 + 1e-4 * float(np.abs(r).max()), "%s: %.3g" % (name, err)
