"""attn_backward on the GPU against the fp64 oracle's backward.

The GPU forward supplies out and lse (as a caller would get them); the
oracle's backward recomputes everything from q, k, v and dout in fp64.
Tolerance (fp32 arithmetic), per gradient tensor: max |gpu - ref| <=
1e-5 + 1e-4 * max |ref| -- the forward's fp32 bound (1e-5 absolute, 1e-4
relative) with the relative part taken against the tensor's largest entry.
Each gradient element is a sum over up to a few thousand rows or keys of
fp32 products, and the softmax is rebuilt from the fp32 (max, log-sum) pair
and the fp32 forward output, whose own errors are of that size.  The
absolute part matters where the exact gradient is 0 (a row with one kept
key has dq = 0; fp32 rounding leaves a few 1e-6).
"""
import numpy as np
import pytest
import torch

from attention_gqa_online_gb300 import synthetic
from helpers import dev

pytestmark = pytest.mark.gpu
CAUSAL, FULL, CROSS = 0, 1, 2
ATOL, RTOL = 1e-5, 1e-4


def gpu_backward(A, q, k, v, dout, q_seq, kv_seq, H, G, D, mask, window=0):
    dq_, dk_, dv_, do_ = dev(q), dev(k) if kv_seq else None, dev(v) if kv_seq else None, dev(dout)
    out = torch.empty((q_seq, H * D), device="cuda")
    lse = torch.empty((q_seq, H, 2), device="cuda")
    A.attn_forward_window(dq_, dk_, dv_, out, lse, q_seq, kv_seq, H, G, D, mask, A.ATTN_FP32, window)
    gq = torch.full((q_seq, H * D), float("nan"), device="cuda")
    gk = torch.full((kv_seq, G * D), float("nan"), device="cuda")
    gv = torch.full((kv_seq, G * D), float("nan"), device="cuda")
    A.attn_backward(dq_, dk_, dv_, out, do_, lse, gq, gk if kv_seq else None, gv if kv_seq else None, q_seq, kv_seq,
                    H, G, D, mask, A.ATTN_FP32, window)
    torch.cuda.synchronize()
    assert A.attn_get_status() == 0
    return gq.cpu().numpy(), gk.cpu().numpy(), gv.cpu().numpy()


def assert_grad_close(got, ref, what):
    assert np.all(np.isfinite(got)), what + ": non-finite gradient"
    err = float(np.abs(got - ref).max())
    tol = ATOL + RTOL * float(np.abs(ref).max())
    assert err <= tol, "%s: max|err| = %.3g > %.3g" % (what, err, tol)


def check(A, orc, q_seq, kv_seq, H, G, D, mask, window=0, seed=0, **kw):
    q, k, v = (x.numpy() for x in synthetic.forward_inputs(q_seq, kv_seq, H, G, D, seed=seed, **kw))
    dout = np.random.default_rng(seed + 1000).standard_normal((q_seq, H * D)).astype(np.float32)
    got = gpu_backward(A, torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), torch.from_numpy(dout),
                       q_seq, kv_seq, H, G, D, mask, window)
    ref = orc.backward(q, k, v, dout, q_seq, kv_seq, H, G, D, mask, window=window)
    where = "q%d kv%d H%d G%d D%d mask%d window%d" % (q_seq, kv_seq, H, G, D, mask, window)
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        if b.size:
            assert_grad_close(a, b, where + " " + name)


@pytest.mark.parametrize("mask,kv", [(CAUSAL, 16), (FULL, 16), (CROSS, 24)])
def test_small_config(cuda_lib, orc, mask, kv):
    """q_seq=16, 4 heads over 2 kv heads, D=64, N(0,1), seed 0."""
    check(cuda_lib, orc, 16, kv, 4, 2, 64, mask)


@pytest.mark.parametrize("q_seq,kv_seq,H,G,D,mask,window", [
    (67, 67, 6, 2, 80, CAUSAL, 0),      # gs = 3, ragged tails in rows and keys
    (67, 67, 6, 2, 80, FULL, 0),
    (45, 131, 8, 8, 64, CROSS, 0),      # MHA, ragged key tail
    (130, 130, 16, 2, 128, CAUSAL, 0),  # gs = 8
    (200, 200, 1, 1, 128, CAUSAL, 0),
    (20, 20, 2, 1, 12, FULL, 0),        # small head_dim
    (1, 1, 4, 2, 64, CAUSAL, 0),        # one query, one key
    (300, 300, 8, 2, 64, CAUSAL, 100),  # sliding windows
    (300, 300, 8, 2, 64, FULL, 65),
    (90, 421, 8, 2, 64, CROSS, 129),
    (150, 150, 4, 2, 64, CAUSAL, 1),
])
def test_shapes(cuda_lib, orc, q_seq, kv_seq, H, G, D, mask, window):
    check(cuda_lib, orc, q_seq, kv_seq, H, G, D, mask, window, seed=q_seq + D + window)


def test_causal_1024_wide_scores(cuda_lib, orc):
    """q_seq 1024, 8 heads over 2 kv heads, D=128, Q,K N(0,3^2): 16 row blocks, 16 key blocks."""
    check(cuda_lib, orc, 1024, 1024, 8, 2, 128, CAUSAL, seed=11, qk_sigma=3.0)


def test_empty_keys(cuda_lib):
    q, _, _ = synthetic.forward_inputs(7, 0, 4, 2, 64, seed=22)
    dout = torch.ones((7, 256))
    gq, gk, gv = gpu_backward(cuda_lib, q, None, None, dout, 7, 0, 4, 2, 64, CROSS)
    assert np.all(gq == 0.0) and gk.size == 0 and gv.size == 0


def test_repeatable_bits(cuda_lib):
    q, k, v = synthetic.forward_inputs(300, 300, 8, 2, 64, seed=5)
    dout = torch.randn((300, 512), generator=torch.Generator().manual_seed(5))
    a = gpu_backward(cuda_lib, q, k, v, dout, 300, 300, 8, 2, 64, CAUSAL)
    b = gpu_backward(cuda_lib, q, k, v, dout, 300, 300, 8, 2, 64, CAUSAL)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_unsupported_forms(cuda_lib):
    q, k, v = synthetic.forward_inputs(8, 8, 2, 1, 6, seed=1)  # head_dim 6: not a multiple of 4
    z = torch.zeros((8, 12), device="cuda")
    lse = torch.zeros((8, 2, 2), device="cuda")
    with pytest.raises(cuda_lib.AttnError) as e:
        cuda_lib.attn_backward(dev(q), dev(k), dev(v), z, z, lse, z.clone(), z[:, :6].clone(), z[:, :6].clone(),
                               8, 8, 2, 1, 6, CAUSAL, cuda_lib.ATTN_FP32)
    assert e.value.code == cuda_lib.ATTN_ERR_UNSUPPORTED
    q, k, v = synthetic.forward_inputs(8, 8, 2, 1, 64, seed=1)
    z = torch.zeros((8, 128), device="cuda")
    with pytest.raises(cuda_lib.AttnError) as e:
        cuda_lib.attn_backward(dev(q), dev(k), dev(v), z, z, lse, z.clone(), z[:, :64].clone(), z[:, :64].clone(),
                               8, 8, 2, 1, 64, CAUSAL, cuda_lib.ATTN_TF32)
    assert e.value.code == cuda_lib.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("window", [0, 4096])
def test_long_causal_properties_and_sampled_rows(cuda_lib, orc, window):
    """q_seq 8192, 32 heads over 8 kv heads, D=128, Q,K N(0,3^2) (the long forward
    workload): properties that hold at any size -- per kv head, the key sums of dv
    equal the summed dout of its query heads and the key sums of dk vanish -- plus
    sampled dq rows, each the oracle's cross-attention backward of that one row
    over its own window."""
    q_seq, H, G, D = 8192, 32, 8, 128
    q, k, v = synthetic.forward_inputs(q_seq, q_seq, H, G, D, seed=5, qk_sigma=3.0)
    dout = torch.from_numpy(np.random.default_rng(77).standard_normal((q_seq, H * D)).astype(np.float32))
    gq, gk, gv = gpu_backward(cuda_lib, q, k, v, dout, q_seq, q_seq, H, G, D, CAUSAL, window)
    dsum = dout.double().numpy().reshape(q_seq, G, H // G, D).sum(axis=(0, 2)).reshape(G * D)
    vs = gv.astype(np.float64).sum(axis=0)
    assert np.abs(vs - dsum).max() <= ATOL + RTOL * np.abs(dsum).max()
    ks = gk.astype(np.float64).sum(axis=0)
    assert np.abs(ks).max() <= ATOL + RTOL * np.abs(gk).sum(axis=0).max()
    qn, kn, vn, dn = q.numpy(), k.numpy(), v.numpy(), dout.numpy()
    for i in (0, 1, 127, 4095, 4096, 6000, 8191):
        n = i + 1
        lo = max(0, n - window) if window else 0
        dq1, _, _ = orc.backward(qn[i:i + 1], kn[lo:n], vn[lo:n], dn[i:i + 1], 1, n - lo, H, G, D, CROSS)
        assert_grad_close(gq[i:i + 1], dq1, "dq row %d window %d" % (i, window))


# ---------------------------------------------------------------- bf16 operands (tensor cores)
BF16_TOL = 2e-2  # per gradient tensor: max|gpu - ref| <= 2e-2 * max|ref| (the forward's bf16 bound)


def gpu_backward_bf16(A, q, k, v, dout, q_seq, kv_seq, H, G, D, mask, window=0):
    dq_, dk_, dv_, do_ = dev(q), dev(k), dev(v), dev(dout)
    out = torch.empty((q_seq, H * D), device="cuda")
    lse = torch.empty((q_seq, H, 2), device="cuda")
    A.attn_forward_window(dq_, dk_, dv_, out, lse, q_seq, kv_seq, H, G, D, mask, A.ATTN_FP32, window)
    gq = torch.full((q_seq, H * D), float("nan"), device="cuda")
    gk = torch.full((kv_seq, G * D), float("nan"), device="cuda")
    gv = torch.full((kv_seq, G * D), float("nan"), device="cuda")
    A.attn_backward(dq_, dk_, dv_, out, do_, lse, gq, gk, gv, q_seq, kv_seq, H, G, D, mask, A.ATTN_BF16, window)
    torch.cuda.synchronize()
    assert A.attn_get_status() == 0
    return gq.cpu().numpy(), gk.cpu().numpy(), gv.cpu().numpy()


@pytest.mark.parametrize("q_seq,kv_seq,H,G,D,mask,window", [
    (16, 16, 4, 2, 64, CAUSAL, 0),
    (16, 24, 4, 2, 64, CROSS, 0),
    (300, 300, 8, 2, 64, CAUSAL, 0),    # 3 row blocks (gs = 4: 32 queries each), ragged tail
    (300, 300, 8, 2, 64, FULL, 0),
    (130, 130, 16, 2, 128, CAUSAL, 0),  # gs = 8
    (200, 200, 1, 1, 128, CAUSAL, 0),   # MHA, one head
    (90, 421, 8, 8, 128, CROSS, 0),     # ragged key tail
    (300, 300, 8, 2, 64, CAUSAL, 100),  # sliding windows
    (90, 421, 8, 2, 64, CROSS, 129),
    (1024, 1024, 8, 2, 128, CAUSAL, 0),
])
def test_bf16_shapes(cuda_lib, orc, q_seq, kv_seq, H, G, D, mask, window):
    q, k, v = (x.numpy() for x in synthetic.forward_inputs(q_seq, kv_seq, H, G, D, seed=q_seq + window))
    dout = np.random.default_rng(q_seq).standard_normal((q_seq, H * D)).astype(np.float32)
    got = gpu_backward_bf16(cuda_lib, *(torch.from_numpy(x) for x in (q, k, v, dout)), q_seq, kv_seq, H, G, D, mask,
                            window)
    ref = orc.backward(q, k, v, dout, q_seq, kv_seq, H, G, D, mask, window=window)
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(a)), name
        err = float(np.abs(a - b).max()) / float(np.abs(b).max())
        assert err <= BF16_TOL, "bf16 backward q%d kv%d mask%d window%d %s: %.3g" % (q_seq, kv_seq, mask, window,
                                                                                     name, err)


def test_bf16_long_causal_properties(cuda_lib, orc):
    """q_seq 8192, 32 / 8 heads, D=128: key sums of dv and dk, and sampled dq rows (oracle,
    one row over its own window as cross attention)."""
    q_seq, H, G, D = 8192, 32, 8, 128
    q, k, v = synthetic.forward_inputs(q_seq, q_seq, H, G, D, seed=5)
    dout = torch.from_numpy(np.random.default_rng(78).standard_normal((q_seq, H * D)).astype(np.float32))
    gq, gk, gv = gpu_backward_bf16(cuda_lib, q, k, v, dout, q_seq, q_seq, H, G, D, CAUSAL)
    dsum = dout.double().numpy().reshape(q_seq, G, H // G, D).sum(axis=(0, 2)).reshape(G * D)
    assert np.abs(gv.astype(np.float64).sum(axis=0) - dsum).max() <= BF16_TOL * np.abs(dsum).max()
    assert np.abs(gk.astype(np.float64).sum(axis=0)).max() <= BF16_TOL * np.abs(gk).sum(axis=0).max()
    qn, kn, vn, dn = q.numpy(), k.numpy(), v.numpy(), dout.numpy()
    rows = (0, 1, 127, 4096, 8191)  # row 0 has one key: its exact dq is 0
    refs = [orc.backward(qn[i:i + 1], kn[:i + 1], vn[:i + 1], dn[i:i + 1], 1, i + 1, H, G, D, CROSS)[0] for i in rows]
    scale = max(float(np.abs(r).max()) for r in refs)
    for i, r in zip(rows, refs):
        assert np.abs(gq[i:i + 1] - r).max() <= BF16_TOL * scale, i
