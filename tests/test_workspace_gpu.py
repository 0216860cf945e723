"""Caller-owned scratch (attn_set_workspace) through the C ABI.

A workspace of exactly the size the query reports serves each call that
needs scratch, the results are bit-identical to the library-pool path, and
the library pool's high-water mark stays at zero meanwhile: the call
allocated nothing.  A workspace one byte short is refused before anything
runs (the output keeps its sentinel), as is a misaligned one."""
import math

import numpy as np
import pytest
import torch

from attention_gqa_online_gb300 import synthetic
from helpers import BF16, FP32, TF32, dev

pytestmark = pytest.mark.gpu
CAUSAL = 0


def forward_call(A, q, k, v, out, lse, n, H, G, D, prec, rope=None, window=0):
    if rope is None:
        A.attn_forward_window(q, k, v, out, lse, n, n, H, G, D, CAUSAL, prec, window)
    else:
        A.attn_forward_rope(q, k, v, out, lse, n, n, H, G, D, CAUSAL, prec, window, rope)


def with_workspace(A, nbytes, fn):
    """Run fn with a fresh workspace of nbytes bound; return the pool's peak use during it."""
    torch.cuda.synchronize()
    A.attn_scratch_peak_bytes(reset=True)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    A.attn_set_workspace(ws, nbytes)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        A.attn_set_workspace(None)
    return A.attn_scratch_peak_bytes()


@pytest.mark.parametrize("prec,use_rope", [(BF16, False), (TF32, False), (BF16, True), (FP32, True)])
def test_forward_with_workspace(cuda_lib, prec, use_rope):
    A = cuda_lib
    n, H, G, D = 300, 8, 2, 128
    q, k, v = (dev(x) for x in synthetic.forward_inputs(n, n, H, G, D, seed=31))
    rope = None
    if use_rope:
        rope = torch.empty((n, D), device="cuda")
        A.attn_rope_table(rope, n, D, 10000.0)
    need = A.attn_forward_workspace_bytes(n, n, H, G, D, CAUSAL, prec, 0, use_rope)
    assert need > 0
    ref, ref_l = torch.empty((n, H * D), device="cuda"), torch.empty((n, H, 2), device="cuda")
    forward_call(A, q, k, v, ref, ref_l, n, H, G, D, prec, rope)
    out = torch.full((n, H * D), float("nan"), device="cuda")
    lse = torch.full((n, H, 2), float("nan"), device="cuda")
    peak = with_workspace(A, need, lambda: forward_call(A, q, k, v, out, lse, n, H, G, D, prec, rope))
    assert peak == 0
    assert torch.equal(out, ref) and torch.equal(lse, ref_l)
    assert A.attn_get_status() == 0


def test_prefill_with_workspace(cuda_lib):
    A = cuda_lib
    nq, H, G, D, max_seq, start = 96, 32, 8, 128, 640, 500
    qb, kc, vc = (dev(x) for x in synthetic.prefill_inputs(nq, H * D, max_seq, G * D, seed=32))
    scale = 1.0 / math.sqrt(D)
    for prec in (BF16, TF32):
        need = A.attn_prefill_workspace_bytes(nq, H, G, D, G * D, max_seq, start, 0, prec)
        assert need > 0
        ref = torch.empty((nq, H * D), device="cuda")
        A.attn_prefill(qb, kc, vc, ref, nq, H, G, D, G * D, max_seq, scale, start, H * D, H * D, 0, prec)
        out = torch.full((nq, H * D), float("nan"), device="cuda")
        peak = with_workspace(A, need, lambda: A.attn_prefill(qb, kc, vc, out, nq, H, G, D, G * D, max_seq, scale,
                                                              start, H * D, H * D, 0, prec))
        assert peak == 0
        assert torch.equal(out, ref)


@pytest.mark.parametrize("prec,use_rope", [(BF16, True), (FP32, False)])
def test_backward_with_workspace(cuda_lib, prec, use_rope):
    A = cuda_lib
    n, H, G, D = 200, 8, 2, 64
    q, k, v = (dev(x) for x in synthetic.forward_inputs(n, n, H, G, D, seed=33))
    dout = dev(torch.from_numpy(np.random.default_rng(33).standard_normal((n, H * D)).astype(np.float32)))
    rope = None
    if use_rope:
        rope = torch.empty((n, D), device="cuda")
        A.attn_rope_table(rope, n, D, 10000.0)
    out, lse = torch.empty((n, H * D), device="cuda"), torch.empty((n, H, 2), device="cuda")
    forward_call(A, q, k, v, out, lse, n, H, G, D, prec, rope)
    need = A.attn_backward_workspace_bytes(n, n, H, G, D, prec, use_rope)
    assert need > 0

    def grads():
        g = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
        if rope is None:
            A.attn_backward(q, k, v, out, dout, lse, *g, n, n, H, G, D, CAUSAL, prec, 0)
        else:
            A.attn_backward_rope(q, k, v, out, dout, lse, *g, n, n, H, G, D, CAUSAL, prec, 0, rope)
        return g
    ref = grads()
    box = []
    peak = with_workspace(A, need, lambda: box.append(grads()))
    assert peak == 0
    for a, b in zip(box[0], ref):
        assert torch.equal(a, b)


def test_short_or_misaligned_workspace_is_refused(cuda_lib):
    A = cuda_lib
    n, H, G, D = 300, 8, 2, 128
    q, k, v = (dev(x) for x in synthetic.forward_inputs(n, n, H, G, D, seed=34))
    need = A.attn_forward_workspace_bytes(n, n, H, G, D, CAUSAL, BF16, 0, False)
    out = torch.full((n, H * D), float("nan"), device="cuda")
    with pytest.raises(A.AttnError) as e:
        with_workspace(A, need - 1, lambda: forward_call(A, q, k, v, out, None, n, H, G, D, BF16))
    assert e.value.code == A.ATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(A.AttnError) as e:
        A.attn_set_workspace(ws[16:], need)
    assert e.value.code == A.ATTN_ERR_INVALID_ARG
    A.attn_set_workspace(None)
