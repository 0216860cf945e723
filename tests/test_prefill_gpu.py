"""attn_prefill on the GPU against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

from attention_gqa_online_gb300 import synthetic
from helpers import BF16, FP32, TF32, assert_out_close, dev, tc_supported

pytestmark = pytest.mark.gpu
PRECS = [FP32, TF32, BF16]


def check(A, orc, n_queries, H, G, D, kv_dim, max_seq, start_pos, q_stride, out_stride, q_base, prec, seed,
          q_rows=None, scale=None):
    q_rows = q_rows or (q_base + n_queries)
    qb, kc, vc = synthetic.prefill_inputs(q_rows, q_stride, max_seq, kv_dim, seed=seed)
    scale = np.float32(1.0 / math.sqrt(D)) if scale is None else np.float32(scale)
    sentinel = 12345.0
    out = torch.full((q_rows, out_stride), sentinel, device="cuda")
    A.attn_prefill(dev(qb), dev(kc), dev(vc), out, n_queries, H, G, D, kv_dim, max_seq, float(scale), start_pos,
                   q_stride, out_stride, q_base, prec)
    torch.cuda.synchronize()
    assert A.attn_get_status() == 0
    got = out.cpu().numpy()
    ref = orc.prefill(qb.numpy(), kc.numpy(), vc.numpy(), q_rows, n_queries, H, G, D, kv_dim, max_seq, scale,
                      start_pos, q_stride, out_stride, q_base)
    written = np.zeros_like(got, dtype=bool)
    written[q_base:q_base + n_queries, :H * D] = True
    assert np.all(got[~written] == sentinel), "prefill wrote outside its rows / head columns"
    where = "nq%d H%d G%d D%d start%d qbase%d" % (n_queries, H, G, D, start_pos, q_base)
    assert_out_close(got[written].reshape(n_queries, H * D), ref[written].reshape(n_queries, H * D), prec,
                     float(vc.abs().max()), where)


@pytest.mark.parametrize("prec", PRECS)
def test_prefill_config(cuda_lib, orc, prec):
    """512 queries from start_pos 1536 into a 2048-row cache, 32 heads over 8, D=128."""
    check(cuda_lib, orc, 512, 32, 8, 128, 1024, 2048, 1536, 4096, 4096, 0, prec, seed=0)


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("n_queries,H,G,D,kv_dim,max_seq,start_pos,q_stride,out_stride,q_base", [
    (37, 6, 2, 80, 200, 300, 100, 500, 520, 5),     # gs = 3, padded strides, q_base
    (64, 32, 8, 128, 1024, 128, 0, 4096, 4096, 64),  # start 0, q_base 64: window ends at row 127
    (1, 4, 2, 64, 128, 1, 0, 256, 256, 0),          # one query, one-row cache
    (129, 8, 1, 64, 96, 1000, 700, 520, 512, 3),    # gs = 8, kv_dim > G*D
    (50, 2, 2, 12, 30, 80, 25, 30, 24, 2),          # small odd head_dim
    (37, 6, 2, 128, 256, 300, 100, 800, 776, 5),    # gs = 3 on the tensor cores
    (70, 10, 2, 64, 136, 400, 250, 648, 640, 1),    # gs = 5, kv_dim > G*D
])
def test_prefill_shapes(cuda_lib, orc, prec, n_queries, H, G, D, kv_dim, max_seq, start_pos, q_stride,
                        out_stride, q_base):
    if prec != FP32 and not tc_supported(H, G, D):
        pytest.skip("tensor-core precisions need D in {64, 128}")
    check(cuda_lib, orc, n_queries, H, G, D, kv_dim, max_seq, start_pos, q_stride, out_stride, q_base, prec,
          seed=n_queries)


@pytest.mark.parametrize("prec", PRECS)
def test_prefill_scale_argument(cuda_lib, orc, prec):
    check(cuda_lib, orc, 40, 4, 2, 64, 128, 100, 30, 256, 256, 0, prec, seed=9, scale=0.37)
