"""Paged-cache entry points (attn_decode_paged, attn_prefill_paged) on the GPU
against the oracle, which gathers the logical cache through the block table
and runs the contiguous computation.

Pools hold the cache's pages in shuffled order among spare pages filled with
NaN that the table never names, so a wrong page or row shows up as NaN or as
a mismatch.
"""
import math

import numpy as np
import pytest
import torch

from helpers import BF16, FP32, TF32, assert_out_close, dev

pytestmark = pytest.mark.gpu
PRECS = [FP32, TF32, BF16]


def paged_pool(seed, max_blocks, page_rows, kv_dim, spare=5):
    """(pool K, pool V, block table): logical page b sits in pool page table[b]."""
    rng = np.random.default_rng(seed)
    num_pages = max_blocks + spare
    table = rng.permutation(num_pages)[:max_blocks].astype(np.uint32)
    kp = np.full((num_pages * page_rows, kv_dim), np.nan, np.float32)
    vp = np.full((num_pages * page_rows, kv_dim), np.nan, np.float32)
    for b in range(max_blocks):
        rows = slice(int(table[b]) * page_rows, (int(table[b]) + 1) * page_rows)
        kp[rows] = rng.standard_normal((page_rows, kv_dim))
        vp[rows] = rng.standard_normal((page_rows, kv_dim))
    return kp, vp, table, num_pages


def table_dev(table):
    return torch.from_numpy(table.astype(np.int64)).to(torch.int32).cuda()


@pytest.mark.parametrize("H,G,D,page_rows,max_blocks", [
    (32, 8, 128, 32, 128),   # split kernel, 32-row pages
    (32, 8, 128, 256, 16),   # split kernel, 256-row pages
    (16, 2, 64, 64, 40),     # split kernel, gs = 8
    (6, 2, 80, 16, 30),      # generic kernel (D = 80, 16-row pages)
    (64, 8, 128, 64, 20),    # split kernel, gs = 8 at D = 128 (two head groups)
])
def test_decode_paged(cuda_lib, orc, H, G, D, page_rows, max_blocks):
    kp, vp, table, num_pages = paged_pool(H + page_rows, max_blocks, page_rows, G * D)
    cap = page_rows * max_blocks
    q = np.random.default_rng(5).standard_normal((1, H * D)).astype(np.float32)
    ws = torch.zeros(cuda_lib.attn_decode_workspace_bytes(H, G, D, cap), dtype=torch.uint8, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    dq, dk, dv, dt = dev(torch.from_numpy(q)), dev(torch.from_numpy(kp)), dev(torch.from_numpy(vp)), table_dev(table)
    vmax = float(np.nanmax(np.abs(vp)))
    for kv_pos, w in ((0, 0), (31, 0), (32, 0), (cap // 3, 0), (cap - 1, 0), (cap - 1, 100), (cap // 2, 33)):
        pos.fill_(kv_pos)
        out = torch.full((1, H * D), float("nan"), device="cuda")
        cuda_lib.attn_decode_paged(dq, dk, dv, dt, pos, out, H, G, D, page_rows, num_pages, max_blocks, ws,
                                   window=w)
        torch.cuda.synchronize()
        assert cuda_lib.attn_get_status() == 0
        ref = orc.decode_paged(q, kp, vp, table, kv_pos, H, G, D, page_rows, window=w)
        assert_out_close(out.cpu().numpy(), ref, FP32, vmax, "paged decode P%d kv_pos=%d window=%d" % (
            page_rows, kv_pos, w))


def test_decode_paged_shared_and_bad_pages(cuda_lib, orc):
    """Two table entries naming one page; then an entry past the pool, which
    reads as zeros and records ATTN_ERR_INVALID_ARG."""
    H, G, D, P = 32, 8, 128, 32
    kp, vp, table, num_pages = paged_pool(9, 8, P, G * D)
    table[5] = table[2]
    q = np.random.default_rng(6).standard_normal((1, H * D)).astype(np.float32)
    ws = torch.zeros(cuda_lib.attn_decode_workspace_bytes(H, G, D, 8 * P), dtype=torch.uint8, device="cuda")
    pos = torch.full((1,), 8 * P - 1, dtype=torch.int32, device="cuda")
    out = torch.empty((1, H * D), device="cuda")
    args = (dev(torch.from_numpy(q)), dev(torch.from_numpy(kp)), dev(torch.from_numpy(vp)))
    cuda_lib.attn_decode_paged(*args, table_dev(table), pos, out, H, G, D, P, num_pages, 8, ws)
    assert cuda_lib.attn_get_status() == 0
    ref = orc.decode_paged(q, kp, vp, table, 8 * P - 1, H, G, D, P)
    assert_out_close(out.cpu().numpy(), ref, FP32, float(np.nanmax(np.abs(vp))), "shared page")
    bad = table.copy()
    bad[3] = num_pages + 7
    cuda_lib.attn_decode_paged(*args, table_dev(bad), pos, out, H, G, D, P, num_pages, 8, ws)
    assert cuda_lib.attn_get_status() == cuda_lib.ATTN_ERR_INVALID_ARG
    assert np.all(np.isfinite(out.cpu().numpy()))


def check_prefill_paged(A, orc, n_queries, H, G, D, kv_dim, page_rows, max_blocks, start_pos, q_stride, q_base, prec,
                        window, seed):
    kp, vp, table, num_pages = paged_pool(seed, max_blocks, page_rows, kv_dim)
    q_rows = q_base + n_queries
    qb = np.random.default_rng(seed + 1).standard_normal((q_rows, q_stride)).astype(np.float32)
    scale = np.float32(1.0 / math.sqrt(D))
    out = torch.full((q_rows, q_stride), 12345.0, device="cuda")
    A.attn_prefill_paged(dev(torch.from_numpy(qb)), dev(torch.from_numpy(kp)), dev(torch.from_numpy(vp)),
                         table_dev(table), out, n_queries, H, G, D, kv_dim, page_rows, num_pages, max_blocks,
                         float(scale), start_pos, q_stride, q_stride, q_base, prec, window)
    torch.cuda.synchronize()
    assert A.attn_get_status() == 0
    got = out.cpu().numpy()
    ref = orc.prefill_paged(qb, kp, vp, table, q_rows, n_queries, H, G, D, kv_dim, page_rows, scale, start_pos,
                            q_stride, q_stride, q_base, window=window)
    assert np.all(got[:q_base] == 12345.0) and np.all(got[:, H * D:] == 12345.0)
    assert_out_close(got[q_base:, :H * D], ref[q_base:, :H * D], prec, float(np.nanmax(np.abs(vp))),
                     "paged prefill P%d prec%d window%d" % (page_rows, prec, window))


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("page_rows,window", [(32, 0), (64, 300), (128, 0), (256, 0), (512, 1000)])
def test_prefill_paged_config(cuda_lib, orc, prec, page_rows, window):
    """512 queries from start_pos 1536, capacity 2048, 32 heads over 8, D=128."""
    check_prefill_paged(cuda_lib, orc, 512, 32, 8, 128, 1024, page_rows, 2048 // page_rows, 1536, 4096, 0, prec,
                        window, seed=page_rows + window)


@pytest.mark.parametrize("prec", PRECS)
def test_prefill_paged_ragged(cuda_lib, orc, prec):
    """gs = 8, kv_dim > G*D, q_base 3, 129 queries from start_pos 700 of a 1024-row capacity."""
    check_prefill_paged(cuda_lib, orc, 129, 8, 1, 64, 96, 64, 16, 700, 520, 3, prec, 0, seed=3)


@pytest.mark.parametrize("prec", [TF32, BF16])
def test_prefill_paged_small_pages(cuda_lib, orc, prec):
    """16-row pages: the fp32 kernel takes them; the tensor-core precisions, whose
    tiles follow pages of 32 rows, run on that kernel too (within their bounds)."""
    check_prefill_paged(cuda_lib, orc, 37, 6, 2, 80, 200, 16, 20, 100, 500, 5, FP32, 0, seed=4)
    check_prefill_paged(cuda_lib, orc, 37, 6, 2, 64, 136, 16, 20, 100, 400, 5, prec, 0, seed=6)
